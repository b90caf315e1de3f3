// a3 + a4: sparse MLA attention over the top-k rows of the paged bf16 latent
// cache, with split-KV partials and their online-softmax merge
// (vLLM PR #38476, Changes 3: split-KV decode with an N-way online-softmax
// merge, a single-pass path, and a finite -1e30 sentinel for masked slots).
//
// For query token t and head h:
//   s_i = scale * q[t,h,:] . kv[i,:]          over the selected rows i
//   out = sum_i softmax(s)_i * kv[i, :Dv]     lse = log sum_i exp(s_i)
//
// The 128 heads are the MMA M dimension. For Dk = 576 a (token, split) is
// one 2-CTA cluster: CTA r owns K-blocks (64 dims each) [4r, 4r+4) and half
// of the rope dims, [512+32r, 544+32r), of every row, gathers only those
// (4-row TMA gathers through the block table, 576 bytes of each row per CTA;
// empty or invalid slots read as zeros and score the sentinel with weight 0),
// and owns value dims [256r, 256r+256), which are its four K-blocks.
// Per 64-key tile, in each CTA:
//   S_r = Q_r K_r^T   tcgen05 kind::f16, M=128, N=64, A (this CTA's q dims)
//                     in tensor memory, B from the swizzled KV stage;
//   exchange          S_r, scaled by softmax_scale * log2(e), goes to the peer
//                     in fp32 over DSMEM (st.async); both CTAs form
//                     S = S_0 + S_1 (log2 units) and agree bit for bit;
//   softmax           thread = head row; two warp groups take alternate
//                     tiles; lazy rescaling of O (only when the row maximum
//                     grows by more than 2^8);
//   O_r += P V_r      M=128, N=256, A = P (bf16) in tensor memory, fp32
//                     accumulator in tensor memory.
// Warp roles: 8 softmax/epilogue warps, 4 producer warps (TMA), 1 MMA warp.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "ptx.cuh"

namespace dsa {
namespace {

using namespace ptx;

constexpr int kThreads = 416;  // warps 0-7 softmax/epilogue, warps 8-11 loads, warp 12 MMA
constexpr int kProdWarp0 = 8;
constexpr int kMmaWarp = 12;
constexpr int kTileKeys = 64;
constexpr int kStages = 4;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.f;  // log2 units
constexpr int kMaxSlots = 2048;           // top-k slots one CTA (one split) may cover
constexpr int kXBufs = 2;                 // score-exchange buffers, one per softmax group
constexpr long long kWaitLimitCycles = 2000000000ll;
static_assert(kMaxSlots <= 256 * 8, "the softmax warps resolve all slots in one pass");
constexpr int kXRow = 64 * 4;             // bytes of one row's 64 fp32 scores in an exchange buffer
constexpr int kXChunk = 128 * 16;         // stride of a 16-byte chunk column (128 rows) in an exchange buffer

// kPair: the two CTAs of a cluster split the Dk dims and the value dims:
// rank r owns value dims [r*kDvc, (r+1)*kDvc) = K-blocks [4r, 4r+4) (64 dims
// each), and half of the rope dims, [512 + 32r, 544 + 32r), which enter QK
// only; both gather 576 bytes of every row. They exchange partial scores
// through DSMEM.
template <int DK, int DV>
struct MlaCfg;
template <>
struct MlaCfg<576, 512> {
  static constexpr bool kPair = true;
  static constexpr int kNkb = 4, kMaxNkb = 4, kDvc = 256, kTmemCols = 512;
  static constexpr bool kRopeHalf = true;  // plus a 32-dim rope half-block (64-byte rows)
  static constexpr int kRopeX = 512;       // first rope dim
};
template <>
struct MlaCfg<80, 64> {
  static constexpr bool kPair = false;
  static constexpr int kNkb = 2, kMaxNkb = 2, kDvc = 64, kTmemCols = 256;
  static constexpr bool kRopeHalf = false;
  static constexpr int kRopeX = 0;
};

// Shared-memory layout. F8: the latent cache is fp8 (e4m3 codes in groups of
// 128 dims with an fp32 scale each, then the rope dims in bf16); its codes
// and scales are gathered into raw stages and dequantised by the producer
// warps into the bf16 operand stages the MMAs read.
template <int DK, int DV, bool F8>
struct MlaSmem {
  using C = MlaCfg<DK, DV>;
  static constexpr int kBStages = F8 ? 3 : kStages;  // bf16 operand stages
  static constexpr int kRStages = F8 ? 2 : 0;        // raw fp8 stages (codes + scales)
  static constexpr int kQStage = F8 ? 1 : 2;         // q is staged in bf16 stages kQStage, kQStage + 1
  static constexpr int kKvKb = kTileKeys * 128;  // one 64-dim K-block of a KV tile
  static constexpr int kKvHalf = C::kMaxNkb * kKvKb;  // the rope half-block: 64 keys x 64 B (SWIZZLE_64B)
  static constexpr int kKvStage = kKvHalf + (C::kRopeHalf ? kTileKeys * 64 : 0);
  static constexpr int kQHalf = C::kRopeHalf ? 128 * 64 : 0;  // q's rope half: 128 heads x 64 B
  static constexpr int kRawCodes = kTileKeys * 256;  // this CTA's 256 codes of each key
  // then the keys' four group scales (16 bytes a key); a 4-row gather writes
  // 64 bytes, and tensor copies need 128-byte aligned destinations, so each
  // group of 4 keys takes a 128-byte slot
  static constexpr int kRawScaleSlot = 128;
  static constexpr int kRawStage = kRawCodes + (kTileKeys / 4) * kRawScaleSlot;
  static constexpr int kKv = 0;
  static constexpr int kRaw = kKv + kBStages * kKvStage;
  static constexpr int kX = kRaw + kRStages * kRawStage;  // [kKv, kX) is idle at write-out
  static constexpr int kXBuf = 128 * kXRow;
  static constexpr int kRow = kX + (C::kPair ? kXBufs * kXBuf : 0);
  static constexpr int kLive = kRow + kMaxSlots * 4;
  static constexpr int kCoordStages = F8 ? kRStages : 0;  // gather rows of the fp8 producer's raw stages
  static constexpr int kCoord = kLive + kBStages * 4 * 2;
  static constexpr int kRed = kCoord + kCoordStages * kTileKeys * 4;
  static constexpr int kTotal = kRed + 6 * 128 * 4 + 1024;
  static_assert(C::kMaxNkb * 16384 + kQHalf <= 2 * kKvStage, "q staging does not fit in two KV stages");
  static_assert(kQStage + 2 <= kBStages, "q staging needs two bf16 stages");
  static_assert(!F8 || (C::kPair && C::kNkb == 4), "the fp8 cache is read by the paired 576/512 kernel only");
  // every TMA destination is 128-byte aligned (stages are 1024-byte multiples)
  static_assert(kKvStage % 1024 == 0 && kRawStage % 1024 == 0 && kRawCodes % 128 == 0 && kRaw % 1024 == 0,
                "TMA destinations must stay 128-byte aligned");
};

struct MlaParams {
  int32_t num_blocks, rows_per_block, total_rows;
  const int32_t* block_table;
  int32_t bt_stride;
  const int32_t* seq_lens;
  const int32_t* qsl;
  const int32_t* topk;
  int32_t B, T, H, K, block_size, splits, per_split;
  float scale_log2;
  uint16_t* out;    // bf16 [T, H, DV]
  float* lse;       // [T, H] or null
  float* o_part;    // [T, H, S, DV]
  float2* ml_part;  // [T, H, S] (max in log2 units, sum)
  int32_t* dev_status;
};

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ int find_request(const int32_t* qsl, int B, int t) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(qsl + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// e4m3 pair (low byte = first value) -> two bf16 of code * scale, packed
// with the first value in the low half.
__device__ __forceinline__ uint32_t dequant_e4m3x2(uint32_t two, float sc) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(static_cast<uint16_t>(two)));
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
  return pack_bf16(f.x * sc, f.y * sc);
}

template <int DK, int DV, bool F8>
__global__ void __launch_bounds__(kThreads, 1) sparse_mla_kernel(const __grid_constant__ MlaParams p,
                                                                 const __grid_constant__ CUtensorMap qmap,
                                                                 const __grid_constant__ CUtensorMap kvmap,
                                                                 const __grid_constant__ CUtensorMap qmap64,
                                                                 const __grid_constant__ CUtensorMap kvmap64,
                                                                 const __grid_constant__ CUtensorMap scmap) {
  // F8: kvmap = the cache rows' code bytes (256-byte boxes), kvmap64 = their
  // rope dims (bf16, 64-byte boxes, SWIZZLE_64B), scmap = their 16 scale bytes
  using C = MlaCfg<DK, DV>;
  using L = MlaSmem<DK, DV, F8>;
  constexpr int kBS = L::kBStages;
  constexpr int kSplitDv = C::kPair ? 2 : 1;
  // tensor-memory columns: S (fp32), O (fp32), Q (bf16 pairs), P (bf16 pairs)
  constexpr uint32_t kColS = 0, kColO = kTileKeys, kColQ = kTileKeys + C::kDvc;
  constexpr uint32_t kColP = kColQ + C::kNkb * 32 + (C::kRopeHalf ? 16 : 0);
  static_assert(kColP + kTileKeys / 2 <= C::kTmemCols, "tensor-memory columns overflow");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t kv_full[kStages], kv_empty[kStages], x_full[kXBufs], x_empty[kXBufs];
  // F8: per raw stage and producer warp, the TMA completion of that warp's
  // codes + scales
  __shared__ uint64_t raw_full[2][4];
  // s_full, o_done and m_bar come in pairs indexed by tile parity, so each
  // softmax group waits on phases of its own tiles only
  __shared__ uint64_t s_full[2], s_free, p_full, o_done[2], o_final, q_full, q_ready, rows_ready, m_bar[2], epi_bar;
  __shared__ uint32_t tmem_holder;
  __shared__ int s_qsl[kThreads + 1], s_sl[kThreads];  // the batch's query_start_loc and seq_lens (B <= kThreads)
  __shared__ int s_last_live;
  __shared__ volatile int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = C::kPair ? static_cast<int>(cluster_ctarank()) : 0;
  const int j = (blockIdx.x / kSplitDv) % p.splits;
  const int t = blockIdx.x / (kSplitDv * p.splits);
  const int kb0 = r * C::kNkb;                     // first K-block (64 dims) this CTA owns
  constexpr int nkb = C::kNkb;                     // K-blocks this CTA owns
  const int rope_x = C::kRopeX + 32 * r;           // its rope half (dims of q), when there is one
  // ... and the same dims in a cache row: bf16 element 512 + 32 r of a bf16
  // row; in an fp8 row the rope follows DV code bytes and DV / 128 scales
  const int rope_kv = F8 ? (DV + 4 * (DV / 128)) / 2 + 32 * r : rope_x;

  uint8_t* kv_sm = smem + L::kKv;
  uint8_t* x_sm = smem + L::kX;
  int* row_sm = reinterpret_cast<int*>(smem + L::kRow);
  uint16_t* live_m = reinterpret_cast<uint16_t*>(smem + L::kLive);  // [stage][producer warp]: live-key bits
  int* coord_sm = reinterpret_cast<int*>(smem + L::kCoord);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      // the four producer warps; F8: each arrives twice, when it issues the
      // stage's rope gather (with its bytes) and when its keys are dequantised
      mbar_init(&kv_full[s], F8 ? 8 : 4);
      mbar_init(&kv_empty[s], 1);
    }
    if constexpr (F8) {
      for (int w = 0; w < 4; ++w)
        for (int s = 0; s < 2; ++s) mbar_init(&raw_full[s][w], 1);
    }
    for (int s = 0; s < kXBufs; ++s) {
      mbar_init(&x_full[s], 1);   // local expect_tx; the peer's st.async deliver the bytes
      mbar_init(&x_empty[s], 4);  // the peer's four reading warps, remotely
    }
    mbar_init(&s_free, 4);
    mbar_init(&p_full, 4);
    mbar_init(&o_final, 1);
    mbar_init(&q_full, 1);
    mbar_init(&q_ready, 8);
    mbar_init(&rows_ready, 8);
    for (int q = 0; q < 2; ++q) {
      mbar_init(&s_full[q], 1);
      mbar_init(&o_done[q], 1);
      mbar_init(&m_bar[q], 4);
    }
    mbar_init(&epi_bar, 256);
    fence_mbar_init();
    s_last_live = -1;
    s_abort = 0;
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&tmem_holder, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  if constexpr (C::kPair) {
    cluster_sync_all();  // both CTAs' barriers exist before any remote arrival
  } else {
    __syncthreads();
  }
  tc_fence_after();
  const uint32_t tmem = tmem_holder;

  // Launched as a programmatic dependent of the top-k. q, query_start_loc and
  // seq_lens are inputs of the step that no kernel of the library writes, so
  // this CTA's q K-blocks (by TMA, into KV stages kQStage..., which tiles 0
  // and 1 leave untouched) and the token's request are fetched before the
  // wait, overlapping the top-k's tail; the top-k slots are read after it.
  uint8_t* q_stage = kv_sm + L::kQStage * L::kKvStage;
  if (tid == kProdWarp0 * 32) {  // first producer thread
    prefetch_tmap(&qmap);
    prefetch_tmap(&kvmap);
    if constexpr (C::kRopeHalf) {
      prefetch_tmap(&qmap64);
      prefetch_tmap(&kvmap64);
    }
    if constexpr (F8) prefetch_tmap(&scmap);
    mbar_arrive_expect_tx(&q_full, nkb * 16384 + L::kQHalf);
    for (int kb = 0; kb < nkb; ++kb)
      tma_load_3d(smem_u32(q_stage + kb * 16384), &qmap, &q_full, (kb0 + kb) * 64, 0, t);
    if constexpr (C::kRopeHalf) tma_load_3d(smem_u32(q_stage + nkb * 16384), &qmap64, &q_full, rope_x, 0, t);
  }
  // the request of token t: the last b with query_start_loc[b] <= t, found in
  // one round of loads when the batch has at most kThreads requests
  int b, q0, q1, sl_b;
  if (p.B <= kThreads) {
    const int qv = tid <= p.B ? __ldg(p.qsl + tid) : 0;
    const int sv = tid < p.B ? __ldg(p.seq_lens + tid) : 0;
    if (tid <= p.B) s_qsl[tid] = qv;
    if (tid < p.B) s_sl[tid] = sv;
    b = max(0, __syncthreads_count(tid < p.B && qv <= t) - 1);
    q0 = s_qsl[b];
    q1 = s_qsl[b + 1];
    sl_b = s_sl[b];
  } else {
    b = find_request(p.qsl, p.B, t);
    q0 = __ldg(p.qsl + b);
    q1 = __ldg(p.qsl + b + 1);
    sl_b = __ldg(p.seq_lens + b);
  }
  int64_t valid64 = static_cast<int64_t>(sl_b) - (q1 - q0) + (t - q0) + 1;
  const int64_t cap = static_cast<int64_t>(p.bt_stride) * p.block_size;
  if (valid64 > cap || valid64 < 1) {
    if (tid == 0 && r == 0 && j == 0) report(p.dev_status, DSA_DEVERR_SEQ_LEN);
    valid64 = max(static_cast<int64_t>(0), min(valid64, cap));
  }
  const int valid = static_cast<int>(valid64);

  asm volatile("griddepcontrol.wait;" ::: "memory");  // the top-k's results are visible from here on
  const int slot0 = j * p.per_split;
  const int n_slots = max(0, min(p.K, slot0 + p.per_split) - slot0);
  const int32_t* idx_row = p.topk + static_cast<int64_t>(t) * p.K + slot0;
  int idx[8];
  if (warp < 8) {
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int sl = u * 256 + tid;
      idx[u] = sl < n_slots ? __ldg(idx_row + sl) : -1;
    }
  }

  auto abort_now = [&](void) {
    s_abort = 1;
    report(p.dev_status, DSA_DEVERR_TIMEOUT);
  };

  if (warp < 8) {
    // the split's top-k slots -> physical rows (-1: empty or invalid)
    const int32_t* bt_row = p.block_table + static_cast<int64_t>(b) * p.bt_stride;
    int blk[8];
#pragma unroll
    for (int u = 0; u < 8; ++u)
      blk[u] = (idx[u] >= 0 && idx[u] < valid) ? __ldg(bt_row + idx[u] / p.block_size) : -1;
    int last = -1;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int sl = u * 256 + tid;
      if (sl >= n_slots) continue;
      int row = -1;
      if (idx[u] >= 0 && idx[u] < valid) {
        if (blk[u] >= 0 && blk[u] < p.num_blocks)
          row = blk[u] * p.rows_per_block + idx[u] % p.block_size;
        else if (r == 0)
          report(p.dev_status, DSA_DEVERR_BLOCK_OOB);
      } else if (idx[u] != -1 && r == 0) {
        report(p.dev_status, DSA_DEVERR_INDEX_OOB);
      }
      row_sm[sl] = row;
      if (row >= 0) last = sl;
    }
    if (last >= 0) atomicMax(&s_last_live, last);
    __syncwarp();
    if (lane == 0) mbar_arrive(&rows_ready);
    // this CTA's q dims -> tensor memory (A operand of QK)
    if (!mbar_wait(&q_full, 0)) {
      if (lane == 0) abort_now();
    } else {
      const int hq = (warp & 3) * 32 + lane;
      const uint32_t lane_q = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + kColQ;
#pragma unroll 1
      for (int kb = warp >> 2; kb < nkb; kb += 2) {  // the two warps of a lane group split the K-blocks
        uint32_t v[16];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 u = *reinterpret_cast<const uint4*>(q_stage + kb * 16384 + sw128_offset(hq, half * 4 + c));
            v[4 * c] = u.x;
            v[4 * c + 1] = u.y;
            v[4 * c + 2] = u.z;
            v[4 * c + 3] = u.w;
          }
          tmem_st16(lane_q + kb * 32 + half * 16, v);
        }
      }
      if constexpr (C::kRopeHalf) {
        if (warp >> 2 == (nkb & 1)) {  // the rope half: 64-byte rows, chunk c at c ^ ((row >> 1) & 3)
          uint32_t v[16];
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 u = *reinterpret_cast<const uint4*>(q_stage + nkb * 16384 + hq * 64 + ((c ^ ((hq >> 1) & 3)) << 4));
            v[4 * c] = u.x;
            v[4 * c + 1] = u.y;
            v[4 * c + 2] = u.z;
            v[4 * c + 3] = u.w;
          }
          tmem_st16(lane_q + nkb * 32, v);
        }
      }
      tmem_st_wait();
      fence_proxy_async_smem();  // the staging stages are refilled by TMA next
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&q_ready);
  }
  if (!mbar_wait(&rows_ready, 0) && lane == 0) abort_now();
  const int n_tiles = s_abort ? 0 : (s_last_live + kTileKeys) / kTileKeys;

  if (F8 && warp >= kProdWarp0 && warp < kMmaWarp) {
    // ---------------- fp8 producer: 4 warps, 16 keys each. Codes + scales of
    // tile i go by 4-row TMA gathers into raw stage i % 2 two tiles ahead;
    // when bf16 stage i % 3 is free its rope half is gathered straight into
    // it (the bytes counted on the stage's barrier, which the MMA waits for),
    // the warp dequantises its 16 keys (code * group scale -> bf16, in the
    // MMA's swizzled layout), hands its part of the stage to the MMA and
    // gathers tile i + 2's codes.
    const int pw = warp - kProdWarp0;
    const int g = pw * 4 + (lane & 3);  // 4-row group a gathering lane issues
    uint32_t live_bits0 = 0u, live_bits1 = 0u;  // live-key bits of the tiles in raw stages 0 and 1
    int codes_issued = 0, codes_done = 0;
    int open_stage = -1;  // a tile whose rope this warp gathered but whose stage it has not handed over
    auto issue_codes = [&](int i) {
      const int rst = i & 1;
      bool live = false;
      if (lane < 16) {
        const int kr = pw * 16 + lane;
        const int sl = i * kTileKeys + kr;
        const int row = sl < n_slots ? row_sm[sl] : -1;
        live = row >= 0;
        coord_sm[rst * kTileKeys + kr] = live ? row : p.total_rows;  // out of range: zero fill
      }
      const uint32_t bits = __ballot_sync(0xFFFFFFFFu, live) & 0xFFFFu;
      if (rst) live_bits1 = bits; else live_bits0 = bits;
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(&raw_full[rst][pw], 16 * (256 + 16));
      __syncwarp();
      const int* cs = coord_sm + rst * kTileKeys + 4 * g;
      uint8_t* raw = smem + L::kRaw + rst * L::kRawStage;
      if (lane < 4)
        tma_gather4(smem_u32(raw + g * 4 * 256), &kvmap, &raw_full[rst][pw], 256 * r, cs[0], cs[1], cs[2], cs[3]);
      else if (lane < 8)
        tma_gather4(smem_u32(raw + L::kRawCodes + g * L::kRawScaleSlot), &scmap, &raw_full[rst][pw], DV, cs[0], cs[1],
                    cs[2], cs[3]);
      codes_issued = i + 1;
    };
    for (int i = 0; i < min(2, n_tiles); ++i) issue_codes(i);
    for (int i = 0; i < n_tiles && !s_abort; ++i) {
      const int bst = i % kBS, rst = i & 1;
      if (i >= kBS && !mbar_wait(&kv_empty[bst], ((i / kBS) - 1) & 1)) {
        if (lane == 0) abort_now();
        break;
      }
      if (i == L::kQStage && !mbar_wait(&q_ready, 0)) {  // q has left its staging stages
        if (lane == 0) abort_now();
        break;
      }
      uint8_t* stage = kv_sm + bst * L::kKvStage;
      // the rope half of this warp's keys, straight into the bf16 stage
      if (lane == 0) mbar_arrive_expect_tx(&kv_full[bst], 16 * 64);
      __syncwarp();
      if (lane < 4) {
        const int* cs = coord_sm + rst * kTileKeys + 4 * g;
        tma_gather4(smem_u32(stage + L::kKvHalf + g * 256), &kvmap64, &kv_full[bst], rope_kv, cs[0], cs[1], cs[2],
                    cs[3]);
      }
      open_stage = i;
      if (!mbar_wait(&raw_full[rst][pw], (i >> 1) & 1)) {
        if (lane == 0) abort_now();
        break;
      }
      codes_done = i + 1;
      {
        // lane: key pw * 16 + lane / 2, group lane % 2 of this CTA's two
        // 128-dim groups (K-blocks 2 grp, 2 grp + 1); 16 codes per step, the
        // step order rotated by lane so that a quarter-warp's loads hit
        // distinct banks
        const int k = pw * 16 + (lane >> 1), grp = lane & 1;
        const uint8_t* raw = smem + L::kRaw + rst * L::kRawStage;
        const uint8_t* src = raw + k * 256 + grp * 128;
        const float sc = *reinterpret_cast<const float*>(raw + L::kRawCodes + (k >> 2) * L::kRawScaleSlot +
                                                         (k & 3) * 16 + (2 * r + grp) * 4);
        uint8_t* dst = stage + (2 * grp) * L::kKvKb + k * 128;
        const uint32_t sw = static_cast<uint32_t>(k & 7);
#pragma unroll 2
        for (int step = 0; step < 8; ++step) {
          const int jj = (step + lane) & 7;  // dims 16 jj .. 16 jj + 15 of the group
          const uint4 c = *reinterpret_cast<const uint4*>(src + jj * 16);
          uint8_t* kb = dst + (jj >> 2) * L::kKvKb;
          const uint32_t c0 = 2u * static_cast<uint32_t>(jj & 3);
          *reinterpret_cast<uint4*>(kb + ((c0 ^ sw) << 4)) =
              make_uint4(dequant_e4m3x2(c.x, sc), dequant_e4m3x2(c.x >> 16, sc), dequant_e4m3x2(c.y, sc),
                         dequant_e4m3x2(c.y >> 16, sc));
          *reinterpret_cast<uint4*>(kb + (((c0 + 1u) ^ sw) << 4)) =
              make_uint4(dequant_e4m3x2(c.z, sc), dequant_e4m3x2(c.z >> 16, sc), dequant_e4m3x2(c.w, sc),
                         dequant_e4m3x2(c.w >> 16, sc));
        }
      }
      if (lane == 0) live_m[bst * 4 + pw] = static_cast<uint16_t>(rst ? live_bits1 : live_bits0);
      fence_proxy_async_smem();  // the MMA reads the stage through the async proxy
      __syncwarp();              // every lane is done with raw stage rst
      if (lane == 0) mbar_arrive(&kv_full[bst]);
      open_stage = -1;
      if (i + 2 < n_tiles) issue_codes(i + 2);
    }
    if (s_abort) {
      // let this warp's gathers in flight land before shared memory is given
      // up: its codes on its own barriers; a rope gather by completing this
      // warp's arrivals on the stage's barrier and waiting for the phase
      for (int i = codes_done; i < codes_issued; ++i) mbar_wait(&raw_full[i & 1][pw], (i >> 1) & 1, 20000000ll);
      if (open_stage >= 0) {
        if (lane == 0) mbar_arrive(&kv_full[open_stage % kBS]);
        mbar_wait(&kv_full[open_stage % kBS], (open_stage / kBS) & 1, 20000000ll);
      }
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  } else if (warp >= kProdWarp0 && warp < kMmaWarp) {
    // ---------------- producer: 4 warps, 16 keys each; 4-row TMA gathers of
    // this CTA's K-blocks only
    const int pw = warp - kProdWarp0;
    const uint32_t tile_bytes = kTileKeys * (nkb * 128 + (C::kRopeHalf ? 64 : 0));
    int issued = 0;
    // row of key pw * 16 + lane of the next tile (lanes 0-15), read before
    // the wait for its stage
    auto tile_row = [&](int i) {
      const int sl = i * kTileKeys + pw * 16 + lane;
      return (lane < 16 && sl < n_slots) ? row_sm[sl] : -1;
    };
    int row_next = n_tiles > 0 ? tile_row(0) : -1;
    for (int i = 0; i < n_tiles && !s_abort; ++i) {
      const int st = i % kBS;
      const int row = row_next;
      if (i + 1 < n_tiles) row_next = tile_row(i + 1);
      if (i >= kBS && !mbar_wait(&kv_empty[st], ((i / kBS) - 1) & 1)) {
        if (lane == 0) abort_now();
        break;
      }
      if (i == L::kQStage && !mbar_wait(&q_ready, 0)) {  // q has left its staging stages
        if (lane == 0) abort_now();
        break;
      }
      const bool live = row >= 0;
      const int crd = live ? row : p.total_rows;  // out of range: zero fill
      const uint32_t mask = __ballot_sync(0xFFFFFFFFu, live);
      if (lane == 0) live_m[st * 4 + pw] = static_cast<uint16_t>(mask);
      // the 4 rows of gather group lane % 4 of this warp
      const int gs = 4 * (lane & 3);
      const int c0 = __shfl_sync(0xFFFFFFFFu, crd, gs), c1 = __shfl_sync(0xFFFFFFFFu, crd, gs + 1),
                c2 = __shfl_sync(0xFFFFFFFFu, crd, gs + 2), c3 = __shfl_sync(0xFFFFFFFFu, crd, gs + 3);
      if (lane == 0) {
        if (pw == 0) mbar_arrive_expect_tx(&kv_full[st], tile_bytes);
        else mbar_arrive(&kv_full[st]);
      }
      if (lane < 4 * nkb) {
        const int g = pw * 4 + (lane & 3), kb = lane >> 2;
        tma_gather4(smem_u32(kv_sm + st * L::kKvStage + kb * L::kKvKb + g * 512), &kvmap, &kv_full[st],
                    (kb0 + kb) * 64, c0, c1, c2, c3);
      } else if (C::kRopeHalf && lane < 4 * nkb + 4) {  // the rope half of the same 4-row groups
        const int g = pw * 4 + (lane & 3);
        tma_gather4(smem_u32(kv_sm + st * L::kKvStage + L::kKvHalf + g * 256), &kvmap64, &kv_full[st], rope_kv, c0,
                    c1, c2, c3);
      }
      issued = i + 1;
    }
    if (s_abort && pw == 0) {
      // let the gathers in flight land before shared memory is given up
      for (int i = max(0, issued - kBS); i < issued; ++i)
        mbar_wait(&kv_full[i % kBS], (i / kBS) & 1, 20000000ll);
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issuer. QK of tile i needs its KV stage and S of
    // tile i-1 read out; PV of tile i needs P of tile i. The two softmax
    // groups finish their tiles out of step, so whichever is ready goes first.
    if (!mbar_wait(&q_ready, 0) && lane == 0) abort_now();
    tc_fence_after();
    const uint32_t idesc_qk = idesc_bf16(128, kTileKeys, false, false);
    const uint32_t idesc_pv = idesc_bf16(128, C::kDvc, false, true);
    auto issue_qk = [&](int i) {  // this CTA's part of S = Q K^T
      const int st = i % kBS;
      // descriptors differ only in the start-address field (16-byte units)
      const uint64_t d0 = smem_desc(smem_u32(kv_sm + st * L::kKvStage), 16, 1024, kSwizzle128B);
#pragma unroll
      for (int kb = 0; kb < nkb; ++kb) {
#pragma unroll
        for (int k4 = 0; k4 < 4; ++k4)
          mma_bf16_ts(tmem + kColS, tmem + kColQ + (kb * 4 + k4) * 8,
                      d0 + static_cast<uint64_t>((kb * L::kKvKb + k4 * 32) >> 4), idesc_qk, (kb | k4) ? 1u : 0u);
      }
      if constexpr (C::kRopeHalf) {  // 64-byte rows: SWIZZLE_64B, 8-row groups 512 bytes apart
        const uint64_t dh = smem_desc(smem_u32(kv_sm + st * L::kKvStage + L::kKvHalf), 16, 512, kSwizzle64B);
#pragma unroll
        for (int k2 = 0; k2 < 2; ++k2)
          mma_bf16_ts(tmem + kColS, tmem + kColQ + (nkb * 4 + k2) * 8, dh + static_cast<uint64_t>((k2 * 32) >> 4),
                      idesc_qk, 1u);
      }
      mma_commit(&s_full[i & 1]);
    };
    auto issue_pv = [&](int i) {  // O += P V
      const int st = i % kBS;
      // value dims = this CTA's first K-blocks
      const uint64_t vd = smem_desc(smem_u32(kv_sm + st * L::kKvStage), L::kKvKb, 1024, kSwizzle128B);
      // A = P from tensor memory: 16 keys (8 columns of bf16 pairs) per MMA
#pragma unroll
      for (int ks = 0; ks < kTileKeys / 16; ++ks)
        mma_bf16_ts(tmem + kColO, tmem + kColP + ks * 8, vd + static_cast<uint64_t>((ks * 2048) >> 4), idesc_pv,
                    (i > 0 || ks > 0) ? 1u : 0u);
      mma_commit(&kv_empty[st]);
      mma_commit(&o_done[i & 1]);
      if (i == n_tiles - 1) mma_commit(&o_final);
    };
    int nq = 0, np = 0;  // next tile to issue QK / PV for
    long long idle_since = clock64();
    while (np < n_tiles && !s_abort) {
      bool progressed = false;
      if (nq < n_tiles) {
        const int st = nq % kBS;
        bool ready = mbar_test_wait(&kv_full[st], (nq / kBS) & 1) &&
                     (nq == 0 || mbar_test_wait(&s_free, (nq - 1) & 1));
        ready = __shfl_sync(0xFFFFFFFFu, ready, 0);
        if (ready) {
          tc_fence_after();
          if (lane == 0) issue_qk(nq);
          __syncwarp();
          ++nq;
          progressed = true;
        }
      }
      if (np < nq) {
        const bool ready = __shfl_sync(0xFFFFFFFFu, mbar_test_wait(&p_full, np & 1), 0);
        if (ready) {
          tc_fence_after();
          if (lane == 0) issue_pv(np);
          __syncwarp();
          ++np;
          progressed = true;
        }
      }
      if (progressed) {
        idle_since = clock64();
      } else if (clock64() - idle_since > kWaitLimitCycles) {
        if (lane == 0) abort_now();
        break;
      } else {
        __nanosleep(20);
      }
    }
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  } else {
    // ---------------- softmax: group g = warp / 4 takes the tiles i with
    // i % 2 == g, so the score exchange and loads of one tile overlap the
    // arithmetic of the other; thread = head row h (its TMEM lane), all 64
    // keys of a tile. The running maximum passes from group to group through
    // shared memory, tile by tile.
    const int g = warp >> 2;
    const int h = (warp & 3) * 32 + lane;
    const bool leader = (tid & 127) == 0;
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    float* m_hand = reinterpret_cast<float*>(smem + L::kRed);  // [group][row]: m after the group's latest tile
    // this group's exchange buffer is chunk-major: 16-byte chunk c (scores
    // 4c..4c+3) of row h sits at c * 2048 + h * 16, so a warp's accesses to
    // one chunk are 512 contiguous bytes
    const uint8_t* x_mine = x_sm + g * L::kXBuf + h * 16;
    uint32_t x_peer = 0, peer_x_full = 0, peer_x_empty = 0;
    if constexpr (C::kPair) {
      x_peer = mapa_shared(smem_u32(x_mine), static_cast<uint32_t>(r ^ 1));
      peer_x_full = mapa_shared(smem_u32(&x_full[g]), static_cast<uint32_t>(r ^ 1));
      peer_x_empty = mapa_shared(smem_u32(&x_empty[g]), static_cast<uint32_t>(r ^ 1));
    }
    float m_own = kNegSentinel, l_part = 0.f;  // l_part is expressed against m_own
    for (int i = g; i < n_tiles && !s_abort; i += 2) {
      const int u = i >> 1;  // tiles this group has finished
      const int st = i % kBS;
      float s[kTileKeys];
      if (!mbar_wait(&s_full[g], u & 1)) {
        if (lane == 0) abort_now();
        break;
      }
      tc_fence_after();
      if constexpr (C::kPair) {
        // this CTA's half-scores, scaled to log2 units, go to the peer in
        // fp32; both CTAs then add the same two fp32 halves (addition is
        // commutative) and agree bit for bit
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t sv[32];
          tmem_ld32_sync(lane_base + kColS + half * 32, sv);
#pragma unroll
          for (int x = 0; x < 32; ++x) s[half * 32 + x] = __uint_as_float(sv[x]) * p.scale_log2;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_free);
        // the peer has read what this group sent for its previous tile (its
        // reads completed before its arrival, so no acquire is needed here)
        if (u >= 1 && !mbar_wait(&x_empty[g], (u - 1) & 1)) {
          if (lane == 0) abort_now();
          break;
        }
        if (leader) mbar_arrive_expect_tx(&x_full[g], 128 * kXRow);  // the peer's whole tile of half-scores
#pragma unroll
        for (int c = 0; c < 16; ++c)
          st_async_v4(x_peer + c * kXChunk, peer_x_full, __float_as_uint(s[4 * c]), __float_as_uint(s[4 * c + 1]),
                      __float_as_uint(s[4 * c + 2]), __float_as_uint(s[4 * c + 3]));
        if (!mbar_wait_cluster(&x_full[g], u & 1)) {
          if (lane == 0) abort_now();
          break;
        }
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float4 f = *reinterpret_cast<const float4*>(x_mine + c * kXChunk);
          s[4 * c] += f.x;
          s[4 * c + 1] += f.y;
          s[4 * c + 2] += f.z;
          s[4 * c + 3] += f.w;
        }
        // the loaded values are consumed above (the empty asm takes the sum of
        // the last chunk, so it cannot issue before that load has returned),
        // so the loads have completed when the (fence-free) arrival tells the
        // peer it may overwrite them
        asm volatile("" ::"f"(s[kTileKeys - 1]) : "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive_remote_relaxed(peer_x_empty);
      } else {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t sv[32];
          tmem_ld32_sync(lane_base + kColS + half * 32, sv);
#pragma unroll
          for (int x = 0; x < 32; ++x) s[half * 32 + x] = __uint_as_float(sv[x]) * p.scale_log2;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_free);
      }
      if (!mbar_wait(&kv_full[st], (i / kBS) & 1)) {  // orders the producers' live masks
        if (lane == 0) abort_now();
        break;
      }
      const uint64_t live = *reinterpret_cast<const uint64_t*>(live_m + st * 4);
      float mt = -INFINITY;  // the tile's row maximum (log2 units)
#pragma unroll
      for (int x = 0; x < kTileKeys; ++x) {
        if (!((live >> x) & 1u)) s[x] = -INFINITY;
        mt = fmaxf(mt, s[x]);
      }
      float m_prev = kNegSentinel;  // what O and the other group's sum are expressed against
      if (i >= 1) {
        if (!mbar_wait(&m_bar[g ^ 1], ((i - 1) >> 1) & 1)) {
          if (lane == 0) abort_now();
          break;
        }
        m_prev = m_hand[(g ^ 1) * 128 + h];
      }
      const bool rescale = mt > m_prev + kRescaleThreshold;
      const float m_new = rescale ? mt : m_prev;
      m_hand[g * 128 + h] = m_new;
      __syncwarp();
      if (lane == 0) mbar_arrive(&m_bar[g]);
      // masked keys are -inf here and get weight exactly 0
      const float neg_m = -m_new;
      uint32_t pw[32];
      float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
      for (int x = 0; x < 32; ++x) {
        const float a = ex2_approx(s[2 * x] + neg_m);
        const float c = ex2_approx(s[2 * x + 1] + neg_m);
        const __nv_bfloat162 pb = __floats2bfloat162_rn(a, c);
        // the normaliser sums the bf16 weights that the PV product uses
        ps0 += __bfloat162float(pb.x);
        ps1 += __bfloat162float(pb.y);
        pw[x] = *reinterpret_cast<const uint32_t*>(&pb);
      }
      if (m_new != m_own) {
        l_part *= ex2_approx(m_own - m_new);
        m_own = m_new;
      }
      l_part += ps0 + ps1;
      // P and O are free once PV of the previous tile is done
      if (i >= 1) {
        if (!mbar_wait(&o_done[g ^ 1], ((i - 1) >> 1) & 1)) {
          if (lane == 0) abort_now();
          break;
        }
        tc_fence_after();
      }
      tmem_st32(lane_base + kColP, pw);  // this row's 64 weights as 32 bf16 pairs
      if (i >= 1 && __any_sync(0xFFFFFFFFu, rescale)) {
        const float alpha = rescale ? ex2_approx(m_prev - m_new) : 1.f;
#pragma unroll 1
        for (int c = 0; c < C::kDvc; c += 32) {
          uint32_t o[32];
          tmem_ld32_sync(lane_base + kColO + c, o);
#pragma unroll
          for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * alpha);
          tmem_st32(lane_base + kColO + c, o);
        }
      }
      tmem_st_wait();  // P (and a rescaled O) are in tensor memory before PV is issued
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full);
    }

    // ---- epilogue: both groups' sums against the final maximum (the larger
    // of the two, as the maximum only grows); each group writes half of this
    // CTA's value columns
    float* epi = m_hand + 2 * 128;  // [group][m, l][row]
    epi[(2 * g) * 128 + h] = m_own;
    epi[(2 * g + 1) * 128 + h] = l_part;
    bool o_valid = n_tiles > 0 && !s_abort;
    float m_fin = kNegSentinel, l_sum = 0.f;
    mbar_arrive(&epi_bar);
    if (mbar_wait(&epi_bar, 0)) {
      const float m0 = epi[h], l0 = epi[128 + h], m1 = epi[256 + h], l1 = epi[384 + h];
      m_fin = fmaxf(m0, m1);
      l_sum = l0 * ex2_approx(m0 - m_fin) + l1 * ex2_approx(m1 - m_fin);
    } else {
      if (lane == 0) abort_now();
      o_valid = false;
    }
    if (o_valid) {
      if (!mbar_wait(&o_final, 0)) {
        if (lane == 0) abort_now();
        o_valid = false;
      }
    }
    o_valid = __all_sync(0xFFFFFFFFu, o_valid) && !s_abort;
    tc_fence_after();
    const bool have = o_valid && l_sum > 0.f;
    // the merge grid (if any) may launch now; it waits for this grid to finish
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // Write-out through shared memory (the KV stages are idle now): each
    // thread stages its row's half of this CTA's value columns, then each
    // warp stores its 32 rows as contiguous segments, 16 bytes per lane.
    constexpr int kHalf = C::kDvc / 2;
    constexpr int kPitch = kHalf * 4 + 16;  // staged row: fp32 or bf16 values + pad
    static_assert(8 * 32 * kPitch <= L::kX, "write-out staging does not fit");
    const bool final_out = p.splits == 1;  // bf16 output, else fp32 partials
    uint8_t* stg = kv_sm + warp * 32 * kPitch;
    {
      const float inv = have ? 1.f / l_sum : 0.f;
      uint8_t* srow = stg + lane * kPitch;
#pragma unroll 1
      for (int c = 0; c < kHalf; c += 32) {
        uint32_t o[32];
        if (o_valid) tmem_ld32_sync(lane_base + kColO + g * kHalf + c, o);
        if (final_out) {
          uint4* d = reinterpret_cast<uint4*>(srow + c * 2);
#pragma unroll
          for (int x = 0; x < 4; ++x) {
            uint32_t w[4];
#pragma unroll
            for (int y = 0; y < 4; ++y)
              w[y] = have ? pack_bf16(__uint_as_float(o[8 * x + 2 * y]) * inv, __uint_as_float(o[8 * x + 2 * y + 1]) * inv)
                          : 0u;
            d[x] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        } else {
          uint4* d = reinterpret_cast<uint4*>(srow + c * 4);
#pragma unroll
          for (int x = 0; x < 8; ++x)
            d[x] = o_valid ? make_uint4(o[4 * x], o[4 * x + 1], o[4 * x + 2], o[4 * x + 3]) : make_uint4(0u, 0u, 0u, 0u);
        }
      }
    }
    __syncwarp();
    {
      const int chunks = final_out ? kHalf * 2 / 16 : kHalf * 4 / 16;  // 16-byte chunks per row segment
      const int rbase = (warp & 3) * 32;
#pragma unroll 4
      for (int e = lane; e < 32 * chunks; e += 32) {
        const int rr = e / chunks, ch = e - rr * chunks;
        const int hh = rbase + rr;
        if (hh >= p.H) continue;
        const uint4 v = *reinterpret_cast<const uint4*>(stg + rr * kPitch + ch * 16);
        const int64_t row = static_cast<int64_t>(t) * p.H + hh;
        uint8_t* gdst = final_out
                            ? reinterpret_cast<uint8_t*>(p.out + row * DV + r * C::kDvc + g * kHalf)
                            : reinterpret_cast<uint8_t*>(p.o_part + (row * p.splits + j) * DV + r * C::kDvc + g * kHalf);
        *reinterpret_cast<uint4*>(gdst + ch * 16) = v;
      }
    }
    if (r == 0 && g == 0 && h < p.H) {
      const int64_t row = static_cast<int64_t>(t) * p.H + h;
      if (final_out) {
        if (p.lse != nullptr) p.lse[row] = have ? (m_fin + log2f(l_sum)) * kLn2 : -INFINITY;
      } else {
        p.ml_part[row * p.splits + j] = make_float2(o_valid ? m_fin : kNegSentinel, o_valid ? l_sum : 0.f);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (C::kPair) cluster_sync_all();  // no remote access may target an exited CTA
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, C::kTmemCols);
}

// a4: out = sum_j 2^(m_j-M) o_j / sum_j 2^(m_j-M) l_j, M = max_j m_j (log2 units).
// A thread merges 8 consecutive values of one (token, head) row; a block of
// 128 threads covers 128 * 8 / DV rows. Launched as a programmatic dependent
// of the split kernel: it waits for that grid's completion before any read.
// NS > 0: the split count is NS, and every (m, l) pair and partial value of
// the thread is loaded before any arithmetic (one round of L2 reads); NS = 0:
// any split count, split by split. The arithmetic, and so every output bit,
// is the same in both.
template <int NS>
__global__ void __launch_bounds__(128) mla_merge_kernel(const float* __restrict__ o_part,
                                                        const float2* __restrict__ ml, int S, int DV, int64_t n_rows,
                                                        uint16_t* __restrict__ out, float* __restrict__ lse) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if constexpr (NS > 0) S = NS;
  const int tpr = DV / 8;  // threads per row
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (128 / tpr) + threadIdx.x / tpr;
  if (row >= n_rows) return;
  const int v = (threadIdx.x % tpr) * 8;
  const float2* mlr = ml + row * S;
  const float* orow = o_part + row * S * DV + v;
  float M = kNegSentinel;
  float den = 0.f;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  auto add = [&](const float2 mlj, const float4 o0, const float4 o1) {
    const float a = exp2f(mlj.x - M);
    den = fmaf(a, mlj.y, den);
    acc[0] = fmaf(a, o0.x, acc[0]);
    acc[1] = fmaf(a, o0.y, acc[1]);
    acc[2] = fmaf(a, o0.z, acc[2]);
    acc[3] = fmaf(a, o0.w, acc[3]);
    acc[4] = fmaf(a, o1.x, acc[4]);
    acc[5] = fmaf(a, o1.y, acc[5]);
    acc[6] = fmaf(a, o1.z, acc[6]);
    acc[7] = fmaf(a, o1.w, acc[7]);
  };
  if constexpr (NS > 0) {
    float2 mlv[NS];
    float4 o0[NS], o1[NS];
#pragma unroll
    for (int j = 0; j < NS; ++j) {
      mlv[j] = mlr[j];
      o0[j] = *reinterpret_cast<const float4*>(orow + static_cast<int64_t>(j) * DV);
      o1[j] = *reinterpret_cast<const float4*>(orow + static_cast<int64_t>(j) * DV + 4);
    }
#pragma unroll
    for (int j = 0; j < NS; ++j) M = fmaxf(M, mlv[j].x);
#pragma unroll
    for (int j = 0; j < NS; ++j) add(mlv[j], o0[j], o1[j]);
  } else {
    for (int j = 0; j < S; ++j) M = fmaxf(M, mlr[j].x);
#pragma unroll 4
    for (int j = 0; j < S; ++j)
      add(mlr[j], *reinterpret_cast<const float4*>(orow + static_cast<int64_t>(j) * DV),
          *reinterpret_cast<const float4*>(orow + static_cast<int64_t>(j) * DV + 4));
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  uint4 w;
  w.x = pack_bf16(acc[0] * inv, acc[1] * inv);
  w.y = pack_bf16(acc[2] * inv, acc[3] * inv);
  w.z = pack_bf16(acc[4] * inv, acc[5] * inv);
  w.w = pack_bf16(acc[6] * inv, acc[7] * inv);
  *reinterpret_cast<uint4*>(out + row * DV + v) = w;
  if (v == 0 && lse != nullptr) lse[row] = den > 0.f ? (M + log2f(den)) * kLn2 : -INFINITY;
}

FuncAttrOnce g_smem_merge[5];

template <int NS>
dsa_status_t launch_merge_ns(const MlaParams& p, int Dv, float* lse, cudaStream_t s, FuncAttrOnce& once) {
  dsa_status_t st = allow_smem(mla_merge_kernel<NS>, 0, once);
  if (st != DSA_OK) return st;
  const int64_t n_rows = static_cast<int64_t>(p.T) * p.H;
  const int rows_per_block = 128 / (Dv / 8);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((n_rows + rows_per_block - 1) / rows_per_block));
  cfg.blockDim = dim3(128);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, mla_merge_kernel<NS>, static_cast<const float*>(p.o_part),
                                     static_cast<const float2*>(p.ml_part), p.splits, Dv, n_rows, p.out, lse);
  if (e != cudaSuccess) return fail(DSA_ERR_CUDA, "mla_merge_kernel launch failed: %s", cudaGetErrorString(e));
  return DSA_OK;
}

// the split counts the automatic choice gives at decode get their own unrolled merge
dsa_status_t launch_merge(const MlaParams& p, int Dv, float* lse, cudaStream_t s) {
  switch (p.splits) {
    case 2: return launch_merge_ns<2>(p, Dv, lse, s, g_smem_merge[0]);
    case 3: return launch_merge_ns<3>(p, Dv, lse, s, g_smem_merge[1]);
    case 4: return launch_merge_ns<4>(p, Dv, lse, s, g_smem_merge[2]);
    case 8: return launch_merge_ns<8>(p, Dv, lse, s, g_smem_merge[3]);
    default: return launch_merge_ns<0>(p, Dv, lse, s, g_smem_merge[4]);
  }
}

FuncAttrOnce g_smem_big, g_smem_tiny, g_smem_f8;

int dv_split_for(int Dv) { return Dv == 512 ? 2 : 1; }

// Bytes of one fp8 cache row: Dv codes, Dv / 128 fp32 scales, the rope in bf16.
constexpr int fp8_row_bytes(int Dk, int Dv) { return Dv + 4 * (Dv / 128) + 2 * (Dk - Dv); }

// q [T, H, Dk] as a 3-D tensor (box: 64 dims x 128 heads x 1 token) and the
// latent cache as 2-D rows (gathered 4 rows at a time). bf16 cache: boxes of
// 64 dims (SWIZZLE_128B, the MMA operand layout) and 32 rope dims
// (SWIZZLE_64B). fp8 cache (f8): 256 code bytes and 16 scale bytes (no
// swizzle; dequantised by the kernel) and 32 rope dims (SWIZZLE_64B).
dsa_status_t launch_mla(const MlaParams& p, const void* q, const void* kv, int Dk, int Dv, bool f8, cudaStream_t s) {
  const int64_t grid = static_cast<int64_t>(p.T) * p.splits * dv_split_for(Dv);
  if (grid > 0x7FFFFFFF) return fail(DSA_ERR_UNSUPPORTED, "sparse_mla: grid too large");
  const uint64_t rows = static_cast<uint64_t>(std::max(p.total_rows, 1));
  CUtensorMap qmap, kvmap, qmap64, kvmap64, scmap;
  memset(&scmap, 0, sizeof(scmap));
  for (int half = 0; half < 2; ++half) {
    const uint32_t w = half ? 32 : 64;
    const CUtensorMapSwizzle sw = half ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
    const uint64_t dims[3] = {static_cast<uint64_t>(Dk), static_cast<uint64_t>(p.H), static_cast<uint64_t>(p.T)};
    const uint64_t strides[2] = {static_cast<uint64_t>(Dk) * 2, static_cast<uint64_t>(p.H) * Dk * 2};
    const uint32_t box[3] = {w, 128, 1};
    dsa_status_t st = make_tmap(half ? &qmap64 : &qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, dims, strides, box, sw);
    if (st != DSA_OK) return st;
  }
  if (!f8) {
    for (int half = 0; half < 2; ++half) {
      const uint32_t w = half ? 32 : 64;
      const CUtensorMapSwizzle sw = half ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
      const uint64_t dims[2] = {static_cast<uint64_t>(Dk), rows};
      const uint64_t strides[1] = {static_cast<uint64_t>(Dk) * 2};
      const uint32_t box[2] = {w, 1};
      dsa_status_t st = make_tmap(half ? &kvmap64 : &kvmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kv, dims, strides, box, sw);
      if (st != DSA_OK) return st;
    }
  } else {
    const uint64_t rb = static_cast<uint64_t>(fp8_row_bytes(Dk, Dv));
    {
      const uint64_t dims[2] = {rb, rows};
      const uint64_t strides[1] = {rb};
      const uint32_t box_codes[2] = {256, 1}, box_scales[2] = {16, 1};
      dsa_status_t st = make_tmap(&kvmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, kv, dims, strides, box_codes,
                                  CU_TENSOR_MAP_SWIZZLE_NONE);
      if (st != DSA_OK) return st;
      st = make_tmap(&scmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, kv, dims, strides, box_scales, CU_TENSOR_MAP_SWIZZLE_NONE);
      if (st != DSA_OK) return st;
    }
    {
      const uint64_t dims[2] = {rb / 2, rows};
      const uint64_t strides[1] = {rb};
      const uint32_t box[2] = {32, 1};
      dsa_status_t st = make_tmap(&kvmap64, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kv, dims, strides, box,
                                  CU_TENSOR_MAP_SWIZZLE_64B);
      if (st != DSA_OK) return st;
    }
  }
  dsa_status_t st;
  if (Dk == 576) {
    const int smem = f8 ? MlaSmem<576, 512, true>::kTotal : MlaSmem<576, 512, false>::kTotal;
    st = f8 ? allow_smem(sparse_mla_kernel<576, 512, true>, smem, g_smem_f8)
            : allow_smem(sparse_mla_kernel<576, 512, false>, smem, g_smem_big);
    if (st != DSA_OK) return st;
    // the two value halves of a (token, split) form a 2-CTA cluster
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = f8 ? cudaLaunchKernelEx(&cfg, sparse_mla_kernel<576, 512, true>, p, qmap, kvmap, qmap64, kvmap64, scmap)
                       : cudaLaunchKernelEx(&cfg, sparse_mla_kernel<576, 512, false>, p, qmap, kvmap, qmap64, kvmap64,
                                            scmap);
    if (e != cudaSuccess) return fail(DSA_ERR_CUDA, "sparse_mla_kernel launch failed: %s", cudaGetErrorString(e));
  } else {
    st = allow_smem(sparse_mla_kernel<80, 64, false>, MlaSmem<80, 64, false>::kTotal, g_smem_tiny);
    if (st != DSA_OK) return st;
    sparse_mla_kernel<80, 64, false><<<static_cast<unsigned>(grid), kThreads, MlaSmem<80, 64, false>::kTotal, s>>>(
        p, qmap, kvmap, qmap64, kvmap64, scmap);
  }
  return check_launch("sparse_mla_kernel");
}

dsa_status_t validate(const void* q, const void* kv_cache, int64_t kv_block_stride, int32_t num_blocks,
                      const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens,
                      const int32_t* query_start_loc, const int32_t* topk_idx, int32_t B, int32_t T, int32_t H,
                      int32_t Dk, int32_t Dv, int32_t index_topk, int32_t block_size, float softmax_scale,
                      const void* out, bool f8, const char* name) {
  if (B < 0 || T < 0 || H <= 0 || index_topk <= 0 || block_size <= 0 || num_blocks < 0 || bt_stride < 0)
    return fail(DSA_ERR_INVALID_ARG, "%s: negative or zero size argument", name);
  if (T > 0 && B == 0) return fail(DSA_ERR_INVALID_ARG, "%s: T > 0 with B == 0", name);
  if (!(Dk == 576 && Dv == 512) && !(Dk == 80 && Dv == 64))
    return fail(DSA_ERR_UNSUPPORTED, "%s: (Dk, Dv) = (%d, %d) not in {(576,512), (80,64)}", name, Dk, Dv);
  if (f8 && !(Dk == 576 && Dv == 512))
    return fail(DSA_ERR_UNSUPPORTED, "%s: the fp8 cache supports (Dk, Dv) = (576, 512) only", name);
  // a cache row in the units of kv_block_stride: Dk bf16 elements, or the
  // bytes of an fp8 row
  const int64_t row = f8 ? fp8_row_bytes(Dk, Dv) : Dk;
  if (H > 128) return fail(DSA_ERR_UNSUPPORTED, "%s: H=%d > 128", name, H);
  if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale))
    return fail(DSA_ERR_INVALID_ARG, "%s: softmax_scale must be positive and finite", name);
  if (T == 0) return DSA_OK;
  if (!q || !kv_cache || !block_table || !seq_lens || !query_start_loc || !topk_idx || !out)
    return fail(DSA_ERR_INVALID_ARG, "%s: null pointer", name);
  if (!aligned16(q) || !aligned16(kv_cache) || !aligned16(out))
    return fail(DSA_ERR_INVALID_ARG, "%s: q, kv_cache and out must be 16-byte aligned", name);
  if (kv_block_stride < static_cast<int64_t>(block_size) * row)
    return fail(DSA_ERR_INVALID_ARG, "%s: kv_block_stride %lld < block_size rows of %lld", name,
                static_cast<long long>(kv_block_stride), static_cast<long long>(row));
  if (kv_block_stride % row)
    return fail(DSA_ERR_UNSUPPORTED, "%s: kv_block_stride %lld is not a whole number of %lld-unit rows", name,
                static_cast<long long>(kv_block_stride), static_cast<long long>(row));
  if (static_cast<int64_t>(num_blocks) * (kv_block_stride / row) >= (int64_t(1) << 31))
    return fail(DSA_ERR_UNSUPPORTED, "%s: the cache holds 2^31 rows or more", name);
  return check_device();
}

MlaParams make_params(int64_t kv_block_stride, int64_t row_units, int32_t num_blocks, const int32_t* block_table,
                      int32_t bt_stride, const int32_t* seq_lens, const int32_t* query_start_loc,
                      const int32_t* topk_idx, int32_t B, int32_t T, int32_t H, int32_t index_topk, int32_t block_size,
                      float softmax_scale, int32_t splits, void* out, float* lse, int32_t* dev_status) {
  MlaParams p;
  p.num_blocks = num_blocks;
  p.rows_per_block = static_cast<int32_t>(kv_block_stride / row_units);
  p.total_rows = static_cast<int32_t>(static_cast<int64_t>(num_blocks) * p.rows_per_block);
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.seq_lens = seq_lens;
  p.qsl = query_start_loc;
  p.topk = topk_idx;
  p.B = B;
  p.T = T;
  p.H = H;
  p.K = index_topk;
  p.block_size = block_size;
  p.splits = splits;
  p.per_split = (index_topk + splits - 1) / splits;
  p.scale_log2 = softmax_scale * kLog2e;
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  p.o_part = nullptr;
  p.ml_part = nullptr;
  p.dev_status = dev_status;
  return p;
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" size_t sparse_mla_workspace_size(int32_t T, int32_t H, int32_t Dv, int32_t num_kv_splits) {
  if (T <= 0 || H <= 0 || Dv <= 0 || num_kv_splits <= 1) return 0;
  return static_cast<size_t>(T) * H * num_kv_splits * (static_cast<size_t>(Dv) * sizeof(float) + sizeof(float2));
}

extern "C" int32_t sparse_mla_auto_splits(int32_t T, int32_t H, int32_t Dv, int32_t index_topk) {
  (void)H;
  if (T <= 0 || index_topk <= 0) return 1;
  const int tiles = (index_topk + 63) / 64;  // work granule of the cost model
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0) sms = v;
  } else {
    cudaGetLastError();
  }
  const int64_t units = static_cast<int64_t>(T) * dv_split_for(Dv);
  int best = (index_topk + kMaxSlots - 1) / kMaxSlots;
  int64_t best_cost = INT64_MAX;
  for (int s = (index_topk + kMaxSlots - 1) / kMaxSlots; s <= std::min(32, tiles); ++s) {
    const int64_t waves = (units * s + sms - 1) / sms;
    const int64_t cost = waves * ((tiles + s - 1) / s + 2);
    if (cost < best_cost) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

extern "C" int32_t sparse_mla_num_splits(int32_t T, int32_t H, int32_t Dv, int32_t index_topk,
                                         int32_t num_kv_splits) {
  if (num_kv_splits > 0) return num_kv_splits;
  if (num_kv_splits == DSA_KV_SPLITS_BATCH_INVARIANT)
    return index_topk > 0 ? (index_topk + kMaxSlots - 1) / kMaxSlots : 1;  // depends on index_topk alone
  return sparse_mla_auto_splits(T, H, Dv, index_topk);
}

namespace dsa {
namespace {

dsa_status_t decode_impl(const void* q, const void* kv_cache, int64_t kv_block_stride, int32_t num_blocks,
                         const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens,
                         const int32_t* query_start_loc, const int32_t* topk_idx, int32_t B, int32_t T, int32_t H,
                         int32_t Dk, int32_t Dv, int32_t index_topk, int32_t block_size, float softmax_scale,
                         int32_t num_kv_splits, void* out, float* lse, void* workspace, size_t ws_bytes,
                         int32_t* dev_status, dsa_stream_t stream, bool f8, const char* name) {
  dsa_status_t st = validate(q, kv_cache, kv_block_stride, num_blocks, block_table, bt_stride, seq_lens,
                             query_start_loc, topk_idx, B, T, H, Dk, Dv, index_topk, block_size, softmax_scale, out, f8,
                             name);
  if (st != DSA_OK || T == 0) return st;
  if (num_kv_splits < DSA_KV_SPLITS_BATCH_INVARIANT || num_kv_splits > 32)
    return fail(DSA_ERR_INVALID_ARG, "%s: num_kv_splits %d not in [-1, 32]", name, num_kv_splits);
  const int splits = sparse_mla_num_splits(T, H, Dv, index_topk, num_kv_splits);
  if ((index_topk + splits - 1) / splits > kMaxSlots)
    return fail(DSA_ERR_UNSUPPORTED, "%s: %d top-k slots per split exceed %d", name, (index_topk + splits - 1) / splits,
                kMaxSlots);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  MlaParams p = make_params(kv_block_stride, f8 ? fp8_row_bytes(Dk, Dv) : Dk, num_blocks, block_table, bt_stride,
                            seq_lens, query_start_loc, topk_idx, B, T, H, index_topk, block_size, softmax_scale,
                            splits, out, lse, dev_status);
  if (splits > 1) {
    const size_t need = sparse_mla_workspace_size(T, H, Dv, splits);
    if (workspace == nullptr || ws_bytes < need || !aligned16(workspace))
      return fail(DSA_ERR_WORKSPACE, "%s: %d splits need %zu workspace bytes (16-byte aligned), got %zu", name, splits,
                  need, ws_bytes);
    p.o_part = static_cast<float*>(workspace);
    p.ml_part = reinterpret_cast<float2*>(p.o_part + static_cast<int64_t>(T) * H * splits * Dv);
  }
  st = launch_mla(p, q, kv_cache, Dk, Dv, f8, s);
  if (st != DSA_OK || splits == 1) return st;
  return launch_merge(p, Dv, lse, s);
}

dsa_status_t prefill_impl(const void* q, const void* kv_cache, int64_t kv_block_stride, int32_t num_blocks,
                          const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens,
                          const int32_t* query_start_loc, const int32_t* topk_idx, int32_t B, int32_t T, int32_t H,
                          int32_t Dk, int32_t Dv, int32_t index_topk, int32_t block_size, float softmax_scale,
                          void* out, float* lse, int32_t* dev_status, dsa_stream_t stream, bool f8, const char* name) {
  dsa_status_t st = validate(q, kv_cache, kv_block_stride, num_blocks, block_table, bt_stride, seq_lens,
                             query_start_loc, topk_idx, B, T, H, Dk, Dv, index_topk, block_size, softmax_scale, out, f8,
                             name);
  if (st != DSA_OK || T == 0) return st;
  if (index_topk > kMaxSlots)
    return fail(DSA_ERR_UNSUPPORTED, "%s: index_topk %d > %d (use the decode entry point with splits)", name, index_topk,
                kMaxSlots);
  MlaParams p = make_params(kv_block_stride, f8 ? fp8_row_bytes(Dk, Dv) : Dk, num_blocks, block_table, bt_stride,
                            seq_lens, query_start_loc, topk_idx, B, T, H, index_topk, block_size, softmax_scale, 1, out,
                            lse, dev_status);
  return launch_mla(p, q, kv_cache, Dk, Dv, f8, reinterpret_cast<cudaStream_t>(stream));
}

}  // namespace
}  // namespace dsa

extern "C" dsa_status_t sparse_mla_decode(const void* q, const void* kv_cache, int64_t kv_block_stride,
                                          int32_t num_blocks, const int32_t* block_table, int32_t bt_stride,
                                          const int32_t* seq_lens, const int32_t* query_start_loc,
                                          const int32_t* topk_idx, int32_t B, int32_t T, int32_t H, int32_t Dk,
                                          int32_t Dv, int32_t index_topk, int32_t block_size, float softmax_scale,
                                          int32_t num_kv_splits, void* out, float* lse, void* workspace,
                                          size_t ws_bytes, int32_t* dev_status, dsa_stream_t stream) {
  return decode_impl(q, kv_cache, kv_block_stride, num_blocks, block_table, bt_stride, seq_lens, query_start_loc,
                     topk_idx, B, T, H, Dk, Dv, index_topk, block_size, softmax_scale, num_kv_splits, out, lse,
                     workspace, ws_bytes, dev_status, stream, false, "sparse_mla_decode");
}

extern "C" dsa_status_t sparse_mla_prefill(const void* q, const void* kv_cache, int64_t kv_block_stride,
                                           int32_t num_blocks, const int32_t* block_table, int32_t bt_stride,
                                           const int32_t* seq_lens, const int32_t* query_start_loc,
                                           const int32_t* topk_idx, int32_t B, int32_t T, int32_t H, int32_t Dk,
                                           int32_t Dv, int32_t index_topk, int32_t block_size, float softmax_scale,
                                           void* out, float* lse, int32_t* dev_status, dsa_stream_t stream) {
  return prefill_impl(q, kv_cache, kv_block_stride, num_blocks, block_table, bt_stride, seq_lens, query_start_loc,
                      topk_idx, B, T, H, Dk, Dv, index_topk, block_size, softmax_scale, out, lse, dev_status, stream,
                      false, "sparse_mla_prefill");
}

extern "C" dsa_status_t sparse_mla_decode_fp8(const void* q, const uint8_t* kv_cache, int64_t kv_block_stride_bytes,
                                              int32_t num_blocks, const int32_t* block_table, int32_t bt_stride,
                                              const int32_t* seq_lens, const int32_t* query_start_loc,
                                              const int32_t* topk_idx, int32_t B, int32_t T, int32_t H, int32_t Dk,
                                              int32_t Dv, int32_t index_topk, int32_t block_size, float softmax_scale,
                                              int32_t num_kv_splits, void* out, float* lse, void* workspace,
                                              size_t ws_bytes, int32_t* dev_status, dsa_stream_t stream) {
  return decode_impl(q, kv_cache, kv_block_stride_bytes, num_blocks, block_table, bt_stride, seq_lens,
                     query_start_loc, topk_idx, B, T, H, Dk, Dv, index_topk, block_size, softmax_scale, num_kv_splits,
                     out, lse, workspace, ws_bytes, dev_status, stream, true, "sparse_mla_decode_fp8");
}

extern "C" dsa_status_t sparse_mla_prefill_fp8(const void* q, const uint8_t* kv_cache, int64_t kv_block_stride_bytes,
                                               int32_t num_blocks, const int32_t* block_table, int32_t bt_stride,
                                               const int32_t* seq_lens, const int32_t* query_start_loc,
                                               const int32_t* topk_idx, int32_t B, int32_t T, int32_t H, int32_t Dk,
                                               int32_t Dv, int32_t index_topk, int32_t block_size, float softmax_scale,
                                               void* out, float* lse, int32_t* dev_status, dsa_stream_t stream) {
  return prefill_impl(q, kv_cache, kv_block_stride_bytes, num_blocks, block_table, bt_stride, seq_lens,
                      query_start_loc, topk_idx, B, T, H, Dk, Dv, index_topk, block_size, softmax_scale, out, lse,
                      dev_status, stream, true, "sparse_mla_prefill_fp8");
}

// ---------------------------------------------------------------------------
// Split-KV decode for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run the step:
// code inside a CUDA-graph capture region, an allocator-free serving runtime
// that owns all device memory up front, or a host environment (a plugin, a
// sandboxed runtime) that is not allowed to create allocations. For them the
// split partials live in the file-scope array below instead of a caller
// workspace. It is reserved when the library is loaded on a device and stays
// resident on every GPU that loads the library until the process exits.
namespace {

constexpr size_t kFixedScratchBytes = size_t(24) << 20;  // 24 MiB
static __device__ __align__(256) unsigned char g_mla_fixed_scratch[kFixedScratchBytes];

constexpr int kScratchMaxDevices = 64;
void* g_fixed_scratch_ptr[kScratchMaxDevices] = {nullptr};
std::mutex g_fixed_scratch_mu;

// Device address of the array on the current device, looked up once per
// device. In host code the array's name is only a host-side stand-in, so the
// kernels are given the address returned here.
dsa_status_t fixed_scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(DSA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kScratchMaxDevices) return fail(DSA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_fixed_scratch_mu);
  if (g_fixed_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_mla_fixed_scratch);
    if (e != cudaSuccess || ptr == nullptr)
      return fail(DSA_ERR_CUDA, "cudaGetSymbolAddress(fixed scratch): %s", cudaGetErrorString(e));
    g_fixed_scratch_ptr[dev] = ptr;
  }
  *out = g_fixed_scratch_ptr[dev];
  return DSA_OK;
}

}  // namespace

extern "C" size_t sparse_mla_fixed_scratch_bytes(void) { return kFixedScratchBytes; }

extern "C" dsa_status_t sparse_mla_decode_fixed_scratch(
    const void* q, const void* kv_cache, int64_t kv_block_stride, int32_t num_blocks, const int32_t* block_table,
    int32_t bt_stride, const int32_t* seq_lens, const int32_t* query_start_loc, const int32_t* topk_idx, int32_t B,
    int32_t T, int32_t H, int32_t Dk, int32_t Dv, int32_t index_topk, int32_t block_size, float softmax_scale,
    int32_t num_kv_splits, void* out, float* lse, int32_t* dev_status, dsa_stream_t stream) {
  if (num_kv_splits < DSA_KV_SPLITS_BATCH_INVARIANT || num_kv_splits > 32)
    return fail(DSA_ERR_INVALID_ARG, "sparse_mla_decode_fixed_scratch: num_kv_splits %d not in [-1, 32]",
                num_kv_splits);
  if (T <= 0 || H <= 0 || Dv <= 0 || index_topk <= 0)  // nothing to split: no scratch needed
    return sparse_mla_decode(q, kv_cache, kv_block_stride, num_blocks, block_table, bt_stride, seq_lens,
                             query_start_loc, topk_idx, B, T, H, Dk, Dv, index_topk, block_size, softmax_scale,
                             num_kv_splits, out, lse, nullptr, 0, dev_status, stream);
  int32_t splits = sparse_mla_num_splits(T, H, Dv, index_topk, num_kv_splits);
  if (num_kv_splits == 0) {
    // automatic count: the largest one, down to the fewest splits the slot
    // limit allows, whose partials fit the fixed scratch
    const int32_t fewest = (index_topk + kMaxSlots - 1) / kMaxSlots;
    while (splits > fewest && sparse_mla_workspace_size(T, H, Dv, splits) > kFixedScratchBytes) --splits;
  }
  const size_t need = sparse_mla_workspace_size(T, H, Dv, splits);
  if (need > kFixedScratchBytes)
    return fail(DSA_ERR_WORKSPACE,
                "sparse_mla_decode_fixed_scratch: %d splits of T=%d H=%d Dv=%d need %zu bytes of partials, more than "
                "the fixed %zu-byte scratch; use fewer splits or sparse_mla_decode with a workspace",
                splits, T, H, Dv, need, kFixedScratchBytes);
  void* scratch = nullptr;
  if (need > 0) {
    dsa_status_t st = fixed_scratch_address(&scratch);
    if (st != DSA_OK) return st;
  }
  // every partial the merge reads is written by the split kernel first, so
  // nothing in the scratch has to start at zero
  return sparse_mla_decode(q, kv_cache, kv_block_stride, num_blocks, block_table, bt_stride, seq_lens,
                           query_start_loc, topk_idx, B, T, H, Dk, Dv, index_topk, block_size, softmax_scale, splits,
                           out, lse, scratch, need, dev_status, stream);
}
