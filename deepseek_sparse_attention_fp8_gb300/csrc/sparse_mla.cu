// a3 + a4: sparse MLA attention over the top-k rows of the paged bf16 latent
// cache, with split-KV partials and their online-softmax merge
// (vLLM PR #38476, Changes 3: split-KV decode with an N-way online-softmax
// merge, a single-pass path, and a finite -1e30 sentinel for masked slots).
//
// For query token t and head h:
//   s_i = scale * q[t,h,:] . kv[i,:]          over the selected rows i
//   out = sum_i softmax(s)_i * kv[i, :Dv]     lse = log sum_i exp(s_i)
//
// One CTA handles (token, value half, split). The 128 heads are the MMA M
// dimension. Per 64-key tile:
//   S  = Q K^T    tcgen05 kind::f16, M=128 heads, N=64 keys, K=Dk; the first
//                 384 q dims are the A operand in tensor memory, the rest in
//                 shared memory;
//   softmax       thread = head row, lazy rescaling of O (only when the row
//                 maximum grows by more than 2^8);
//   O += P V      M=128 heads, N=256 value dims (MN-major view of the same
//                 shared-memory KV tile), fp32 accumulator in tensor memory.
// The 512 value dims are split across two CTAs because O for 128 heads x 512
// dims would fill the whole tensor memory of an SM; both CTAs compute S.
// Selected rows are gathered through the block table with 16-byte cp.async;
// empty or invalid slots are zero-filled and score the sentinel with weight 0.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cmath>
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
constexpr int kXBufs = 2;                 // score-exchange buffers in flight
constexpr int kXPitch = 64 * 2 + 16;      // bytes per row of an exchange buffer (fp16 scores)

// kPair: the two CTAs of a cluster split the Dk dims (rank 0: K-blocks
// [0, kNkb0), rank 1: the rest) and the value dims (rank r: values
// [r*kDvc, (r+1)*kDvc)), and exchange partial scores through DSMEM.
template <int DK, int DV>
struct MlaCfg;
template <>
struct MlaCfg<576, 512> {
  static constexpr bool kPair = true;
  static constexpr int kNkb0 = 4, kNkb1 = 5, kMaxNkb = 5, kDvc = 256, kTmemCols = 512;
};
template <>
struct MlaCfg<80, 64> {
  static constexpr bool kPair = false;
  static constexpr int kNkb0 = 2, kNkb1 = 0, kMaxNkb = 2, kDvc = 64, kTmemCols = 256;
};

template <int DK, int DV>
struct MlaSmem {
  using C = MlaCfg<DK, DV>;
  static constexpr int kKvKb = kTileKeys * 128;  // one 64-dim K-block of a KV tile
  static constexpr int kKvStage = C::kMaxNkb * kKvKb;
  static constexpr int kKv = 0;
  static constexpr int kP = kKv + kStages * kKvStage;
  static constexpr int kX = kP + 16384;
  static constexpr int kXBuf = 128 * kXPitch;
  static constexpr int kRow = kX + (C::kPair ? kXBufs * kXBuf : 0);
  static constexpr int kLive = kRow + kMaxSlots * 4;
  static constexpr int kCoord = kLive + kStages * kTileKeys;
  static constexpr int kRed = kCoord + kStages * kTileKeys * 4;
  static constexpr int kTotal = kRed + 2 * 2 * 128 * 4 + 1024;
  static_assert(C::kMaxNkb * 16384 <= kStages * kKvStage, "q staging does not fit");
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

__device__ __forceinline__ uint32_t pack_f16_sat(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float2 unpack_f16(uint32_t v) {
  return __half22float2(*reinterpret_cast<const __half2*>(&v));
}

__device__ __forceinline__ int find_request(const int32_t* qsl, int B, int t) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(qsl + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

template <int DK, int DV>
__global__ void __launch_bounds__(kThreads, 1) sparse_mla_kernel(const __grid_constant__ MlaParams p,
                                                                 const __grid_constant__ CUtensorMap qmap,
                                                                 const __grid_constant__ CUtensorMap kvmap) {
  using C = MlaCfg<DK, DV>;
  using L = MlaSmem<DK, DV>;
  constexpr int kSplitDv = C::kPair ? 2 : 1;
  constexpr uint32_t kColS = 0, kColO = kTileKeys, kColQ = kTileKeys + C::kDvc;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t kv_full[kStages], kv_empty[kStages], x_full[kXBufs];
  __shared__ uint64_t s_full, s_free, p_full, o_done, q_full, pair_bar[4];
  __shared__ uint32_t tmem_holder;
  __shared__ int s_last_live;
  __shared__ volatile int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = C::kPair ? static_cast<int>(cluster_ctarank()) : 0;
  const int j = (blockIdx.x / kSplitDv) % p.splits;
  const int t = blockIdx.x / (kSplitDv * p.splits);
  const int kb0 = r == 0 ? 0 : C::kNkb0;          // first K-block (64 dims) this CTA owns
  const int nkb = r == 0 ? C::kNkb0 : C::kNkb1;   // K-blocks this CTA owns
  const int b = find_request(p.qsl, p.B, t);
  const int q0 = __ldg(p.qsl + b), q1 = __ldg(p.qsl + b + 1);
  int64_t valid64 = static_cast<int64_t>(__ldg(p.seq_lens + b)) - (q1 - q0) + (t - q0) + 1;
  const int64_t cap = static_cast<int64_t>(p.bt_stride) * p.block_size;
  if (valid64 > cap || valid64 < 1) {
    if (tid == 0 && r == 0 && j == 0) report(p.dev_status, DSA_DEVERR_SEQ_LEN);
    valid64 = max(static_cast<int64_t>(0), min(valid64, cap));
  }
  const int valid = static_cast<int>(valid64);
  const int slot0 = j * p.per_split;
  const int n_slots = max(0, min(p.K, slot0 + p.per_split) - slot0);

  uint8_t* kv_sm = smem + L::kKv;
  uint8_t* p_sm = smem + L::kP;
  uint8_t* x_sm = smem + L::kX;
  int* row_sm = reinterpret_cast<int*>(smem + L::kRow);
  uint8_t* live_sm = smem + L::kLive;
  int* coord_sm = reinterpret_cast<int*>(smem + L::kCoord);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int s = 0; s < kXBufs; ++s) mbar_init(&x_full[s], 1);  // local expect_tx; the peer's st.async deliver the bytes
    mbar_init(&s_full, 1);
    mbar_init(&s_free, 8);
    mbar_init(&p_full, 8);
    mbar_init(&o_done, 1);
    mbar_init(&q_full, 1);
    for (int q = 0; q < 4; ++q) mbar_init(&pair_bar[q], 64);
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

  auto abort_now = [&](void) {
    s_abort = 1;
    report(p.dev_status, DSA_DEVERR_TIMEOUT);
  };

  // ---- prologue: this CTA's q K-blocks by TMA into the idle KV stage area;
  // the softmax warps resolve the split's top-k slots to physical rows
  if (tid == kProdWarp0 * 32) {  // first producer thread
    prefetch_tmap(&qmap);
    prefetch_tmap(&kvmap);
    mbar_arrive_expect_tx(&q_full, nkb * 16384);
    for (int kb = 0; kb < nkb; ++kb)
      tma_load_3d(smem_u32(kv_sm + kb * 16384), &qmap, &q_full, (kb0 + kb) * 64, 0, t);
  }
  if (warp < 8) {
    const int32_t* bt_row = p.block_table + static_cast<int64_t>(b) * p.bt_stride;
    const int32_t* idx_row = p.topk + static_cast<int64_t>(t) * p.K + slot0;
    int last = -1;
    for (int base = 0; base < n_slots; base += 256 * 8) {
      int idx[8], blk[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int sl = base + u * 256 + tid;
        idx[u] = sl < n_slots ? __ldg(idx_row + sl) : -1;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u)
        blk[u] = (idx[u] >= 0 && idx[u] < valid) ? __ldg(bt_row + idx[u] / p.block_size) : -1;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int sl = base + u * 256 + tid;
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
    }
    if (last >= 0) atomicMax(&s_last_live, last);
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
            const uint4 u = *reinterpret_cast<const uint4*>(kv_sm + kb * 16384 + sw128_offset(hq, half * 4 + c));
            v[4 * c] = u.x;
            v[4 * c + 1] = u.y;
            v[4 * c + 2] = u.z;
            v[4 * c + 3] = u.w;
          }
          tmem_st16(lane_q + kb * 32 + half * 16, v);
        }
      }
      tmem_st_wait();
      fence_proxy_async_smem();  // the staging area is refilled by TMA next
    }
  }
  tc_fence_before();
  __syncthreads();  // q in place, slots resolved, staging area free
  tc_fence_after();
  const int n_tiles = s_abort ? 0 : (s_last_live + kTileKeys) / kTileKeys;

  if (warp >= kProdWarp0 && warp < kMmaWarp) {
    // ---------------- producer: 4 warps, 16 keys each; 4-row TMA gathers of
    // this CTA's K-blocks only
    const int pw = warp - kProdWarp0;
    const uint32_t tile_bytes = kTileKeys * nkb * 128;
    for (int i = 0; i < n_tiles && !s_abort; ++i) {
      const int st = i % kStages;
      if (i >= kStages && !mbar_wait(&kv_empty[st], ((i / kStages) - 1) & 1)) {
        if (lane == 0) abort_now();
        break;
      }
      if (lane < 16) {
        const int kr = pw * 16 + lane;
        const int sl = i * kTileKeys + kr;
        const int row = sl < n_slots ? row_sm[sl] : -1;
        live_sm[st * kTileKeys + kr] = row >= 0 ? 1 : 0;
        coord_sm[st * kTileKeys + kr] = row >= 0 ? row : p.total_rows;  // out of range: zero fill
      }
      __syncwarp();
      if (pw == 0 && lane == 0) mbar_arrive_expect_tx(&kv_full[st], tile_bytes);
      if (lane < 4 * nkb) {
        const int g = pw * 4 + (lane & 3), kb = lane >> 2;
        const int* cs = coord_sm + st * kTileKeys + 4 * g;
        tma_gather4(smem_u32(kv_sm + st * L::kKvStage + kb * L::kKvKb + g * 512), &kvmap, &kv_full[st],
                    (kb0 + kb) * 64, cs[0], cs[1], cs[2], cs[3]);
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issuer
    if (!mbar_wait(&q_full, 0) && lane == 0) abort_now();
    const uint32_t idesc_qk = idesc_bf16(128, kTileKeys, false, false);
    const uint32_t idesc_pv = idesc_bf16(128, C::kDvc, false, true);
    const uint32_t p0s = smem_u32(p_sm);
    auto issue_pv = [&](int i) {
      const int st = i % kStages;
      // value dims = this CTA's first K-blocks
      const uint64_t vd = smem_desc(smem_u32(kv_sm + st * L::kKvStage), L::kKvKb, 1024, kSwizzle128B);
      const uint64_t pd = smem_desc(p0s, 16, 1024, kSwizzle128B);
#pragma unroll
      for (int ks = 0; ks < kTileKeys / 16; ++ks)
        mma_bf16_ss(tmem + kColO, pd + static_cast<uint64_t>((ks * 32) >> 4), vd + static_cast<uint64_t>((ks * 2048) >> 4),
                    idesc_pv, (i > 0 || ks > 0) ? 1u : 0u);
      mma_commit(&kv_empty[st]);
      mma_commit(&o_done);
    };
    for (int i = 0; i < n_tiles && !s_abort; ++i) {
      const int st = i % kStages;
      bool ok = mbar_wait(&kv_full[st], (i / kStages) & 1);
      if (ok && i >= 1) ok = mbar_wait(&s_free, (i - 1) & 1);
      if (!ok) {
        if (lane == 0) abort_now();
        break;
      }
      tc_fence_after();
      if (lane == 0) {  // this CTA's part of S = Q K^T
        // descriptors differ only in the start-address field (16-byte units)
        const uint64_t d0 = smem_desc(smem_u32(kv_sm + st * L::kKvStage), 16, 1024, kSwizzle128B);
#pragma unroll
        for (int kb = 0; kb < C::kMaxNkb; ++kb) {
          if (kb >= nkb) break;
#pragma unroll
          for (int k4 = 0; k4 < 4; ++k4)
            mma_bf16_ts(tmem + kColS, tmem + kColQ + (kb * 4 + k4) * 8,
                        d0 + static_cast<uint64_t>((kb * L::kKvKb + k4 * 32) >> 4), idesc_qk, (kb | k4) ? 1u : 0u);
        }
        mma_commit(&s_full);
      }
      __syncwarp();
      if (i >= 1) {  // O += P V for the previous tile
        if (!mbar_wait(&p_full, (i - 1) & 1)) {
          if (lane == 0) abort_now();
          break;
        }
        tc_fence_after();
        if (lane == 0) issue_pv(i - 1);
        __syncwarp();
      }
    }
    if (n_tiles > 0 && !s_abort) {
      const int i = n_tiles - 1;
      if (!mbar_wait(&p_full, i & 1)) {
        if (lane == 0) abort_now();
      } else {
        tc_fence_after();
        if (lane == 0) issue_pv(i);
        __syncwarp();
      }
    }
  } else {
    // ---------------- softmax: warps w and w+4 share TMEM lanes 32*(w%4).. (one
    // head row per thread) and take keys [32*kh, 32*kh+32) of each tile
    const int kh = warp >> 2;            // key half
    const int h = (warp & 3) * 32 + lane;  // head row
    const uint32_t lane_base = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    uint64_t* pbar = &pair_bar[warp & 3];  // joins the two warps of this lane group
    float* red = reinterpret_cast<float*>(smem + L::kRed);  // [parity][key half][128 rows]
    uint32_t x_peer = 0;
    if constexpr (C::kPair) x_peer = mapa_shared(smem_u32(x_sm + h * kXPitch + kh * 64), static_cast<uint32_t>(r ^ 1));
    const uint8_t* x_mine = x_sm + h * kXPitch + kh * 64;
    uint32_t peer_x_full[kXBufs] = {};
    if constexpr (C::kPair) {
      for (int q = 0; q < kXBufs; ++q) peer_x_full[q] = mapa_shared(smem_u32(&x_full[q]), static_cast<uint32_t>(r ^ 1));
    }
    float m_ref = kNegSentinel, l_part = 0.f;
    uint32_t prev[16];  // this CTA's fp16 partial scores of the tile waiting for the peer's
    // The peer's buffer X[i % 2] is free again when tile i is sent: this CTA
    // has received the peer's tile i-1, which the peer sends only after it has
    // finished reading X[i % 2] (tile i-2).
    constexpr int kLag = 0;
    for (int step = 0; step < n_tiles + kLag && !s_abort; ++step) {
      uint32_t sv[32];
      uint32_t hv[16];
      if (step < n_tiles) {
        if (!mbar_wait(&s_full, step & 1)) {
          if (lane == 0) abort_now();
          break;
        }
        tc_fence_after();
        tmem_ld32_sync(lane_base + kColS + kh * 32, sv);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&s_free);
        if constexpr (C::kPair) {
          const int xb = step % kXBufs;
          if (tid == 0) mbar_arrive_expect_tx(&x_full[xb], 128 * 64 * 2);  // the peer's whole partial tile
#pragma unroll
          for (int x = 0; x < 16; ++x) hv[x] = pack_f16_sat(__uint_as_float(sv[2 * x]), __uint_as_float(sv[2 * x + 1]));
#pragma unroll
          for (int c = 0; c < 4; ++c)
            st_async_v4(x_peer + xb * L::kXBuf + c * 16, peer_x_full[xb], hv[4 * c], hv[4 * c + 1], hv[4 * c + 2],
                        hv[4 * c + 3]);
        }
      }
      if (step < kLag) {
#pragma unroll
        for (int x = 0; x < 16; ++x) prev[x] = hv[x];
        continue;
      }
      const int i = step - kLag;  // the tile finished in this step
      const int st = i % kStages;
      if constexpr (C::kPair) {
        uint32_t cur[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) {
          cur[x] = kLag ? prev[x] : hv[x];
          prev[x] = hv[x];
        }
        const int xb = i % kXBufs;
        if (!mbar_wait_cluster(&x_full[xb], (i / kXBufs) & 1)) {
          if (lane == 0) abort_now();
          break;
        }
        // S = own partial + the peer's, both rounded to fp16 for the exchange,
        // so the two CTAs add the same two values and agree bit for bit
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 u = *reinterpret_cast<const uint4*>(x_mine + xb * L::kXBuf + c * 16);
          const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int y = 0; y < 4; ++y) {
            const float2 f = unpack_f16(w[y]);
            const float2 o = unpack_f16(cur[4 * c + y]);
            sv[8 * c + 2 * y] = __float_as_uint(o.x + f.x);
            sv[8 * c + 2 * y + 1] = __float_as_uint(o.y + f.y);
          }
        }
      }
      if (!mbar_wait(&kv_full[st], (i / kStages) & 1)) {  // live flags of this tile
        if (lane == 0) abort_now();
        break;
      }
      const uint32_t* lw = reinterpret_cast<const uint32_t*>(live_sm + st * kTileKeys + kh * 32);
      uint32_t live_bits = 0;
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        const uint32_t w4 = lw[x];
#pragma unroll
        for (int y = 0; y < 4; ++y) live_bits |= ((w4 >> (8 * y)) & 1u) << (4 * x + y);
      }
      float mt = kNegSentinel;
#pragma unroll
      for (int x = 0; x < 32; ++x) {
        const float s = ((live_bits >> x) & 1u) ? __uint_as_float(sv[x]) * p.scale_log2 : kNegSentinel;
        sv[x] = __float_as_uint(s);
        mt = fmaxf(mt, s);
      }
      // the row maximum over both key halves (slots alternate by tile parity, so
      // one join per tile suffices)
      red[(i & 1) * 256 + kh * 128 + h] = mt;
      mbar_arrive(pbar);
      if (!mbar_wait(pbar, i & 1)) {
        if (lane == 0) abort_now();
        break;
      }
      mt = fmaxf(mt, red[(i & 1) * 256 + (kh ^ 1) * 128 + h]);
      float alpha = 1.f;
      const bool rescale = mt > m_ref + kRescaleThreshold;
      if (rescale) {
        alpha = ex2_approx(m_ref - mt);
        m_ref = mt;
        l_part *= alpha;
      }
      uint32_t pw[16];
      float psum = 0.f;
#pragma unroll
      for (int x = 0; x < 16; ++x) {
        const float a = ((live_bits >> (2 * x)) & 1u) ? ex2_approx(__uint_as_float(sv[2 * x]) - m_ref) : 0.f;
        const float c = ((live_bits >> (2 * x + 1)) & 1u) ? ex2_approx(__uint_as_float(sv[2 * x + 1]) - m_ref) : 0.f;
        const __nv_bfloat162 pb = __floats2bfloat162_rn(a, c);
        // the normaliser sums the bf16 weights that the PV product uses
        psum += __bfloat162float(pb.x) + __bfloat162float(pb.y);
        pw[x] = *reinterpret_cast<const uint32_t*>(&pb);
      }
      l_part += psum;
      // P and O are free once PV of the previous tile is done
      if (i >= 1) {
        if (!mbar_wait(&o_done, (i - 1) & 1)) {
          if (lane == 0) abort_now();
          break;
        }
        tc_fence_after();
      }
#pragma unroll
      for (int c = 0; c < 4; ++c)
        *reinterpret_cast<uint4*>(p_sm + sw128_offset(h, kh * 4 + c)) =
            make_uint4(pw[4 * c], pw[4 * c + 1], pw[4 * c + 2], pw[4 * c + 3]);
      if (i >= 1 && __any_sync(0xFFFFFFFFu, rescale)) {  // each warp of the pair scales half of O
#pragma unroll 1
        for (int c = kh * (C::kDvc / 2); c < (kh + 1) * (C::kDvc / 2); c += 32) {
          uint32_t o[32];
          tmem_ld32_sync(lane_base + kColO + c, o);
#pragma unroll
          for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * alpha);
          tmem_st32(lane_base + kColO + c, o);
        }
        tmem_st_wait();
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&p_full);
    }

    // ---- epilogue: l = l_half0 + l_half1; each warp of the pair writes half of the columns
    bool o_valid = n_tiles > 0 && !s_abort;
    float l_sum = 0.f;
    {
      const int e = n_tiles & 1;  // the join after the last tile
      red[e * 256 + kh * 128 + h] = l_part;
      mbar_arrive(pbar);
      if (mbar_wait(pbar, n_tiles & 1)) {
        l_sum = red[e * 256 + h] + red[e * 256 + 128 + h];
      } else {
        if (lane == 0) abort_now();
        o_valid = false;
      }
    }
    if (o_valid) {
      if (!mbar_wait(&o_done, (n_tiles - 1) & 1)) {
        if (lane == 0) abort_now();
        o_valid = false;
      }
    }
    o_valid = __all_sync(0xFFFFFFFFu, o_valid) && !s_abort;
    tc_fence_after();
    const bool have = o_valid && l_sum > 0.f;
    constexpr int kHalf = C::kDvc / 2;
    if (p.splits == 1) {
      const float inv = have ? 1.f / l_sum : 0.f;
      uint16_t* dst = p.out + (static_cast<int64_t>(t) * p.H + h) * DV + r * C::kDvc;
#pragma unroll 1
      for (int c = kh * kHalf; c < (kh + 1) * kHalf; c += 32) {
        uint32_t o[32];
        if (o_valid) tmem_ld32_sync(lane_base + kColO + c, o);
        if (h < p.H) {
          uint32_t w[16];
#pragma unroll
          for (int x = 0; x < 16; ++x)
            w[x] = have ? pack_bf16(__uint_as_float(o[2 * x]) * inv, __uint_as_float(o[2 * x + 1]) * inv) : 0u;
          uint4* d4 = reinterpret_cast<uint4*>(dst + c);
#pragma unroll
          for (int x = 0; x < 4; ++x) d4[x] = make_uint4(w[4 * x], w[4 * x + 1], w[4 * x + 2], w[4 * x + 3]);
        }
      }
      if (r == 0 && kh == 0 && h < p.H && p.lse != nullptr)
        p.lse[static_cast<int64_t>(t) * p.H + h] = have ? (m_ref + log2f(l_sum)) * kLn2 : -INFINITY;
    } else {
      const int64_t row = (static_cast<int64_t>(t) * p.H + h) * p.splits + j;
      float* dst = p.o_part + row * DV + r * C::kDvc;
#pragma unroll 1
      for (int c = kh * kHalf; c < (kh + 1) * kHalf; c += 32) {
        uint32_t o[32];
        if (o_valid) tmem_ld32_sync(lane_base + kColO + c, o);
        if (h < p.H) {
          float4* d4 = reinterpret_cast<float4*>(dst + c);
#pragma unroll
          for (int x = 0; x < 8; ++x)
            d4[x] = o_valid ? make_float4(__uint_as_float(o[4 * x]), __uint_as_float(o[4 * x + 1]),
                                          __uint_as_float(o[4 * x + 2]), __uint_as_float(o[4 * x + 3]))
                            : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
      if (r == 0 && kh == 0 && h < p.H)
        p.ml_part[row] = make_float2(o_valid ? m_ref : kNegSentinel, o_valid ? l_sum : 0.f);
    }
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (C::kPair) cluster_sync_all();  // no remote access may target an exited CTA
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, C::kTmemCols);
}

// a4: out = sum_j 2^(m_j-M) o_j / sum_j 2^(m_j-M) l_j, M = max_j m_j (log2 units).
__global__ void __launch_bounds__(128) mla_merge_kernel(const float* __restrict__ o_part,
                                                        const float2* __restrict__ ml, int S, int DV,
                                                        uint16_t* __restrict__ out, float* __restrict__ lse) {
  const int64_t row = blockIdx.x;  // t * H + h
  const float2* mlr = ml + row * S;
  float M = kNegSentinel;
  for (int j = 0; j < S; ++j) M = fmaxf(M, mlr[j].x);
  float den = 0.f;
  for (int j = 0; j < S; ++j) den += exp2f(mlr[j].x - M) * mlr[j].y;
  const float inv = den > 0.f ? 1.f / den : 0.f;
  for (int v = threadIdx.x * 4; v < DV; v += blockDim.x * 4) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < S; ++j) {
      const float a = exp2f(mlr[j].x - M);
      const float4 o = *reinterpret_cast<const float4*>(o_part + (row * S + j) * DV + v);
      acc.x = fmaf(a, o.x, acc.x);
      acc.y = fmaf(a, o.y, acc.y);
      acc.z = fmaf(a, o.z, acc.z);
      acc.w = fmaf(a, o.w, acc.w);
    }
    uint2 w;
    w.x = pack_bf16(acc.x * inv, acc.y * inv);
    w.y = pack_bf16(acc.z * inv, acc.w * inv);
    *reinterpret_cast<uint2*>(out + row * DV + v) = w;
  }
  if (threadIdx.x == 0 && lse != nullptr) lse[row] = den > 0.f ? (M + log2f(den)) * kLn2 : -INFINITY;
}

bool g_smem_big = false, g_smem_tiny = false;

int dv_split_for(int Dv) { return Dv == 512 ? 2 : 1; }

// q [T, H, Dk] as a 3-D tensor (box: 64 dims x 128 heads x 1 token) and the
// latent cache as 2-D rows of Dk (box: 64 dims x 1 row, gathered 4 rows at a
// time); both 128-byte swizzled to match the MMA operand layout.
dsa_status_t launch_mla(const MlaParams& p, const void* q, const void* kv, int Dk, int Dv, cudaStream_t s) {
  const int64_t grid = static_cast<int64_t>(p.T) * p.splits * dv_split_for(Dv);
  if (grid > 0x7FFFFFFF) return fail(DSA_ERR_UNSUPPORTED, "sparse_mla: grid too large");
  CUtensorMap qmap, kvmap;
  {
    const uint64_t dims[3] = {static_cast<uint64_t>(Dk), static_cast<uint64_t>(p.H), static_cast<uint64_t>(p.T)};
    const uint64_t strides[2] = {static_cast<uint64_t>(Dk) * 2, static_cast<uint64_t>(p.H) * Dk * 2};
    const uint32_t box[3] = {64, 128, 1};
    dsa_status_t st = make_tmap(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, q, dims, strides, box,
                                CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != DSA_OK) return st;
  }
  {
    const uint64_t dims[2] = {static_cast<uint64_t>(Dk), static_cast<uint64_t>(std::max(p.total_rows, 1))};
    const uint64_t strides[1] = {static_cast<uint64_t>(Dk) * 2};
    const uint32_t box[2] = {64, 1};
    dsa_status_t st = make_tmap(&kvmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kv, dims, strides, box,
                                CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != DSA_OK) return st;
  }
  dsa_status_t st;
  if (Dk == 576) {
    st = allow_smem(sparse_mla_kernel<576, 512>, MlaSmem<576, 512>::kTotal, g_smem_big);
    if (st != DSA_OK) return st;
    // the two value halves of a (token, split) form a 2-CTA cluster
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = MlaSmem<576, 512>::kTotal;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, sparse_mla_kernel<576, 512>, p, qmap, kvmap);
    if (e != cudaSuccess) return fail(DSA_ERR_CUDA, "sparse_mla_kernel launch failed: %s", cudaGetErrorString(e));
  } else {
    st = allow_smem(sparse_mla_kernel<80, 64>, MlaSmem<80, 64>::kTotal, g_smem_tiny);
    if (st != DSA_OK) return st;
    sparse_mla_kernel<80, 64><<<static_cast<unsigned>(grid), kThreads, MlaSmem<80, 64>::kTotal, s>>>(p, qmap, kvmap);
  }
  return check_launch("sparse_mla_kernel");
}

dsa_status_t validate(const void* q, const void* kv_cache, int64_t kv_block_stride, int32_t num_blocks,
                      const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens,
                      const int32_t* query_start_loc, const int32_t* topk_idx, int32_t B, int32_t T, int32_t H,
                      int32_t Dk, int32_t Dv, int32_t index_topk, int32_t block_size, float softmax_scale,
                      const void* out, const char* name) {
  if (B < 0 || T < 0 || H <= 0 || index_topk <= 0 || block_size <= 0 || num_blocks < 0 || bt_stride < 0)
    return fail(DSA_ERR_INVALID_ARG, "%s: negative or zero size argument", name);
  if (T > 0 && B == 0) return fail(DSA_ERR_INVALID_ARG, "%s: T > 0 with B == 0", name);
  if (!(Dk == 576 && Dv == 512) && !(Dk == 80 && Dv == 64))
    return fail(DSA_ERR_UNSUPPORTED, "%s: (Dk, Dv) = (%d, %d) not in {(576,512), (80,64)}", name, Dk, Dv);
  if (H > 128) return fail(DSA_ERR_UNSUPPORTED, "%s: H=%d > 128", name, H);
  if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale))
    return fail(DSA_ERR_INVALID_ARG, "%s: softmax_scale must be positive and finite", name);
  if (T == 0) return DSA_OK;
  if (!q || !kv_cache || !block_table || !seq_lens || !query_start_loc || !topk_idx || !out)
    return fail(DSA_ERR_INVALID_ARG, "%s: null pointer", name);
  if (!aligned16(q) || !aligned16(kv_cache) || !aligned16(out))
    return fail(DSA_ERR_INVALID_ARG, "%s: q, kv_cache and out must be 16-byte aligned", name);
  if (kv_block_stride < static_cast<int64_t>(block_size) * Dk)
    return fail(DSA_ERR_INVALID_ARG, "%s: kv_block_stride %lld < block_size*Dk", name,
                static_cast<long long>(kv_block_stride));
  if (kv_block_stride % Dk)
    return fail(DSA_ERR_UNSUPPORTED, "%s: kv_block_stride %lld is not a whole number of %d-element rows", name,
                static_cast<long long>(kv_block_stride), Dk);
  if (static_cast<int64_t>(num_blocks) * (kv_block_stride / Dk) >= (int64_t(1) << 31))
    return fail(DSA_ERR_UNSUPPORTED, "%s: the cache holds 2^31 rows or more", name);
  return check_device();
}

MlaParams make_params(int64_t kv_block_stride, int32_t Dk, int32_t num_blocks, const int32_t* block_table,
                      int32_t bt_stride, const int32_t* seq_lens, const int32_t* query_start_loc,
                      const int32_t* topk_idx, int32_t B, int32_t T, int32_t H, int32_t index_topk, int32_t block_size,
                      float softmax_scale, int32_t splits, void* out, float* lse, int32_t* dev_status) {
  MlaParams p;
  p.num_blocks = num_blocks;
  p.rows_per_block = static_cast<int32_t>(kv_block_stride / Dk);
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

extern "C" dsa_status_t sparse_mla_decode(const void* q, const void* kv_cache, int64_t kv_block_stride,
                                          int32_t num_blocks, const int32_t* block_table, int32_t bt_stride,
                                          const int32_t* seq_lens, const int32_t* query_start_loc,
                                          const int32_t* topk_idx, int32_t B, int32_t T, int32_t H, int32_t Dk,
                                          int32_t Dv, int32_t index_topk, int32_t block_size, float softmax_scale,
                                          int32_t num_kv_splits, void* out, float* lse, void* workspace,
                                          size_t ws_bytes, int32_t* dev_status, dsa_stream_t stream) {
  dsa_status_t st = validate(q, kv_cache, kv_block_stride, num_blocks, block_table, bt_stride, seq_lens,
                             query_start_loc, topk_idx, B, T, H, Dk, Dv, index_topk, block_size, softmax_scale, out,
                             "sparse_mla_decode");
  if (st != DSA_OK || T == 0) return st;
  if (num_kv_splits < 0 || num_kv_splits > 32)
    return fail(DSA_ERR_INVALID_ARG, "sparse_mla_decode: num_kv_splits %d not in [0, 32]", num_kv_splits);
  int splits = num_kv_splits == 0 ? sparse_mla_auto_splits(T, H, Dv, index_topk) : num_kv_splits;
  if ((index_topk + splits - 1) / splits > kMaxSlots)
    return fail(DSA_ERR_UNSUPPORTED, "sparse_mla_decode: %d top-k slots per split exceed %d", (index_topk + splits - 1) / splits,
                kMaxSlots);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  MlaParams p = make_params(kv_block_stride, Dk, num_blocks, block_table, bt_stride, seq_lens, query_start_loc,
                            topk_idx, B, T, H, index_topk, block_size, softmax_scale, splits, out, lse, dev_status);
  if (splits > 1) {
    const size_t need = sparse_mla_workspace_size(T, H, Dv, splits);
    if (workspace == nullptr || ws_bytes < need || !aligned16(workspace))
      return fail(DSA_ERR_WORKSPACE, "sparse_mla_decode: %d splits need %zu workspace bytes (16-byte aligned), got %zu",
                  splits, need, ws_bytes);
    p.o_part = static_cast<float*>(workspace);
    p.ml_part = reinterpret_cast<float2*>(p.o_part + static_cast<int64_t>(T) * H * splits * Dv);
  }
  st = launch_mla(p, q, kv_cache, Dk, Dv, s);
  if (st != DSA_OK || splits == 1) return st;
  mla_merge_kernel<<<static_cast<unsigned>(static_cast<int64_t>(T) * H), 128, 0, s>>>(p.o_part, p.ml_part, splits, Dv,
                                                                                    p.out, lse);
  return check_launch("mla_merge_kernel");
}

extern "C" dsa_status_t sparse_mla_prefill(const void* q, const void* kv_cache, int64_t kv_block_stride,
                                           int32_t num_blocks, const int32_t* block_table, int32_t bt_stride,
                                           const int32_t* seq_lens, const int32_t* query_start_loc,
                                           const int32_t* topk_idx, int32_t B, int32_t T, int32_t H, int32_t Dk,
                                           int32_t Dv, int32_t index_topk, int32_t block_size, float softmax_scale,
                                           void* out, float* lse, int32_t* dev_status, dsa_stream_t stream) {
  dsa_status_t st = validate(q, kv_cache, kv_block_stride, num_blocks, block_table, bt_stride, seq_lens,
                             query_start_loc, topk_idx, B, T, H, Dk, Dv, index_topk, block_size, softmax_scale, out,
                             "sparse_mla_prefill");
  if (st != DSA_OK || T == 0) return st;
  if (index_topk > kMaxSlots)
    return fail(DSA_ERR_UNSUPPORTED, "sparse_mla_prefill: index_topk %d > %d (use sparse_mla_decode with splits)",
                index_topk, kMaxSlots);
  MlaParams p = make_params(kv_block_stride, Dk, num_blocks, block_table, bt_stride, seq_lens, query_start_loc,
                            topk_idx, B, T, H, index_topk, block_size, softmax_scale, 1, out, lse, dev_status);
  return launch_mla(p, q, kv_cache, Dk, Dv, reinterpret_cast<cudaStream_t>(stream));
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
  if (num_kv_splits < 0 || num_kv_splits > 32)
    return fail(DSA_ERR_INVALID_ARG, "sparse_mla_decode_fixed_scratch: num_kv_splits %d not in [0, 32]",
                num_kv_splits);
  if (T <= 0 || H <= 0 || Dv <= 0 || index_topk <= 0)  // nothing to split: no scratch needed
    return sparse_mla_decode(q, kv_cache, kv_block_stride, num_blocks, block_table, bt_stride, seq_lens,
                             query_start_loc, topk_idx, B, T, H, Dk, Dv, index_topk, block_size, softmax_scale,
                             num_kv_splits, out, lse, nullptr, 0, dev_status, stream);
  const int32_t splits = num_kv_splits == 0 ? sparse_mla_auto_splits(T, H, Dv, index_topk) : num_kv_splits;
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
