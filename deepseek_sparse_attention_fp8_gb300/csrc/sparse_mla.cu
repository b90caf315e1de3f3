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

#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "ptx.cuh"

namespace dsa {
namespace {

using namespace ptx;

constexpr int kThreads = 128;
constexpr int kTileKeys = 64;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.f;  // log2 units

template <int DK, int DV>
struct MlaCfg;
template <>
struct MlaCfg<576, 512> {
  static constexpr int kDvSplit = 2, kDvc = 256, kDkTmem = 384, kNkb = 9, kQsmKb = 3, kStages = 2, kTmemCols = 512;
};
template <>
struct MlaCfg<80, 64> {
  static constexpr int kDvSplit = 1, kDvc = 64, kDkTmem = 64, kNkb = 2, kQsmKb = 1, kStages = 2, kTmemCols = 256;
};

template <int DK, int DV>
struct MlaSmem {
  using C = MlaCfg<DK, DV>;
  static constexpr int kQ = 0;
  static constexpr int kKv = kQ + C::kQsmKb * 16384;
  static constexpr int kKvStage = C::kNkb * 8192;
  static constexpr int kP = kKv + C::kStages * kKvStage;
  static constexpr int kLive = kP + 16384;
  static constexpr int kTotal = kLive + C::kStages * kTileKeys + 1024;
};

struct MlaParams {
  const uint16_t* q;   // bf16 [T, H, DK]
  const uint16_t* kv;  // bf16 paged
  int64_t kv_block_stride;
  int32_t num_blocks;
  const int32_t* block_table;
  int32_t bt_stride;
  const int32_t* seq_lens;
  const int32_t* qsl;
  const int32_t* topk;
  int32_t B, T, H, K, block_size, splits, per_split;
  float scale_log2;
  uint16_t* out;     // bf16 [T, H, DV]
  float* lse;        // [T, H] or null
  float* o_part;     // [T, H, S, DV]
  float2* ml_part;   // [T, H, S] (max in log2 units, sum)
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

template <int DK, int DV>
__global__ void __launch_bounds__(kThreads, 1) sparse_mla_kernel(const MlaParams p) {
  using C = MlaCfg<DK, DV>;
  using L = MlaSmem<DK, DV>;
  constexpr int kChunksRow = DK * 2 / 16;       // 16-byte chunks per KV row
  constexpr uint32_t kColS = 0, kColO = 64, kColQ = 64 + C::kDvc;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t bar_s, bar_o;
  __shared__ uint32_t tmem_holder;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int r = blockIdx.x % C::kDvSplit;
  const int j = (blockIdx.x / C::kDvSplit) % p.splits;
  const int t = blockIdx.x / (C::kDvSplit * p.splits);
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
  const int slot1 = min(p.K, slot0 + p.per_split);
  const int n_tiles = slot1 > slot0 ? (slot1 - slot0 + kTileKeys - 1) / kTileKeys : 0;

  uint8_t* q_sm = smem + L::kQ;
  uint8_t* kv_sm = smem + L::kKv;
  uint8_t* p_sm = smem + L::kP;
  uint8_t* live_sm = smem + L::kLive;

  // ---- set-up: zero the KV stages when rows are narrower than the K-blocks
  if constexpr (DK % 64 != 0) {
    for (int i = tid; i < C::kStages * L::kKvStage / 16; i += kThreads)
      reinterpret_cast<uint4*>(kv_sm)[i] = make_uint4(0, 0, 0, 0);
  }
  if (warp == 0) {
    tmem_alloc(&tmem_holder, C::kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) {
    mbar_init(&bar_s, 1);
    mbar_init(&bar_o, 1);
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_holder;
  const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);

  // ---- q: dims [0, kDkTmem) into tensor memory, the rest into shared memory
  {
    const int h = tid;
    const uint4* src = reinterpret_cast<const uint4*>(p.q + (static_cast<int64_t>(t) * p.H + h) * DK);
#pragma unroll 1
    for (int c = 0; c < C::kDkTmem / 32; ++c) {
      uint32_t v[16];
      if (h < p.H) {
#pragma unroll
        for (int x = 0; x < 4; ++x) {
          const uint4 u = __ldg(src + c * 4 + x);
          v[4 * x] = u.x; v[4 * x + 1] = u.y; v[4 * x + 2] = u.z; v[4 * x + 3] = u.w;
        }
      } else {
#pragma unroll
        for (int x = 0; x < 16; ++x) v[x] = 0u;
      }
      tmem_st16(lane_base + kColQ + c * 16, v);
    }
    tmem_st_wait();
    constexpr int kQChunks = C::kQsmKb * 8;
    for (int i = tid; i < 128 * kQChunks; i += kThreads) {
      const int row = i / kQChunks, c = i % kQChunks;
      const int dim = C::kDkTmem + c * 8;
      const bool ok = row < p.H && dim < DK;
      const uint16_t* g = ok ? p.q + (static_cast<int64_t>(t) * p.H + row) * DK + dim : p.q;
      cp_async_16(smem_u32(q_sm + (c / 8) * 16384 + sw128_offset(row, c % 8)), g, ok ? 16u : 0u);
    }
  }

  const int32_t* bt_row = p.block_table + static_cast<int64_t>(b) * p.bt_stride;
  const int32_t* idx_row = p.topk + static_cast<int64_t>(t) * p.K;

  // Gathers the rows of tile `i` into stage `st`; records which slots are live.
  auto load_tile = [&](int i, int st) {
    uint8_t* dst = kv_sm + st * L::kKvStage;
    const uint16_t* row_ptr = p.kv;
    bool live = false;
    if (lane < 16) {
      const int kr = warp + 4 * lane;
      const int slot = slot0 + i * kTileKeys + kr;
      if (slot < slot1) {
        const int idx = __ldg(idx_row + slot);
        if (idx >= 0 && idx < valid) {
          const int blk = __ldg(bt_row + idx / p.block_size);
          if (blk >= 0 && blk < p.num_blocks) {
            live = true;
            row_ptr = p.kv + static_cast<int64_t>(blk) * p.kv_block_stride + static_cast<int64_t>(idx % p.block_size) * DK;
          } else {
            report(p.dev_status, DSA_DEVERR_BLOCK_OOB);
          }
        } else if (idx != -1) {
          report(p.dev_status, DSA_DEVERR_INDEX_OOB);
        }
      }
      live_sm[st * kTileKeys + kr] = live ? 1 : 0;
    }
#pragma unroll 1
    for (int m = 0; m < 16; ++m) {
      const int kr = warp + 4 * m;
      const uint16_t* rp = reinterpret_cast<const uint16_t*>(
          __shfl_sync(0xFFFFFFFFu, reinterpret_cast<unsigned long long>(row_ptr), m));
      const bool lv = __shfl_sync(0xFFFFFFFFu, live, m);
#pragma unroll
      for (int c0 = 0; c0 < kChunksRow; c0 += 32) {
        const int c = c0 + lane;
        if (c < kChunksRow)
          cp_async_16(smem_u32(dst + (c / 8) * 8192 + sw128_offset(kr, c % 8)), lv ? rp + c * 8 : p.kv, lv ? 16u : 0u);
      }
    }
  };

  const uint32_t idesc_qk = idesc_bf16(128, kTileKeys, false, false);
  const uint32_t idesc_pv = idesc_bf16(128, C::kDvc, false, true);

  float m_ref = kNegSentinel, l_sum = 0.f;
  bool o_valid = false, pv_pending = false, aborted = false;
  uint32_t s_phase = 0, o_phase = 0;

  if (n_tiles > 0) load_tile(0, 0);
  cp_async_commit();

  for (int i = 0; i < n_tiles; ++i) {
    const int st = i % C::kStages;
    cp_async_wait<0>();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t* lw = reinterpret_cast<const uint32_t*>(live_sm + st * kTileKeys);
    uint32_t any = 0;
#pragma unroll
    for (int x = 0; x < kTileKeys / 4; ++x) any |= lw[x];
    const uint8_t* kv_st = kv_sm + st * L::kKvStage;

    if (any && tid == 0) {  // S = Q K^T
      const uint32_t kv0 = smem_u32(kv_st), qs0 = smem_u32(q_sm);
#pragma unroll 1
      for (int ks = 0; ks < C::kDkTmem / 16; ++ks)
        mma_bf16_ts(tmem + kColS, tmem + kColQ + ks * 8,
                    smem_desc(kv0 + (ks / 4) * 8192 + (ks % 4) * 32, 16, 1024, kSwizzle128B), idesc_qk, ks > 0 ? 1u : 0u);
#pragma unroll 1
      for (int kk = 0; kk < (DK - C::kDkTmem) / 16; ++kk)
        mma_bf16_ss(tmem + kColS, smem_desc(qs0 + (kk / 4) * 16384 + (kk % 4) * 32, 16, 1024, kSwizzle128B),
                    smem_desc(kv0 + (C::kDkTmem / 64 + kk / 4) * 8192 + (kk % 4) * 32, 16, 1024, kSwizzle128B),
                    idesc_qk, 1u);
      mma_commit(&bar_s);
    }
    // the previous PV must be done before its stage is refilled
    if (pv_pending) {
      const bool ok = mbar_wait(&bar_o, o_phase & 1);
      ++o_phase;
      pv_pending = false;
      if (__syncthreads_or(!ok)) { aborted = true; break; }
    }
    if (i + 1 < n_tiles) load_tile(i + 1, (i + 1) % C::kStages);
    cp_async_commit();
    if (!any) continue;

    {
      const bool ok = mbar_wait(&bar_s, s_phase & 1);
      ++s_phase;
      if (__syncthreads_or(!ok)) { aborted = true; break; }
    }
    tc_fence_after();

    // ---- softmax over this tile (thread = head row)
    uint32_t sv[64];
    {
      uint32_t a[32], c[32];
      tmem_ld32_sync(lane_base + kColS, a);
      tmem_ld32_sync(lane_base + kColS + 32, c);
#pragma unroll
      for (int x = 0; x < 32; ++x) { sv[x] = a[x]; sv[32 + x] = c[x]; }
    }
    const uint8_t* live_t = live_sm + st * kTileKeys;
    float mt = kNegSentinel;
#pragma unroll
    for (int x = 0; x < 64; ++x) {
      const float s = live_t[x] ? __uint_as_float(sv[x]) * p.scale_log2 : kNegSentinel;
      sv[x] = __float_as_uint(s);
      mt = fmaxf(mt, s);
    }
    float alpha = 1.f;
    const bool rescale = mt > m_ref + kRescaleThreshold;
    if (rescale) {
      alpha = exp2f(m_ref - mt);
      m_ref = mt;
      l_sum *= alpha;
    }
    uint32_t pw[32];
    float psum = 0.f;
#pragma unroll
    for (int x = 0; x < 32; ++x) {
      const float p0 = live_t[2 * x] ? exp2f(__uint_as_float(sv[2 * x]) - m_ref) : 0.f;
      const float p1 = live_t[2 * x + 1] ? exp2f(__uint_as_float(sv[2 * x + 1]) - m_ref) : 0.f;
      const __nv_bfloat162 pb = __floats2bfloat162_rn(p0, p1);
      // the normaliser adds the bf16 weights that the PV product uses
      psum += __bfloat162float(pb.x) + __bfloat162float(pb.y);
      pw[x] = *reinterpret_cast<const uint32_t*>(&pb);
    }
    l_sum += psum;
#pragma unroll
    for (int c = 0; c < 8; ++c)
      *reinterpret_cast<uint4*>(p_sm + sw128_offset(tid, c)) = make_uint4(pw[4 * c], pw[4 * c + 1], pw[4 * c + 2], pw[4 * c + 3]);
    if (o_valid && __any_sync(0xFFFFFFFFu, rescale)) {
#pragma unroll 1
      for (int c = 0; c < C::kDvc; c += 32) {
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
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {  // O += P V
      const uint32_t p0 = smem_u32(p_sm), v0 = smem_u32(kv_st) + (r * C::kDvc / 64) * 8192;
#pragma unroll
      for (int ks = 0; ks < kTileKeys / 16; ++ks)
        mma_bf16_ss(tmem + kColO, smem_desc(p0 + ks * 32, 16, 1024, kSwizzle128B),
                    smem_desc(v0 + ks * 2048, 8192, 1024, kSwizzle128B), idesc_pv, (o_valid || ks > 0) ? 1u : 0u);
      mma_commit(&bar_o);
    }
    o_valid = true;
    pv_pending = true;
  }
  cp_async_wait<0>();
  if (pv_pending && !aborted) {
    const bool ok = mbar_wait(&bar_o, o_phase & 1);
    if (__syncthreads_or(!ok)) aborted = true;
  }
  tc_fence_after();
  if (aborted) {
    if (tid == 0) report(p.dev_status, DSA_DEVERR_TIMEOUT);
    o_valid = false;
    l_sum = 0.f;
  }

  // ---- epilogue
  const int h = tid;
  const bool have = o_valid && l_sum > 0.f;
  if (p.splits == 1) {
    const float inv = have ? 1.f / l_sum : 0.f;
    uint16_t* dst = p.out + (static_cast<int64_t>(t) * p.H + h) * DV + r * C::kDvc;
#pragma unroll 1
    for (int c = 0; c < C::kDvc; c += 32) {
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
    if (r == 0 && h < p.H && p.lse != nullptr)
      p.lse[static_cast<int64_t>(t) * p.H + h] = have ? (m_ref + log2f(l_sum)) * kLn2 : -INFINITY;
  } else {
    const int64_t row = (static_cast<int64_t>(t) * p.H + h) * p.splits + j;
    float* dst = p.o_part + row * DV + r * C::kDvc;
#pragma unroll 1
    for (int c = 0; c < C::kDvc; c += 32) {
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
    if (r == 0 && h < p.H) p.ml_part[row] = make_float2(o_valid ? m_ref : kNegSentinel, o_valid ? l_sum : 0.f);
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, C::kTmemCols);
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

dsa_status_t launch_mla(const MlaParams& p, int Dk, int Dv, cudaStream_t s) {
  const int64_t grid = static_cast<int64_t>(p.T) * p.splits * dv_split_for(Dv);
  if (grid > 0x7FFFFFFF) return fail(DSA_ERR_UNSUPPORTED, "sparse_mla: grid too large");
  dsa_status_t st;
  if (Dk == 576) {
    st = allow_smem(sparse_mla_kernel<576, 512>, MlaSmem<576, 512>::kTotal, g_smem_big);
    if (st != DSA_OK) return st;
    sparse_mla_kernel<576, 512><<<static_cast<unsigned>(grid), kThreads, MlaSmem<576, 512>::kTotal, s>>>(p);
  } else {
    st = allow_smem(sparse_mla_kernel<80, 64>, MlaSmem<80, 64>::kTotal, g_smem_tiny);
    if (st != DSA_OK) return st;
    sparse_mla_kernel<80, 64><<<static_cast<unsigned>(grid), kThreads, MlaSmem<80, 64>::kTotal, s>>>(p);
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
  if (kv_block_stride < static_cast<int64_t>(block_size) * Dk || kv_block_stride % 8)
    return fail(DSA_ERR_INVALID_ARG, "%s: kv_block_stride %lld must be >= block_size*Dk and a multiple of 8", name,
                static_cast<long long>(kv_block_stride));
  return check_device();
}

MlaParams make_params(const void* q, const void* kv_cache, int64_t kv_block_stride, int32_t num_blocks,
                      const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens,
                      const int32_t* query_start_loc, const int32_t* topk_idx, int32_t B, int32_t T, int32_t H,
                      int32_t index_topk, int32_t block_size, float softmax_scale, int32_t splits, void* out,
                      float* lse, int32_t* dev_status) {
  MlaParams p;
  p.q = static_cast<const uint16_t*>(q);
  p.kv = static_cast<const uint16_t*>(kv_cache);
  p.kv_block_stride = kv_block_stride;
  p.num_blocks = num_blocks;
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
  const int tiles = (index_topk + kTileKeys - 1) / kTileKeys;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0) sms = v;
  } else {
    cudaGetLastError();
  }
  const int64_t units = static_cast<int64_t>(T) * dv_split_for(Dv);
  int best = 1;
  int64_t best_cost = INT64_MAX;
  for (int s = 1; s <= std::min(32, tiles); ++s) {
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
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  MlaParams p = make_params(q, kv_cache, kv_block_stride, num_blocks, block_table, bt_stride, seq_lens,
                            query_start_loc, topk_idx, B, T, H, index_topk, block_size, softmax_scale, splits, out,
                            lse, dev_status);
  if (splits > 1) {
    const size_t need = sparse_mla_workspace_size(T, H, Dv, splits);
    if (workspace == nullptr || ws_bytes < need || !aligned16(workspace))
      return fail(DSA_ERR_WORKSPACE, "sparse_mla_decode: %d splits need %zu workspace bytes (16-byte aligned), got %zu",
                  splits, need, ws_bytes);
    p.o_part = static_cast<float*>(workspace);
    p.ml_part = reinterpret_cast<float2*>(p.o_part + static_cast<int64_t>(T) * H * splits * Dv);
  }
  st = launch_mla(p, Dk, Dv, s);
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
  MlaParams p = make_params(q, kv_cache, kv_block_stride, num_blocks, block_table, bt_stride, seq_lens,
                            query_start_loc, topk_idx, B, T, H, index_topk, block_size, softmax_scale, 1, out, lse,
                            dev_status);
  return launch_mla(p, Dk, Dv, reinterpret_cast<cudaStream_t>(stream));
}
