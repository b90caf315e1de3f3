// a2: exact per-row top-k by radix select.
//
// Each fp32 logit maps to a 32-bit key whose unsigned order is the float
// order (-0.0 is folded onto +0.0 first, so the two tie). Four 8-bit radix
// passes find the exact key T of the k-th largest element and how many
// elements equal to T are needed; a final pass compacts, in position order,
// every element above T plus the first `need` elements equal to T. The
// output is therefore the exact top-k set with ties resolved toward the lower
// position, listed in ascending position.
//
// Long rows use two exact stages: the top-k of every 8192-key chunk, then
// the top-k of the concatenated candidates. Any element of the global top-k
// is in its chunk's top-k, and the candidates stay in position order, so the
// second stage sees the same ties in the same order (vLLM PR #38476 review
// thread: the global top-k is recoverable from per-chunk top-k candidates).
#include <algorithm>

#include "common.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kChunk = 8192;       // keys per first-stage CTA
constexpr int kCacheCap = 32768;   // rows up to this many keys are staged in shared memory

struct TopkShared {
  uint32_t hist[kWarps][256];
  uint32_t total[256];
  uint32_t scan[kWarps];
  uint32_t sel_digit, sel_gt;
};

__device__ __forceinline__ uint32_t order_key(float v) {
  uint32_t b = __float_as_uint(v);
  b = (b == 0x80000000u) ? 0u : b;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// position of token t inside its request: (request index, valid length)
__device__ __forceinline__ int valid_length(const int32_t* seq_lens, const int32_t* qsl, int B, int t, int64_t ld) {
  int lo = 0, hi = B - 1;  // last request with qsl[b] <= t
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(qsl + mid) <= t) lo = mid; else hi = mid - 1;
  }
  const int q0 = __ldg(qsl + lo), q1 = __ldg(qsl + lo + 1);
  const int64_t v = static_cast<int64_t>(__ldg(seq_lens + lo)) - (q1 - q0) + (t - q0) + 1;
  return static_cast<int>(max(static_cast<int64_t>(0), min(v, ld)));
}

// Exclusive block scan of `v` (1024 threads); returns the prefix, sets `total`.
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t& total, TopkShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) sh.scan[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint32_t s = sh.scan[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, s, off);
      if (lane >= off) s += y;
    }
    sh.scan[lane] = s;  // inclusive over warps
  }
  __syncthreads();
  const uint32_t before_warp = warp > 0 ? sh.scan[warp - 1] : 0u;
  total = sh.scan[kWarps - 1];
  const uint32_t r = before_warp + x - v;
  __syncthreads();  // sh.scan is reused by the next call
  return r;
}

// Selects the k largest of n values (position i holds vals[i]; ids[i] < 0
// marks an empty candidate). Writes min(k, n) results in position order to
// out_idx (ids[i], or base + i when ids is null) and out_val (if non-null),
// then pads up to k with -1 / -inf.
__device__ void block_select(const float* __restrict__ vals, const int32_t* __restrict__ ids, int n, int k,
                             int32_t base, int32_t* __restrict__ out_idx, float* __restrict__ out_val,
                             uint32_t* kcache, TopkShared& sh) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto make_key = [&](int i) -> uint32_t {
    if (ids != nullptr && __ldg(ids + i) < 0) return 0u;
    return order_key(__ldg(vals + i));
  };
  auto emit = [&](int i, int pos) {
    out_idx[pos] = ids != nullptr ? __ldg(ids + i) : base + i;
    if (out_val != nullptr) out_val[pos] = __ldg(vals + i);
  };
  if (n <= k) {
    for (int i = tid; i < n; i += kThreads) emit(i, i);
    for (int i = n + tid; i < k; i += kThreads) {
      out_idx[i] = -1;
      if (out_val != nullptr) out_val[i] = -INFINITY;
    }
    return;
  }
  if (kcache != nullptr) {
    // eight independent loads per thread in flight at a time
    for (int base = 0; base < n; base += 8 * kThreads) {
      uint32_t kk[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = base + u * kThreads + tid;
        kk[u] = i < n ? make_key(i) : 0u;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = base + u * kThreads + tid;
        if (i < n) kcache[i] = kk[u];
      }
    }
    __syncthreads();
  }
  auto key_at = [&](int i) -> uint32_t { return kcache != nullptr ? kcache[i] : make_key(i); };

  uint32_t prefix = 0, mask = 0;
  int need = k;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = tid; i < kWarps * 256; i += kThreads) (&sh.hist[0][0])[i] = 0u;
    __syncthreads();
    for (int i = tid; i < n; i += kThreads) {
      const uint32_t key = key_at(i);
      if ((key & mask) == prefix) atomicAdd(&sh.hist[warp][(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    uint32_t suffix = 0;  // elements whose digit is >= tid, within this warp's 32 digits
    if (tid < 256) {
      uint32_t s = 0;
#pragma unroll 8
      for (int w = 0; w < kWarps; ++w) s += sh.hist[w][tid];
      sh.total[tid] = s;
      suffix = s;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_down_sync(0xFFFFFFFFu, suffix, off);
        if (lane + off < 32) suffix += y;
      }
      if (lane == 0) sh.scan[warp] = suffix;
    }
    __syncthreads();
    if (tid < 256) {
      uint32_t above = 0;  // elements in digits of higher warps
      for (int w = warp + 1; w < 8; ++w) above += sh.scan[w];
      const uint32_t incl = suffix + above;  // elements with digit >= tid
      const uint32_t gt = incl - sh.total[tid];        // elements with digit > tid
      if (gt < static_cast<uint32_t>(need) && static_cast<uint32_t>(need) <= incl) {
        sh.sel_digit = tid;
        sh.sel_gt = gt;
      }
    }
    __syncthreads();
    need -= static_cast<int>(sh.sel_gt);
    prefix |= sh.sel_digit << shift;
    mask |= 255u << shift;
    __syncthreads();
  }
  const uint32_t thr = prefix;

  // ordered compaction: everything above thr, then the first `need` equal to thr
  if (kcache != nullptr) {
    // staged rows: each thread owns one contiguous segment, one block scan
    const int seg = (n + kThreads - 1) / kThreads;
    const int lo = min(n, tid * seg), hi = min(n, lo + seg);
    uint32_t cg = 0, ce = 0;
    for (int i = lo; i < hi; ++i) {
      const uint32_t key = kcache[i];
      cg += key > thr;
      ce += key == thr;
    }
    uint32_t total;
    const uint32_t before = block_exclusive_scan(cg | (ce << 16), total, sh);
    uint32_t g = before & 0xFFFFu, e = before >> 16;
    for (int i = lo; i < hi; ++i) {
      const uint32_t key = kcache[i];
      if (key > thr) {
        emit(i, static_cast<int>(g + min(e, static_cast<uint32_t>(need))));
        ++g;
      } else if (key == thr) {
        if (e < static_cast<uint32_t>(need)) emit(i, static_cast<int>(g + e));
        ++e;
      }
    }
    return;
  }
  uint32_t run_gt = 0, run_eq = 0;
  for (int start = 0; start < n; start += kThreads) {
    const int i = start + tid;
    uint32_t key = 0;
    bool gt = false, eq = false;
    if (i < n) {
      key = key_at(i);
      gt = key > thr;
      eq = key == thr;
    }
    uint32_t total;
    const uint32_t before = block_exclusive_scan((gt ? 1u : 0u) | (eq ? 0x10000u : 0u), total, sh);
    const uint32_t gt_before = run_gt + (before & 0xFFFFu);
    const uint32_t eq_before = run_eq + (before >> 16);
    if (gt) emit(i, static_cast<int>(gt_before + min(eq_before, static_cast<uint32_t>(need))));
    if (eq && eq_before < static_cast<uint32_t>(need)) emit(i, static_cast<int>(gt_before + eq_before));
    run_gt += total & 0xFFFFu;
    run_eq += total >> 16;
  }
}

struct TopkParams {
  const float* logits;
  int64_t ld;
  const int32_t* seq_lens;
  const int32_t* qsl;
  int B, k, nchunks;
  int32_t* out;
  int32_t* cand_idx;
  float* cand_val;
  int use_cache;
};

__global__ void __launch_bounds__(kThreads) topk_single_kernel(const TopkParams p) {
  extern __shared__ uint32_t kcache[];
  __shared__ TopkShared sh;
  const int t = blockIdx.x;
  const int n = valid_length(p.seq_lens, p.qsl, p.B, t, p.ld);
  block_select(p.logits + static_cast<int64_t>(t) * p.ld, nullptr, n, p.k, 0, p.out + static_cast<int64_t>(t) * p.k,
               nullptr, (p.use_cache && n <= kCacheCap) ? kcache : nullptr, sh);
}

__global__ void __launch_bounds__(kThreads) topk_stage1_kernel(const TopkParams p) {
  extern __shared__ uint32_t kcache[];
  __shared__ TopkShared sh;
  const int c = blockIdx.x, t = blockIdx.y;
  const int valid = valid_length(p.seq_lens, p.qsl, p.B, t, p.ld);
  if (valid <= p.k) return;  // the second stage writes such rows directly
  const int begin = c * kChunk;
  const int n = max(0, min(valid - begin, kChunk));
  const int64_t slot = (static_cast<int64_t>(t) * p.nchunks + c) * p.k;
  block_select(p.logits + static_cast<int64_t>(t) * p.ld + begin, nullptr, n, p.k, begin, p.cand_idx + slot,
               p.cand_val + slot, kcache, sh);
}

__global__ void __launch_bounds__(kThreads) topk_stage2_kernel(const TopkParams p) {
  extern __shared__ uint32_t kcache[];
  __shared__ TopkShared sh;
  const int t = blockIdx.x;
  const int valid = valid_length(p.seq_lens, p.qsl, p.B, t, p.ld);
  int32_t* out = p.out + static_cast<int64_t>(t) * p.k;
  if (valid <= p.k) {
    block_select(p.logits + static_cast<int64_t>(t) * p.ld, nullptr, valid, p.k, 0, out, nullptr, nullptr, sh);
    return;
  }
  const int n = p.nchunks * p.k;
  const int64_t slot = static_cast<int64_t>(t) * n;
  block_select(p.cand_val + slot, p.cand_idx + slot, n, p.k, 0, out, nullptr, (p.use_cache && n <= kCacheCap) ? kcache : nullptr,
               sh);
}

bool g_smem_single = false, g_smem_s1 = false, g_smem_s2 = false;

bool use_two_stage(int32_t T, int64_t ld, int32_t k) {
  return ld > 2 * kChunk && k < kChunk && T < 2 * num_sms();
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" size_t dsa_topk_workspace_size(int32_t T, int64_t ld, int32_t index_topk) {
  if (T <= 0 || ld <= 0 || index_topk <= 0) return 0;
  if (!use_two_stage(T, ld, index_topk)) return 0;
  const int64_t nchunks = (ld + kChunk - 1) / kChunk;
  return static_cast<size_t>(T) * nchunks * index_topk * (sizeof(int32_t) + sizeof(float));
}

extern "C" dsa_status_t dsa_topk(const float* logits, int64_t ld, const int32_t* seq_lens,
                                 const int32_t* query_start_loc, int32_t B, int32_t T, int32_t index_topk,
                                 int32_t* topk_idx, void* workspace, size_t ws_bytes, dsa_stream_t stream) {
  if (B < 0 || T < 0 || ld <= 0 || index_topk <= 0)
    return fail(DSA_ERR_INVALID_ARG, "dsa_topk: bad sizes B=%d T=%d ld=%lld k=%d", B, T, (long long)ld, index_topk);
  if (T == 0) return DSA_OK;
  if (B == 0) return fail(DSA_ERR_INVALID_ARG, "dsa_topk: T > 0 with B == 0");
  if (!logits || !seq_lens || !query_start_loc || !topk_idx) return fail(DSA_ERR_INVALID_ARG, "dsa_topk: null pointer");
  if (index_topk > 65535) return fail(DSA_ERR_UNSUPPORTED, "dsa_topk: index_topk %d > 65535", index_topk);
  dsa_status_t st = check_device();
  if (st != DSA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  TopkParams p;
  p.logits = logits;
  p.ld = ld;
  p.seq_lens = seq_lens;
  p.qsl = query_start_loc;
  p.B = B;
  p.k = index_topk;
  p.out = topk_idx;
  p.cand_idx = nullptr;
  p.cand_val = nullptr;
  p.nchunks = 0;
  p.use_cache = 1;
  if (use_two_stage(T, ld, index_topk)) {
    const size_t need = dsa_topk_workspace_size(T, ld, index_topk);
    if (workspace == nullptr || ws_bytes < need)
      return fail(DSA_ERR_WORKSPACE, "dsa_topk: needs %zu workspace bytes, got %zu", need, ws_bytes);
    p.nchunks = static_cast<int>((ld + kChunk - 1) / kChunk);
    p.cand_idx = static_cast<int32_t*>(workspace);
    p.cand_val = reinterpret_cast<float*>(p.cand_idx + static_cast<int64_t>(T) * p.nchunks * index_topk);
    const int s1 = kChunk * 4;
    st = allow_smem(topk_stage1_kernel, s1, g_smem_s1);
    if (st != DSA_OK) return st;
    topk_stage1_kernel<<<dim3(p.nchunks, T), kThreads, s1, s>>>(p);
    st = check_launch("topk_stage1_kernel");
    if (st != DSA_OK) return st;
    const int n2 = p.nchunks * index_topk;
    const int s2 = (n2 <= kCacheCap ? n2 : 0) * 4;
    p.use_cache = n2 <= kCacheCap;
    st = allow_smem(topk_stage2_kernel, kCacheCap * 4, g_smem_s2);
    if (st != DSA_OK) return st;
    topk_stage2_kernel<<<T, kThreads, s2, s>>>(p);
    return check_launch("topk_stage2_kernel");
  }
  const int64_t cache_keys = ld <= kCacheCap ? ld : 0;
  p.use_cache = cache_keys > 0;
  st = allow_smem(topk_single_kernel, kCacheCap * 4, g_smem_single);
  if (st != DSA_OK) return st;
  topk_single_kernel<<<T, kThreads, static_cast<int>(cache_keys * 4), s>>>(p);
  return check_launch("topk_single_kernel");
}
