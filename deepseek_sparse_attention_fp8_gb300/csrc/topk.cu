// a2: exact per-row top-k.
//
// Each fp32 logit maps to a 32-bit key whose unsigned order is the float
// order (-0.0 is folded onto +0.0 first, so the two tie). The selection
// finds the exact key T of the k-th largest element and how many elements
// equal to T are needed; a final pass compacts, in position order, every
// element above T plus the first `need` elements equal to T. The output is
// therefore the exact top-k set with ties resolved toward the lower
// position, listed in ascending position.
//
// Rows of at most 32768 keys, when one CTA per row already fills the GPU,
// take topk_row_kernel: one CTA holds the whole row in registers (each warp a
// contiguous run), so the steps below need no staging and no cluster.
// Otherwise a row is cut into P contiguous parts (P = 1..8), one CTA each, the P CTAs
// of a row forming a thread-block cluster that combines its histograms and
// counts through distributed shared memory:
//   1. each CTA stages its part's keys in shared memory and finds the part's
//      finite minimum and maximum; the cluster's range gives 2048 bins that
//      are linear in the value (outside values clamp to the end bins);
//   2. the cluster's histogram of those bins gives, from its suffix sums, the
//      bin holding the k-th largest key. The binning is monotonic, so every
//      element of a higher bin is larger than every element of a lower one;
//   3. T is the exact rank selection among that bin's elements (tens, for
//      logits of a smooth distribution, gathered into every CTA), whose
//      positions and the parts' counts above the bin also give each part's
//      output offset. A bin of more than 1024 elements is refined instead by
//      histograms over its key interval, each level shrinking the interval
//      2048-fold, until it holds one key; the parts then exchange counts;
//   4. an ordered compaction writes each part's selected positions.
// (vLLM PR #38476 review thread: index_topk selection, one exact top-k per
// query row.)
#include <algorithm>

#include "common.cuh"
#include "ptx.cuh"

namespace dsa {
namespace {

using namespace ptx;

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxParts = 8;     // CTAs per row (portable cluster size)
constexpr int kSegCap = 32768;   // keys of one part staged in shared memory
constexpr int kBins = 2048;      // histogram bins
constexpr int kCandCap = kThreads;  // threshold-bin elements ranked directly (one per thread)
constexpr int kListCap = 512;       // candidate positions one warp may record (cached cluster kernel)
constexpr int kFilterRatio = 8;     // rows with valid >= 8 k record candidates above a sampled bin

struct TopkShared {
  uint32_t hist[kBins];   // this CTA's histogram (read by the peers)
  uint32_t ghist[kBins];  // the row's histogram (slices written by the owners)
  uint32_t cand_key[kCandCap];  // the threshold bin's elements of the whole row
  int32_t cand_pos[kCandCap];
  uint32_t loc_key[kCandCap];   // ... of this part
  int32_t loc_pos[kCandCap];
  uint32_t part_above[kMaxParts];  // per part: elements in bins above the threshold bin
  uint32_t part_kmin[kMaxParts], part_kmax[kMaxParts];
  uint32_t part_gt[kMaxParts], part_eq[kMaxParts];
  uint32_t push_base[kMaxParts];
  uint32_t cand_n, loc_n;
  uint64_t scan[kWarps];
  float red_f[2][kWarps];
  uint32_t red_u[3][kWarps];
  uint32_t part_ovf[1];              // a warp's candidate list overflowed in this part
  uint32_t bsel, above, thr, gtotal;
  uint32_t thr_gt;  // threshold-bin elements above the threshold key (row kernel)
  int32_t qsl_s[kThreads + 1], sl_s[kThreads];  // the batch's query_start_loc and seq_lens (B <= kThreads)
};

__device__ __forceinline__ uint32_t order_key(float v) {
  uint32_t b = __float_as_uint(v);
  b = (b == 0x80000000u) ? 0u : b;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
// float value of an order key (the inverse map; -0.0 comes back as +0.0)
__device__ __forceinline__ float key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}
// Monotonic bin of v: v <= u implies bin(v) <= bin(u). NaNs go to the end
// bin on the side their order key puts them.
__device__ __forceinline__ int lin_bin(float v, float lo, float inv_w) {
  if (v != v) return (__float_as_uint(v) & 0x80000000u) ? 0 : kBins - 1;
  const float x = __fmul_rn(__fsub_rn(v, lo), inv_w);
  return static_cast<int>(fminf(fmaxf(x, 0.f), static_cast<float>(kBins - 1)));
}

__device__ __forceinline__ void st_cluster_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t atom_add_cluster_u32(uint32_t addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(addr), "r"(v) : "memory");
  return old;
}

// valid(t): the number of leading positions of row t that are ranked. Every
// thread of the block calls it: the request of token t is the last b with
// query_start_loc[b] <= t, counted over the block. Up to kThreads requests,
// query_start_loc and seq_lens arrive in one round of loads.
struct TopkShared;
__device__ int valid_length(const int32_t* seq_lens, const int32_t* qsl, int B, int t, int64_t ld, TopkShared& sh);

// Exclusive block scan of `v`; returns the prefix and sets `total`. Two
// 32-bit counts can travel packed in one 64-bit value.
__device__ __forceinline__ uint64_t block_exclusive_scan(uint64_t v, uint64_t& total, TopkShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint64_t x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint64_t y = __shfl_up_sync(0xFFFFFFFFu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) sh.scan[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint64_t s = lane < kWarps ? sh.scan[lane] : 0ull;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint64_t y = __shfl_up_sync(0xFFFFFFFFu, s, off);
      if (lane >= off) s += y;
    }
    if (lane < kWarps) sh.scan[lane] = s;  // inclusive over warps
  }
  __syncthreads();
  const uint64_t before_warp = warp > 0 ? sh.scan[warp - 1] : 0ull;
  total = sh.scan[kWarps - 1];
  const uint64_t r = before_warp + x - v;
  __syncthreads();  // sh.scan is reused by the next call
  return r;
}

// The block-wide minimum and maximum of the warps' partials in red_f (after
// a barrier that follows their writes): each warp reduces the 32 partials
// with shuffles.
static_assert(kWarps == 32, "one partial per lane");
__device__ __forceinline__ void block_range(float& lo, float& hi, const TopkShared& sh) {
  lo = sh.red_f[0][threadIdx.x & 31];
  hi = sh.red_f[1][threadIdx.x & 31];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    lo = fminf(lo, __shfl_xor_sync(0xFFFFFFFFu, lo, off));
    hi = fmaxf(hi, __shfl_xor_sync(0xFFFFFFFFu, hi, off));
  }
}

__device__ int valid_length(const int32_t* seq_lens, const int32_t* qsl, int B, int t, int64_t ld, TopkShared& sh) {
  const int tid = static_cast<int>(threadIdx.x);
  int b, q0, q1, sl;
  if (B <= kThreads) {
    const int qv = tid <= B ? __ldg(qsl + tid) : 0;
    const int sv = tid < B ? __ldg(seq_lens + tid) : 0;
    if (tid <= B) sh.qsl_s[tid] = qv;
    if (tid < B) sh.sl_s[tid] = sv;
    b = max(0, __syncthreads_count(tid < B && qv <= t) - 1);
    q0 = sh.qsl_s[b];
    q1 = sh.qsl_s[b + 1];
    sl = sh.sl_s[b];
  } else {
    int cnt = 0;
    for (int j0 = 0; j0 < B; j0 += kThreads) {
      const int j = j0 + tid;
      cnt += __syncthreads_count(j < B && __ldg(qsl + j) <= t);
    }
    b = max(0, cnt - 1);
    q0 = __ldg(qsl + b);
    q1 = __ldg(qsl + b + 1);
    sl = __ldg(seq_lens + b);
  }
  const int64_t v = static_cast<int64_t>(sl) - (q1 - q0) + (t - q0) + 1;
  return static_cast<int>(max(static_cast<int64_t>(0), min(v, ld)));
}

// The bin of the row histogram `ghist` holding the `need`-th largest element
// (bins scanned from the top): sets sh.bsel and sh.above (elements in higher
// bins) when 1 <= need <= the histogram's total, which goes to sh.gtotal.
__device__ void find_bin(TopkShared& sh, uint32_t need) {
  const int tid = threadIdx.x;
  constexpr int kPer = kBins / kThreads;  // bins per thread, descending
  uint32_t h[kPer], sum = 0;
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    h[u] = sh.ghist[kBins - 1 - (kPer * tid + u)];
    sum += h[u];
  }
  uint64_t tot;
  uint32_t before = static_cast<uint32_t>(block_exclusive_scan(sum, tot, sh));
#pragma unroll
  for (int u = 0; u < kPer; ++u) {
    if (before < need && need <= before + h[u]) {
      sh.bsel = kBins - 1 - (kPer * tid + u);
      sh.above = before;
    }
    before += h[u];
  }
  if (tid == 0) sh.gtotal = static_cast<uint32_t>(tot);
  __syncthreads();
}

// Output modes. kPositions: the selected positions of each row, -1 padded
// (dsa_topk). kWindow: the row is one window of the keys, starting at key
// key_begin; its n = min(k, valid keys in the window) selections go, with
// their values, to the candidate arrays at the window's offset (window index
// x kcand, kcand = min(k, win)), no padding. kFinal: the row is the
// candidate array itself (positions = candidate slots, ascending in key);
// the selected slots' keys are written, -1 padded.
enum TopkMode { kPositions = 0, kWindow = 1, kFinal = 2 };

struct TopkParams {
  const float* logits;
  int64_t ld;
  const int32_t* seq_lens;
  const int32_t* qsl;
  int B, k, parts;
  int32_t* out;
  int mode;
  int64_t key_begin;
  int32_t win, kcand, cand_stride;
  float* cand_val;
  int32_t* cand_idx;
};

// The row's length in the mode's own positions, from the token's valid
// length v (keys 0..v-1) clipped to ld.
template <int MODE>
__device__ __forceinline__ int row_length(const TopkParams& p, int v) {
  if constexpr (MODE == kWindow) return static_cast<int>(max(static_cast<int64_t>(0), min(static_cast<int64_t>(v) - p.key_begin, p.ld)));
  if constexpr (MODE == kFinal) {
    const int full = v / p.win, rem = v - full * p.win;
    return static_cast<int>(min(static_cast<int64_t>(full) * p.kcand + min(p.kcand, rem), p.ld));
  }
  return static_cast<int>(min(static_cast<int64_t>(v), p.ld));
}

// Writes selection `slot` (position `pos` of row t, value `val`) in the mode's form.
template <int MODE>
__device__ __forceinline__ void emit(const TopkParams& p, int t, int slot, int pos, float val) {
  if constexpr (MODE == kWindow) {
    const int64_t at = static_cast<int64_t>(t) * p.cand_stride + (p.key_begin / p.win) * p.kcand + slot;
    p.cand_idx[at] = static_cast<int32_t>(p.key_begin + pos);
    p.cand_val[at] = val;
  } else if constexpr (MODE == kFinal) {
    p.out[static_cast<int64_t>(t) * p.k + slot] = __ldg(p.cand_idx + static_cast<int64_t>(t) * p.cand_stride + pos);
  } else {
    (void)val;
    p.out[static_cast<int64_t>(t) * p.k + slot] = pos;
  }
}
// An empty slot (slot >= the row's length): -1, except in window mode.
template <int MODE>
__device__ __forceinline__ void emit_empty(const TopkParams& p, int t, int slot) {
  if constexpr (MODE != kWindow) p.out[static_cast<int64_t>(t) * p.k + slot] = -1;
}

// kCached: the part's keys are staged in shared memory (else re-read)
template <bool kCached, int MODE>
__global__ void __launch_bounds__(kThreads) topk_kernel(const TopkParams p) {
  extern __shared__ uint32_t kc[];  // this part's keys (when cached)
  __shared__ TopkShared sh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int P = p.parts;
  const int r = static_cast<int>(cluster_ctarank());
  const int t = blockIdx.x / P;
  const int k = p.k;
  // Launched as a programmatic dependent of the logits producer. The row's
  // valid length comes from the step's inputs, which that kernel does not
  // write, so it is found first; then wait for the logits and let the next
  // kernel's CTAs be scheduled.
  const int n = row_length<MODE>(p, valid_length(p.seq_lens, p.qsl, p.B, t, 0x7FFFFFFF, sh));
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const float* row = p.logits + static_cast<int64_t>(t) * p.ld;
  // The row's parts are cut by ld, so the first values are loaded whatever
  // valid(t) is; positions at or past valid(t) are ignored afterwards.
  const int ld = static_cast<int>(p.ld);
  const int seg = (ld + P - 1) / P;
  const int s0 = min(ld, r * seg);
  const int m_ld = min(ld, s0 + seg) - s0;
  const int m = max(0, min(n - s0, m_ld));  // this part's valid length (may be 0)
  // warp w stages (and later compacts) the contiguous run [w0, w1) of the part
  const int wrun = (((m + kWarps - 1) / kWarps) + 31) & ~31;
  const int w0 = min(m, warp * wrun), w1 = min(m, w0 + wrun);
  constexpr int kFirst = 4;  // values loaded before the samples, overlapping their latency
  float v_first[kFirst];
#pragma unroll
  for (int u = 0; u < kFirst; ++u) {
    const int i = w0 + 32 * u + lane;
    v_first[u] = i < w1 ? __ldg(row + s0 + i) : 0.f;
  }
  if (n <= k) {  // every valid position, then -1 (the same branch for the whole cluster)
    const int o0 = static_cast<int>(static_cast<int64_t>(r) * k / P);
    const int o1 = static_cast<int>(static_cast<int64_t>(r + 1) * k / P);
    for (int i = o0 + tid; i < o1; i += kThreads) {
      if (i < n) emit<MODE>(p, t, i, i, MODE == kWindow ? __ldg(row + i) : 0.f);
      else emit_empty<MODE>(p, t, i);
    }
    return;
  }
  // Rows that keep a small fraction of their keys record, per warp and in
  // position order, the positions whose bin is at least a bin taken from the
  // row's samples (a 1.25x margin on k/valid); the later passes then visit
  // those candidates only. The same in every CTA of the row.
  const bool use_filter = kCached && static_cast<int64_t>(n) >= static_cast<int64_t>(kFilterRatio) * k;
  uint16_t* lst = reinterpret_cast<uint16_t*>(kc + ((seg + 7) & ~7)) + warp * kListCap;  // this warp's list
  auto key_at = [&](int i) -> uint32_t {
    if constexpr (kCached) return kc[i];
    else return order_key(__ldg(row + s0 + i));
  };
  auto remote = [&](const void* ptr, int q) -> uint32_t { return mapa_shared(smem_u32(ptr), static_cast<uint32_t>(q)); };
  // barrier over the row's CTAs (a CTA barrier when the row has one CTA)
  auto row_sync = [&]() {
    if (P == 1) __syncthreads();
    else cluster_sync_all();
  };

  // ---- 1. bin range: the finite min and max of 1024 evenly spaced samples of
  // the row, the same in every CTA of the row
  for (int b = tid; b < kBins; b += kThreads) sh.hist[b] = 0u;
  if (tid == 0) {
    sh.cand_n = 0u;
    sh.loc_n = 0u;
  }
  float lo = INFINITY, hi = -INFINITY;
  const int ns = min(n, 1024);
  static_assert(kThreads == 1024, "one sample per thread");
  const float v_smp = tid < ns ? __ldg(row + static_cast<int64_t>(tid) * n / ns) : 0.f;
  {
    if (tid < ns && isfinite(v_smp)) {
      lo = v_smp;
      hi = v_smp;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      lo = fminf(lo, __shfl_xor_sync(0xFFFFFFFFu, lo, off));
      hi = fmaxf(hi, __shfl_xor_sync(0xFFFFFFFFu, hi, off));
    }
    if (lane == 0) {
      sh.red_f[0][warp] = lo;
      sh.red_f[1][warp] = hi;
    }
    __syncthreads();
    lo = INFINITY;
    hi = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      lo = fminf(lo, sh.red_f[0][w]);
      hi = fmaxf(hi, sh.red_f[1][w]);
    }
  }
  float inv_w = hi > lo ? static_cast<float>(kBins) / (hi - lo) : 0.f;
  if (!isfinite(inv_w)) inv_w = 0.f;
  if (!(lo <= hi)) lo = 0.f;
  int b_tau = 0;  // candidates: bin >= b_tau
  if (use_filter) {
    for (int b = tid; b < kBins; b += kThreads) sh.ghist[b] = 0u;
    __syncthreads();
    if (tid < ns) atomicAdd(&sh.ghist[lin_bin(key_value(order_key(v_smp)), lo, inv_w)], 1u);
    __syncthreads();
    const int64_t want = (static_cast<int64_t>(ns) * k * 5 + static_cast<int64_t>(n) * 4 - 1) / (static_cast<int64_t>(n) * 4) + 8;
    find_bin(sh, static_cast<uint32_t>(want < ns ? want : static_cast<int64_t>(ns)));
    b_tau = static_cast<int>(sh.bsel);
  }

  // ---- 2. stage the keys and count them into the part's histogram; CTA r
  // then sums its slice of bins over the cluster and writes the sums into
  // every CTA
  const uint32_t lt = (1u << lane) - 1u;
  int cnt_w = 0;  // candidates this warp saw (the list keeps the first kListCap)
  for (int base = w0; base < w1; base += 8 * 32) {
    float v[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = base + 32 * u + lane;
      v[u] = (base == w0 && u < kFirst) ? v_first[u < kFirst ? u : 0] : (i < w1 ? __ldg(row + s0 + i) : 0.f);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int i = base + 32 * u + lane;
      const bool ok = i < w1;
      const uint32_t key = order_key(v[u]);
      const int b = lin_bin(key_value(key), lo, inv_w);
      if constexpr (kCached) {
        if (ok) kc[i] = key;
      }
      const bool cand = ok && b >= b_tau;  // every valid key when there is no filter
      if (cand) atomicAdd(&sh.hist[b], 1u);
      if (use_filter) {
        const uint32_t msk = __ballot_sync(0xFFFFFFFFu, cand);
        const int slot = cnt_w + __popc(msk & lt);
        if (cand && slot < kListCap) lst[slot] = static_cast<uint16_t>(i);
        cnt_w += __popc(msk);
      }
    }
  }
  if (use_filter) {  // this part's flag, read by the row's CTAs after the next cluster barrier
    const int ovf = __syncthreads_or(cnt_w > kListCap);
    if (tid == 0) sh.part_ovf[0] = static_cast<uint32_t>(ovf);
  }
  const int sl0 = r * (kBins / P), sl1 = (r + 1) * (kBins / P);
  auto reduce_hist = [&]() {
    row_sync();  // every local histogram is complete
    for (int b = sl0 + tid; b < sl1; b += kThreads) {
      uint32_t s = 0;
      for (int q = 0; q < P; ++q) s += ld_cluster_u32(remote(&sh.hist[b], q));
      for (int q = 0; q < P; ++q) st_cluster_u32(remote(&sh.ghist[b], q), s);
    }
    row_sync();  // every CTA holds the whole row histogram
  };
  reduce_hist();
  find_bin(sh, static_cast<uint32_t>(k));
  // the candidate lists serve when the row's candidates hold the top k and
  // no warp's list overflowed; otherwise the passes below visit every key
  bool fast = false;
  if (use_filter) {
    uint32_t any_ovf = 0;
    for (int q = 0; q < P; ++q) any_ovf |= ld_cluster_u32(remote(&sh.part_ovf[0], q));
    const bool enough = sh.gtotal >= static_cast<uint32_t>(k);
    fast = enough && any_ovf == 0;
    if (!enough) {  // the sampled bin was too high: count the remaining keys too
      for (int i = tid; i < m; i += kThreads) {
        const int b = lin_bin(key_value(key_at(i)), lo, inv_w);
        if (b < b_tau) atomicAdd(&sh.hist[b], 1u);
      }
      reduce_hist();
      find_bin(sh, static_cast<uint32_t>(k));
    }
  }
  const int n_lst = min(cnt_w, kListCap);  // this warp's candidates (all of them when fast)
  const int bsel = static_cast<int>(sh.bsel);
  const uint32_t c = sh.ghist[bsel];
  const bool direct = c <= static_cast<uint32_t>(kCandCap);  // the same in every CTA
  int need = k - static_cast<int>(sh.above);  // elements still to take from the bin: 1..c

  // ---- 3. the part's elements of the threshold bin go to every CTA, with
  // the part's count above that bin and its key range within it
  {
    uint32_t kmin = 0xFFFFFFFFu, kmax = 0u, above = 0u;
    auto visit = [&](int i, uint32_t key) {
      const int b = lin_bin(key_value(key), lo, inv_w);
      above += b > bsel;
      if (b != bsel) return;
      kmin = min(kmin, key);
      kmax = max(kmax, key);
      if (direct) {
        const uint32_t slot = atomicAdd(&sh.loc_n, 1u);
        sh.loc_key[slot] = key;
        sh.loc_pos[slot] = s0 + i;
      }
    };
    if (fast) {  // keys outside the lists lie in bins below b_tau <= bsel
      for (int j = lane; j < n_lst; j += 32) {
        const int i = lst[j];
        visit(i, key_at(i));
      }
    } else {
      for (int i0 = 0; i0 < m; i0 += 4 * kThreads) {
        uint32_t kk[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = i0 + u * kThreads + tid;
          kk[u] = i < m ? key_at(i) : 0u;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = i0 + u * kThreads + tid;
          if (i < m) visit(i, kk[u]);
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      kmin = min(kmin, __shfl_xor_sync(0xFFFFFFFFu, kmin, off));
      kmax = max(kmax, __shfl_xor_sync(0xFFFFFFFFu, kmax, off));
      above += __shfl_xor_sync(0xFFFFFFFFu, above, off);
    }
    if (lane == 0) {
      sh.red_u[0][warp] = kmin;
      sh.red_u[1][warp] = kmax;
      sh.red_u[2][warp] = above;
    }
    __syncthreads();
    const uint32_t ln = sh.loc_n;
    if (tid < P) {
      uint32_t a = 0xFFFFFFFFu, b = 0u, ab = 0u;
      for (int w = 0; w < kWarps; ++w) {
        a = min(a, sh.red_u[0][w]);
        b = max(b, sh.red_u[1][w]);
        ab += sh.red_u[2][w];
      }
      st_cluster_u32(remote(&sh.part_kmin[r], tid), a);
      st_cluster_u32(remote(&sh.part_kmax[r], tid), b);
      st_cluster_u32(remote(&sh.part_above[r], tid), ab);
      if (direct) sh.push_base[tid] = atom_add_cluster_u32(remote(&sh.cand_n, tid), ln);  // slots in CTA tid
    }
    __syncthreads();
    if (direct) {
      for (int e = tid; e < static_cast<int>(ln) * P; e += kThreads) {
        const int q = e / static_cast<int>(ln), j = e - q * static_cast<int>(ln);
        const uint32_t slot = sh.push_base[q] + j;
        st_cluster_u32(remote(&sh.cand_key[slot], q), sh.loc_key[j]);
        st_cluster_u32(remote(&sh.cand_pos[slot], q), static_cast<uint32_t>(sh.loc_pos[j]));
      }
    }
    row_sync();  // after this, no CTA reads or writes another's shared memory
                         // unless the bin is refined below
  }

  // ---- 4. the threshold key T and, per part, the output offsets
  uint32_t thr;
  uint32_t g_base = 0, e_base = 0;  // elements > T and == T in the parts before this one
  if (direct) {
    // rank of each candidate: larger key first, then lower position
    if (tid < static_cast<int>(c)) {
      const uint32_t key = sh.cand_key[tid];
      const int pos = sh.cand_pos[tid];
      int rank = 0;
      for (int j = 0; j < static_cast<int>(c); ++j) {
        const uint32_t kj = sh.cand_key[j];
        rank += (kj > key) || (kj == key && sh.cand_pos[j] < pos);
      }
      if (rank == need - 1) sh.thr = key;
    }
    __syncthreads();
    thr = sh.thr;
    const bool mine = tid < static_cast<int>(c);
    need -= __syncthreads_count(mine && sh.cand_key[tid] > thr);
    for (int q = 0; q < r; ++q) g_base += sh.part_above[q];
    g_base += __syncthreads_count(mine && sh.cand_pos[tid] < s0 && sh.cand_key[tid] > thr);
    e_base = __syncthreads_count(mine && sh.cand_pos[tid] < s0 && sh.cand_key[tid] == thr);
  } else {
    // refine over the bin's key interval [klo, khi] until it holds one key
    uint32_t klo = 0xFFFFFFFFu, khi = 0u;
    for (int q = 0; q < P; ++q) {
      klo = min(klo, sh.part_kmin[q]);
      khi = max(khi, sh.part_kmax[q]);
    }
    while (klo < khi) {  // the same trip count in every CTA of the row
      const uint64_t R = static_cast<uint64_t>(khi - klo) + 1;
      for (int b = tid; b < kBins; b += kThreads) sh.hist[b] = 0u;
      __syncthreads();
      for (int i = tid; i < m; i += kThreads) {
        const uint32_t key = key_at(i);
        if (key >= klo && key <= khi)
          atomicAdd(&sh.hist[static_cast<int>((static_cast<uint64_t>(key - klo) * kBins) / R)], 1u);
      }
      reduce_hist();
      find_bin(sh, static_cast<uint32_t>(need));
      const uint64_t b = sh.bsel;
      need -= static_cast<int>(sh.above);
      const uint32_t nlo = klo + static_cast<uint32_t>((b * R + kBins - 1) / kBins);
      const uint32_t nhi = klo + static_cast<uint32_t>(((b + 1) * R + kBins - 1) / kBins) - 1u;
      klo = nlo;
      khi = nhi;
    }
    thr = klo;
  }

  // ---- 5. ordered compaction: warp w takes a contiguous run of the part,
  // 32 consecutive keys at a time; ballots give the order within a step
  // (with candidate lists: warp w takes its list, which holds every selected
  // key of its run in position order)
  const int c0 = fast ? 0 : w0, c1 = fast ? n_lst : w1;
  auto pos_at = [&](int c) -> int { return fast ? static_cast<int>(lst[c]) : c; };
  uint32_t cg = 0, ce = 0;
  for (int base = c0; base < c1; base += 32) {
    const int c = base + lane;
    const uint32_t key = c < c1 ? key_at(pos_at(c)) : 0u;
    cg += __popc(__ballot_sync(0xFFFFFFFFu, c < c1 && key > thr));
    ce += __popc(__ballot_sync(0xFFFFFFFFu, c < c1 && key == thr));
  }
  uint64_t tot;
  const uint64_t wpre = block_exclusive_scan(lane == 0 ? (static_cast<uint64_t>(cg) | (static_cast<uint64_t>(ce) << 32)) : 0ull,
                                             tot, sh);
  const uint64_t wbefore = __shfl_sync(0xFFFFFFFFu, wpre, 0);
  if (!direct) {  // the parts' counts give the offsets
    if (tid < P) {
      st_cluster_u32(remote(&sh.part_gt[r], tid), static_cast<uint32_t>(tot));
      st_cluster_u32(remote(&sh.part_eq[r], tid), static_cast<uint32_t>(tot >> 32));
    }
    row_sync();  // no shared-memory access between the CTAs after this
    for (int q = 0; q < r; ++q) {
      g_base += sh.part_gt[q];
      e_base += sh.part_eq[q];
    }
  }
  uint32_t g = g_base + static_cast<uint32_t>(wbefore), e = e_base + static_cast<uint32_t>(wbefore >> 32);
  const uint32_t nq = static_cast<uint32_t>(need);
  for (int base = c0; base < c1; base += 32) {
    const int c = base + lane;
    const int i = c < c1 ? pos_at(c) : 0;
    const uint32_t key = c < c1 ? key_at(i) : 0u;
    const bool gt = c < c1 && key > thr, eq = c < c1 && key == thr;
    const uint32_t bg = __ballot_sync(0xFFFFFFFFu, gt), be = __ballot_sync(0xFFFFFFFFu, eq);
    const uint32_t gi = g + __popc(bg & lt), ei = e + __popc(be & lt);
    if (gt) emit<MODE>(p, t, static_cast<int>(gi + min(ei, nq)), s0 + i, key_value(key));
    if (eq && ei < nq) emit<MODE>(p, t, static_cast<int>(gi + ei), s0 + i, key_value(key));
    g += __popc(bg);
    e += __popc(be);
  }
}

// One CTA per row, the row in registers (rows of up to 32 * VPT * 32 keys).
// Warp w owns the contiguous run [w * 32 * VPT, (w + 1) * 32 * VPT), lane l
// its keys at w * 32 * VPT + 32 u + l, so loads are coalesced and the ordered
// compaction needs only ballots within a warp and one scan over the warps.
// The bins span the row's exact finite range; the steps are those of
// topk_kernel with P = 1.
template <int VPT, int MODE>
__global__ void __launch_bounds__(kThreads) topk_row_kernel(const TopkParams p) {
  __shared__ TopkShared sh;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t = blockIdx.x;
  const int k = p.k;
  // the row's valid length comes from the step's inputs, which the logits
  // producer does not write: it is found while that kernel may still run
  const int n = row_length<MODE>(p, valid_length(p.seq_lens, p.qsl, p.B, t, 0x7FFFFFFF, sh));
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const float* row = p.logits + static_cast<int64_t>(t) * p.ld;
  if (n <= k) {
    for (int i = tid; i < k; i += kThreads) {
      if (i < n) emit<MODE>(p, t, i, i, MODE == kWindow ? __ldg(row + i) : 0.f);
      else emit_empty<MODE>(p, t, i);
    }
    return;
  }
  const int ld = static_cast<int>(p.ld);
  const int base = warp * 32 * VPT + lane;  // position of key[0]; key[u] sits at base + 32 u
  uint32_t key[VPT];
#pragma unroll
  for (int u = 0; u < VPT; ++u) key[u] = base + 32 * u < ld ? order_key(__ldg(row + base + 32 * u)) : 0u;
  auto valid = [&](int u) { return base + 32 * u < n; };

  // ---- exact finite range of the row; histogram over 2048 bins linear in it
  float lo = INFINITY, hi = -INFINITY;
#pragma unroll
  for (int u = 0; u < VPT; ++u) {
    const float v = key_value(key[u]);
    if (valid(u) && isfinite(v)) {
      lo = fminf(lo, v);
      hi = fmaxf(hi, v);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    lo = fminf(lo, __shfl_xor_sync(0xFFFFFFFFu, lo, off));
    hi = fmaxf(hi, __shfl_xor_sync(0xFFFFFFFFu, hi, off));
  }
  if (lane == 0) {
    sh.red_f[0][warp] = lo;
    sh.red_f[1][warp] = hi;
  }
  for (int b = tid; b < kBins; b += kThreads) sh.ghist[b] = 0u;
  if (tid == 0) sh.cand_n = 0u;
  __syncthreads();
  block_range(lo, hi, sh);
  float inv_w = hi > lo ? static_cast<float>(kBins) / (hi - lo) : 0.f;
  if (!isfinite(inv_w)) inv_w = 0.f;
  if (!(lo <= hi)) lo = 0.f;
#pragma unroll
  for (int u = 0; u < VPT; ++u)
    if (valid(u)) atomicAdd(&sh.ghist[lin_bin(key_value(key[u]), lo, inv_w)], 1u);
  __syncthreads();
  find_bin(sh, static_cast<uint32_t>(k));
  const int bsel = static_cast<int>(sh.bsel);
  const uint32_t c = sh.ghist[bsel];
  const bool direct = c <= static_cast<uint32_t>(kCandCap);
  int need = k - static_cast<int>(sh.above);

  // ---- the threshold key within the bin
  uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
#pragma unroll
  for (int u = 0; u < VPT; ++u) {
    if (!valid(u) || lin_bin(key_value(key[u]), lo, inv_w) != bsel) continue;
    kmin = min(kmin, key[u]);
    kmax = max(kmax, key[u]);
    if (direct) {
      const uint32_t slot = atomicAdd(&sh.cand_n, 1u);
      sh.cand_key[slot] = key[u];
      sh.cand_pos[slot] = base + 32 * u;
    }
  }
  uint32_t thr;
  if (direct) {
    __syncthreads();
    if (tid < static_cast<int>(c)) {
      const uint32_t kk = sh.cand_key[tid];
      const int pos = sh.cand_pos[tid];
      int rank = 0, above_kk = 0;
      for (int j = 0; j < static_cast<int>(c); ++j) {
        const uint32_t kj = sh.cand_key[j];
        above_kk += kj > kk;
        rank += (kj > kk) || (kj == kk && sh.cand_pos[j] < pos);
      }
      if (rank == need - 1) {  // exactly one element has this rank
        sh.thr = kk;
        sh.thr_gt = static_cast<uint32_t>(above_kk);
      }
    }
    __syncthreads();
    thr = sh.thr;
    need -= static_cast<int>(sh.thr_gt);
  } else {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      kmin = min(kmin, __shfl_xor_sync(0xFFFFFFFFu, kmin, off));
      kmax = max(kmax, __shfl_xor_sync(0xFFFFFFFFu, kmax, off));
    }
    if (lane == 0) {
      sh.red_u[0][warp] = kmin;
      sh.red_u[1][warp] = kmax;
    }
    __syncthreads();
    uint32_t klo = 0xFFFFFFFFu, khi = 0u;
    for (int w = 0; w < kWarps; ++w) {
      klo = min(klo, sh.red_u[0][w]);
      khi = max(khi, sh.red_u[1][w]);
    }
    // refine over the bin's key interval until it holds one key
    while (klo < khi) {
      const uint64_t R = static_cast<uint64_t>(khi - klo) + 1;
      __syncthreads();  // every thread has read the previous level's histogram
      for (int b = tid; b < kBins; b += kThreads) sh.ghist[b] = 0u;
      __syncthreads();
#pragma unroll
      for (int u = 0; u < VPT; ++u)
        if (valid(u) && key[u] >= klo && key[u] <= khi)
          atomicAdd(&sh.ghist[static_cast<int>((static_cast<uint64_t>(key[u] - klo) * kBins) / R)], 1u);
      __syncthreads();
      find_bin(sh, static_cast<uint32_t>(need));
      const uint64_t b = sh.bsel;
      need -= static_cast<int>(sh.above);
      const uint32_t nlo = klo + static_cast<uint32_t>((b * R + kBins - 1) / kBins);
      const uint32_t nhi = klo + static_cast<uint32_t>(((b + 1) * R + kBins - 1) / kBins) - 1u;
      klo = nlo;
      khi = nhi;
    }
    thr = klo;
  }

  // ---- ordered compaction: warp counts by ballots, one scan over the warps
  uint32_t cg = 0, ce = 0;
#pragma unroll
  for (int u = 0; u < VPT; ++u) {
    cg += __popc(__ballot_sync(0xFFFFFFFFu, valid(u) && key[u] > thr));
    ce += __popc(__ballot_sync(0xFFFFFFFFu, valid(u) && key[u] == thr));
  }
  uint64_t tot;
  const uint64_t wpre = block_exclusive_scan(lane == 0 ? (static_cast<uint64_t>(cg) | (static_cast<uint64_t>(ce) << 32)) : 0ull,
                                             tot, sh);
  const uint64_t wbefore = __shfl_sync(0xFFFFFFFFu, wpre, 0);
  uint32_t g = static_cast<uint32_t>(wbefore), e = static_cast<uint32_t>(wbefore >> 32);
  const uint32_t nq = static_cast<uint32_t>(need);
  const uint32_t lt = (1u << lane) - 1u;
#pragma unroll
  for (int u = 0; u < VPT; ++u) {
    const bool gt = valid(u) && key[u] > thr, eq = valid(u) && key[u] == thr;
    const uint32_t bg = __ballot_sync(0xFFFFFFFFu, gt), be = __ballot_sync(0xFFFFFFFFu, eq);
    const uint32_t gi = g + __popc(bg & lt), ei = e + __popc(be & lt);
    if (gt) emit<MODE>(p, t, static_cast<int>(gi + min(ei, nq)), base + 32 * u, key_value(key[u]));
    if (eq && ei < nq) emit<MODE>(p, t, static_cast<int>(gi + ei), base + 32 * u, key_value(key[u]));
    g += __popc(bg);
    e += __popc(be);
  }
}

FuncAttrOnce g_smem[3], g_smem_u[3];  // per output mode

// CTAs per row: more only for long rows (at least 8192 keys per CTA) while
// they fill the GPU once (at most 8), and enough that a part fits the
// shared-memory stage where possible. A cluster barrier costs about as much
// as a short row's whole selection, so short rows keep one CTA.
int parts_for(int32_t T, int64_t ld) {
  int P = 1;
  while (P < kMaxParts && static_cast<int64_t>(T) * P * 2 <= num_sms() && (ld + 2 * P - 1) / (2 * P) >= 8192) P *= 2;
  while (P < kMaxParts && (ld + P - 1) / P > kSegCap) P *= 2;
  return P;
}

// Launches the top-k of rows 0..T-1 described by p in output mode MODE.
template <int MODE>
dsa_status_t topk_launch_mode(TopkParams p, int32_t T, cudaStream_t stream) {
  dsa_status_t st;
  const int64_t ld = p.ld;
  p.parts = parts_for(T, ld);
  if (p.parts == 1 && ld <= 32 * 32 * 32) {  // one CTA per row, the row in registers
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(T));
    cfg.blockDim = dim3(kThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = ld <= 32 * 8 * 32 ? cudaLaunchKernelEx(&cfg, topk_row_kernel<8, MODE>, p)
                                            : cudaLaunchKernelEx(&cfg, topk_row_kernel<32, MODE>, p);
    if (e != cudaSuccess) return fail(DSA_ERR_CUDA, "topk_row_kernel launch failed: %s", cudaGetErrorString(e));
    return DSA_OK;
  }
  const int64_t seg = (ld + p.parts - 1) / p.parts;
  const bool cached = seg <= kSegCap;
  // the part's keys, then one candidate list per warp (16-bit positions)
  constexpr int kListBytes = kWarps * kListCap * 2;
  const int smem = cached ? static_cast<int>(((seg + 7) & ~7) * 4) + kListBytes : 0;
  st = cached ? allow_smem(topk_kernel<true, MODE>, kSegCap * 4 + kListBytes, g_smem[MODE])
              : allow_smem(topk_kernel<false, MODE>, 0, g_smem_u[MODE]);
  if (st != DSA_OK) return st;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(static_cast<int64_t>(T) * p.parts));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.parts;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = cached ? cudaLaunchKernelEx(&cfg, topk_kernel<true, MODE>, p)
                         : cudaLaunchKernelEx(&cfg, topk_kernel<false, MODE>, p);
  if (e != cudaSuccess) return fail(DSA_ERR_CUDA, "topk_kernel launch failed: %s", cudaGetErrorString(e));
  return DSA_OK;
}

dsa_status_t topk_launch(const TopkParams& p, int32_t T, cudaStream_t stream) {
  switch (p.mode) {
    case kWindow: return topk_launch_mode<kWindow>(p, T, stream);
    case kFinal: return topk_launch_mode<kFinal>(p, T, stream);
    default: return topk_launch_mode<kPositions>(p, T, stream);
  }
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" size_t dsa_topk_workspace_size(int32_t T, int64_t ld, int32_t index_topk) {
  (void)T;
  (void)ld;
  (void)index_topk;
  return 0;  // the CTAs of a row combine their counts in distributed shared memory
}

extern "C" dsa_status_t dsa_topk(const float* logits, int64_t ld, const int32_t* seq_lens,
                                 const int32_t* query_start_loc, int32_t B, int32_t T, int32_t index_topk,
                                 int32_t* topk_idx, void* workspace, size_t ws_bytes, dsa_stream_t stream) {
  (void)workspace;
  (void)ws_bytes;
  if (B < 0 || T < 0 || ld <= 0 || index_topk <= 0)
    return fail(DSA_ERR_INVALID_ARG, "dsa_topk: bad sizes B=%d T=%d ld=%lld k=%d", B, T, (long long)ld, index_topk);
  if (T == 0) return DSA_OK;
  if (B == 0) return fail(DSA_ERR_INVALID_ARG, "dsa_topk: T > 0 with B == 0");
  if (!logits || !seq_lens || !query_start_loc || !topk_idx) return fail(DSA_ERR_INVALID_ARG, "dsa_topk: null pointer");
  if (index_topk > 65535) return fail(DSA_ERR_UNSUPPORTED, "dsa_topk: index_topk %d > 65535", index_topk);
  if (ld > 0x7FFFFFFF) return fail(DSA_ERR_UNSUPPORTED, "dsa_topk: ld %lld does not fit int32 positions", (long long)ld);
  if (static_cast<int64_t>(T) * kMaxParts > 0x7FFFFFFF) return fail(DSA_ERR_UNSUPPORTED, "dsa_topk: T too large");
  dsa_status_t st = check_device();
  if (st != DSA_OK) return st;
  TopkParams p = {};
  p.logits = logits;
  p.ld = ld;
  p.seq_lens = seq_lens;
  p.qsl = query_start_loc;
  p.B = B;
  p.k = index_topk;
  p.out = topk_idx;
  p.mode = kPositions;
  return topk_launch(p, T, reinterpret_cast<cudaStream_t>(stream));
}


// ---------------------------------------------------------------------------
// a1 + a2 over key windows (vLLM PR #38476 review thread: the decode logits
// buffer is [batch, max_seq_len] fp32; windowing the keys, a top-k per window
// giving (score, global id) candidates and one final top-k over the
// concatenated candidates bound it, and recover the global top-k exactly,
// since any key of the global top-k is in its window's top-k).
namespace dsa {
namespace {

struct WindowPlan {
  int64_t W, n_win, kcand, stride;  // window, windows, candidates per window, candidate row stride
  size_t logits_bytes, cand_bytes, total;
};

WindowPlan window_plan(int32_t T, int64_t max_seq_len, int32_t window, int32_t index_topk) {
  WindowPlan w = {};
  w.W = window > 0 ? window : (max_seq_len + 127) / 128 * 128;
  w.n_win = (max_seq_len + w.W - 1) / w.W;
  w.kcand = std::min<int64_t>(index_topk, w.W);
  w.stride = (w.n_win * w.kcand + 3) / 4 * 4;
  auto up = [](size_t b) { return (b + 255) / 256 * 256; };
  w.logits_bytes = up(static_cast<size_t>(T) * w.W * 4);
  w.cand_bytes = up(static_cast<size_t>(T) * w.stride * 4);
  w.total = w.logits_bytes + (w.n_win > 1 ? 2 * w.cand_bytes : 0);
  return w;
}

}  // namespace
}  // namespace dsa

extern "C" size_t dsa_indexer_topk_workspace_size(int32_t T, int64_t max_seq_len, int32_t window,
                                                  int32_t index_topk) {
  if (T <= 0 || max_seq_len <= 0 || index_topk <= 0 || window < 0) return 0;
  return window_plan(T, max_seq_len, window, index_topk).total;
}

extern "C" dsa_status_t dsa_indexer_topk(const void* q_idx, int64_t q_stride_t, const float* w,
                                         const uint8_t* k_cache, int64_t k_block_stride_bytes, int32_t num_blocks,
                                         const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens,
                                         const int32_t* query_start_loc, int32_t B, int32_t T, int32_t Hi, int32_t Di,
                                         int32_t block_size, int32_t max_q_len, int64_t max_seq_len, int32_t window,
                                         int32_t index_topk, int32_t* topk_idx, void* workspace, size_t ws_bytes,
                                         int32_t* dev_status, dsa_stream_t stream) {
  const IndexerCall c = {q_idx, q_stride_t, w, k_cache, k_block_stride_bytes, num_blocks, block_table, bt_stride,
                         seq_lens, query_start_loc, B, T, Hi, Di, block_size, max_q_len, dev_status};
  dsa_status_t st = indexer_validate(c, "dsa_indexer_topk");
  if (st != DSA_OK) return st;
  if (max_seq_len <= 0 || index_topk <= 0 || window < 0)
    return fail(DSA_ERR_INVALID_ARG, "dsa_indexer_topk: max_seq_len, index_topk must be positive and window >= 0");
  if (B == 0 || T == 0) return DSA_OK;
  if (!topk_idx) return fail(DSA_ERR_INVALID_ARG, "dsa_indexer_topk: null pointer");
  if (window % 128 || window % block_size)
    return fail(DSA_ERR_INVALID_ARG, "dsa_indexer_topk: window %d must be a multiple of 128 and of block_size", window);
  if (index_topk > 65535) return fail(DSA_ERR_UNSUPPORTED, "dsa_indexer_topk: index_topk %d > 65535", index_topk);
  const WindowPlan pl = window_plan(T, max_seq_len, window, index_topk);
  if (pl.n_win * pl.W > 0x7FFFFFFF || pl.stride > 0x7FFFFFFF)
    return fail(DSA_ERR_UNSUPPORTED, "dsa_indexer_topk: positions beyond int32");
  if (workspace == nullptr || ws_bytes < pl.total || !aligned16(workspace))
    return fail(DSA_ERR_WORKSPACE, "dsa_indexer_topk: %zu workspace bytes needed (16-byte aligned), got %zu", pl.total,
                ws_bytes);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  float* logits = static_cast<float*>(workspace);
  const int64_t key_cap = pl.n_win * pl.W;
  TopkParams p = {};
  p.seq_lens = seq_lens;
  p.qsl = query_start_loc;
  p.B = B;
  p.k = index_topk;
  p.out = topk_idx;
  if (pl.n_win == 1) {  // one window: the plain logits + top-k on the workspace row
    st = indexer_launch(c, logits, pl.W, 0, key_cap, s);
    if (st != DSA_OK) return st;
    p.logits = logits;
    p.ld = pl.W;
    p.mode = kPositions;
    return topk_launch(p, T, s);
  }
  float* cand_val = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + pl.logits_bytes);
  int32_t* cand_idx = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + pl.logits_bytes + pl.cand_bytes);
  p.win = static_cast<int32_t>(pl.W);
  p.kcand = static_cast<int32_t>(pl.kcand);
  p.cand_stride = static_cast<int32_t>(pl.stride);
  p.cand_val = cand_val;
  p.cand_idx = cand_idx;
  for (int64_t wi = 0; wi < pl.n_win; ++wi) {
    // the window's logits reuse one buffer: the logits kernel is not a
    // programmatic dependent, so it starts after the previous window's top-k
    st = indexer_launch(c, logits, pl.W, wi * pl.W, key_cap, s);
    if (st != DSA_OK) return st;
    p.logits = logits;
    p.ld = pl.W;
    p.mode = kWindow;
    p.key_begin = wi * pl.W;
    st = topk_launch(p, T, s);
    if (st != DSA_OK) return st;
  }
  p.logits = cand_val;
  p.ld = pl.stride;
  p.mode = kFinal;
  p.key_begin = 0;
  return topk_launch(p, T, s);
}
