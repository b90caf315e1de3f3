// a0 + a1: per-(token, head) e4m3 quantisation of the indexer query and the
// lightning-indexer logits over the paged fp8 key cache.
//
//   logits[t, s] = sk[s] * sum_h (w[t,h] * sq[t,h]) * ReLU( sum_d q8[t,h,d] * k8[s,d] )
//
// which equals sum_h w * ReLU(dequant(q) . dequant(k)) because both scales are
// positive (vLLM PR #38476, Changes 2: fp8 MQA logits with the K scale applied
// to the fp32 dot output; review thread: per_token_group_quant_fp8 of the
// indexer q). Keys outside the causal range get -inf and every entry of a
// row up to ld is written (the PR's clean_logits contract).
//
// tcgen05 e4m3 MMAs per 128-key tile: A = the key tile (M = 128 keys,
// K = head_dim bytes, 128-byte swizzled), B = the quantised queries of up to
// four tokens of one request (N = 64 heads x tokens, or one MMA per token
// pair with four tokens of 64 heads). Each TMEM lane then holds one key, so
// the ReLU-weighted head sum is an in-thread loop over columns; two
// accumulators let one epilogue warp group sum one unit while the other
// unit's MMA runs. Key tiles come through the block table into a ring of
// shared-memory stages (TMA page loads for 128-dim keys, 16-byte cp.async
// otherwise); two CTAs share an SM so one CTA's epilogue overlaps the other's
// loads and MMAs.
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "ptx.cuh"

namespace dsa {
namespace {

using namespace ptx;

constexpr int kThreads = 320;       // 8 epilogue warps, 1 load warp, 1 MMA warp
constexpr int kEpiThreads = 256;
constexpr int kProdWarp = 8, kMmaWarp = 9;
constexpr int kQuantThreads = 128;
constexpr int kTileKeys = 128;
constexpr int kMaxStages = 6;
constexpr int kTileBytes = kTileKeys * 128;  // rows padded to 128 bytes in shared memory
constexpr int kMaxTokensPerCta = 4;
constexpr int kMaxTilesPerCta = 64;
constexpr int kMaxBlocksPerCta = kMaxTilesPerCta * kTileKeys / 64 + 2;  // block_size >= 64

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// x / s correctly rounded, given y = RN(1/s): q = RN(x y) is within one ulp
// of x / s, the remainder x - s q is exact in one FMA, and RN(q + (x - s q) y)
// is the correctly rounded quotient (P. Markstein, "Computation of elementary
// functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1),
// 1990). A zero x is returned as x * y so that -0 keeps its sign.
__device__ __forceinline__ float div_by_recip(float x, float s, float y) {
  const float q = x * y;
  if (q == 0.f) return q;
  return fmaf(fmaf(-q, s, x), y, q);
}

// a0 for 16 consecutive dims of one (token, head) row. The row is spread
// over an aligned group of 8 lanes (lane % 8 = 16-dim chunk, chunks past the
// head dim hold zeros); the row amax is reduced with shuffles.
// scale = amax/448 (1 if amax == 0); code = e4m3_rn_satfinite(x / scale), the
// division correctly rounded (by div_by_recip, or IEEE division when 1/scale
// is not a normal number).
__device__ __forceinline__ uint4 quant_chunk16(uint4 a, uint4 b, float& scale) {
  const uint32_t u[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(u[i])), fabsf(bf16_hi(u[i]))));
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
  amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 4));
  scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  const float y = __frcp_rn(scale);
  uint32_t out[4];
  if (y < 0x1p126f) {  // 1/scale normal (scale is positive): the reciprocal path is exact
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint16_t p0 = cvt_e4m3x2(div_by_recip(bf16_lo(u[2 * i]), scale, y), div_by_recip(bf16_hi(u[2 * i]), scale, y));
      const uint16_t p1 =
          cvt_e4m3x2(div_by_recip(bf16_lo(u[2 * i + 1]), scale, y), div_by_recip(bf16_hi(u[2 * i + 1]), scale, y));
      out[i] = static_cast<uint32_t>(p0) | (static_cast<uint32_t>(p1) << 16);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint16_t p0 = cvt_e4m3x2(__fdiv_rn(bf16_lo(u[2 * i]), scale), __fdiv_rn(bf16_hi(u[2 * i]), scale));
      const uint16_t p1 = cvt_e4m3x2(__fdiv_rn(bf16_lo(u[2 * i + 1]), scale), __fdiv_rn(bf16_hi(u[2 * i + 1]), scale));
      out[i] = static_cast<uint32_t>(p0) | (static_cast<uint32_t>(p1) << 16);
    }
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

// One thread per 16-dim chunk; 8 consecutive threads per (token, head) row.
__global__ void __launch_bounds__(kQuantThreads) quant_q_kernel(const uint16_t* q, int64_t q_stride_t, int T, int Hi,
                                                           int Di, uint8_t* q8, float* sq) {
  const int64_t g = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t row = g / 8;
  const int c = static_cast<int>(g % 8);
  const bool row_ok = row < static_cast<int64_t>(T) * Hi;
  const bool have = row_ok && c < Di / 16;
  uint4 a = make_uint4(0, 0, 0, 0), b = a;
  if (have) {
    const int64_t t = row / Hi, h = row % Hi;
    const uint4* src = reinterpret_cast<const uint4*>(q + t * q_stride_t + h * Di) + 2 * c;
    a = __ldg(src);
    b = __ldg(src + 1);
  }
  float scale;
  const uint4 codes = quant_chunk16(a, b, scale);
  if (have) reinterpret_cast<uint4*>(q8 + row * Di)[c] = codes;
  if (row_ok && c == 0) sq[row] = scale;
}

struct IndexerParams {
  const uint16_t* q;  // bf16 bits [T, Hi, Di]
  int64_t q_stride_t;
  const float* w;  // [T, Hi]
  const uint8_t* k_cache;
  int64_t k_block_stride;
  int32_t num_blocks;
  const int32_t* block_table;
  int32_t bt_stride;
  const int32_t* seq_lens;
  const int32_t* qsl;
  int32_t B, Hi, Di, block_size;
  int32_t tb;      // tokens per CTA
  int32_t n_tb;    // token blocks per request (upper bound)
  int32_t hi_pad;  // heads rounded up to 16: columns per token
  int32_t tiles_per_cta;
  int32_t n_tiles;  // ceil(ld / 128)
  int32_t stages;
  float* logits;
  int64_t ld;
  int64_t key_begin;  // key of logits column 0 (a window of the keys; a multiple of 128 and of block_size)
  int64_t key_cap;    // requests are clipped to keys below this (ld for the whole-row call)
  int32_t* dev_status;
  int32_t lpt;  // hand out the (row, chunk) pairs longest work first (rows <= kThreads)
};

struct SmemOffsets {
  int k, sc, q, w, total;
};
__host__ __device__ inline SmemOffsets indexer_smem(int n_cols, int stages) {
  SmemOffsets o;
  o.k = 0;
  o.sc = o.k + stages * kTileBytes;
  o.q = (o.sc + stages * kTileKeys * 4 + 1023) & ~1023;
  o.w = o.q + n_cols * 128;
  o.total = o.w + n_cols * 4 + 1024;  // + slack for 1024-byte alignment of the base
  return o;
}
// two CTAs per SM: stages sized so that 2 x smem stays within 228 KB
__host__ __device__ inline int indexer_stages(int n_cols) { return n_cols <= 64 ? 6 : (n_cols <= 128 ? 5 : 4); }
// three or four tokens of 64 heads: one MMA per token pair (see the kernel)
__host__ __device__ inline bool indexer_pair_split(int hi_pad, int tb) { return hi_pad == 64 && tb > 2; }
// query rows staged as the MMA's B operand: every pair's rows, so that with
// an odd token count the last pair's MMA reads zero rows, not past the region
__host__ __device__ inline int indexer_q_rows(int hi_pad, int tb) {
  return indexer_pair_split(hi_pad, tb) ? 2 * ((tb + 1) / 2) * hi_pad : hi_pad * tb;
}

// Warp roles: warps 0-7 quantise the queries, then run the epilogue (warps w
// and w + 4 read TMEM lanes 32(w%4)..+31 = keys of the tile); warp 8 loads key
// tiles (TMA for 128-byte rows from lanes 0 and 1, cp.async otherwise); warp 9
// issues the MMAs.
template <int DI>
__global__ void __launch_bounds__(kThreads, 2) indexer_logits_kernel(const __grid_constant__ IndexerParams p,
                                                                     const __grid_constant__ CUtensorMap kmap) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full_bar[kMaxStages], empty_bar[kMaxStages], acc_full[2], acc_empty[2], q_ready;
  __shared__ uint32_t tmem_holder;
  __shared__ int s_tok[kMaxTokensPerCta];
  __shared__ int s_valid[kMaxTokensPerCta];
  __shared__ int s_blk[kMaxBlocksPerCta];
  __shared__ volatile int s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // the top-k kernel may be scheduled now; it waits for this grid's results
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // the CTA's row (request b, token block tblk) and chunk of tiles
  int b, tblk, chunk;
  if (p.lpt) {
    // Longest work first: the grid's (row, chunk) pairs, in the order the
    // block scheduler starts CTAs, are every row's full chunks, then each
    // row's partial last chunk, then the chunks past its last key (which only
    // write -inf), so that with requests of different lengths the long rows'
    // chunks start early and the last CTAs to start are short ones. The order
    // only permutes the pairs; each CTA derives its bounds below as before.
    // Thread i < rows counts row i's chunks (rows * gridDim.x < 2^21).
    __shared__ uint64_t s_wsum[kThreads / 32];
    __shared__ int s_row, s_chunk;
    const int R = p.B * p.n_tb, nx = static_cast<int>(gridDim.x), tpc = p.tiles_per_cta;
    int full = 0, part = 0, empty = 0;
    if (tid < R) {
      const int bi = tid / p.n_tb, ti = tid - bi * p.n_tb;
      const int q0i = __ldg(p.qsl + bi), q1i = __ldg(p.qsl + bi + 1), tok0i = q0i + ti * p.tb;
      int tiles = 0;
      if (tok0i < q1i) {
        const int last = min(tok0i + p.tb, q1i) - 1;  // the block's last token
        const int64_t vmax = static_cast<int64_t>(__ldg(p.seq_lens + bi)) - (q1i - q0i) + (last - q0i) + 1;
        const int64_t v = min(vmax, p.key_cap) - p.key_begin;
        tiles = static_cast<int>(max(static_cast<int64_t>(0), min((v + kTileKeys - 1) / kTileKeys,
                                                                  static_cast<int64_t>(p.n_tiles))));
      }
      full = min(tiles / tpc, nx);
      part = (full < nx && tiles % tpc != 0) ? 1 : 0;
      empty = nx - full - part;
    }
    constexpr uint64_t kM = (1u << 21) - 1;
    const uint64_t v = static_cast<uint64_t>(full) | (static_cast<uint64_t>(part) << 21) |
                       (static_cast<uint64_t>(empty) << 42);
    uint64_t x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint64_t y = __shfl_up_sync(0xFFFFFFFFu, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) s_wsum[warp] = x;
    __syncthreads();
    uint64_t before = 0, total = 0;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) {
      const uint64_t ws = s_wsum[w];
      if (w < warp) before += ws;
      total += ws;
    }
    const uint64_t ex = before + x - v;
    const int fi = static_cast<int>(ex & kM), pi = static_cast<int>((ex >> 21) & kM), ei = static_cast<int>(ex >> 42);
    const int F = static_cast<int>(total & kM), P = static_cast<int>((total >> 21) & kM);
    const int L = static_cast<int>(blockIdx.y) * nx + static_cast<int>(blockIdx.x);
    if (tid < R) {
      int c = -1;
      if (L < F) {
        if (L >= fi && L < fi + full) c = L - fi;
      } else if (L < F + P) {
        if (part && L - F == pi) c = full;
      } else if (L - F - P >= ei && L - F - P < ei + empty) {
        c = full + part + (L - F - P - ei);
      }
      if (c >= 0) {
        s_row = tid;
        s_chunk = c;
      }
    }
    __syncthreads();
    b = s_row / p.n_tb;
    tblk = s_row - b * p.n_tb;
    chunk = s_chunk;
  } else {
    b = blockIdx.y / p.n_tb;
    tblk = blockIdx.y % p.n_tb;
    chunk = blockIdx.x;
  }
  // tiles are counted in logits columns; tile i holds keys key_begin + 128 i ..
  const int t_begin = chunk * p.tiles_per_cta;
  const int t_end = min(t_begin + p.tiles_per_cta, p.n_tiles);
  const int kb = static_cast<int>(p.key_begin);
  // block ids of every key the CTA's tiles can address (warps 8 and 9), read
  // before the request's length is known; entries past it are never used
  // because every use first checks the key against seq_len
  const int* bt_row = p.block_table + static_cast<int64_t>(b) * p.bt_stride;
  const int blk0 = (kb + t_begin * kTileKeys) / p.block_size;
  const int n_blk = max(0, min((kb + t_end * kTileKeys + p.block_size - 1) / p.block_size, p.bt_stride) - blk0);
  constexpr int kBlkPerThread = (kMaxBlocksPerCta + 63) / 64;
  int blk_v[kBlkPerThread];
  if (warp >= 8) {
#pragma unroll
    for (int u = 0; u < kBlkPerThread; ++u) {
      const int i = tid - kEpiThreads + 64 * u;
      blk_v[u] = i < n_blk ? __ldg(bt_row + blk0 + i) : -1;
    }
  }
  const int q0 = __ldg(p.qsl + b), q1 = __ldg(p.qsl + b + 1);
  const int tok0 = q0 + tblk * p.tb;
  if (tok0 >= q1) return;  // this request has fewer token blocks (uniform exit)
  const int ntok = min(p.tb, q1 - tok0);
  const int q_len = q1 - q0;
  int seq_len = __ldg(p.seq_lens + b);
  // clip the request to what the logits row and the block table can address
  const int64_t cap = min(p.key_cap, static_cast<int64_t>(p.bt_stride) * p.block_size);
  if (seq_len < q_len || seq_len > cap) {
    if (tid == 0 && chunk == 0) report(p.dev_status, DSA_DEVERR_SEQ_LEN);
    seq_len = max(q_len, static_cast<int>(min(static_cast<int64_t>(seq_len), cap)));
  }
  const int max_valid = min(static_cast<int64_t>(seq_len - q_len + (tok0 + ntok - 1 - q0) + 1), cap);

  const int t_comp_end = min(t_end, (max_valid - kb + kTileKeys - 1) / kTileKeys);  // tiles needing an MMA
  const int n_comp = max(0, t_comp_end - t_begin);
  const int n_cols = indexer_q_rows(p.hi_pad, p.tb);  // staged query rows (the MMA N without pairs)
  const int S = p.stages;
  // MMA units: a unit is one MMA of a key tile against unit_cols query
  // columns into one of nbuf accumulators. When all the CTA's columns fit
  // twice in its 256 TMEM columns, a unit is the whole tile (nbuf = 2). With
  // three or four tokens of 64 heads they fit once, so a unit is one pair of
  // tokens: the key tile stays for both pairs and one pair's epilogue overlaps
  // the next pair's MMA, which a single 256-column accumulator would serialise.
  const bool pair_split = indexer_pair_split(p.hi_pad, p.tb);
  const int n_units = pair_split ? (ntok + 1) / 2 : 1;  // MMA units per key tile
  const int unit_cols = pair_split ? 2 * p.hi_pad : n_cols;
  const int nbuf = 2 * unit_cols <= 256 ? 2 : 1;
  // one token and two accumulators: the two epilogue warp groups take
  // alternate tiles, each the whole head sum of its keys, so the latency of
  // one tile's epilogue overlaps the next tile's
  // with two accumulators the two epilogue warp groups take alternate units
  // (each warp every token of its unit), so one group's head sums run while
  // the other group's accumulator is refilled; with one accumulator both
  // groups take alternate tokens of every tile
  const bool alt_units = nbuf == 2;
  // epilogue warps that read one tile's scales (two groups when a tile has two units)
  const int epi_warps = alt_units ? 4 * n_units : 8;
  const int acc_release = alt_units ? 4 : 8;  // warps that release one accumulator

  const SmemOffsets so = indexer_smem(n_cols, S);
  uint8_t* sk = smem + so.k;
  float* ssc = reinterpret_cast<float*>(smem + so.sc);
  uint8_t* sq = smem + so.q;
  float* sw = reinterpret_cast<float*>(smem + so.w);

  if (tid < ntok) {
    s_tok[tid] = tok0 + tid;
    s_valid[tid] = min(static_cast<int64_t>(seq_len - q_len + (tok0 + tid - q0) + 1), cap);
  }
  if (tid == 0) s_abort = 0;

  uint32_t tmem = 0;
  const uint32_t acc_cols = unit_cols <= 32 ? 32 : (unit_cols <= 64 ? 64 : (unit_cols <= 128 ? 128 : 256));
  const uint32_t tmem_cols = acc_cols * nbuf;
  auto abort_now = [&](void) {
    s_abort = 1;
    report(p.dev_status, DSA_DEVERR_TIMEOUT);
  };
  auto block_id_ok = [&](int blk) { return blk >= 0 && blk < p.num_blocks; };
  auto block_ok = [&](int s) {  // key s < seq_len lies in a valid block
    return block_id_ok(s_blk[s / p.block_size - blk0]);
  };
  // keys that later token blocks of the request read again stay in L2
  const bool keep_keys = p.n_tb > 1;
  // tile i: two TMA loads of 64 keys x 128 B (one page each) plus their
  // scales, completing on full_bar[st]; keys past seq_len are neither loaded
  // nor counted. Issued by lanes 0 and 1 of the producer warp together, lane u
  // the half of keys 64u.. (one instruction issues both halves' copies), for
  // tiles in order: each lane's block and offset in it advance with the tile
  // (block_size is a multiple of 64) instead of being divided out per tile.
  int iss_blk = 0, iss_off = 0;
  {
    const int s0 = kb + t_begin * kTileKeys + 64 * (lane & 1);
    iss_blk = s0 / p.block_size - blk0;
    iss_off = s0 - (iss_blk + blk0) * p.block_size;
  }
  auto issue_keys = [&](int i, int st) {
    const int s0 = kb + (t_begin + i) * kTileKeys + 64 * lane;
    int blk = -1;
    bool bad = false;
    if (s0 < seq_len) {
      const int b = s_blk[iss_blk];
      if (block_id_ok(b)) blk = b;
      else bad = true;
    }
    const uint32_t halves = __ballot_sync(0x3u, blk >= 0);
    if (lane == 0) mbar_arrive_expect_tx(&full_bar[st], __popc(halves) * (64 * 128 + 64 * 4));
    __syncwarp(0x3u);
    if (blk >= 0) {
      if (keep_keys)
        tma_load_3d_hint(smem_u32(sk + st * kTileBytes + lane * 8192), &kmap, &full_bar[st], 0, iss_off, blk,
                         l2_policy_evict_last());
      else
        tma_load_3d(smem_u32(sk + st * kTileBytes + lane * 8192), &kmap, &full_bar[st], 0, iss_off, blk);
      bulk_copy_g2s(smem_u32(ssc + st * kTileKeys + lane * 64),
                    p.k_cache + static_cast<int64_t>(blk) * p.k_block_stride +
                        static_cast<int64_t>(p.block_size) * 128 + iss_off * 4,
                    256, &full_bar[st]);
    }
    if (bad) report(p.dev_status, DSA_DEVERR_BLOCK_OOB);
    for (iss_off += kTileKeys; iss_off >= p.block_size; iss_off -= p.block_size) ++iss_blk;
  };
  // tiles whose loads the producer issues before the CTA barrier (TMA path):
  // one, so that its latency overlaps the prologue; issuing every stage this
  // early delays the query loads the first MMA also waits for
  const int n_early = DI == 128 ? min(1, n_comp) : 0;

  // ---- prologue, before one CTA barrier: warps 0-7 load and quantise the
  // queries (a0) into the B operand; warp 8 stores the block ids, initialises
  // the barriers and issues the first key tile; warp 9 allocates TMEM.
  if (n_comp > 0) {
    if constexpr (DI < 128) {  // row padding past Di is never written by the loads
      for (int i = tid; i < S * kTileBytes / 16; i += kThreads) reinterpret_cast<uint4*>(sk)[i] = make_uint4(0, 0, 0, 0);
    }
    if (warp < 8) {
      // a0 takes 32 (token, head) rows per pass, 8 lanes per row; the loads of
      // kQPass passes are in flight together
      constexpr int kQPass = 2;
      for (int base0 = 0; base0 < n_cols; base0 += kQPass * 32) {
        uint4 qa[kQPass], qb[kQPass];
        float qw[kQPass];
#pragma unroll
        for (int u = 0; u < kQPass; ++u) {
          const int n = base0 + u * 32 + tid / 8, c = tid % 8;
          const int j = n / p.hi_pad, h = n % p.hi_pad;
          qa[u] = make_uint4(0, 0, 0, 0);
          qb[u] = qa[u];
          qw[u] = 0.f;
          if (n < n_cols && j < ntok && h < p.Hi) {
            if (c < DI / 16) {
              const uint4* src =
                  reinterpret_cast<const uint4*>(p.q + (tok0 + j) * p.q_stride_t + static_cast<int64_t>(h) * DI) + 2 * c;
              qa[u] = __ldg(src);
              qb[u] = __ldg(src + 1);
            }
            if (c == 0) qw[u] = __ldg(p.w + static_cast<int64_t>(tok0 + j) * p.Hi + h);
          }
        }
#pragma unroll
        for (int u = 0; u < kQPass; ++u) {
          const int n = base0 + u * 32 + tid / 8, c = tid % 8;
          if (n >= n_cols) break;  // uniform within a warp (n_cols is a multiple of 16)
          float scale;
          const uint4 codes = quant_chunk16(qa[u], qb[u], scale);
          *reinterpret_cast<uint4*>(sq + sw128_offset(n, c)) = codes;
          if (c == 0) sw[n] = qw[u] * scale;  // zero for padded rows
        }
      }
      fence_proxy_async_smem();  // the MMA reads the codes through the async proxy
    } else {
#pragma unroll
      for (int u = 0; u < kBlkPerThread; ++u) {
        const int i = tid - kEpiThreads + 64 * u;
        if (i < n_blk) s_blk[i] = blk_v[u];
      }
      __syncwarp();
      if (warp == kProdWarp && lane == 0) {
        for (int s = 0; s < S; ++s) {
          mbar_init(&full_bar[s], DI == 128 ? 1 : 32);
          mbar_init(&empty_bar[s], 1 + epi_warps);
        }
        for (int s = 0; s < 2; ++s) {
          mbar_init(&acc_full[s], 1);
          mbar_init(&acc_empty[s], acc_release);
        }
        mbar_init(&q_ready, 8);
        fence_mbar_init();
      }
      // the tiles' block ids were stored by this warp (its first 32 entries
      // cover the first 16 tiles: block_size >= 64), the barriers initialised
      // by its lane 0
      if constexpr (DI == 128) {
        __syncwarp();
        if (warp == kProdWarp && lane < 2)
          for (int i = 0; i < n_early; ++i) issue_keys(i, i);
      }
      if (warp == kMmaWarp) {
        tmem_alloc(&tmem_holder, tmem_cols);
        tmem_relinquish();
      }
    }
    if (DI < 128) fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (n_comp > 0) tmem = tmem_holder;
  if (n_comp > 0 && warp < 8) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&q_ready);
  }


  if (n_comp > 0 && warp == kProdWarp) {
    // ---------------- producer (the first tile went out before the CTA barrier)
    // stage of tile i and how many times the ring has wrapped before it
    int st = n_early, wraps = 0;
    for (int i = n_early; i < n_comp && !s_abort; ++i) {
      if (i >= S && !mbar_wait(&empty_bar[st], (wraps - 1) & 1)) {
        if (lane == 0) abort_now();
        break;
      }
      const int key0 = kb + (t_begin + i) * kTileKeys;
      if constexpr (DI == 128) {
        if (lane < 2) issue_keys(i, st);
      } else {
        constexpr int kChunks = DI / 16;
        uint8_t* dst_base = sk + st * kTileBytes;
        for (int c = lane; c < kTileKeys * kChunks; c += 32) {
          const int r = c / kChunks, ch = c % kChunks;
          const int s = key0 + r;
          const uint8_t* src = p.k_cache;
          uint32_t bytes = 0;
          if (s < seq_len && block_ok(s)) {
            src = p.k_cache + static_cast<int64_t>(s_blk[s / p.block_size - blk0]) * p.k_block_stride +
                  (s % p.block_size) * DI + ch * 16;
            bytes = 16;
          }
          cp_async_16(smem_u32(dst_base + sw128_offset(r, ch)), src, bytes);
        }
        {  // 4 consecutive keys per 16-byte scale chunk (block_size % 64 == 0)
          const int s = key0 + lane * 4;
          const uint8_t* src = p.k_cache;
          uint32_t bytes = 0;
          if (s < seq_len) {
            if (block_ok(s)) {
              src = p.k_cache + static_cast<int64_t>(s_blk[s / p.block_size - blk0]) * p.k_block_stride +
                    static_cast<int64_t>(p.block_size) * DI + (s % p.block_size) * 4;
              bytes = 16;
            } else {
              report(p.dev_status, DSA_DEVERR_BLOCK_OOB);
            }
          }
          cp_async_16(smem_u32(ssc + st * kTileKeys + lane * 4), src, bytes);
        }
        cp_async_mbar_arrive(&full_bar[st]);
      }
      if (++st == S) {
        st = 0;
        ++wraps;
      }
    }
  } else if (n_comp > 0 && warp == kMmaWarp) {
    // ---------------- MMA issuer
    const uint32_t idesc = idesc_e4m3(128, unit_cols);
    if (!mbar_wait(&q_ready, 0) && lane == 0) abort_now();
    int st = 0, wraps = 0;  // stage of tile i and how many times the ring has wrapped before it
    for (int i = 0; i < n_comp && !s_abort; ++i) {
      bool ok = mbar_wait(&full_bar[st], wraps & 1);
      for (int pp = 0; ok && pp < n_units; ++pp) {
        const int u = i * n_units + pp;
        const int buf = nbuf == 2 ? u & 1 : 0, use = nbuf == 2 ? u >> 1 : u;  // accumulator, its use count
        if (u >= nbuf) ok = mbar_wait(&acc_empty[buf], (use - 1) & 1);
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          // unit pp takes the query rows pp * unit_cols.. (whole 1024-byte swizzle atoms)
          const uint32_t a0 = smem_u32(sk + st * kTileBytes), b0 = smem_u32(sq + pp * unit_cols * 128);
#pragma unroll
          for (int ks = 0; ks < DI / 32; ++ks)
            mma_e4m3_ss(tmem + buf * acc_cols, smem_desc(a0 + ks * 32, 16, 1024, kSwizzle128B),
                        smem_desc(b0 + ks * 32, 16, 1024, kSwizzle128B), idesc, ks > 0 ? 1u : 0u);
          if (pp == n_units - 1) mma_commit(&empty_bar[st]);  // the tile's last MMA has read the stage
          mma_commit(&acc_full[buf]);
        }
        __syncwarp();
      }
      if (!ok) {
        if (lane == 0) abort_now();
        break;
      }
      if (++st == S) {
        st = 0;
        ++wraps;
      }
    }
  } else if (n_comp > 0) {
    // ---------------- epilogue: thread = key row = TMEM lane. Warps w and
    // w+4 (warp group g = w / 4) share the lanes 32(w%4)..: with two
    // accumulators they take alternate units, with one alternate tokens.
    const int g = warp >> 2;
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    // sum over heads [h0, h1) of token j (h1 - h0 a multiple of 16): four
    // independent chains, head h on chain h % 4; chains 0, 1 and chains 2, 3
    // advance together by one packed FMA each (each lane rounded once, as an
    // fmaf of its own). ReLU(x) is taken as (x + |x|) / 2 on the FMA pipe:
    // for finite x, x + |x| is exactly 2x or +0, so every chain holds exactly
    // twice the sum of w * ReLU(x) (scaling by 2 commutes with rounding) and
    // one halving at the end gives the same bits as max(x, 0) would; a NaN
    // score (a NaN key code) stays NaN, as in the definition
    auto head_sum = [&](uint32_t col, int j, int h0, int h1) -> float {  // token j's heads from TMEM column col
      float2 a01 = make_float2(0.f, 0.f), a23 = make_float2(0.f, 0.f);
      const float4* w4 = reinterpret_cast<const float4*>(sw + j * p.hi_pad);
      auto step4 = [&](const float4 w, uint32_t v0, uint32_t v1, uint32_t v2, uint32_t v3) {
        const float x0 = __uint_as_float(v0), x1 = __uint_as_float(v1), x2 = __uint_as_float(v2),
                    x3 = __uint_as_float(v3);
        a01 = __ffma2_rn(make_float2(w.x, w.y), make_float2(x0 + fabsf(x0), x1 + fabsf(x1)), a01);
        a23 = __ffma2_rn(make_float2(w.z, w.w), make_float2(x2 + fabsf(x2), x3 + fabsf(x3)), a23);
      };
      // 16 columns per tensor-memory load: measured faster than 32 (fewer
      // registers held across the wait) and than 8 at every shape
      for (int hc = h0; hc < h1; hc += 16) {
        uint32_t v[16];
        tmem_ld16_sync(lane_addr + col + hc, v);
#pragma unroll
        for (int x = 0; x < 4; ++x) step4(w4[hc / 4 + x], v[4 * x], v[4 * x + 1], v[4 * x + 2], v[4 * x + 3]);
      }
      return 0.5f * ((a01.x + a01.y) + (a23.x + a23.y));
    };
    // two accumulators: group g takes the units u = g, g + 2, .. (with two
    // token pairs per tile, pair g of every tile; otherwise alternate tiles),
    // always in accumulator g, every token of the unit; the accumulator goes
    // back to the MMA before the unit's last logits are stored. The tokens of
    // a group's units are the same in every tile, so their logits rows and
    // causal limits are read once.
    if (alt_units) {
      const int di = n_units == 2 ? 1 : 2;  // tiles from one unit of the group to its next
      const int j0 = n_units == 2 ? 2 * g : 0;
      const int j_end = pair_split ? min(j0 + 2, ntok) : ntok;
      float* row0 = p.logits + static_cast<int64_t>(s_tok[j0]) * p.ld;
      float* row1 = p.logits + static_cast<int64_t>(s_tok[min(j0 + 1, ntok - 1)]) * p.ld;
      const int valid0 = s_valid[j0], valid1 = s_valid[min(j0 + 1, ntok - 1)];
      const uint32_t acc_col = g * acc_cols;
      int i = n_units == 2 ? 0 : g;
      int st = i % S;
      // the block of this warp's 32 keys (one block: block_size is a multiple
      // of 64), advanced with the tile instead of divided out per tile
      const int key_w = kb + (t_begin + i) * kTileKeys + (warp & 3) * 32;
      int blk_rel = key_w / p.block_size - blk0;
      int blk_off = key_w - (blk_rel + blk0) * p.block_size;
      for (int k = 0; i < n_comp && !s_abort; ++k) {
        if (!mbar_wait(&acc_full[g], k & 1)) {
          if (lane == 0) abort_now();
          break;
        }
        tc_fence_after();
        const int col = (t_begin + i) * kTileKeys + r;  // logits column of this lane's key
        const int s = kb + col;
        const float scale_k = ssc[st * kTileKeys + r];
        const bool bad = s < seq_len && !block_id_ok(s_blk[blk_rel]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[st]);  // this warp is done with the stage's scales
        if (pair_split) {  // 64 heads: constant trip counts
          const bool two = j0 + 1 < j_end;
          const float acc0 = head_sum(acc_col, j0, 0, 64);
          const float acc1 = two ? head_sum(acc_col + 64, j0 + 1, 0, 64) : 0.f;
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&acc_empty[g]);
          if (col < p.ld) {
            __stcs(row0 + col, (s < valid0 && !bad) ? acc0 * scale_k : -INFINITY);
            if (two) __stcs(row1 + col, (s < valid1 && !bad) ? acc1 * scale_k : -INFINITY);
          }
        } else {
          for (int j = 0; j < ntok; ++j) {
            const float acc = head_sum(acc_col + j * p.hi_pad, j, 0, p.hi_pad);
            if (j + 1 == ntok) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&acc_empty[g]);
            }
            if (col < p.ld)
              __stcs(p.logits + static_cast<int64_t>(s_tok[j]) * p.ld + col,
                     (s < s_valid[j] && !bad) ? acc * scale_k : -INFINITY);
          }
        }
        i += di;
        st += di;
        if (st >= S) st -= S;
        for (blk_off += di * kTileKeys; blk_off >= p.block_size; blk_off -= p.block_size) ++blk_rel;
      }
    }
    // one accumulator (more than 128 columns of fewer than 64 heads): both
    // groups read every tile, warp w the tokens g, g + 2, ..
    for (int i = 0; !alt_units && i < n_comp && !s_abort; ++i) {
      const int st = i % S;
      if (!mbar_wait(&acc_full[0], i & 1)) {
        if (lane == 0) abort_now();
        break;
      }
      tc_fence_after();
      const int col = (t_begin + i) * kTileKeys + r;  // logits column of this lane's key
      const int s = kb + col;
      const float scale_k = ssc[st * kTileKeys + r];
      const bool bad = s < seq_len && !block_ok(s);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty_bar[st]);  // this warp is done with the stage's scales
      for (int j = g; j < ntok; j += 2) {
        const float acc = head_sum(j * p.hi_pad, j, 0, p.hi_pad);
        if (col < p.ld)
          __stcs(p.logits + static_cast<int64_t>(s_tok[j]) * p.ld + col,
                 (s < s_valid[j] && !bad) ? acc * scale_k : -INFINITY);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[0]);
    }
  }

  // tiles entirely past every token's valid range: -inf only
  if (warp < 4) {
    for (int tile = t_begin + n_comp; tile < t_end; ++tile) {
      const int col = tile * kTileKeys + tid;
      if (col < p.ld)
        for (int j = 0; j < ntok; ++j) __stcs(p.logits + static_cast<int64_t>(s_tok[j]) * p.ld + col, -INFINITY);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (n_comp > 0 && warp == kMmaWarp) tmem_dealloc(tmem, tmem_cols);
}

FuncAttrOnce g_smem_set[3];

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" dsa_status_t dsa_quant_q(const void* q_idx, int64_t q_stride_t, int32_t T, int32_t Hi, int32_t Di,
                                    uint8_t* q8, float* sq, dsa_stream_t stream) {
  if (T < 0 || Hi <= 0 || Di <= 0) return fail(DSA_ERR_INVALID_ARG, "dsa_quant_q: bad sizes T=%d Hi=%d Di=%d", T, Hi, Di);
  if (Di != 32 && Di != 64 && Di != 128) return fail(DSA_ERR_UNSUPPORTED, "dsa_quant_q: Di must be 32, 64 or 128");
  if (T == 0) return DSA_OK;
  if (!q_idx || !q8 || !sq) return fail(DSA_ERR_INVALID_ARG, "dsa_quant_q: null pointer");
  if (!aligned16(q_idx) || !aligned16(q8) || q_stride_t < static_cast<int64_t>(Hi) * Di || q_stride_t % 8)
    return fail(DSA_ERR_INVALID_ARG, "dsa_quant_q: q must be 16-byte aligned with a token stride >= Hi*Di, multiple of 8");
  dsa_status_t st = check_device();
  if (st != DSA_OK) return st;
  const int rows = T * Hi;
  quant_q_kernel<<<(rows * 8 + kQuantThreads - 1) / kQuantThreads, kQuantThreads, 0,
                   reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint16_t*>(q_idx), q_stride_t, T, Hi, Di, q8, sq);
  return check_launch("quant_q_kernel");
}

namespace dsa {

dsa_status_t indexer_validate(const IndexerCall& c, const char* name) {
  if (c.B < 0 || c.T < 0 || c.Hi <= 0 || c.Di <= 0 || c.block_size <= 0 || c.max_q_len < 0 || c.num_blocks < 0 ||
      c.bt_stride < 0)
    return fail(DSA_ERR_INVALID_ARG, "%s: negative or zero size argument", name);
  if (c.B == 0 || c.T == 0) return DSA_OK;
  if (!c.q_idx || !c.w || !c.k_cache || !c.block_table || !c.seq_lens || !c.query_start_loc)
    return fail(DSA_ERR_INVALID_ARG, "%s: null pointer", name);
  if (c.max_q_len < 1) return fail(DSA_ERR_INVALID_ARG, "%s: max_q_len must be >= 1 when T > 0", name);
  if (c.Hi > 64) return fail(DSA_ERR_UNSUPPORTED, "%s: Hi=%d > 64", name, c.Hi);
  if (c.Di != 32 && c.Di != 64 && c.Di != 128) return fail(DSA_ERR_UNSUPPORTED, "%s: Di=%d not in {32,64,128}", name, c.Di);
  if (c.block_size % 64) return fail(DSA_ERR_UNSUPPORTED, "%s: block_size %d not a multiple of 64", name, c.block_size);
  if (c.k_block_stride_bytes < static_cast<int64_t>(c.block_size) * (c.Di + 4) || c.k_block_stride_bytes % 16)
    return fail(DSA_ERR_INVALID_ARG, "%s: k_block_stride_bytes %lld must be >= block_size*(Di+4) and a multiple of 16",
                name, static_cast<long long>(c.k_block_stride_bytes));
  if (!aligned16(c.q_idx) || !aligned16(c.k_cache) || c.q_stride_t < static_cast<int64_t>(c.Hi) * c.Di ||
      c.q_stride_t % 8)
    return fail(DSA_ERR_INVALID_ARG,
                "%s: q_idx/k_cache must be 16-byte aligned, q token stride >= Hi*Di and a multiple of 8", name);
  if (!aligned4(c.w)) return fail(DSA_ERR_INVALID_ARG, "%s: misaligned w", name);
  return check_device();
}

dsa_status_t indexer_launch(const IndexerCall& c, float* logits, int64_t ld, int64_t key_begin, int64_t key_cap,
                            cudaStream_t s) {
  IndexerParams p;
  p.q = static_cast<const uint16_t*>(c.q_idx);
  p.q_stride_t = c.q_stride_t;
  p.w = c.w;
  p.k_cache = c.k_cache;
  p.k_block_stride = c.k_block_stride_bytes;
  p.num_blocks = c.num_blocks;
  p.block_table = c.block_table;
  p.bt_stride = c.bt_stride;
  p.seq_lens = c.seq_lens;
  p.qsl = c.query_start_loc;
  p.B = c.B;
  p.Hi = c.Hi;
  p.Di = c.Di;
  p.block_size = c.block_size;
  p.hi_pad = (c.Hi + 15) / 16 * 16;
  p.tb = std::min(std::min(c.max_q_len, kMaxTokensPerCta), 256 / p.hi_pad);
  p.n_tb = (c.max_q_len + p.tb - 1) / p.tb;
  p.n_tiles = static_cast<int32_t>((ld + kTileKeys - 1) / kTileKeys);
  p.logits = logits;
  p.ld = ld;
  p.key_begin = key_begin;
  p.key_cap = key_cap;
  p.dev_status = c.dev_status;
  const int64_t rows = static_cast<int64_t>(c.B) * p.n_tb;
  if (rows > 65535) return fail(DSA_ERR_UNSUPPORTED, "indexer: B * token blocks = %lld > 65535", (long long)rows);
  if (key_begin + ld > 0x7FFFFFFF) return fail(DSA_ERR_UNSUPPORTED, "indexer: key positions beyond int32");
  const int64_t slots = 2LL * num_sms();
  const int64_t total_tiles = rows * p.n_tiles;
  // Several tokens per request and few rows (batches of short multi-token
  // steps, whose requests' lengths differ and are on the device only): chunks
  // of about 1 / 2.5 of an even share of the rows' key ranges, handed out
  // longest work first, so that chunks of the long requests start early and
  // the ones past the short requests' keys cost a launch each. Otherwise one
  // wave of two CTAs per SM when the work allows it, at least two tiles per
  // CTA (the ordering's extra round trip for every row's length costs a
  // decode batch more than it saves on even lengths: measured).
  const bool lpt = c.max_q_len >= 2 && rows <= kThreads;
  int64_t tpc;
  if (lpt) {
    tpc = std::max<int64_t>(4, (2 * total_tiles + 5 * slots - 1) / (5 * slots));
  } else {
    tpc = std::max<int64_t>(2, (total_tiles + slots - 1) / slots);
    while (tpc < kMaxTilesPerCta && rows * ((p.n_tiles + tpc - 1) / tpc) > slots) ++tpc;
  }
  p.tiles_per_cta = static_cast<int32_t>(std::min<int64_t>(tpc, kMaxTilesPerCta));
  const int64_t grid_x = (p.n_tiles + p.tiles_per_cta - 1) / p.tiles_per_cta;
  p.lpt = lpt && rows * grid_x < (int64_t{1} << 21) ? 1 : 0;
  const int n_cols = indexer_q_rows(p.hi_pad, p.tb);
  p.stages = indexer_stages(n_cols);
  const SmemOffsets so = indexer_smem(n_cols, p.stages);
  const int max_smem = std::max(indexer_smem(64, indexer_stages(64)).total,
                                std::max(indexer_smem(128, indexer_stages(128)).total, indexer_smem(256, indexer_stages(256)).total));
  CUtensorMap kmap;
  memset(&kmap, 0, sizeof(kmap));
  dsa_status_t st;
  if (c.Di == 128) {
    const uint64_t dims[3] = {128, static_cast<uint64_t>(c.block_size), static_cast<uint64_t>(std::max(c.num_blocks, 1))};
    const uint64_t strides[2] = {128, static_cast<uint64_t>(c.k_block_stride_bytes)};
    const uint32_t box[3] = {128, 64, 1};
    st = make_tmap(&kmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, c.k_cache, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    if (st != DSA_OK) return st;
  }
  dim3 grid((p.n_tiles + p.tiles_per_cta - 1) / p.tiles_per_cta, static_cast<unsigned>(rows));
  switch (c.Di) {
    case 128:
      st = allow_smem(indexer_logits_kernel<128>, max_smem, g_smem_set[0]);
      if (st != DSA_OK) return st;
      indexer_logits_kernel<128><<<grid, kThreads, so.total, s>>>(p, kmap);
      break;
    case 64:
      st = allow_smem(indexer_logits_kernel<64>, max_smem, g_smem_set[1]);
      if (st != DSA_OK) return st;
      indexer_logits_kernel<64><<<grid, kThreads, so.total, s>>>(p, kmap);
      break;
    default:
      st = allow_smem(indexer_logits_kernel<32>, max_smem, g_smem_set[2]);
      if (st != DSA_OK) return st;
      indexer_logits_kernel<32><<<grid, kThreads, so.total, s>>>(p, kmap);
      break;
  }
  return check_launch("indexer_logits_kernel");
}

}  // namespace dsa

extern "C" dsa_status_t dsa_indexer_logits(const void* q_idx, int64_t q_stride_t, const float* w,
                                           const uint8_t* k_cache, int64_t k_block_stride_bytes, int32_t num_blocks,
                                           const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens,
                                           const int32_t* query_start_loc, int32_t B, int32_t T, int32_t Hi,
                                           int32_t Di, int32_t block_size, int32_t max_q_len, float* logits,
                                           int64_t ld, int32_t* dev_status, dsa_stream_t stream) {
  const IndexerCall c = {q_idx, q_stride_t, w, k_cache, k_block_stride_bytes, num_blocks, block_table, bt_stride,
                         seq_lens, query_start_loc, B, T, Hi, Di, block_size, max_q_len, dev_status};
  if (ld <= 0) return fail(DSA_ERR_INVALID_ARG, "dsa_indexer_logits: ld must be positive");
  dsa_status_t st = indexer_validate(c, "dsa_indexer_logits");
  if (st != DSA_OK || B == 0 || T == 0) return st;
  if (!logits) return fail(DSA_ERR_INVALID_ARG, "dsa_indexer_logits: null pointer");
  if (!aligned4(logits)) return fail(DSA_ERR_INVALID_ARG, "dsa_indexer_logits: misaligned logits");
  return indexer_launch(c, logits, ld, 0, ld, reinterpret_cast<cudaStream_t>(stream));
}
