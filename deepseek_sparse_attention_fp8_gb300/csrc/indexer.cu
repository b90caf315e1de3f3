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
// One tcgen05 e4m3 MMA per 128-key tile: A = the key tile (M = 128 keys,
// K = head_dim bytes, 128-byte swizzled), B = the quantised queries of up to
// four tokens of one request (N = 64 heads x tokens). Each TMEM lane then holds
// one key, so the ReLU-weighted head sum is an in-thread loop over columns.
// Key tiles are gathered through the block table with 16-byte cp.async into a
// ring of shared-memory stages; two CTAs share an SM so one CTA's epilogue
// overlaps the other's loads and MMAs.
#include <cuda_bf16.h>

#include <algorithm>

#include "common.cuh"
#include "ptx.cuh"

namespace dsa {
namespace {

using namespace ptx;

constexpr int kThreads = 128;
constexpr int kTileKeys = 128;
constexpr int kStages = 4;
constexpr int kTileBytes = kTileKeys * 128;  // rows padded to 128 bytes in shared memory
constexpr int kMaxTokensPerCta = 4;

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
  float* logits;
  int64_t ld;
  int32_t* dev_status;
};

struct SmemOffsets {
  int k, sc, bad, q, w, total;
};
__host__ __device__ inline SmemOffsets indexer_smem(int n_cols) {
  SmemOffsets o;
  o.k = 0;
  o.sc = o.k + kStages * kTileBytes;
  o.bad = o.sc + kStages * kTileKeys * 4;
  o.q = (o.bad + kStages * 16 + 1023) & ~1023;
  o.w = o.q + n_cols * 128;
  o.total = o.w + n_cols * 4 + 1024;  // + slack for 1024-byte alignment of the base
  return o;
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Quantises one (token, head) row of Di bf16 values. Calls emit(chunk, uint4)
// for every 16-code chunk and returns the fp32 scale (amax/448, 1 if amax==0).
template <typename Emit>
__device__ __forceinline__ float quant_row(const uint16_t* src, int Di, Emit emit) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  float amax = 0.f;
  for (int c = 0; c < Di / 8; ++c) {
    uint4 v = __ldg(s4 + c);
    uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(u[i])), fabsf(bf16_hi(u[i]))));
  }
  const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  for (int c = 0; c < Di / 16; ++c) {
    uint4 a = __ldg(s4 + 2 * c), b = __ldg(s4 + 2 * c + 1);
    uint32_t u[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t out[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint16_t p0 = cvt_e4m3x2(__fdiv_rn(bf16_lo(u[2 * i]), scale), __fdiv_rn(bf16_hi(u[2 * i]), scale));
      uint16_t p1 = cvt_e4m3x2(__fdiv_rn(bf16_lo(u[2 * i + 1]), scale), __fdiv_rn(bf16_hi(u[2 * i + 1]), scale));
      out[i] = static_cast<uint32_t>(p0) | (static_cast<uint32_t>(p1) << 16);
    }
    emit(c, make_uint4(out[0], out[1], out[2], out[3]));
  }
  return scale;
}

__global__ void __launch_bounds__(kThreads) quant_q_kernel(const uint16_t* q, int64_t q_stride_t, int T, int Hi,
                                                           int Di, uint8_t* q8, float* sq) {
  const int row = blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= T * Hi) return;
  const int t = row / Hi, h = row % Hi;
  uint4* dst = reinterpret_cast<uint4*>(q8 + static_cast<int64_t>(row) * Di);
  sq[row] = quant_row(q + t * q_stride_t + static_cast<int64_t>(h) * Di, Di, [&](int c, uint4 v) { dst[c] = v; });
}

__global__ void __launch_bounds__(kThreads, 2) indexer_logits_kernel(const IndexerParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t mma_bar;
  __shared__ uint32_t tmem_holder;
  __shared__ int s_tok[kMaxTokensPerCta];
  __shared__ int s_valid[kMaxTokensPerCta];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int b = blockIdx.y / p.n_tb;
  const int tblk = blockIdx.y % p.n_tb;
  const int q0 = __ldg(p.qsl + b), q1 = __ldg(p.qsl + b + 1);
  const int tok0 = q0 + tblk * p.tb;
  if (tok0 >= q1) return;  // this request has fewer token blocks (uniform exit)
  const int ntok = min(p.tb, q1 - tok0);
  const int q_len = q1 - q0;
  int seq_len = __ldg(p.seq_lens + b);
  // clip the request to what the logits row and the block table can address
  const int64_t cap = min(p.ld, static_cast<int64_t>(p.bt_stride) * p.block_size);
  if (seq_len < q_len || seq_len > cap) {
    if (tid == 0 && blockIdx.x == 0) report(p.dev_status, DSA_DEVERR_SEQ_LEN);
    seq_len = max(q_len, static_cast<int>(min(static_cast<int64_t>(seq_len), cap)));
  }
  const int max_valid = min(static_cast<int64_t>(seq_len - q_len + (tok0 + ntok - 1 - q0) + 1), cap);

  const int t_begin = blockIdx.x * p.tiles_per_cta;
  const int t_end = min(t_begin + p.tiles_per_cta, p.n_tiles);
  const int t_comp_end = min(t_end, (max_valid + kTileKeys - 1) / kTileKeys);  // tiles needing an MMA
  const int n_comp = max(0, t_comp_end - t_begin);
  const int n_cols = p.hi_pad * p.tb;  // MMA N

  const SmemOffsets so = indexer_smem(n_cols);
  uint8_t* sk = smem + so.k;
  float* ssc = reinterpret_cast<float*>(smem + so.sc);
  uint32_t* sbad = reinterpret_cast<uint32_t*>(smem + so.bad);
  uint8_t* sq = smem + so.q;
  float* sw = reinterpret_cast<float*>(smem + so.w);

  if (tid < ntok) {
    s_tok[tid] = tok0 + tid;
    s_valid[tid] = min(static_cast<int64_t>(seq_len - q_len + (tok0 + tid - q0) + 1), cap);
  }

  uint32_t tmem = 0;
  const uint32_t tmem_cols = n_cols <= 32 ? 32 : (n_cols <= 64 ? 64 : (n_cols <= 128 ? 128 : 256));
  if (n_comp > 0) {
    // zero the key stages once: columns past Di are never written by the loads
    if (p.Di < 128) {
      for (int i = tid; i < kStages * kTileBytes / 16; i += kThreads)
        reinterpret_cast<uint4*>(sk)[i] = make_uint4(0, 0, 0, 0);
    }
    // a0: quantise the token block's queries into the B operand (N rows x 128 B)
    for (int n = tid; n < n_cols; n += kThreads) {
      const int j = n / p.hi_pad, h = n % p.hi_pad;
      uint8_t* row = sq;
      if (j < ntok && h < p.Hi) {
        const int tok = tok0 + j;
        const float scale = quant_row(p.q + tok * p.q_stride_t + static_cast<int64_t>(h) * p.Di, p.Di,
                                      [&](int c, uint4 v) {
                                        *reinterpret_cast<uint4*>(row + sw128_offset(n, c)) = v;
                                      });
        for (int c = p.Di / 16; c < 8; ++c) *reinterpret_cast<uint4*>(row + sw128_offset(n, c)) = make_uint4(0, 0, 0, 0);
        sw[n] = __ldg(p.w + static_cast<int64_t>(tok) * p.Hi + h) * scale;
      } else {
        for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(row + sw128_offset(n, c)) = make_uint4(0, 0, 0, 0);
        sw[n] = 0.f;
      }
    }
    fence_proxy_async_smem();
    if (warp == 0) {
      tmem_alloc(&tmem_holder, tmem_cols);
      tmem_relinquish();
    }
    if (tid == 0) {
      mbar_init(&mma_bar, 1);
      fence_mbar_init();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (n_comp > 0) tmem = tmem_holder;

  const int* bt_row = p.block_table + static_cast<int64_t>(b) * p.bt_stride;
  const int chunks_per_row = p.Di / 16;

  // Issues the cp.async loads of key tile `tile` into stage `st`.
  auto load_tile = [&](int tile, int st) {
    const int key0 = tile * kTileKeys;
    uint8_t* dst_base = sk + st * kTileBytes;
    const int total = kTileKeys * chunks_per_row;
    for (int c = tid; c < total; c += kThreads) {
      const int r = c / chunks_per_row, ch = c % chunks_per_row;
      const int s = key0 + r;
      const uint8_t* src = p.k_cache;
      uint32_t bytes = 0;
      if (s < seq_len) {
        const int blk = __ldg(bt_row + s / p.block_size);
        if (blk >= 0 && blk < p.num_blocks) {
          src = p.k_cache + static_cast<int64_t>(blk) * p.k_block_stride + (s % p.block_size) * p.Di + ch * 16;
          bytes = 16;
        }
      }
      cp_async_16(smem_u32(dst_base + sw128_offset(r, ch)), src, bytes);
    }
    // scales: 4 consecutive keys per 16-byte chunk (block_size % 64 == 0);
    // warp 0 loads them and records which keys sit in an out-of-range block
    if (warp == 0) {
      const int s = key0 + tid * 4;
      const uint8_t* src = p.k_cache;
      uint32_t bytes = 0;
      bool bad = false;
      if (s < seq_len) {
        const int blk = __ldg(bt_row + s / p.block_size);
        if (blk >= 0 && blk < p.num_blocks) {
          src = p.k_cache + static_cast<int64_t>(blk) * p.k_block_stride +
                static_cast<int64_t>(p.block_size) * p.Di + (s % p.block_size) * 4;
          bytes = 16;
        } else {
          bad = true;
        }
      }
      cp_async_16(smem_u32(ssc + st * kTileKeys + tid * 4), src, bytes);
      const uint32_t bal = __ballot_sync(0xFFFFFFFFu, bad);
      if (lane < 4) {  // word `lane` covers keys 32*lane .. +31 = lanes 8*lane .. +7
        uint32_t word = 0;
        for (int k = 0; k < 8; ++k)
          if ((bal >> (8 * lane + k)) & 1u) word |= 0xFu << (4 * k);
        sbad[st * 4 + lane] = word;
      }
      if (bad) report(p.dev_status, DSA_DEVERR_BLOCK_OOB);
    }
  };

  const uint32_t idesc = idesc_e4m3(128, n_cols);
  const int ksteps = p.Di / 32;
  bool aborted = false;

  // prologue: fill kStages-1 stages
  for (int i = 0; i < kStages - 1; ++i) {
    if (i < n_comp) load_tile(t_begin + i, i);
    cp_async_commit();
  }
  for (int i = 0; i < n_comp; ++i) {
    const int st = i % kStages;
    // the stage refilled below was read by the previous tile's epilogue
    if (i > 0) __syncthreads();
    if (i + kStages - 1 < n_comp) load_tile(t_begin + i + kStages - 1, (i + kStages - 1) % kStages);
    cp_async_commit();
    cp_async_wait<kStages - 1>();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) {
      const uint32_t a0 = smem_u32(sk + st * kTileBytes), b0 = smem_u32(sq);
      for (int ks = 0; ks < ksteps; ++ks)
        mma_e4m3_ss(tmem, smem_desc(a0 + ks * 32, 16, 1024, kSwizzle128B), smem_desc(b0 + ks * 32, 16, 1024, kSwizzle128B),
                    idesc, ks > 0 ? 1u : 0u);
      mma_commit(&mma_bar);
    }
    __syncwarp();
    const bool ok = mbar_wait(&mma_bar, i & 1);
    if (__syncthreads_or(!ok)) {
      aborted = true;
      break;
    }
    tc_fence_after();
    // epilogue: thread = key row = TMEM lane
    const int r = warp * 32 + lane;
    const int s = (t_begin + i) * kTileKeys + r;
    const float scale_k = ssc[st * kTileKeys + r];
    const bool bad = (sbad[st * 4 + (r >> 5)] >> (r & 31)) & 1u;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    for (int j = 0; j < ntok; ++j) {
      float acc = 0.f;
      for (int hc = 0; hc < p.hi_pad; hc += 32) {
        if (hc + 32 <= p.hi_pad) {
          uint32_t v[32];
          tmem_ld32_sync(lane_addr + j * p.hi_pad + hc, v);
#pragma unroll
          for (int x = 0; x < 32; ++x) acc = fmaf(sw[j * p.hi_pad + hc + x], fmaxf(__uint_as_float(v[x]), 0.f), acc);
        } else {
          uint32_t v[16];
          tmem_ld16_sync(lane_addr + j * p.hi_pad + hc, v);
#pragma unroll
          for (int x = 0; x < 16; ++x) acc = fmaf(sw[j * p.hi_pad + hc + x], fmaxf(__uint_as_float(v[x]), 0.f), acc);
        }
      }
      const float out = (s < s_valid[j] && !bad) ? acc * scale_k : -INFINITY;
      if (s < p.ld) p.logits[static_cast<int64_t>(s_tok[j]) * p.ld + s] = out;
    }
    tc_fence_before();
  }
  cp_async_wait<0>();
  if (aborted && tid == 0) report(p.dev_status, DSA_DEVERR_TIMEOUT);

  // tiles entirely past every token's valid range: -inf only
  for (int tile = t_begin + n_comp; tile < t_end; ++tile) {
    const int s = tile * kTileKeys + tid;
    if (s < p.ld)
      for (int j = 0; j < ntok; ++j) p.logits[static_cast<int64_t>(s_tok[j]) * p.ld + s] = -INFINITY;
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (n_comp > 0 && warp == 0) tmem_dealloc(tmem, tmem_cols);
}

bool g_smem_set = false;

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
  quant_q_kernel<<<(rows + kThreads - 1) / kThreads, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint16_t*>(q_idx), q_stride_t, T, Hi, Di, q8, sq);
  return check_launch("quant_q_kernel");
}

extern "C" dsa_status_t dsa_indexer_logits(const void* q_idx, int64_t q_stride_t, const float* w,
                                           const uint8_t* k_cache, int64_t k_block_stride_bytes, int32_t num_blocks,
                                           const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens,
                                           const int32_t* query_start_loc, int32_t B, int32_t T, int32_t Hi,
                                           int32_t Di, int32_t block_size, int32_t max_q_len, float* logits,
                                           int64_t ld, int32_t* dev_status, dsa_stream_t stream) {
  if (B < 0 || T < 0 || Hi <= 0 || Di <= 0 || block_size <= 0 || max_q_len < 0 || ld <= 0 || num_blocks < 0 ||
      bt_stride < 0)
    return fail(DSA_ERR_INVALID_ARG, "dsa_indexer_logits: negative or zero size argument");
  if (B == 0 || T == 0) return DSA_OK;
  if (!q_idx || !w || !k_cache || !block_table || !seq_lens || !query_start_loc || !logits)
    return fail(DSA_ERR_INVALID_ARG, "dsa_indexer_logits: null pointer");
  if (max_q_len < 1) return fail(DSA_ERR_INVALID_ARG, "dsa_indexer_logits: max_q_len must be >= 1 when T > 0");
  if (Hi > 64) return fail(DSA_ERR_UNSUPPORTED, "dsa_indexer_logits: Hi=%d > 64", Hi);
  if (Di != 32 && Di != 64 && Di != 128) return fail(DSA_ERR_UNSUPPORTED, "dsa_indexer_logits: Di=%d not in {32,64,128}", Di);
  if (block_size % 64) return fail(DSA_ERR_UNSUPPORTED, "dsa_indexer_logits: block_size %d not a multiple of 64", block_size);
  if (k_block_stride_bytes < static_cast<int64_t>(block_size) * (Di + 4) || k_block_stride_bytes % 16)
    return fail(DSA_ERR_INVALID_ARG, "dsa_indexer_logits: k_block_stride_bytes %lld must be >= block_size*(Di+4) and a multiple of 16",
                static_cast<long long>(k_block_stride_bytes));
  if (!aligned16(q_idx) || !aligned16(k_cache) || q_stride_t < static_cast<int64_t>(Hi) * Di || q_stride_t % 8)
    return fail(DSA_ERR_INVALID_ARG, "dsa_indexer_logits: q_idx/k_cache must be 16-byte aligned, q token stride >= Hi*Di and a multiple of 8");
  if (!aligned4(w) || !aligned4(logits)) return fail(DSA_ERR_INVALID_ARG, "dsa_indexer_logits: misaligned w/logits");
  dsa_status_t st = check_device();
  if (st != DSA_OK) return st;

  IndexerParams p;
  p.q = static_cast<const uint16_t*>(q_idx);
  p.q_stride_t = q_stride_t;
  p.w = w;
  p.k_cache = k_cache;
  p.k_block_stride = k_block_stride_bytes;
  p.num_blocks = num_blocks;
  p.block_table = block_table;
  p.bt_stride = bt_stride;
  p.seq_lens = seq_lens;
  p.qsl = query_start_loc;
  p.B = B;
  p.Hi = Hi;
  p.Di = Di;
  p.block_size = block_size;
  p.hi_pad = (Hi + 15) / 16 * 16;
  p.tb = std::min(std::min(max_q_len, kMaxTokensPerCta), 256 / p.hi_pad);
  p.n_tb = (max_q_len + p.tb - 1) / p.tb;
  p.n_tiles = static_cast<int32_t>((ld + kTileKeys - 1) / kTileKeys);
  p.logits = logits;
  p.ld = ld;
  p.dev_status = dev_status;
  const int64_t rows = static_cast<int64_t>(B) * p.n_tb;
  if (rows > 65535) return fail(DSA_ERR_UNSUPPORTED, "dsa_indexer_logits: B * token blocks = %lld > 65535", (long long)rows);
  // about four CTAs per SM in total, at least two tiles each
  const int64_t total_tiles = rows * p.n_tiles;
  const int64_t target = 4LL * num_sms();
  p.tiles_per_cta = static_cast<int32_t>(std::max<int64_t>(2, std::min<int64_t>(64, (total_tiles + target - 1) / target)));
  const int n_cols = p.hi_pad * p.tb;
  const SmemOffsets so = indexer_smem(n_cols);
  st = allow_smem(indexer_logits_kernel, indexer_smem(256).total, g_smem_set);  // the largest N any call uses
  if (st != DSA_OK) return st;
  dim3 grid((p.n_tiles + p.tiles_per_cta - 1) / p.tiles_per_cta, static_cast<unsigned>(rows));
  indexer_logits_kernel<<<grid, kThreads, so.total, reinterpret_cast<cudaStream_t>(stream)>>>(p);
  return check_launch("indexer_logits_kernel");
}
