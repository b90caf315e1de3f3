// Producer side of the indexer key cache: the new tokens' indexer keys are
// quantised to e4m3 with one fp32 scale per token and stored into the paged
// fp8 cache that the logits kernel reads ("vllm-dsa-mtp-sm80" README, "The
// skew fixes", item 0: indexer_k_quant_and_cache writes the 132-byte-per-token
// indexer page and, like every op on that cache, addresses blocks through the
// cache's block stride).
//
// Quantisation rule, the same as a0's for the query (vLLM PR #38476 review
// thread: per_token_group_quant_fp8 with one group per head_dim values):
//   scale = amax(|k[t,:]|) / 448 (1 when amax == 0), code = e4m3_rn_satfinite(k / scale),
// both divisions IEEE-rounded fp32.
//
// One warp per token: lane l holds Di/32 consecutive dims, the amax is reduced
// with shuffles, and the 32 lanes' codes are the token's Di-byte row, written
// as one coalesced store; lane 0 writes the scale.
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 256;  // 8 tokens per CTA

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

template <int DI>
__global__ void __launch_bounds__(kThreads) k_quant_cache_kernel(const uint16_t* k, int64_t k_stride_t, int T,
                                                                  uint8_t* k_cache, int64_t k_block_stride,
                                                                  int num_blocks, const int32_t* block_table,
                                                                  int bt_stride, const int32_t* seq_lens,
                                                                  const int32_t* qsl, int B, int block_size,
                                                                  int32_t* dev_status) {
  constexpr int E = DI / 32;  // dims per lane: 4, 2 or 1
  const int t = static_cast<int>((static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;  // uniform per warp

  // the token's Di values, E consecutive bf16 per lane
  float x[E];
  const uint16_t* src = k + static_cast<int64_t>(t) * k_stride_t + lane * E;
  if constexpr (E == 4) {
    const uint2 v = __ldg(reinterpret_cast<const uint2*>(src));
    x[0] = bf16_bits_to_f32(v.x & 0xFFFFu);
    x[1] = bf16_bits_to_f32(v.x >> 16);
    x[2] = bf16_bits_to_f32(v.y & 0xFFFFu);
    x[3] = bf16_bits_to_f32(v.y >> 16);
  } else if constexpr (E == 2) {
    const uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(src));
    x[0] = bf16_bits_to_f32(v & 0xFFFFu);
    x[1] = bf16_bits_to_f32(v >> 16);
  } else {
    x[0] = bf16_bits_to_f32(__ldg(src));
  }

  // request of token t: the last b with query_start_loc[b] <= t, counted by
  // the warp's lanes over strided entries (independent loads, one round)
  int cnt = 0;
#pragma unroll 4
  for (int j = lane; j < B; j += 32) cnt += __ldg(qsl + j) <= t ? 1 : 0;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) cnt += __shfl_xor_sync(0xFFFFFFFFu, cnt, off);
  const int b = max(0, cnt - 1);
  const int q0 = __ldg(qsl + b), q1 = __ldg(qsl + b + 1);
  const int64_t pos = static_cast<int64_t>(__ldg(seq_lens + b)) - (q1 - q0) + (t - q0);

  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
  const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;

  if (pos < 0 || pos >= static_cast<int64_t>(bt_stride) * block_size) {
    if (lane == 0) report(dev_status, DSA_DEVERR_SEQ_LEN);
    return;
  }
  const int blk = __ldg(block_table + static_cast<int64_t>(b) * bt_stride + pos / block_size);
  if (blk < 0 || blk >= num_blocks) {
    if (lane == 0) report(dev_status, DSA_DEVERR_BLOCK_OOB);
    return;
  }
  const int off = static_cast<int>(pos % block_size);
  uint8_t* page = k_cache + static_cast<int64_t>(blk) * k_block_stride;
  uint8_t* dst = page + static_cast<int64_t>(off) * DI + lane * E;
  if constexpr (E == 4) {
    const uint32_t lo16 = ptx::cvt_e4m3x2(__fdiv_rn(x[0], scale), __fdiv_rn(x[1], scale));
    const uint32_t hi16 = ptx::cvt_e4m3x2(__fdiv_rn(x[2], scale), __fdiv_rn(x[3], scale));
    *reinterpret_cast<uint32_t*>(dst) = lo16 | (hi16 << 16);
  } else if constexpr (E == 2) {
    *reinterpret_cast<uint16_t*>(dst) = ptx::cvt_e4m3x2(__fdiv_rn(x[0], scale), __fdiv_rn(x[1], scale));
  } else {
    // pair with the next lane's value so one conversion yields both bytes
    const float y = __fdiv_rn(x[0], scale);
    const float y_next = __shfl_down_sync(0xFFFFFFFFu, y, 1);
    const uint16_t two = ptx::cvt_e4m3x2(y, y_next);
    if ((lane & 1) == 0) *reinterpret_cast<uint16_t*>(dst) = two;
  }
  if (lane == 0) *reinterpret_cast<float*>(page + static_cast<int64_t>(block_size) * DI + off * 4) = scale;
}

// Producer side of the fp8 latent cache: the new tokens' latent rows
// (Dk = 576 bf16: 512 latent + 64 rope) are written as fp8 rows of 656
// bytes: 512 e4m3 codes in four groups of 128 dims, each group quantised with
// the rule above (scale = amax/448, 1 when amax == 0), then the four fp32
// scales, then the 64 rope values' bf16 bits unchanged. vLLM PR #38476
// (Limitations; review thread) names fp8 latent caches for SM90+/SM12x parts
// without printing a layout; this is the layout the attention kernels read.
// One warp per token: lane l quantises latent dims 16 l .. 16 l + 15 (eight
// lanes per group, amax by shuffles) and stores their 16 code bytes; lanes
// 0, 8, 16, 24 store the group scales and lanes 0-7 copy the rope bytes.
constexpr int kF8Dk = 576, kF8Dv = 512, kF8RowBytes = 656;

__global__ void __launch_bounds__(kThreads) mla_kv_fp8_cache_kernel(const uint16_t* kv, int64_t kv_stride_t, int T,
                                                                     uint8_t* cache, int64_t block_stride,
                                                                     int num_blocks, const int32_t* block_table,
                                                                     int bt_stride, const int32_t* seq_lens,
                                                                     const int32_t* qsl, int B, int block_size,
                                                                     int32_t* dev_status) {
  const int t = static_cast<int>((static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5);
  const int lane = threadIdx.x & 31;
  if (t >= T) return;  // uniform per warp
  const uint16_t* src = kv + static_cast<int64_t>(t) * kv_stride_t;
  const uint4 a = __ldg(reinterpret_cast<const uint4*>(src + 16 * lane));
  const uint4 c = __ldg(reinterpret_cast<const uint4*>(src + 16 * lane + 8));
  uint4 rope = make_uint4(0u, 0u, 0u, 0u);
  if (lane < 8) rope = __ldg(reinterpret_cast<const uint4*>(src + kF8Dv + 8 * lane));
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
  float x[16];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = bf16_bits_to_f32(w[i] & 0xFFFFu);
    x[2 * i + 1] = bf16_bits_to_f32(w[i] >> 16);
  }

  // request and position of token t (as for the indexer keys above)
  int cnt = 0;
#pragma unroll 4
  for (int j = lane; j < B; j += 32) cnt += __ldg(qsl + j) <= t ? 1 : 0;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) cnt += __shfl_xor_sync(0xFFFFFFFFu, cnt, off);
  const int b = max(0, cnt - 1);
  const int q0 = __ldg(qsl + b), q1 = __ldg(qsl + b + 1);
  const int64_t pos = static_cast<int64_t>(__ldg(seq_lens + b)) - (q1 - q0) + (t - q0);

  // the group's amax over its eight lanes
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < 16; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
  for (int off = 1; off < 8; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
  const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;

  if (pos < 0 || pos >= static_cast<int64_t>(bt_stride) * block_size) {
    if (lane == 0) report(dev_status, DSA_DEVERR_SEQ_LEN);
    return;
  }
  const int blk = __ldg(block_table + static_cast<int64_t>(b) * bt_stride + pos / block_size);
  if (blk < 0 || blk >= num_blocks) {
    if (lane == 0) report(dev_status, DSA_DEVERR_BLOCK_OOB);
    return;
  }
  uint8_t* row = cache + static_cast<int64_t>(blk) * block_stride + (pos % block_size) * kF8RowBytes;
  uint32_t code[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = ptx::cvt_e4m3x2(__fdiv_rn(x[4 * i], scale), __fdiv_rn(x[4 * i + 1], scale));
    const uint32_t hi = ptx::cvt_e4m3x2(__fdiv_rn(x[4 * i + 2], scale), __fdiv_rn(x[4 * i + 3], scale));
    code[i] = lo | (hi << 16);
  }
  *reinterpret_cast<uint4*>(row + 16 * lane) = make_uint4(code[0], code[1], code[2], code[3]);
  if ((lane & 7) == 0) *reinterpret_cast<float*>(row + kF8Dv + 4 * (lane >> 3)) = scale;
  if (lane < 8) *reinterpret_cast<uint4*>(row + kF8Dv + 16 + 16 * lane) = rope;
}

}  // namespace
}  // namespace dsa

using namespace dsa;

extern "C" dsa_status_t dsa_mla_kv_fp8_quant_and_cache(const void* kv, int64_t kv_stride_t, int32_t T, int32_t Dk,
                                                       int32_t Dv, uint8_t* kv_cache, int64_t kv_block_stride_bytes,
                                                       int32_t num_blocks, const int32_t* block_table,
                                                       int32_t bt_stride, const int32_t* seq_lens,
                                                       const int32_t* query_start_loc, int32_t B, int32_t block_size,
                                                       int32_t* dev_status, dsa_stream_t stream) {
  if (T < 0 || B < 0 || block_size <= 0 || num_blocks < 0 || bt_stride < 0)
    return fail(DSA_ERR_INVALID_ARG, "dsa_mla_kv_fp8_quant_and_cache: negative or zero size argument");
  if (Dk != kF8Dk || Dv != kF8Dv)
    return fail(DSA_ERR_UNSUPPORTED, "dsa_mla_kv_fp8_quant_and_cache: (Dk, Dv) = (%d, %d), only (576, 512)", Dk, Dv);
  if (block_size % 64)
    return fail(DSA_ERR_UNSUPPORTED, "dsa_mla_kv_fp8_quant_and_cache: block_size %d not a multiple of 64", block_size);
  if (T == 0) return DSA_OK;
  if (B == 0) return fail(DSA_ERR_INVALID_ARG, "dsa_mla_kv_fp8_quant_and_cache: T > 0 tokens but no request");
  if (!kv || !kv_cache || !block_table || !seq_lens || !query_start_loc)
    return fail(DSA_ERR_INVALID_ARG, "dsa_mla_kv_fp8_quant_and_cache: null pointer");
  if (kv_block_stride_bytes < static_cast<int64_t>(block_size) * kF8RowBytes || kv_block_stride_bytes % kF8RowBytes)
    return fail(DSA_ERR_INVALID_ARG,
                "dsa_mla_kv_fp8_quant_and_cache: kv_block_stride_bytes %lld must be a whole number (>= block_size) "
                "of 656-byte rows",
                static_cast<long long>(kv_block_stride_bytes));
  if (!aligned16(kv) || !aligned16(kv_cache) || kv_stride_t < Dk || kv_stride_t % 8)
    return fail(DSA_ERR_INVALID_ARG,
                "dsa_mla_kv_fp8_quant_and_cache: kv/kv_cache must be 16-byte aligned, token stride >= Dk and a "
                "multiple of 8");
  dsa_status_t st = check_device();
  if (st != DSA_OK) return st;
  const unsigned grid = static_cast<unsigned>((static_cast<int64_t>(T) * 32 + kThreads - 1) / kThreads);
  mla_kv_fp8_cache_kernel<<<grid, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint16_t*>(kv), kv_stride_t, T, kv_cache, kv_block_stride_bytes, num_blocks, block_table,
      bt_stride, seq_lens, query_start_loc, B, block_size, dev_status);
  return check_launch("mla_kv_fp8_cache_kernel");
}

extern "C" dsa_status_t dsa_indexer_k_quant_and_cache(const void* k, int64_t k_stride_t, int32_t T, int32_t Di,
                                                      uint8_t* k_cache, int64_t k_block_stride_bytes,
                                                      int32_t num_blocks, const int32_t* block_table,
                                                      int32_t bt_stride, const int32_t* seq_lens,
                                                      const int32_t* query_start_loc, int32_t B, int32_t block_size,
                                                      int32_t* dev_status, dsa_stream_t stream) {
  if (T < 0 || B < 0 || Di <= 0 || block_size <= 0 || num_blocks < 0 || bt_stride < 0)
    return fail(DSA_ERR_INVALID_ARG, "dsa_indexer_k_quant_and_cache: negative or zero size argument");
  if (Di != 32 && Di != 64 && Di != 128)
    return fail(DSA_ERR_UNSUPPORTED, "dsa_indexer_k_quant_and_cache: Di=%d not in {32,64,128}", Di);
  if (block_size % 64)
    return fail(DSA_ERR_UNSUPPORTED, "dsa_indexer_k_quant_and_cache: block_size %d not a multiple of 64", block_size);
  if (T == 0) return DSA_OK;
  if (B == 0) return fail(DSA_ERR_INVALID_ARG, "dsa_indexer_k_quant_and_cache: T > 0 tokens but no request");
  if (!k || !k_cache || !block_table || !seq_lens || !query_start_loc)
    return fail(DSA_ERR_INVALID_ARG, "dsa_indexer_k_quant_and_cache: null pointer");
  if (k_block_stride_bytes < static_cast<int64_t>(block_size) * (Di + 4) || k_block_stride_bytes % 16)
    return fail(DSA_ERR_INVALID_ARG,
                "dsa_indexer_k_quant_and_cache: k_block_stride_bytes %lld must be >= block_size*(Di+4) and a multiple of 16",
                static_cast<long long>(k_block_stride_bytes));
  if (!aligned16(k) || !aligned16(k_cache) || k_stride_t < Di || k_stride_t % 8)
    return fail(DSA_ERR_INVALID_ARG,
                "dsa_indexer_k_quant_and_cache: k/k_cache must be 16-byte aligned, token stride >= Di and a multiple of 8");
  dsa_status_t st = check_device();
  if (st != DSA_OK) return st;
  const unsigned grid = static_cast<unsigned>((static_cast<int64_t>(T) * 32 + kThreads - 1) / kThreads);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const uint16_t* kk = static_cast<const uint16_t*>(k);
  switch (Di) {
    case 128:
      k_quant_cache_kernel<128><<<grid, kThreads, 0, s>>>(kk, k_stride_t, T, k_cache, k_block_stride_bytes, num_blocks,
                                                          block_table, bt_stride, seq_lens, query_start_loc, B,
                                                          block_size, dev_status);
      break;
    case 64:
      k_quant_cache_kernel<64><<<grid, kThreads, 0, s>>>(kk, k_stride_t, T, k_cache, k_block_stride_bytes, num_blocks,
                                                         block_table, bt_stride, seq_lens, query_start_loc, B,
                                                         block_size, dev_status);
      break;
    default:
      k_quant_cache_kernel<32><<<grid, kThreads, 0, s>>>(kk, k_stride_t, T, k_cache, k_block_stride_bytes, num_blocks,
                                                         block_table, bt_stride, seq_lens, query_start_loc, B,
                                                         block_size, dev_status);
      break;
  }
  return check_launch("k_quant_cache_kernel");
}
