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

}  // namespace
}  // namespace dsa

using namespace dsa;

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
