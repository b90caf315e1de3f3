/*
 * dsa.h -- C ABI of libdsa, the DeepSeek-Sparse-Attention (DSA) step on one
 * GB300 (sm_103a).
 *
 * The step, per attention layer and batch of query tokens:
 *   a0  quantise the indexer query to e4m3, one fp32 scale per (token, head)
 *   a1  lightning-indexer logits over a paged fp8 key cache
 *         logits[t,s] = sum_h w[t,h] * ReLU(q[t,h,:] . dequant(k[s,:]))
 *   a2  top-k of each logits row
 *   a3  sparse MLA attention over the selected rows of a paged bf16 latent
 *       KV cache, optionally split into KV splits
 *   a4  online-softmax merge of the split partials
 *
 * Sources: vLLM PR #38476 "[Feature] TRITON_MLA_SPARSE backend for
 * SM8x/11x/12x DSA Sparse MLA Support" (Changes 2: fp8 MQA logits, prefill and
 * paged decode, the K scale applied to the fp32 dot; Changes 3: split-KV
 * sparse-MLA decode, N-way online-softmax merge, single-pass path, -1e30
 * sentinel for masked slots; Changes 4: CUDA-graph capture; Tests:
 * clean/dirty logits; review thread: top-k after the indexer,
 * per_token_group_quant_fp8 of the indexer q, chunked exact top-k) and the
 * "vllm-dsa-mtp-sm80" README ("The skew fixes", item 0: the 132-byte indexer
 * page per token, blocks addressed through the cache's block stride).
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller. The library
 *     never allocates, frees or synchronises; every call only enqueues kernels
 *     on `stream`.
 *   - Arguments are validated on the host before any launch. A bad argument
 *     returns DSA_ERR_INVALID_ARG (or DSA_ERR_UNSUPPORTED for a valid but
 *     unimplemented shape) and launches nothing; dsa_last_error() then holds
 *     a one-line reason (thread-local, valid until the next call on the
 *     thread).
 *   - Values that only the device sees (block-table entries, top-k indices,
 *     seq_lens) are checked in the kernels. A bad one never traps: the access
 *     is skipped (masked / zero-filled) and the matching DSA_DEVERR_* bit is
 *     OR-ed into *dev_status when dev_status is non-NULL.
 *   - Every wait inside a kernel is bounded (about one second); a wait that
 *     runs out sets DSA_DEVERR_TIMEOUT and the kernel returns.
 *   - The top-k, attention and merge kernels are launched as programmatic
 *     dependents of the kernel before them on the stream. Before waiting for
 *     it they read only inputs that no kernel of this library writes (q,
 *     seq_lens, query_start_loc); a caller's kernel placed directly before
 *     them that lets its dependents start early must not write those.
 *   - Request b owns query tokens [query_start_loc[b], query_start_loc[b+1]);
 *     q_len_b is their count. seq_lens[b] counts the request's cached keys
 *     INCLUDING its q_len_b new tokens, so query token t of request b sits at
 *     position pos(t) = seq_lens[b] - q_len_b + (t - query_start_loc[b]) and
 *     attends causally to keys 0..pos(t); valid(t) = pos(t) + 1.
 *   - block_size must be a multiple of 64. Block table row b (stride
 *     bt_stride int32 entries) maps logical block i of request b to a
 *     physical block in [0, num_blocks).
 *
 * Paged cache layouts
 *   Indexer key cache (fp8): block p starts at byte p * k_block_stride_bytes
 *   (>= block_size * (Di + 4), a multiple of 16). Inside it: block_size rows
 *   of Di e4m3 bytes (token-major), then block_size fp32 scales. The key of
 *   token s is dequant(k[s,:]) = e4m3(k[s,:]) * scale[s]. With Di = 128 this
 *   is the 132-byte-per-token page.
 *   Latent KV cache (bf16): block p starts at element p * kv_block_stride;
 *   inside it block_size rows of Dk bf16 (Dk = 576: 512 latent + 64 rope).
 *   The value vector of a row is its first Dv elements.
 *   Latent KV cache (fp8, Dk = 576, Dv = 512): block p starts at byte
 *   p * kv_block_stride_bytes (a whole number, >= block_size, of 656-byte
 *   rows); inside it block_size rows of 656 bytes: 512 e4m3 codes of the
 *   latent dims, then 4 fp32 scales (one per 128-dim group, little-endian),
 *   then the 64 rope dims as bf16. A latent value is e4m3(code) * scale of
 *   its group; a group is quantised with scale = amax/448 (1 when amax == 0)
 *   and code = e4m3_rn_satfinite(x / scale). vLLM PR #38476 (Limitations,
 *   review thread) names FP8-KV sparse-MLA backends for SM90+/SM12x parts but
 *   prints no layout; this is the layout this library reads and writes.
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* dsa_stream_t; /* same type as cudaStream_t; NULL = legacy default stream */

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1, /* null pointer, negative size, inconsistent strides ... */
  DSA_ERR_UNSUPPORTED = 2, /* not an sm_103 device, or dims outside the compiled set */
  DSA_ERR_WORKSPACE = 3,   /* workspace missing or smaller than the *_workspace_size() figure */
  DSA_ERR_CUDA = 4         /* a CUDA runtime call failed (launch error, ...) */
} dsa_status_t;

/* Bits OR-ed into *dev_status by the kernels. */
#define DSA_DEVERR_BLOCK_OOB 1u /* a block-table entry outside [0, num_blocks) was needed */
#define DSA_DEVERR_INDEX_OOB 2u /* a top-k index outside [-1, valid(t)) was given */
#define DSA_DEVERR_TIMEOUT 4u   /* a bounded wait inside a kernel ran out */
#define DSA_DEVERR_SEQ_LEN 8u   /* seq_lens[b] < q_len_b, or larger than the block table can hold */

/* num_kv_splits value of sparse_mla_decode that makes the split count depend
 * on index_topk alone, so a token's out and lse do not depend on the batch. */
#define DSA_KV_SPLITS_BATCH_INVARIANT (-1)

/* One-line reason for the last non-OK status returned on this thread. */
const char* dsa_last_error(void);

/* Library version string. */
const char* dsa_version(void);

/*
 * a0 on its own: quantise q_idx [T, Hi, Di] (bf16, token stride q_stride_t
 * elements, contiguous heads and dims) to e4m3 codes q8 [T, Hi, Di] and fp32
 * scales sq [T, Hi], scale = amax/448 (1 when amax == 0), code =
 * e4m3_rn_satfinite(x / scale). dsa_indexer_logits performs the same
 * quantisation internally; this entry point exposes it so its codes can be
 * compared bit for bit. (vLLM PR #38476 review thread: per_token_group_quant_fp8
 * quantises the indexer q per token group.)
 */
dsa_status_t dsa_quant_q(const void* q_idx, int64_t q_stride_t, int32_t T, int32_t Hi, int32_t Di, uint8_t* q8,
                         float* sq, dsa_stream_t stream);

/*
 * a0 + a1: indexer logits over the paged fp8 key cache.
 *   q_idx  bf16 [T, Hi, Di], token stride q_stride_t elements
 *   w      fp32 [T, Hi] head weights
 *   logits fp32 [T, ld] output. For every token t all ld entries are
 *          written: the logit for s < valid(t), -inf for valid(t) <= s < ld
 *          (the clean-logits contract). ld >= max_b seq_lens[b] is required
 *          (a longer request sets DSA_DEVERR_SEQ_LEN and is clipped to ld).
 * max_q_len is an upper bound of q_len_b over the batch (1 or 2 for decode,
 * larger for prefill). Supported: Hi <= 64, Di in {32, 64, 128}.
 * (vLLM PR #38476 Changes 2.)
 */
dsa_status_t dsa_indexer_logits(const void* q_idx, int64_t q_stride_t, const float* w, const uint8_t* k_cache,
                                int64_t k_block_stride_bytes, int32_t num_blocks, const int32_t* block_table,
                                int32_t bt_stride, const int32_t* seq_lens, const int32_t* query_start_loc, int32_t B,
                                int32_t T, int32_t Hi, int32_t Di, int32_t block_size, int32_t max_q_len,
                                float* logits, int64_t ld, int32_t* dev_status, dsa_stream_t stream);

/*
 * Producer side of the indexer key cache (the op indexer_k_quant_and_cache
 * of the "vllm-dsa-mtp-sm80" README, "The skew fixes", item 0): quantise the
 * keys of the T new query tokens and store them in the paged fp8 cache that
 * dsa_indexer_logits reads.
 *   k        bf16 [T, Di], token stride k_stride_t elements (>= Di, a multiple
 *            of 8; 16-byte aligned), one row per query token in query order
 *   k_cache  the indexer key cache (layout above), written in place: for each
 *            token t of request b, the Di code bytes and the fp32 scale of key
 *            position pos(t) = seq_lens[b] - q_len_b + (t - query_start_loc[b])
 *            in block block_table[b, pos(t) / block_size]. Nothing else of the
 *            cache is touched.
 * Per token: scale = amax(|k[t,:]|)/448 (1 when amax == 0) and code =
 * e4m3_rn_satfinite(k / scale), both divisions IEEE-rounded fp32: the rule of
 * a0 applied to the key row (finite inputs). A position outside the block
 * table (DSA_DEVERR_SEQ_LEN) or a block id outside [0, num_blocks)
 * (DSA_DEVERR_BLOCK_OOB) skips that token. Supported: Di in {32, 64, 128};
 * block_size a multiple of 64. Tokens must not share a position (each writes
 * its row without ordering against the others).
 */
dsa_status_t dsa_indexer_k_quant_and_cache(const void* k, int64_t k_stride_t, int32_t T, int32_t Di, uint8_t* k_cache,
                                           int64_t k_block_stride_bytes, int32_t num_blocks,
                                           const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens,
                                           const int32_t* query_start_loc, int32_t B, int32_t block_size,
                                           int32_t* dev_status, dsa_stream_t stream);

/*
 * a2: top-k of each logits row.
 * Row t ranks logits[t, 0:valid(t)] (fp32, compared as floats so -0.0 equals
 * +0.0); the n = min(index_topk, valid(t)) largest are selected, equal values
 * resolved toward the lower position. topk_idx [T, index_topk] receives the n
 * selected positions in ascending position order, then -1 in the remaining
 * slots. A row is shared by up to 8 CTAs of one cluster, which combine their
 * histograms in distributed shared memory: dsa_topk_workspace_size() is 0 and
 * `workspace` may be NULL (both stay in the interface for callers that size a
 * workspace generically). Requires ld < 2^31 and index_topk <= 65535.
 * (vLLM PR #38476 review thread: index_topk selection.)
 */
size_t dsa_topk_workspace_size(int32_t T, int64_t ld, int32_t index_topk);
dsa_status_t dsa_topk(const float* logits, int64_t ld, const int32_t* seq_lens, const int32_t* query_start_loc,
                      int32_t B, int32_t T, int32_t index_topk, int32_t* topk_idx, void* workspace, size_t ws_bytes,
                      dsa_stream_t stream);

/*
 * a1 + a2 with a bounded logits buffer: the indexer logits and the top-k
 * computed over windows of `window` keys (vLLM PR #38476 review thread: the
 * [batch, max_seq_len] fp32 decode logits buffer is bounded by windowing the
 * keys, taking a top-k per window as (score, key) candidates and one final
 * top-k over the concatenated candidates; any key of the global top-k is in
 * its window's top-k, so the result is exact).
 * Arguments as dsa_indexer_logits, then:
 *   max_seq_len  upper bound of seq_lens (a longer request is clipped to the
 *                windows covering it and sets DSA_DEVERR_SEQ_LEN)
 *   window       keys per window, a multiple of 128 and of block_size; 0 =
 *                one window of max_seq_len (rounded up to 128)
 *   topk_idx     int32 [T, index_topk], exactly dsa_topk's result on the
 *                logits of dsa_indexer_logits (the same selection, ascending
 *                key positions, -1 padded)
 *   workspace    dsa_indexer_topk_workspace_size(T, max_seq_len, window,
 *                index_topk) bytes, 16-byte aligned: a [T, window] fp32 logits
 *                buffer and, with several windows, the candidates (value and
 *                key, [T, windows * min(index_topk, window)] each).
 * Kernels per call: a logits kernel and a top-k kernel per window, and one
 * final top-k when there are several windows.
 */
size_t dsa_indexer_topk_workspace_size(int32_t T, int64_t max_seq_len, int32_t window, int32_t index_topk);
dsa_status_t dsa_indexer_topk(const void* q_idx, int64_t q_stride_t, const float* w, const uint8_t* k_cache,
                              int64_t k_block_stride_bytes, int32_t num_blocks, const int32_t* block_table,
                              int32_t bt_stride, const int32_t* seq_lens, const int32_t* query_start_loc, int32_t B,
                              int32_t T, int32_t Hi, int32_t Di, int32_t block_size, int32_t max_q_len,
                              int64_t max_seq_len, int32_t window, int32_t index_topk, int32_t* topk_idx,
                              void* workspace, size_t ws_bytes, int32_t* dev_status, dsa_stream_t stream);

/*
 * a3 (+ a4): sparse MLA decode with split-KV.
 *   q         bf16 [T, H, Dk] (contiguous)
 *   kv_cache  bf16 paged latent cache (layout above)
 *   topk_idx  int32 [T, index_topk]: logical key positions of the token's
 *             request, -1 = empty slot. An index outside [-1, valid(t)) is
 *             treated as empty and sets DSA_DEVERR_INDEX_OOB.
 *   out       bf16 [T, H, Dv]: softmax(scale * q . kv[sel]) @ kv[sel, :Dv]
 *   lse       fp32 [T, H] natural-log sum-exp of the scaled scores, or NULL.
 * num_kv_splits: the number S of KV splits.
 *   1..32  that many splits;
 *   0      chosen from T, H, Dv, index_topk and the SM count
 *          (sparse_mla_auto_splits). The count then depends on the batch
 *          size, and so do the bf16 roundings of a token's out and lse;
 *   DSA_KV_SPLITS_BATCH_INVARIANT (-1)
 *          ceil(index_topk / 2048) splits, fixed by index_topk alone: a
 *          token's out and lse are bit-identical in any batch (every kernel
 *          of the step works on one token of one request at a time). With
 *          index_topk <= 2048 this is the single-pass path (the batch-invariant
 *          mode of vLLM PR #38476, Limitations: force one KV split).
 * sparse_mla_num_splits() resolves 0 and -1 to the count a call will use.
 * With S > 1 the top-k slots are cut into S contiguous ranges of
 * ceil(index_topk / S); each split writes fp32 partials to `workspace`
 * (sparse_mla_workspace_size(T, H, Dv, S) bytes) and a merge kernel combines
 * them. Empty slots score the finite sentinel -1e30 and carry weight 0, so an
 * all-empty split contributes nothing and no NaN appears; a token with no
 * selected row gets out = 0 and lse = -inf.
 * Score arithmetic (Dk = 576): the dims of a row are split between two CTAs
 * (latent [0,256) with rope [512,544), latent [256,512) with rope [544,576));
 * each CTA's half-score comes from an fp32 tensor-core accumulator, is scaled
 * by softmax_scale * log2(e) in fp32 and exchanged in fp32, and the two
 * halves are added in fp32 (no input-range limit beyond fp32's).
 * Supported: H <= 128, (Dk, Dv) in {(576, 512), (80, 64)}, 1 <= S and
 * ceil(index_topk / S) <= 2048.
 * (vLLM PR #38476 Changes 3.)
 */
/* Workspace bytes of S = num_kv_splits splits (an actual count: 0 when S <= 1). */
size_t sparse_mla_workspace_size(int32_t T, int32_t H, int32_t Dv, int32_t num_kv_splits);
/* The automatic split count: a wave-count cost model over the SM count. */
int32_t sparse_mla_auto_splits(int32_t T, int32_t H, int32_t Dv, int32_t index_topk);
/* The split count sparse_mla_decode uses for this num_kv_splits argument. */
int32_t sparse_mla_num_splits(int32_t T, int32_t H, int32_t Dv, int32_t index_topk, int32_t num_kv_splits);
dsa_status_t sparse_mla_decode(const void* q, const void* kv_cache, int64_t kv_block_stride, int32_t num_blocks,
                               const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens,
                               const int32_t* query_start_loc, const int32_t* topk_idx, int32_t B, int32_t T,
                               int32_t H, int32_t Dk, int32_t Dv, int32_t index_topk, int32_t block_size,
                               float softmax_scale, int32_t num_kv_splits, void* out, float* lse, void* workspace,
                               size_t ws_bytes, int32_t* dev_status, dsa_stream_t stream);

/*
 * a3 for prefill / many query tokens: the single-pass path (no splits, no
 * workspace). Same arguments and results as sparse_mla_decode with
 * num_kv_splits = 1. (vLLM PR #38476 Changes 3, single-pass path.)
 */
dsa_status_t sparse_mla_prefill(const void* q, const void* kv_cache, int64_t kv_block_stride, int32_t num_blocks,
                                const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens,
                                const int32_t* query_start_loc, const int32_t* topk_idx, int32_t B, int32_t T,
                                int32_t H, int32_t Dk, int32_t Dv, int32_t index_topk, int32_t block_size,
                                float softmax_scale, void* out, float* lse, int32_t* dev_status,
                                dsa_stream_t stream);

/*
 * a3 (+ a4) over the fp8 latent cache (layout above): the same calls,
 * arguments and results as sparse_mla_decode / sparse_mla_prefill, with
 * kv_cache the fp8 cache and its block stride in bytes. Each CTA gathers the
 * 256 code bytes of its half of the latent dims, the row's 16 scale bytes and
 * its 32 rope dims (336 of the row's 656 bytes; 576 of 1152 for bf16) and
 * dequantises the codes to bf16 (code * scale, rounded to nearest even) in
 * shared memory before the bf16 tensor-core products. Supported: (Dk, Dv) =
 * (576, 512), H <= 128. (vLLM PR #38476 Limitations and review thread: FP8
 * latent caches on SM90+ parts.)
 */
dsa_status_t sparse_mla_decode_fp8(const void* q, const uint8_t* kv_cache, int64_t kv_block_stride_bytes,
                                   int32_t num_blocks, const int32_t* block_table, int32_t bt_stride,
                                   const int32_t* seq_lens, const int32_t* query_start_loc, const int32_t* topk_idx,
                                   int32_t B, int32_t T, int32_t H, int32_t Dk, int32_t Dv, int32_t index_topk,
                                   int32_t block_size, float softmax_scale, int32_t num_kv_splits, void* out,
                                   float* lse, void* workspace, size_t ws_bytes, int32_t* dev_status,
                                   dsa_stream_t stream);
dsa_status_t sparse_mla_prefill_fp8(const void* q, const uint8_t* kv_cache, int64_t kv_block_stride_bytes,
                                    int32_t num_blocks, const int32_t* block_table, int32_t bt_stride,
                                    const int32_t* seq_lens, const int32_t* query_start_loc, const int32_t* topk_idx,
                                    int32_t B, int32_t T, int32_t H, int32_t Dk, int32_t Dv, int32_t index_topk,
                                    int32_t block_size, float softmax_scale, void* out, float* lse,
                                    int32_t* dev_status, dsa_stream_t stream);

/*
 * Producer side of the fp8 latent cache: quantise the latent rows of the T
 * new query tokens and store them in the fp8 cache (layout above), the way
 * dsa_indexer_k_quant_and_cache stores indexer keys.
 *   kv       bf16 [T, Dk], token stride kv_stride_t elements (>= Dk, a
 *            multiple of 8; 16-byte aligned), one row per query token
 *   kv_cache the fp8 latent cache, written in place: token t of request b
 *            goes to row pos(t) % block_size of block
 *            block_table[b, pos(t) / block_size]; nothing else is touched.
 * Per token: four 128-dim groups of the 512 latent dims, each with scale =
 * amax/448 (1 when amax == 0) and code = e4m3_rn_satfinite(x / scale), both
 * divisions IEEE-rounded fp32; the 64 rope dims keep their bf16 bits. A
 * position outside the block table (DSA_DEVERR_SEQ_LEN) or a block id outside
 * [0, num_blocks) (DSA_DEVERR_BLOCK_OOB) skips that token. Supported: (Dk, Dv)
 * = (576, 512), block_size a multiple of 64.
 */
dsa_status_t dsa_mla_kv_fp8_quant_and_cache(const void* kv, int64_t kv_stride_t, int32_t T, int32_t Dk, int32_t Dv,
                                            uint8_t* kv_cache, int64_t kv_block_stride_bytes, int32_t num_blocks,
                                            const int32_t* block_table, int32_t bt_stride, const int32_t* seq_lens,
                                            const int32_t* query_start_loc, int32_t B, int32_t block_size,
                                            int32_t* dev_status, dsa_stream_t stream);

/*
 * Split-KV sparse MLA decode that allocates nothing. It serves callers that
 * may not call cudaMalloc when they run the step: serving runtimes that hand
 * all device memory to their own allocator at start-up and forbid later
 * allocations, and host environments (plugins, sandboxed runtimes) that are
 * not allowed to create device allocations. The pages have no counterpart of
 * this entry point; it is a deployment convenience.
 *
 * Same arguments and results as sparse_mla_decode, minus the workspace: the
 * split partials go to a fixed scratch array of sparse_mla_fixed_scratch_bytes()
 * bytes (24 MiB) that the library reserves in device memory on every GPU that
 * loads it, held until the process exits. With num_kv_splits = 0 the
 * automatic count is lowered, down to the fewest splits allowed, until the
 * partials fit. A request whose partials (sparse_mla_workspace_size for the
 * resulting number of splits) still exceed the array is rejected with
 * DSA_ERR_WORKSPACE and launches nothing.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) for that device; make that first call before any
 *     stream capture that includes this entry point.
 *   - All calls share the one array, which keeps the last call's contents.
 *     Calls that may overlap on the GPU (on different streams, or in parallel
 *     graphs) race on it and must be serialised by the caller.
 *   - Nothing in the array needs to start at zero: every partial the merge
 *     reads is written first in the same call.
 */
size_t sparse_mla_fixed_scratch_bytes(void);
dsa_status_t sparse_mla_decode_fixed_scratch(const void* q, const void* kv_cache, int64_t kv_block_stride,
                                             int32_t num_blocks, const int32_t* block_table, int32_t bt_stride,
                                             const int32_t* seq_lens, const int32_t* query_start_loc,
                                             const int32_t* topk_idx, int32_t B, int32_t T, int32_t H, int32_t Dk,
                                             int32_t Dv, int32_t index_topk, int32_t block_size, float softmax_scale,
                                             int32_t num_kv_splits, void* out, float* lse, int32_t* dev_status,
                                             dsa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H_ */
