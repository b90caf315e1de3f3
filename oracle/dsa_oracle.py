"""CPU oracle for the DeepSeek-Sparse-Attention (DSA) step.

TEST INFRASTRUCTURE ONLY. Only the test suite, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module. The product path (the CUDA library and its Python binding) never calls
it, and this module imports nothing from the product.

What it computes is the plain definition of each step of the method, in
float64 with numpy, one query token at a time:

  a0  per-(token, head) fp8 quantisation of the indexer query
  a1  lightning-indexer logits over a paged fp8 key cache, causally masked
  a2  per-query top-k selection (ties to the lower index, -1 padding)
  a3  sparse MLA attention over the selected rows of a paged bf16 latent cache,
      single pass or split into KV splits
  a4  merge of the split partials by online softmax
  and, on the producer side, the new tokens' indexer keys quantised into the
  paged fp8 key cache (indexer_k_quant_and_cache)
  the fp8 variant of the latent cache: its row layout, the quantisation of new
  latent rows into it, and its decoding (a3 then runs on the decoded rows)

Sources (web pages; cited by title and section):
  [PR]     vLLM PR #38476, "[Feature] TRITON_MLA_SPARSE backend for SM8x/11x/12x
           DSA Sparse MLA Support" -- Changes 2 (indexer fp8 MQA logits, scale
           applied to the fp32 dot, paged decode, 256-entry fp8 decode),
           Changes 3 (split-KV decode, N-way online-softmax merge, single-pass
           path, -1e30 masked sentinel), Tests (clean/dirty logits), and the
           review thread (skip_topk_buffer_clear / top-k, per_token_group_quant_fp8
           for the indexer q, the chunked exact top-k argument, the
           [batch, max_seq_len] fp32 decode logits buffer).
  [README] "vllm-dsa-mtp-sm80" README, "The skew fixes" item 0 (132-byte
           indexer page per token, 96:11 page ratio against the 576-dim bf16
           MLA page, blocks addressed by the cache's block stride).
  The step's formulas: logits[t,s] = sum_h w[t,h] * ReLU(q[t,h,:] . dequant(k[s,:]));
  top-k of each logits row; softmax attention over the selected rows.

Readings where the pages are silent:
  * e4m3 is OCP E4M3FN: bias 7, max 448, no infinities, S.1111.111 is NaN.
  * q quantisation: per (token, head) group of head_dim values,
    scale = amax / 448 in fp32; codes = e4m3_rn_sat(fp32(x / scale)); amax == 0
    gives scale 1 and all-zero codes.
  * Indexer page layout inside one block of block_size tokens: block_size x 128
    e4m3 bytes (token-major) followed by block_size fp32 scales.
  * The new tokens' keys are quantised with the q rule (one group = a key's Di
    values) and stored at the tokens' own positions (below).
  * seq_lens include the new tokens, whose keys are already in the cache;
    query token t of request b sits at position seq_len_b - q_len_b + (t - qsl_b)
    and sees keys s <= that position.
  * Top-k ranks by fp32 value compared as floats (so -0.0 == +0.0), ties go to
    the lower index, min(K, valid) entries are kept and the rest are -1.
  * Top-k indices are logical positions inside the request; attention maps them
    through the block table. The value vector is the first Dv dims of the
    Dk-dim latent row.
  * An empty selection gives output 0 and lse -inf.
  * Split j covers top-k slots [j*ceil(K/S), min(K, (j+1)*ceil(K/S))); a -1
    slot scores the -1e30 sentinel and carries weight 0.
  * fp8 latent cache ([PR] Limitations and review thread: the FP8-KV sparse-MLA
    backends of SM90+/SM12x parts; the pages print no layout). One token's row
    holds its Dv latent values as e4m3 codes in groups of 128 with one fp32
    scale per group (the q rule: amax/448, 1 when amax == 0), then its Dk - Dv
    rope values unchanged in bf16: [Dv code bytes][Dv/128 fp32 scales]
    [(Dk-Dv) bf16], 656 bytes at Dk = 576, Dv = 512. A decoded latent value is
    e4m3(code) * scale of its group.
"""
from __future__ import annotations

import math

import numpy as np

NEG_SENTINEL = -1e30
E4M3_MAX = 448.0

# ----------------------------------------------------------------------------
# e4m3 (OCP E4M3FN)
# ----------------------------------------------------------------------------


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """Value of each e4m3 byte, float64.

    [PR] Changes 2 decodes all 256 fp8 codes through a table; this is the
    format's definition: sign S, exponent E (bias 7), mantissa M.
      E > 0 : (-1)^S * 2^(E-7) * (1 + M/8)
      E == 0: (-1)^S * 2^-6 * (M/8)        (subnormal)
      E == 15 and M == 7: NaN               (no infinities)
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = (c >> 7) & 1
    e = (c >> 3) & 0xF
    m = c & 7
    mag = np.where(e == 0, np.ldexp(m / 8.0, -6), np.ldexp(1.0 + m / 8.0, e - 7))
    val = np.where(s == 1, -mag, mag)
    return np.where((e == 15) & (m == 7), np.nan, val)


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """Round finite float values to e4m3 codes: nearest, ties to even, and
    saturation to +-448 for magnitudes beyond it (the satfinite rule).

    Works on the exact value of each input (float64 holds any fp32 exactly).
    Zero keeps its sign. NaN input is not expected and maps to 0x7F.
    """
    x = np.asarray(x, dtype=np.float64)
    sign = np.where(np.signbit(x), 0x80, 0x00).astype(np.int64)
    # magnitudes past 2^10 all saturate; clipping keeps the arithmetic finite
    a = np.minimum(np.abs(np.nan_to_num(x, nan=0.0)), 1024.0)
    out = np.zeros(a.shape, dtype=np.int64)
    # exponent of the binade: a in [2^e, 2^(e+1))
    _, fe = np.frexp(np.where(a > 0, a, 1.0))
    e = fe.astype(np.int64) - 1
    sub = a < 2.0**-6
    # subnormal range: multiples of 2^-9; rint rounds half to even
    q_sub = np.rint(a / 2.0**-9).astype(np.int64)  # may reach 8 == code of 2^-6
    # normal range: 3 mantissa bits
    frac = np.where(sub, 0.0, a / np.ldexp(1.0, np.clip(e, -6, 8)) - 1.0)
    q = np.rint(frac * 8.0).astype(np.int64)
    e_adj = np.where(q == 8, e + 1, e)
    q = np.where(q == 8, 0, q)
    normal_code = ((e_adj + 7) << 3) | q
    out = np.where(sub, q_sub, normal_code)
    out = np.where(a >= E4M3_MAX, 0x7E, out)
    out = np.where(out > 0x7E, 0x7E, out)
    out = np.where(np.isnan(x), 0x7F, out | sign)
    return out.astype(np.uint8)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float64 values to bf16 (nearest, ties to even), returned as float64.

    Rounds the exact value directly to 8 significant bits (no fp32 detour).
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, copy=True)
    fin = np.isfinite(x) & (x != 0)
    mant, ex = np.frexp(x[fin])  # |mant| in [0.5, 1)
    # bf16 keeps 8 significant bits: mant * 2^8 rounded to an integer
    r = np.rint(mant * 256.0) / 256.0
    val = np.ldexp(r, ex)
    # below the bf16 normal range the spacing is fixed at 2^-133
    tiny = np.abs(x[fin]) < 2.0**-126
    val = np.where(tiny, np.rint(x[fin] / 2.0**-133) * 2.0**-133, val)
    out[fin] = val
    return out


# ----------------------------------------------------------------------------
# a0: per-(token, head) quantisation of the indexer query
# ----------------------------------------------------------------------------


def quantize_groups(x: np.ndarray):
    """Quantise each row of the last axis to e4m3 with one fp32 scale.

    [PR] review thread: the unfused per_token_group_quant_fp8 op quantises the
    indexer q per token group; the group is one head's head_dim values.
    scale = amax/448 (fp32 division, correctly rounded); codes are the e4m3
    rounding of fp32(x/scale). amax == 0 gives scale 1.0.
    Returns (codes uint8 [..., D], scales float32 [...]).
    """
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.max(np.abs(x32), axis=-1)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    y = (x32 / scale[..., None]).astype(np.float32)  # IEEE fp32 division
    return e4m3_encode(y), scale


# ----------------------------------------------------------------------------
# paged cache helpers
# ----------------------------------------------------------------------------


def token_positions(seq_lens, query_start_loc):
    """For every query token t: (request b, absolute position pos(t)).

    Reading: seq_len_b counts the request's new tokens, so the q_len_b new
    tokens occupy positions seq_len_b - q_len_b .. seq_len_b - 1 and token t
    may attend to keys 0..pos(t) (valid(t) = pos(t) + 1).
    """
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    qsl = np.asarray(query_start_loc, dtype=np.int64)
    T = int(qsl[-1])
    req = np.zeros(T, dtype=np.int64)
    pos = np.zeros(T, dtype=np.int64)
    for b in range(len(seq_lens)):
        q_len = qsl[b + 1] - qsl[b]
        for i in range(q_len):
            t = qsl[b] + i
            req[t] = b
            pos[t] = seq_lens[b] - q_len + i
    return req, pos


def indexer_k_quant_and_cache(k, k_cache, k_block_stride, block_table, seq_lens, query_start_loc, block_size):
    """Producer side of the indexer key cache: a copy of k_cache with the T
    new tokens' keys stored.

    [README] "The skew fixes" item 0 names indexer_k_quant_and_cache as the op
    that writes the indexer page (block_size rows of Di e4m3 bytes, then
    block_size fp32 scales) and addresses blocks through the cache's block
    stride. Each key row k[t] (bf16 values, exact in fp32) is quantised with
    the a0 rule of quantize_groups; token t of request b lands at position
    pos(t) of token_positions: block block_table[b, pos // block_size], row
    pos % block_size. A position past the block-table row or a block id
    outside the cache skips the token (the device code reports it).
    """
    k = np.asarray(k, dtype=np.float32)
    T, Di = k.shape
    codes, scales = quantize_groups(k)
    out = np.array(k_cache, dtype=np.uint8, copy=True).reshape(-1, k_block_stride)
    bt = np.asarray(block_table)
    req, pos = token_positions(seq_lens, query_start_loc)
    for t in range(T):
        b, p = int(req[t]), int(pos[t])
        if p < 0 or p >= bt.shape[1] * block_size:
            continue
        blk = int(bt[b, p // block_size])
        if blk < 0 or blk >= out.shape[0]:
            continue
        off = p % block_size
        out[blk, off * Di:(off + 1) * Di] = codes[t]
        sc0 = block_size * Di + off * 4
        out[blk, sc0:sc0 + 4] = np.array([scales[t]], dtype=np.float32).view(np.uint8)
    return out.reshape(np.shape(k_cache))


def gather_index_keys(k_cache: np.ndarray, block_stride: int, block_table_row, n_keys: int, block_size: int, head_dim: int):
    """Read the first n_keys keys of one request from the paged indexer cache.

    [README] "The skew fixes" item 0: one token takes 132 bytes (128 e4m3 +
    one fp32 scale) and blocks are addressed through the cache's block stride.
    Reading: inside a block, block_size*head_dim value bytes come first
    (token-major), then block_size fp32 scales.
    Returns (codes uint8 [n, head_dim], scales float32 [n]).
    """
    flat = np.asarray(k_cache, dtype=np.uint8).reshape(-1)
    codes = np.empty((n_keys, head_dim), dtype=np.uint8)
    scales = np.empty(n_keys, dtype=np.float32)
    for s in range(n_keys):
        blk = int(block_table_row[s // block_size])
        off = s % block_size
        base = blk * block_stride
        codes[s] = flat[base + off * head_dim: base + (off + 1) * head_dim]
        sb = base + block_size * head_dim + off * 4
        scales[s] = flat[sb: sb + 4].view(np.float32)[0]
    return codes, scales


def gather_kv_rows(kv_cache: np.ndarray, block_stride_elems: int, block_table_row, positions, block_size: int, dk: int):
    """Rows of the paged bf16 latent cache (given as float values) at the
    logical positions of one request. Layout [block][block_size][dk] with the
    block stride in elements; row i lives in block block_table[i // bs]."""
    flat = np.asarray(kv_cache).reshape(-1)
    out = np.empty((len(positions), dk), dtype=np.float64)
    for r, i in enumerate(positions):
        blk = int(block_table_row[int(i) // block_size])
        base = blk * block_stride_elems + (int(i) % block_size) * dk
        out[r] = flat[base: base + dk]
    return out


# ----------------------------------------------------------------------------
# a1: indexer logits
# ----------------------------------------------------------------------------


def indexer_logits(q_codes, q_scales, w, k_cache, k_block_stride, block_table, seq_lens, query_start_loc,
                   block_size, ld, rows=None):
    """logits[t, s] = sum_h w[t,h] * ReLU( dq[t,h,:] . dk[s,:] )   for s < valid(t)
                    = -inf                                        for valid(t) <= s < ld

    dq = e4m3(q) * q_scale and dk = e4m3(k) * k_scale are the fp8-decoded
    inputs; the sum is taken in float64 and rounded to fp32 once.
    [PR] Changes 2 (fp8 MQA logits over paged K; the K scale multiplies the
    fp32 dot), Tests (every logits position is written: clean_logits).
    `rows` restricts the computation to a subset of query tokens (others NaN).
    """
    q_codes = np.asarray(q_codes)
    T, Hi, Di = q_codes.shape
    req, pos = token_positions(seq_lens, query_start_loc)
    out = np.full((T, ld), np.nan, dtype=np.float32)
    dq_all = e4m3_decode(q_codes) * np.asarray(q_scales, dtype=np.float64)[..., None]
    w = np.asarray(w, dtype=np.float64)
    cache = {}
    for t in (range(T) if rows is None else rows):
        b = int(req[t])
        valid = int(pos[t]) + 1
        if b not in cache:
            codes, sc = gather_index_keys(k_cache, k_block_stride, block_table[b], int(seq_lens[b]), block_size, Di)
            cache = {b: e4m3_decode(codes) * sc.astype(np.float64)[:, None]}
        dk = cache[b][:valid]
        dots = dq_all[t] @ dk.T  # [Hi, valid]
        row = w[t] @ np.maximum(dots, 0.0)
        out[t, :valid] = row.astype(np.float32)
        out[t, valid:] = -np.inf
    return out


# ----------------------------------------------------------------------------
# a2: top-k
# ----------------------------------------------------------------------------


def topk_row(values: np.ndarray, k: int) -> np.ndarray:
    """The min(k, len(values)) positions with the largest values, largest
    first, equal values in increasing position order; -1 fills up to k.

    Values compare as floats, so -0.0 and +0.0 tie. A stable sort on the
    negated values gives exactly that order.
    """
    v = np.asarray(values, dtype=np.float32)
    order = np.argsort(-v, kind="stable")
    n = min(k, len(v))
    out = np.full(k, -1, dtype=np.int32)
    out[:n] = order[:n]
    return out


def topk(logits, seq_lens, query_start_loc, index_topk, rows=None):
    """[PR] review thread (index_topk selection after the indexer; the global
    top-k of a row is recoverable from per-chunk top-k candidates).
    Row t ranks logits[t, :valid(t)]."""
    logits = np.asarray(logits)
    T = logits.shape[0]
    _, pos = token_positions(seq_lens, query_start_loc)
    out = np.full((T, index_topk), -1, dtype=np.int32)
    for t in (range(T) if rows is None else rows):
        out[t] = topk_row(logits[t, : int(pos[t]) + 1], index_topk)
    return out


# ----------------------------------------------------------------------------
# a3 / a4: sparse MLA attention
# ----------------------------------------------------------------------------


def _selected_rows(kv_cache, kv_block_stride, block_table, b, idx_row, block_size, dk):
    sel = [int(i) for i in idx_row if int(i) != -1]
    rows = gather_kv_rows(kv_cache, kv_block_stride, block_table[b], sel, block_size, dk)
    return sel, rows


def sparse_mla(q, kv_cache, kv_block_stride, block_table, seq_lens, query_start_loc, topk_idx, softmax_scale, dv,
               block_size, rows=None):
    """Single-pass sparse MLA for each query token t and head h:

      s_i   = softmax_scale * sum_{d<Dk} q[t,h,d] * kv[i,d]     for i in idx[t], i != -1
      p     = softmax(s) over the selected rows
      out   = sum_i p_i * kv[i, :Dv]          lse = log sum_i exp(s_i)

    [PR] Changes 3 (sparse MLA over the top-k rows, single-pass path).
    Returns (out float64 [T,H,Dv], lse float64 [T,H]).
    """
    q = np.asarray(q, dtype=np.float64)
    T, H, dk = q.shape
    req, _ = token_positions(seq_lens, query_start_loc)
    out = np.full((T, H, dv), np.nan)
    lse = np.full((T, H), np.nan)
    for t in (range(T) if rows is None else rows):
        _, kv = _selected_rows(kv_cache, kv_block_stride, block_table, int(req[t]), topk_idx[t], block_size, dk)
        if kv.shape[0] == 0:
            out[t] = 0.0
            lse[t] = -np.inf
            continue
        s = softmax_scale * (q[t] @ kv.T)  # [H, n]
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        den = e.sum(axis=1, keepdims=True)
        out[t] = (e / den) @ kv[:, :dv]
        lse[t] = (m + np.log(den))[:, 0]
    return out, lse


def split_bounds(k: int, num_splits: int):
    """Slot range of each split: [j*ceil(k/S), min(k, (j+1)*ceil(k/S)))."""
    per = -(-k // num_splits)
    return [(j * per, min(k, (j + 1) * per)) for j in range(num_splits)]


def sparse_mla_partials(q_t, kv_cache, kv_block_stride, block_table_row, idx_row, softmax_scale, dv, block_size,
                        num_splits):
    """Per-split online-softmax partials for one token (all heads).

    [PR] Changes 3: split-KV decode with a finite -1e30 sentinel for masked
    slots so an all-masked split yields no NaN. A -1 slot scores -1e30 and
    carries weight 0, so an empty split gives m = -1e30, l = 0, o = 0.
    Returns m [S,H], l [S,H], o [S,H,Dv] (o unnormalised).
    """
    q_t = np.asarray(q_t, dtype=np.float64)
    H, dk = q_t.shape
    S = num_splits
    m = np.full((S, H), NEG_SENTINEL)
    l = np.zeros((S, H))
    o = np.zeros((S, H, dv))
    for j, (lo, hi) in enumerate(split_bounds(len(idx_row), S)):
        slots = [int(i) for i in idx_row[lo:hi]]
        live = [i for i in slots if i != -1]
        if not live:
            continue
        kv = gather_kv_rows(kv_cache, kv_block_stride, block_table_row, live, block_size, dk)
        s = softmax_scale * (q_t @ kv.T)
        m[j] = np.maximum(NEG_SENTINEL, s.max(axis=1))
        e = np.exp(s - m[j][:, None])
        l[j] = e.sum(axis=1)
        o[j] = e @ kv[:, :dv]
    return m, l, o


def merge_partials(m, l, o):
    """N-way online-softmax merge ([PR] Changes 3):
      M = max_j m_j;  out = sum_j e^{m_j-M} o_j / sum_j e^{m_j-M} l_j;
      lse = M + log sum_j e^{m_j-M} l_j.  All l_j == 0 gives out 0, lse -inf.
    """
    M = m.max(axis=0)
    a = np.exp(m - M[None, :])
    den = (a * l).sum(axis=0)
    num = (a[..., None] * o).sum(axis=0)
    safe = den > 0
    out = np.where(safe[:, None], num / np.where(safe, den, 1.0)[:, None], 0.0)
    lse = np.where(safe, M + np.log(np.where(safe, den, 1.0)), -np.inf)
    return out, lse


def sparse_mla_split(q, kv_cache, kv_block_stride, block_table, seq_lens, query_start_loc, topk_idx, softmax_scale,
                     dv, block_size, num_splits, rows=None):
    """Split-KV sparse MLA followed by the merge; equals `sparse_mla`."""
    q = np.asarray(q, dtype=np.float64)
    T, H, dk = q.shape
    req, _ = token_positions(seq_lens, query_start_loc)
    out = np.full((T, H, dv), np.nan)
    lse = np.full((T, H), np.nan)
    for t in (range(T) if rows is None else rows):
        b = int(req[t])
        m, l, o = sparse_mla_partials(q[t], kv_cache, kv_block_stride, block_table[b], topk_idx[t], softmax_scale, dv,
                                      block_size, num_splits)
        out[t], lse[t] = merge_partials(m, l, o)
    return out, lse


def dense_mla(q_t, kv_rows, softmax_scale, dv):
    """Dense MLA attention of one token over all given rows (brute force):
    out[h] = sum_i softmax_i(scale * q[h] . kv[i]) kv[i, :dv]."""
    q_t = np.asarray(q_t, dtype=np.float64)
    kv_rows = np.asarray(kv_rows, dtype=np.float64)
    out = np.zeros((q_t.shape[0], dv))
    for h in range(q_t.shape[0]):
        s = [softmax_scale * float(np.dot(q_t[h], kv_rows[i])) for i in range(kv_rows.shape[0])]
        mx = max(s)
        e = [math.exp(v - mx) for v in s]
        z = sum(e)
        for i in range(kv_rows.shape[0]):
            out[h] += (e[i] / z) * kv_rows[i, :dv]
    return out


# ----------------------------------------------------------------------------
# fp8 latent KV cache (the FP8-KV variant of a3)
# ----------------------------------------------------------------------------

MLA_FP8_GROUP = 128


def mla_fp8_row_bytes(dk: int, dv: int) -> int:
    """Bytes of one token's row: dv e4m3 codes, dv/128 fp32 scales, and the
    dk - dv rope values in bf16 (656 at dk = 576, dv = 512)."""
    return dv + 4 * (dv // MLA_FP8_GROUP) + 2 * (dk - dv)


def _bf16_bits_of(values) -> np.ndarray:
    """bf16 bit patterns of values that are bf16 already (exact)."""
    v = np.asarray(values, dtype=np.float32)
    bits = v.view(np.uint32)
    assert np.all((bits & 0xFFFF) == 0), "rope values must be bf16 values"
    return (bits >> 16).astype(np.uint16)


def mla_fp8_quantize_rows(kv, dv):
    """Rows [n, dk] of bf16 latent values -> their fp8 cache rows [n, bytes].

    The latent part is quantised in groups of 128 with the rule of
    quantize_groups; the rope part keeps its bf16 bits.
    """
    kv = np.asarray(kv, dtype=np.float32)
    n, dk = kv.shape
    assert dv % MLA_FP8_GROUP == 0
    ng = dv // MLA_FP8_GROUP
    codes, scales = quantize_groups(kv[:, :dv].reshape(n, ng, MLA_FP8_GROUP))
    out = np.zeros((n, mla_fp8_row_bytes(dk, dv)), dtype=np.uint8)
    out[:, :dv] = codes.reshape(n, dv)
    out[:, dv:dv + 4 * ng] = np.ascontiguousarray(scales.astype(np.float32)).view(np.uint8).reshape(n, 4 * ng)
    out[:, dv + 4 * ng:] = np.ascontiguousarray(_bf16_bits_of(kv[:, dv:])).view(np.uint8).reshape(n, 2 * (dk - dv))
    return out


def mla_fp8_decode_rows(rows, dk, dv):
    """fp8 cache rows [..., bytes] -> latent rows [..., dk] in float64:
    e4m3(code) * scale of the code's group for the first dv values, the bf16
    rope values for the rest."""
    rows = np.asarray(rows, dtype=np.uint8)
    lead = rows.shape[:-1]
    r = rows.reshape(-1, rows.shape[-1])
    ng = dv // MLA_FP8_GROUP
    scales = np.ascontiguousarray(r[:, dv:dv + 4 * ng]).view(np.float32).astype(np.float64)  # [n, ng]
    lat = e4m3_decode(r[:, :dv]).reshape(-1, ng, MLA_FP8_GROUP) * scales[:, :, None]
    rope_bits = np.ascontiguousarray(r[:, dv + 4 * ng:dv + 4 * ng + 2 * (dk - dv)]).view(np.uint16)
    rope = (rope_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    out = np.concatenate([lat.reshape(-1, dv), rope], axis=1)
    return out.reshape(lead + (dk,))


def mla_kv_fp8_quant_and_cache(kv, kv_cache_fp8, block_table, seq_lens, query_start_loc, block_size, dv):
    """Producer side of the fp8 latent cache: a copy of the cache
    [num_blocks, block_size, row_bytes] with the T new tokens' latent rows
    kv [T, dk] (bf16 values) quantised by mla_fp8_quantize_rows and stored at
    the tokens' positions pos(t) (block block_table[b, pos // block_size],
    row pos % block_size), as indexer_k_quant_and_cache places keys. A position
    past the block-table row or a block id outside the cache skips the token.
    """
    kv = np.asarray(kv, dtype=np.float32)
    T, dk = kv.shape
    rows = mla_fp8_quantize_rows(kv, dv)
    out = np.array(kv_cache_fp8, dtype=np.uint8, copy=True)
    bt = np.asarray(block_table)
    req, pos = token_positions(seq_lens, query_start_loc)
    for t in range(T):
        b, p = int(req[t]), int(pos[t])
        if p < 0 or p >= bt.shape[1] * block_size:
            continue
        blk = int(bt[b, p // block_size])
        if blk < 0 or blk >= out.shape[0]:
            continue
        out[blk, p % block_size] = rows[t]
    return out


def mla_fp8_decode_cache(kv_cache_fp8, dk, dv):
    """The whole fp8 latent cache [num_blocks, block_size, bytes] decoded to
    float64 rows [num_blocks, block_size, dk]; a3 on the fp8 cache is
    sparse_mla / sparse_mla_split over these rows."""
    return mla_fp8_decode_rows(kv_cache_fp8, dk, dv)
