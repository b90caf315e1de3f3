"""Pins for the CPU oracle: closed forms, hand-derived examples, library
routines and invariants that fix what each oracle function must return.
CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import logsumexp, softmax

from oracle import dsa_oracle as O

with open(os.path.join(os.path.dirname(__file__), "golden", "hand_examples.json")) as _f:
    GOLDEN = json.load(_f)


def _f(v):
    return float("-inf") if v == "-inf" else float(v)


# --------------------------------------------------------------------- e4m3
def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.e4m3_decode(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))


def test_e4m3_decode_closed_forms():
    d = O.e4m3_decode(np.array([0x7E, 0x08, 0x01, 0x38, 0x40, 0xB8, 0x07, 0x7F, 0xFF, 0x80, 0x00], dtype=np.uint8))
    assert d[0] == 448.0 and d[1] == 2.0**-6 and d[2] == 2.0**-9 and d[3] == 1.0
    assert d[4] == 2.0 and d[5] == -1.0 and d[6] == 7 * 2.0**-9
    assert np.isnan(d[7]) and np.isnan(d[8])
    assert d[9] == 0.0 and np.signbit(d[9]) and d[10] == 0.0 and not np.signbit(d[10])


def test_e4m3_encode_roundtrip_all_codes():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    assert np.array_equal(O.e4m3_encode(O.e4m3_decode(codes)), codes)


def test_e4m3_encode_ties_and_random_match_torch_rne():
    vals = O.e4m3_decode(np.arange(0, 0x7E, dtype=np.uint8))
    mids = (vals[:-1] + vals[1:]) / 2.0
    rng = np.random.default_rng(5)
    rnd = rng.uniform(-448, 448, 20000)
    small = rng.uniform(-0.05, 0.05, 20000)
    x = np.concatenate([mids, -mids, np.nextafter(mids, 1e9), np.nextafter(mids, -1e9), rnd, small]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = O.e4m3_encode(x.astype(np.float64))
    assert np.array_equal(got, ref)
    # exact midpoints go to the even mantissa
    for m, lo in zip(mids[:20], range(20)):
        c = int(O.e4m3_encode(np.array([m]))[0])
        assert c % 2 == 0 and c in (lo, lo + 1)


def test_e4m3_encode_saturates():
    got = O.e4m3_encode(np.array([448.0, 449.0, 463.9, 464.0, 500.0, 1e30, -1e30, -460.0]))
    assert list(got) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE]


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(5000) * 10.0 ** rng.integers(-30, 30, 5000), [1.0 + 2**-8, 1.0 + 3 * 2**-9]])
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).to(torch.float64).numpy()
    # torch rounds from fp32; compare on values exactly representable in fp32
    got = O.bf16_round(x.astype(np.float32).astype(np.float64))
    assert np.array_equal(got, ref)


# --------------------------------------------------------------------- a0
def test_quantize_hand_example():
    g = GOLDEN["indexer"]
    codes, scales = O.quantize_groups(np.array(g["q_heads"], dtype=np.float32))
    assert codes.tolist() == g["q_codes_expected"]
    assert scales[0] == np.float32(2.0) / np.float32(448.0)
    assert scales[1] == np.float32(4.0) / np.float32(448.0)


def test_quantize_power_of_two_scale_is_exact():
    vals = O.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))
    row = np.concatenate([vals, -vals[:10]]) * 2.0**-5  # amax = 448 * 2^-5
    codes, scale = O.quantize_groups(row[None, :].astype(np.float32))
    assert scale[0] == np.float32(2.0**-5)
    assert np.array_equal(O.e4m3_decode(codes[0]) * float(scale[0]), row)


def test_quantize_zero_row():
    codes, scale = O.quantize_groups(np.zeros((2, 8), dtype=np.float32))
    assert np.all(codes == 0) and np.all(scale == 1.0)


def test_quantize_error_within_format_bound():
    rng = np.random.default_rng(7)
    x = rng.standard_normal((64, 128)).astype(np.float32)
    codes, scale = O.quantize_groups(x)
    dq = O.e4m3_decode(codes) * scale[:, None].astype(np.float64)
    # half a unit in the last place: 2^-4 relative for normals, 2^-10 * scale
    # absolute in the subnormal range; plus the fp32 rounding of x/scale
    bound = np.maximum(np.abs(x) * 2.0**-4, 2.0**-10 * scale[:, None]) * (1 + 1e-6)
    assert np.all(np.abs(dq - x) <= bound)
    assert np.all(np.abs(O.e4m3_decode(codes)).max(axis=1) == 448.0)


# --------------------------------------------------------------------- a1
def _pack_index_cache(codes_rows, scales, block_size, head_dim, table):
    """Lay keys out in the paged indexer format (values then scales per block)."""
    n = len(codes_rows)
    nblk = max(table) + 1
    stride = block_size * (head_dim + 4)
    cache = np.zeros((nblk, stride), dtype=np.uint8)
    for s in range(n):
        blk, off = table[s // block_size], s % block_size
        cache[blk, off * head_dim:(off + 1) * head_dim] = codes_rows[s]
        cache[blk, block_size * head_dim + off * 4: block_size * head_dim + off * 4 + 4] = \
            np.array([scales[s]], dtype=np.float32).view(np.uint8)
    return cache, stride


def _golden_indexer(q_len):
    g = GOLDEN["indexer"]
    codes, qs = O.quantize_groups(np.array(g["q_heads"], dtype=np.float32))
    cache, stride = _pack_index_cache(np.array(g["key_codes"], dtype=np.uint8), g["key_scales"], g["block_size"],
                                      g["head_dim"], [0])
    T = q_len
    qc = np.repeat(codes[None], T, axis=0)
    qsc = np.repeat(qs[None], T, axis=0)
    w = np.repeat(np.array(g["w"], dtype=np.float32)[None], T, axis=0)
    return O.indexer_logits(qc, qsc, w, cache, stride, np.array([[0]]), np.array([g["seq_len"]]), np.array([0, T]),
                            g["block_size"], g["ld"])


@pytest.mark.parametrize("q_len", [1, 2])
def test_indexer_hand_example(q_len):
    g = GOLDEN["indexer"]
    got = _golden_indexer(q_len)
    exp = np.array([[_f(v) for v in row] for row in g["logits_q_len%d" % q_len]])
    fin = np.isfinite(exp)
    assert np.array_equal(np.isinf(got), ~fin)
    assert np.allclose(got[fin], exp[fin], rtol=1e-6, atol=0)


def test_indexer_unit_keys_pick_one_coordinate():
    # one head, w = 1, key s = e_{s mod D} with scale sk: logit = sk * ReLU(dq[d])
    D, n, bs = 8, 16, 4
    rng = np.random.default_rng(11)
    q = rng.standard_normal((1, 1, D)).astype(np.float32)
    qc, qs = O.quantize_groups(q)
    codes = np.zeros((n, D), dtype=np.uint8)
    for s in range(n):
        codes[s, s % D] = 0x38  # 1.0
    sk = rng.uniform(0.5, 2.0, n).astype(np.float32)
    cache, stride = _pack_index_cache(codes, sk, bs, D, [3, 0, 2, 1])
    out = O.indexer_logits(qc, qs, np.ones((1, 1), np.float32), cache, stride, np.array([[3, 0, 2, 1]]),
                           np.array([n]), np.array([0, 1]), bs, n)
    dq = O.e4m3_decode(qc[0, 0]) * float(qs[0, 0])
    exp = np.array([float(sk[s]) * max(0.0, dq[s % D]) for s in range(n)], dtype=np.float32)
    assert np.array_equal(out[0], exp)


def test_indexer_negative_dots_give_zero_and_scale_is_linear():
    D, n, bs = 16, 8, 8
    qc = np.full((1, 2, D), 0x38, dtype=np.uint8)  # q = +1 everywhere
    qs = np.ones((1, 2), np.float32)
    codes = np.full((n, D), 0xB8, dtype=np.uint8)  # k = -1 everywhere
    cache, stride = _pack_index_cache(codes, np.ones(n, np.float32), bs, D, [0])
    w = np.array([[1.0, -3.0]], np.float32)
    out = O.indexer_logits(qc, qs, w, cache, stride, np.array([[0]]), np.array([n]), np.array([0, 1]), bs, n)
    assert np.all(out[0] == 0.0)
    rng = np.random.default_rng(2)
    codes = O.e4m3_encode(rng.uniform(-8, 8, (n, D)))
    qc = O.e4m3_encode(rng.uniform(-8, 8, (1, 2, D)))
    c1, _ = _pack_index_cache(codes, np.ones(n, np.float32), bs, D, [0])
    c2, _ = _pack_index_cache(codes, np.full(n, 2.0, np.float32), bs, D, [0])
    o1 = O.indexer_logits(qc, qs, w, c1, stride, np.array([[0]]), np.array([n]), np.array([0, 1]), bs, n)
    o2 = O.indexer_logits(qc, qs, w, c2, stride, np.array([[0]]), np.array([n]), np.array([0, 1]), bs, n)
    assert np.array_equal(o2, 2 * o1) and np.any(o1 != 0)


def test_indexer_brute_force_and_folded_algebra():
    """Per-element loops (scale inside the dot) agree with the oracle, and with
    the folded form sk * sum_h (w*sq) ReLU(sum_d code_q*code_k) that the GPU
    kernel evaluates (exact because both scales are positive)."""
    rng = np.random.default_rng(4)
    Hi, D, n, bs = 3, 8, 10, 4
    q = rng.standard_normal((2, Hi, D)).astype(np.float32)
    qc, qs = O.quantize_groups(q)
    kc, ks = O.quantize_groups(rng.standard_normal((n, D)).astype(np.float32))
    w = rng.standard_normal((2, Hi)).astype(np.float32)
    table = [1, 0, 2]
    cache, stride = _pack_index_cache(kc, ks, bs, D, table)
    out = O.indexer_logits(qc, qs, w, cache, stride, np.array([table]), np.array([n]), np.array([0, 2]), bs, 12)
    dec = O.e4m3_decode
    for t in range(2):
        valid = n - 2 + t + 1
        for s in range(12):
            if s >= valid:
                assert out[t, s] == -np.inf
                continue
            direct = 0.0
            folded = 0.0
            for h in range(Hi):
                dot = sum((dec(qc[t, h, d]) * qs[t, h]) * (dec(kc[s, d]) * ks[s]) for d in range(D))
                direct += w[t, h] * max(0.0, dot)
                raw = sum(dec(qc[t, h, d]) * dec(kc[s, d]) for d in range(D))
                folded += (float(w[t, h]) * float(qs[t, h])) * max(0.0, raw)
            folded *= float(ks[s])
            assert abs(out[t, s] - direct) <= 1e-6 * (1 + abs(direct))
            assert abs(folded - direct) <= 1e-9 * (1 + abs(direct))


def test_indexer_paging_is_transparent():
    rng = np.random.default_rng(9)
    D, n, bs = 8, 20, 4
    kc, ks = O.quantize_groups(rng.standard_normal((n, D)).astype(np.float32))
    qc, qs = O.quantize_groups(rng.standard_normal((1, 2, D)).astype(np.float32))
    w = rng.standard_normal((1, 2)).astype(np.float32)
    ident = list(range(5))
    perm = [4, 2, 0, 3, 1]
    c1, st = _pack_index_cache(kc, ks, bs, D, ident)
    c2, _ = _pack_index_cache(kc, ks, bs, D, perm)
    args = (np.array([n]), np.array([0, 1]), bs, 24)
    o1 = O.indexer_logits(qc, qs, w, c1, st, np.array([ident]), *args)
    o2 = O.indexer_logits(qc, qs, w, c2, st, np.array([perm]), *args)
    assert np.array_equal(o1, o2)


# ------------------------------------------------- producer: key cache writes
def test_k_quant_and_cache_worked_example():
    """Request of 130 keys whose last 3 are new; block size 64, table [4, 0, 2]:
    positions 127, 128, 129 -> block 0 row 63, block 2 rows 0 and 1."""
    bs, Di = 64, 128
    stride = bs * (Di + 4)
    cache = np.full((5, stride), 0xA5, dtype=np.uint8)
    k = np.random.default_rng(3).standard_normal((3, Di)).astype(np.float32)
    out = O.indexer_k_quant_and_cache(k, cache, stride, np.array([[4, 0, 2]]), np.array([130]), np.array([0, 3]), bs)
    codes, scales = O.quantize_groups(k)
    want = cache.copy()
    for (blk, row), t in (((0, 63), 0), ((2, 0), 1), ((2, 1), 2)):
        want[blk, row * Di:(row + 1) * Di] = codes[t]
        want[blk, bs * Di + 4 * row: bs * Di + 4 * row + 4] = np.frombuffer(np.float32(scales[t]).tobytes(), np.uint8)
    assert np.array_equal(out, want)
    assert np.array_equal(out[[1, 3, 4]], cache[[1, 3, 4]])  # other blocks untouched


def test_k_quant_and_cache_fills_the_page_the_indexer_reads():
    """Writing every key of two prompts (seq_len == q_len) gives the cache the
    test's own packer lays out by key index, so the indexer reads them back."""
    rng = np.random.default_rng(11)
    bs, Di = 4, 8
    lens = [9, 6]
    tables = [[3, 0, 5], [1, 4]]
    keys = [rng.standard_normal((n, Di)).astype(np.float32) for n in lens]
    stride = bs * (Di + 4)
    bt = np.full((2, 3), -1, dtype=np.int32)
    for b, tb in enumerate(tables):
        bt[b, :len(tb)] = tb
    qsl = np.array([0, lens[0], lens[0] + lens[1]])
    out = O.indexer_k_quant_and_cache(np.concatenate(keys), np.zeros((6, stride), np.uint8), stride, bt, np.array(lens),
                                      qsl, bs)
    want = np.zeros((6, stride), np.uint8)
    for b in range(2):
        kc, ks = O.quantize_groups(keys[b])
        packed, _ = _pack_index_cache(kc, ks, bs, Di, tables[b])
        used = sorted(set(tables[b]))
        want[used] = packed[used]
    assert np.array_equal(out, want)


def test_k_quant_matches_the_torch_cast_recipe():
    """The key rule: scale = fp32(amax / 448) and codes = e4m3fn cast of
    fp32(x / scale), the recipe of PyTorch's own float8 cast."""
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((256, 128)) * rng.uniform(1e-3, 1e3, (256, 1))).astype(np.float32)
    codes, scales = O.quantize_groups(x)
    amax = np.abs(x).max(axis=1)
    s_ref = (amax / np.float32(448.0)).astype(np.float32)
    c_ref = torch.from_numpy((x / s_ref[:, None]).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(scales, s_ref)
    assert np.array_equal(codes, c_ref)


# --------------------------------------------------------------------- a2
def test_topk_hand_example():
    g = GOLDEN["topk"]
    v = np.array(g["values"], np.float32)
    for k in (4, 5, 9):
        assert O.topk_row(v, k).tolist() == g["k%d" % k]


def test_topk_matches_full_sort_with_ties():
    rng = np.random.default_rng(1)
    for trial in range(200):
        n = int(rng.integers(1, 60))
        k = int(rng.integers(1, 70))
        v = rng.integers(-3, 4, n).astype(np.float32)
        v[rng.random(n) < 0.2] = -0.0
        ref = sorted(range(n), key=lambda i: (-float(v[i]), i))[:k]
        got = O.topk_row(v, k)
        assert got[: len(ref)].tolist() == ref
        assert np.all(got[len(ref):] == -1)


def test_topk_rows_use_causal_valid_length():
    logits = np.array([[5, 4, -np.inf, -np.inf], [1, 2, 3, -np.inf]], np.float32)
    out = O.topk(logits, np.array([3]), np.array([0, 2]), 3)
    assert out[0].tolist() == [0, 1, -1]
    assert out[1].tolist() == [2, 1, 0]


def test_topk_chunked_candidates_are_exact():
    """The global top-K equals the top-K of the union of per-chunk top-K
    (vLLM PR #38476 review thread, chunked top-k argument)."""
    rng = np.random.default_rng(8)
    for trial in range(20):
        n, K, chunk = 3000, 100, 256
        v = rng.integers(-20, 20, n).astype(np.float32)
        glob = O.topk_row(v, K)
        cand = []
        for c0 in range(0, n, chunk):
            loc = O.topk_row(v[c0:c0 + chunk], K)
            cand += [c0 + i for i in loc if i >= 0]
        cand = np.array(sorted(cand))
        sub = O.topk_row(v[cand], K)
        assert np.array_equal(cand[sub], glob)


# --------------------------------------------------------------------- a3/a4
def _one_request_cache(rows, bs, table):
    n, dk = rows.shape
    nblk = max(table) + 1
    cache = np.full((nblk, bs, dk), np.nan)
    for i in range(n):
        cache[table[i // bs], i % bs] = rows[i]
    return cache, bs * dk


def test_attention_hand_example():
    g = GOLDEN["attention"]
    rows = np.array(g["rows"])
    cache, st = _one_request_cache(rows, 2, [0])
    out, lse = O.sparse_mla(np.array([g["q"]]), cache, st, np.array([[0]]), np.array([2]), np.array([0, 1]),
                            np.array([[1, 0]]), g["softmax_scale"], g["dv"], 2)
    assert np.allclose(out[0], g["out"], rtol=1e-15, atol=0)
    assert np.allclose(lse[0], g["lse"], rtol=1e-15, atol=0)


def _rand_case(rng, n=40, H=3, dk=12, dv=8, bs=4):
    rows = rng.standard_normal((n, dk))
    nblk_used = (n + bs - 1) // bs
    table = list(rng.permutation(nblk_used + 3)[:nblk_used])
    cache, st = _one_request_cache(rows, bs, table)  # unused blocks hold NaN
    q = rng.standard_normal((1, H, dk))
    return rows, cache, st, np.array([table]), q


def test_attention_full_selection_equals_dense_brute_force():
    rng = np.random.default_rng(12)
    rows, cache, st, bt, q = _rand_case(rng)
    n = rows.shape[0]
    idx = np.full((1, 64), -1, np.int32)
    idx[0, :n] = rng.permutation(n)
    out, lse = O.sparse_mla(q, cache, st, bt, np.array([n]), np.array([0, 1]), idx, 0.3, 8, 4)
    dense = O.dense_mla(q[0], rows, 0.3, 8)
    assert np.allclose(out[0], dense, rtol=1e-12, atol=1e-14)
    s = 0.3 * q[0] @ rows.T
    assert np.allclose(out[0], softmax(s, axis=1) @ rows[:, :8], rtol=1e-12, atol=1e-14)
    assert np.allclose(lse[0], logsumexp(s, axis=1), rtol=1e-13)


def test_attention_closed_forms():
    rng = np.random.default_rng(13)
    rows, cache, st, bt, q = _rand_case(rng)
    n = rows.shape[0]
    sel = [3, 17, 5, 30]
    idx = np.array([sel + [-1] * 4], np.int32)
    args = (cache, st, bt, np.array([n]), np.array([0, 1]))
    # q = 0: uniform weights -> mean of the selected value rows, lse = log(count)
    out, lse = O.sparse_mla(np.zeros_like(q), *args, idx, 0.5, 8, 4)
    assert np.allclose(out[0], np.tile(rows[sel, :8].mean(axis=0), (3, 1)), rtol=1e-13)
    assert np.allclose(lse[0], math.log(4))
    # one selected row: its value vector exactly
    out, _ = O.sparse_mla(q, *args, np.array([[-1, 9, -1]], np.int32), 0.5, 8, 4)
    assert np.array_equal(out[0], np.tile(rows[9, :8], (3, 1)))
    # a constant-1 value column reads back 1 (weights sum to 1)
    rows2 = rows.copy()
    rows2[:, 2] = 1.0
    cache2, _ = _one_request_cache(rows2, 4, list(bt[0]))
    out, _ = O.sparse_mla(q, cache2, st, bt, np.array([n]), np.array([0, 1]), idx, 0.5, 8, 4)
    assert np.allclose(out[0][:, 2], 1.0, rtol=0, atol=1e-14)
    # permuting the selection changes nothing
    o1, _ = O.sparse_mla(q, *args, idx, 0.5, 8, 4)
    o2, _ = O.sparse_mla(q, *args, np.array([[-1, 30, 5, -1, 3, -1, 17, -1]], np.int32), 0.5, 8, 4)
    assert np.allclose(o1, o2, rtol=1e-13, atol=1e-15)
    assert np.all(np.isfinite(o1))  # NaN-poisoned unused blocks never leak


def test_attention_empty_selection():
    rng = np.random.default_rng(14)
    rows, cache, st, bt, q = _rand_case(rng)
    out, lse = O.sparse_mla(q, cache, st, bt, np.array([40]), np.array([0, 1]), np.full((1, 8), -1, np.int32), 1.0, 8,
                            4)
    assert np.all(out == 0) and np.all(lse == -np.inf)


@pytest.mark.parametrize("splits", [1, 2, 3, 8, 32])
def test_split_merge_equals_single_pass(splits):
    rng = np.random.default_rng(15 + splits)
    rows, cache, st, bt, q = _rand_case(rng, n=40)
    idx = np.full((1, 48), -1, np.int32)
    idx[0, :40] = rng.permutation(40)
    idx[0] = idx[0, rng.permutation(48)]  # -1 slots scattered, some splits all -1
    args = (cache, st, bt, np.array([40]), np.array([0, 1]), idx, 0.4, 8, 4)
    o1, l1 = O.sparse_mla(q, *args)
    o2, l2 = O.sparse_mla_split(q, *args, splits)
    assert np.allclose(o1, o2, rtol=1e-12, atol=1e-14)
    assert np.allclose(l1, l2, rtol=1e-12, atol=1e-14)


def test_split_all_masked_partial_uses_sentinel():
    rng = np.random.default_rng(21)
    rows, cache, st, bt, q = _rand_case(rng, n=8)
    idx = np.array([0, 1, 2, 3, -1, -1, -1, -1], np.int32)
    m, l, o = O.sparse_mla_partials(q[0], cache, st, bt[0], idx, 1.0, 8, 4, 2)
    assert np.all(m[1] == O.NEG_SENTINEL) and np.all(l[1] == 0) and np.all(o[1] == 0)
    assert np.all(np.isfinite(m)) and np.all(np.isfinite(o))
    out, lse = O.merge_partials(m, l, o)
    ref, rl = O.sparse_mla(q, cache, st, bt, np.array([8]), np.array([0, 1]), idx[None], 1.0, 8, 4)
    assert np.allclose(out, ref[0], rtol=1e-13) and np.allclose(lse, rl[0], rtol=1e-13)
    # every split empty: output 0, lse -inf
    m = np.full((3, 2), O.NEG_SENTINEL)
    out, lse = O.merge_partials(m, np.zeros((3, 2)), np.zeros((3, 2, 4)))
    assert np.all(out == 0) and np.all(lse == -np.inf)


def test_split_bounds_cover_every_slot_once():
    for k in (1, 7, 64, 2048):
        for s in (1, 2, 3, 8, 32):
            b = O.split_bounds(k, s)
            covered = [i for lo, hi in b for i in range(lo, hi)]
            assert covered == list(range(k))
