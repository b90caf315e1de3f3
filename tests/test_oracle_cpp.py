"""The plain C++ oracle (CPU) against the hand-worked examples and against the
numpy oracle on the pin workloads: a0 codes and scales bit for bit, a1 logits
within one fp32 rounding (both sum in double, in different orders), a2
selections exactly on the same logits, a3 outputs to 1e-12."""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from oracle import dsa_oracle as O  # noqa: E402
from oracle import ref as R  # noqa: E402
from deepseek_sparse_attention_fp8_gb300.inputs import bf16_bits_to_float, make_workload  # noqa: E402

HAND = json.load(open(os.path.join(ROOT, "tests", "golden", "hand_examples.json")))


def _bits(vals):
    import torch

    return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_quant_matches_hand_codes_and_all_magnitudes():
    ex = HAND["indexer"]
    codes, _ = R.quant_q(_bits(ex["q_heads"]))
    assert codes.tolist() == ex["q_codes_expected"]
    # every bf16 magnitude class: random rows spanning 1e-6 .. 1e4
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((300, 128)) * np.exp(rng.uniform(-14, 9, (300, 1)))).astype(np.float32)
    x[7] = 0.0
    bits = _bits(x)
    c_ref, s_ref = O.quantize_groups(bf16_bits_to_float(bits))
    c, s = R.quant_q(bits)
    assert np.array_equal(c, c_ref)
    assert np.array_equal(s.view(np.uint32), s_ref.view(np.uint32))


def test_topk_hand_example():
    ex = HAND["topk"]
    vals = np.array(ex["values"], dtype=np.float32)[None]
    sl = np.array([len(ex["values"])], dtype=np.int32)
    qsl = np.array([0, 1], dtype=np.int32)
    for k, key in ((4, "k4"), (5, "k5"), (9, "k9")):
        assert R.topk(vals, sl, qsl, k)[0].tolist() == ex[key]


def _close_logits(a, b):
    fin = np.isfinite(b)
    assert np.array_equal(np.isneginf(a), np.isneginf(b))
    ulp = np.spacing(np.abs(b[fin]).astype(np.float32))
    assert np.all(np.abs(a[fin] - b[fin]) <= ulp)


def test_step_matches_numpy_oracle_tiny():
    wl = make_workload("tiny")
    lg = R.indexer_logits(wl, threads=2)
    codes, scales = O.quantize_groups(bf16_bits_to_float(wl.q_idx))
    ref = O.indexer_logits(codes, scales, wl.w, wl.k_cache, wl.k_block_stride, wl.block_table, wl.seq_lens,
                           wl.query_start_loc, wl.block_size, wl.ld)
    _close_logits(lg, ref)
    idx = R.topk(ref, wl.seq_lens, wl.query_start_loc, wl.index_topk, threads=2)
    assert np.array_equal(idx, O.topk(ref, wl.seq_lens, wl.query_start_loc, wl.index_topk))
    out, lse = R.sparse_mla(wl, idx, threads=2)
    o_ref, l_ref = O.sparse_mla(bf16_bits_to_float(wl.q), bf16_bits_to_float(wl.kv_cache), wl.kv_block_stride,
                                wl.block_table, wl.seq_lens, wl.query_start_loc, idx, wl.softmax_scale, wl.Dv,
                                wl.block_size)
    assert np.allclose(out, o_ref, rtol=1e-12, atol=1e-14) and np.allclose(lse, l_ref, rtol=1e-12)


def test_step_matches_numpy_oracle_decode_rows():
    """Three tokens of a decode batch (ragged lengths, K = 2048), an MTP pair
    and a request with an empty selection."""
    wl = make_workload("decode_b32_l8192", B=3, lens=[1000, 2500, 777], index_topk=2048)
    rows = [0, 1, 2]
    lg = R.indexer_logits(wl, rows=rows, threads=3)
    codes, scales = O.quantize_groups(bf16_bits_to_float(wl.q_idx))
    ref = O.indexer_logits(codes, scales, wl.w, wl.k_cache, wl.k_block_stride, wl.block_table, wl.seq_lens,
                           wl.query_start_loc, wl.block_size, wl.ld, rows=rows)
    _close_logits(lg, ref)
    idx = R.topk(ref, wl.seq_lens, wl.query_start_loc, wl.index_topk, rows=rows)
    assert np.array_equal(idx, O.topk(ref, wl.seq_lens, wl.query_start_loc, wl.index_topk, rows=rows))
    idx[2] = -1  # an empty selection: out 0, lse -inf
    out, lse = R.sparse_mla(wl, idx, rows=rows, threads=3)
    o_ref, l_ref = O.sparse_mla(bf16_bits_to_float(wl.q), bf16_bits_to_float(wl.kv_cache), wl.kv_block_stride,
                                wl.block_table, wl.seq_lens, wl.query_start_loc, idx, wl.softmax_scale, wl.Dv,
                                wl.block_size, rows=rows)
    assert np.allclose(out[:2], o_ref[:2], rtol=1e-10, atol=1e-13)
    assert np.all(out[2] == 0) and np.all(np.isneginf(lse[2]))
    assert np.allclose(lse[:2], l_ref[:2], rtol=1e-12)


def test_mtp_pair_positions():
    wl = make_workload("mixed_b64_mtp2", lens=[300, 129], index_topk=64)
    lg = R.indexer_logits(wl)
    # token 0 of request 0 sits at position 298 (valid 299), token 1 at 299
    assert np.isneginf(lg[0, 299]) and np.isfinite(lg[0, 298]) and np.isfinite(lg[1, 299])
    codes, scales = O.quantize_groups(bf16_bits_to_float(wl.q_idx))
    ref = O.indexer_logits(codes, scales, wl.w, wl.k_cache, wl.k_block_stride, wl.block_table, wl.seq_lens,
                           wl.query_start_loc, wl.block_size, wl.ld)
    _close_logits(lg, ref)


def test_threads_do_not_change_results():
    wl = make_workload("tiny")
    a = R.step(wl, rows=[0], threads=1)
    b = R.step(wl, rows=[0], threads=4)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
