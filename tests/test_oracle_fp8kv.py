"""Pins of the oracle's fp8 latent cache (CPU): the row layout and its
quantisation against a hand-derived row, the placement of new tokens against
hand-derived blocks and rows, the e4m3 rounding bound, PyTorch's own float8
cast, and sparse attention over decoded rows against brute force."""
import json
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from oracle import dsa_oracle as O  # noqa: E402

GOLD = json.load(open(os.path.join(ROOT, "tests", "golden", "mla_fp8_row.json")))


def _bf16(x):
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).float().numpy()


def _hand_row():
    dk, dv = GOLD["dk"], GOLD["dv"]
    row = np.zeros(dk, dtype=np.float32)
    row[:len(GOLD["latent_first"])] = GOLD["latent_first"]
    row[dv:] = GOLD["rope"]
    row[6] = -0.0
    return row


def test_row_bytes_of_the_workload_shape():
    assert O.mla_fp8_row_bytes(576, 512) == 656
    assert O.mla_fp8_row_bytes(GOLD["dk"], GOLD["dv"]) == GOLD["row_bytes"]


def test_hand_derived_row():
    dk, dv = GOLD["dk"], GOLD["dv"]
    got = O.mla_fp8_quantize_rows(_hand_row()[None], dv)[0]
    n = len(GOLD["codes_first"])
    assert got.shape == (GOLD["row_bytes"],)
    assert list(got[:n]) == GOLD["codes_first"]
    assert not got[n:dv].any()
    assert list(got[dv:dv + 8]) == GOLD["scale_bytes"]
    assert list(got[dv + 8:]) == GOLD["rope_bytes"]
    dec = O.mla_fp8_decode_rows(got[None], dk, dv)[0]
    want = np.zeros(dk)
    want[:n] = GOLD["decoded_first"]
    want[dv:] = GOLD["rope"]
    assert np.array_equal(dec, want)
    assert np.signbit(dec[6])  # -0.0 keeps its sign through the code 0x80


def test_codes_match_pytorch_float8_cast():
    """The codes of each group are PyTorch's float8_e4m3fn cast (round to
    nearest even) of fp32(x / scale), scale = fp32(amax / 448)."""
    rng = np.random.default_rng(5)
    kv = _bf16(rng.standard_normal((64, 576)) * rng.uniform(1e-3, 30, (64, 1)))
    kv[3, :128] = 0.0  # an all-zero group
    rows = O.mla_fp8_quantize_rows(kv, 512)
    g = kv[:, :512].reshape(64, 4, 128).astype(np.float32)
    amax = np.abs(g).max(axis=-1)
    scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
    want = torch.from_numpy((g / scale[..., None]).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8)
    assert np.array_equal(rows[:, :512], want.numpy().reshape(64, 512))
    assert np.array_equal(rows[:, 512:528].view(np.float32), scale)


def test_round_trip_within_the_e4m3_bound():
    """Decoded latent values lie within half an e4m3 ulp of the input: 2^-4 of
    the value in the normal range, 2^-10 of the group scale below it; rope
    values come back exactly."""
    rng = np.random.default_rng(9)
    kv = _bf16(rng.standard_normal((200, 576)) * 0.5)
    dec = O.mla_fp8_decode_rows(O.mla_fp8_quantize_rows(kv, 512), 576, 512)
    scale = np.abs(kv[:, :512].reshape(200, 4, 128)).max(axis=-1) / 448.0
    bound = np.maximum(np.abs(kv[:, :512]) * 2.0 ** -4, np.repeat(scale, 128, axis=1) * 2.0 ** -10) * (1 + 1e-6)
    assert np.all(np.abs(dec[:, :512] - kv[:, :512]) <= bound)
    assert np.array_equal(dec[:, 512:], kv[:, 512:].astype(np.float64))


def test_new_tokens_land_at_hand_derived_blocks_and_rows():
    """Request 0: seq_len 70, one new token -> position 69 = block_table[0][1]
    (block 1), row 5. Request 1: seq_len 65, two new tokens -> positions 63 and
    64 = block 0 row 63 and block 2 row 0. Every other byte is unchanged."""
    bs, dk, dv = 64, 576, 512
    rng = np.random.default_rng(2)
    nb = 4
    cache = rng.integers(0, 256, (nb, bs, 656), dtype=np.uint8)
    bt = np.array([[3, 1], [0, 2]], dtype=np.int32)
    seq = np.array([70, 65], dtype=np.int32)
    qsl = np.array([0, 1, 3], dtype=np.int32)
    kv = _bf16(rng.standard_normal((3, dk)))
    out = O.mla_kv_fp8_quant_and_cache(kv, cache, bt, seq, qsl, bs, dv)
    rows = O.mla_fp8_quantize_rows(kv, dv)
    want = cache.copy()
    want[1, 5] = rows[0]
    want[0, 63] = rows[1]
    want[2, 0] = rows[2]
    assert np.array_equal(out, want)


def test_sparse_attention_over_decoded_rows_is_dense_brute_force():
    """index_topk >= valid: sparse MLA over the decoded fp8 cache equals dense
    MLA (a plain loop) over the decoded rows of every position."""
    rng = np.random.default_rng(4)
    bs, dk, dv, H, L = 64, 576, 512, 3, 100
    kv = _bf16(rng.standard_normal((2 * bs, dk)) * 0.5)
    cache = O.mla_fp8_quantize_rows(kv, dv).reshape(2, bs, 656)
    bt = np.array([[1, 0]], dtype=np.int32)
    dec = O.mla_fp8_decode_cache(cache, dk, dv)
    q = _bf16(rng.standard_normal((1, H, dk)))
    idx = np.arange(128, dtype=np.int32)[None]
    idx[0, L:] = -1
    out, _ = O.sparse_mla(q, dec, bs * dk, bt, np.array([L]), np.array([0, 1]), idx, 1 / 24, dv, bs)
    rows = [dec[bt[0, s // bs], s % bs] for s in range(L)]
    assert np.allclose(out[0], O.dense_mla(q[0], np.array(rows), 1 / 24, dv), rtol=1e-12, atol=1e-14)
