"""Shared helpers for the parity tests: oracle-side evaluation of a workload
and the comparison rules (tolerances as stated for the DSA step)."""
from __future__ import annotations

import numpy as np

from deepseek_sparse_attention_fp8_gb300.inputs import bf16_bits_to_float
from oracle import dsa_oracle as O

# Indexer logits: max relative error 2e-2. A relative error is meaningless on
# logits near zero (signed head weights cancel), so the reference magnitude is
# floored at 1e-2 of the row's rms.
LOGIT_RTOL = 2e-2
LOGIT_FLOOR = 1e-2
# Attention output (bf16): max abs 2e-2, mean abs 2e-3. At index_topk = 2048
# the outputs are small (|out| ~ 1e-2), so the error relative to the output's
# rms is bounded too: bf16 output rounding alone gives ~2e-3, and the kernel's
# bf16 softmax weights add about as much again.
ATT_MAX_ABS = 2e-2
ATT_MEAN_ABS = 2e-3
ATT_RMS_REL = 1e-2
# lse: the kernel's softmax normaliser sums the bf16-rounded weights that its
# PV product uses, each within a relative 2^-9 of the exact weight, so ln l
# may be off by up to ln(1 + 2^-9) = 1.95e-3 (reached when a row has a few
# dominant keys); beyond |lse| = 2.5 the bound is 1e-3 relative.
LSE_ABS = 2.5e-3
LSE_REL = 1e-3


def oracle_q_quant(wl):
    return O.quantize_groups(bf16_bits_to_float(wl.q_idx))


def oracle_logits(wl, rows=None):
    codes, scales = oracle_q_quant(wl)
    return O.indexer_logits(codes, scales, wl.w, wl.k_cache, wl.k_block_stride, wl.block_table, wl.seq_lens,
                            wl.query_start_loc, wl.block_size, wl.ld, rows=rows)


def check_logits(got, ref, rows):
    """Exact -inf on masked positions, relative error on the rest."""
    worst = 0.0
    for t in rows:
        g, r = got[t].astype(np.float64), ref[t].astype(np.float64)
        masked = np.isneginf(r)
        assert np.array_equal(np.isneginf(g), masked), f"row {t}: -inf pattern differs"
        v = ~masked
        if not v.any():
            continue
        assert np.all(np.isfinite(g[v])), f"row {t}: non-finite logits"
        rms = np.sqrt(np.mean(r[v] ** 2))
        denom = np.maximum(np.abs(r[v]), LOGIT_FLOOR * rms)
        err = np.max(np.abs(g[v] - r[v]) / denom)
        worst = max(worst, err)
        assert err <= LOGIT_RTOL, f"row {t}: relative error {err:.3g}"
    return worst


def check_topk_sets(got, ref, rows):
    for t in rows:
        g = np.sort(got[t][got[t] >= 0])
        r = np.sort(ref[t][ref[t] >= 0])
        assert np.array_equal(g, r), f"row {t}: top-k sets differ ({len(np.setdiff1d(g, r))} entries)"
        assert np.sum(got[t] >= 0) == np.sum(ref[t] >= 0)
        assert np.all(got[t][len(g):] == -1), f"row {t}: -1 padding missing"


def oracle_attention(wl, topk_idx, rows=None, splits=1):
    q = bf16_bits_to_float(wl.q)
    kv = bf16_bits_to_float(wl.kv_cache)
    if splits == 1:
        return O.sparse_mla(q, kv, wl.kv_block_stride, wl.block_table, wl.seq_lens, wl.query_start_loc, topk_idx,
                            wl.softmax_scale, wl.Dv, wl.block_size, rows=rows)
    return O.sparse_mla_split(q, kv, wl.kv_block_stride, wl.block_table, wl.seq_lens, wl.query_start_loc, topk_idx,
                              wl.softmax_scale, wl.Dv, wl.block_size, splits, rows=rows)


def check_attention(got, ref, rows, got_lse=None, ref_lse=None):
    """Max and mean absolute error and rms(g - r) / rms(r) within bounds;
    returns the three."""
    g = got[rows].astype(np.float64)
    r = ref[rows]
    assert np.all(np.isfinite(g)), "non-finite attention output"
    err = np.abs(g - r)
    assert err.max() <= ATT_MAX_ABS, f"max abs error {err.max():.3g}"
    assert err.mean() <= ATT_MEAN_ABS, f"mean abs error {err.mean():.3g}"
    rms_r = np.sqrt(np.mean(r ** 2))
    rms_rel = float(np.sqrt(np.mean(err ** 2)) / rms_r) if rms_r > 0 else 0.0
    if rms_r > 0:
        assert rms_rel <= ATT_RMS_REL, f"rms(g - r) / rms(r) = {rms_rel:.3g}"
    if got_lse is not None:
        gl, rl = got_lse[rows].astype(np.float64), ref_lse[rows]
        fin = np.isfinite(rl)
        assert np.array_equal(np.isfinite(gl), fin)
        bound = np.maximum(LSE_ABS, LSE_REL * np.abs(rl[fin]))
        assert np.all(np.abs(gl[fin] - rl[fin]) <= bound), \
            f"lse error {np.max(np.abs(gl[fin] - rl[fin]) - bound):.3g} over the bound"
    return float(err.max()), float(err.mean()), rms_rel
