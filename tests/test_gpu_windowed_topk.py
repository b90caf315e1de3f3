"""GPU checks of the windowed indexer + top-k (dsa_indexer_topk), through the
C ABI (GB300 only). Its logits are those of dsa_indexer_logits key for key,
so its selection must equal dsa_topk's on those logits exactly (same
positions, same order) whatever the window, and the oracle's top-k of the
same logits (vLLM PR #38476 review thread: the global top-k is recovered
exactly from per-window top-k candidates)."""
import numpy as np
import pytest
import torch

from oracle import dsa_oracle as O
from deepseek_sparse_attention_fp8_gb300.inputs import make_workload

from dsa_testlib import check_logits, check_topk_sets, oracle_logits

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from deepseek_sparse_attention_fp8_gb300 import api
    from deepseek_sparse_attention_fp8_gb300.step import DsaStep

CASES = {
    "decode_small": ("decode_b32_l8192", dict(B=3, lens=[1000, 2500, 777], index_topk=2048)),
    "decode_topk256": ("decode_b32_l8192", dict(lens=[300, 129, 64, 4000, 2600], index_topk=256)),
    "mtp2_small": ("mixed_b64_mtp2", dict(lens=[1500, 2049, 3000, 65], index_topk=2048)),
    "prefill_small": ("prefill_4096_of_65536", dict(L=2300, q_len=260, index_topk=512)),
    "ragged_q3": ("mixed_b64_mtp2", dict(lens=[50, 5000, 700, 12000, 3, 2048], q_lens=[1, 3, 2, 3, 1, 2],
                                         index_topk=512)),
}


def _windowed(step, wl, window):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = api.dsa_indexer_topk(step.q_idx, step.w, step.k_cache, step.block_table, step.seq_lens, step.qsl,
                               wl.block_size, wl.max_q_len, wl.ld, window, wl.index_topk, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return got


@pytest.mark.parametrize("name", sorted(CASES))
@pytest.mark.parametrize("window", [0, 128, 512, 1024, 4096])
def test_windowed_topk_equals_plain_topk(name, window):
    base, kw = CASES[name]
    wl = make_workload(base, **kw)
    step = DsaStep(wl)
    step.run()
    torch.cuda.synchronize()
    got = _windowed(step, wl, window)
    assert torch.equal(got, step.topk_idx)
    # and the oracle's selection on those logits
    logits = step.logits.cpu().numpy()
    ref = O.topk(logits, wl.seq_lens, wl.query_start_loc, wl.index_topk)
    check_topk_sets(got.cpu().numpy(), ref, range(wl.T))


def test_windowed_logits_match_the_oracle():
    """The logits behind the windowed selection: the plain call's logits
    against the oracle (the windowed call computes each key the same way)."""
    base, kw = CASES["decode_small"]
    wl = make_workload(base, **kw)
    step = DsaStep(wl)
    step.indexer()
    torch.cuda.synchronize()
    check_logits(step.logits.cpu().numpy(), oracle_logits(wl), range(wl.T))


def test_windowed_topk_long_rows():
    """decode_b8_l131072 at full size with 32768-key windows (4 windows, a
    [8, 32768] logits buffer instead of [8, 131072]): the same selection as
    the plain path."""
    wl = make_workload("decode_b8_l131072")
    step = DsaStep(wl, num_kv_splits=8)
    step.run()
    torch.cuda.synchronize()
    got = _windowed(step, wl, 32768)
    assert torch.equal(got, step.topk_idx)
    need = api.dsa_indexer_topk_workspace_size(wl.T, wl.ld, 32768, wl.index_topk)
    assert need < wl.T * wl.ld * 4  # bounded by the window, not the context


def test_windowed_topk_rejects_bad_windows():
    base, kw = CASES["decode_small"]
    wl = make_workload(base, **kw)
    step = DsaStep(wl)
    with pytest.raises(api.DsaError) as e:
        _windowed(step, wl, 100)
    assert e.value.status == api.DSA_ERR_INVALID_ARG
