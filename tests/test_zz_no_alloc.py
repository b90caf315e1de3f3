"""The split-KV decode entry point that allocates nothing.

Some callers may not call cudaMalloc while they run the attention step:
serving runtimes that hand all device memory to their own allocator at
start-up and forbid later allocations, and host environments (plugins,
sandboxed runtimes) that may not create device allocations at all. For them
libdsa keeps the split partials in a fixed device scratch array instead of a
caller workspace. These checks call that
entry point through the C ABI twice in a row and compare each result with the
workspace-based entry point on the same inputs. This file sorts last so that a
stop-at-first-failure run has already run every other test.
"""
import numpy as np
import pytest
import torch

from deepseek_sparse_attention_fp8_gb300.inputs import make_workload

from dsa_testlib import ATT_MAX_ABS, ATT_MEAN_ABS

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from deepseek_sparse_attention_fp8_gb300 import api
    from deepseek_sparse_attention_fp8_gb300.step import DsaStep


def _compare(got, ref, got_lse, ref_lse):
    g = got.float().cpu().numpy()
    r = ref.float().cpu().numpy()
    err = np.abs(g - r)
    assert np.all(np.isfinite(g))
    assert err.max() <= ATT_MAX_ABS and err.mean() <= ATT_MEAN_ABS
    gl, rl = got_lse.cpu().numpy(), ref_lse.cpu().numpy()
    assert np.array_equal(np.isfinite(gl), np.isfinite(rl))
    fin = np.isfinite(rl)
    assert np.all(np.abs(gl[fin] - rl[fin]) <= 1e-3 * np.maximum(1.0, np.abs(rl[fin])))


@pytest.mark.parametrize("splits", [4, 0])
def test_fixed_scratch_matches_workspace_entry_point_twice(splits):
    wl = make_workload("decode_b32_l8192", B=3, lens=[1000, 2500, 777], index_topk=2048)
    step = DsaStep(wl, num_kv_splits=4)
    step.run()
    torch.cuda.synchronize()
    ref = torch.empty_like(step.out)
    ref_lse = torch.empty_like(step.lse)
    api.sparse_mla_decode(step.q, step.kv_cache, step.block_table, step.seq_lens, step.qsl, step.topk_idx,
                          wl.softmax_scale, wl.Dv, ref, ref_lse, num_kv_splits=splits or 4, workspace=step.ws_mla)
    for call in range(2):
        out = torch.full_like(step.out, float("nan"))
        lse = torch.full_like(step.lse, float("nan"))
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        api.sparse_mla_decode_fixed_scratch(step.q, step.kv_cache, step.block_table, step.seq_lens, step.qsl,
                                            step.topk_idx, wl.softmax_scale, wl.Dv, out, lse,
                                            num_kv_splits=splits, dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        _compare(out, ref, lse, ref_lse)


def test_fixed_scratch_rejects_requests_beyond_its_size():
    wl = make_workload("decode_b32_l8192", B=3, lens=[1000, 2500, 777], index_topk=2048)
    step = DsaStep(wl, num_kv_splits=1)
    limit = api.sparse_mla_fixed_scratch_bytes()
    T, H, Dv = 1024, 128, 512
    assert api.sparse_mla_workspace_size(T, H, Dv, 32) > limit
    q = torch.zeros((T, H, wl.Dk), dtype=torch.bfloat16, device="cuda")
    idx = torch.full((T, wl.index_topk), -1, dtype=torch.int32, device="cuda")
    out = torch.empty((T, H, Dv), dtype=torch.bfloat16, device="cuda")
    seq = torch.full((1,), 2048, dtype=torch.int32, device="cuda")
    qsl = torch.tensor([0, T], dtype=torch.int32, device="cuda")
    with pytest.raises(api.DsaError) as e:
        api.sparse_mla_decode_fixed_scratch(q, step.kv_cache, step.block_table[:1], seq, qsl, idx, wl.softmax_scale,
                                            Dv, out, num_kv_splits=32)
    assert e.value.status == api.DSA_ERR_WORKSPACE
    assert "fixed" in str(e.value)
