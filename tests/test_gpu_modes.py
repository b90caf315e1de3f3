"""GPU checks of the attention call's modes and input ranges, through the C ABI
(GB300 only): the batch-invariant split mode, one top-k selection shared by
several attention calls, and queries large enough that the scaled scores
reach hundreds of log2 units."""
import dataclasses

import numpy as np
import pytest
import torch

from deepseek_sparse_attention_fp8_gb300.inputs import make_workload

from dsa_testlib import check_attention, oracle_attention

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from deepseek_sparse_attention_fp8_gb300 import api
    from deepseek_sparse_attention_fp8_gb300.step import DsaStep


def _sub_batch(wl, reqs):
    """The workload restricted to the given requests (same caches)."""
    qsl = wl.query_start_loc
    toks = np.concatenate([np.arange(qsl[b], qsl[b + 1]) for b in reqs])
    lens = [int(qsl[b + 1] - qsl[b]) for b in reqs]
    return dataclasses.replace(wl, B=len(reqs), T=len(toks), seq_lens=wl.seq_lens[reqs].copy(),
                               query_start_loc=np.concatenate([[0], np.cumsum(lens)]).astype(np.int32),
                               block_table=wl.block_table[reqs].copy(), q_idx=wl.q_idx[toks].copy(),
                               w=wl.w[toks].copy(), q=wl.q[toks].copy()), toks


def test_batch_invariant_mode():
    """Under DSA_KV_SPLITS_BATCH_INVARIANT a request's logits, top-k, output
    and lse are bit-identical alone and inside two batches of other sizes,
    although the automatic split count differs between those batch sizes
    (vLLM PR #38476, Limitations: batch invariance forces the split count)."""
    lens = [300 + (i * 977) % 7000 for i in range(40)]
    wl = make_workload("decode_b32_l8192", lens=lens, index_topk=2048)
    target = 7
    batches = [[target], [3, 5, target, 11, 12], list(range(40))]
    auto = {len(r): api.sparse_mla_auto_splits(len(r), wl.H, wl.Dv, wl.index_topk) for r in batches}
    assert len(set(auto.values())) > 1, f"automatic split counts do not vary: {auto}"
    results = []
    for reqs in batches:
        sub, _ = _sub_batch(wl, reqs)
        step = DsaStep(sub, num_kv_splits=api.DSA_KV_SPLITS_BATCH_INVARIANT)
        assert step.splits == 1
        step.run()
        torch.cuda.synchronize()
        assert int(step.dev_status.item()) == 0
        t = reqs.index(target)
        results.append((step.logits[t].clone(), step.topk_idx[t].clone(), step.out[t].clone(), step.lse[t].clone()))
    for other in results[1:]:
        for a, b in zip(results[0], other):
            assert torch.equal(a, b)
    # the batch-invariant result is also the oracle's
    sub, _ = _sub_batch(wl, [target])
    ref, ref_lse = oracle_attention(sub, results[0][1].cpu().numpy()[None])
    check_attention(results[0][2].float().cpu().numpy()[None], ref, np.array([0]),
                    results[0][3].cpu().numpy()[None], ref_lse)


def test_batch_invariant_split_count_follows_index_topk():
    for K, want in ((64, 1), (2048, 1), (2049, 2), (4096, 2), (6000, 3)):
        for T in (1, 8, 300):
            assert api.sparse_mla_num_splits(T, 128, 512, K, api.DSA_KV_SPLITS_BATCH_INVARIANT) == want


def test_topk_selection_reused_by_a_second_layer():
    """One indexer + top-k selection serves two attention calls with different
    queries and latent caches (cross-layer reuse of the top-k indices, the
    IndexShare note of the vLLM PR #38476 review thread)."""
    wl = make_workload("decode_b32_l8192", B=3, lens=[1000, 2500, 777], index_topk=2048)
    step = DsaStep(wl, num_kv_splits=4)
    step.run()
    torch.cuda.synchronize()
    idx = step.topk_idx.clone()
    layer2 = make_workload("decode_b32_l8192", seed=99, B=3, lens=[1000, 2500, 777], index_topk=2048)
    # same paging, the second layer's own queries and cache contents
    layer2 = dataclasses.replace(layer2, block_table=wl.block_table, num_blocks=wl.num_blocks)
    q2 = torch.from_numpy(layer2.q.view(np.int16)).view(torch.bfloat16).cuda()
    kv2 = torch.from_numpy(layer2.kv_cache[:wl.num_blocks].view(np.int16)).view(torch.bfloat16).cuda()
    out2 = torch.empty_like(step.out)
    lse2 = torch.empty_like(step.lse)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for splits in (1, 2, 4):
        api.sparse_mla_decode(q2, kv2, step.block_table, step.seq_lens, step.qsl, idx, wl.softmax_scale, wl.Dv,
                              out2, lse2, num_kv_splits=splits, dev_status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(step.topk_idx, idx)  # the selection is only read
        l2 = dataclasses.replace(layer2, kv_cache=layer2.kv_cache[:wl.num_blocks])
        ref, ref_lse = oracle_attention(l2, idx.cpu().numpy())
        check_attention(out2.float().cpu().numpy(), ref, np.arange(wl.T), lse2.cpu().numpy(), ref_lse)
    # the first layer's own output is unchanged by the second call
    ref1, _ = oracle_attention(wl, idx.cpu().numpy())
    check_attention(step.out.float().cpu().numpy(), ref1, np.arange(wl.T))


@pytest.mark.parametrize("q_std", [30.0, 100.0, 1000.0])
@pytest.mark.parametrize("splits", [1, 4])
def test_attention_with_large_scores(q_std, splits):
    """Queries of standard deviation 30..1000 against KV of 0.5: the scaled
    scores have a standard deviation of 15..500 (natural-log units) and the
    half-scores of the two CTAs of a pair reach thousands in log2 units,
    cancelling in part. The pair exchanges its half-scores in fp32, so the
    output still meets the attention tolerance."""
    wl = make_workload("decode_b32_l8192", B=3, lens=[1000, 2500, 777], index_topk=2048, q_std=q_std)
    step = DsaStep(wl, num_kv_splits=splits)
    step.run()
    torch.cuda.synchronize()
    assert int(step.dev_status.item()) == 0
    idx = step.topk_idx.cpu().numpy()
    ref, ref_lse = oracle_attention(wl, idx)
    check_attention(step.out.float().cpu().numpy(), ref, np.arange(wl.T), step.lse.cpu().numpy(), ref_lse)


def test_split_count_from_the_environment(monkeypatch):
    """DSA_NUM_KV_SPLITS sets the split count of a step built with the
    automatic count; an explicit count keeps precedence."""
    wl = make_workload("decode_b32_l8192", B=3, lens=[1000, 2500, 777], index_topk=2048)
    monkeypatch.setenv("DSA_NUM_KV_SPLITS", "4")
    assert DsaStep(wl).splits == 4
    assert DsaStep(wl, num_kv_splits=2).splits == 2
    monkeypatch.delenv("DSA_NUM_KV_SPLITS")
    assert DsaStep(wl).splits == api.sparse_mla_num_splits(wl.T, wl.H, wl.Dv, wl.index_topk, 0)


def test_step_from_host_buffers_matches_the_resident_step():
    """run_host (indexer inputs copied first, the attention queries copied on a
    side stream during indexer and top-k, outputs read back) gives the same
    bits as the step over resident inputs, also for changed inputs."""
    wl = make_workload("decode_b32_l8192", B=3, lens=[1000, 2500, 777], index_topk=2048)
    step = DsaStep(wl)
    step.run()
    torch.cuda.synchronize()
    want = step.outputs.cpu()
    host_in = step.inputs.cpu().pin_memory()
    host_q = step.inputs_q.cpu().pin_memory()
    host_out = torch.empty_like(step.outputs, device="cpu").pin_memory()
    step.outputs.zero_()
    step.inputs_q.zero_()
    step.run_host(host_in, host_q, host_out)
    torch.cuda.synchronize()
    assert torch.equal(host_out, want)
    # new queries through the host path equal a resident step over the same queries
    host_q.view(torch.bfloat16).mul_(0.5)
    step.run_host(host_in, host_q, host_out)
    torch.cuda.synchronize()
    got = host_out.clone()
    step.inputs_q.copy_(host_q)
    step.run()
    torch.cuda.synchronize()
    assert torch.equal(got, step.outputs.cpu())
    assert int(step.dev_status.item()) == 0


def test_nvtx_ranges_leave_results_unchanged(monkeypatch):
    """DSA_NVTX=1 wraps each call in an NVTX range; the step's results are the
    same bits as without."""
    wl = make_workload("decode_b32_l8192", B=3, lens=[1000, 2500, 777], index_topk=2048)
    plain = DsaStep(wl)
    plain.run()
    monkeypatch.setenv("DSA_NVTX", "1")
    marked = DsaStep(wl)
    assert marked.nvtx
    marked.run()
    torch.cuda.synchronize()
    assert torch.equal(plain.outputs, marked.outputs) and torch.equal(plain.topk_idx, marked.topk_idx)
