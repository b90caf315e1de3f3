"""GPU parity of the fp8 latent cache through the C ABI (GB300 only): sparse
MLA over the fp8 cache against the oracle's attention over the decoded rows,
and the cache writer bit-exact against the oracle's."""
import numpy as np
import pytest
import torch

from oracle import dsa_oracle as O
from deepseek_sparse_attention_fp8_gb300.inputs import bf16_bits_to_float, make_workload

from dsa_testlib import check_attention

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from deepseek_sparse_attention_fp8_gb300 import api
    from deepseek_sparse_attention_fp8_gb300.step import DsaStep

CASES = {
    "decode_small": ("decode_b32_l8192", dict(B=3, lens=[1000, 2500, 777], index_topk=2048)),
    "mtp2_small": ("mixed_b64_mtp2", dict(lens=[1500, 2049, 3000, 65], index_topk=2048)),
    "prefill_small": ("prefill_4096_of_65536", dict(L=2300, q_len=260, index_topk=512)),
    "decode_topk_small": ("decode_b32_l8192", dict(lens=[300, 129, 64, 4000], index_topk=256)),
    "ragged_q3": ("mixed_b64_mtp2", dict(lens=[50, 5000, 700, 12000, 3, 2048], q_lens=[1, 3, 2, 3, 1, 2],
                                         index_topk=512)),
    "bs192": ("decode_b32_l8192", dict(lens=[3000, 1111, 200], index_topk=512, block_size=192)),
}


def oracle_fp8_attention(wl, idx, rows=None, splits=1):
    q = bf16_bits_to_float(wl.q)
    kv = O.mla_fp8_decode_cache(wl.kv_cache_fp8, wl.Dk, wl.Dv)
    if splits == 1:
        return O.sparse_mla(q, kv, wl.kv_block_stride, wl.block_table, wl.seq_lens, wl.query_start_loc, idx,
                            wl.softmax_scale, wl.Dv, wl.block_size, rows=rows)
    return O.sparse_mla_split(q, kv, wl.kv_block_stride, wl.block_table, wl.seq_lens, wl.query_start_loc, idx,
                              wl.softmax_scale, wl.Dv, wl.block_size, splits, rows=rows)


@pytest.mark.parametrize("name", sorted(CASES))
def test_fp8_cache_attention(name):
    base, kw = CASES[name]
    wl = make_workload(base, kv_fp8=True, **kw)
    step = DsaStep(wl, kv_fp8=True)
    step.run()
    torch.cuda.synchronize()
    assert int(step.dev_status.item()) == 0
    idx = step.topk_idx.cpu().numpy()
    ref, ref_lse = oracle_fp8_attention(wl, idx)
    check_attention(step.out.float().cpu().numpy(), ref, np.arange(wl.T), step.lse.cpu().numpy(), ref_lse)


@pytest.mark.parametrize("splits", [1, 2, 4, 8])
def test_fp8_cache_splits(splits):
    base, kw = CASES["decode_small"]
    wl = make_workload(base, kv_fp8=True, **kw)
    step = DsaStep(wl, kv_fp8=True, num_kv_splits=splits)
    step.run()
    torch.cuda.synchronize()
    assert int(step.dev_status.item()) == 0
    idx = step.topk_idx.cpu().numpy()
    ref, ref_lse = oracle_fp8_attention(wl, idx)
    check_attention(step.out.float().cpu().numpy(), ref, np.arange(wl.T), step.lse.cpu().numpy(), ref_lse)


def test_fp8_cache_empty_and_invalid_selection():
    base, kw = CASES["decode_small"]
    wl = make_workload(base, kv_fp8=True, **kw)
    step = DsaStep(wl, kv_fp8=True, num_kv_splits=4)
    step.run()
    idx = step.topk_idx.clone()
    idx[0] = -1  # token 0: nothing selected -> out 0, lse -inf
    idx[1, :5] = torch.tensor([10**6, -7, 3, 3, 2499], dtype=torch.int32)
    step.topk_idx.copy_(idx)
    step.dev_status.zero_()
    for splits in (1, 2, 4):
        step.splits = splits
        step.attention()
        torch.cuda.synchronize()
        out = step.out.float().cpu().numpy()
        assert np.all(out[0] == 0) and np.all(np.isneginf(step.lse.cpu().numpy()[0]))
        assert int(step.dev_status.item()) & api.DSA_DEVERR_INDEX_OOB
        clean = idx.cpu().numpy().copy()
        clean[1][(clean[1] < -1) | (clean[1] >= 2500)] = -1
        ref, _ = oracle_fp8_attention(wl, clean, rows=[1])
        check_attention(out, ref, np.array([1]))


def _fp8_cache_case(seq, q_lens, seed, bs=64):
    rng = np.random.default_rng(seed)
    B, T = len(seq), sum(q_lens)
    qsl = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    nblk = [max(1, -(-s // bs)) for s in seq]
    num_blocks = sum(nblk) + 3
    phys = rng.permutation(num_blocks).astype(np.int32)
    bt = np.full((B, max(nblk) + 1), -1, dtype=np.int32)
    cur = 0
    for b, n in enumerate(nblk):
        bt[b, :n] = phys[cur:cur + n]
        cur += n
    cache = rng.integers(0, 256, (num_blocks, bs, 656), dtype=np.uint8)  # untouched rows must stay as they are
    kf = (rng.standard_normal((T, 576)) * rng.uniform(1e-3, 1e2, (T, 1))).astype(np.float32)
    kf[min(1, T - 1), 128:256] = 0.0  # an all-zero group: scale 1, codes 0
    kv = torch.from_numpy(kf).to(torch.bfloat16)
    return dict(kv=kv, cache=cache, bt=bt, seq=np.array(seq, dtype=np.int32), qsl=qsl)


def _run_fp8_cache(c, bs=64):
    dev = torch.device("cuda")
    cache = torch.from_numpy(c["cache"]).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    api.dsa_mla_kv_fp8_quant_and_cache(c["kv"].to(dev), cache, torch.from_numpy(c["bt"]).to(dev),
                                       torch.from_numpy(c["seq"]).to(dev), torch.from_numpy(c["qsl"]).to(dev), bs,
                                       dev_status=status)
    torch.cuda.synchronize()
    want = O.mla_kv_fp8_quant_and_cache(c["kv"].float().numpy(), c["cache"], c["bt"], c["seq"], c["qsl"], bs, 512)
    return cache.cpu().numpy(), want, int(status.item())


def test_fp8_cache_writer_bit_exact():
    # decode, an MTP pair, a 5-token chunk, and a request made of new tokens only
    c = _fp8_cache_case(seq=[70, 129, 200, 3], q_lens=[1, 2, 5, 3], seed=31)
    got, want, st = _run_fp8_cache(c)
    assert st == 0
    assert np.array_equal(got, want)


def test_fp8_cache_writer_skips_and_reports_bad_targets():
    c = _fp8_cache_case(seq=[70, 129, 1], q_lens=[1, 2, 2], seed=6)
    c["bt"][1, 127 // 64] = int(c["bt"].max()) + 1000  # request 1's first new token -> block outside the cache
    got, want, st = _run_fp8_cache(c)
    assert st & api.DSA_DEVERR_BLOCK_OOB and st & api.DSA_DEVERR_SEQ_LEN
    assert np.array_equal(got, want)


def test_fp8_cache_written_by_the_writer_feeds_attention():
    """Rows stored by the writer are read back by the attention kernel: a
    cache filled through dsa_mla_kv_fp8_quant_and_cache equals the
    generator's fp8 cache of the same bf16 rows, byte for byte."""
    base, kw = CASES["decode_small"]
    wl = make_workload(base, kv_fp8=True, **kw)
    dev = torch.device("cuda")
    rows = torch.from_numpy(wl.kv_cache.reshape(-1, wl.Dk).view(np.int16)).view(torch.bfloat16).to(dev)
    nb, bs = wl.num_blocks, wl.block_size
    # every physical row written once: one request per block, block_size new tokens each
    bt = torch.arange(nb, dtype=torch.int32, device=dev)[:, None]
    seq = torch.full((nb,), bs, dtype=torch.int32, device=dev)
    qsl = torch.arange(0, (nb + 1) * bs, bs, dtype=torch.int32, device=dev)
    cache = torch.zeros((nb, bs, 656), dtype=torch.uint8, device=dev)
    api.dsa_mla_kv_fp8_quant_and_cache(rows, cache, bt, seq, qsl, bs)
    torch.cuda.synchronize()
    assert np.array_equal(cache.cpu().numpy(), wl.kv_cache_fp8)
