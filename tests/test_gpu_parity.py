"""GPU-vs-oracle parity of every step, through the C ABI (GB300 only)."""
import numpy as np
import pytest
import torch

from oracle import dsa_oracle as O
from deepseek_sparse_attention_fp8_gb300.inputs import bf16_bits_to_float, make_workload

from dsa_testlib import (check_attention, check_logits, check_topk_sets, oracle_attention, oracle_logits,
                         oracle_q_quant)

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from deepseek_sparse_attention_fp8_gb300 import api
    from deepseek_sparse_attention_fp8_gb300.step import DsaStep

# Small cases the oracle finishes in seconds, spanning several tiles and a
# ragged tail: (workload, overrides)
SMALL = {
    "tiny": ("tiny", {}),
    "decode_small": ("decode_b32_l8192", dict(B=3, lens=[1000, 2500, 777], index_topk=2048)),
    "decode_topk_small": ("decode_b32_l8192", dict(lens=[300, 129, 64, 4000], index_topk=256)),
    "mtp2_small": ("mixed_b64_mtp2", dict(lens=[1500, 2049, 3000, 65], index_topk=2048)),
    "prefill_small": ("prefill_4096_of_65536", dict(L=2300, q_len=260, index_topk=512)),
    "decode_bs128": ("decode_b32_l8192", dict(lens=[3000, 1111], index_topk=2048, block_size=128)),
}


def _wl(name):
    base, kw = SMALL[name]
    return make_workload(base, **kw)


@pytest.fixture(scope="module", params=sorted(SMALL))
def run_small(request):
    wl = _wl(request.param)
    step = DsaStep(wl)
    step.logits.fill_(float("nan"))  # dirty buffer: every entry must be rewritten
    step.run()
    torch.cuda.synchronize()
    return wl, step


def test_quant_q_bit_exact():
    for name in ("tiny", "decode_small"):
        wl = _wl(name)
        step = DsaStep(wl)
        q8, sq = api.dsa_quant_q(step.q_idx)
        codes, scales = oracle_q_quant(wl)
        assert np.array_equal(q8.cpu().numpy(), codes)
        assert np.array_equal(sq.cpu().numpy().view(np.uint32), scales.view(np.uint32))


def test_quant_q_bit_exact_across_magnitudes():
    """a0's division by the scale (a reciprocal with one FMA correction, or
    IEEE division when 1/scale is not normal) gives the correctly rounded
    quotient, so the codes equal the oracle's (IEEE fp32 division) bit for
    bit: rows of every bf16 magnitude from 1e-38 to 1e38, rows with
    power-of-two scales whose quotients hit e4m3 rounding midpoints exactly,
    signed zeros and all-zero rows."""
    rng = np.random.default_rng(11)
    T, Hi, Di = 512, 16, 128
    mag = np.exp(rng.uniform(-87, 87, (T, Hi, 1)))  # per-row magnitude
    x = (rng.standard_normal((T, Hi, Di)) * mag).astype(np.float32)
    # power-of-two scales: amax = 448 * 2^e, values on and next to e4m3 midpoints
    e = rng.integers(-20, 20, (T // 4, Hi, 1))
    mids = np.array([1.0625, 1.1875, 1.3125, 1.4375, 1.5625, 1.6875, 1.8125, 1.9375], np.float32)
    v = mids[rng.integers(0, 8, (T // 4, Hi, Di))] * np.exp2(rng.integers(-6, 8, (T // 4, Hi, Di)))
    v *= rng.choice([-1.0, 1.0], v.shape)
    v[..., 0] = 448.0
    x[: T // 4] = (v * np.exp2(e)).astype(np.float32)
    x[T // 4, 0] = 0.0
    x[T // 4, 1, ::2] = -0.0
    q = torch.from_numpy(x).to(torch.bfloat16).cuda()
    q8, sq = api.dsa_quant_q(q)
    codes, scales = O.quantize_groups(q.float().cpu().numpy())
    assert np.array_equal(sq.cpu().numpy().view(np.uint32), scales.view(np.uint32))
    got = q8.cpu().numpy()
    bad = np.argwhere(got != codes)
    assert bad.size == 0, f"{len(bad)} codes differ, first at {bad[0].tolist()}"


def test_indexer_logits(run_small):
    wl, step = run_small
    got = step.logits.cpu().numpy()
    ref = oracle_logits(wl)
    check_logits(got, ref, range(wl.T))
    assert int(step.dev_status.item()) == 0


HEAD_SHAPES = {
    "decode": ("decode_b32_l8192", dict(lens=[700, 1500, 333])),
    "mtp2": ("mixed_b64_mtp2", dict(lens=[900, 1300, 65])),
    "mtp3": ("mixed_b64_mtp2", dict(lens=[900, 1300, 65], q_len=3)),
    "prefill": ("prefill_4096_of_65536", dict(L=900, q_len=13)),
    "prefill14": ("prefill_4096_of_65536", dict(L=900, q_len=14)),
    "prefill15": ("prefill_4096_of_65536", dict(L=900, q_len=15)),
}


@pytest.mark.parametrize("Hi,Di", [(64, 128), (48, 128), (16, 128), (64, 64), (32, 64), (64, 32), (48, 32)])
@pytest.mark.parametrize("shape", sorted(HEAD_SHAPES))
def test_indexer_logits_head_shapes(shape, Hi, Di):
    """The logits kernel over indexer head counts (padded to multiples of 16)
    and head dims 32, 64 and 128 (TMA key pages for 128, 16-byte copies
    otherwise), for one, two, three and four tokens per CTA: two accumulators taken
    by the two epilogue warp groups in turn (whole tiles, or token pairs for
    three or four tokens of 64 heads), or one accumulator read by both groups
    when fewer than 64 heads of four tokens fill more than 128 columns; the
    13-, 14- and 15-token prefills end in a block of one, two and three
    tokens. Checked against the oracle; the top-k of the same logits is exact."""
    base, kw = HEAD_SHAPES[shape]
    wl = make_workload(base, Hi=Hi, Di=Di, index_topk=256, **kw)
    step = DsaStep(wl)
    step.logits.fill_(float("nan"))  # dirty buffer: every entry must be rewritten
    step.indexer()
    step.topk()
    torch.cuda.synchronize()
    assert int(step.dev_status.item()) == 0
    got = step.logits.cpu().numpy()
    check_logits(got, oracle_logits(wl), range(wl.T))
    idx = step.topk_idx.cpu().numpy()
    check_topk_sets(idx, O.topk(got, wl.seq_lens, wl.query_start_loc, wl.index_topk), range(wl.T))


RAGGED_STEPS = {
    # requests of one to three query tokens and very different lengths (one
    # token block each): chunks of the longest-work-first order of every kind
    "q3": dict(lens=[50, 5000, 700, 12000, 3, 2048], q_lens=[1, 3, 2, 3, 1, 2]),
    # up to six tokens (token blocks of four): second blocks of one or two
    # tokens, and rows with no second block
    "q6": dict(lens=[6, 9000, 130, 4100, 2500], q_lens=[6, 5, 1, 4, 2]),
}


@pytest.mark.parametrize("bs", [192, 256])
@pytest.mark.parametrize("base,kw", [("decode_b32_l8192", dict(lens=[3000, 1111, 200])),
                                     ("mixed_b64_mtp2", dict(lens=[900, 5000, 65], q_lens=[3, 2, 1]))],
                         ids=["decode", "ragged"])
def test_other_block_sizes(base, kw, bs):
    """Block sizes other than 64 and 128 (any multiple of 64 is accepted):
    the whole step against the oracle."""
    wl = make_workload(base, index_topk=512, block_size=bs, **kw)
    step = DsaStep(wl)
    step.logits.fill_(float("nan"))
    step.run()
    torch.cuda.synchronize()
    assert int(step.dev_status.item()) == 0
    got = step.logits.cpu().numpy()
    check_logits(got, oracle_logits(wl), range(wl.T))
    idx = step.topk_idx.cpu().numpy()
    check_topk_sets(idx, O.topk(got, wl.seq_lens, wl.query_start_loc, wl.index_topk), range(wl.T))
    ref, ref_lse = oracle_attention(wl, idx)
    check_attention(step.out.float().cpu().numpy(), ref, np.arange(wl.T), step.lse.cpu().numpy(), ref_lse)


@pytest.mark.parametrize("H", [16, 64, 100])
@pytest.mark.parametrize("splits", [1, 2])
def test_fewer_mla_heads(H, splits):
    """MLA head counts below the kernel's 128 rows (16 per GPU is DeepSeek's
    128 under 8-way tensor parallelism; 100 is not a multiple of 16): the
    attention against the oracle, split and unsplit."""
    wl = make_workload("decode_b32_l8192", H=H, index_topk=512, lens=[3000, 1111, 200])
    step = DsaStep(wl, num_kv_splits=splits)
    step.run()
    torch.cuda.synchronize()
    assert int(step.dev_status.item()) == 0
    idx = step.topk_idx.cpu().numpy()
    ref, ref_lse = oracle_attention(wl, idx)
    check_attention(step.out.float().cpu().numpy(), ref, np.arange(wl.T), step.lse.cpu().numpy(), ref_lse)


@pytest.mark.parametrize("kv_fp8", [False, True])
@pytest.mark.parametrize("H", [16, 100])
def test_fewer_mla_heads_prefill_entry(H, kv_fp8):
    """Fewer MLA heads through the prefill entry point (a batch of up to three
    query tokens per request) and over the fp8 latent cache."""
    wl = make_workload("mixed_b64_mtp2", H=H, index_topk=512, lens=[900, 5000, 65], q_lens=[3, 2, 1],
                       kv_fp8=kv_fp8)
    step = DsaStep(wl, kv_fp8=kv_fp8)
    assert step.prefill
    step.run()
    torch.cuda.synchronize()
    assert int(step.dev_status.item()) == 0
    idx = step.topk_idx.cpu().numpy()
    if kv_fp8:
        q = bf16_bits_to_float(wl.q)
        kv = O.mla_fp8_decode_cache(wl.kv_cache_fp8, wl.Dk, wl.Dv)
        ref, ref_lse = O.sparse_mla(q, kv, wl.kv_block_stride, wl.block_table, wl.seq_lens, wl.query_start_loc, idx,
                                    wl.softmax_scale, wl.Dv, wl.block_size)
    else:
        ref, ref_lse = oracle_attention(wl, idx)
    check_attention(step.out.float().cpu().numpy(), ref, np.arange(wl.T), step.lse.cpu().numpy(), ref_lse)


@pytest.mark.parametrize("K,splits", [(4096, 0), (6000, 3), (6000, 8)])
def test_index_topk_above_one_split(K, splits):
    """index_topk above the 2048 slots one split may cover (automatic and
    explicit split counts): the top-k exact and the attention against the
    oracle."""
    wl = make_workload("decode_b32_l8192", index_topk=K, lens=[9000, 5000, 700])
    step = DsaStep(wl, num_kv_splits=splits)
    step.run()
    torch.cuda.synchronize()
    assert int(step.dev_status.item()) == 0
    got = step.logits.cpu().numpy()
    idx = step.topk_idx.cpu().numpy()
    check_topk_sets(idx, O.topk(got, wl.seq_lens, wl.query_start_loc, wl.index_topk), range(wl.T))
    ref, ref_lse = oracle_attention(wl, idx)
    check_attention(step.out.float().cpu().numpy(), ref, np.arange(wl.T), step.lse.cpu().numpy(), ref_lse)


@pytest.mark.parametrize("K", [100, 2047])
def test_unpadded_logits_rows_and_odd_topk(K):
    """Logits rows exactly as long as the longest request (ld = 2999, not a
    multiple of the 128-key tile nor of 16 bytes) and an index_topk that is
    not a multiple of the 64-key attention tile: the whole step against the
    oracle, every logit written."""
    wl = make_workload("decode_b32_l8192", index_topk=K, lens=[2999, 1001, 77, 2100], ld_pad=1)
    assert wl.ld == 2999
    step = DsaStep(wl)
    step.logits.fill_(float("nan"))
    step.run()
    torch.cuda.synchronize()
    assert int(step.dev_status.item()) == 0
    got = step.logits.cpu().numpy()
    assert not np.isnan(got).any(), "logits left unwritten"
    check_logits(got, oracle_logits(wl), range(wl.T))
    idx = step.topk_idx.cpu().numpy()
    check_topk_sets(idx, O.topk(got, wl.seq_lens, wl.query_start_loc, wl.index_topk), range(wl.T))
    ref, ref_lse = oracle_attention(wl, idx)
    check_attention(step.out.float().cpu().numpy(), ref, np.arange(wl.T), step.lse.cpu().numpy(), ref_lse)


def test_more_requests_than_any_cta_has_threads():
    """1100 short requests (more than any kernel's threads per CTA, so the
    request lookups take their loop paths, the top-k's included): the whole
    step against the oracle
    on sampled rows, every logit checked."""
    rng = np.random.default_rng(11)
    lens = rng.integers(64, 700, 1100)
    wl = make_workload("decode_b32_l8192", index_topk=64, lens=lens.tolist())
    step = DsaStep(wl)
    step.logits.fill_(float("nan"))
    step.run()
    torch.cuda.synchronize()
    assert int(step.dev_status.item()) == 0
    rows = sorted(set(rng.integers(0, wl.T, 48).tolist()) | {0, wl.T - 1})
    got = step.logits.cpu().numpy()
    assert not np.isnan(got).any(), "logits left unwritten"
    check_logits(got, oracle_logits(wl, rows=rows), rows)
    idx = step.topk_idx.cpu().numpy()
    check_topk_sets(idx, O.topk(got, wl.seq_lens, wl.query_start_loc, wl.index_topk, rows=rows), rows)
    ref, ref_lse = oracle_attention(wl, idx, rows=rows)
    check_attention(step.out.float().cpu().numpy(), ref, np.array(rows), step.lse.cpu().numpy(), ref_lse)


@pytest.mark.parametrize("case", sorted(RAGGED_STEPS))
def test_ragged_multi_token_batch(case):
    """A batch of requests with different query counts and lengths (the
    indexer hands out its work longest first there): every logit against the
    oracle on a dirty buffer, the top-k of the same logits exact, and the
    attention against the oracle."""
    wl = make_workload("mixed_b64_mtp2", index_topk=512, **RAGGED_STEPS[case])
    step = DsaStep(wl)
    step.logits.fill_(float("nan"))
    step.run()
    torch.cuda.synchronize()
    assert int(step.dev_status.item()) == 0
    got = step.logits.cpu().numpy()
    check_logits(got, oracle_logits(wl), range(wl.T))
    idx = step.topk_idx.cpu().numpy()
    check_topk_sets(idx, O.topk(got, wl.seq_lens, wl.query_start_loc, wl.index_topk), range(wl.T))
    ref, ref_lse = oracle_attention(wl, idx)
    check_attention(step.out.float().cpu().numpy(), ref, np.arange(wl.T), step.lse.cpu().numpy(), ref_lse)


def test_topk_exact_on_same_logits(run_small):
    wl, step = run_small
    logits = step.logits.cpu().numpy()
    got = step.topk_idx.cpu().numpy()
    ref = O.topk(logits, wl.seq_lens, wl.query_start_loc, wl.index_topk)
    check_topk_sets(got, ref, range(wl.T))
    # the library lists positions in ascending order
    for t in range(wl.T):
        g = got[t][got[t] >= 0]
        assert np.all(np.diff(g) > 0)


def test_attention(run_small):
    wl, step = run_small
    idx = step.topk_idx.cpu().numpy()
    ref, ref_lse = oracle_attention(wl, idx)
    got = step.out.float().cpu().numpy()
    check_attention(got, ref, np.arange(wl.T), step.lse.cpu().numpy(), ref_lse)


def test_topk_ties_and_signed_zero():
    """Integer-valued logits with many ties, and -0.0/+0.0 ties, against a full sort."""
    T, ld, K = 6, 5000, 700
    rng = np.random.default_rng(3)
    vals = rng.integers(-3, 4, (T, ld)).astype(np.float32)
    vals[rng.random((T, ld)) < 0.3] = -0.0
    seq = np.array([5000, 4000, 1000, 700, 699, 3], np.int32)
    qsl = np.arange(T + 1, dtype=np.int32)
    dev = torch.from_numpy(vals).cuda()
    got = api.dsa_topk(dev, torch.from_numpy(seq).cuda(), torch.from_numpy(qsl).cuda(), K).cpu().numpy()
    ref = O.topk(vals, seq, qsl, K)
    check_topk_sets(got, ref, range(T))


@pytest.mark.parametrize("T,ld,K,dist", [(5, 8192, 2048, "normal"), (4, 32768, 2048, "normal"),
                                         (304, 36000, 2048, "normal"), (4, 8192, 100, "normal"),
                                         (4, 8192, 2048, "outliers"), (4, 8192, 2048, "constant_bins"),
                                         (2, 32768, 2048, "ties_across_parts")])
def test_topk_histogram_paths(T, ld, K, dist):
    """Logits of a smooth distribution (the threshold bin holds few keys), rows
    staged in shared memory and rows read from global memory (T >= 2 x SMs),
    a small k; two cases that force the refinement of the threshold bin:
    +-1e30 outliers inside the sampled range (one bin holds almost
    everything) and values of a few distinct levels; and equal values spread
    over all the CTAs of a row, ranked by position in the direct path."""
    rng = np.random.default_rng(T * 7 + ld + K)
    vals = rng.standard_normal((T, ld)).astype(np.float32)
    if dist == "outliers":
        vals[:, 0] = 1e30
        vals[:, 8] = -1e30
        vals[:, 16] = np.inf
    elif dist == "constant_bins":
        vals = np.round(vals * 2).astype(np.float32)
    elif dist == "ties_across_parts":  # ~80 copies of each of 400 levels, spread over the whole row
        vals = rng.integers(-200, 200, (T, ld)).astype(np.float32)
    seq = np.full(T, ld, np.int32)
    seq[-1] = ld - 777
    qsl = np.arange(T + 1, dtype=np.int32)
    got = api.dsa_topk(torch.from_numpy(vals).cuda(), torch.from_numpy(seq).cuda(), torch.from_numpy(qsl).cuda(),
                       K).cpu().numpy()
    ref = O.topk(vals, seq, qsl, K)
    check_topk_sets(got, ref, range(T))
    for t in range(T):
        g = got[t][got[t] >= 0]
        assert np.all(np.diff(g) > 0)


@pytest.mark.parametrize("ld", [40000, 131072])
def test_topk_long_rows_match_full_sort(ld):
    """Long rows shared by a cluster of CTAs, integer-valued (heavy ties
    across the CTAs of a row)."""
    T, K = 3, 2048
    rng = np.random.default_rng(ld)
    vals = rng.integers(-50, 50, (T, ld)).astype(np.float32)
    seq = np.array([ld, ld - 12345, 3000], np.int32)
    qsl = np.arange(T + 1, dtype=np.int32)
    got = api.dsa_topk(torch.from_numpy(vals).cuda(), torch.from_numpy(seq).cuda(), torch.from_numpy(qsl).cuda(),
                       K).cpu().numpy()
    ref = O.topk(vals, seq, qsl, K)
    check_topk_sets(got, ref, range(T))


def test_many_requests():
    """More requests than one CTA has threads: the kernels find a token's
    request by a search over query_start_loc instead of a single round of
    loads. Sampled tokens against the oracle."""
    lens = [64 + (i * 37) % 200 for i in range(450)]
    wl = make_workload("decode_b32_l8192", B=len(lens), lens=lens, index_topk=128)
    step = DsaStep(wl)
    step.logits.fill_(float("nan"))
    step.run()
    torch.cuda.synchronize()
    assert int(step.dev_status.item()) == 0
    rows = [0, 223, 449]
    logits = step.logits.cpu().numpy()
    check_logits(logits, oracle_logits(wl, rows=rows), rows)
    idx = step.topk_idx.cpu().numpy()
    check_topk_sets(idx, O.topk(logits, wl.seq_lens, wl.query_start_loc, wl.index_topk, rows=rows), rows)
    ref, ref_lse = oracle_attention(wl, idx, rows=rows)
    check_attention(step.out.float().cpu().numpy(), ref, np.array(rows), step.lse.cpu().numpy(), ref_lse)


@pytest.mark.parametrize("splits", [1, 2, 3, 4, 8, 32])
def test_attention_splits(splits):
    wl = _wl("decode_small")
    step = DsaStep(wl, num_kv_splits=splits)
    step.run()
    idx = step.topk_idx.cpu().numpy()
    ref, ref_lse = oracle_attention(wl, idx)
    check_attention(step.out.float().cpu().numpy(), ref, np.arange(wl.T), step.lse.cpu().numpy(), ref_lse)


def test_attention_empty_and_invalid_selection():
    wl = _wl("decode_small")
    step = DsaStep(wl, num_kv_splits=4)
    step.run()
    idx = step.topk_idx.clone()
    idx[0] = -1  # token 0: nothing selected -> out 0, lse -inf
    idx[1, :5] = torch.tensor([10**6, -7, 3, 3, 2499], dtype=torch.int32)  # out of range entries are skipped
    step.topk_idx.copy_(idx)
    step.dev_status.zero_()
    for splits in (1, 2, 4):
        step.splits = splits
        step.attention()
        torch.cuda.synchronize()
        out = step.out.float().cpu().numpy()
        lse = step.lse.cpu().numpy()
        assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
        st = int(step.dev_status.item())
        assert st & api.DSA_DEVERR_INDEX_OOB
        host_idx = idx.cpu().numpy()
        clean = host_idx.copy()
        clean[1][(clean[1] < -1) | (clean[1] >= 2500)] = -1
        ref, _ = oracle_attention(wl, clean, rows=[1])
        check_attention(out, ref, np.array([1]))


def test_bad_block_ids_are_masked_and_reported():
    wl = _wl("decode_small")
    step = DsaStep(wl)
    bt = step.block_table.clone()
    bt[0, 2] = wl.num_blocks + 5  # logical block 2 of request 0 -> out of range
    step.block_table.copy_(bt)
    step.dev_status.zero_()
    step.indexer()
    torch.cuda.synchronize()
    assert int(step.dev_status.item()) & api.DSA_DEVERR_BLOCK_OOB
    lg = step.logits.cpu().numpy()
    assert np.all(np.isneginf(lg[0, 128:192]))  # keys of the bad block
    assert np.all(np.isfinite(lg[0, :128]))


@pytest.mark.parametrize("shape,bs", [("decode", 64), ("mtp2", 64), ("prefill", 64), ("prefill", 128),
                                      ("prefill15", 128)])
def test_bad_block_ids_are_masked_in_every_epilogue_shape(shape, bs):
    """A bad block id in request 0's table masks exactly that block's keys to
    -inf for every token of the request, whichever epilogue shape the CTA takes
    (one token, two tokens, token pairs), and reports BLOCK_OOB; every other
    logit is bit-identical to the run with the clean table."""
    base, kw = HEAD_SHAPES[shape]
    wl = make_workload(base, index_topk=256, block_size=bs, **kw)
    step = DsaStep(wl)
    step.indexer()
    torch.cuda.synchronize()
    clean = step.logits.cpu().numpy().copy()
    bt = step.block_table.clone()
    lb = 128 // bs  # the logical block holding key 128
    bt[0, lb] = wl.num_blocks + 5
    step.block_table.copy_(bt)
    step.dev_status.zero_()
    step.logits.fill_(float("nan"))
    step.indexer()
    torch.cuda.synchronize()
    assert int(step.dev_status.item()) & api.DSA_DEVERR_BLOCK_OOB
    lg = step.logits.cpu().numpy()
    k0, k1 = lb * bs, (lb + 1) * bs
    rows0 = range(int(wl.query_start_loc[0]), int(wl.query_start_loc[1]))
    for t in rows0:
        assert np.all(np.isneginf(lg[t, k0:k1])), f"row {t}: bad block not masked"
    keep = np.ones_like(lg, dtype=bool)
    keep[list(rows0), k0:k1] = False
    assert np.array_equal(lg[keep].view(np.uint32), clean[keep].view(np.uint32))


def test_unused_block_table_entries_are_ignored():
    """Entries of a request's block-table row past its length may hold anything:
    the kernels may read them but never use them, so results are unchanged and
    no error is reported."""
    wl = _wl("decode_small")
    step = DsaStep(wl)
    step.run()
    torch.cuda.synchronize()
    ref = (step.logits.clone(), step.topk_idx.clone(), step.out.clone())
    bt = step.block_table.cpu().numpy().copy()
    garbage = np.array([wl.num_blocks + 7, 0, wl.num_blocks - 1, 2**30, -5], dtype=np.int32)
    touched = 0
    for b in range(bt.shape[0]):
        used = -(-int(wl.seq_lens[b]) // wl.block_size)
        n = bt.shape[1] - used
        bt[b, used:] = np.resize(garbage, n)
        touched += n
    assert touched > 0
    step.block_table.copy_(torch.from_numpy(bt))
    step.dev_status.zero_()
    step.logits.fill_(float("nan"))
    step.run()
    torch.cuda.synchronize()
    assert int(step.dev_status.item()) == 0
    assert torch.equal(step.logits, ref[0])
    assert torch.equal(step.topk_idx, ref[1])
    assert torch.equal(step.out, ref[2])


def _k_cache_case(Di, bs, seq, q_lens, seed):
    """A small paged key cache of random bytes (so untouched bytes are checked
    too), a permuted block table and new keys of varied magnitudes."""
    rng = np.random.default_rng(seed)
    B, T = len(seq), sum(q_lens)
    qsl = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    nblk = [max(1, -(-s // bs)) for s in seq]
    num_blocks = sum(nblk) + 5
    phys = rng.permutation(num_blocks).astype(np.int32)
    bt = np.full((B, max(nblk) + 1), -1, dtype=np.int32)
    cur = 0
    for b, n in enumerate(nblk):
        bt[b, :n] = phys[cur:cur + n]
        cur += n
    stride = bs * (Di + 4) + 16  # a padded page: bytes past the layout stay as they were
    cache = rng.integers(0, 256, (num_blocks, stride), dtype=np.uint8)
    kf = (rng.standard_normal((T, Di)) * rng.uniform(1e-2, 1e2, (T, 1))).astype(np.float32)
    kf[min(2, T - 1)] = 0.0  # amax == 0: scale 1, codes 0
    k = torch.from_numpy(kf).to(torch.bfloat16)
    return dict(k=k, cache=cache, bt=bt, seq=np.array(seq, dtype=np.int32), qsl=qsl, stride=stride)


def _run_k_cache(c, bs):
    dev = torch.device("cuda")
    cache = torch.from_numpy(c["cache"]).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    api.dsa_indexer_k_quant_and_cache(c["k"].to(dev), cache, torch.from_numpy(c["bt"]).to(dev),
                                      torch.from_numpy(c["seq"]).to(dev), torch.from_numpy(c["qsl"]).to(dev), bs,
                                      dev_status=status)
    torch.cuda.synchronize()
    want = O.indexer_k_quant_and_cache(c["k"].float().numpy(), c["cache"], c["stride"], c["bt"], c["seq"], c["qsl"], bs)
    return cache.cpu().numpy(), want, int(status.item())


@pytest.mark.parametrize("Di,bs", [(128, 64), (64, 128), (32, 64)])
def test_k_quant_and_cache_bit_exact(Di, bs):
    # decode, MTP pair, a 5-token chunk, and a request made of new tokens only
    c = _k_cache_case(Di, bs, seq=[70, 129, 200, 3], q_lens=[1, 2, 5, 3], seed=21 + Di)
    got, want, st = _run_k_cache(c, bs)
    assert st == 0
    assert np.array_equal(got, want)


def test_k_quant_and_cache_skips_and_reports_bad_targets():
    bs = 64
    c = _k_cache_case(128, bs, seq=[70, 129, 1], q_lens=[1, 2, 2], seed=5)
    c["bt"][1, 127 // bs] = int(c["bt"].max()) + 1000  # request 1's first new key -> block outside the cache
    got, want, st = _run_k_cache(c, bs)
    # request 2 has seq_len 1 < q_len 2: its first token has no position
    assert st & api.DSA_DEVERR_BLOCK_OOB and st & api.DSA_DEVERR_SEQ_LEN
    assert np.array_equal(got, want)  # the oracle skips the same tokens


def test_batch_invariance_with_fixed_splits():
    """With the split count fixed, a request's logits, top-k and attention
    output do not depend on which other requests share the batch (every
    kernel works on one token or one token block at a time)."""
    import dataclasses

    wl = _wl("mtp2_small")
    full = DsaStep(wl, num_kv_splits=2)
    full.run()
    torch.cuda.synchronize()
    qsl = wl.query_start_loc
    for b in (1, 3):
        t0, t1 = int(qsl[b]), int(qsl[b + 1])
        sub = dataclasses.replace(wl, B=1, T=t1 - t0, seq_lens=wl.seq_lens[b:b + 1].copy(),
                                  query_start_loc=np.array([0, t1 - t0], dtype=np.int32),
                                  block_table=wl.block_table[b:b + 1].copy(), q_idx=wl.q_idx[t0:t1].copy(),
                                  w=wl.w[t0:t1].copy(), q=wl.q[t0:t1].copy())
        one = DsaStep(sub, num_kv_splits=2)
        one.run()
        torch.cuda.synchronize()
        assert int(one.dev_status.item()) == 0
        assert torch.equal(one.logits, full.logits[t0:t1])
        assert torch.equal(one.topk_idx, full.topk_idx[t0:t1])
        assert torch.equal(one.out, full.out[t0:t1])
        assert torch.equal(one.lse, full.lse[t0:t1])


@pytest.mark.parametrize("case", ["sample_misses_the_tail", "ascending_row", "descending_row", "mixed_rows"])
def test_topk_candidate_lists_and_their_fallbacks(case):
    """Rows shared by a cluster that keep under 1/8 of their keys record
    candidates above a bin taken from 1024 samples. These rows defeat that
    estimate: the sampled positions hold the largest values, so the sampled
    bin admits fewer than k keys (the histogram is completed and every key
    visited); sorted rows put all candidates in a few warps' runs (their
    lists overflow); and a batch mixing such rows with smooth ones."""
    # 80 rows: two CTAs per row (32768 keys each, 1024-key runs per warp)
    T, ld, K = 80, 65536, 2048
    rng = np.random.default_rng(17)
    vals = rng.random((T, ld), dtype=np.float32)
    sampled = (np.arange(1024, dtype=np.int64) * ld) // 1024
    if case == "sample_misses_the_tail":
        vals[:, sampled] = 9.0 + rng.random((T, 1024), dtype=np.float32)
    elif case == "ascending_row":
        vals = np.tile(np.arange(ld, dtype=np.float32), (T, 1)) * 1e-3
    elif case == "descending_row":
        vals = np.tile(np.arange(ld, 0, -1, dtype=np.float32), (T, 1)) * 1e-3
    else:
        vals[0, sampled] = 9.0
        vals[2] = np.arange(ld, dtype=np.float32)
    seq = np.full(T, ld, np.int32)
    qsl = np.arange(T + 1, dtype=np.int32)
    got = api.dsa_topk(torch.from_numpy(vals).cuda(), torch.from_numpy(seq).cuda(), torch.from_numpy(qsl).cuda(),
                       K).cpu().numpy()
    ref = O.topk(vals, seq, qsl, K)
    check_topk_sets(got, ref, range(T))
    for t in range(T):
        g = got[t][got[t] >= 0]
        assert len(g) == K and np.all(np.diff(g) > 0)
