"""Host-side pieces of bench.py that need no GPU: the algorithmic byte counts
behind the roofline, the bounded oracle sample and the host description."""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from deepseek_sparse_attention_fp8_gb300.inputs import make_workload  # noqa: E402


def test_decode_bytes_match_the_workload_arithmetic():
    """decode_b32_l8192: 32 requests of 8192 keys, one new token each."""
    wl = make_workload("decode_b32_l8192")
    alg = bench.algorithmic_bytes(wl)
    T, L, K = 32, 8192, 2048
    # key pages (128 code bytes + a 4-byte scale per key), q_idx bf16, w fp32, logits written
    assert alg["indexer"] == T * L * 132 + T * 64 * 128 * 2 + T * 64 * 4 + T * L * 4
    # logits read, indices written
    assert alg["topk"] == T * L * 4 + T * K * 4
    # K gathered 576-dim bf16 rows per token, q, out, indices, lse
    assert alg["attention"] == T * K * 576 * 2 + T * 128 * 576 * 2 + T * 128 * 512 * 2 + T * K * 4 + T * 128 * 4
    assert alg["flops_attention"] == T * K * 128 * (2 * 576 + 2 * 512)


def test_oracle_sample_is_bounded_and_evenly_spaced():
    rows = bench.oracle_rows(4096, 3)
    assert rows == [0, 1365, 2730]
    assert bench.oracle_rows(32, 1000) == list(range(32))  # never more than the workload
    assert bench.oracle_rows(32, 0) == [0]                  # at least one token
    r = bench.oracle_rows(4096, 100)
    assert len(r) == 100 and r == sorted(set(r)) and np.all(np.diff(r) >= 40)


def test_cpu_model_names_the_host():
    name = bench.cpu_model()
    assert isinstance(name, str) and name.strip()


def test_config_index_selects_the_workload(monkeypatch):
    from deepseek_sparse_attention_fp8_gb300.inputs import CONFIG_WORKLOADS, WORKLOADS

    assert set(CONFIG_WORKLOADS) == set(WORKLOADS)
    for n, name in enumerate(CONFIG_WORKLOADS):
        monkeypatch.setattr(sys, "argv", ["bench.py", "--config", str(n), "--seed", "7"])
        args = bench.parse()
        assert args.workload == name and args.seed == 7
    monkeypatch.setattr(sys, "argv", ["bench.py", "--config", "5"])
    try:
        bench.parse()
    except SystemExit:
        pass
    else:
        raise AssertionError("an out-of-range --config must be refused")
