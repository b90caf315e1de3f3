"""Benchmark of one DSA step (indexer logits -> top-k -> sparse MLA + merge).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME | --config N] [--splits S] [--seed S] [--kv-fp8]

Default workload: decode_b32_l8192 (32 requests x 1 query token, 8192 cached
tokens each, 64x128 fp8 indexer, top-2048, 128-head 576/512 MLA). Prints one
JSON line. `value` is decode tokens/s over the device-timed step with inputs
resident in HBM and L2 flushed between steps; `e2e` repeats it through the
public API with per-step inputs copied from pinned host memory (the attention
queries on a side stream while the indexer and top-k run) and the output read
back. Times are medians over the timed steps (p10 / p90 beside them).
`kernels` times each phase alone (medians; their sum must stay within 1.3x of
the step median), `roofline` relates the dominant one to its peak (HBM at
decode, the e4m3 or bf16 tensor peak at prefill), `workloads` repeats the
measurement for the other four workloads (the long-context decode at 1, 8 and
32 KV splits), `producer` times the key-cache writer (outside the step) and
`cpu_baseline` the oracle on a bounded sample of the workload's tokens.
Under torchrun every rank runs an independent replica (the step has no
exchange), ranks are timed with a barrier and the max is taken.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse-MLA decode tokens/s + indexer/attention HBM GB/s vs roofline (1 GB300)"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode_b32_l8192")
    ap.add_argument("--config", type=int, default=None, metavar="N",
                    help="workload by configuration index (0 tiny, 1 decode_b32_l8192, 2 decode_b8_l131072, "
                         "3 prefill_4096_of_65536, 4 mixed_b64_mtp2); overrides --workload")
    ap.add_argument("--seed", type=int, default=None, help="input seed (default: the workload's own)")
    ap.add_argument("--splits", type=int, default=0)
    ap.add_argument("--kv-fp8", action="store_true", help="run the step over the fp8 latent cache")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-clock-load", action="store_true", help="skip the one-second load before the timed steps")
    ap.add_argument("--no-other-workloads", action="store_true",
                    help="time only --workload (by default the other workloads are timed too and reported under "
                         "'workloads')")
    ap.add_argument("--oracle-seconds", type=int, default=0, metavar="N",
                    help="print the oracle's seconds for N evenly spaced query tokens of the workload and exit (no GPU)")
    args = ap.parse_args()
    if args.config is not None:
        from deepseek_sparse_attention_fp8_gb300.inputs import CONFIG_WORKLOADS

        if not 0 <= args.config < len(CONFIG_WORKLOADS):
            ap.error(f"--config must be in 0..{len(CONFIG_WORKLOADS) - 1}")
        args.workload = CONFIG_WORKLOADS[args.config]
    return args


def dist_info():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def algorithmic_bytes(wl, topk_idx_host=None, kv_row_bytes=None):
    """Bytes each kernel must move at minimum: its inputs read once, its outputs
    written once (gathered rows counted once per selected valid slot; a latent
    row is Dk bf16 values, or kv_row_bytes for the fp8 cache)."""
    T, ld, K = wl.T, wl.ld, wl.index_topk
    qsl = wl.query_start_loc
    valid = []
    for b in range(wl.B):
        ql = qsl[b + 1] - qsl[b]
        for i in range(ql):
            valid.append(int(wl.seq_lens[b]) - ql + i + 1)
    valid = np.array(valid, dtype=np.int64)
    key_bytes = int(np.sum(wl.seq_lens.astype(np.int64))) * (wl.Di + 4)
    indexer = key_bytes + T * wl.Hi * wl.Di * 2 + T * wl.Hi * 4 + T * ld * 4
    topk = int(np.sum(valid)) * 4 + T * K * 4
    live = np.minimum(valid, K) if topk_idx_host is None else np.sum(topk_idx_host >= 0, axis=1)
    row = wl.Dk * 2 if kv_row_bytes is None else kv_row_bytes
    attention = int(np.sum(live)) * row + T * wl.H * wl.Dk * 2 + T * wl.H * wl.Dv * 2 + T * K * 4 + T * wl.H * 4
    flops_att = int(np.sum(live)) * wl.H * (2 * wl.Dk + 2 * wl.Dv)
    flops_idx = int(np.sum(valid)) * wl.Hi * wl.Di * 2
    return dict(indexer=indexer, topk=topk, attention=attention, flops_attention=flops_att, flops_indexer=flops_idx)


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            with open(p) as f:
                d = json.load(f)
            hbm = d.get("hbm_gbs") or d.get("hbm_GBs")
            return float(hbm), "measured", d
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback", None


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        # the raw samples go to DSA_BENCH_OUT (default: the system temp directory)
        out_dir = os.environ.get("DSA_BENCH_OUT") or tempfile.gettempdir()
        os.makedirs(out_dir, exist_ok=True)
        self.path = os.path.join(out_dir, f"clocks_rank{self.gpu}.csv")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def cpu_oracle_step(wl, rows, threads=0):
    """The plain C++ oracle's DSA step (a0-a3) for the given query rows on
    `threads` host threads (0 = all hardware threads); returns seconds."""
    from oracle import ref as R

    t0 = time.perf_counter()
    R.step(wl, rows, threads=threads)
    return time.perf_counter() - t0


def cpu_model() -> str:
    """The host CPU's name as /proc/cpuinfo gives it (x86 or Arm)."""
    import platform

    try:
        fields = {}
        with open("/proc/cpuinfo") as f:
            for line in f:
                k, _, v = line.partition(":")
                fields.setdefault(k.strip(), v.strip())
        if fields.get("model name"):
            return fields["model name"]
        if fields.get("CPU part"):
            return f"{platform.machine()} implementer {fields.get('CPU implementer', '?')} part {fields['CPU part']}"
    except OSError:
        pass
    return platform.processor() or platform.machine()


def oracle_rows(T: int, n: int):
    """n evenly spaced query tokens of T."""
    n = max(1, min(T, n))
    return sorted({(i * T) // n for i in range(n)})


def oracle_timed(wl, budget_s: float = 10.0):
    """The C++ oracle on a bounded sample of the workload's query tokens, about
    budget_s seconds on every hardware thread: (rows, seconds, threads,
    seconds of one token on one thread)."""
    from oracle import ref as R

    threads = R.hardware_threads()
    one = cpu_oracle_step(wl, [0], threads=1)
    n = int(max(1, min(wl.T, budget_s * threads / max(one, 1e-6))))
    rows = oracle_rows(wl.T, n)
    sec = cpu_oracle_step(wl, rows, threads=threads)
    return rows, sec, threads, one


def run_reference(args, wl):
    """The C++ oracle timed on the host cores: each step is a bounded sample of
    query tokens of the workload (sized so the whole run stays within a few
    minutes), scaled to tokens/s."""
    from oracle import ref as R

    threads = R.hardware_threads()
    one = cpu_oracle_step(wl, [0], threads=1)
    budget = 150.0 / max(1, args.steps + args.warmup)
    n = int(max(1, min(wl.T, budget * threads / max(one, 1e-6))))
    rows = oracle_rows(wl.T, n)
    for _ in range(args.warmup):
        cpu_oracle_step(wl, rows, threads=threads)
    times = [cpu_oracle_step(wl, rows, threads=threads) for _ in range(args.steps)]
    sec = float(np.median(times))
    value = len(rows) / sec
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3 * wl.T / len(rows),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "B": wl.B, "T": wl.T, "context": int(wl.seq_lens.max()),
                       "index_topk": wl.index_topk, "Hi": wl.Hi, "Di": wl.Di, "H": wl.H, "Dk": wl.Dk, "Dv": wl.Dv,
                       "block_size": wl.block_size},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                             "sample": f"{len(rows)} of {wl.T} query tokens per step, evenly spaced (full indexer "
                                       f"row, top-k, attention), plain C++17 oracle, {threads} std::threads",
                             "cpu_model": cpu_model()},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def pct(xs, q):
    return float(np.percentile(np.asarray(xs, dtype=np.float64), q))


def summary(xs):
    """Median and 10th / 90th percentiles of a list of milliseconds."""
    return {"ms": pct(xs, 50), "p10_ms": pct(xs, 10), "p90_ms": pct(xs, 90)}


def fp8_peak_tflops(peaks_doc):
    """Dense e4m3 tensor peak: twice the measured bf16 burst (the nominal
    fp8:bf16 ratio of this part; only bf16 is measured)."""
    if peaks_doc and peaks_doc.get("bf16_tflops"):
        return 2.0 * float(peaks_doc["bf16_tflops"]), "2 x measured bf16 burst (nominal fp8:bf16 ratio)"
    return 2.0 * FALLBACK_BF16_TFLOPS, "2 x fallback bf16 (nominal fp8:bf16 ratio)"


def bf16_peak_tflops(peaks_doc):
    if peaks_doc and peaks_doc.get("bf16_tflops"):
        return float(peaks_doc["bf16_tflops"]), "measured bf16 burst"
    return FALLBACK_BF16_TFLOPS, "fallback bf16"


def kernel_table(wl, phase_ms, alg, peaks_doc):
    """Per-kernel achieved rate against its roofline: HBM bytes for the decode
    shapes, tensor-core flops for the prefill indexer (e4m3) and prefill
    attention (bf16)."""
    hbm, _, _ = load_peaks()
    prefill = wl.max_q_len > 2
    fp8, fp8_src = fp8_peak_tflops(peaks_doc)
    bf16, bf16_src = bf16_peak_tflops(peaks_doc)
    rows = {
        "indexer_logits": (alg["indexer"], alg["flops_indexer"], fp8, fp8_src),
        "topk": (alg["topk"], 0, None, None),
        "sparse_mla": (alg["attention"], alg["flops_attention"], bf16, bf16_src),
    }
    out = {}
    for name, (nbytes, flops, tpeak, tsrc) in rows.items():
        st = phase_ms[name]
        sec = st["ms"] / 1e3
        d = dict(st)
        d["bytes"] = int(nbytes)
        d["GBps"] = nbytes / sec / 1e9
        d["hbm_frac"] = d["GBps"] / hbm
        if flops:
            d["flops"] = int(flops)
            d["TFLOPs"] = flops / sec / 1e12
            d["tensor_frac"] = d["TFLOPs"] / tpeak
            d["tensor_peak"] = tpeak
            d["tensor_peak_source"] = tsrc
        tensor_bound = prefill and name != "topk"
        d["bound"] = "tensor" if tensor_bound else "hbm"
        d["frac"] = d["tensor_frac"] if tensor_bound else d["hbm_frac"]
        out[name] = d
    return out


def main():
    args = parse()
    rank, world, local = dist_info()
    from deepseek_sparse_attention_fp8_gb300.inputs import make_workload

    if args.oracle_seconds:
        wl = make_workload(args.workload, seed=args.seed)
        print(cpu_oracle_step(wl, oracle_rows(wl.T, args.oracle_seconds), threads=1), flush=True)
        return
    if args.impl == "reference":
        if rank != 0:
            return
        run_reference(args, make_workload(args.workload, seed=args.seed))
        return

    import torch

    import __graft_entry__

    __graft_entry__.build()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    from deepseek_sparse_attention_fp8_gb300.step import DsaStep

    wl = make_workload(args.workload, seed=args.seed, kv_fp8=args.kv_fp8)
    step = DsaStep(wl, device=f"cuda:{local}", num_kv_splits=args.splits, kv_fp8=args.kv_fp8)
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=step.device)
    flush_rd = torch.ones(256 * 1024 * 1024 // 4, dtype=torch.float32, device=step.device)

    def flush_l2():
        # write 256 MiB (evicts every line of the step's inputs), then read
        # another 256 MiB so that the dirty lines are written back here and
        # not inside the next timed step
        flush.zero_()
        flush_rd.sum()

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    def warm(st, n):
        for _ in range(max(3, n)):
            st.run()
        torch.cuda.synchronize()
        assert int(st.dev_status.item()) == 0, "device status bits set during warm-up"
        assert torch.isfinite(st.out.float()).all(), "non-finite output"

    def time_steps(st, n):
        # events only at step boundaries, so that nothing sits between the
        # step's kernels (each is launched as a programmatic dependent of the
        # one before); L2 flushed before every step
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
        barrier()
        for k in range(n):
            flush_l2()
            ev[k][0].record(stream)
            st.run()
            ev[k][1].record(stream)
        barrier()
        return [e[0].elapsed_time(e[1]) for e in ev]

    def time_phases(st, n):
        # each phase timed alone after its own L2 flush (its inputs are the
        # previous phase's outputs, already in place)
        evb = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(n)]
        for k in range(n):
            e = evb[k]
            for ph, fn in enumerate((st.indexer, st.topk, st.attention)):
                flush_l2()
                e[2 * ph].record(stream)
                fn()
                e[2 * ph + 1].record(stream)
        barrier()
        return {name: summary([evb[k][2 * ph].elapsed_time(evb[k][2 * ph + 1]) for k in range(n)])
                for ph, name in enumerate(("indexer_logits", "topk", "sparse_mla"))}

    def phases_consistent(st, t_step_ms, n):
        """Phase medians whose sum is within 1.3x of the step median (each phase
        alone pays its own launch and ramp, the chained step does not); one
        re-measurement, then a hard failure."""
        for _ in range(2):
            ph = time_phases(st, n)
            total = sum(v["ms"] for v in ph.values())
            if total <= 1.3 * t_step_ms:
                return ph, total
        raise SystemExit(f"bench: phase medians sum to {total:.4f} ms, more than 1.3 x the step median "
                         f"{t_step_ms:.4f} ms: the breakdown does not describe the step")

    peak, peak_kind, peaks_doc = load_peaks()

    warm(step, args.warmup)
    # clocks: sampler runs through a one-second sustained load and the timed steps
    sampler = ClockSampler(local)
    sampler.start()
    t_end = time.time() + (0.0 if args.no_clock_load else 1.0)
    while time.time() < t_end:
        for _ in range(20):
            step.run()
        torch.cuda.synchronize()

    K = args.steps
    wall0 = time.perf_counter()
    t_step = time_steps(step, K)
    wall = time.perf_counter() - wall0
    clocks = sampler.stop()
    step_stats = summary(t_step)
    Kb = max(5, min(K, 50))
    phase_ms, phase_sum = phases_consistent(step, step_stats["ms"], Kb)

    # producer side, not part of the step: the new tokens' indexer keys
    # quantised into a scratch copy of the key cache
    from deepseek_sparse_attention_fp8_gb300 import api

    gen = torch.Generator(device=step.device).manual_seed(1234)
    k_new = torch.randn((wl.T, wl.Di), generator=gen, device=step.device).to(torch.bfloat16)
    k_scratch = step.k_cache.clone()
    evp = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(Kb)]
    for k in range(Kb):
        flush_l2()
        evp[k][0].record(stream)
        api.dsa_indexer_k_quant_and_cache(k_new, k_scratch, step.block_table, step.seq_lens, step.qsl, wl.block_size,
                                          dev_status=step.dev_status)
        evp[k][1].record(stream)
    barrier()
    t_prod = summary([evp[k][0].elapsed_time(evp[k][1]) for k in range(Kb)])
    del k_scratch
    from deepseek_sparse_attention_fp8_gb300.replicas import aggregate

    ms, _, value = aggregate(step_stats["ms"], wl.T, step.device)

    # warm-L2 (no flush) for context
    ew = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ew[0].record(stream)
    for _ in range(20):
        step.run()
    ew[1].record(stream)
    torch.cuda.synchronize()
    ms_warm = ew[0].elapsed_time(ew[1]) / 20

    # e2e through the public API with host buffers: per-step inputs (queries,
    # head weights, block table, lengths) copied from pinned memory, output and
    # lse read back; the caches stay resident like a serving engine's KV cache.
    # DsaStep.run_host copies the indexer's inputs first and the attention
    # queries on a side stream while the indexer and top-k run.
    e2e = None
    if not args.no_e2e:
        host_in = step.inputs.cpu().pin_memory()
        host_q = step.inputs_q.cpu().pin_memory()
        host_out = torch.empty_like(step.outputs, device="cpu").pin_memory()
        h2d = host_in.numel() * host_in.element_size() + host_q.numel() * host_q.element_size()
        d2h = host_out.numel() * host_out.element_size()
        Ke = max(10, min(K, 200))
        eve = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(Ke)]
        barrier()
        for k in range(Ke):
            flush_l2()
            eve[k][0].record(stream)
            step.run_host(host_in, host_q, host_out)
            eve[k][1].record(stream)
        barrier()
        e2e_stats = summary([e[0].elapsed_time(e[1]) for e in eve])
        ms_e2e, _, v_e2e = aggregate(e2e_stats["ms"], wl.T, step.device)
        e2e = {"value": v_e2e, "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "ms_per_step": ms_e2e, "p10_ms": e2e_stats["p10_ms"],
               "p90_ms": e2e_stats["p90_ms"]}

    alg = algorithmic_bytes(wl, step.topk_idx.cpu().numpy(), wl.kv_row_bytes_fp8 if args.kv_fp8 else None)
    kern = kernel_table(wl, phase_ms, alg, peaks_doc)
    # bf16 keys read, codes and scales written
    prod_bytes = wl.T * (wl.Di * 2 + wl.Di + 4)
    producer = {"indexer_k_quant_and_cache": dict(t_prod, bytes=prod_bytes,
                                                  GBps=prod_bytes / (t_prod["ms"] / 1e3) / 1e9)}
    producer["indexer_k_quant_and_cache"]["frac"] = producer["indexer_k_quant_and_cache"]["GBps"] / peak
    dom = max(kern, key=lambda k_: kern[k_]["ms"])
    traffic = load_traffic(dom, wl.name + ("_fp8kv" if args.kv_fp8 else ""))
    step_bytes = alg["indexer"] + alg["topk"] + alg["attention"]
    launches_per_step = step.kernel_launches()
    splits_used = step.splits
    del step

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms, "p10_ms": step_stats["p10_ms"], "p90_ms": step_stats["p90_ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3+bf16", "data": "synthetic",
        "config": {"workload": wl.name, "B": wl.B, "T": wl.T, "context": int(wl.seq_lens.max()),
                   "index_topk": wl.index_topk, "Hi": wl.Hi, "Di": wl.Di, "H": wl.H, "Dk": wl.Dk, "Dv": wl.Dv,
                   "block_size": wl.block_size, "num_kv_splits": splits_used,
                   "kv_cache": "fp8 (656 B/row)" if args.kv_fp8 else "bf16",
                   "l2": "flushed between steps (256 MiB write + 256 MiB read)",
                   "seed": "workload default" if args.seed is None else args.seed,
                   "parallelism": "replicas" if world > 1 else "1 GPU"},
        "roofline": {"bound": kern[dom]["bound"], "kernel": dom,
                     "achieved": kern[dom]["GBps"] if kern[dom]["bound"] == "hbm" else kern[dom]["TFLOPs"],
                     "peak": peak if kern[dom]["bound"] == "hbm" else kern[dom]["tensor_peak"],
                     "unit": "GB/s" if kern[dom]["bound"] == "hbm" else "TFLOP/s",
                     "frac": kern[dom]["frac"], "peak_source": peak_kind, "traffic": traffic,
                     "step_GBps": step_bytes / (ms / 1e3) / 1e9, "step_frac": step_bytes / (ms / 1e3) / 1e9 / peak},
        "kernels": kern,
        "phase_sum_ms": phase_sum,
        "producer": producer,
        "warm_l2_ms_per_step": ms_warm,
        "gpu_launches": launches_per_step * K,
        "clocks": clocks,
        "wall_s": wall,
    }
    if e2e is not None:
        line["e2e"] = e2e

    # the other workloads, each measured the same way (median of flushed
    # steps, phases alone), on rank 0 at N=1 only
    if world == 1 and not args.no_other_workloads:
        others = {}
        for name, splits_list, fp8 in OTHER_WORKLOADS:
            if name == wl.name and not fp8:
                continue
            owl = make_workload(name, kv_fp8=fp8)
            for sp in splits_list:
                ost = DsaStep(owl, device=step_device(local), num_kv_splits=sp, kv_fp8=fp8)
                warm(ost, 3)
                n = max(5, min(K, 30))
                ts = summary(time_steps(ost, n))
                oph, osum = phases_consistent(ost, ts["ms"], max(5, min(n, 10)))
                oalg = algorithmic_bytes(owl, ost.topk_idx.cpu().numpy(), owl.kv_row_bytes_fp8 if fp8 else None)
                okern = kernel_table(owl, oph, oalg, peaks_doc)
                odom = max(okern, key=lambda k_: okern[k_]["ms"])
                obytes = oalg["indexer"] + oalg["topk"] + oalg["attention"]
                key = (name if len(splits_list) == 1 else f"{name}_splits{sp}") + ("_fp8kv" if fp8 else "")
                others[key] = {
                    "config": {"workload": name, "B": owl.B, "T": owl.T, "context": int(owl.seq_lens.max()),
                               "index_topk": owl.index_topk, "num_kv_splits": ost.splits,
                               "prefill": bool(ost.prefill), "kv_cache": "fp8 (656 B/row)" if fp8 else "bf16"},
                    "value": owl.T / (ts["ms"] / 1e3), "unit": "tokens/s", "steps": n, **ts,
                    "step_GBps": obytes / (ts["ms"] / 1e3) / 1e9,
                    "step_frac": obytes / (ts["ms"] / 1e3) / 1e9 / peak,
                    "dominant": odom, "kernels": okern, "phase_sum_ms": osum,
                    "traffic": load_traffic(odom, name + ("_fp8kv" if fp8 else "")) if len(splits_list) == 1 else None,
                }
                del ost
                torch.cuda.empty_cache()
        line["workloads"] = others

    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        rows, sec, threads, one = oracle_timed(wl)
        line["cpu_baseline"] = {"value": len(rows) / sec, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                                "sample": f"{len(rows)} of {wl.T} query tokens, evenly spaced (full indexer row, "
                                          f"top-k, attention), plain C++17 oracle on {threads} std::threads, "
                                          f"{sec:.1f} s",
                                "cpu_model": cpu_model(), "one_thread_value": 1.0 / one}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def step_device(local):
    return f"cuda:{local}"


# Workloads measured beside the headline one: (name, split counts, fp8 latent
# cache); the long-context decode runs at the three split counts its parity
# test forces, and two decode shapes run over the fp8 latent cache as well.
OTHER_WORKLOADS = (
    ("decode_b32_l8192", (0,), False),
    ("decode_b8_l131072", (1, 8, 32), False),
    ("prefill_4096_of_65536", (0,), False),
    ("mixed_b64_mtp2", (0,), False),
    ("decode_b32_l8192", (0,), True),
    ("decode_b8_l131072", (0,), True),
)


def load_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if one exists for
    this kernel and workload (null otherwise)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        with open(p) as f:
            d = json.load(f)
        return d.get(workload, {}).get(kernel)
    except Exception:
        return None


if __name__ == "__main__":
    main()
