"""One DSA step on the device: indexer logits -> top-k -> sparse MLA.

`DsaStep` owns the device copies of one workload's inputs and the output,
logits and workspace buffers, so that `run()` only enqueues the library's
kernels (no allocation, no host synchronisation). It is the call a user
makes per attention layer and batch; the tests and the benchmark drive it.

The per-step inputs the indexer and top-k read (q_idx, w, block_table,
seq_lens, query_start_loc) are views into one device buffer, `inputs`; the
attention queries q into a second, `inputs_q`; the outputs (out, lse) into a
third, `outputs`; each tensor at a 256-byte aligned offset. A caller that
stages a step's inputs in host memory moves them with one copy per buffer
(`run_host` overlaps the queries' copy with the indexer and top-k). The
caches stay resident in their own buffers.
"""
from __future__ import annotations

import contextlib
import os

import numpy as np
import torch

from . import api


_ALIGN = 256


def _packed(specs, device):
    """One uint8 device buffer holding tensors of the given (shape, dtype), each
    at a 256-byte aligned offset; returns (buffer, [views])."""
    offs, total = [], 0
    for shape, dtype in specs:
        nbytes = int(np.prod(shape)) * torch.tensor([], dtype=dtype).element_size()
        offs.append((total, nbytes))
        total += (nbytes + _ALIGN - 1) // _ALIGN * _ALIGN
    buf = torch.empty(max(total, _ALIGN), dtype=torch.uint8, device=device)
    views = [buf[o:o + n].view(dtype).view(shape) for (o, n), (shape, dtype) in zip(offs, specs)]
    return buf, views


def _host(a, dtype):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype == torch.bfloat16:
        t = t.view(torch.int16).view(torch.bfloat16)
    return t if t.dtype == dtype else t.to(dtype)


def _dev(a, dtype, device):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype in (torch.bfloat16,):
        t = t.view(torch.int16).view(torch.bfloat16)
    return t.to(device=device, dtype=dtype) if t.dtype != dtype else t.to(device)


def _nvtx_enabled() -> bool:
    return os.environ.get("DSA_NVTX", "0") not in ("", "0")


class DsaStep:
    """One DSA step over a workload's device buffers: indexer logits (a0 + a1),
    top-k (a2), sparse MLA with its split merge (a3 + a4).

    num_kv_splits: 0 automatic, -1 batch-invariant (fixed by index_topk), n > 0
    that many; when 0 and the environment sets DSA_NUM_KV_SPLITS, that value.
    DSA_NVTX=1 wraps each call in an NVTX range (for profilers)."""

    def __init__(self, wl, device="cuda", num_kv_splits: int = 0, prefill: bool | None = None, kv_fp8: bool = False):
        if num_kv_splits == 0 and os.environ.get("DSA_NUM_KV_SPLITS"):
            num_kv_splits = int(os.environ["DSA_NUM_KV_SPLITS"])
        self.nvtx = _nvtx_enabled()
        self.wl = wl
        self.device = torch.device(device)
        d = self.device
        # per-step inputs in two buffers: what the indexer and top-k read, and
        # the attention queries (copied from the host in parallel with those
        # kernels by run_host)
        ins = [(wl.q_idx, torch.bfloat16), (wl.w, torch.float32), (wl.block_table, torch.int32),
               (wl.seq_lens, torch.int32), (wl.query_start_loc, torch.int32)]
        self.inputs, views = _packed([(np.shape(a), dt) for a, dt in ins], d)
        for v, (a, dt) in zip(views, ins):
            v.copy_(_host(a, dt))
        self.q_idx, self.w, self.block_table, self.seq_lens, self.qsl = views
        self.inputs_q, (self.q,) = _packed([(np.shape(wl.q), torch.bfloat16)], d)
        self.q.copy_(_host(wl.q, torch.bfloat16))
        self._side = None
        self.k_cache = _dev(wl.k_cache, torch.uint8, d)
        # the latent cache: bf16 rows, or (kv_fp8) the workload's fp8 rows
        self.kv_fp8 = kv_fp8
        if kv_fp8:
            if wl.kv_cache_fp8 is None:
                raise ValueError("the workload was built without kv_fp8=True")
            self.kv_cache = _dev(wl.kv_cache_fp8, torch.uint8, d)
        else:
            self.kv_cache = _dev(wl.kv_cache, torch.bfloat16, d)
        self.logits = torch.empty((wl.T, wl.ld), dtype=torch.float32, device=d)
        self.topk_idx = torch.empty((wl.T, wl.index_topk), dtype=torch.int32, device=d)
        self.outputs, (self.out, self.lse) = _packed([((wl.T, wl.H, wl.Dv), torch.bfloat16),
                                                      ((wl.T, wl.H), torch.float32)], d)
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=d)
        self.prefill = (wl.max_q_len > 2) if prefill is None else prefill
        # num_kv_splits: 0 automatic, -1 batch-invariant (fixed by index_topk), n > 0 that many
        self.splits = 1 if self.prefill else api.sparse_mla_num_splits(wl.T, wl.H, wl.Dv, wl.index_topk,
                                                                         num_kv_splits)
        ws_topk = api.dsa_topk_workspace_size(wl.T, wl.ld, wl.index_topk)
        ws_mla = api.sparse_mla_workspace_size(wl.T, wl.H, wl.Dv, self.splits)
        self.ws_topk = torch.empty(max(ws_topk, 16), dtype=torch.uint8, device=d)
        self.ws_mla = torch.empty(max(ws_mla, 16), dtype=torch.uint8, device=d)

    def _range(self, name):
        return torch.cuda.nvtx.range(name) if self.nvtx else contextlib.nullcontext()

    def indexer(self, stream=None):
        with self._range("dsa_indexer_logits"):
            self._indexer(stream)

    def topk(self, stream=None):
        with self._range("dsa_topk"):
            self._topk(stream)

    def attention(self, stream=None):
        with self._range("sparse_mla"):
            self._attention(stream)

    def _indexer(self, stream=None):
        wl = self.wl
        api.dsa_indexer_logits(self.q_idx, self.w, self.k_cache, self.block_table, self.seq_lens, self.qsl,
                               wl.block_size, wl.max_q_len, self.logits, self.dev_status, stream)

    def _topk(self, stream=None):
        api.dsa_topk(self.logits, self.seq_lens, self.qsl, self.wl.index_topk, self.topk_idx, self.ws_topk, stream)

    def _attention(self, stream=None):
        wl = self.wl
        prefill = api.sparse_mla_prefill_fp8 if self.kv_fp8 else api.sparse_mla_prefill
        decode = api.sparse_mla_decode_fp8 if self.kv_fp8 else api.sparse_mla_decode
        if self.prefill:
            prefill(self.q, self.kv_cache, self.block_table, self.seq_lens, self.qsl, self.topk_idx, wl.softmax_scale,
                    wl.Dv, self.out, self.lse, self.dev_status, stream)
        else:
            decode(self.q, self.kv_cache, self.block_table, self.seq_lens, self.qsl, self.topk_idx, wl.softmax_scale,
                   wl.Dv, self.out, self.lse, self.splits, self.ws_mla, self.dev_status, stream)

    def run(self, stream=None):
        self.indexer(stream)
        self.topk(stream)
        self.attention(stream)
        return self.out

    def run_host(self, host_inputs, host_q, host_outputs):
        """One step from pinned host memory on the current stream: the
        indexer's inputs (`host_inputs`, laid out like `inputs`) are copied
        first; the attention queries (`host_q`, like `inputs_q`) are copied on
        a side stream while the indexer and top-k run; out and lse come back
        into `host_outputs` (like `outputs`)."""
        main = torch.cuda.current_stream(self.device)
        if self._side is None:
            self._side = torch.cuda.Stream(self.device)
            self._q_copied = torch.cuda.Event()
        self._side.wait_stream(main)  # the previous step's attention has read q
        with torch.cuda.stream(self._side):
            self.inputs_q.copy_(host_q, non_blocking=True)
            self._q_copied.record(self._side)
        self.inputs.copy_(host_inputs, non_blocking=True)
        self.indexer()
        self.topk()
        main.wait_event(self._q_copied)
        self.attention()
        host_outputs.copy_(self.outputs, non_blocking=True)
        return host_outputs

    def kernel_launches(self) -> int:
        """Kernels one run() enqueues."""
        n = 1  # indexer
        n += 2 if api.dsa_topk_workspace_size(self.wl.T, self.wl.ld, self.wl.index_topk) else 1
        n += 1 if (self.prefill or self.splits == 1) else 2
        return n
