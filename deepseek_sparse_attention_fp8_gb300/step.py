"""One DSA step on the device: indexer logits -> top-k -> sparse MLA.

`DsaStep` owns the device copies of one workload's inputs and the output,
logits and workspace buffers, so that `run()` only enqueues the library's
kernels (no allocation, no host synchronisation). It is the call a user
makes per attention layer and batch; the tests and the benchmark drive it.
"""
from __future__ import annotations

import numpy as np
import torch

from . import api


def _dev(a, dtype, device):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype in (torch.bfloat16,):
        t = t.view(torch.int16).view(torch.bfloat16)
    return t.to(device=device, dtype=dtype) if t.dtype != dtype else t.to(device)


class DsaStep:
    def __init__(self, wl, device="cuda", num_kv_splits: int = 0, prefill: bool | None = None):
        self.wl = wl
        self.device = torch.device(device)
        d = self.device
        self.q_idx = _dev(wl.q_idx, torch.bfloat16, d)
        self.w = _dev(wl.w, torch.float32, d)
        self.k_cache = _dev(wl.k_cache, torch.uint8, d)
        self.q = _dev(wl.q, torch.bfloat16, d)
        self.kv_cache = _dev(wl.kv_cache, torch.bfloat16, d)
        self.block_table = _dev(wl.block_table, torch.int32, d)
        self.seq_lens = _dev(wl.seq_lens, torch.int32, d)
        self.qsl = _dev(wl.query_start_loc, torch.int32, d)
        self.logits = torch.empty((wl.T, wl.ld), dtype=torch.float32, device=d)
        self.topk_idx = torch.empty((wl.T, wl.index_topk), dtype=torch.int32, device=d)
        self.out = torch.empty((wl.T, wl.H, wl.Dv), dtype=torch.bfloat16, device=d)
        self.lse = torch.empty((wl.T, wl.H), dtype=torch.float32, device=d)
        self.dev_status = torch.zeros(1, dtype=torch.int32, device=d)
        self.prefill = (wl.max_q_len > 2) if prefill is None else prefill
        self.splits = 1 if self.prefill else (num_kv_splits or api.sparse_mla_auto_splits(wl.T, wl.H, wl.Dv,
                                                                                          wl.index_topk))
        ws_topk = api.dsa_topk_workspace_size(wl.T, wl.ld, wl.index_topk)
        ws_mla = api.sparse_mla_workspace_size(wl.T, wl.H, wl.Dv, self.splits)
        self.ws_topk = torch.empty(max(ws_topk, 16), dtype=torch.uint8, device=d)
        self.ws_mla = torch.empty(max(ws_mla, 16), dtype=torch.uint8, device=d)

    def indexer(self, stream=None):
        wl = self.wl
        api.dsa_indexer_logits(self.q_idx, self.w, self.k_cache, self.block_table, self.seq_lens, self.qsl,
                               wl.block_size, wl.max_q_len, self.logits, self.dev_status, stream)

    def topk(self, stream=None):
        api.dsa_topk(self.logits, self.seq_lens, self.qsl, self.wl.index_topk, self.topk_idx, self.ws_topk, stream)

    def attention(self, stream=None):
        wl = self.wl
        if self.prefill:
            api.sparse_mla_prefill(self.q, self.kv_cache, self.block_table, self.seq_lens, self.qsl, self.topk_idx,
                                   wl.softmax_scale, wl.Dv, self.out, self.lse, self.dev_status, stream)
        else:
            api.sparse_mla_decode(self.q, self.kv_cache, self.block_table, self.seq_lens, self.qsl, self.topk_idx,
                                  wl.softmax_scale, wl.Dv, self.out, self.lse, self.splits, self.ws_mla,
                                  self.dev_status, stream)

    def run(self, stream=None):
        self.indexer(stream)
        self.topk(stream)
        self.attention(stream)
        return self.out

    def kernel_launches(self) -> int:
        """Kernels one run() enqueues."""
        n = 1  # indexer
        n += 2 if api.dsa_topk_workspace_size(self.wl.T, self.wl.ld, self.wl.index_topk) else 1
        n += 1 if (self.prefill or self.splits == 1) else 2
        return n
