"""ctypes loader of the plain C++ oracle (oracle/dsa_oracle_ref.cpp).

TEST INFRASTRUCTURE ONLY (tests and the benchmark's CPU legs). Functions take
a workload's host arrays and return numpy results; `threads` is the number of
std::threads over query tokens (0 = the host's hardware threads).
"""
from __future__ import annotations

import ctypes

import numpy as np

from .build_ref import build

_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        _lib.oracle_hardware_threads.restype = ctypes.c_int
    return _lib


def _p(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def hardware_threads() -> int:
    return int(lib().oracle_hardware_threads())


def _threads(n):
    return hardware_threads() if not n else int(n)


def quant_q(q_bits: np.ndarray):
    """a0: (codes uint8 [..., Di], scales float32 [...]) of bf16 bits q [..., Di]."""
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    Di = q.shape[-1]
    rows = q.size // Di
    codes = np.zeros(q.shape, dtype=np.uint8)
    scales = np.zeros(q.shape[:-1], dtype=np.float32)
    lib().oracle_quant_q(_p(q), ctypes.c_int(rows), ctypes.c_int(Di), _p(codes), _p(scales))
    return codes, scales


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


def indexer_logits(wl, rows=None, threads=0):
    """a0 + a1: logits float32 [T, ld] for the listed tokens (others NaN)."""
    rows = _i32(np.arange(wl.T) if rows is None else rows)
    out = np.full((wl.T, wl.ld), np.nan, dtype=np.float32)
    q = np.ascontiguousarray(wl.q_idx, dtype=np.uint16)
    w = np.ascontiguousarray(wl.w, dtype=np.float32)
    kc = np.ascontiguousarray(wl.k_cache, dtype=np.uint8)
    bt, sl, qsl = _i32(wl.block_table), _i32(wl.seq_lens), _i32(wl.query_start_loc)
    lib().oracle_indexer_logits(_p(q), _p(w), _p(kc), ctypes.c_int64(wl.k_block_stride), _p(bt),
                                ctypes.c_int(bt.shape[1]), _p(sl), _p(qsl), ctypes.c_int(wl.B), ctypes.c_int(wl.Hi),
                                ctypes.c_int(wl.Di), ctypes.c_int(wl.block_size), ctypes.c_int64(wl.ld), _p(rows),
                                ctypes.c_int(len(rows)), _p(out), ctypes.c_int(_threads(threads)))
    return out


def topk(logits, seq_lens, query_start_loc, index_topk, rows=None, threads=0):
    """a2: top-k [T, K] (largest first, ties by position, -1 padded)."""
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    T, ld = lg.shape
    rows = _i32(np.arange(T) if rows is None else rows)
    out = np.full((T, index_topk), -1, dtype=np.int32)
    sl, qsl = _i32(seq_lens), _i32(query_start_loc)
    lib().oracle_topk(_p(lg), ctypes.c_int64(ld), _p(sl), _p(qsl), ctypes.c_int(len(sl)), ctypes.c_int(index_topk),
                      _p(rows), ctypes.c_int(len(rows)), _p(out), ctypes.c_int(_threads(threads)))
    return out


def sparse_mla(wl, topk_idx, rows=None, threads=0):
    """a3: (out float64 [T, H, Dv], lse float64 [T, H]) for the listed tokens."""
    rows = _i32(np.arange(wl.T) if rows is None else rows)
    out = np.full((wl.T, wl.H, wl.Dv), np.nan)
    lse = np.full((wl.T, wl.H), np.nan)
    q = np.ascontiguousarray(wl.q, dtype=np.uint16)
    kv = np.ascontiguousarray(wl.kv_cache, dtype=np.uint16)
    idx = _i32(topk_idx)
    bt, sl, qsl = _i32(wl.block_table), _i32(wl.seq_lens), _i32(wl.query_start_loc)
    lib().oracle_sparse_mla(_p(q), _p(kv), ctypes.c_int64(wl.kv_block_stride), _p(bt), ctypes.c_int(bt.shape[1]),
                            _p(sl), _p(qsl), ctypes.c_int(wl.B), ctypes.c_int(wl.H), ctypes.c_int(wl.Dk),
                            ctypes.c_int(wl.Dv), _p(idx), ctypes.c_int(idx.shape[1]),
                            ctypes.c_double(wl.softmax_scale), ctypes.c_int(wl.block_size), _p(rows),
                            ctypes.c_int(len(rows)), _p(out), _p(lse), ctypes.c_int(_threads(threads)))
    return out, lse


def step(wl, rows, threads=0):
    """The whole step (a0-a3) for the listed query tokens."""
    logits = indexer_logits(wl, rows=rows, threads=threads)
    idx = topk(logits, wl.seq_lens, wl.query_start_loc, wl.index_topk, rows=rows, threads=threads)
    return sparse_mla(wl, idx, rows=rows, threads=threads)
