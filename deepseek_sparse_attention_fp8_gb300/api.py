"""Python binding of libdsa (include/dsa.h): argument marshalling only.

Every function here has the name of the C entry point it calls. Tensors are
torch CUDA tensors (PyTorch provides device memory and streams); the binding
checks dtypes, shapes and contiguity, passes raw pointers and the current
CUDA stream, and raises DsaError on a non-OK status. All arithmetic happens
in the CUDA kernels of libdsa. Importing this module loads libdsa.so and
raises if it has not been built (run ``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB

_H = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "dsa.h")

if not os.path.exists(LIB):
    raise RuntimeError(f"libdsa.so is not built ({LIB} missing): run __graft_entry__.build() first")
lib = ctypes.CDLL(LIB)

DSA_OK, DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED, DSA_ERR_WORKSPACE, DSA_ERR_CUDA = range(5)
DSA_DEVERR_BLOCK_OOB, DSA_DEVERR_INDEX_OOB, DSA_DEVERR_TIMEOUT, DSA_DEVERR_SEQ_LEN = 1, 2, 4, 8
DSA_KV_SPLITS_BATCH_INVARIANT = -1

_p = ctypes.c_void_p
_i32 = ctypes.c_int32
_i64 = ctypes.c_int64
_f32 = ctypes.c_float
_sz = ctypes.c_size_t

_SIGS = {
    "dsa_last_error": ([], ctypes.c_char_p),
    "dsa_version": ([], ctypes.c_char_p),
    "dsa_quant_q": ([_p, _i64, _i32, _i32, _i32, _p, _p, _p], _i32),
    "dsa_indexer_logits": ([_p, _i64, _p, _p, _i64, _i32, _p, _i32, _p, _p, _i32, _i32, _i32, _i32, _i32, _i32, _p,
                            _i64, _p, _p], _i32),
    "dsa_indexer_k_quant_and_cache": ([_p, _i64, _i32, _i32, _p, _i64, _i32, _p, _i32, _p, _p, _i32, _i32, _p, _p],
                                      _i32),
    "dsa_topk_workspace_size": ([_i32, _i64, _i32], _sz),
    "dsa_indexer_topk_workspace_size": ([_i32, _i64, _i32, _i32], _sz),
    "dsa_indexer_topk": ([_p, _i64, _p, _p, _i64, _i32, _p, _i32, _p, _p, _i32, _i32, _i32, _i32, _i32, _i32, _i64,
                          _i32, _i32, _p, _p, _sz, _p, _p], _i32),
    "dsa_topk": ([_p, _i64, _p, _p, _i32, _i32, _i32, _p, _p, _sz, _p], _i32),
    "sparse_mla_workspace_size": ([_i32, _i32, _i32, _i32], _sz),
    "sparse_mla_auto_splits": ([_i32, _i32, _i32, _i32], _i32),
    "sparse_mla_num_splits": ([_i32, _i32, _i32, _i32, _i32], _i32),
    "sparse_mla_decode": ([_p, _p, _i64, _i32, _p, _i32, _p, _p, _p, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _f32,
                           _i32, _p, _p, _p, _sz, _p, _p], _i32),
    "sparse_mla_fixed_scratch_bytes": ([], _sz),
    "sparse_mla_decode_fixed_scratch": ([_p, _p, _i64, _i32, _p, _i32, _p, _p, _p, _i32, _i32, _i32, _i32, _i32, _i32,
                                         _i32, _f32, _i32, _p, _p, _p, _p], _i32),
    "sparse_mla_prefill": ([_p, _p, _i64, _i32, _p, _i32, _p, _p, _p, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _f32,
                            _p, _p, _p, _p], _i32),
    "sparse_mla_decode_fp8": ([_p, _p, _i64, _i32, _p, _i32, _p, _p, _p, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
                               _f32, _i32, _p, _p, _p, _sz, _p, _p], _i32),
    "sparse_mla_prefill_fp8": ([_p, _p, _i64, _i32, _p, _i32, _p, _p, _p, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
                                _f32, _p, _p, _p, _p], _i32),
    "dsa_mla_kv_fp8_quant_and_cache": ([_p, _i64, _i32, _i32, _i32, _p, _i64, _i32, _p, _i32, _p, _p, _i32, _i32, _p,
                                        _p], _i32),
}

MLA_FP8_ROW_BYTES = 656  # fp8 latent cache row at Dk = 576, Dv = 512
for _name, (_args, _res) in _SIGS.items():
    _fn = getattr(lib, _name)
    _fn.argtypes = _args
    _fn.restype = _res


class DsaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: status {status}: {lib.dsa_last_error().decode()}")


def _check(status: int, where: str):
    if status != DSA_OK:
        raise DsaError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, dtype, name, dims=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dims is not None and t.dim() != dims:
        raise ValueError(f"{name} must have {dims} dims, got {t.dim()}")


def dsa_version() -> str:
    return lib.dsa_version().decode()


def dsa_quant_q(q_idx, q8=None, sq=None, stream=None):
    """a0: e4m3 codes [T,Hi,Di] (uint8) and fp32 scales [T,Hi] of the indexer q."""
    _need(q_idx, torch.bfloat16, "q_idx", 3)
    T, Hi, Di = q_idx.shape
    q8 = torch.empty((T, Hi, Di), dtype=torch.uint8, device=q_idx.device) if q8 is None else q8
    sq = torch.empty((T, Hi), dtype=torch.float32, device=q_idx.device) if sq is None else sq
    _need(q8, torch.uint8, "q8", 3)
    _need(sq, torch.float32, "sq", 2)
    _check(lib.dsa_quant_q(_ptr(q_idx), Hi * Di, T, Hi, Di, _ptr(q8), _ptr(sq), _stream(stream)), "dsa_quant_q")
    return q8, sq


def dsa_indexer_k_quant_and_cache(k, k_cache, block_table, seq_lens, query_start_loc, block_size, dev_status=None,
                                  stream=None):
    """Quantises the new tokens' indexer keys k [T, Di] (bf16) to e4m3 with one
    fp32 scale per token and stores them into the paged fp8 key cache
    k_cache [num_blocks, k_block_stride_bytes] (uint8) in place."""
    _need(k, torch.bfloat16, "k", 2)
    _need(k_cache, torch.uint8, "k_cache", 2)
    _need(block_table, torch.int32, "block_table", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _need(query_start_loc, torch.int32, "query_start_loc", 1)
    if dev_status is not None:
        _need(dev_status, torch.int32, "dev_status")
    T, Di = k.shape
    st = lib.dsa_indexer_k_quant_and_cache(_ptr(k), Di, T, Di, _ptr(k_cache), k_cache.shape[1], k_cache.shape[0],
                                           _ptr(block_table), block_table.shape[1], _ptr(seq_lens),
                                           _ptr(query_start_loc), seq_lens.shape[0], block_size, _ptr(dev_status),
                                           _stream(stream))
    _check(st, "dsa_indexer_k_quant_and_cache")
    return k_cache


def dsa_indexer_logits(q_idx, w, k_cache, block_table, seq_lens, query_start_loc, block_size, max_q_len, logits,
                       dev_status=None, stream=None):
    """a0 + a1: fills logits [T, ld] (fp32) for the paged fp8 key cache
    k_cache [num_blocks, k_block_stride_bytes] (uint8)."""
    _need(q_idx, torch.bfloat16, "q_idx", 3)
    _need(w, torch.float32, "w", 2)
    _need(k_cache, torch.uint8, "k_cache", 2)
    _need(block_table, torch.int32, "block_table", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _need(query_start_loc, torch.int32, "query_start_loc", 1)
    _need(logits, torch.float32, "logits", 2)
    T, Hi, Di = q_idx.shape
    B = seq_lens.shape[0]
    if dev_status is not None:
        _need(dev_status, torch.int32, "dev_status")
    st = lib.dsa_indexer_logits(_ptr(q_idx), Hi * Di, _ptr(w), _ptr(k_cache), k_cache.shape[1], k_cache.shape[0],
                                _ptr(block_table), block_table.shape[1], _ptr(seq_lens), _ptr(query_start_loc), B, T,
                                Hi, Di, block_size, max_q_len, _ptr(logits), logits.shape[1], _ptr(dev_status),
                                _stream(stream))
    _check(st, "dsa_indexer_logits")
    return logits


def dsa_indexer_topk_workspace_size(T: int, max_seq_len: int, window: int, index_topk: int) -> int:
    return int(lib.dsa_indexer_topk_workspace_size(T, max_seq_len, window, index_topk))


def dsa_indexer_topk(q_idx, w, k_cache, block_table, seq_lens, query_start_loc, block_size, max_q_len, max_seq_len,
                     window, index_topk, topk_idx=None, workspace=None, dev_status=None, stream=None):
    """a1 + a2 over key windows of `window` keys (0 = one window): topk_idx
    [T, index_topk] (int32), the exact top-k of the indexer logits, with a
    logits buffer of [T, window] instead of [T, max_seq_len]."""
    _need(q_idx, torch.bfloat16, "q_idx", 3)
    _need(w, torch.float32, "w", 2)
    _need(k_cache, torch.uint8, "k_cache", 2)
    _need(block_table, torch.int32, "block_table", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _need(query_start_loc, torch.int32, "query_start_loc", 1)
    T, Hi, Di = q_idx.shape
    if topk_idx is None:
        topk_idx = torch.empty((T, index_topk), dtype=torch.int32, device=q_idx.device)
    _need(topk_idx, torch.int32, "topk_idx", 2)
    if dev_status is not None:
        _need(dev_status, torch.int32, "dev_status")
    need = dsa_indexer_topk_workspace_size(T, max_seq_len, window, index_topk)
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q_idx.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib.dsa_indexer_topk(_ptr(q_idx), Hi * Di, _ptr(w), _ptr(k_cache), k_cache.shape[1], k_cache.shape[0],
                              _ptr(block_table), block_table.shape[1], _ptr(seq_lens), _ptr(query_start_loc),
                              seq_lens.shape[0], T, Hi, Di, block_size, max_q_len, max_seq_len, window, index_topk,
                              _ptr(topk_idx), _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream))
    _check(st, "dsa_indexer_topk")
    return topk_idx


def dsa_topk_workspace_size(T: int, ld: int, index_topk: int) -> int:
    return int(lib.dsa_topk_workspace_size(T, ld, index_topk))


def dsa_topk(logits, seq_lens, query_start_loc, index_topk, topk_idx=None, workspace=None, stream=None):
    """a2: topk_idx [T, index_topk] (int32, ascending positions, -1 padded)."""
    _need(logits, torch.float32, "logits", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _need(query_start_loc, torch.int32, "query_start_loc", 1)
    T, ld = logits.shape
    if topk_idx is None:
        topk_idx = torch.empty((T, index_topk), dtype=torch.int32, device=logits.device)
    _need(topk_idx, torch.int32, "topk_idx", 2)
    need = dsa_topk_workspace_size(T, ld, index_topk)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=logits.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.dsa_topk(_ptr(logits), ld, _ptr(seq_lens), _ptr(query_start_loc), seq_lens.shape[0], T, index_topk,
                      _ptr(topk_idx), _ptr(workspace), ws_bytes, _stream(stream))
    _check(st, "dsa_topk")
    return topk_idx


def sparse_mla_workspace_size(T: int, H: int, Dv: int, num_kv_splits: int) -> int:
    return int(lib.sparse_mla_workspace_size(T, H, Dv, num_kv_splits))


def sparse_mla_auto_splits(T: int, H: int, Dv: int, index_topk: int) -> int:
    return int(lib.sparse_mla_auto_splits(T, H, Dv, index_topk))


def sparse_mla_num_splits(T: int, H: int, Dv: int, index_topk: int, num_kv_splits: int) -> int:
    """The split count sparse_mla_decode uses for num_kv_splits (0 = automatic,
    DSA_KV_SPLITS_BATCH_INVARIANT = fixed by index_topk alone, n = n)."""
    return int(lib.sparse_mla_num_splits(T, H, Dv, index_topk, num_kv_splits))


def _mla_common(q, kv_cache, block_table, seq_lens, query_start_loc, topk_idx, out, lse, dev_status):
    _need(q, torch.bfloat16, "q", 3)
    _need(kv_cache, torch.bfloat16, "kv_cache", 3)
    _need(block_table, torch.int32, "block_table", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _need(query_start_loc, torch.int32, "query_start_loc", 1)
    _need(topk_idx, torch.int32, "topk_idx", 2)
    _need(out, torch.bfloat16, "out", 3)
    if lse is not None:
        _need(lse, torch.float32, "lse", 2)
    if dev_status is not None:
        _need(dev_status, torch.int32, "dev_status")
    num_blocks, block_size, Dk = kv_cache.shape
    T, H, _ = q.shape
    return num_blocks, block_size, Dk, T, H


def sparse_mla_decode(q, kv_cache, block_table, seq_lens, query_start_loc, topk_idx, softmax_scale, dv, out,
                      lse=None, num_kv_splits=0, workspace=None, dev_status=None, stream=None):
    """a3 + a4: out [T,H,Dv] (bf16) of sparse MLA over kv_cache [blocks, block_size, Dk].
    num_kv_splits: 0 automatic (depends on the batch size), -1
    (DSA_KV_SPLITS_BATCH_INVARIANT) fixed by index_topk alone, or a count."""
    num_blocks, block_size, Dk, T, H = _mla_common(q, kv_cache, block_table, seq_lens, query_start_loc, topk_idx,
                                                   out, lse, dev_status)
    K = topk_idx.shape[1]
    splits = sparse_mla_num_splits(T, H, dv, K, num_kv_splits)
    need = sparse_mla_workspace_size(T, H, dv, splits)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.sparse_mla_decode(_ptr(q), _ptr(kv_cache), block_size * Dk, num_blocks, _ptr(block_table),
                               block_table.shape[1], _ptr(seq_lens), _ptr(query_start_loc), _ptr(topk_idx),
                               seq_lens.shape[0], T, H, Dk, dv, K, block_size, softmax_scale, num_kv_splits, _ptr(out),
                               _ptr(lse), _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream))
    _check(st, "sparse_mla_decode")
    return out


def sparse_mla_fixed_scratch_bytes() -> int:
    return int(lib.sparse_mla_fixed_scratch_bytes())


def sparse_mla_decode_fixed_scratch(q, kv_cache, block_table, seq_lens, query_start_loc, topk_idx, softmax_scale, dv,
                                    out, lse=None, num_kv_splits=0, dev_status=None, stream=None):
    """a3 + a4 without any allocation: the split partials live in the
    library's fixed device scratch (for callers that cannot allocate; calls
    that overlap on the GPU race on the shared scratch)."""
    num_blocks, block_size, Dk, T, H = _mla_common(q, kv_cache, block_table, seq_lens, query_start_loc, topk_idx,
                                                   out, lse, dev_status)
    K = topk_idx.shape[1]
    st = lib.sparse_mla_decode_fixed_scratch(_ptr(q), _ptr(kv_cache), block_size * Dk, num_blocks, _ptr(block_table),
                                             block_table.shape[1], _ptr(seq_lens), _ptr(query_start_loc),
                                             _ptr(topk_idx), seq_lens.shape[0], T, H, Dk, dv, K, block_size,
                                             softmax_scale, num_kv_splits, _ptr(out), _ptr(lse), _ptr(dev_status),
                                             _stream(stream))
    _check(st, "sparse_mla_decode_fixed_scratch")
    return out


def sparse_mla_prefill(q, kv_cache, block_table, seq_lens, query_start_loc, topk_idx, softmax_scale, dv, out,
                       lse=None, dev_status=None, stream=None):
    """a3 single pass (no splits, no workspace)."""
    num_blocks, block_size, Dk, T, H = _mla_common(q, kv_cache, block_table, seq_lens, query_start_loc, topk_idx,
                                                   out, lse, dev_status)
    K = topk_idx.shape[1]
    st = lib.sparse_mla_prefill(_ptr(q), _ptr(kv_cache), block_size * Dk, num_blocks, _ptr(block_table),
                                block_table.shape[1], _ptr(seq_lens), _ptr(query_start_loc), _ptr(topk_idx),
                                seq_lens.shape[0], T, H, Dk, dv, K, block_size, softmax_scale, _ptr(out), _ptr(lse),
                                _ptr(dev_status), _stream(stream))
    _check(st, "sparse_mla_prefill")
    return out


def header_functions():
    """Names of the functions include/dsa.h declares (for export checks)."""
    import re

    with open(_H) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const char\*|dsa_status_t|size_t|int32_t)\s+(\w+)\s*\(", text, re.M)))


def _mla_fp8_common(q, kv_cache, block_table, seq_lens, query_start_loc, topk_idx, out, lse, dev_status):
    _need(q, torch.bfloat16, "q", 3)
    _need(kv_cache, torch.uint8, "kv_cache", 3)
    _need(block_table, torch.int32, "block_table", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _need(query_start_loc, torch.int32, "query_start_loc", 1)
    _need(topk_idx, torch.int32, "topk_idx", 2)
    _need(out, torch.bfloat16, "out", 3)
    if lse is not None:
        _need(lse, torch.float32, "lse", 2)
    if dev_status is not None:
        _need(dev_status, torch.int32, "dev_status")
    num_blocks, block_size, row_bytes = kv_cache.shape
    T, H, Dk = q.shape
    return num_blocks, block_size, row_bytes, T, H, Dk


def sparse_mla_decode_fp8(q, kv_cache, block_table, seq_lens, query_start_loc, topk_idx, softmax_scale, dv, out,
                          lse=None, num_kv_splits=0, workspace=None, dev_status=None, stream=None):
    """a3 + a4 over the fp8 latent cache kv_cache [blocks, block_size, 656] (uint8)."""
    num_blocks, block_size, rb, T, H, Dk = _mla_fp8_common(q, kv_cache, block_table, seq_lens, query_start_loc,
                                                           topk_idx, out, lse, dev_status)
    K = topk_idx.shape[1]
    splits = sparse_mla_num_splits(T, H, dv, K, num_kv_splits)
    need = sparse_mla_workspace_size(T, H, dv, splits)
    if need and (workspace is None or workspace.numel() * workspace.element_size() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.sparse_mla_decode_fp8(_ptr(q), _ptr(kv_cache), block_size * rb, num_blocks, _ptr(block_table),
                                   block_table.shape[1], _ptr(seq_lens), _ptr(query_start_loc), _ptr(topk_idx),
                                   seq_lens.shape[0], T, H, Dk, dv, K, block_size, softmax_scale, num_kv_splits,
                                   _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream))
    _check(st, "sparse_mla_decode_fp8")
    return out


def sparse_mla_prefill_fp8(q, kv_cache, block_table, seq_lens, query_start_loc, topk_idx, softmax_scale, dv, out,
                           lse=None, dev_status=None, stream=None):
    """a3 single pass over the fp8 latent cache."""
    num_blocks, block_size, rb, T, H, Dk = _mla_fp8_common(q, kv_cache, block_table, seq_lens, query_start_loc,
                                                           topk_idx, out, lse, dev_status)
    K = topk_idx.shape[1]
    st = lib.sparse_mla_prefill_fp8(_ptr(q), _ptr(kv_cache), block_size * rb, num_blocks, _ptr(block_table),
                                    block_table.shape[1], _ptr(seq_lens), _ptr(query_start_loc), _ptr(topk_idx),
                                    seq_lens.shape[0], T, H, Dk, dv, K, block_size, softmax_scale, _ptr(out), _ptr(lse),
                                    _ptr(dev_status), _stream(stream))
    _check(st, "sparse_mla_prefill_fp8")
    return out


def dsa_mla_kv_fp8_quant_and_cache(kv, kv_cache, block_table, seq_lens, query_start_loc, block_size, dv=512,
                                   dev_status=None, stream=None):
    """Quantises the new tokens' latent rows kv [T, Dk] (bf16) into the fp8
    latent cache kv_cache [num_blocks, block_size, 656] (uint8) in place."""
    _need(kv, torch.bfloat16, "kv", 2)
    _need(kv_cache, torch.uint8, "kv_cache", 3)
    _need(block_table, torch.int32, "block_table", 2)
    _need(seq_lens, torch.int32, "seq_lens", 1)
    _need(query_start_loc, torch.int32, "query_start_loc", 1)
    if dev_status is not None:
        _need(dev_status, torch.int32, "dev_status")
    T, Dk = kv.shape
    nb, bs, rb = kv_cache.shape
    if bs != block_size:
        raise ValueError("kv_cache's second dim must be block_size")
    st = lib.dsa_mla_kv_fp8_quant_and_cache(_ptr(kv), Dk, T, Dk, dv, _ptr(kv_cache), bs * rb, nb, _ptr(block_table),
                                            block_table.shape[1], _ptr(seq_lens), _ptr(query_start_loc),
                                            seq_lens.shape[0], block_size, _ptr(dev_status), _stream(stream))
    _check(st, "dsa_mla_kv_fp8_quant_and_cache")
    return kv_cache
