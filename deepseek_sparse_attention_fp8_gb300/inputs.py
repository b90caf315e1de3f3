"""Seeded synthetic inputs for the DSA step, shaped like the five workloads.

This module draws random tensors and lays them out in the paged formats the
step consumes. It performs none of the step's arithmetic: the e4m3 key codes
are produced by PyTorch's own float8_e4m3fn cast, and the bf16 values by
PyTorch's bfloat16 cast. Both the CUDA path and the CPU oracle consume the
same arrays.

Layouts (host numpy arrays):
  q_idx        bf16 bits  uint16 [T, Hi, Di]
  w            float32    [T, Hi]
  k_cache      uint8      [num_blocks, k_block_stride]; inside a block:
               block_size*Di e4m3 bytes (token-major) then block_size fp32 scales
  q            bf16 bits  uint16 [T, H, Dk]
  kv_cache     bf16 bits  uint16 [num_blocks, block_size, Dk]
  block_table  int32      [B, max_blocks]   (-1 where unused)
  seq_lens     int32      [B]   (includes the new tokens)
  query_start_loc int32   [B+1]

Distributions (the five workloads): q_idx ~ N(0,1); indexer keys ~ N(0,1) rows
quantised per token with scale amax/448; w ~ N(0,1)/sqrt(Hi); MLA q ~ N(0,1);
KV ~ N(0,1) (tiny workload) or N(0, 0.5^2); permuted or fragmented block
tables; unused blocks poisoned with NaN.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch


@dataclasses.dataclass
class Workload:
    name: str
    B: int
    T: int
    Hi: int
    Di: int
    H: int
    Dk: int
    Dv: int
    index_topk: int
    block_size: int
    softmax_scale: float
    seq_lens: np.ndarray
    query_start_loc: np.ndarray
    block_table: np.ndarray
    num_blocks: int
    k_block_stride: int  # bytes
    kv_block_stride: int  # elements
    ld: int
    q_idx: np.ndarray
    w: np.ndarray
    k_cache: np.ndarray
    q: np.ndarray
    kv_cache: np.ndarray
    kv_cache_fp8: np.ndarray | None = None  # uint8 [num_blocks, block_size, 656] when drawn

    @property
    def kv_row_bytes_fp8(self) -> int:
        return self.Dv + 4 * (self.Dv // 128) + 2 * (self.Dk - self.Dv)

    @property
    def max_q_len(self) -> int:
        return int(np.max(np.diff(self.query_start_loc))) if self.B else 0


# the five configurations of the benchmark in their fixed order (config 0 .. 4)
CONFIG_WORKLOADS = ("tiny", "decode_b32_l8192", "decode_b8_l131072", "prefill_4096_of_65536", "mixed_b64_mtp2")

WORKLOADS = {
    # name: (B, L or (lo, hi), q_len, Hi, Di, H, Dk, Dv, topk, kv_std, w_div, table kind, seed)
    "tiny": dict(B=1, L=256, q_len=1, Hi=4, Di=32, H=4, Dk=80, Dv=64, topk=64, kv_std=1.0, table="identity", seed=0),
    "decode_b32_l8192": dict(B=32, L=8192, q_len=1, Hi=64, Di=128, H=128, Dk=576, Dv=512, topk=2048, kv_std=0.5,
                             table="permuted", seed=1),
    "decode_b8_l131072": dict(B=8, L=131072, q_len=1, Hi=64, Di=128, H=128, Dk=576, Dv=512, topk=2048, kv_std=0.5,
                              table="permuted", seed=2),
    "prefill_4096_of_65536": dict(B=1, L=65536, q_len=4096, Hi=64, Di=128, H=128, Dk=576, Dv=512, topk=2048,
                                  kv_std=0.5, table="permuted", seed=3),
    "mixed_b64_mtp2": dict(B=64, L=(1024, 32768), q_len=2, Hi=64, Di=128, H=128, Dk=576, Dv=512, topk=2048,
                           kv_std=0.5, table="fragmented", seed=4),
}


def _bf16_bits(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_float(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 values (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _e4m3_codes(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.float8_e4m3fn)
    return t.view(torch.uint8).numpy()


def make_workload(name: str, seed: int | None = None, *, B: int | None = None, L=None, q_len: int | None = None,
                  index_topk: int | None = None, ld_pad: int = 128, lens=None, block_size: int = 64,
                  q_std: float = 1.0, kv_fp8: bool = False, Hi: int | None = None, Di: int | None = None,
                  q_lens=None, H: int | None = None) -> Workload:
    """Build one of the named workloads (optionally overriding a few sizes
    for smaller parity cases). `lens` gives explicit per-request lengths and
    `q_lens` per-request query counts (with `lens`, one entry per request);
    `q_std` the standard deviation of the MLA queries (1 in every workload);
    `kv_fp8` also lays the latent rows out as an fp8 latent cache; `Hi` and
    `Di` change the indexer's head count and head dim, `H` the MLA head count."""
    spec = dict(WORKLOADS[name])
    if Hi is not None:
        spec["Hi"] = Hi
    if Di is not None:
        spec["Di"] = Di
    if H is not None:
        spec["H"] = H
    if B is not None:
        spec["B"] = B
    if L is not None:
        spec["L"] = L
    if q_len is not None:
        spec["q_len"] = q_len
    if index_topk is not None:
        spec["topk"] = index_topk
    rng = np.random.Generator(np.random.PCG64(spec["seed"] if seed is None else seed))
    Bn, qn = spec["B"], spec["q_len"]
    Hi, Di, H, Dk, Dv = spec["Hi"], spec["Di"], spec["H"], spec["Dk"], spec["Dv"]
    bs = block_size

    if lens is not None:
        seq_lens = np.asarray(lens, dtype=np.int32)
        Bn = len(seq_lens)
    elif isinstance(spec["L"], tuple):
        lo, hi = spec["L"]
        seq_lens = rng.integers(lo, hi + 1, size=Bn).astype(np.int32)
        # at least two requests shorter than index_topk, so that some KV splits
        # are entirely masked
        if Bn >= 2 and np.sum(seq_lens < spec["topk"]) < 2:
            seq_lens[0], seq_lens[1] = min(1024, spec["topk"] - 1), min(1500, spec["topk"] - 1)
    else:
        seq_lens = np.full(Bn, spec["L"], dtype=np.int32)
    seq_lens = np.maximum(seq_lens, qn).astype(np.int32)

    if q_lens is not None:
        q_lens = np.asarray(q_lens, dtype=np.int32)
        assert len(q_lens) == Bn and np.all(q_lens >= 1)
        seq_lens = np.maximum(seq_lens, q_lens).astype(np.int32)
    else:
        q_lens = np.full(Bn, qn, dtype=np.int32)
    qsl = np.zeros(Bn + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(q_lens)
    T = int(qsl[-1])

    blocks_per = [(int(l) + bs - 1) // bs for l in seq_lens]
    max_blocks = max(blocks_per) if Bn else 1
    needed = sum(blocks_per)
    table = spec["table"]
    if table == "fragmented":
        num_blocks = needed + max(8, needed // 4)
    else:
        num_blocks = needed
    if table == "identity":
        phys = np.arange(num_blocks)
    else:
        phys = rng.permutation(num_blocks)
    block_table = np.full((Bn, max_blocks), -1, dtype=np.int32)
    cur = 0
    for b in range(Bn):
        block_table[b, : blocks_per[b]] = phys[cur: cur + blocks_per[b]]
        cur += blocks_per[b]
    used = np.zeros(num_blocks, dtype=bool)
    used[phys[:cur]] = True

    # indexer key cache: rows ~ N(0,1) quantised per token (scale = amax/448)
    k_block_stride = bs * (Di + 4)
    k_cache = np.full((num_blocks, k_block_stride), 0x7F, dtype=np.uint8)  # unused: e4m3 NaN bytes
    keys = rng.standard_normal((num_blocks, bs, Di), dtype=np.float32)
    amax = np.abs(keys).max(axis=-1)
    kscale = (amax / np.float32(448.0)).astype(np.float32)
    codes = _e4m3_codes(keys / kscale[..., None]).reshape(num_blocks, bs * Di)
    k_cache[used, : bs * Di] = codes[used]
    sc_bytes = kscale.astype(np.float32).view(np.uint8).reshape(num_blocks, bs * 4)
    k_cache[used, bs * Di:] = sc_bytes[used]

    # latent KV cache: bf16 rows, unused blocks hold NaN
    kv_cache = np.empty((num_blocks, bs, Dk), dtype=np.uint16)
    for c0 in range(0, num_blocks, 1024):
        c1 = min(num_blocks, c0 + 1024)
        kv = rng.standard_normal((c1 - c0, bs, Dk), dtype=np.float32) * np.float32(spec["kv_std"])
        kv_cache[c0:c1] = _bf16_bits(kv)
    kv_cache[~used] = 0x7FC0

    kv_cache_fp8 = None
    if kv_fp8:
        # the same latent rows as an fp8 cache: per token, the Dv latent values
        # as e4m3 codes in groups of 128 with one fp32 scale each (amax/448,
        # codes from PyTorch's float8 cast), then the rope values' bf16 bits;
        # unused blocks hold e4m3 NaN bytes
        assert Dv % 128 == 0
        ng = Dv // 128
        row_bytes = Dv + 4 * ng + 2 * (Dk - Dv)
        kv_cache_fp8 = np.full((num_blocks, bs, row_bytes), 0x7F, dtype=np.uint8)
        for c0 in range(0, num_blocks, 1024):
            c1 = min(num_blocks, c0 + 1024)
            u = used[c0:c1]
            lat = bf16_bits_to_float(kv_cache[c0:c1][u, :, :Dv]).reshape(-1, bs, ng, 128)
            amax = np.abs(lat).max(axis=-1)
            scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
            codes = _e4m3_codes(lat / scale[..., None]).reshape(-1, bs, Dv)
            blk = np.empty((int(u.sum()), bs, row_bytes), dtype=np.uint8)
            blk[:, :, :Dv] = codes
            blk[:, :, Dv:Dv + 4 * ng] = np.ascontiguousarray(scale).view(np.uint8).reshape(-1, bs, 4 * ng)
            blk[:, :, Dv + 4 * ng:] = np.ascontiguousarray(kv_cache[c0:c1][u, :, Dv:]).view(np.uint8).reshape(
                -1, bs, 2 * (Dk - Dv))
            kv_cache_fp8[c0:c1][u] = blk

    q_idx = _bf16_bits(rng.standard_normal((T, Hi, Di), dtype=np.float32))
    w = (rng.standard_normal((T, Hi), dtype=np.float32) / np.float32(math.sqrt(Hi))).astype(np.float32)
    q = _bf16_bits(rng.standard_normal((T, H, Dk), dtype=np.float32) * np.float32(q_std))

    ld = int(max(seq_lens)) if Bn else 1
    ld = (ld + ld_pad - 1) // ld_pad * ld_pad

    return Workload(name=name, B=Bn, T=T, Hi=Hi, Di=Di, H=H, Dk=Dk, Dv=Dv, index_topk=spec["topk"], block_size=bs,
                    softmax_scale=1.0 / math.sqrt(Dk), seq_lens=seq_lens, query_start_loc=qsl,
                    block_table=block_table, num_blocks=num_blocks, k_block_stride=k_block_stride,
                    kv_block_stride=bs * Dk, ld=ld, q_idx=q_idx, w=w, k_cache=k_cache, q=q, kv_cache=kv_cache,
                    kv_cache_fp8=kv_cache_fp8)
