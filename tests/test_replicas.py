"""The multi-GPU path runs independent replicas; only the timing bookkeeping
crosses ranks. World-size-2 gloo run on CPU."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from deepseek_sparse_attention_fp8_gb300.replicas import aggregate

    ms_local = [0.25, 0.40][rank]
    tokens_local = [32, 32][rank]
    ms, tokens, value = aggregate(ms_local, tokens_local)
    out[rank] = (ms, tokens, value)
    dist.barrier()
    dist.destroy_process_group()


def test_two_replicas_take_the_slowest_rank_and_add_tokens():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()  # no fork of this (multi-threaded) process
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    for rank in range(world):
        ms, tokens, value = out[rank]
        assert ms == 0.40
        assert tokens == 64
        assert abs(value - 64 / 0.40e-3) < 1e-6 * value
    mgr.shutdown()


def test_single_process_is_unchanged():
    from deepseek_sparse_attention_fp8_gb300.replicas import aggregate

    ms, tokens, value = aggregate(0.5, 32)
    assert (ms, tokens) == (0.5, 32) and abs(value - 64000.0) < 1e-9
