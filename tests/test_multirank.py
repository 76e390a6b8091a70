"""Cross-rank timing logic of bench.py on CPU with two gloo ranks: every rank
reports its own step time and rank 0 takes the maximum (weak scaling: each
rank runs a full copy of the workload; the dense path has no collective)."""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    w, r, _ = bench.dist_setup()
    assert (w, r) == (world, rank)
    bench.barrier(w)
    t = bench.reduce_max(1.5 + rank, w)
    out[rank] = t
    import torch.distributed as dist
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max_time():
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    assert dict(out) == {0: 2.5, 1: 2.5}


def test_deterministic_mode_guard_on_host():
    import softmax_attention_backward_gb300 as A
    torch.use_deterministic_algorithms(True)
    try:
        x = torch.zeros(1)
        with pytest.raises(RuntimeError, match="not bitwise reproducible; use dq_mode=ATTN_DQ_SPLIT"):
            A.attn_bwd(x, x, x, x, x, x, mode=A.ATTN_DQ_ATOMIC, workspace=x)
        with pytest.raises(RuntimeError, match="not bitwise reproducible; use sparse_attn_bwd_deterministic"):
            A.sparse_attn_bwd(x, x, x, x, x, x)
        # the reproducible paths pass the guard (and fail later on the dummy tensors)
        for call in (lambda: A.attn_bwd(x, x, x, x, x, x, mode=A.ATTN_DQ_SPLIT, workspace=x),
                     lambda: A.sparse_attn_bwd_deterministic(x, x, x, x, x, x)):
            with pytest.raises(Exception) as e:
                call()
            assert "bitwise" not in str(e.value)
    finally:
        torch.use_deterministic_algorithms(False)
