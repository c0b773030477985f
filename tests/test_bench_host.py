"""CPU checks of bench.py's host logic: algorithmic byte counts and the
max-over-ranks timing reduction of the replicated (N > 1) run, on two gloo
ranks."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def test_algorithmic_bytes_of_the_named_shapes():
    # CQ 2-bit 32768 x 512, group 128: packed + norms + codebook + x + y
    assert bench.cq_matvec_bytes(32768, 512, 128, 2) == 4_589_584
    assert bench.cq_matvec_bytes(512, 512, 64, 4) == 143_424
    assert [bench.cq_matvec_bytes(2048, 512, 64, b) for b in (2, 3, 4, 5)] == \
        [305_168, 436_256, 567_360, 698_496]
    assert bench.cq_matvec_bytes(2048, 512, 64, 2, batch=4) == 335_888
    # F8 E4M3 head 245760 x 4096 with scales [1920, 32]
    assert bench.f8_bytes(245760, 4096, 1920, 32) == 1_007_693_824
    assert bench.f8_bytes(4096, 4096, 32, 32) == 16_811_008
    assert bench.f8_bytes(245760, 4096, 1920, 32, batch=8) == 1_014_689_792


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    w, r, _ = bench.dist_env()
    d = bench.init_dist(w, "gloo")
    bench.barrier(d)
    got = bench.max_over_ranks(0.5 + rank, d)
    q.put((rank, got))
    d.destroy_process_group()


def test_max_over_ranks_on_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 1.5, 1: 1.5}


def test_single_rank_reduction_is_identity():
    assert bench.max_over_ranks(2.25, None) == 2.25
