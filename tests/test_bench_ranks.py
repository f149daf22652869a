"""The benchmark's multi-rank path (weak scaling, no collective on the data
path) on CPU with two gloo ranks: timings are reduced with a max and the
whole-job value counts the tokens of every rank."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local = [10.0 + rank * 5.0, 3.0 - rank]
        got = bench.max_over_ranks(local)
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    world = 2
    mgr = mp.get_context("spawn").Manager()     # no fork: other tests may have started threads
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    assert out[0] == [15.0, 3.0] and out[1] == [15.0, 3.0]


def test_whole_job_rate_counts_all_ranks():
    assert bench.whole_job_rate(1000, 4, 2.0) == pytest.approx(2e6)
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]     # single process: identity


def test_traffic_digest_ignores_comments_only():
    """The DRAM-traffic line is keyed by the scan kernel's sources without
    comments: editing a comment keeps it, changing code does not."""
    src = 'int a = 1; // note\n/* block\n comment */ const char *s = "x//y";\n'
    assert bench._strip_comments(src) == 'int a = 1; const char *s = "x//y";'
    assert bench._strip_comments(src.replace("note", "other note")) == bench._strip_comments(src)
    assert bench._strip_comments(src.replace("a = 1", "a = 2")) != bench._strip_comments(src)
