"""bench.py's multi-rank host logic on CPU: two gloo ranks (one process each) combine
their timings as the whole-job numbers (slowest rank's times, summed tokens), and each
rank draws its own batch. No GPU."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        ms = [10.0, 12.5][rank]
        tokens = [320, 288][rank]
        e2e_s = [0.5, 0.4][rank]
        e2e_tok = [640, 600][rank]
        q.put((rank, bench.combine_ranks(ms, tokens, e2e_s, e2e_tok, world, "cpu")))
    finally:
        dist.destroy_process_group()


def test_two_ranks_combine_on_gloo():
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
    for r in (0, 1):
        assert res[r] == pytest.approx((12.5, 608.0, 0.5, 1240.0))


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.combine_ranks(3.0, 7, 1.5, 9, 1, "cpu") == (3.0, 7.0, 1.5, 9.0)


def test_each_rank_draws_its_own_batch():
    sys.path.insert(0, ROOT)
    import bench
    from synth import CONFIGS, make_prompts
    cfg = CONFIGS["b32"]
    p0 = make_prompts(bench.rank_config(cfg, 0))
    p1 = make_prompts(bench.rank_config(cfg, 1))
    assert bench.rank_config(cfg, 0) is cfg
    assert len(p0) == len(p1) == cfg.batch
    assert any(len(a) != len(b) or (a != b).any() for a, b in zip(p0, p1))
