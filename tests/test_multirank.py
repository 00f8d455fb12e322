"""The N > 1 host path of bench.py on CPU: two gloo ranks on 127.0.0.1.

Every rank runs its own part of the batch (no data-path collective; the split itself
is checked in tests/test_shard.py); ranks only agree on the timing and the totals: a
barrier around the timed region, the maximum elapsed time over ranks and the sum of
the bytes they moved.  The reference arm runs on rank 0 alone; other ranks exit
without work.
"""
from __future__ import annotations

import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    w, r, local = bench.dist_env()
    assert (w, r, local) == (world, rank, rank)
    dist = bench.init_dist(world, "gloo")
    bench.barrier(dist)
    # each rank reports a different elapsed time; all must agree on the largest
    got = bench.max_over_ranks(1.0 + rank * 0.25, dist)
    # ... and on the bytes all of them moved: each rank's own part of the batch
    spec = bench.workloads.get_spec("many_small")
    part, ps = bench.rank_part(spec, world, rank)
    total = bench.sum_over_ranks(float(bench.step_bytes(ps)), dist)
    bench.barrier(dist)
    out.put((rank, (got, total, part.requests[0], part.requests[-1])))
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_max_elapsed_time_and_the_bytes_moved():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res[0][0] == res[1][0] == 1.25
    # the parts' bytes add up to the whole batch's step, and the parts follow each other
    spec = bench.workloads.get_spec("many_small")
    assert res[0][1] == res[1][1] == float(bench.step_bytes(spec))
    assert res[0][2] == 0 and res[1][2] == res[0][3] + 1 and res[1][3] == spec.n_req - 1


def test_single_rank_needs_no_process_group():
    assert bench.init_dist(1, "gloo") is None
    assert bench.max_over_ranks(3.5, None) == 3.5


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    assert bench.main(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"]) == 0
    assert capsys.readouterr().out == ""


def test_warmup_below_three_is_refused():
    with pytest.raises(SystemExit):
        bench.parse_args(["--warmup", "2"])
