"""The replicated (N > 1) bench path on the host: two gloo ranks on 127.0.0.1
time different amounts and the job's figures must be the slowest rank's
time over every rank's tokens, identical on both ranks. No GPU: the op has
no collective of its own (every (sequence, head) chain is independent), so
the only multi-rank logic is this aggregation plus rank 0 alone printing."""
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


def _rank_main(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(ws), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        ms = [10.0, 12.5][rank]         # rank 1 is the slower replica
        ms_e2e = [20.0, 15.0][rank]     # rank 0 is slower end to end
        got = bench.aggregate_over_ranks(ms, ms_e2e, tokens_per_step=64, K=100, ws=ws,
                                         device=torch.device("cpu"))
        env = bench.dist_env()
        q.put((rank, got, env))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_max_time_and_all_tokens():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.SimpleQueue()
    procs = [ctx.Process(target=_rank_main, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict((r, (got, env)) for r, got, env in (q.get() for _ in range(ws)))
    tokens_all = 64 * 100 * ws
    for r in range(ws):
        (ms_max, ms_e2e_max, value, e2e), env = res[r]
        assert env == (ws, r, r)
        assert ms_max == 12.5 and ms_e2e_max == 20.0
        assert value == pytest.approx(tokens_all / 12.5e-3)
        assert e2e == pytest.approx(tokens_all / 20e-3)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    called = []

    class Wl:
        def __init__(self):
            called.append(1)

    # a non-zero rank returns 0 at once, without touching the oracle or a workload
    assert bench.reference_arm(None, Wl) == 0
