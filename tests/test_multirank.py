"""The bench's multi-rank host path on two CPU ranks (gloo): rank discovery
from the launcher's environment, the barrier, the max-over-ranks step time,
the whole-job throughput of weak-scaled replicas, and the reference arm that
only rank 0 runs. No rank exchanges decode data (replicas only)."""
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    r, w, local = bench.dist_info()
    bench.dist_init(w, "gloo")
    bench.dist_barrier(w)
    # rank r measured (r + 1) ms per step; the job takes the slowest rank's time
    ms_max = bench.dist_max(float(r + 1), w)
    gbps = bench.whole_job_gbps(w, 1_000_000_000, ms_max)

    class Args:
        config, steps, warmup = "tiny_bf16", 1, 0

    ref = bench.run_reference(Args) if r != 0 else None   # only rank 0 runs (and prints) the oracle arm
    bench.dist_barrier(w)
    dist.destroy_process_group()
    out.put((r, w, local, ms_max, gbps, ref))


def test_two_ranks_gloo():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [x[:3] for x in res] == [(0, 2, 0), (1, 2, 1)]
    assert all(x[3] == 2.0 for x in res)                     # max over ranks
    assert all(abs(x[4] - 2 * 1.0 / 2e-3) < 1e-6 for x in res)  # 2 GB in 2 ms = 1000 GB/s
    assert res[1][5] is None                                 # rank 1 does no reference work


def test_single_rank_defaults(monkeypatch):
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    sys.path.insert(0, ROOT)
    import bench
    assert bench.dist_info() == (0, 1, 0)
    assert bench.dist_max(3.5, 1) == 3.5
    assert bench.whole_job_gbps(1, 6_000_000_000, 1.0) == pytest.approx(6000.0)
