"""The N > 1 path of bench.py on CPU ranks (gloo, world size 2): replicas that
share nothing on the data path; the host side only synchronises and takes the
maximum time over ranks, which these tests check."""
import multiprocessing as mp
import socket

import pytest

import _dist_worker

pytestmark = pytest.mark.cpu


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("world", [2, 3])
def test_max_over_ranks_with_gloo(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_dist_worker.run, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in results] == list(range(world))
    assert all(r[1] == world for r in results)
    # every rank sees the slowest rank's time
    assert all(r[3] == 1.5 + (world - 1) * 10.0 for r in results)


def test_single_process_is_rank_zero(monkeypatch):
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    d = bench.Dist("gloo")
    assert (d.ws, d.rank, d.local) == (1, 0, 0)
    assert d.max(3.25) == 3.25
    d.barrier()
    d.close()
