"""Child process of tests/test_dist.py: one gloo rank running bench.py's
distributed helpers (barrier, max over ranks) on the CPU."""
import os
import sys


def run(rank, world, port, q):
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if root not in sys.path:
        sys.path.insert(0, root)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import bench
    d = bench.Dist("gloo")
    d.barrier()
    # each rank times a different amount of work; the job's time is the slowest rank's
    m = d.max(1.5 + rank * 10.0)
    d.barrier()
    q.put((rank, d.ws, d.rank, m))
    d.close()
