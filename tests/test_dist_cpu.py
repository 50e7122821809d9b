"""The N > 1 path of bench.py on CPU: two gloo ranks join the group the way `torchrun` starts
them, meet at the barrier, take the maximum of their timings (the whole-job clock), and only
rank 0 of the reference arm prints.  The GEMM itself has no exchange step (rows are
independent), so N GPUs run N replicas."""
import io
import multiprocessing as mp
import os
import socket
import sys
from contextlib import redirect_stdout

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank), BI_DIST_BACKEND="gloo")
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    r, w, local = bench.dist_init()
    bench.barrier(w)
    ms = bench.max_over_ranks(10.0 * (rank + 1), w)       # each rank's elapsed time
    par = bench.config_obj(w)["parallelism"]
    bench.barrier(w)
    dist.destroy_process_group()
    q.put((r, w, local, ms, par))


def test_two_gloo_ranks_share_the_max_clock():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [o[0] for o in out] == [0, 1] and all(o[1] == 2 for o in out)
    assert all(o[3] == 20.0 for o in out)              # max over ranks, the same on both
    assert all(o[4] == "replicas x2" for o in out)


def test_reference_arm_prints_on_rank_zero_only():
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        steps, warmup = 1, 1

    buf = io.StringIO()
    with redirect_stdout(buf):
        assert bench.run_reference(Args(), rank=1, world=2) is None
    assert buf.getvalue() == ""
