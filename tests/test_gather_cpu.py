"""The exchange of the gather + GEMM over ranks (all-gather matmul, batch-invariance test issue,
"Background"), on CPU: two and three gloo ranks each hold a row block of x with its own row
count (one of them empty); all_gather_rows returns every rank's block, in rank order, with its
rows and bytes intact, on every rank.  The multiplication itself runs on the GPU
(tests/test_gpu_k_gather.py); here the oracle checks that the gathered rows give each rank's
own rows of y (the row-wise definition the kernel relies on)."""
import multiprocessing as mp
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
K, N = 64, 24
ROWS = {2: [3, 5], 3: [4, 0, 7]}


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _block(rank, rows):
    import inputgen as ig
    return ig.normal_bf16(100 + rank, rows, K) if rows else np.zeros((0, K), np.uint16)


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    from invariant_bi_gemm_gb300.gather import all_gather_rows
    dist.init_process_group("gloo")
    x = torch.from_numpy(_block(rank, ROWS[world][rank]).view(np.int16)).view(torch.bfloat16)
    blocks = all_gather_rows(x)
    got = [b.view(torch.int16).numpy().view(np.uint16).copy() for b in blocks]
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, [g.shape[0] for g in got], [g.tobytes() for g in got]))


@pytest.mark.parametrize("world", [2, 3])
def test_all_gather_rows_rank_order_and_bytes(world):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    sys.path.insert(0, ROOT)
    import inputgen as ig  # noqa: F401
    import oracle
    want = [_block(r, ROWS[world][r]) for r in range(world)]
    w = ig.normal_bf16(ig.SEED_W, K, N, std=0.05)
    for rank, rows, data in out:
        assert rows == ROWS[world]
        for r in range(world):
            assert data[r] == want[r].tobytes(), (rank, r)
        # the gathered x, multiplied as one batch, gives each rank its own rows of y
        xg = np.concatenate([np.frombuffer(d, np.uint16).reshape(-1, K) for d in data])
        y_all = oracle.gemm_bf16(xg, w, "bf16")[0]
        off = 0
        for r in range(world):
            if ROWS[world][r]:
                y_own = oracle.gemm_bf16(want[r], w, "bf16")[0]
                assert np.array_equal(y_all[off:off + ROWS[world][r]], y_own)
            off += ROWS[world][r]
