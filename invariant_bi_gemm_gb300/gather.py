"""Row-block exchange for the gather + GEMM (all-gather matmul) over ranks.

Each rank holds a row block of x; ``all_gather_rows`` gathers every rank's block into this
process, in rank order, with ``torch.distributed`` (NCCL for CUDA tensors, gloo for CPU ones);
blocks may have different row counts.  ``BiGemm.run_gathered`` then copies the blocks into one
x in this GPU's memory and multiplies them with the handle's one kernel configuration, so a
row's bits do not depend on which rank it came from (the local-versus-gathered defect of the
batch-invariance test issue, "Background").  This module moves data only; no arithmetic of the
product runs here.
"""
from __future__ import annotations


def all_gather_rows(x_local, group=None):
    """Gather the [rows_r, ...] blocks of every rank of `group`; returns the list of blocks in
    rank order (views into one buffer), rank r's block with its own row count."""
    import torch
    import torch.distributed as dist

    world = dist.get_world_size(group)
    dtype = x_local.dtype
    dev = x_local.device
    # moved as raw bytes (the last dimension times the element size): every backend carries uint8
    shape_b = tuple(x_local.shape[:-1]) + (int(x_local.shape[-1]) * x_local.element_size(),)
    if x_local.numel():
        x_local = x_local.contiguous().view(torch.uint8)
    else:
        x_local = torch.empty(shape_b, dtype=torch.uint8, device=dev)
    n = torch.tensor([int(x_local.shape[0])], dtype=torch.int64, device=dev)
    counts = [torch.zeros_like(n) for _ in range(world)]
    dist.all_gather(counts, n, group=group)
    rows = [int(c.item()) for c in counts]
    cap = max(rows)
    tail = tuple(x_local.shape[1:])
    padded = torch.zeros((cap,) + tail, dtype=x_local.dtype, device=dev)
    if rows[dist.get_rank(group)] > 0:
        padded[: x_local.shape[0]] = x_local
    out = torch.empty((world * cap,) + tail, dtype=x_local.dtype, device=dev)
    parts = list(out.view((world, cap) + tail).unbind(0))
    dist.all_gather(parts, padded, group=group)
    return [parts[r][: rows[r]].view(dtype) for r in range(world)]


__all__ = ["all_gather_rows"]
