"""Helpers shared by the GPU tests: host<->device marshalling of raw bit patterns, the
tolerance check against the oracle, and the byte-diff batch-invariance harness (bi_check).

bi_check follows the cell contract of the batch-invariance test issue ("Test methodology"):
variant A fixes target row i to content C and draws the other rows from seed_A, variant B
the same with seed_B, and the cell passes only if byte(y_A[i]) == byte(y_B[i]); the cell's
result is a byte-diff count, and any count > 0 fails ("ATK integration", item 3).
"""
from __future__ import annotations

import ctypes

import numpy as np
import torch

import inputgen as ig
import oracle
from invariant_bi_gemm_gb300 import build as bgbuild

DEV = "cuda"


def dev_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(DEV).view(torch.bfloat16)


def dev_u8(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).to(DEV)


def host_bits(y: torch.Tensor) -> np.ndarray:
    """Raw output: uint16 bf16 patterns or float32 values."""
    if y.dtype == torch.bfloat16:
        return y.view(torch.int16).cpu().numpy().view(np.uint16)
    return y.cpu().numpy()


def to_f64(y: np.ndarray) -> np.ndarray:
    if y.dtype == np.uint16:
        return oracle.bf16_array_to_f64(y)
    return y.astype(np.float64)


def byte_diffs(a: np.ndarray, b: np.ndarray) -> int:
    a = np.ascontiguousarray(a).view(np.uint8)
    b = np.ascontiguousarray(b).view(np.uint8)
    assert a.shape == b.shape
    return int(np.count_nonzero(a != b))


def oracle_rows(fn, rows, chunks=None):
    """Run an oracle call `fn(rows) -> (y, acc, sabs)` over `rows` split across host threads (the
    C oracle releases the interpreter lock; rows are independent, so the result is the same as one
    call) and stack the pieces in the order of `rows`."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    rows = np.asarray(list(rows), dtype=np.int64)
    n = chunks or max(1, min(len(rows), os.cpu_count() or 1))
    parts = [np.arange(i, len(rows), n) for i in range(n)]
    parts = [p for p in parts if p.size]
    with ThreadPoolExecutor(max_workers=len(parts)) as ex:
        outs = list(ex.map(lambda p: fn(rows[p]), parts))
    res = []
    for k in range(3):
        first = outs[0][k]
        full = np.empty((len(rows),) + first.shape[1:], dtype=first.dtype)
        for p, o in zip(parts, outs):
            full[p] = o[k]
        res.append(full)
    return tuple(res)


def check_tolerance(y_gpu: np.ndarray, y_ref: np.ndarray, sabs: np.ndarray, tol: float, what: str):
    """|y - y_ref| <= tol * S_abs elementwise; returns the max ratio for reporting."""
    bad, ratio = oracle.tolerance_violations(to_f64(y_gpu), to_f64(y_ref), sabs, tol)
    assert bad == 0, f"{what}: {bad} elements outside {tol:g}*S_abs (max ratio {ratio:.3g})"
    return ratio


def bi_check(run, rows_a: torch.Tensor, rows_b: torch.Tensor, content: torch.Tensor, M: int,
             golden_row: np.ndarray | None = None):
    """Run the A/B cells for targets {0, mid, last} at batch size M.

    run(x) -> y (device tensors); rows_a / rows_b hold at least M rows drawn from seed_A /
    seed_B; content is the fixed row C.  Returns a list of (target, diffs_AB, diffs_golden)
    where diffs_golden compares y_A[target] against `golden_row` (C's row at M = 1) if given.
    """
    out = []
    for t in ig.target_rows(M):
        xa = rows_a[:M].clone()
        xa[t] = content
        xb = rows_b[:M].clone()
        xb[t] = content
        ya = host_bits(run(xa)[t:t + 1])
        yb = host_bits(run(xb)[t:t + 1])
        dg = byte_diffs(ya, golden_row) if golden_row is not None else 0
        out.append((t, byte_diffs(ya, yb), dg))
    return out


class Controls:
    """ctypes view of the test-only libbi_gemm_controls.so (tests/include/bi_gemm_controls.h)."""

    def __init__(self):
        L = ctypes.CDLL(bgbuild.lib_path("libbi_gemm_controls.so"))
        P, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.bi_ctl_create.argtypes = [ctypes.POINTER(P), I64, I64, I32, I32, ctypes.c_int32, ctypes.c_uint64]
        L.bi_ctl_destroy.argtypes = [P]
        L.bi_ctl_get_device_error.argtypes = [P, P]
        L.bi_ctl_run.argtypes = [P, P, I64, P, P, P, P]
        L.bi_ctl_msplit_count.argtypes = [P, I64]
        L.bi_ctl_run_msplit.argtypes = [P, P, I64, P, P, P, P]
        L.bi_ctl_run_smallm_fork.argtypes = [P, P, I64, P, P, P]
        L.bi_ctl_run_stall.argtypes = [P, P, I64, P, P, P, P]
        L.bi_ctl_run_skip_arrival.argtypes = [P, P, I64, P, P, P, P]
        L.bi_ctl_rmsnorm_f32.argtypes = [P, I64, I64, P, ctypes.c_float, P, ctypes.c_int32, P]
        L.bi_ctl_attention_stall.argtypes = [P, P, I64, P, P, P, P, I64, P, I64, I64, I64, P, ctypes.c_uint64, P]
        L.bi_ctl_attention_create.argtypes = [ctypes.POINTER(P), I64, I64, I64, I64, ctypes.c_float, I64]
        L.bi_ctl_attention_run.argtypes = [P, P, I64, P, P, P, P, I64, P, I64, I64, I64, P, P]
        L.bi_ctl_attention_get_device_error.argtypes = [P, P]
        L.bi_ctl_attention_destroy.argtypes = [P]
        L.bi_ctl_attention_run_kernel.argtypes = [P, P, I64, P, P, P, P, I64, P, I64, I64, I64, P, ctypes.c_int32, P]
        for n in ("bi_ctl_create", "bi_ctl_destroy", "bi_ctl_get_device_error", "bi_ctl_run",
                  "bi_ctl_msplit_count", "bi_ctl_run_msplit", "bi_ctl_run_smallm_fork", "bi_ctl_run_stall",
                  "bi_ctl_run_skip_arrival", "bi_ctl_rmsnorm_f32", "bi_ctl_attention_stall", "bi_ctl_attention_create",
                  "bi_ctl_attention_run", "bi_ctl_attention_get_device_error", "bi_ctl_attention_destroy",
                  "bi_ctl_attention_run_kernel"):
            getattr(L, n).restype = I32
        self.L = L

    def create(self, K, N, dtype, layout=0, split_k=0, timeout_ns=0):
        h = ctypes.c_void_p()
        rc = self.L.bi_ctl_create(ctypes.byref(h), K, N, dtype, layout, split_k, timeout_ns)
        assert rc == 0, rc
        return h.value


def stream_ptr() -> int:
    return torch.cuda.current_stream().cuda_stream
