"""bi_gemm_run_noalloc: the allocation-free entry point, for callers that may not allocate device
memory when they run a GEMM (their device memory is owned by another framework's pool, or the
call sits in a loop that must not enter the allocator).  Its split-K scratch lives in the
library's fixed per-device array instead of a workspace grown with cudaMallocAsync.

The test calls it through the C ABI on the split-K handle of the small-N long-K workload
(K=16384, N=24, S=32) and checks two calls in a row against bi_gemm_run on the same inputs:
within the fp32 tolerance the other tests use, and byte for byte (same kernel, same
configuration).  It also checks that a run too large for the fixed array is refused.  This
file is collected last, so a run that stops at the first failure has run everything else."""
import ctypes

import numpy as np
import pytest
import torch

import inputgen as ig
import oracle
import invariant_bi_gemm_gb300 as bg
from gpu_util import dev_bf16, host_bits, stream_ptr

pytestmark = pytest.mark.gpu

K, N = 16384, 24


def _call(L, h, x, M, w, y, s):
    return L.bi_gemm_run_noalloc(ctypes.c_void_p(h), ctypes.c_void_p(x.data_ptr()), M,
                                 ctypes.c_void_p(w.data_ptr()), None, ctypes.c_void_p(y.data_ptr()),
                                 ctypes.c_void_p(s))


def test_noalloc_matches_bi_gemm_run_twice():
    L = bg.library()
    M = 200
    x_np = ig.scaled_rows_bf16(ig.SEED_X, M, K)
    w_np = ig.normal_bf16(ig.SEED_W, K, N, std=0.02)
    x, w = dev_bf16(x_np), dev_bf16(w_np)
    h = bg.bi_gemm_create(K, N, bg.BI_BF16_OUT_F32)
    try:
        assert bg.bi_gemm_get_config(h)["split_k"] == 32      # the path that needs scratch
        s = stream_ptr()
        y_ref = torch.empty((M, N), dtype=torch.float32, device="cuda")
        bg.bi_gemm_run(h, x.data_ptr(), M, w.data_ptr(), None, y_ref.data_ptr(), s)
        ref = host_bits(y_ref)
        # |y_noalloc - y_run| <= 1e-5 * S_abs with S_abs from the oracle, on two calls in a row
        _, _, sabs = oracle.gemm_bf16(x_np, w_np, "f32")
        for _ in range(2):
            y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
            assert _call(L, h, x, M, w, y, s) == bg.BI_GEMM_OK
            got = host_bits(y)
            bad, ratio = oracle.tolerance_violations(got.astype(np.float64), ref.astype(np.float64), sabs,
                                                     oracle.TOL_F32)
            assert bad == 0, f"{bad} elements differ from bi_gemm_run beyond tolerance (max ratio {ratio:.3g})"
            assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
        assert bg.bi_gemm_get_device_error(h, s) == bg.BI_GEMM_OK
    finally:
        bg.bi_gemm_destroy(h)


def test_noalloc_refuses_runs_beyond_its_scratch():
    L = bg.library()
    M = 1024                          # 8 tiles x 32 splits x 128 x 64 x 4 B = 8 MiB > 8 MiB - 4 KiB
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((K, N), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    h = bg.bi_gemm_create(K, N, bg.BI_BF16_OUT_F32)
    try:
        assert _call(L, h, x, M, w, y, stream_ptr()) == bg.BI_GEMM_ERR_SCRATCH_LIMIT
        assert "scratch" in bg.bi_gemm_strerror(bg.BI_GEMM_ERR_SCRATCH_LIMIT)
        assert bg.bi_gemm_get_device_error(h, stream_ptr()) == bg.BI_GEMM_OK
    finally:
        bg.bi_gemm_destroy(h)
