"""bi_gemm_run_noalloc: the allocation-free entry point, for callers that may not allocate device
memory when they run a GEMM (their device memory is owned by another framework's pool, or the
call sits in a loop that must not enter the allocator).  Its split-K scratch lives in the
library's fixed per-device array instead of a workspace grown with cudaMallocAsync.

Every case calls it through the C ABI on a fresh handle that only this entry point touches, so
that no workspace of the handle can stand in for the array, and checks two calls in a row:
byte for byte against bi_gemm_run on a second handle of the same configuration (same kernel),
within the tolerance of the other tests against the oracle, and with the device's free memory
unchanged across the calls.  The cases cover both merge paths of the split-K kernel (the last
CTA to arrive merges alone; the split CTAs share the merge), the largest run the array accepts,
a split CTA-pair MXFP8 tile, and the refusal of a run one tile too large.  This file is
collected last, so a run that stops at the first failure has run everything else."""
import ctypes

import numpy as np
import pytest
import torch

import inputgen as ig
import oracle
import invariant_bi_gemm_gb300 as bg
from gpu_util import dev_bf16, dev_u8, host_bits, stream_ptr

pytestmark = pytest.mark.gpu

K, N = 16384, 24      # the small-N long-K workload: S = 32, 128 x 64 tiles on single CTAs


def _noalloc(L, h, x, M, w, y, s, scales=None):
    sc = ctypes.byref(scales) if scales is not None else None
    return L.bi_gemm_run_noalloc(ctypes.c_void_p(h), ctypes.c_void_p(x.data_ptr()), M,
                                 ctypes.c_void_p(w.data_ptr()), sc, ctypes.c_void_p(y.data_ptr()),
                                 ctypes.c_void_p(s))


def _free_bytes():
    torch.cuda.synchronize()
    return torch.cuda.mem_get_info()[0]


def _run_case(K, N, dtype, M, x, w, ref_f64, sabs, tol, split_k=0, scales=None, out_dtype=torch.float32,
              expect_coop=None):
    """noalloc twice on a fresh handle vs bi_gemm_run on another handle; returns the merge path."""
    L = bg.library()
    s = stream_ptr()
    opts = bg.bi_gemm_options(split_k, 0, 0, 0, 0) if split_k else None
    layout = bg.BI_SCALES_E8M0_K32 if scales is not None else bg.BI_SCALES_NONE
    h_ref = bg.bi_gemm_create(K, N, dtype, layout, opts)
    h = bg.bi_gemm_create(K, N, dtype, layout, opts)
    try:
        cfg = bg.bi_gemm_get_config(h)
        assert cfg["split_k"] > 1                                  # the path that needs scratch
        units = -(-M // cfg["block_m"]) * -(-N // cfg["block_n"]) * cfg["split_k"]
        coop = units <= cfg["max_groups"]
        y_ref = torch.empty((M, N), dtype=out_dtype, device="cuda")
        bg.bi_gemm_run(h_ref, x.data_ptr(), M, w.data_ptr(), scales, y_ref.data_ptr(), s)
        ref = host_bits(y_ref)
        ys = [torch.full((M, N), float("nan"), dtype=out_dtype, device="cuda") for _ in range(2)]
        before = _free_bytes()
        for y in ys:
            assert _noalloc(L, h, x, M, w, y, s, scales) == bg.BI_GEMM_OK
        after = _free_bytes()
        assert after == before, f"device free memory changed by {before - after} bytes across the calls"
        for y in ys:
            got = host_bits(y)
            assert np.array_equal(got.view(np.uint8), ref.view(np.uint8)), "differs from bi_gemm_run"
            got_f64 = oracle.bf16_array_to_f64(got) if got.dtype == np.uint16 else got.astype(np.float64)
            bad, ratio = oracle.tolerance_violations(got_f64, ref_f64, sabs, tol)
            assert bad == 0, f"{bad} elements outside the oracle tolerance (max ratio {ratio:.3g})"
        assert bg.bi_gemm_get_device_error(h, s) == bg.BI_GEMM_OK
        assert bg.bi_gemm_get_device_error(h_ref, s) == bg.BI_GEMM_OK
        return coop
    finally:
        bg.bi_gemm_destroy(h)
        bg.bi_gemm_destroy(h_ref)


@pytest.fixture(scope="module")
def small_n_long_k():
    x_np = ig.scaled_rows_bf16(ig.SEED_X, 896, K)
    w_np = ig.normal_bf16(ig.SEED_W, K, N, std=0.02)
    return x_np, w_np, dev_bf16(x_np), dev_bf16(w_np)


# M = 8: one CTA merges (a small sub-tile); 200: the split CTAs share the merge; 640: more split
# units than resident CTAs, so the last CTA to arrive merges; 896: 7 tiles x 32 splits x 32 KiB,
# the largest run that fits the array.
@pytest.mark.parametrize("M,coop", [(8, None), (200, True), (640, False), (896, False)])
def test_noalloc_small_n_long_k(small_n_long_k, M, coop):
    x_np, w_np, x, w = small_n_long_k
    y_ref, _, sabs = oracle.gemm_bf16(x_np[:M], w_np, "f32")
    got_coop = _run_case(K, N, bg.BI_BF16_OUT_F32, M, x[:M], w, y_ref.astype(np.float64), sabs, oracle.TOL_F32)
    if coop is not None:
        assert got_coop == coop


def test_noalloc_mxfp8_pair_tile_split():
    Kf, Nf, M = 2048, 256, 300        # 256 x 256 pair tiles, S = 4: 4 sub-tiles x 4 x 128 KiB = 2 MiB
    x_np = ig.normal_e4m3(ig.SEED_X, M, Kf)
    sx_np = ig.e8m0_scales("VAR", ig.SEED_X, M, Kf // 32)
    w_np = ig.normal_e4m3(ig.SEED_W, Kf, Nf)
    sw_np = ig.e8m0_scales("VAR", ig.SEED_W, Kf // 32, Nf)
    x, sx, w, sw = dev_u8(x_np), dev_u8(sx_np), dev_u8(w_np), dev_u8(sw_np)
    sc = bg.bi_gemm_scales(sx.data_ptr(), sw.data_ptr())
    y_ref, _, sabs = oracle.gemm_mxfp8(x_np, sx_np, w_np, sw_np)
    _run_case(Kf, Nf, bg.BI_MXFP8E4M3_OUT_BF16, M, x, w, oracle.bf16_array_to_f64(y_ref), sabs, oracle.TOL_BF16,
              split_k=4, scales=sc, out_dtype=torch.bfloat16)


def test_noalloc_refuses_runs_beyond_its_scratch():
    L = bg.library()
    M = 897                           # 8 tiles x 32 splits x 128 x 64 x 4 B = 8 MiB > 8 MiB - 4 KiB
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((K, N), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    h = bg.bi_gemm_create(K, N, bg.BI_BF16_OUT_F32)
    try:
        assert _noalloc(L, h, x, M, w, y, stream_ptr()) == bg.BI_GEMM_ERR_SCRATCH_LIMIT
        assert "scratch" in bg.bi_gemm_strerror(bg.BI_GEMM_ERR_SCRATCH_LIMIT)
        assert bg.bi_gemm_get_device_error(h, stream_ptr()) == bg.BI_GEMM_OK
    finally:
        bg.bi_gemm_destroy(h)
