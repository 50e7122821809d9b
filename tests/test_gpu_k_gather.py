"""Gather + GEMM over ranks (the all-gather matmul of the batch-invariance test issue,
"Background"; its test matrix, "Test methodology": world sizes 2, 4 and 8) through
bi_gemm_run_gathered on one GPU: the ranks' row blocks are separate device buffers, gathered
into one x and multiplied with the handle's one kernel configuration.  Checks: the gathered x
is the blocks' bytes in order; every row's output is bitwise the one its block gives alone
(LOCAL) and the one the concatenated batch gives through bi_gemm_run (GATHER); every element
against the oracle; MXFP8 with K-varying scales; empty and ragged blocks; bad block tables."""
import ctypes

import numpy as np
import pytest
import torch

import inputgen as ig
import invariant_bi_gemm_gb300 as bg
import oracle
from gpu_util import check_tolerance, dev_bf16, dev_u8, host_bits, stream_ptr
from invariant_bi_gemm_gb300 import BiGemm

pytestmark = pytest.mark.gpu


def _blocks_bf16(rows, K, seed0=200):
    return [ig.normal_bf16(seed0 + r, n, K) if n else np.zeros((0, K), np.uint16) for r, n in enumerate(rows)]


@pytest.mark.parametrize("ws,mr", [(2, 1), (2, 64), (4, 8), (4, 17), (8, 16), (8, 64)])
def test_gathered_bf16_equals_local_and_concatenated(ws, mr):
    K, N = 4096, 1024
    rows = [mr + (r % 3) for r in range(ws)]               # ragged: blocks differ in rows
    xs = _blocks_bf16(rows, K)
    w = ig.normal_bf16(ig.SEED_W, K, N, std=0.02)
    g = BiGemm(K, N, "bf16")
    wd = dev_bf16(w)
    blocks = [dev_bf16(x) for x in xs]
    y, x_out, _ = g.run_gathered(blocks, wd)
    xcat = np.concatenate(xs)
    assert np.array_equal(host_bits(x_out), xcat)                      # the gather moves bytes only
    y_cat = host_bits(g(dev_bf16(xcat), wd))
    got = host_bits(y)
    assert np.array_equal(got, y_cat)                                  # GATHER path == one batch
    off = 0
    for r, x in enumerate(xs):
        y_loc = host_bits(g(blocks[r], wd))                            # LOCAL path: the block alone
        assert np.array_equal(got[off:off + len(x)], y_loc), r
        off += len(x)
    y_ref, _, sabs = oracle.gemm_bf16(xcat, w, "bf16")
    check_tolerance(got, y_ref, sabs, oracle.TOL_BF16, f"gathered ws={ws}")
    assert g.device_error() == 0
    g.close()


@pytest.mark.parametrize("ws,mr", [(2, 4), (4, 32), (8, 8)])
def test_gathered_mxfp8_k_varying_scales(ws, mr):
    K, N = 2048, 512
    rows = [mr] * ws
    xs = [ig.normal_e4m3(300 + r, mr, K) for r in range(ws)]
    sxs = [ig.e8m0_scales("VAR", 300 + r, mr, K // 32) for r in range(ws)]
    w = ig.normal_e4m3(ig.SEED_W, K, N)
    sw = ig.e8m0_scales("VAR", ig.SEED_W, K // 32, N)
    g = BiGemm(K, N, "mxfp8")
    wd, swd = dev_u8(w), dev_u8(sw)
    blocks, sblocks = [dev_u8(x) for x in xs], [dev_u8(s) for s in sxs]
    y, x_out, sx_out = g.run_gathered(blocks, wd, sx_blocks=sblocks, sw=swd)
    xcat, sxcat = np.concatenate(xs), np.concatenate(sxs)
    assert np.array_equal(x_out.cpu().numpy(), xcat) and np.array_equal(sx_out.cpu().numpy(), sxcat)
    got = host_bits(y)
    assert np.array_equal(got, host_bits(g(dev_u8(xcat), wd, sx=dev_u8(sxcat), sw=swd)))
    for r in range(ws):
        y_loc = host_bits(g(blocks[r], wd, sx=sblocks[r], sw=swd))
        assert np.array_equal(got[r * mr:(r + 1) * mr], y_loc), r
    y_ref, _, sabs = oracle.gemm_mxfp8(xcat, sxcat, w, sw)
    check_tolerance(got, y_ref, sabs, oracle.TOL_BF16, f"gathered MXFP8 ws={ws}")
    assert g.device_error() == 0
    g.close()


def test_gathered_empty_blocks_and_bad_tables():
    K, N = 256, 128
    g = BiGemm(K, N, "bf16")
    xs = _blocks_bf16([0, 5, 0, 3], K)
    w = ig.normal_bf16(ig.SEED_W, K, N, std=0.05)
    wd = dev_bf16(w)
    blocks = [dev_bf16(x) if len(x) else torch.empty((0, K), dtype=torch.bfloat16, device="cuda") for x in xs]
    y, _, _ = g.run_gathered(blocks, wd)
    assert np.array_equal(host_bits(y), host_bits(g(dev_bf16(np.concatenate(xs)), wd)))
    L = bg.library()
    x_out = torch.empty((8, K), dtype=torch.bfloat16, device="cuda")
    y_out = torch.empty((8, N), dtype=torch.bfloat16, device="cuda")
    def call(arr, n):
        return L.bi_gemm_run_gathered(ctypes.c_void_p(g.handle), arr, n, ctypes.c_void_p(x_out.data_ptr()), None,
                                      ctypes.c_void_p(wd.data_ptr()), None, ctypes.c_void_p(y_out.data_ptr()),
                                      ctypes.c_void_p(stream_ptr()))
    arr = (bg.bi_gemm_block * 2)()
    arr[0].x, arr[0].rows = blocks[1].data_ptr(), 5
    arr[1].x, arr[1].rows = blocks[3].data_ptr(), -1                  # negative rows
    assert call(arr, 2) == bg.BI_GEMM_ERR_INVALID_ARG
    arr[1].rows = 3
    assert call(arr, 0) == bg.BI_GEMM_ERR_INVALID_ARG                 # no blocks
    assert call(arr, 257) == bg.BI_GEMM_ERR_INVALID_ARG               # more than the table holds
    arr[1].x = blocks[3].data_ptr() + 2                                # misaligned block
    assert call(arr, 2) == bg.BI_GEMM_ERR_ALIGNMENT
    arr[1].x = blocks[3].data_ptr()
    assert call(arr, 2) == bg.BI_GEMM_OK
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(y_out), host_bits(y)[0:8])
    assert g.device_error() == 0
    g.close()
