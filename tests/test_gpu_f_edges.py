"""Edge cases: empty batch, ragged tails in M, N and K, guard bands around the output (no
write outside [0, M) x [0, N)), a very large M, argument errors, weight-pointer changes."""
import ctypes

import numpy as np
import pytest
import torch

import inputgen as ig
import oracle
from gpu_util import check_tolerance, dev_bf16, host_bits, stream_ptr
import invariant_bi_gemm_gb300 as bg
from invariant_bi_gemm_gb300 import BiGemm, BiGemmError

pytestmark = pytest.mark.gpu


def test_empty_batch_is_noop():
    g = BiGemm(256, 128, "bf16")
    bg.bi_gemm_run(g.handle, 0, 0, 0, None, 0, stream_ptr())   # M = 0 with null pointers
    assert g.device_error() == 0
    g.close()


@pytest.mark.parametrize("K,N,kind,M", [
    (200, 200, "bf16", 131),       # K, N and M all ragged (K not a multiple of 64)
    (72, 8, "bf16_f32", 5),        # smallest N, tiny K
    (1032, 264, "bf16", 257),      # N just above one 256 tile
    (4096, 520, "bf16_f32", 300),
    (8, 64, "bf16", 1),            # K = 8: one partial k-block
    (1024, 4000, "bf16", 300),     # N ends inside the second (peer) half of the last pair tile
    (1024, 4000, "bf16_f32", 77),
    # pair tile at M <= 64 (stages of two k-blocks): an odd k-block count (the last stage holds
    # one), a partial last k-block, a single k-block, a single stage, ragged N
    (1032, 264, "bf16", 57),
    (200, 200, "bf16", 13),
    (8, 264, "bf16", 1),
    (72, 264, "bf16_f32", 3),
    (4096, 520, "bf16_f32", 64),
    # more N tiles than CTA pairs (80 and 81 tiles on 76 pairs): some pairs run two tiles, in
    # both pipelines, the second tile's accumulator double-buffered behind the first
    (512, 20480, "bf16", 40),
    (520, 20488, "bf16_f32", 64),
    (512, 20480, "bf16", 200),
])
def test_ragged_shapes(K, N, kind, M):
    x = ig.normal_bf16(21, M, K)
    w = ig.normal_bf16(22, K, N, std=0.05)
    out = "f32" if kind == "bf16_f32" else "bf16"
    y_ref, _, sabs = oracle.gemm_bf16(x, w, out)
    g = BiGemm(K, N, kind)
    y = host_bits(g(dev_bf16(x), dev_bf16(w)))
    check_tolerance(y, y_ref, sabs, oracle.TOL_F32 if out == "f32" else oracle.TOL_BF16, f"{K},{N},{M}")
    g.close()


@pytest.mark.parametrize("kind,N,split,M", [("bf16", 200, 0, 77), ("bf16_f32", 24, 0, 77), ("bf16_f32", 40, 4, 77),
                                            ("bf16", 520, 0, 33)])
def test_guard_bands(kind, N, split, M):
    K = 1024
    x = dev_bf16(ig.normal_bf16(31, M, K))
    w = dev_bf16(ig.normal_bf16(32, K, N, std=0.05))
    g = BiGemm(K, N, kind, split_k=split)
    esz = 4 if kind == "bf16_f32" else 2
    pad = 4096                                   # bytes of guard on each side
    buf = torch.full((pad * 2 + M * N * esz,), 0xA5, dtype=torch.uint8, device="cuda")
    y_view = buf[pad:pad + M * N * esz].view(torch.float32 if esz == 4 else torch.bfloat16).view(M, N)
    g(x, w, y_view)
    torch.cuda.synchronize()
    b = buf.cpu().numpy()
    assert np.all(b[:pad] == 0xA5) and np.all(b[pad + M * N * esz:] == 0xA5)
    ref = g(x, w)
    assert torch.equal(y_view.view(torch.uint8), ref.view(torch.uint8))
    g.close()


def test_large_m():
    K, N, M = 64, 64, 1 << 17
    x = ig.normal_bf16(41, M, K)
    w = ig.normal_bf16(42, K, N)
    g = BiGemm(K, N, "bf16_f32")
    y = host_bits(g(dev_bf16(x), dev_bf16(w)))
    rows = [0, 1, 65535, 65536, M - 1]
    y_ref, _, sabs = oracle.gemm_bf16(x, w, "f32", rows=rows)
    check_tolerance(y[rows], y_ref, sabs, oracle.TOL_F32, "large M")
    y_last = host_bits(g(dev_bf16(x[-1:]), dev_bf16(w)))
    assert np.array_equal(y_last.view(np.uint32), y[-1:].view(np.uint32))
    g.close()


def test_weight_pointer_change_reencodes():
    K, N, M = 512, 256, 33
    x = ig.normal_bf16(51, M, K)
    w1 = ig.normal_bf16(52, K, N)
    w2 = ig.normal_bf16(53, K, N)
    g = BiGemm(K, N, "bf16")
    xd, w1d, w2d = dev_bf16(x), dev_bf16(w1), dev_bf16(w2)
    for w, wd in ((w1, w1d), (w2, w2d), (w1, w1d)):
        y_ref, _, sabs = oracle.gemm_bf16(x, w, "bf16")
        check_tolerance(host_bits(g(xd, wd)), y_ref, sabs, oracle.TOL_BF16, "W swap")
    g.close()


def test_argument_errors():
    g = BiGemm(256, 128, "bf16")
    x = torch.zeros((4, 256), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((256, 128), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((4 * 128 + 8,), dtype=torch.bfloat16, device="cuda")
    s = stream_ptr()
    with pytest.raises(BiGemmError) as e:
        bg.bi_gemm_run(g.handle, x.data_ptr(), 4, w.data_ptr(), None, y.data_ptr() + 2, s)
    assert e.value.code == bg.BI_GEMM_ERR_ALIGNMENT
    with pytest.raises(BiGemmError) as e:
        bg.bi_gemm_run(g.handle, x.data_ptr(), -1, w.data_ptr(), None, y.data_ptr(), s)
    assert e.value.code == bg.BI_GEMM_ERR_INVALID_ARG
    with pytest.raises(BiGemmError) as e:
        bg.bi_gemm_run(g.handle, 0, 4, w.data_ptr(), None, y.data_ptr(), s)
    assert e.value.code == bg.BI_GEMM_ERR_INVALID_ARG
    with pytest.raises(BiGemmError) as e:
        bg.bi_gemm_run(g.handle, x.data_ptr(), 4, w.data_ptr(), bg.bi_gemm_scales(x.data_ptr(), 0), y.data_ptr(), s)
    assert e.value.code == bg.BI_GEMM_ERR_INVALID_ARG
    f = BiGemm(256, 128, "mxfp8")
    xs = torch.zeros((4, 256), dtype=torch.uint8, device="cuda")
    ws = torch.zeros((256, 128), dtype=torch.uint8, device="cuda")
    sxs = torch.zeros((4 * 8 + 4,), dtype=torch.uint8, device="cuda")
    with pytest.raises(BiGemmError) as e:
        bg.bi_gemm_run(f.handle, xs.data_ptr(), 4, ws.data_ptr(), None, y.data_ptr(), s)
    assert e.value.code == bg.BI_GEMM_ERR_INVALID_ARG
    with pytest.raises(BiGemmError) as e:
        bg.bi_gemm_run(f.handle, xs.data_ptr(), 4, ws.data_ptr(),
                       bg.bi_gemm_scales(sxs.data_ptr() + 1, sxs.data_ptr()), y.data_ptr(), s)
    assert e.value.code == bg.BI_GEMM_ERR_ALIGNMENT
    for off in (2, 4, 8):   # W scales are copied in 16-byte chunks
        with pytest.raises(BiGemmError) as e:
            bg.bi_gemm_run(f.handle, xs.data_ptr(), 4, ws.data_ptr(),
                           bg.bi_gemm_scales(sxs.data_ptr(), sxs.data_ptr() + off), y.data_ptr(), s)
        assert e.value.code == bg.BI_GEMM_ERR_ALIGNMENT
    assert g.device_error() == 0 and f.device_error() == 0
    g.close()
    f.close()


def test_workspace_size_reported():
    g = BiGemm(16384, 24, "bf16_f32")
    assert g.workspace_size(0) == 0
    assert g.workspace_size(256) >= 2 * 32 * 128 * 64 * 4
    assert BiGemm(4096, 14336, "bf16").workspace_size(8192) == 0
    g.close()


@pytest.mark.parametrize("kind,out", [("bf16", "bf16"), ("bf16_f32", "f32")])
def test_forced_split_on_pair_tile(kind, out):
    """A fixed split count on the 256 x 256 CTA-pair tile: each CTA merges its own 128 rows."""
    K, N, M = 4096, 512, 300
    x = ig.normal_bf16(81, M, K)
    w = ig.normal_bf16(82, K, N, std=0.02)
    y_ref, _, sabs = oracle.gemm_bf16(x, w, out)
    g = BiGemm(K, N, kind, split_k=4)
    assert g.config["ctas_per_tile"] == 2 and g.config["split_k"] == 4
    xd, wd = dev_bf16(x), dev_bf16(w)
    y = host_bits(g(xd, wd))
    check_tolerance(y, y_ref, sabs, oracle.TOL_F32 if out == "f32" else oracle.TOL_BF16, "pair split")
    for M2 in (1, 129, 257):
        y2 = host_bits(g(xd[:M2].contiguous(), wd))
        assert np.array_equal(y2.view(np.uint8), y[:M2].view(np.uint8)), M2
    assert g.device_error() == 0
    g.close()
