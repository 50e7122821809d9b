"""mHC pre-norm projection ("[BI][DSv4] Make mHC tilelang ops batch invariant": the pre-norm GEMM
with its fused RMSNorm) on the GPU through include/bi_prenorm.h: every element against the
oracle within |y - v| <= TOL_PRENORM_ABS * sabs + 2^-15 |v|, rows bitwise identical for every
M = 1..256, the A/B cells and golden rows at the page's batch boundaries, and the page's defect
as a negative control (the K split chosen from the token count).

Workload: the flattened streams of four 4096-wide residual streams (K = 16384), 24 mixing
coefficients (N = 4 x 6), rows scaled by the page's checkpoint magnitudes 2.08 / 0.019 / 0.245
in turn, W ~ N(0, 0.02)."""
import ctypes

import numpy as np
import pytest
import torch

import inputgen as ig
import invariant_bi_gemm_gb300 as bg
import oracle
from gpu_util import bi_check, byte_diffs, dev_bf16, host_bits, stream_ptr
from invariant_bi_gemm_gb300 import BiPreNorm

pytestmark = pytest.mark.gpu

EPS = float(np.float32(1e-6))
BOUNDARIES = [1, 7, 8, 15, 16, 17, 63, 64, 65, 128, 129, 192, 193, 256]


def check(y, v, sabs, what):
    err = np.abs(y.astype(np.float64) - v)
    tol = oracle.TOL_PRENORM_ABS * sabs + 2.0**-15 * np.abs(v)
    bad = ~(err <= tol)
    assert not bad.any(), f"{what}: {int(bad.sum())} outside the tolerance, first at {np.argwhere(bad)[0]}"
    return float(np.max(err / tol))


@pytest.mark.parametrize("K,N,M,chunk", [
    (16384, 24, 256, 0), (16384, 24, 1, 0), (4096, 32, 40, 0), (1000, 8, 33, 0),
    (16384, 24, 17, 64), (16384, 16, 100, 1024), (2056, 24, 19, 512),
])
def test_parity_every_element(K, N, M, chunk):
    x = ig.scaled_rows_bf16(ig.SEED_X, M, K)
    w = ig.normal_bf16(ig.SEED_W, K, N, std=0.02)
    h = BiPreNorm(K, N, EPS, chunk)
    y = h(dev_bf16(x), dev_bf16(w)).cpu().numpy()
    _, v, sabs = oracle.prenorm_gemm(x, w, EPS)
    worst = check(y, v, sabs, f"K={K} N={N} M={M} chunk={chunk}")
    h.close()
    print(f"prenorm K={K} N={N} M={M} chunk={chunk}: max err/tol {worst:.3g}")


def test_rows_identical_for_every_m():
    K, N, MMAX = 16384, 24, 256
    x = dev_bf16(ig.scaled_rows_bf16(ig.SEED_X, MMAX, K))
    w = dev_bf16(ig.normal_bf16(ig.SEED_W, K, N, std=0.02))
    h = BiPreNorm(K, N, EPS)
    full = host_bits(h(x, w))
    for M in range(1, MMAX + 1):
        assert np.array_equal(host_bits(h(x[:M].contiguous(), w)).view(np.uint32), full[:M].view(np.uint32)), M
    h.close()


def test_x_written_by_the_preceding_kernel():
    """Both kernels of a call start while the kernel before them finishes: x written by a kernel
    into the same buffer right before every call, alternating two contents, back to back over the
    page's batch boundaries, gives the bits of the same calls made after a synchronisation."""
    K, N = 16384, 24
    w = dev_bf16(ig.normal_bf16(ig.SEED_W, K, N, std=0.02))
    srcs = [dev_bf16(ig.scaled_rows_bf16(sd, 256, K)) for sd in (ig.SEED_X, ig.SEED_A)]
    h = BiPreNorm(K, N, EPS)
    refs = [h(src, w).clone() for src in srcs]
    torch.cuda.synchronize()
    xbuf = torch.empty_like(srcs[0])
    outs = []
    for M in BOUNDARIES:
        for which in (0, 1):
            torch.mul(srcs[which][:M], 1, out=xbuf[:M])     # exact; a kernel on the stream
            outs.append((M, which, h(xbuf[:M], w)))
    torch.cuda.synchronize()
    for M, which, y in outs:
        assert torch.equal(y.view(torch.int32), refs[which][:M].view(torch.int32)), (M, which)
    h.close()


def test_bi_cells_at_the_pages_batch_boundaries():
    K, N = 16384, 24
    h = BiPreNorm(K, N, EPS)
    w = dev_bf16(ig.normal_bf16(ig.SEED_W, K, N, std=0.02))
    A = dev_bf16(ig.scaled_rows_bf16(ig.SEED_A, 256, K))
    B = dev_bf16(ig.scaled_rows_bf16(ig.SEED_B, 256, K))
    C = dev_bf16(ig.scaled_rows_bf16(ig.SEED_C, 1, K))[0]
    golden = host_bits(h(C[None].contiguous(), w))
    total = 0
    for M in BOUNDARIES:
        for t, d_ab, d_g in bi_check(lambda xx: h(xx, w), A, B, C, M, golden):
            total += d_ab + d_g
    assert total == 0
    h.close()


def test_large_batch_sampled_rows():
    K, N, M = 16384, 24, 4096
    x = ig.scaled_rows_bf16(ig.SEED_X, M, K)
    w = ig.normal_bf16(ig.SEED_W, K, N, std=0.02)
    h = BiPreNorm(K, N, EPS)
    xd, wd = dev_bf16(x), dev_bf16(w)
    y = h(xd, wd).cpu().numpy()
    rows = sorted(set([0, M // 2, M - 1] + list(ig.uniform_int(7, 0, 29, 0, M - 1))))
    _, v, sabs = oracle.prenorm_gemm(x[rows], w, EPS)
    check(y[rows], v, sabs, "M=4096 sample")
    for r in rows[:8]:
        assert np.array_equal(h(xd[r:r + 1].contiguous(), wd).cpu().numpy().view(np.uint32), y[r:r + 1].view(np.uint32))
    h.close()


def test_negative_control_split_from_token_count_is_caught():
    """The page's defect: a split chosen from the number of tokens (here chunks of 128 up to 64
    tokens, 512 above) moves the bits of the same rows between batch sizes; the fixed chunk
    does not."""
    K, N = 16384, 24
    x = dev_bf16(ig.scaled_rows_bf16(ig.SEED_X, 256, K))
    w = dev_bf16(ig.normal_bf16(ig.SEED_W, K, N, std=0.02))
    small, large, fixed = BiPreNorm(K, N, EPS, 128), BiPreNorm(K, N, EPS, 512), BiPreNorm(K, N, EPS)
    keyed = steady = 0
    for M_small, M_large in ((1, 65), (64, 256), (16, 129)):
        m = min(M_small, M_large)
        a = host_bits(small(x[:M_small].contiguous(), w))[:m]
        b = host_bits(large(x[:M_large].contiguous(), w))[:m]
        keyed += byte_diffs(a, b)
        c = host_bits(fixed(x[:M_small].contiguous(), w))[:m]
        d = host_bits(fixed(x[:M_large].contiguous(), w))[:m]
        steady += byte_diffs(c, d)
    assert steady == 0 and keyed > 0
    print(f"prenorm control: fixed split diffs {steady}, token-keyed split diffs {keyed}")
    for hh in (small, large, fixed):
        hh.close()


def test_empty_and_misaligned():
    h = BiPreNorm(4096, 24, EPS)
    buf = torch.zeros(8192 + 64, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(64, dtype=torch.float32, device="cuda")
    L, V = bg.library(), ctypes.c_void_p
    assert L.bi_prenorm_run(V(h.handle), V(buf.data_ptr()), 0, V(buf.data_ptr()), V(y.data_ptr()), V(stream_ptr())) == 0
    assert L.bi_prenorm_run(V(h.handle), V(buf.data_ptr() + 2), 1, V(buf.data_ptr()), V(y.data_ptr()),
                            V(stream_ptr())) == bg.BI_GEMM_ERR_ALIGNMENT
    assert L.bi_prenorm_run(V(h.handle), V(buf.data_ptr()), 1, V(buf.data_ptr() + 8), V(y.data_ptr()),
                            V(stream_ptr())) == bg.BI_GEMM_ERR_ALIGNMENT
    assert L.bi_prenorm_run(V(h.handle), V(buf.data_ptr()), 1, V(buf.data_ptr()), V(y.data_ptr() + 4),
                            V(stream_ptr())) == bg.BI_GEMM_ERR_ALIGNMENT
    assert h.config == {"K": 4096, "N": 24, "chunk": 512, "splits": 8, "tile_rows": 16}
    h.close()
