"""Batch-invariant RMSNorm ("Batch-invariant RMSNorm", nondeterminism article) on the GPU,
through the C ABI of include/bi_rmsnorm.h: every element against the oracle within
|y - v| <= (2^-8 + 2^-16)|v| (v the oracle's unrounded fp64 value), rows bitwise identical for
every batch size, the A/B cells and cross-M golden row of the batch-invariance harness, edge
cases, and the negative control (a thread count keyed on M) that the harness must catch.

Rows: N(0, 1) scaled by 2.08 / 0.019 / 0.245 in turn (the mHC page's checkpoint magnitudes);
weight g = 1 + 0.1 N(0, 1); eps = fp32(1e-6)."""
import ctypes

import numpy as np
import pytest
import torch

import inputgen as ig
import invariant_bi_gemm_gb300 as bg
import oracle
from gpu_util import Controls, bi_check, byte_diffs, dev_bf16, host_bits, stream_ptr
from invariant_bi_gemm_gb300 import BiRmsNorm

pytestmark = pytest.mark.gpu

EPS = float(np.float32(1e-6))


def check_rms(y_bits: np.ndarray, v: np.ndarray, what: str) -> float:
    """|y - v| <= TOL_RMSNORM_REL * |v| elementwise; returns the max of |y - v| / |v|."""
    y = ig.bf16_bits_to_f32(y_bits).astype(np.float64)
    d = np.abs(y - v)
    bad = ~(d <= oracle.TOL_RMSNORM_REL * np.abs(v))
    assert not bad.any(), f"{what}: {int(bad.sum())} elements outside tolerance, first at {np.argwhere(bad)[0]}"
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(v != 0, d / np.abs(v), 0.0)
    return float(r.max()) if r.size else 0.0


def inputs(d: int, M: int, seed: int = ig.SEED_X):
    return ig.scaled_rows_bf16(seed, M, d), ig.rmsnorm_weight_bf16(ig.SEED_W, d)


@pytest.mark.parametrize("d", [8, 40, 1000, 4096, 4104, 7168, 16384, 32768])
def test_parity_every_element(d):
    M = 130
    x, g = inputs(d, M)
    y_ref, v = oracle.rmsnorm_bf16(x, g, EPS)
    n = BiRmsNorm(d, EPS)
    y = host_bits(n(dev_bf16(x), dev_bf16(g)))
    worst = check_rms(y, v, f"d={d}")
    same = float(np.mean(y == y_ref))
    for M2 in (1, 3, 129):
        y2 = host_bits(n(dev_bf16(x[:M2]), dev_bf16(g)))
        assert np.array_equal(y2, y[:M2]), (d, M2)
    n.close()
    print(f"RMSNorm d={d}: max |y-v|/|v| = {worst:.3g}, bits equal to the oracle's rounding {same:.5f}")


def test_configuration_depends_on_d_only():
    for d, threads in ((8, 128), (4096, 128), (4104, 160), (7168, 224), (16384, 512), (32768, 1024)):
        c = BiRmsNorm(d, EPS).config
        assert c["threads"] == threads and c["vectors_per_thread"] <= 4 and c["d"] == d
        assert c["max_ctas"] >= c["num_sms"]


def test_rows_identical_for_every_m():
    d, MMAX = 4096, 300
    x, g = inputs(d, MMAX)
    n = BiRmsNorm(d, EPS)
    xd, gd = dev_bf16(x), dev_bf16(g)
    y_full = host_bits(n(xd, gd))
    for M in range(1, MMAX + 1):
        yM = host_bits(n(xd[:M].contiguous(), gd))
        assert np.array_equal(yM, y_full[:M]), M
    n.close()


def test_bi_cells_and_golden_row_across_batch_sizes():
    """A/B cells at targets {0, mid, last} and the content row C byte-equal to its M = 1 output,
    for batch sizes on both sides of every resident-block boundary of the persistent grid."""
    d = 7168
    n = BiRmsNorm(d, EPS)
    maxc = n.config["max_ctas"]
    g = dev_bf16(ig.rmsnorm_weight_bf16(ig.SEED_W, d))
    Mmax = 2 * maxc + 3
    A = dev_bf16(ig.scaled_rows_bf16(ig.SEED_A, Mmax, d))
    B = dev_bf16(ig.scaled_rows_bf16(ig.SEED_B, Mmax, d))
    C = dev_bf16(ig.scaled_rows_bf16(ig.SEED_C, 1, d))[0]
    golden = host_bits(n(C[None].contiguous(), g))
    total = 0
    for M in (1, 2, 16, 17, 151, 152, 153, maxc - 1, maxc, maxc + 1, 2 * maxc + 3):
        for t, d_ab, d_g in bi_check(lambda xx: n(xx, g), A, B, C, M, golden):
            total += d_ab + d_g
    assert total == 0
    n.close()


def test_large_batch_sampled_rows():
    """M = 8192 at d = 4096 (the LLM projection's width): 64 sampled rows against the oracle,
    and each equal to the same row normalised alone."""
    d, M = 4096, 8192
    x, g = inputs(d, M)
    n = BiRmsNorm(d, EPS)
    xd, gd = dev_bf16(x), dev_bf16(g)
    y = host_bits(n(xd, gd))
    rows = sorted(set([0, M // 2, M - 1] + list(ig.uniform_int(5, 0, 61, 0, M - 1))))
    _, v = oracle.rmsnorm_bf16(x, g, EPS, rows=rows)
    check_rms(y[rows], v, "M=8192 sample")
    for r in rows[:16]:
        assert np.array_equal(host_bits(n(xd[r:r + 1].contiguous(), gd)), y[r:r + 1]), r
    # batches just past the persistent grid's resident blocks (each row then has a block of its
    # own, without the next-row prefetch): the same bits as in the batch of 8192
    maxc = n.config["max_ctas"]
    for M2 in (maxc + 1, 2000, 2 * maxc):
        assert np.array_equal(host_bits(n(xd[:M2].contiguous(), gd)), y[:M2]), M2
    n.close()


def test_repeat_runs_identical():
    d, M = 4096, 64
    x, g = inputs(d, M)
    n = BiRmsNorm(d, EPS)
    xd, gd = dev_bf16(x), dev_bf16(g)
    first = host_bits(n(xd, gd))
    out = torch.empty_like(xd)
    for _ in range(200):
        n(xd, gd, out)
        assert np.array_equal(host_bits(out), first)
    n.close()


def test_edge_cases():
    d = 4096
    n = BiRmsNorm(d, EPS)
    g1 = torch.full((d,), 1.0, dtype=torch.bfloat16, device="cuda")
    # M = 0 queues nothing and leaves y alone
    y = torch.full((4, d), 7.0, dtype=torch.bfloat16, device="cuda")
    bg.bi_rmsnorm_run(n.handle, y.data_ptr(), 0, g1.data_ptr(), y.data_ptr(), stream_ptr())
    torch.cuda.synchronize()
    assert torch.all(y == 7.0)
    # zero row -> zeros (r = 1/sqrt(eps) finite); constant rows: closed forms of the oracle pins
    x = torch.zeros((3, d), dtype=torch.bfloat16, device="cuda")
    x[1] = 0.5
    x[2] = -0.5
    out = host_bits(n(x, g1))
    assert np.all(out[0] == 0) and np.all(out[1] == 0x3F80) and np.all(out[2] == 0xBF80)
    # in place gives the bits of the out-of-place run
    xs, gs = inputs(d, 33)
    xd, gd = dev_bf16(xs), dev_bf16(gs)
    ref = host_bits(n(xd, gd))
    n(xd, gd, xd)
    assert np.array_equal(host_bits(xd), ref)
    # row magnitudes 2^-40 .. 2^40 (sums of squares well inside fp32)
    f = ig.bf16_bits_to_f32(ig.normal_bf16(9, 6, d)).astype(np.float64)
    xw = ig.to_bf16_bits(f * np.exp2(np.array([-40, -20, -1, 1, 20, 40]))[:, None])
    _, v = oracle.rmsnorm_bf16(xw, gs, EPS)
    check_rms(host_bits(n(dev_bf16(xw), gd)), v, "wide magnitudes")
    n.close()


def test_misaligned_pointers_refused():
    d = 4096
    n = BiRmsNorm(d, EPS)
    buf = torch.zeros(3 * d + 16, dtype=torch.bfloat16, device="cuda")
    base = buf.data_ptr()
    for xo, go, yo in ((2, 0, 0), (0, 8, 0), (0, 0, 4)):
        rc = bg.library().bi_rmsnorm_run(ctypes.c_void_p(n.handle), ctypes.c_void_p(base + xo), 1,
                                         ctypes.c_void_p(base + 2 * d * 2 + go), ctypes.c_void_p(base + d * 2 + yo),
                                         ctypes.c_void_p(stream_ptr()))
        assert rc == bg.BI_GEMM_ERR_ALIGNMENT, (xo, go, yo)
    assert bg.library().bi_rmsnorm_run(ctypes.c_void_p(n.handle), ctypes.c_void_p(base), -1, ctypes.c_void_p(base),
                                       ctypes.c_void_p(base), ctypes.c_void_p(stream_ptr())) == bg.BI_GEMM_ERR_INVALID_ARG
    n.close()


def _control_rows(mkeyed: int, M: int, xd, gd, d):
    L = Controls().L
    y = torch.empty((M, d), dtype=torch.float32, device="cuda")
    rc = L.bi_ctl_rmsnorm_f32(ctypes.c_void_p(xd.data_ptr()), M, d, ctypes.c_void_p(gd.data_ptr()), EPS,
                              ctypes.c_void_p(y.data_ptr()), mkeyed, ctypes.c_void_p(stream_ptr()))
    assert rc == 0, rc
    return y.cpu().numpy().view(np.uint32)


def test_negative_control_m_keyed_threads_is_caught():
    """fp32 output before rounding: with threads per row fixed from d every row is the same at
    M = 1..16 as at M = 300; with threads keyed on M (1024 while M <= 16) the byte diffs are
    non-zero, so the harness can fail.  The fixed-tree control's values also stay within the
    fp32 part of the tolerance against the oracle."""
    d, MM = 4096, 300
    x, g = inputs(d, MM)
    xd, gd = dev_bf16(x), dev_bf16(g)
    fixed_full = _control_rows(0, MM, xd, gd, d)
    keyed_full = _control_rows(1, MM, xd, gd, d)
    assert np.array_equal(fixed_full, keyed_full)            # both use 128 threads above M = 16
    diffs_fixed = diffs_keyed = 0
    for M in (1, 2, 5, 16):
        diffs_fixed += byte_diffs(_control_rows(0, M, xd[:M].contiguous(), gd, d), fixed_full[:M])
        diffs_keyed += byte_diffs(_control_rows(1, M, xd[:M].contiguous(), gd, d), keyed_full[:M])
    assert diffs_fixed == 0
    assert diffs_keyed > 0
    _, v = oracle.rmsnorm_bf16(x[:8], g, EPS)
    vf = fixed_full[:8].view(np.float32).astype(np.float64)
    assert np.all(np.abs(vf - v) <= 2.0**-16 * np.abs(v))
    print(f"RMSNorm control: fixed-tree diffs {diffs_fixed}, M-keyed diffs {diffs_keyed}")
