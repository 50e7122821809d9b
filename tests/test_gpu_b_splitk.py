"""Small-N long-K GEMM, the split-K-tempting shape of "[BI][DSv4] Make mHC tilelang ops batch
invariant": fp32 out of bf16 x[M,16384]·W[16384,24], rows of x scaled by 2.08 / 0.019 / 0.245
in turn (the page's checkpoint-realistic magnitudes), W~N(0,0.02), M = 1..256 every value.
The handle pins the split count to 32 with an ordered serial merge; every row must be
bitwise the same at every M, and within 1e-5 * S_abs of the oracle."""
import numpy as np
import pytest

import inputgen as ig
import oracle
from gpu_util import bi_check, check_tolerance, dev_bf16, host_bits
from invariant_bi_gemm_gb300 import BiGemm

pytestmark = pytest.mark.gpu

K, N, MMAX = 16384, 24, 256


@pytest.fixture(scope="module")
def setup():
    W = ig.normal_bf16(ig.SEED_W, K, N, std=0.02)
    X = ig.scaled_rows_bf16(ig.SEED_X, MMAX, K)
    g = BiGemm(K, N, "bf16_f32")
    y_ref, _, sabs = oracle.gemm_bf16(X, W, "f32")
    yield g, dev_bf16(W), dev_bf16(X), y_ref, sabs
    g.close()


def test_split_is_pinned(setup):
    c = setup[0].config
    assert c["split_k"] == 32 and c["block_n"] == 64


def test_parity_and_rows_identical_for_every_m(setup):
    g, Wd, Xd, y_ref, sabs = setup
    y_full = host_bits(g(Xd, Wd))
    worst = check_tolerance(y_full, y_ref, sabs, oracle.TOL_F32, "M=256")
    for M in range(1, MMAX + 1):
        yM = host_bits(g(Xd[:M].contiguous(), Wd))
        assert np.array_equal(yM.view(np.uint32), y_full[:M].view(np.uint32)), f"M={M}"
    assert g.device_error() == 0
    print(f"split-K fp32 max |y-y_ref|/S_abs = {worst:.3g}")


def test_bi_cells_across_batch_boundaries(setup):
    g, Wd, Xd, _, _ = setup
    C = dev_bf16(ig.scaled_rows_bf16(ig.SEED_C, 1, K))[0]
    A = dev_bf16(ig.scaled_rows_bf16(ig.SEED_A, MMAX, K))
    B = dev_bf16(ig.scaled_rows_bf16(ig.SEED_B, MMAX, K))
    golden = host_bits(g(C[None].contiguous(), Wd))
    total = 0
    for M in (1, 7, 8, 15, 16, 17, 63, 64, 65, 127, 128, 129, 192, 193, 255, 256):
        for t, d_ab, d_g in bi_check(lambda x: g(x, Wd), A, B, C, M, golden):
            total += d_ab + d_g
    assert total == 0


def test_forced_split_counts_agree_with_oracle(setup):
    """Any fixed split count is a valid configuration; each stays within tolerance."""
    _, Wd, Xd, y_ref, sabs = setup
    for s in (1, 2, 8, 64, 256):
        g = BiGemm(K, N, "bf16_f32", split_k=s)
        assert g.config["split_k"] == s
        y = host_bits(g(Xd[:130].contiguous(), Wd))
        check_tolerance(y, y_ref[:130], sabs[:130], oracle.TOL_F32, f"S={s}")
        g.close()


@pytest.mark.parametrize("max_ctas", [4, 16, 31])
def test_merge_paths_give_identical_bits(setup, max_ctas):
    """With every split unit resident the 32 split CTAs share a tile's merge; with the grid
    capped below the unit count the last CTA to arrive merges it alone.  Both sum every element
    in split order, so the outputs are bitwise identical (and the capped grid also exercises
    CTAs that carry several units)."""
    g, Wd, Xd, _, _ = setup
    capped = BiGemm(K, N, "bf16_f32", max_ctas=max_ctas)
    assert capped.config["split_k"] == 32 and capped.config["max_groups"] == max_ctas
    for M in (1, 64, 129, 256):
        xs = Xd[:M].contiguous()
        a = host_bits(g(xs, Wd))
        b = host_bits(capped(xs, Wd))
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), (M, max_ctas)
    assert capped.device_error() == 0 and g.device_error() == 0
    capped.close()


def test_split_too_large_for_merge_staging():
    """A fixed split of 4096 k-ranges: one item's partials (64 KB) no longer fit the epilogue
    staging, so the merge takes its register-batch path; still every element against the
    oracle and rows bitwise equal across M."""
    K, N, M = 262144, 24, 8
    x = ig.scaled_rows_bf16(91, M, K)
    w = ig.normal_bf16(92, K, N, std=0.02)
    g = BiGemm(K, N, "bf16_f32", split_k=4096)
    assert g.config["split_k"] == 4096
    xd, wd = dev_bf16(x), dev_bf16(w)
    y = host_bits(g(xd, wd))
    y_ref, _, sabs = oracle.gemm_bf16(x, w, "f32")
    check_tolerance(y, y_ref, sabs, oracle.TOL_F32, "S=4096")
    y1 = host_bits(g(xd[3:4].contiguous(), wd))
    assert np.array_equal(y1.view(np.uint32), y[3:4].view(np.uint32))
    assert g.device_error() == 0
    g.close()


@pytest.mark.parametrize("kind", ["bf16", "bf16_f32"])
def test_pair_tile_split_across_both_pipelines(kind):
    """A wide single N tile with a long K (N = 256, K = 16384) runs the CTA-pair tile with the
    fixed split of 32: rows of up to 64 take the pair tile's small-M pipeline (stages of two
    k-blocks), larger batches the other one.  Every row of the M = 200 run against the oracle,
    and every row bitwise the same at M = 1, 40, 64, 65 and 200, across the switch."""
    K2, N2, M2 = 16384, 256, 200
    x = ig.scaled_rows_bf16(71, M2, K2)
    w = ig.normal_bf16(72, K2, N2, std=0.02)
    g = BiGemm(K2, N2, kind)
    c = g.config
    assert c["ctas_per_tile"] == 2 and c["split_k"] == 32
    out = "f32" if kind == "bf16_f32" else "bf16"
    xd, wd = dev_bf16(x), dev_bf16(w)
    y = host_bits(g(xd, wd))
    y_ref, _, sabs = oracle.gemm_bf16(x, w, out)
    check_tolerance(y, y_ref, sabs, oracle.TOL_F32 if out == "f32" else oracle.TOL_BF16, f"pair split {kind}")
    view = np.uint32 if out == "f32" else np.uint16
    for M in (1, 40, 64, 65):
        yM = host_bits(g(xd[:M].contiguous(), wd))
        assert np.array_equal(yM.view(view), y[:M].view(view)), (kind, M)
    assert g.device_error() == 0
    g.close()
