"""Linspace stress GEMM of the nondeterminism article ("Batch invariance"):
a = linspace(-1000, 1000, 2048*4096) as [2048, 4096], b = linspace(-1000, 1000, 4096^2) as
[4096, 4096], bf16 in, fp32 out.  The page's library GEMM gave rows that differ by up to
1669.25 between mm(a[:1], b) and mm(a, b)[:1]; here they must be bitwise equal."""
import numpy as np
import pytest

import inputgen as ig
import oracle
from gpu_util import check_tolerance, dev_bf16, host_bits, oracle_rows
from invariant_bi_gemm_gb300 import BiGemm

pytestmark = pytest.mark.gpu

B_ROWS, D = 2048, 4096


@pytest.fixture(scope="module")
def setup():
    a = ig.linspace_bf16(-1000, 1000, B_ROWS, D)
    b = ig.linspace_bf16(-1000, 1000, D, D)
    g = BiGemm(D, D, "bf16_f32")
    yield g, a, b, dev_bf16(a), dev_bf16(b)
    g.close()


def test_first_row_alone_equals_first_row_of_full(setup):
    g, a, b, ad, bd = setup
    y_full = host_bits(g(ad, bd))
    y_one = host_bits(g(ad[:1].contiguous(), bd))
    assert np.array_equal(y_one.view(np.uint32), y_full[:1].view(np.uint32))
    # every prefix batch, and the last row alone, agree too
    for M in (2, 127, 128, 129, 1000):
        yM = host_bits(g(ad[:M].contiguous(), bd))
        assert np.array_equal(yM.view(np.uint32), y_full[:M].view(np.uint32)), M
    y_last = host_bits(g(ad[-1:].contiguous(), bd))
    assert np.array_equal(y_last.view(np.uint32), y_full[-1:].view(np.uint32))


def sample_rows():
    """64 rows of the M = 2048 output: tile and batch boundaries, {0, mid, last}, seeded rows."""
    rows = {0, 1, 2, 63, 64, 127, 128, 255, 256, 1023, 1024, 2046, 2047}
    rng = np.random.default_rng(20240611)
    while len(rows) < 64:
        rows.add(int(rng.integers(0, B_ROWS)))
    return sorted(rows)


def test_parity_sampled_rows(setup):
    """64 sampled rows of the full M = 2048 launch, every column, against the oracle."""
    g, a, b, ad, bd = setup
    rows = sample_rows()
    y_ref, _, sabs = oracle_rows(lambda r: oracle.gemm_bf16(a, b, "f32", rows=r), rows)
    y = host_bits(g(ad, bd))[rows]
    worst = check_tolerance(y, y_ref, sabs, oracle.TOL_F32, "linspace")
    print(f"linspace fp32 max |y-y_ref|/S_abs = {worst:.3g}")


@pytest.mark.parametrize("M", [1, 17, 64])
def test_parity_every_element_small_m(setup, M):
    """Every element of the launches with M <= 64 rows against the oracle."""
    g, a, b, ad, bd = setup
    y_ref, _, sabs = oracle_rows(lambda r: oracle.gemm_bf16(a[:M], b, "f32", rows=r), list(range(M)))
    y = host_bits(g(ad[:M].contiguous(), bd))
    worst = check_tolerance(y, y_ref, sabs, oracle.TOL_F32, f"linspace M={M}")
    print(f"linspace M={M} fp32 max |y-y_ref|/S_abs = {worst:.3g}")
