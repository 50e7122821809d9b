"""Tiny bf16 GEMM x[M,256]·W[256,128], x~N(0,1), W~N(0,0.05), bf16 out, M in 1..16:
parity with the oracle on every element, and batch invariance (A/B cells at rows
{0, mid, last}, and C's row at M=1 byte-equal to its row at every other M and position)."""
import numpy as np
import pytest
import torch

import inputgen as ig
import oracle
from gpu_util import bi_check, check_tolerance, dev_bf16, host_bits
from invariant_bi_gemm_gb300 import BiGemm

pytestmark = pytest.mark.gpu

K, N = 256, 128


@pytest.fixture(scope="module")
def setup():
    W = ig.normal_bf16(ig.SEED_W, K, N, std=0.05)
    X = ig.normal_bf16(ig.SEED_X, 16, K)
    g = BiGemm(K, N, "bf16")
    yield g, W, X, dev_bf16(W), dev_bf16(X)
    g.close()


def test_config_is_fixed(setup):
    g = setup[0]
    c = g.config
    assert (c["block_m"], c["mma_m"], c["split_k"]) == (128, 128, 1)
    assert c["block_n"] == c["mma_n"] == 128 and c["mma_k"] == 16


def test_parity_every_m(setup):
    g, W, X, Wd, Xd = setup
    y_ref, _, sabs = oracle.gemm_bf16(X, W, "bf16")
    y16 = host_bits(g(Xd, Wd))
    check_tolerance(y16, y_ref, sabs, oracle.TOL_BF16, "M=16")
    for M in range(1, 17):
        yM = host_bits(g(Xd[:M].contiguous(), Wd))
        check_tolerance(yM, y_ref[:M], sabs[:M], oracle.TOL_BF16, f"M={M}")
        assert np.array_equal(yM.view(np.uint8), y16[:M].view(np.uint8)), f"rows moved at M={M}"
    assert g.device_error() == 0


def test_bi_cells(setup):
    g, W, X, Wd, Xd = setup
    C = dev_bf16(ig.normal_bf16(ig.SEED_C, 1, K))[0]
    A = dev_bf16(ig.normal_bf16(ig.SEED_A, 16, K))
    B = dev_bf16(ig.normal_bf16(ig.SEED_B, 16, K))
    golden = host_bits(g(C[None].contiguous(), Wd))
    total = 0
    for M in range(1, 17):
        for t, d_ab, d_g in bi_check(lambda x: g(x, Wd), A, B, C, M, golden):
            total += d_ab + d_g
    assert total == 0


def test_device_error_clear(setup):
    assert setup[0].device_error() == 0
