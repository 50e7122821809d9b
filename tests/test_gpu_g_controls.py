"""Negative controls must fail the batch-invariance harness, and the bounded waits must turn a
withheld pipeline stage into an error status instead of a hang.

The controls are the two defects of "[BI][DSv4] Make mHC tilelang ops batch invariant"
("What"): N1, a split count n_sms // cdiv(M, 64); N2, a second implementation for M <= 16.
They run at the page's checkpoint-realistic row magnitudes (2.08 / 0.019 / 0.245): the page
warns that tiny synthetic magnitudes made a control pass vacuously."""
import ctypes

import numpy as np
import pytest
import torch

import inputgen as ig
import oracle
from gpu_util import Controls, byte_diffs, check_tolerance, dev_bf16, host_bits, stream_ptr
from invariant_bi_gemm_gb300 import BI_BF16_OUT_BF16, BI_BF16_OUT_F32, BI_GEMM_ERR_TIMEOUT

pytestmark = pytest.mark.gpu

M_SWEEP = [1, 7, 8, 15, 16, 17, 63, 64, 65, 128, 129, 192, 193, 256]


def _row0_across_m(run, C, A, N, out_dtype):
    """Bytes of content C's output row at position 0 for every M of the sweep."""
    rows = []
    for M in M_SWEEP:
        x = A[:M].clone()
        x[0] = C
        y = torch.empty((M, N), dtype=out_dtype, device="cuda")
        run(x, M, y)
        rows.append(host_bits(y[:1]))
    return rows


def _diffs_vs_first(rows):
    return sum(byte_diffs(r, rows[0]) for r in rows[1:])


@pytest.fixture(scope="module")
def ctl():
    return Controls()


def test_n1_msplit_control_fails_and_product_passes(ctl):
    K, N = 16384, 24
    W = dev_bf16(ig.normal_bf16(ig.SEED_W, K, N, std=0.02))
    C = dev_bf16(ig.scaled_rows_bf16(ig.SEED_C, 1, K))[0]
    A = dev_bf16(ig.scaled_rows_bf16(ig.SEED_A, 256, K))
    h = ctl.create(K, N, BI_BF16_OUT_F32)
    L, s = ctl.L, stream_ptr()
    counts = {ctl.L.bi_ctl_msplit_count(h, M) for M in M_SWEEP}
    assert len(counts) > 1                      # the control's split count does move with M

    def run_ctl(x, M, y):
        assert L.bi_ctl_run_msplit(h, x.data_ptr(), M, W.data_ptr(), None, y.data_ptr(), s) == 0

    def run_prod(x, M, y):
        assert L.bi_ctl_run(h, x.data_ptr(), M, W.data_ptr(), None, y.data_ptr(), s) == 0

    bad = _diffs_vs_first(_row0_across_m(run_ctl, C, A, N, torch.float32))
    good = _diffs_vs_first(_row0_across_m(run_prod, C, A, N, torch.float32))
    assert good == 0
    assert bad > 0, "the M-dependent split control passed: the harness cannot see a broken kernel"
    assert L.bi_ctl_get_device_error(h, s) == 0
    L.bi_ctl_destroy(h)


def test_n2_small_m_fork_control_fails(ctl):
    K, N = 4096, 14336
    W = dev_bf16(ig.normal_bf16(ig.SEED_W, K, N, std=0.02))
    C = dev_bf16(ig.scaled_rows_bf16(ig.SEED_C, 1, K))[0]
    A = dev_bf16(ig.scaled_rows_bf16(ig.SEED_A, 256, K))
    h = ctl.create(K, N, BI_BF16_OUT_BF16)
    L, s = ctl.L, stream_ptr()

    def run_ctl(x, M, y):
        assert L.bi_ctl_run_smallm_fork(h, x.data_ptr(), M, W.data_ptr(), y.data_ptr(), s) == 0

    rows = _row0_across_m(run_ctl, C, A, N, torch.bfloat16)
    small = [r for M, r in zip(M_SWEEP, rows) if M <= 16]
    large = [r for M, r in zip(M_SWEEP, rows) if M > 16]
    assert _diffs_vs_first(small) == 0 and _diffs_vs_first(large) == 0   # each side is consistent
    assert byte_diffs(small[0], large[0]) > 0, "small-M fork control passed vacuously"
    L.bi_ctl_destroy(h)


@pytest.mark.parametrize("M", [200, 40])   # the pair tile's two pipelines (M = 40: two k-blocks a stage)
def test_stalled_pipeline_reports_timeout_and_context_survives(ctl, M):
    K, N = 1024, 256
    x = ig.normal_bf16(61, M, K)
    w = ig.normal_bf16(62, K, N, std=0.05)
    xd, wd = dev_bf16(x), dev_bf16(w)
    h = ctl.create(K, N, BI_BF16_OUT_BF16, timeout_ns=50_000_000)     # 50 ms limit
    L, s = ctl.L, stream_ptr()
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    assert L.bi_ctl_run_stall(h, xd.data_ptr(), M, wd.data_ptr(), None, y.data_ptr(), s) == 0
    assert L.bi_ctl_get_device_error(h, s) == BI_GEMM_ERR_TIMEOUT
    assert L.bi_ctl_get_device_error(h, s) == 0                       # status word was cleared
    assert L.bi_ctl_run(h, xd.data_ptr(), M, wd.data_ptr(), None, y.data_ptr(), s) == 0
    assert L.bi_ctl_get_device_error(h, s) == 0
    y_ref, _, sabs = oracle.gemm_bf16(x, w, "bf16")
    check_tolerance(host_bits(y), y_ref, sabs, oracle.TOL_BF16, "after timeout")
    L.bi_ctl_destroy(h)


def test_stalled_split_run_recovers(ctl):
    """A timed-out split-K run may leave arrival counters behind; the next run resets them."""
    K, N, M = 16384, 24, 100
    x = ig.scaled_rows_bf16(71, M, K)
    w = ig.normal_bf16(72, K, N, std=0.02)
    xd, wd = dev_bf16(x), dev_bf16(w)
    h = ctl.create(K, N, BI_BF16_OUT_F32, timeout_ns=50_000_000)
    L, s = ctl.L, stream_ptr()
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    assert L.bi_ctl_run_stall(h, xd.data_ptr(), M, wd.data_ptr(), None, y.data_ptr(), s) == 0
    assert L.bi_ctl_get_device_error(h, s) == BI_GEMM_ERR_TIMEOUT
    for _ in range(2):
        assert L.bi_ctl_run(h, xd.data_ptr(), M, wd.data_ptr(), None, y.data_ptr(), s) == 0
        assert L.bi_ctl_get_device_error(h, s) == 0
        y_ref, _, sabs = oracle.gemm_bf16(x, w, "f32")
        check_tolerance(host_bits(y), y_ref, sabs, oracle.TOL_F32, "split after timeout")
    L.bi_ctl_destroy(h)


def test_shared_merge_wait_times_out_and_recovers(ctl):
    """The split CTAs of a tile wait for each other before a shared merge; when one never
    arrives the others' bounded waits expire, the run reports a timeout, and the next run (which
    resets the arrival counters) is correct."""
    K, N, M = 16384, 24, 100             # 32 resident split CTAs, 300 KB of partials: shared merge
    x = ig.scaled_rows_bf16(73, M, K)
    w = ig.normal_bf16(74, K, N, std=0.02)
    xd, wd = dev_bf16(x), dev_bf16(w)
    h = ctl.create(K, N, BI_BF16_OUT_F32, timeout_ns=50_000_000)
    L, s = ctl.L, stream_ptr()
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    assert L.bi_ctl_run_skip_arrival(h, xd.data_ptr(), M, wd.data_ptr(), None, y.data_ptr(), s) == 0
    assert L.bi_ctl_get_device_error(h, s) == BI_GEMM_ERR_TIMEOUT
    y_ref, _, sabs = oracle.gemm_bf16(x, w, "f32")
    for _ in range(2):
        assert L.bi_ctl_run(h, xd.data_ptr(), M, wd.data_ptr(), None, y.data_ptr(), s) == 0
        assert L.bi_ctl_get_device_error(h, s) == 0
        check_tolerance(host_bits(y), y_ref, sabs, oracle.TOL_F32, "shared merge after timeout")
    L.bi_ctl_destroy(h)
