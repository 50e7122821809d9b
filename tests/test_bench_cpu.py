"""The figures bench.py reports are built from a few closed forms; check them on the CPU against
hand-computed values for the workloads they describe (no GPU)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def test_gemm_flops_and_bytes_of_the_llm_projection():
    # x[1,4096] . W[4096,14336], bf16 in and out: 2*M*K*N flops, W and x read once, y written once
    assert bench.flops(1) == 2 * 4096 * 14336
    assert bench.algo_bytes(1) == 2 * (4096 + 4096 * 14336) + 2 * 14336 == 117_477_376
    # fp32 out and MXFP8 (one E8M0 byte per 32 elements of x and of W)
    assert bench.algo_bytes(8192, out_bytes=4) == 2 * (8192 * 4096 + 4096 * 14336) + 4 * 8192 * 14336
    assert bench.algo_bytes(64, in_bytes=1, scale_bytes=1 / 32) == (64 * 4096 + 4096 * 14336) * (1 + 1 / 32) + 2 * 64 * 14336


def test_roofline_regimes_of_the_sweep():
    """With the measured peaks the LLM shape is HBM-bound up to M = 256 and tensor-bound from
    M = 512 (the ridge is near 280 FLOP per byte)."""
    peaks = {"hbm_gbs": 6774.2, "bf16_tflops": 1895.0}
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    assert 270 < ridge < 290
    for M in bench.M_SWEEP:
        intensity = bench.flops(M) / bench.algo_bytes(M)
        assert (intensity < ridge) == (M <= 256), M


def test_attention_and_rmsnorm_bytes():
    # batch 32 x context 4096, 8 KV heads of 128: K and V once (bf16), q and o of 32 heads
    assert bench.attention_bytes(32, 4096) == 2 * 32 * 4096 * 8 * 128 * 2 + 2 * 32 * 32 * 128 * 2 == 537_395_200
    # RMSNorm of x[8192, 4096] bf16: x read, y written, the weight read
    assert bench.rmsnorm_bytes(8192) == 2 * 8192 * 4096 * 2 + 2 * 4096
