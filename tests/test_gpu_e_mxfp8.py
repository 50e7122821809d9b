"""MXFP8 block-scaled GEMM: E4M3 x[ws*Mr, K] and W[K, N] with E8M0 scales per 32 K
(identity or K-varying, all four combinations), bf16 out, over the batch-invariance matrix of
the batch-invariance test issue ("Test methodology"): ws in {2,4,8} row blocks concatenated
on one GPU, Mr in {1,4,8,16,32,64}, K in {128..2048}, N in {64..512}.

Checks: every element against the oracle; rows bitwise identical across every ws*Mr; each
row block run alone bitwise equal to the same rows of the concatenated run (the LOCAL vs
GATHER defect of that issue's "Background", reduced to one GPU); A/B cells."""
import itertools

import numpy as np
import pytest
import torch

import inputgen as ig
import oracle
from gpu_util import byte_diffs, check_tolerance, dev_u8, host_bits, oracle_rows
from invariant_bi_gemm_gb300 import BiGemm

pytestmark = pytest.mark.gpu

KS = [128, 256, 512, 1024, 2048]
NS = [64, 128, 256, 512]
COMBOS = [("ID", "ID"), ("ID", "VAR"), ("VAR", "ID"), ("VAR", "VAR")]
WS = [2, 4, 8]
MR = [1, 4, 8, 16, 32, 64]
MMAX = 512
BLOCK_CHECKS = [(2, 4), (8, 1), (4, 16), (8, 64), (2, 64)]


def inputs(K, N, combo, rows=MMAX, seed_x=ig.SEED_X):
    x = ig.normal_e4m3(seed_x, rows, K)
    sx = ig.e8m0_scales(combo[0], seed_x, rows, K // 32)
    w = ig.normal_e4m3(ig.SEED_W, K, N)
    sw = ig.e8m0_scales(combo[1], ig.SEED_W, K // 32, N)
    return x, sx, w, sw


@pytest.mark.parametrize("K,N", list(itertools.product(KS, NS)))
def test_mxfp8_matrix(K, N):
    g = BiGemm(K, N, "mxfp8")
    worst = 0.0
    for combo in COMBOS:
        x, sx, w, sw = inputs(K, N, combo)
        y_ref, _, sabs = oracle.gemm_mxfp8(x, sx, w, sw)
        xd, sxd, wd, swd = dev_u8(x), dev_u8(sx), dev_u8(w), dev_u8(sw)
        y_full = g(xd, wd, sx=sxd, sw=swd)
        worst = max(worst, check_tolerance(host_bits(y_full), y_ref, sabs, oracle.TOL_BF16, f"K={K} N={N} {combo}"))
        for ws, mr in itertools.product(WS, MR):
            M = ws * mr
            yM = g(xd[:M], wd, sx=sxd[:M], sw=swd)
            assert torch.equal(yM.view(torch.int16), y_full[:M].view(torch.int16)), (combo, ws, mr)
            if (ws, mr) in BLOCK_CHECKS:
                for b in range(ws):
                    yb = g(xd[b * mr:(b + 1) * mr], wd, sx=sxd[b * mr:(b + 1) * mr], sw=swd)
                    assert torch.equal(yb.view(torch.int16), yM[b * mr:(b + 1) * mr].view(torch.int16)), \
                        ("block", combo, ws, mr, b)
    assert g.device_error() == 0
    g.close()
    print(f"MXFP8 K={K} N={N} max ratio {worst:.3g}")


@pytest.mark.parametrize("combo", COMBOS)
def test_mxfp8_bi_cells(combo):
    K, N = 2048, 256
    g = BiGemm(K, N, "mxfp8")
    x, sx, w, sw = inputs(K, N, combo)
    wd, swd = dev_u8(w), dev_u8(sw)
    cx, csx, _, _ = inputs(K, N, combo, rows=1, seed_x=ig.SEED_C)
    ax, asx, _, _ = inputs(K, N, combo, seed_x=ig.SEED_A)
    bx, bsx, _, _ = inputs(K, N, combo, seed_x=ig.SEED_B)
    golden = host_bits(g(dev_u8(cx), wd, sx=dev_u8(csx), sw=swd))
    total = 0
    for ws, mr in [(2, 1), (2, 4), (4, 8), (8, 16), (8, 64)]:
        M = ws * mr
        for t in ig.target_rows(M):
            outs = []
            for rx, rsx in ((ax, asx), (bx, bsx)):
                xv = ig.bi_variant(rx[:M], t, cx[0])
                sv = ig.bi_variant(rsx[:M], t, csx[0])
                outs.append(host_bits(g(dev_u8(xv), wd, sx=dev_u8(sv), sw=swd))[t:t + 1])
            total += byte_diffs(outs[0], outs[1]) + byte_diffs(outs[0], golden)
    assert total == 0
    g.close()


def test_mxfp8_llm_shape():
    """The LLM projection shape in MXFP8 with K-varying scales on both sides."""
    K, N, MM = 4096, 14336, 2048
    x, sx, w, sw = inputs(K, N, ("VAR", "VAR"), rows=MM)
    g = BiGemm(K, N, "mxfp8")
    xd, sxd, wd, swd = dev_u8(x), dev_u8(sx), dev_u8(w), dev_u8(sw)
    y_full = g(xd, wd, sx=sxd, sw=swd)
    for M in (1, 17, 129, 1000):
        yM = g(xd[:M], wd, sx=sxd[:M], sw=swd)
        assert torch.equal(yM.view(torch.int16), y_full[:M].view(torch.int16)), M
    # every element of rows 0..63 (the M <= 64 launches are bitwise those rows), and 64 sampled rows
    # of the rest: tile and batch boundaries, {mid, last} and seeded rows
    rows = set(range(64)) | {127, 128, 255, 256, 511, 1023, 1024, 2047}
    rng = np.random.default_rng(20240612)
    while len(rows) < 128:
        rows.add(int(rng.integers(64, MM)))
    rows = sorted(rows)
    y_ref, _, sabs = oracle_rows(lambda r: oracle.gemm_mxfp8(x, sx, w, sw, rows=r), rows)
    check_tolerance(host_bits(y_full)[rows], y_ref, sabs, oracle.TOL_BF16, "MXFP8 LLM shape")
    g.close()


def test_mxfp8_static_w_with_x_written_just_before():
    """MXFP8 with BI_GEMM_FLAG_STATIC_W on the LLM shape: x and its scales written by kernels into
    the same buffers right before every launch, alternating between two contents, back to back
    at batch sizes on both sides of the pipeline switches: the bits of the same rows without the
    flag."""
    K, N, MM = 4096, 14336, 2048
    xa, sxa, w, sw = inputs(K, N, ("VAR", "VAR"), rows=MM)
    xb, sxb, _, _ = inputs(K, N, ("VAR", "VAR"), rows=MM, seed_x=ig.SEED_A)
    g = BiGemm(K, N, "mxfp8")
    gs = BiGemm(K, N, "mxfp8", static_w=True)
    wd, swd = dev_u8(w), dev_u8(sw)
    src = [(dev_u8(xa), dev_u8(sxa)), (dev_u8(xb), dev_u8(sxb))]
    refs = [g(x, wd, sx=sx, sw=swd) for x, sx in src]
    xbuf, sxbuf = torch.empty_like(src[0][0]), torch.empty_like(src[0][1])
    outs = []
    for M in (1, 17, 64, 65, 256, 1000, 2048):
        for which in (0, 1):
            torch.bitwise_or(src[which][0][:M], 0, out=xbuf[:M])     # kernels on the stream
            torch.bitwise_or(src[which][1][:M], 0, out=sxbuf[:M])
            outs.append((M, which, gs(xbuf[:M], wd, sx=sxbuf[:M], sw=swd)))
    torch.cuda.synchronize()
    assert gs.device_error() == 0
    for M, which, y in outs:
        assert torch.equal(y.view(torch.int16), refs[which][:M].view(torch.int16)), (M, which)
    g.close()
    gs.close()


@pytest.mark.parametrize("K,N,M,split", [
    (512, 272, 300, 0),     # last pair tile: 16 columns in the leader's half, none in the peer's
    (1024, 400, 257, 0),    # last pair tile ends inside the peer's half; M one past a pair tile
    (2048, 4000, 77, 0),
    (4096, 512, 300, 4),    # fixed split count on the pair tile
    (4096, 256, 129, 0),    # one N tile: the automatic split (S = 4 at 152 SMs)
])
def test_mxfp8_ragged_and_split(K, N, M, split):
    """Ragged M and N on the 256 x 256 MXFP8 CTA-pair tile, against the oracle, with the rows
    of smaller batches bitwise equal to the same rows of the full batch."""
    x, sx, w, sw = inputs(K, N, ("VAR", "VAR"), rows=M)
    y_ref, _, sabs = oracle.gemm_mxfp8(x, sx, w, sw)
    g = BiGemm(K, N, "mxfp8", split_k=split)
    assert g.config["ctas_per_tile"] == 2 and g.config["block_m"] == 256
    if split:
        assert g.config["split_k"] == split
    xd, sxd, wd, swd = dev_u8(x), dev_u8(sx), dev_u8(w), dev_u8(sw)
    y = g(xd, wd, sx=sxd, sw=swd)
    check_tolerance(host_bits(y), y_ref, sabs, oracle.TOL_BF16, f"MXFP8 K={K} N={N} M={M}")
    for M2 in (1, 2, 128, 129, 256):
        if M2 < M:
            y2 = g(xd[:M2], wd, sx=sxd[:M2], sw=swd)
            assert torch.equal(y2.view(torch.int16), y[:M2].view(torch.int16)), M2
    assert g.device_error() == 0
    g.close()


def test_mxfp8_pair_split_too_large_for_merge_staging():
    """MXFP8 on the CTA-pair tile with a fixed split of 1024: one item's partials exceed the
    epilogue staging, so the merge takes its register-batch path."""
    K, N, M = 131072, 256, 8
    x, sx, w, sw = inputs(K, N, ("VAR", "VAR"), rows=M)
    g = BiGemm(K, N, "mxfp8", split_k=1024)
    assert g.config["split_k"] == 1024 and g.config["ctas_per_tile"] == 2
    xd, sxd, wd, swd = dev_u8(x), dev_u8(sx), dev_u8(w), dev_u8(sw)
    y = g(xd, wd, sx=sxd, sw=swd)
    y_ref, _, sabs = oracle.gemm_mxfp8(x, sx, w, sw)
    check_tolerance(host_bits(y), y_ref, sabs, oracle.TOL_BF16, "MXFP8 S=1024")
    y1 = g(xd[5:6], wd, sx=sxd[5:6], sw=swd)
    assert torch.equal(y1.view(torch.int16), y[5:6].view(torch.int16))
    assert g.device_error() == 0
    g.close()
