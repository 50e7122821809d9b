"""Batch-invariant decode attention ("Batch-invariant attention", nondeterminism article) on the
GPU through the C ABI of include/bi_attention.h: every element against the oracle within
oracle.attention_tolerance, a request's output bitwise independent of its batch, its index, its
page placement and page size, and of whether its earlier tokens ran in the same call (chunked
prefill); the A/B cells of the batch-invariance harness; bad inputs caught by the kernels; and
the negative control the harness must catch (a split size chosen from the batch size).

Workload: q, K, V ~ N(0, 1) in bf16, each request's content from its own stream; physical pages
handed out by a seeded permutation; the main shape is 32 query heads on 8 KV heads of 128
(grouped, G = 4) with 16-position pages."""
import ctypes

import numpy as np
import pytest
import torch

import inputgen as ig
import invariant_bi_gemm_gb300 as bg
import oracle
from gpu_util import byte_diffs, stream_ptr
from invariant_bi_gemm_gb300 import BiAttention

pytestmark = pytest.mark.gpu

SEED = 11


class Batch:
    """Requests (seed, id, length), query tokens (request index, position), a paged cache."""

    def __init__(self, reqs, tokens, Hq, Hkv, D, page_size, page_seed=1, spare=3):
        self.keys = [ig.kv_rows_bf16(sd, rid, L, Hkv, D, 0) for sd, rid, L in reqs]
        self.vals = [ig.kv_rows_bf16(sd, rid, L, Hkv, D, 1) for sd, rid, L in reqs]
        self.kc, self.vc, self.table = ig.paged_cache(self.keys, self.vals, page_size, page_seed, spare_pages=spare)
        self.q = np.stack([ig.query_bf16(reqs[b][0], reqs[b][1], p, Hq, D) for b, p in tokens])
        self.q_seq = np.array([b for b, _ in tokens], np.int32)
        self.q_pos = np.array([p for _, p in tokens], np.int32)
        self.max_pos = int(self.q_pos.max())

    def run(self, attn: BiAttention, max_pos=None):
        d = {k: torch.from_numpy(getattr(self, k)).cuda() for k in ("q_seq", "q_pos", "table")}
        bf = {k: torch.from_numpy(getattr(self, k).view(np.int16)).cuda().view(torch.bfloat16) for k in ("q", "kc", "vc")}
        o = attn(bf["q"], d["q_seq"], d["q_pos"], bf["kc"], bf["vc"], d["table"],
                 self.max_pos if max_pos is None else max_pos)
        return o.view(torch.int16).cpu().numpy().view(np.uint16)

    def oracle(self, scale):
        return oracle.attention_bf16(self.q, self.q_seq, self.q_pos, self.kc, self.vc, self.table, scale)


def decode_batch(lens, Hq, Hkv, D, page_size, seed=SEED, page_seed=1):
    reqs = [(seed, i, L) for i, L in enumerate(lens)]
    return Batch(reqs, [(i, L - 1) for i, L in enumerate(lens)], Hq, Hkv, D, page_size, page_seed)


def within(o_bits, v, a, e, D, L):
    tol = oracle.attention_tolerance(v, a, e, D, L)
    y = ig.bf16_bits_to_f32(o_bits).astype(np.float64)
    err = np.abs(y - v)
    bad = ~(err <= tol)
    assert not bad.any(), f"{int(bad.sum())} elements outside the tolerance, first at {np.argwhere(bad)[0]}"
    return float(np.max(err / np.maximum(tol, 1e-300)))


@pytest.mark.parametrize("Hq,Hkv,D,page,split", [
    (32, 8, 128, 16, 256),
    (8, 8, 64, 7, 128),
    (16, 2, 64, 16, 256),
    (8, 1, 128, 5, 512),
    (4, 4, 128, 16, 128),
    (16, 8, 128, 8, 512),
])
def test_parity_every_element(Hq, Hkv, D, page, split):
    lens = [1, 2, 127, 128, 129, 255, 256, 257, 700, 1500]
    bt = decode_batch(lens, Hq, Hkv, D, page)
    attn = BiAttention(Hq, Hkv, D, page, split_size=split)
    scale = attn.scale
    o = bt.run(attn)
    assert attn.device_error() == 0
    o_ref, v, a, e = bt.oracle(np.float32(scale))
    worst = within(o, v, a, e, D, bt.q_pos + 1)
    same = float(np.mean(o == o_ref))
    attn.close()
    print(f"attention Hq={Hq} Hkv={Hkv} D={D} page={page} split={split}: max err/tol {worst:.3g}, "
          f"bits equal to the oracle's rounding {same:.4f}")


def test_request_independent_of_batch_index_and_pages():
    """The same request (its own content stream) alone, at index 17 of a batch of 24 others,
    with its pages permuted differently, and with 32-position pages: identical bits."""
    Hq, Hkv, D = 32, 8, 128
    target = (SEED, 999, 1000)
    alone = Batch([target], [(0, 999)], Hq, Hkv, D, 16)
    a16 = BiAttention(Hq, Hkv, D, 16)
    golden = alone.run(a16)
    others = [(SEED + 1, i, int(L)) for i, L in enumerate(ig.uniform_int(3, 0, 24, 1, 1500))]
    reqs = others[:17] + [target] + others[17:]
    tokens = [(i, r[2] - 1) for i, r in enumerate(reqs)]
    for page_seed in (2, 3):
        big = Batch(reqs, tokens, Hq, Hkv, D, 16, page_seed=page_seed)
        o = big.run(a16)
        assert byte_diffs(o[17:18], golden) == 0
    a32 = BiAttention(Hq, Hkv, D, 32)
    big32 = Batch(reqs, tokens, Hq, Hkv, D, 32, page_seed=4)
    assert byte_diffs(big32.run(a32)[17:18], golden) == 0
    assert a16.device_error() == 0 and a32.device_error() == 0
    a16.close()
    a32.close()


def test_chunked_prefill_matches_single_token_steps():
    """Positions 500..599 of one request as one chunk of 100 query tokens (next to another
    request's decode token) give the bits of 100 single-token calls."""
    Hq, Hkv, D = 32, 8, 128
    reqs = [(SEED, 5, 600), (SEED, 6, 3000)]
    chunk = [(0, p) for p in range(500, 600)] + [(1, 2999)]
    attn = BiAttention(Hq, Hkv, D, 16)
    o_chunk = Batch(reqs, chunk, Hq, Hkv, D, 16).run(attn)
    for k, (b, p) in enumerate(chunk):
        if k % 9 and k != len(chunk) - 1:
            continue
        o1 = Batch(reqs, [(b, p)], Hq, Hkv, D, 16, page_seed=7).run(attn)
        assert byte_diffs(o1[0:1], o_chunk[k:k + 1]) == 0, (b, p)
    assert attn.device_error() == 0
    attn.close()


def test_bi_cells_across_batch_sizes():
    """A/B cells: the target slot holds the fixed request C, every other slot a request from
    seed A or seed B (different lengths too); C's output is the same in both and equal to C run
    alone, for targets {0, mid, last}."""
    Hq, Hkv, D = 16, 4, 64
    attn = BiAttention(Hq, Hkv, D, 16)
    C = (ig.SEED_C, 0, 777)
    golden = Batch([C], [(0, 776)], Hq, Hkv, D, 16).run(attn)
    total = 0
    for M in (1, 2, 7, 64, 129):
        la = ig.uniform_int(ig.SEED_A, 0, M, 1, 900)
        lb = ig.uniform_int(ig.SEED_B, 0, M, 1, 900)
        for t in ig.target_rows(M):
            outs = []
            for seed, lens in ((ig.SEED_A, la), (ig.SEED_B, lb)):
                reqs = [(seed, i, int(L)) for i, L in enumerate(lens)]
                reqs[t] = C
                tokens = [(i, r[2] - 1) for i, r in enumerate(reqs)]
                outs.append(Batch(reqs, tokens, Hq, Hkv, D, 16, page_seed=seed).run(attn)[t:t + 1])
            total += byte_diffs(outs[0], outs[1]) + byte_diffs(outs[0], golden)
    assert total == 0
    assert attn.device_error() == 0
    attn.close()


def test_negative_control_batch_keyed_split_size_is_caught():
    """A split size chosen from the batch size (128 positions for a batch of at most 16 tokens,
    512 above: more parallelism when the batch is small, the strategy the article warns about)
    changes the targets' bits between batch sizes; the fixed split size does not."""
    Hq, Hkv, D = 32, 8, 128
    small, large, fixed = (BiAttention(Hq, Hkv, D, 16, split_size=s) for s in (128, 512, 256))
    targets = [(SEED, 40 + i, 3000 - 37 * i) for i in range(12)]
    others = [(SEED + 2, i, 500) for i in range(20)]
    tok = lambda reqs: [(i, r[2] - 1) for i, r in enumerate(reqs)]
    alone = [Batch([tg], tok([tg]), Hq, Hkv, D, 16) for tg in targets]
    crowd = Batch(targets + others, tok(targets + others), Hq, Hkv, D, 16)
    out_large, out_fixed = crowd.run(large), crowd.run(fixed)
    keyed = steady = 0
    for i, b in enumerate(alone):
        keyed += byte_diffs(b.run(small)[0:1], out_large[i:i + 1])
        steady += byte_diffs(b.run(fixed)[0:1], out_fixed[i:i + 1])
    assert steady == 0 and keyed > 0
    print(f"attention control: fixed split size diffs {steady}, batch-keyed split size diffs {keyed}")
    for a in (small, large, fixed):
        a.close()


@pytest.mark.parametrize("lens", [[32768, 8192, 1], [32768], [4096] * 8])
def test_long_context_sampled(lens):
    """Long contexts against the oracle: a call of 648 units (the three-block TMA kernel over
    more than one round) and two calls of 512 units (one round of the four-block build)."""
    Hq, Hkv, D = 32, 8, 128
    bt = decode_batch(lens, Hq, Hkv, D, 16)
    attn = BiAttention(Hq, Hkv, D, 16)
    o = bt.run(attn)
    assert attn.device_error() == 0
    _, v, a, e = bt.oracle(np.float32(attn.scale))
    within(o, v, a, e, D, bt.q_pos + 1)
    attn.close()


def test_merge_of_long_split_lists():
    """Contexts past 64 splits (the merge's four groups then hold more than 16 splits each and are
    summed over several batches of loads, in the same order): every element against the oracle,
    and the long request's bits unchanged alone and beside a short one."""
    Hq, Hkv, D = 32, 8, 128
    lens = [40000, 33000, 100]
    bt = decode_batch(lens, Hq, Hkv, D, 16)
    attn = BiAttention(Hq, Hkv, D, 16)
    o = bt.run(attn)
    assert attn.device_error() == 0
    _, v, a, e = bt.oracle(np.float32(attn.scale))
    within(o, v, a, e, D, bt.q_pos + 1)
    alone = decode_batch(lens[:1], Hq, Hkv, D, 16).run(attn)
    assert byte_diffs(alone, o[:1]) == 0
    attn.close()


def test_positions_written_by_the_preceding_kernel():
    """The tokens' positions written on the stream by a kernel right before each call, as a serving
    loop's scheduler does: each output equals that of the same call with the positions written
    and the device synchronised first (the attention and merge kernels start before the kernel
    before them has finished and must still read the new positions), for a small batch (unit
    records derived in the attention kernel) and a larger one (the plan kernel first)."""
    Hq, Hkv, D = 32, 8, 128
    for lens in ([5000, 3000], [700] * 40):
        bt = decode_batch(lens, Hq, Hkv, D, 16)
        attn = BiAttention(Hq, Hkv, D, 16)
        d = {k: torch.from_numpy(getattr(bt, k)).cuda() for k in ("q_seq", "q_pos", "table")}
        bf = {k: torch.from_numpy(getattr(bt, k).view(np.int16)).cuda().view(torch.bfloat16)
              for k in ("q", "kc", "vc")}
        sets = [bt.q_pos, bt.q_pos // 2, np.maximum(bt.q_pos - 777, 0)]
        srcs = [torch.from_numpy(ps.astype(np.int32)).cuda() for ps in sets]
        refs = []
        for src in srcs:
            d["q_pos"].copy_(src)
            torch.cuda.synchronize()
            refs.append(attn.run(bf["q"], d["q_seq"], d["q_pos"], bf["kc"], bf["vc"], d["table"], bt.max_pos).clone())
            torch.cuda.synchronize()
        outs = []
        for i in range(9):
            torch.add(srcs[i % 3], 0, out=d["q_pos"])      # a kernel on the stream writes the positions
            outs.append(attn.run(bf["q"], d["q_seq"], d["q_pos"], bf["kc"], bf["vc"], d["table"], bt.max_pos))
        torch.cuda.synchronize()
        assert attn.device_error() == 0
        for i, o in enumerate(outs):
            assert torch.equal(o.view(torch.int16), refs[i % 3].view(torch.int16)), (lens[:2], i)
        attn.close()


def test_repeat_runs_identical():
    bt = decode_batch([300, 5000, 17, 1024], 32, 8, 128, 16)
    attn = BiAttention(32, 8, 128, 16)
    first = bt.run(attn)
    for _ in range(50):
        assert np.array_equal(bt.run(attn), first)
    attn.close()


def test_bad_inputs_are_caught_by_the_kernels():
    """A position above max_pos and a page-table entry of -1 are reported by
    bi_attention_get_device_error (the kernels skip them); the handle keeps working."""
    Hq, Hkv, D = 8, 2, 64
    bt = decode_batch([100, 300], Hq, Hkv, D, 16)
    attn = BiAttention(Hq, Hkv, D, 16)
    good = bt.run(attn)
    assert attn.device_error() == 0
    bt.run(attn, max_pos=50)                       # q_pos 99 and 299 exceed the bound
    assert attn.device_error() == bg.BI_GEMM_ERR_INVALID_ARG
    saved = bt.table.copy()
    bt.table[1, 3] = -1
    bt.run(attn)
    assert attn.device_error() == bg.BI_GEMM_ERR_INVALID_ARG
    bt.table = saved
    assert np.array_equal(bt.run(attn), good) and attn.device_error() == 0
    attn.close()


def test_empty_batch_and_misaligned_pointers():
    import ctypes
    attn = BiAttention(8, 2, 64, 16)
    z = torch.zeros(64, dtype=torch.int32, device="cuda")
    zb = torch.zeros(4096, dtype=torch.bfloat16, device="cuda")
    L, V = bg.library(), ctypes.c_void_p
    assert L.bi_attention_run(V(attn.handle), V(zb.data_ptr()), 0, V(z.data_ptr()), V(z.data_ptr()), V(zb.data_ptr()),
                              V(zb.data_ptr()), 1, V(z.data_ptr()), 1, 1, 0, V(zb.data_ptr()), V(stream_ptr())) == 0
    assert L.bi_attention_run(V(attn.handle), V(zb.data_ptr() + 2), 1, V(z.data_ptr()), V(z.data_ptr()),
                              V(zb.data_ptr()), V(zb.data_ptr()), 1, V(z.data_ptr()), 1, 1, 0, V(zb.data_ptr()),
                              V(stream_ptr())) == bg.BI_GEMM_ERR_ALIGNMENT
    assert L.bi_attention_run(V(attn.handle), V(zb.data_ptr()), 1, V(z.data_ptr() + 2), V(z.data_ptr()),
                              V(zb.data_ptr()), V(zb.data_ptr()), 1, V(z.data_ptr()), 1, 1, 0, V(zb.data_ptr()),
                              V(stream_ptr())) == bg.BI_GEMM_ERR_ALIGNMENT
    attn.close()


def run_pinned(bt, Hq, Hkv, D, page, kernel, split=512):
    """bt on a handle of the test-only controls library with the kernel pinned (1: TMA page boxes,
    2: row copies), whichever the product would pick for the call."""
    from gpu_util import Controls
    L = Controls().L
    P, V = ctypes.c_void_p, ctypes.c_void_p
    h = P()
    assert L.bi_ctl_attention_create(ctypes.byref(h), Hq, Hkv, D, page, ctypes.c_float(float(D) ** -0.5), split) == 0
    d = {k: torch.from_numpy(getattr(bt, k)).cuda() for k in ("q_seq", "q_pos", "table")}
    bf = {k: torch.from_numpy(getattr(bt, k).view(np.int16)).cuda().view(torch.bfloat16) for k in ("q", "kc", "vc")}
    o = torch.full_like(bf["q"], float("nan"))
    rc = L.bi_ctl_attention_run_kernel(h, V(bf["q"].data_ptr()), bf["q"].shape[0], V(d["q_seq"].data_ptr()),
                                       V(d["q_pos"].data_ptr()), V(bf["kc"].data_ptr()), V(bf["vc"].data_ptr()),
                                       bf["kc"].shape[0], V(d["table"].data_ptr()), d["table"].shape[0],
                                       d["table"].shape[1], bt.max_pos, V(o.data_ptr()), kernel, stream_ptr())
    assert rc == 0, rc
    assert L.bi_ctl_attention_get_device_error(h, stream_ptr()) == 0
    assert L.bi_ctl_attention_destroy(h) == 0
    return o.view(torch.int16).cpu().numpy().view(np.uint16)


def test_tma_page_boxes_and_row_copies_give_the_same_bits():
    """Page sizes 8, 16, 32 and 64 can run the kernel whose producer warp loads pages as TMA
    boxes; every page size the kernel whose threads copy rows.  Their arithmetic is the same, so
    the same requests give the same bits whichever runs (each kernel pinned through the test
    controls), including ragged last stages (lengths that end inside a page and inside a
    16-position step) and single-key splits; the product's own choice gives them too."""
    Hq, Hkv, D = 32, 8, 128
    lens = [1, 15, 17, 63, 64, 65, 200, 511, 512, 513, 1000, 2049]
    outs, flags = {}, {}
    for page in (8, 16, 32, 64, 12, 1):
        attn = BiAttention(Hq, Hkv, D, page, split_size=512)
        flags[page] = attn.config["tma_pages"]
        bt = decode_batch(lens, Hq, Hkv, D, page, page_seed=page)
        outs[page] = bt.run(attn)
        assert attn.device_error() == 0
        attn.close()
        if flags[page]:
            assert byte_diffs(run_pinned(bt, Hq, Hkv, D, page, 1), outs[page]) == 0, ("TMA", page)
        assert byte_diffs(run_pinned(bt, Hq, Hkv, D, page, 2), outs[page]) == 0, ("rows", page)
    assert flags == {8: 1, 16: 1, 32: 1, 64: 1, 12: 0, 1: 0}
    for page in (16, 32, 64, 12, 1):
        assert byte_diffs(outs[page], outs[8]) == 0, page


@pytest.mark.parametrize("lens", [[32768], [4096] * 8, [28672], [3000] * 20])
def test_kernel_choice_changes_no_bit(lens):
    """A call whose units fit in one round of the TMA kernel's four-block variant but not of its
    three-block one runs the four-block variant (batch 1 x 32768 and 8 x 4096: 512 units);
    smaller calls run the three-block variant in one round (batch 1 x 28672: 448 units), larger
    ones persistently (20 x 3000).  Whichever the product picks, the bits are those of the TMA
    and the row-copy kernels pinned, and the request alone (batch 1) gives the same bits as
    inside its batch."""
    Hq, Hkv, D = 32, 8, 128
    bt = decode_batch(lens, Hq, Hkv, D, 16)
    attn = BiAttention(Hq, Hkv, D, 16)
    auto = bt.run(attn)
    assert attn.device_error() == 0
    assert byte_diffs(run_pinned(bt, Hq, Hkv, D, 16, 1), auto) == 0
    assert byte_diffs(run_pinned(bt, Hq, Hkv, D, 16, 2), auto) == 0
    one = decode_batch(lens[:1], Hq, Hkv, D, 16).run(attn)
    assert byte_diffs(one, auto[:1]) == 0
    attn.close()


@pytest.mark.parametrize("D,G", [(64, 8), (64, 1), (128, 2)])
def test_tma_page_boxes_other_head_shapes(D, G):
    """The TMA kernel for other head dimensions and group sizes against the row-copy kernel."""
    Hkv = 4
    lens = [3, 64, 129, 777]
    a = BiAttention(G * Hkv, Hkv, D, 16, split_size=256)
    b = BiAttention(G * Hkv, Hkv, D, 4, split_size=256)
    assert a.config["tma_pages"] == 1 and b.config["tma_pages"] == 0
    oa = decode_batch(lens, G * Hkv, Hkv, D, 16).run(a)
    ob = decode_batch(lens, G * Hkv, Hkv, D, 4).run(b)
    assert a.device_error() == 0 and b.device_error() == 0
    assert byte_diffs(oa, ob) == 0
    a.close()
    b.close()


def test_tma_ring_wait_expires_reports_timeout_and_handle_survives():
    """Failure injection (test controls): block 0's producer never issues its first load, so its
    consumers' bounded waits on the ring expire after 50 ms; the run reports BI_GEMM_ERR_TIMEOUT
    through bi_attention_get_device_error, and the next ordinary run on the same handle gives
    the golden bits.  The handle lives in the controls library (each library has its own CUDA
    runtime, so a handle is used only with the library that made it)."""
    from gpu_util import Controls
    L = Controls().L
    P = ctypes.c_void_p
    Hq, Hkv, D = 32, 8, 128
    bt = decode_batch([700, 1500, 64], Hq, Hkv, D, 16)
    attn = BiAttention(Hq, Hkv, D, 16)
    assert attn.config["tma_pages"] == 1
    golden = bt.run(attn)
    assert attn.device_error() == 0
    h = P()
    assert L.bi_ctl_attention_create(ctypes.byref(h), Hq, Hkv, D, 16, ctypes.c_float(attn.scale), 0) == 0
    d = {k: torch.from_numpy(getattr(bt, k)).cuda() for k in ("q_seq", "q_pos", "table")}
    bf = {k: torch.from_numpy(getattr(bt, k).view(np.int16)).cuda().view(torch.bfloat16) for k in ("q", "kc", "vc")}
    o = torch.empty_like(bf["q"])
    V = ctypes.c_void_p
    args = (V(bf["q"].data_ptr()), bf["q"].shape[0], V(d["q_seq"].data_ptr()), V(d["q_pos"].data_ptr()),
            V(bf["kc"].data_ptr()), V(bf["vc"].data_ptr()), bf["kc"].shape[0], V(d["table"].data_ptr()),
            d["table"].shape[0], d["table"].shape[1], bt.max_pos, V(o.data_ptr()))
    bits = lambda: o.view(torch.int16).cpu().numpy().view(np.uint16)
    assert L.bi_ctl_attention_run(h, *args, V(stream_ptr())) == 0
    assert L.bi_ctl_attention_get_device_error(h, V(stream_ptr())) == 0
    assert np.array_equal(bits(), golden)
    o.zero_()
    assert L.bi_ctl_attention_stall(h, *args, 50_000_000, V(stream_ptr())) == 0
    assert L.bi_ctl_attention_get_device_error(h, V(stream_ptr())) == bg.BI_GEMM_ERR_TIMEOUT
    assert L.bi_ctl_attention_run(h, *args, V(stream_ptr())) == 0
    assert L.bi_ctl_attention_get_device_error(h, V(stream_ptr())) == 0
    assert np.array_equal(bits(), golden)
    L.bi_ctl_attention_destroy(h)
    attn.close()
