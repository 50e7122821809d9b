"""Pins of the attention oracle (``oracle.attention_bf16``) to what the mathematics fixes, not to
itself: a single key returns its value, equal keys give the exact mean of the values, two keys
the closed-form logistic weight, tiny cases against 50-digit decimal arithmetic, invariance
under the physical placement of pages, the causal mask, independence of query tokens, and
torch's own scaled_dot_product_attention in fp64 with grouped KV heads.  Planted mistakes (KV
head h % Hkv instead of h / G, an off-by-one causal bound, a dropped scale) fail the torch
comparison.  Definition: "Batch-invariant attention", nondeterminism article."""
import decimal
from decimal import Decimal
from fractions import Fraction

import numpy as np
import pytest
import torch

import inputgen as ig
import oracle
from exact import bf16_value, to_bf16_bits_exact

SEED = 5


def make(lens, Hq, Hkv, D, page_size, seed=SEED, positions=None):
    """Requests of the given lengths; one query token per request at its last position unless
    `positions` lists (request, position) pairs."""
    keys = [ig.kv_rows_bf16(seed, b, L, Hkv, D, 0) for b, L in enumerate(lens)]
    vals = [ig.kv_rows_bf16(seed, b, L, Hkv, D, 1) for b, L in enumerate(lens)]
    kc, vc, table = ig.paged_cache(keys, vals, page_size, seed + 1, spare_pages=2)
    if positions is None:
        positions = [(b, L - 1) for b, L in enumerate(lens)]
    q = np.stack([ig.query_bf16(seed, b, p, Hq, D) for b, p in positions])
    q_seq = np.array([b for b, _ in positions], np.int32)
    q_pos = np.array([p for _, p in positions], np.int32)
    return q, q_seq, q_pos, kc, vc, table, keys, vals


def f64(bits):
    return ig.bf16_bits_to_f32(np.asarray(bits, np.uint16)).astype(np.float64)


def torch_reference(q, q_seq, q_pos, keys, vals, scale):
    """fp64 torch SDPA per query token over its own keys 0..p, KV heads repeated for the group."""
    T, Hq, D = q.shape
    out = np.empty((T, Hq, D))
    for t in range(T):
        b, p = int(q_seq[t]), int(q_pos[t])
        K = torch.from_numpy(f64(keys[b][: p + 1])).permute(1, 0, 2)      # [Hkv, L, D]
        V = torch.from_numpy(f64(vals[b][: p + 1])).permute(1, 0, 2)
        G = Hq // K.shape[0]
        K = K.repeat_interleave(G, dim=0)
        V = V.repeat_interleave(G, dim=0)
        Q = torch.from_numpy(f64(q[t]))[:, None, :]                         # [Hq, 1, D]
        out[t] = torch.nn.functional.scaled_dot_product_attention(Q, K, V, scale=scale)[:, 0, :].numpy()
    return out


def test_single_key_returns_its_value():
    q, q_seq, q_pos, kc, vc, table, keys, vals = make([1, 1, 1], 4, 2, 16, 4)
    o, v, a, e = oracle.attention_bf16(q, q_seq, q_pos, kc, vc, table, 0.25)
    for t in range(3):
        want = np.repeat(vals[t][0], 2, axis=0)                              # KV head h // 2
        assert np.array_equal(o[t], want) and np.array_equal(v[t], f64(want))


def test_equal_keys_give_the_exact_mean():
    """All keys equal: every weight is exactly 1, the output is the mean of the values (one fp64
    rounding of an exact sum), and its bf16 rounding is that of the rational mean."""
    L, Hkv, D = 37, 1, 8
    k = np.tile(ig.kv_rows_bf16(1, 0, 1, Hkv, D, 0), (L, 1, 1))
    vv = ig.kv_rows_bf16(1, 0, L, Hkv, D, 1)
    kc, vc, table = ig.paged_cache([k], [vv], 8, 3)
    q = ig.query_bf16(1, 0, 0, 2, D)[None]
    o, v, _, _ = oracle.attention_bf16(q, np.array([0], np.int32), np.array([L - 1], np.int32), kc, vc, table, 0.3)
    for h in range(2):
        for i in range(D):
            mean = sum((bf16_value(int(vv[j, 0, i])) for j in range(L)), Fraction(0)) / L
            assert abs(Fraction(v[0, h, i]) - mean) <= abs(mean) * Fraction(1, 2**52)
            assert int(o[0, h, i]) == to_bf16_bits_exact(mean)


def test_two_keys_closed_form():
    """Two keys: the weight of the first is 1 / (1 + exp(s1 - s0)), evaluated in 50 digits."""
    D = 8
    q, q_seq, q_pos, kc, vc, table, keys, vals = make([2], 1, 1, D, 2)
    scale = 0.35
    _, v, a, _ = oracle.attention_bf16(q, q_seq, q_pos, kc, vc, table, scale)
    decimal.getcontext().prec = 50
    qd = [Decimal(float(x)) for x in f64(q[0, 0])]
    s = [Decimal(scale) * sum(qd[i] * Decimal(float(f64(keys[0][j, 0, i]))) for i in range(D)) for j in range(2)]
    w0 = 1 / (1 + (s[1] - s[0]).exp())
    for i in range(D):
        v0, v1 = (Decimal(float(f64(vals[0][j, 0, i]))) for j in range(2))
        want = float(w0 * v0 + (1 - w0) * v1)
        assert abs(v[0, 0, i] - want) <= 1e-15 * a[0, 0, i]


def test_tiny_cases_against_50_digit_decimal():
    lens = [1, 3, 6, 4]
    Hq, Hkv, D, scale = 4, 2, 4, 0.5
    q, q_seq, q_pos, kc, vc, table, keys, vals = make(lens, Hq, Hkv, D, 2)
    o, v, a, _ = oracle.attention_bf16(q, q_seq, q_pos, kc, vc, table, scale)
    decimal.getcontext().prec = 50
    for t in range(len(lens)):
        b, p = int(q_seq[t]), int(q_pos[t])
        for h in range(Hq):
            kh = h // (Hq // Hkv)
            qd = [Decimal(float(x)) for x in f64(q[t, h])]
            s = [Decimal(scale) * sum(qd[i] * Decimal(float(f64(keys[b][j, kh, i]))) for i in range(D))
                 for j in range(p + 1)]
            m = max(s)
            w = [(sj - m).exp() for sj in s]
            l = sum(w)
            for i in range(D):
                num = sum(w[j] * Decimal(float(f64(vals[b][j, kh, i]))) for j in range(p + 1))
                exact = num / l
                assert abs(Decimal(v[t, h, i]) - exact) <= Decimal(1e-14) * Decimal(a[t, h, i])
                assert int(o[t, h, i]) == to_bf16_bits_exact(Fraction(exact)), (t, h, i)


def test_page_placement_and_page_size_do_not_change_a_bit():
    lens = [50, 9, 33]
    q, q_seq, q_pos, kc, vc, table, keys, vals = make(lens, 4, 2, 16, 8)
    o1, v1, _, _ = oracle.attention_bf16(q, q_seq, q_pos, kc, vc, table, 0.25)
    for page_size, seed in ((8, 77), (16, 3), (5, 11)):
        kc2, vc2, table2 = ig.paged_cache(keys, vals, page_size, seed, spare_pages=5)
        o2, v2, _, _ = oracle.attention_bf16(q, q_seq, q_pos, kc2, vc2, table2, 0.25)
        assert np.array_equal(o1, o2) and np.array_equal(v1, v2)


def test_causal_mask_ignores_later_keys():
    lens = [40]
    positions = [(0, 0), (0, 17), (0, 39)]
    q, q_seq, q_pos, kc, vc, table, keys, vals = make(lens, 2, 1, 16, 8, positions=positions)
    o1, v1, _, _ = oracle.attention_bf16(q, q_seq, q_pos, kc, vc, table, 0.25)
    keys2 = [keys[0].copy()]
    vals2 = [vals[0].copy()]
    keys2[0][18:] ^= 0x1234
    vals2[0][18:] ^= 0x0F0F
    kc2, vc2, table2 = ig.paged_cache(keys2, vals2, 8, SEED + 1, spare_pages=2)
    o2, v2, _, _ = oracle.attention_bf16(q, q_seq, q_pos, kc2, vc2, table2, 0.25)
    assert np.array_equal(v1[:2], v2[:2]) and not np.array_equal(v1[2], v2[2])


def test_query_tokens_are_independent():
    lens = [30, 12, 7]
    positions = [(0, 29), (1, 11), (0, 3), (2, 6), (1, 0)]
    q, q_seq, q_pos, kc, vc, table, _, _ = make(lens, 4, 2, 8, 4, positions=positions)
    o, v, _, _ = oracle.attention_bf16(q, q_seq, q_pos, kc, vc, table, 0.25)
    for t in range(len(positions)):
        ot, vt, _, _ = oracle.attention_bf16(q[t:t + 1], q_seq[t:t + 1], q_pos[t:t + 1], kc, vc, table, 0.25)
        assert np.array_equal(ot[0], o[t]) and np.array_equal(vt[0], v[t])


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (8, 2), (32, 8)])
def test_against_torch_sdpa_fp64(Hq, Hkv):
    lens = [1, 16, 100, 257]
    D = 64
    q, q_seq, q_pos, kc, vc, table, keys, vals = make(lens, Hq, Hkv, D, 16)
    scale = float(np.float32(1.0 / np.sqrt(D)))
    _, v, a, _ = oracle.attention_bf16(q, q_seq, q_pos, kc, vc, table, scale)
    ref = torch_reference(q, q_seq, q_pos, keys, vals, scale)
    assert np.all(np.abs(v - ref) <= 1e-13 * a)


def _mutant(kind, q, q_seq, q_pos, keys, vals, scale):
    T, Hq, D = q.shape
    Hkv = keys[0].shape[1]
    G = Hq // Hkv
    out = np.empty((T, Hq, D))
    for t in range(T):
        b, p = int(q_seq[t]), int(q_pos[t])
        n = p if kind == "off_by_one" else p + 1
        n = max(n, 1)
        for h in range(Hq):
            kh = h % Hkv if kind == "head_modulo" else h // G
            K = f64(keys[b][:n, kh])
            V = f64(vals[b][:n, kh])
            s = K @ f64(q[t, h]) * (1.0 if kind == "no_scale" else scale)
            w = np.exp(s - s.max())
            out[t, h] = (w @ V) / w.sum()
    return out


@pytest.mark.parametrize("kind", ["head_modulo", "off_by_one", "no_scale"])
def test_planted_mistakes_fail_the_torch_check(kind):
    lens = [5, 40]
    q, q_seq, q_pos, kc, vc, table, keys, vals = make(lens, 8, 2, 32, 8)
    scale = 0.125
    _, v, a, _ = oracle.attention_bf16(q, q_seq, q_pos, kc, vc, table, scale)
    ref = torch_reference(q, q_seq, q_pos, keys, vals, scale)
    assert np.all(np.abs(v - ref) <= 1e-13 * a)
    bad = _mutant(kind, q, q_seq, q_pos, keys, vals, scale)
    assert not np.all(np.abs(bad - ref) <= 1e-13 * a)


def test_tolerance_covers_fp32_evaluation_then_bf16_rounding():
    """An fp32 evaluation (sequential dot products and sums, exp perturbed by 2 ulp either way)
    rounded to bf16 stays inside oracle.attention_tolerance for every element."""
    lens = [1, 64, 700, 2048]
    Hq, Hkv, D = 8, 2, 128
    q, q_seq, q_pos, kc, vc, table, keys, vals = make(lens, Hq, Hkv, D, 16)
    scale = np.float32(1.0 / np.sqrt(D))
    _, v, a, e = oracle.attention_bf16(q, q_seq, q_pos, kc, vc, table, float(scale))
    tol = oracle.attention_tolerance(v, a, e, D, q_pos + 1)
    G = Hq // Hkv
    for ulps in (-2, 2):
        for t in range(len(lens)):
            b, p = int(q_seq[t]), int(q_pos[t])
            for h in range(Hq):
                K = ig.bf16_bits_to_f32(keys[b][: p + 1, h // G])
                V = ig.bf16_bits_to_f32(vals[b][: p + 1, h // G])
                qf = ig.bf16_bits_to_f32(q[t, h])
                s = np.zeros(p + 1, np.float32)
                for i in range(D):
                    s = (s + K[:, i] * qf[i]).astype(np.float32)
                s = (s * scale).astype(np.float32)
                w = np.exp((s - s.max()).astype(np.float32)).astype(np.float32)
                w = (w * np.float32(1 + ulps * 2.0**-23)).astype(np.float32)
                l = np.float32(0)
                acc = np.zeros(D, np.float32)
                for j in range(p + 1):
                    l = np.float32(l + w[j])
                    acc = (acc + w[j] * V[j]).astype(np.float32)
                y = ig.bf16_bits_to_f32(ig.to_bf16_bits((acc / l).astype(np.float32))).astype(np.float64)
                assert np.all(np.abs(y - v[t, h]) <= tol[t, h]), (t, h)


def test_bad_arguments_rejected():
    q, q_seq, q_pos, kc, vc, table, _, _ = make([4], 4, 2, 8, 4)
    with pytest.raises(ValueError):
        oracle.attention_bf16(q, q_seq, np.array([4], np.int32), kc, vc, table, 0.1)   # position past the table
    with pytest.raises(ValueError):
        oracle.attention_bf16(q, np.array([1], np.int32), q_pos, kc, vc, table, 0.1)   # no such request
    bad = table.copy()
    bad[0, 0] = 99
    with pytest.raises(ValueError):
        oracle.attention_bf16(q, q_seq, q_pos, kc, vc, bad, 0.1)
    with pytest.raises(ValueError):
        oracle.attention_bf16(np.zeros((1, 3, 8), np.uint16), q_seq, q_pos, kc, vc, table, 0.1)   # Hq % Hkv
