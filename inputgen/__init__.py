"""Seeded synthetic inputs for the batch-invariant GEMM y = x·W.

This module is the only code shared by the CPU oracle's tests and the CUDA
path's tests and benchmark.  It draws random numbers and encodes them into the
input formats (bf16, OCP E4M3FN, E8M0); it holds none of the GEMM's arithmetic
(no products, no sums, no output rounding).

Generator definitions (all counter-based, so any element can be regenerated
alone and row i of a matrix never depends on how many rows were drawn):

* SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014, with Vigna's published finaliser constants):
  ``word(seed, i) = mix(seed + (i + 1) * 0x9E3779B97F4A7C15)`` where
  ``mix(z) = z ^ (z >> 31)`` after ``z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9``
  and ``z = (z ^ (z >> 27)) * 0x94D049BB133111EB`` (all mod 2^64).
* Box–Muller: element i of a normal stream uses words 2i and 2i+1:
  ``u1 = ((w0 >> 11) + 1) * 2^-53`` in (0, 1], ``u2 = (w1 >> 11) * 2^-53``,
  ``z = sqrt(-2 ln u1) * cos(2 pi u2)``.
* Row-addressed matrices: element (r, c) of an [rows, cols] matrix drawn with
  seed s is stream element ``r * cols + c``; a row with fixed content C is drawn
  from seed C at row index 0, so it is the same bytes at any position.

Encodings:
* bf16: fp64 -> fp32 (IEEE round-to-nearest-even) -> bf16 (round-to-nearest-even
  on the fp32 bit pattern).  Returned as uint16 bit patterns.
* E4M3FN (OCP 8-bit float, bias 7, max 448, S.1111.111 = NaN, no infinities):
  round-to-nearest-even onto the finite grid, saturating to +-448.  uint8 codes.
* E8M0 scales: uint8 biased exponents (value 2^(e-127)); 127 is 1.0.
"""
from __future__ import annotations

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# Named seeds of the workloads (x, W, fixed target content C, variants A and B).
SEED_X = 1
SEED_W = 2
SEED_C = 3
SEED_A = 0xA
SEED_B = 0xB


def splitmix64(seed: int, idx: np.ndarray) -> np.ndarray:
    """SplitMix64 output word for counter values ``idx`` (uint64 array)."""
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + (idx.astype(np.uint64) + np.uint64(1)) * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


_CHUNK = 1 << 20


def _normal_chunk(seed: int, start: int, count: int) -> np.ndarray:
    i = np.arange(start, start + count, dtype=np.uint64)
    w0 = splitmix64(seed, np.uint64(2) * i)
    w1 = splitmix64(seed, np.uint64(2) * i + np.uint64(1))
    u1 = ((w0 >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0**-53
    u2 = (w1 >> np.uint64(11)).astype(np.float64) * 2.0**-53
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def normal(seed: int, start: int, count: int) -> np.ndarray:
    """``count`` standard normal samples (fp64), stream elements start..start+count-1."""
    out = np.empty(count, np.float64)
    for c0 in range(0, count, _CHUNK):
        c1 = min(count, c0 + _CHUNK)
        out[c0:c1] = _normal_chunk(seed, start + c0, c1 - c0)
    return out


def uniform_int(seed: int, start: int, count: int, lo: int, hi: int) -> np.ndarray:
    """Integers in [lo, hi] (inclusive) from the SplitMix64 words (modulo reduction)."""
    i = np.arange(start, start + count, dtype=np.uint64)
    w = splitmix64(seed, i)
    span = np.uint64(hi - lo + 1)
    return (w % span).astype(np.int64) + lo


# ----------------------------------------------------------------------------- encoders

def to_bf16_bits(v: np.ndarray) -> np.ndarray:
    """fp64 -> fp32 (RNE) -> bf16 (RNE on the fp32 pattern); uint16 bit patterns."""
    f = np.ascontiguousarray(v, dtype=np.float64).astype(np.float32)
    b = f.view(np.uint32)
    nan = np.isnan(f)
    lsb = (b >> np.uint32(16)) & np.uint32(1)
    with np.errstate(over="ignore"):
        r = (b + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    r = np.where(nan, np.uint32(0x7FC0), r)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 values (exact); for building inputs only."""
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _e4m3_grid() -> np.ndarray:
    """The 127 non-negative finite E4M3FN values, ordered by code 0x00..0x7E."""
    vals = []
    for code in range(0x7F):
        e, m = code >> 3, code & 7
        vals.append(m * 2.0**-9 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7))
    return np.array(vals, dtype=np.float64)


_E4M3_POS = _e4m3_grid()


def to_e4m3_codes(v: np.ndarray) -> np.ndarray:
    """fp64 -> E4M3FN codes, round-to-nearest-even on the finite grid, saturating at 448."""
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v), 448.0)
    # quantum of the binade holding a (subnormal binade below 2^-6 has quantum 2^-9)
    e = np.floor(np.log2(np.maximum(a, 2.0**-6)))
    step = 2.0 ** (e - 3.0)
    q = np.minimum(np.rint(a / step) * step, 448.0)
    code = np.searchsorted(_E4M3_POS, q).astype(np.uint8)
    sign = np.where(np.signbit(v) & (code != 0), np.uint8(0x80), np.uint8(0))
    return (code | sign).astype(np.uint8)


# ----------------------------------------------------------------------------- matrices

def normal_bf16(seed: int, rows: int, cols: int, std: float = 1.0, row0: int = 0) -> np.ndarray:
    """[rows, cols] bf16 bit patterns of N(0, std^2), rows row0.. of the seed's stream."""
    n = rows * cols
    out = np.empty(n, np.uint16)
    for c0 in range(0, n, _CHUNK):
        c1 = min(n, c0 + _CHUNK)
        out[c0:c1] = to_bf16_bits(_normal_chunk(seed, row0 * cols + c0, c1 - c0) * std)
    return out.reshape(rows, cols)


def normal_e4m3(seed: int, rows: int, cols: int, row0: int = 0) -> np.ndarray:
    """[rows, cols] E4M3FN codes of N(0, 1) samples."""
    z = normal(seed, row0 * cols, rows * cols)
    return to_e4m3_codes(z).reshape(rows, cols)


def e8m0_scales(kind: str, seed: int, rows: int, cols: int, row0: int = 0) -> np.ndarray:
    """E8M0 scale matrix: 'ID' = all 127 (2^0); 'VAR' = 127 + U{-4..4} per entry."""
    if kind == "ID":
        return np.full((rows, cols), 127, dtype=np.uint8)
    if kind == "VAR":
        s = uniform_int(seed ^ 0x5CA1E, row0 * cols, rows * cols, -4, 4) + 127
        return s.astype(np.uint8).reshape(rows, cols)
    raise ValueError(f"unknown scale kind {kind!r}")


def linspace_bf16(lo: float, hi: float, rows: int, cols: int) -> np.ndarray:
    """linspace(lo, hi, rows*cols) reshaped [rows, cols], value i = lo + i*(hi-lo)/(n-1) in fp64, -> bf16."""
    n = rows * cols
    i = np.arange(n, dtype=np.float64)
    v = lo + i * ((hi - lo) / (n - 1))
    return to_bf16_bits(v).reshape(rows, cols)


ROW_SCALES_C4 = (2.08, 0.019, 0.245)


def scaled_rows_bf16(seed: int, rows: int, cols: int, scales=ROW_SCALES_C4, row0: int = 0) -> np.ndarray:
    """N(0,1) rows scaled by scales[(row0 + r) % len(scales)], -> bf16."""
    z = normal(seed, row0 * cols, rows * cols).reshape(rows, cols)
    s = np.array([scales[(row0 + r) % len(scales)] for r in range(rows)], dtype=np.float64)
    return to_bf16_bits(z * s[:, None])


def bi_variant(base_rows: np.ndarray, target: int, content: np.ndarray) -> np.ndarray:
    """Copy of ``base_rows`` with row ``target`` replaced by ``content`` (one row)."""
    out = np.array(base_rows, copy=True)
    out[target] = content
    return out


def target_rows(m: int) -> list[int]:
    """Target positions {0, mid, last} with mid = m // 2, last = m - 1 (deduplicated)."""
    out = []
    for r in (0, m // 2, m - 1):
        if r not in out:
            out.append(r)
    return out


def rmsnorm_weight_bf16(seed: int, d: int) -> np.ndarray:
    """RMSNorm weight g[d]: 1 + 0.1 * N(0, 1), rounded to bf16 (weights of a trained norm sit
    near 1; the pages give no distribution)."""
    return to_bf16_bits(1.0 + 0.1 * normal(seed, 0, d))


# ----------------------------------------------------------------------------- attention inputs

def kv_rows_bf16(seed: int, req: int, length: int, heads: int, dim: int, which: int) -> np.ndarray:
    """Keys (which = 0) or values (which = 1) of one request, [length, heads, dim] bf16 ~ N(0, 1).
    Element (j, h, i) is stream element ((j * heads + h) * dim + i) of the request's own stream,
    so a request's content does not depend on its batch, its index or where its pages sit."""
    s = (seed * 1_000_003 + req * 7_919 + which * 104_729) & 0xFFFFFFFF
    return to_bf16_bits(normal(s, 0, length * heads * dim)).reshape(length, heads, dim)


def query_bf16(seed: int, req: int, pos: int, heads: int, dim: int) -> np.ndarray:
    """Query of request `req` at position `pos`, [heads, dim] bf16 ~ N(0, 1)."""
    s = (seed * 1_000_003 + req * 7_919 + 3 * 104_729) & 0xFFFFFFFF
    return to_bf16_bits(normal(s, pos * heads * dim, heads * dim)).reshape(heads, dim)


def paged_cache(keys: list, values: list, page_size: int, seed: int, spare_pages: int = 0):
    """Place each request's [L_b, Hkv, D] keys and values into pages of `page_size` positions,
    the physical pages of all requests shuffled by `seed` (a seeded permutation, as a paged
    allocator would hand them out).  Returns (k_cache, v_cache [P, page_size, Hkv, D] uint16,
    page_table int32 [B, max_pages]); unused table entries are -1, unused page slots zero."""
    heads, dim = keys[0].shape[1], keys[0].shape[2]
    need = [(k.shape[0] + page_size - 1) // page_size for k in keys]
    total = sum(need) + spare_pages
    max_pages = max(need) if need else 0
    perm = np.argsort(splitmix64(seed, np.arange(total, dtype=np.uint64)), kind="stable")
    kc = np.zeros((total, page_size, heads, dim), np.uint16)
    vc = np.zeros_like(kc)
    table = np.full((len(keys), max(1, max_pages)), -1, np.int32)
    nxt = 0
    for b, (k, v) in enumerate(zip(keys, values)):
        for pg in range(need[b]):
            phys = int(perm[nxt])
            nxt += 1
            table[b, pg] = phys
            rows = slice(pg * page_size, min((pg + 1) * page_size, k.shape[0]))
            n = rows.stop - rows.start
            kc[phys, :n] = k[rows]
            vc[phys, :n] = v[rows]
    return kc, vc, table
