"""Pins for the CPU oracle: checks against facts fixed by the number format,
by hand-built blocks with known values, and by exact arithmetic.

Each ``pin_*`` function takes an oracle handle and raises AssertionError on
a mismatch.  ``test_oracle.py`` runs them against the oracle; the mutation
test runs them against deliberately broken copies of it to show that every
planted mistake is caught by at least one pin.

Block layouts pinned here are the GGUF convention for Q8_0 / Q4_K / Q6_K and
Q4_0 / Q5_0 / Q5_1 / Q5_K, plus the float weights F32 / F16 / BF16 (stored
little-endian, one element each); the pages name the types and block sizes (and
Q5_0's fields) only ("05 · 8p — Persistent f16 weight cache + fused
dequant-in-GEMM", sections 1 and 2).  Hand-built blocks below
are written byte by byte from that layout, independently of the oracle's
decoder and of its encoders.
"""
from __future__ import annotations

import os
from fractions import Fraction

import numpy as np

F32, F16, BF16 = 0, 1, 30
Q4_0, Q5_0, Q5_1, Q8_0, Q4_K, Q5_K, Q6_K = 2, 6, 7, 8, 12, 13, 14
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

ONE = 0x3C00        # f16 1.0
MINUS_ONE = 0xBC00  # f16 -1.0
TWO = 0x4000        # f16 2.0
HALF = 0x3800       # f16 0.5


def f16bits(x: float) -> int:
    """Bits of an exactly representable binary16 value."""
    v = np.float16(x)
    assert float(v) == x, x
    return int(np.array(v).view(np.uint16))


def le16(v: int) -> list[int]:
    return [v & 0xFF, (v >> 8) & 0xFF]


def q4k_bytes(d: int, dmin: int, S, qs) -> np.ndarray:
    assert len(S) == 12 and len(qs) == 128
    return np.array(le16(d) + le16(dmin) + list(S) + list(qs), dtype=np.uint8)


def q6k_bytes(ql, qh, sc, d: int) -> np.ndarray:
    assert len(ql) == 128 and len(qh) == 64 and len(sc) == 16
    return np.array(list(ql) + list(qh) + [s & 0xFF for s in sc] + le16(d), dtype=np.uint8)


def q80_bytes(d: int, q) -> np.ndarray:
    assert len(q) == 32
    return np.array(le16(d) + [v & 0xFF for v in q], dtype=np.uint8)


def ints_to_f16bits(v) -> np.ndarray:
    """Small integers (|v| <= 2048) are exact in binary16."""
    a = np.asarray(v, dtype=np.float64)
    assert np.all(np.abs(a) <= 2048) and np.all(a == np.round(a))
    return a.astype(np.float16).view(np.uint16)


# ---------------------------------------------------------------------------
# O1: binary16 conversion
# ---------------------------------------------------------------------------

def read_golden_f16():
    rows = []
    with open(os.path.join(GOLDEN, "f16_rounding.txt")) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            a, b, *_ = line.split()
            rows.append((int(a, 16), int(b, 16)))
    return rows


def pin_f16_golden(orc):
    rows = read_golden_f16()
    f = np.array([a for a, _ in rows], dtype=np.uint32).view(np.float32)
    got = orc.f32_to_f16(f)
    exp = np.array([b for _, b in rows], dtype=np.uint16)
    bad = np.nonzero(got != exp)[0]
    assert bad.size == 0, [(hex(rows[i][0]), hex(int(got[i])), hex(rows[i][1])) for i in bad]


def pin_f16_to_f32_all(orc):
    """All 65536 binary16 encodings widen exactly (numpy's widening is an
    independent implementation of the same exact map)."""
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = orc.f16_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def pin_f16_roundtrip_all(orc):
    """Every non-NaN binary16 value survives widen -> narrow unchanged."""
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    keep = ~np.isnan(h.view(np.float16))
    back = orc.f32_to_f16(orc.f16_to_f32(h[keep]))
    assert np.array_equal(back, h[keep])


def pin_f16_sample_vs_numpy(orc):
    """2^21 random binary32 patterns plus every tie point between adjacent
    binary16 values against numpy's (independent) conversion."""
    g = np.random.Generator(np.random.PCG64(1234))
    bits = g.integers(0, 2**32, 1 << 21, dtype=np.uint64).astype(np.uint32)
    h = np.arange(0, 0x7C00, dtype=np.uint32).astype(np.uint16)
    lo = h[:-1].view(np.float16).astype(np.float64)
    hi = h[1:].view(np.float16).astype(np.float64)
    ties = ((lo + hi) / 2).astype(np.float32)   # exact: midpoints need <= 12 bits
    assert np.all(ties.astype(np.float64) == (lo + hi) / 2)
    f = np.concatenate([bits.view(np.float32), ties, -ties])
    f = f[~np.isnan(f)]
    with np.errstate(over="ignore"):
        ref = f.astype(np.float16).view(np.uint16)
    got = orc.f32_to_f16(f)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(hex(int(f[i:i + 1].view(np.uint32)[0])), hex(int(got[i])), hex(int(ref[i])))
                           for i in bad[:8]]


# ---------------------------------------------------------------------------
# O2: Q8_0
# ---------------------------------------------------------------------------

def pin_q8_0_identity(orc):
    """d = 1: every int8 quant decodes to itself; d = -2 gives -2q; q = 0
    with negative d gives -0 (the sign of an exact zero product)."""
    qs = np.arange(-128, 128).reshape(8, 32)
    blocks = [q80_bytes(ONE, row) for row in qs]
    blocks += [q80_bytes(f16bits(-2.0), row) for row in qs]
    out = orc.decode(Q8_0, np.concatenate(blocks)).reshape(16, 32)
    assert np.array_equal(out[:8].reshape(-1), ints_to_f16bits(qs.reshape(-1)))
    neg = -2 * qs.reshape(-1)
    exp = ints_to_f16bits(neg)
    exp[neg == 0] = 0x8000
    assert np.array_equal(out[8:].reshape(-1), exp)


def pin_q8_0_rounding_tie(orc):
    """d = 1+2^-10, q = 3: the binary32 product 3+3*2^-10 is exact and is a
    binary16 tie; it must round to even, 3+2^-8 (0x4202)."""
    q = [3] + [0] * 31
    out = orc.decode(Q8_0, q80_bytes(0x3C01, q))
    assert int(out[0]) == 0x4202, hex(int(out[0]))
    assert np.all(out[1:] == 0)


# ---------------------------------------------------------------------------
# O2: Q4_K
# ---------------------------------------------------------------------------

# sc = 1 and m = 0 for all eight sub-blocks, written byte by byte:
# bytes 0..3 hold sc[0..3] (low 6 bits) and the top 2 bits of sc[4..7];
# bytes 4..7 hold m[0..3] and the top 2 bits of m[4..7];
# bytes 8..11 hold the low 4 bits of sc[4..7] and (high nibble) of m[4..7].
S_SC1_M0 = [1, 1, 1, 1, 0, 0, 0, 0, 1, 1, 1, 1]


def q4k_nibble_positions(j: int) -> tuple[int, int]:
    """Elements fed by byte j of qs: (low nibble, high nibble)."""
    p, i = divmod(j, 32)
    return 64 * p + i, 64 * p + 32 + i


def pin_q4k_nibbles(orc):
    """d = 1, dmin = 0, all scales 1: the block decodes to its nibbles."""
    g = np.random.Generator(np.random.PCG64(7))
    qs = g.integers(0, 256, 128).tolist()
    out = orc.decode(Q4_K, q4k_bytes(ONE, 0, S_SC1_M0, qs))
    exp = np.zeros(256, dtype=np.int64)
    for j, byte in enumerate(qs):
        lo, hi = q4k_nibble_positions(j)
        exp[lo] = byte & 15
        exp[hi] = byte >> 4
    assert np.array_equal(out, ints_to_f16bits(exp))


def pin_q4k_single_byte(orc):
    """One nonzero qs byte 0x5A lights exactly two elements: 10 at the
    low-nibble position and 5 at the high-nibble position."""
    blocks, exps = [], []
    for j in range(128):
        qs = [0] * 128
        qs[j] = 0x5A
        blocks.append(q4k_bytes(ONE, 0, S_SC1_M0, qs))
        e = np.zeros(256, dtype=np.int64)
        lo, hi = q4k_nibble_positions(j)
        e[lo], e[hi] = 10, 5
        exps.append(e)
    out = orc.decode(Q4_K, np.concatenate(blocks)).reshape(128, 256)
    assert np.array_equal(out, ints_to_f16bits(np.stack(exps)).reshape(128, 256))


def q4k_expected_scale_min(S) -> list[tuple[int, int]]:
    """(sc, m) of the 8 sub-blocks from 12 packed bytes, bit by bit."""
    res = []
    for s in range(8):
        if s < 4:
            sc = S[s] & 0x3F
            m = S[s + 4] & 0x3F
        else:
            j = s - 4
            sc = (S[j + 8] & 0x0F) | ((S[j] >> 6) << 4)
            m = (S[j + 8] >> 4) | ((S[j + 4] >> 6) << 4)
        res.append((sc, m))
    return res


def pin_q4k_scale_bytes(orc):
    """Random scale bytes, all nibbles 1, d = 2, dmin = 1/2: sub-block s
    decodes to 2*sc_s - m_s/2, exact in binary16 for 6-bit sc and m."""
    g = np.random.Generator(np.random.PCG64(11))
    blocks, exps = [], []
    for _ in range(64):
        S = g.integers(0, 256, 12).tolist()
        blocks.append(q4k_bytes(TWO, HALF, S, [0x11] * 128))
        e = []
        for s, (sc, m) in enumerate(q4k_expected_scale_min(S)):
            e += [2 * sc - m / 2] * 32
        exps.append(e)
    out = orc.decode(Q4_K, np.concatenate(blocks)).reshape(64, 256)
    exp = np.array(exps).astype(np.float16).view(np.uint16)
    assert np.array_equal(out, exp)


def pin_q4k_pack_roundtrip(orc):
    """Every (sc, m) pair of 6-bit values in every sub-block slot, packed by
    the independent encoder and decoded: q = 1, d = 2, dmin = 1/2 gives
    2*sc - m/2 in that sub-block and 0 elsewhere (sc = m = 0 there)."""
    # First: the encoder reproduces hand-built bytes.
    enc = orc.pack_q4_K(ONE, 0, [1] * 8, [0] * 8, [3] * 256)
    assert np.array_equal(enc, q4k_bytes(ONE, 0, S_SC1_M0, [0x33] * 128))
    sc_v, m_v = np.meshgrid(np.arange(64), np.arange(64), indexing="ij")
    sc_v, m_v = sc_v.reshape(-1), m_v.reshape(-1)
    for s in range(8):
        blocks = []
        q = np.zeros(256, dtype=np.uint8)
        q[32 * s: 32 * s + 32] = 1
        for sc, m in zip(sc_v, m_v):
            scs = np.zeros(8, np.uint8)
            ms = np.zeros(8, np.uint8)
            scs[s], ms[s] = sc, m
            blocks.append(orc.pack_q4_K(TWO, HALF, scs, ms, q))
        out = orc.decode(Q4_K, np.concatenate(blocks)).reshape(-1, 256)
        exp = np.zeros((sc_v.size, 256))
        exp[:, 32 * s: 32 * s + 32] = (2 * sc_v - m_v / 2)[:, None]
        assert np.array_equal(out, exp.astype(np.float16).view(np.uint16)), s


def pin_q4k_double_rounding(orc):
    """Binary32 first, then binary16.  d = 293/2048, q = 7, sc = 1 gives
    d*sc*q = 1+3*2^-11 exactly; dmin = 2^-24, m = 1.  The exact difference
    1+3*2^-11-2^-24 rounds in binary32 (a tie, to even) to 1+3*2^-11, a
    binary16 tie that goes to even 1+2^-9 (0x3C02).  Rounding the exact
    value straight to binary16 would give 1+2^-10 (0x3C01).  Elements with
    q = 0 give -2^-24 (0x8001)."""
    d = f16bits(293 / 2048)
    dmin = 0x0001
    S = [1, 0, 0, 0, 1, 0, 0, 0, 0, 0, 0, 0]  # sub-block 0: sc = 1, m = 1
    qs = [7] + [0] * 127
    out = orc.decode(Q4_K, q4k_bytes(d, dmin, S, qs))
    assert int(out[0]) == 0x3C02, hex(int(out[0]))
    assert np.all(out[1:32] == 0x8001)
    assert np.all(out[32:] == 0)


def pin_q4k_signed_zero(orc):
    """d = -1, sc = 1, q = 0, m = 0: (-1*1)*0 - 0 = -0 - (+0) = -0."""
    out = orc.decode(Q4_K, q4k_bytes(MINUS_ONE, ONE, S_SC1_M0, [0] * 128))
    assert np.all(out == 0x8000)


# ---------------------------------------------------------------------------
# O2: Q6_K
# ---------------------------------------------------------------------------

QH_ZERO = [0xAA] * 64   # every 2-bit high field = 2, so with ql = 0 every q6 = 32-32 = 0


def q6k_ql_positions(j: int) -> tuple[int, int]:
    """Elements fed by ql byte j: (low nibble, high nibble)."""
    h, jj = divmod(j, 64)
    return 128 * h + jj, 128 * h + 64 + jj


def q6k_qh_position(j: int, t: int) -> int:
    """Element fed by bits 2t..2t+1 of qh byte j."""
    h, l = divmod(j, 32)
    return 128 * h + 32 * t + l


def pin_q6k_zero_and_sign(orc):
    """All q6 = 0: a positive scale gives +0, a negative one -0."""
    sc = [5, -5] * 8
    out = orc.decode(Q6_K, q6k_bytes([0] * 128, QH_ZERO, sc, ONE))
    exp = np.array([0x0000 if sc[e // 16] > 0 else 0x8000 for e in range(256)], dtype=np.uint16)
    assert np.array_equal(out, exp)


def pin_q6k_single_ql(orc):
    """A single ql nibble of 1 (high bits 2) makes q6 = 1 at one element."""
    blocks, exps = [], []
    for j in range(128):
        for nib in (0x01, 0x10):
            ql = [0] * 128
            ql[j] = nib
            blocks.append(q6k_bytes(ql, QH_ZERO, [1] * 16, ONE))
            e = np.zeros(256, dtype=np.int64)
            lo, hi = q6k_ql_positions(j)
            e[lo if nib == 0x01 else hi] = 1
            exps.append(e)
    out = orc.decode(Q6_K, np.concatenate(blocks)).reshape(-1, 256)
    assert np.array_equal(out, ints_to_f16bits(np.stack(exps)).reshape(-1, 256))


def pin_q6k_single_qh(orc):
    """A single 2-bit qh field of 3 (ql = 0) makes q6 = 48-32 = 16 at one element."""
    blocks, exps = [], []
    for j in range(64):
        for t in range(4):
            qh = list(QH_ZERO)
            qh[j] = (0xAA & ~(3 << (2 * t))) | (3 << (2 * t))
            blocks.append(q6k_bytes([0] * 128, qh, [1] * 16, ONE))
            e = np.zeros(256, dtype=np.int64)
            e[q6k_qh_position(j, t)] = 16
            exps.append(e)
    out = orc.decode(Q6_K, np.concatenate(blocks)).reshape(-1, 256)
    assert np.array_equal(out, ints_to_f16bits(np.stack(exps)).reshape(-1, 256))


def pin_q6k_scales(orc):
    """All q6 = 1 (ql nibbles 1, high bits 2): element e decodes to its
    group's int8 scale sc[e // 16], sign included."""
    sc = [-128, 127, -1, 1, 37, -37, 64, -64, 3, -3, 100, -100, 0, 2, -2, 90]
    out = orc.decode(Q6_K, q6k_bytes([0x11] * 128, QH_ZERO, sc, ONE))
    exp = ints_to_f16bits([sc[e // 16] for e in range(256)])
    exp[[e for e in range(256) if sc[e // 16] == 0]] = 0x0000
    assert np.array_equal(out, exp)


def pin_q6k_roundtrip(orc):
    """Independent encoder -> decoder: d = 1, all scales 1 returns q6."""
    g = np.random.Generator(np.random.PCG64(5))
    enc = orc.pack_q6_K(ONE, [1] * 16, [0] * 256)
    assert np.array_equal(enc, q6k_bytes([0] * 128, QH_ZERO, [1] * 16, ONE))
    blocks, exps = [], []
    for _ in range(64):
        q6 = g.integers(-32, 32, 256)
        blocks.append(orc.pack_q6_K(ONE, [1] * 16, q6))
        exps.append(q6)
    out = orc.decode(Q6_K, np.concatenate(blocks)).reshape(-1, 256)
    exp = np.stack(exps).astype(np.float64)
    e16 = exp.astype(np.float16).view(np.uint16)
    assert np.array_equal(out, e16)


def pin_q6k_rounding_tie(orc):
    """d = 1+2^-10, sc = 3, q6 = 1: the exact binary32 value 3+3*2^-10 is a
    binary16 tie and rounds to even 3+2^-8 (0x4202)."""
    ql = [0x01] + [0] * 127
    out = orc.decode(Q6_K, q6k_bytes(ql, QH_ZERO, [3] * 16, 0x3C01))
    assert int(out[0]) == 0x4202, hex(int(out[0]))
    assert np.all(out[1:] == 0)


# ---------------------------------------------------------------------------
# O4: GEMM
# ---------------------------------------------------------------------------

def f16_exact_int(h: int) -> int:
    """binary16 value as an integer multiple of 2^-24 (every finite binary16
    value is one)."""
    s = -1 if h & 0x8000 else 1
    e = (h >> 10) & 0x1F
    m = h & 0x3FF
    assert e != 0x1F
    mag = m if e == 0 else (1024 + m) << (e - 1)
    return s * mag


def random_f16(g, shape, scale_exp=(-16, 8)):
    """Finite binary16 values over a wide exponent range, subnormals included."""
    e = g.integers(0, 31, shape)
    m = g.integers(0, 1024, shape)
    s = g.integers(0, 2, shape)
    return ((s << 15) | (e << 10) | m).astype(np.uint16)


def pin_gemm_exact_tiny(orc):
    """Brute force against exact integer arithmetic: products of binary16
    values are integer multiples of 2^-48, so the sum is exact in Python
    integers.  The f64 result must lie within the recursive-summation bound
    gamma_K * sum|x*w|, gamma_K = K*u/(1-K*u), u = 2^-53."""
    g = np.random.Generator(np.random.PCG64(3))
    for (M, N, K) in [(1, 1, 1), (3, 5, 7), (8, 8, 64), (5, 2, 33)]:
        X = random_f16(g, (M, K))
        W = random_f16(g, (N, K))
        Y = orc.gemm_f64(X, W)
        u = Fraction(1, 2**53)
        gam = K * u / (1 - K * u)
        for m in range(M):
            xi = [f16_exact_int(int(v)) for v in X[m]]
            for n in range(N):
                wi = [f16_exact_int(int(v)) for v in W[n]]
                exact = Fraction(sum(a * b for a, b in zip(xi, wi)), 2**48)
                absum = Fraction(sum(abs(a * b) for a, b in zip(xi, wi)), 2**48)
                err = abs(Fraction(Y[m, n]) - exact)
                assert err <= gam * absum, (M, N, K, m, n, float(err), float(gam * absum))


def pin_gemm_onehot(orc):
    """X = identity (M = K): Y = W^T exactly (one nonzero product per
    output).  N != K so a transposed operand cannot pass."""
    g = np.random.Generator(np.random.PCG64(4))
    K, N = 48, 20
    W = random_f16(g, (N, K))
    X = np.zeros((K, K), dtype=np.uint16)
    X[np.arange(K), np.arange(K)] = ONE
    Y = orc.gemm_f64(X, W)
    Wf = W.view(np.float16).astype(np.float64)
    assert np.array_equal(Y, Wf.T)


def pin_gemm_zero_and_ones(orc):
    """X = 0 gives Y = 0; X = ones gives exact row sums of W (all terms are
    multiples of 2^-24 below 2^16*K, so the f64 sums here are exact)."""
    g = np.random.Generator(np.random.PCG64(6))
    N, K = 9, 40
    e = g.integers(1, 20, (N, K))          # moderate exponents: sums stay exact in f64
    m = g.integers(0, 1024, (N, K))
    s = g.integers(0, 2, (N, K))
    W = ((s << 15) | (e << 10) | m).astype(np.uint16)
    Y0 = orc.gemm_f64(np.zeros((3, K), np.uint16), W)
    assert np.all(Y0 == 0)
    Y1 = orc.gemm_f64(np.full((2, K), ONE, np.uint16), W)
    for n in range(N):
        exact = Fraction(sum(f16_exact_int(int(v)) for v in W[n]), 2**24)
        assert Fraction(Y1[0, n]) == exact and Fraction(Y1[1, n]) == exact


def pin_gemm_sampled_matches_full(orc):
    """The sampled form sums in the same order, so it matches bit for bit."""
    g = np.random.Generator(np.random.PCG64(8))
    M, N, K = 7, 11, 96
    X = (g.standard_normal((M, K)).astype(np.float16)).view(np.uint16)
    W = (g.standard_normal((N, K)).astype(np.float16)).view(np.uint16)
    Y = orc.gemm_f64(X, W)
    mi = g.integers(0, M, 50)
    ni = g.integers(0, N, 50)
    ys = orc.gemm_f64_sampled(X, W, mi, ni)
    assert np.array_equal(ys, Y[mi, ni])


# ---------------------------------------------------------------------------
# O2: Q4_0 / Q5_0 / Q5_1 (32-element blocks)
# ---------------------------------------------------------------------------

def q40_bytes(d: int, qs) -> np.ndarray:
    assert len(qs) == 16
    return np.array(le16(d) + list(qs), dtype=np.uint8)


def q50_bytes(d: int, qh: int, qs) -> np.ndarray:
    assert len(qs) == 16
    return np.array(le16(d) + [(qh >> (8 * i)) & 0xFF for i in range(4)] + list(qs), dtype=np.uint8)


def q51_bytes(d: int, m: int, qh: int, qs) -> np.ndarray:
    assert len(qs) == 16
    return np.array(le16(d) + le16(m) + [(qh >> (8 * i)) & 0xFF for i in range(4)] + list(qs), dtype=np.uint8)


def nibble_of(qs, e: int) -> int:
    """Element e of a 32-element block: low nibble of byte e (e < 16), high
    nibble of byte e-16."""
    return (qs[e] & 15) if e < 16 else (qs[e - 16] >> 4)


def pin_q4_0_values(orc):
    """d = 1: element e decodes to its nibble - 8 (low nibbles first)."""
    g = np.random.Generator(np.random.PCG64(21))
    blocks, exps = [], []
    for _ in range(32):
        qs = g.integers(0, 256, 16).tolist()
        blocks.append(q40_bytes(ONE, qs))
        exps += [nibble_of(qs, e) - 8 for e in range(32)]
    out = orc.decode(Q4_0, np.concatenate(blocks))
    assert np.array_equal(out, ints_to_f16bits(exps))


def pin_q4_0_sign_and_tie(orc):
    """Nibble 8 with d = -1 gives -0; d = 1+2^-10 with nibble 11 (q = 3)
    gives the binary16 tie 3+3*2^-10, rounded to even 0x4202."""
    out = orc.decode(Q4_0, q40_bytes(MINUS_ONE, [0x88] * 16))
    assert np.all(out == 0x8000)
    out = orc.decode(Q4_0, q40_bytes(0x3C01, [0x8B] + [0x88] * 15))
    assert int(out[0]) == 0x4202 and np.all(out[1:] == 0)


def pin_q5_0_values(orc):
    """d = 1: element e decodes to (nibble | bit e of qh << 4) - 16."""
    g = np.random.Generator(np.random.PCG64(22))
    blocks, exps = [], []
    for _ in range(32):
        qs = g.integers(0, 256, 16).tolist()
        qh = int(g.integers(0, 2**32))
        blocks.append(q50_bytes(ONE, qh, qs))
        exps += [(nibble_of(qs, e) | (((qh >> e) & 1) << 4)) - 16 for e in range(32)]
    out = orc.decode(Q5_0, np.concatenate(blocks))
    assert np.array_equal(out, ints_to_f16bits(exps))


def pin_q5_0_single_qh_bit(orc):
    """With every nibble 0, one set bit e of qh lifts exactly element e from
    -16 to 0 (d = 1)."""
    blocks = [q50_bytes(ONE, 1 << e, [0] * 16) for e in range(32)]
    out = orc.decode(Q5_0, np.concatenate(blocks)).reshape(32, 32)
    exp = np.full((32, 32), -16)
    np.fill_diagonal(exp, 0)
    assert np.array_equal(out, ints_to_f16bits(exp).reshape(32, 32))


def pin_q5_0_tie(orc):
    """q5 = 19 (q = 3), d = 1+2^-10: the tie 3+3*2^-10 rounds to 0x4202."""
    out = orc.decode(Q5_0, q50_bytes(0x3C01, 1, [0x03] + [0] * 15))
    assert int(out[0]) == 0x4202, hex(int(out[0]))


def pin_q5_1_values(orc):
    """d = 1, m = 1/2: element e decodes to q5 + 1/2 (no offset in Q5_1)."""
    g = np.random.Generator(np.random.PCG64(23))
    blocks, exps = [], []
    for _ in range(32):
        qs = g.integers(0, 256, 16).tolist()
        qh = int(g.integers(0, 2**32))
        blocks.append(q51_bytes(ONE, HALF, qh, qs))
        exps += [(nibble_of(qs, e) | (((qh >> e) & 1) << 4)) + 0.5 for e in range(32)]
    out = orc.decode(Q5_1, np.concatenate(blocks))
    assert np.array_equal(out, np.array(exps).astype(np.float16).view(np.uint16))


def pin_q5_1_double_rounding(orc):
    """d = 293/2048, q5 = 7 gives d*q = 1+3*2^-11 exactly; m = -2^-24.  The
    binary32 sum rounds (a tie, to even) to 1+3*2^-11, a binary16 tie that
    goes to 0x3C02; rounding the exact sum straight to binary16 would give
    0x3C01.  q5 = 0 elements give 0*d + m = -2^-24 (0x8001)."""
    out = orc.decode(Q5_1, q51_bytes(f16bits(293 / 2048), 0x8001, 0, [0x07] + [0] * 15))
    assert int(out[0]) == 0x3C02, hex(int(out[0]))
    assert np.all(out[1:] == 0x8001)


# ---------------------------------------------------------------------------
# O2: Q5_K
# ---------------------------------------------------------------------------

def q5k_bytes(d: int, dmin: int, S, qh, qs) -> np.ndarray:
    assert len(S) == 12 and len(qh) == 32 and len(qs) == 128
    return np.array(le16(d) + le16(dmin) + list(S) + list(qh) + list(qs), dtype=np.uint8)


def pin_q5k_values(orc):
    """d = 1, dmin = 0, every scale 1: element 64p+i is the low nibble of
    qs[32p+i] plus 16 * bit 2p of qh[i]; element 64p+32+i the high nibble
    plus 16 * bit 2p+1 of qh[i]."""
    g = np.random.Generator(np.random.PCG64(24))
    blocks, exps = [], []
    for _ in range(16):
        qs = g.integers(0, 256, 128).tolist()
        qh = g.integers(0, 256, 32).tolist()
        blocks.append(q5k_bytes(ONE, 0, S_SC1_M0, qh, qs))
        e = [0] * 256
        for p in range(4):
            for i in range(32):
                e[64 * p + i] = (qs[32 * p + i] & 15) + 16 * ((qh[i] >> (2 * p)) & 1)
                e[64 * p + 32 + i] = (qs[32 * p + i] >> 4) + 16 * ((qh[i] >> (2 * p + 1)) & 1)
        exps += e
    out = orc.decode(Q5_K, np.concatenate(blocks))
    assert np.array_equal(out, ints_to_f16bits(exps))


def pin_q5k_single_qh_bit(orc):
    """With all nibbles 0, bit s of qh byte i lights exactly element 32s+i
    (sub-block s, position i) with 16."""
    blocks, exps = [], []
    for s in range(8):
        for i in range(32):
            qh = [0] * 32
            qh[i] = 1 << s
            blocks.append(q5k_bytes(ONE, 0, S_SC1_M0, qh, [0] * 128))
            e = np.zeros(256, dtype=np.int64)
            e[32 * s + i] = 16
            exps.append(e)
    out = orc.decode(Q5_K, np.concatenate(blocks)).reshape(256, 256)
    assert np.array_equal(out, ints_to_f16bits(np.stack(exps)).reshape(256, 256))


def pin_q5k_scale_bytes(orc):
    """Random scale bytes (packed as in Q4_K), nibbles 1 and qh 0, d = 2,
    dmin = 1/2: sub-block s decodes to 2*sc_s - m_s/2."""
    g = np.random.Generator(np.random.PCG64(25))
    blocks, exps = [], []
    for _ in range(64):
        S = g.integers(0, 256, 12).tolist()
        blocks.append(q5k_bytes(TWO, HALF, S, [0] * 32, [0x11] * 128))
        e = []
        for s, (sc, m) in enumerate(q4k_expected_scale_min(S)):
            e += [2 * sc - m / 2] * 32
        exps.append(e)
    out = orc.decode(Q5_K, np.concatenate(blocks)).reshape(64, 256)
    assert np.array_equal(out, np.array(exps).astype(np.float16).view(np.uint16))


def pin_q5k_double_rounding(orc):
    """As for Q4_K: d*sc*q = 1+3*2^-11 (d = 293/2048, sc = 1, q = 7),
    dmin*m = 2^-24: binary32 first gives 0x3C02, the exact value 0x3C01."""
    S = [1, 0, 0, 0, 1, 0, 0, 0, 0, 0, 0, 0]
    out = orc.decode(Q5_K, q5k_bytes(f16bits(293 / 2048), 0x0001, S, [0] * 32, [7] + [0] * 127))
    assert int(out[0]) == 0x3C02, hex(int(out[0]))
    assert np.all(out[1:32] == 0x8001) and np.all(out[32:] == 0)


def _decode_words(orc, qtype, words, width):
    raw = b"".join(int(w).to_bytes(width, "little") for w in words)
    return orc.decode(qtype, np.frombuffer(raw, dtype=np.uint8))


def pin_f16_passthrough(orc):
    """An F16 weight's f16 value is the element itself: all 65536 patterns,
    stored little-endian, come back unchanged (NaN payloads included)."""
    allbits = np.arange(65536, dtype=np.uint32)
    assert np.array_equal(_decode_words(orc, F16, allbits, 2), allbits.astype(np.uint16))


# (bfloat16 bits, binary16 bits, reason)
BF16_CASES = [
    (0x3F80, 0x3C00, "1.0"),
    (0xBF80, 0xBC00, "-1.0"),
    (0x3F81, 0x3C08, "1 + 2^-7: exact, mantissa 8 * 2^-10"),
    (0x477F, 0x7BF8, "65280 = 255 * 2^8: exact, exponent 15, mantissa 1016 / 1024"),
    (0x4780, 0x7C00, "65536: past the binary16 maximum 65504 and the half-way point 65520: infinity"),
    (0xFF80, 0xFC00, "-infinity"),
    (0x8000, 0x8000, "-0 keeps its sign"),
    (0x3880, 0x0400, "2^-14: the smallest binary16 normal"),
    (0x3380, 0x0001, "2^-24: the smallest binary16 subnormal"),
    (0x3300, 0x0000, "2^-25: half the smallest subnormal, a tie, to even 0"),
    (0x3340, 0x0001, "0.75 * 2^-24: above the half-way point, up"),
    (0x3420, 0x0002, "2.5 * 2^-24: a tie, to even 2"),
    (0x3460, 0x0004, "3.5 * 2^-24: a tie, to even 4"),
    (0x35FF, 0x0020, "31.875 * 2^-24 (2^-20 * 255/128): rounds to 32 * 2^-24"),
]

# (binary32 bits, binary16 bits, reason)
F32_CASES = [
    (0x3F800000, 0x3C00, "1.0"),
    (0xC0490FDB, 0xC248, "-pi: mantissa (pi/2 - 1) * 1024 = 584.495 rounds to 584, -3.140625"),
    (0x477FEFFF, 0x7BFF, "65519.996: just below the half-way point to infinity, 65504"),
    (0x477FF000, 0x7C00, "65520: a tie between 65504 (odd significand) and 2^16, to even: infinity"),
    (0x80000000, 0x8000, "-0"),
    (0x3F801000, 0x3C00, "1 + 2^-11: a tie, to even 1.0"),
    (0x3F803000, 0x3C02, "1 + 3 * 2^-11: a tie, to even 1 + 2^-9"),
    (0x33000000, 0x0000, "2^-25: a tie, to even 0"),
    (0x33000001, 0x0001, "2^-25 (1 + 2^-23): above the tie, the smallest subnormal"),
    (0x7F800000, 0x7C00, "infinity"),
]


def pin_bf16_values(orc):
    """BF16 elements: the upper half of a binary32, rounded to binary16 as
    the table's reasons say (decoded as one little-endian stream)."""
    got = _decode_words(orc, BF16, [c[0] for c in BF16_CASES], 2)
    for (src, want, why), g in zip(BF16_CASES, got):
        assert int(g) == want, f"bf16 0x{src:04x} ({why}): got 0x{int(g):04x} want 0x{want:04x}"


def pin_f32_values(orc):
    """F32 elements rounded to binary16 as the table's reasons say (decoded
    as one little-endian stream, four bytes per element)."""
    got = _decode_words(orc, F32, [c[0] for c in F32_CASES], 4)
    for (src, want, why), g in zip(F32_CASES, got):
        assert int(g) == want, f"f32 0x{src:08x} ({why}): got 0x{int(g):04x} want 0x{want:04x}"


def pin_float_nan_stays_nan(orc):
    """A NaN element (F32 or BF16) decodes to a binary16 NaN."""
    for qt, words, width in ((F32, [0x7FC00000, 0xFF800001, 0x7F800400], 4), (BF16, [0x7FC0, 0xFF81], 2)):
        out = _decode_words(orc, qt, words, width)
        assert np.all((out & 0x7C00) == 0x7C00) and np.all((out & 0x03FF) != 0), (qt, out)


# (binary32 value, e4m3 code, reason) -- OCP e4m3: bias 7, 3 mantissa bits,
# largest finite 448, subnormals m * 2^-9, round to nearest even, clamp.
E4M3_CASES = [
    (1.0, 0x38, "1.0: exponent field 7"),
    (448.0, 0x7E, "448 = 1.75 * 2^8, the largest finite"),
    (0.5, 0x30, "0.5: exponent field 6"),
    (2.0 ** -9, 0x01, "the smallest subnormal"),
    (2.0 ** -10, 0x00, "half the smallest subnormal: a tie, to even 0"),
    (3 * 2.0 ** -10, 0x02, "1.5 * 2^-9: a tie between 1 and 2 units, to even 2"),
    (2.0 ** -6, 0x08, "the smallest normal"),
    (0.97 * 2.0 ** -6, 0x08, "7.76 units of 2^-9 round up to the smallest normal"),
    (1.0625, 0x38, "halfway between 1 and 1.125: to even 1"),
    (1.1875, 0x3A, "halfway between 1.125 and 1.25: to even 1.25"),
    (240.0, 0x77, "240 = 1.875 * 2^7"),
    (232.0, 0x76, "232 halfway between 224 and 240: to even 224"),
    (464.0, 0x7E, "halfway between 448 and 480 (480 is not finite): to even 448"),
    (480.0, 0x7E, "past 448 after rounding: clamped to 448"),
    (1e9, 0x7E, "far past the range: clamped"),
    (-1e9, 0xFE, "negative: clamped to -448"),
    (-0.0, 0x80, "-0 keeps its sign"),
    (-2.0 ** -11, 0x80, "a negative value that rounds to zero keeps its sign"),
    (-224.0, 0xF6, "-224 = -1.75 * 2^7"),
]


def pin_e4m3_values(orc):
    got = orc.f32_to_e4m3([c[0] for c in E4M3_CASES])
    for (v, want, why), g in zip(E4M3_CASES, got):
        assert int(g) == want, f"e4m3({v!r}) ({why}): got 0x{int(g):02x} want 0x{want:02x}"
    assert int(orc.f32_to_e4m3([float("nan")])[0]) == 0x7F


def pin_e4m3_decode(orc):
    """Every code decodes to (8+m)*2^(e-10) (e > 0) or m*2^-9 (e = 0) with
    its sign, 0x7F / 0xFF are NaN, and encoding a decoded value returns the
    code (-0 included)."""
    codes = np.arange(256, dtype=np.uint8)
    vals = orc.e4m3_to_f64(codes)
    for c, v in zip(codes.tolist(), vals.tolist()):
        e, m = (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            assert np.isnan(v)
            continue
        mag = (8 + m) * 2.0 ** (e - 10) if e else m * 2.0 ** -9
        assert v == (-mag if c & 0x80 else mag) and np.signbit(v) == bool(c & 0x80), c
    finite = codes[~np.isnan(vals)]
    assert np.array_equal(orc.f32_to_e4m3(orc.e4m3_to_f64(finite).astype(np.float32)), finite)


def pin_e4m3_matches_torch(orc):
    """Within +-464 (where no clamping happens) the encoder agrees with
    PyTorch's CPU float8_e4m3fn conversion on every code's value, every
    midpoint between neighbouring codes, the binary32 neighbours of each
    midpoint, and 20000 log-uniform random values."""
    torch = __import__("pytest").importorskip("torch")
    vals = np.sort(orc.e4m3_to_f64(np.arange(0, 0x7F, dtype=np.uint8)))
    mids = (vals[:-1] + vals[1:]) / 2
    mids = np.append(mids, 464.0)
    m32 = mids.astype(np.float32)
    pts = np.concatenate([vals.astype(np.float32), m32, np.nextafter(m32, np.float32(0)),
                          np.nextafter(m32, np.float32(1e9))])
    g = np.random.Generator(np.random.PCG64(31))
    rnd = (np.exp(g.uniform(np.log(2.0 ** -12), np.log(464.0), 20000))).astype(np.float32)
    pts = np.concatenate([pts, rnd])
    pts = pts[np.abs(pts) <= 464.0]
    pts = np.concatenate([pts, -pts])
    ref = torch.from_numpy(pts).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = orc.f32_to_e4m3(pts)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first {pts[bad[0]]!r}: 0x{got[bad[0]]:02x} vs 0x{ref[bad[0]]:02x}"


def pin_quantize_rows(orc):
    """Hand rows: [2, -1, 0.5, 0] has amax 2, scale RN32(2/448), inv = 224 and
    codes e4m3(448) = 0x7E, e4m3(-224) = 0xF6, e4m3(112) = 0x6E, 0; an all-zero
    row has scale 1 and zero codes; a row whose amax is 448 keeps its values
    (inv = 1); the amax is of magnitudes (a large negative value sets it)."""
    rows = np.array([[2.0, -1.0, 0.5, 0.0], [0.0, 0.0, 0.0, 0.0], [448.0, 1.0, -3.0, 0.25],
                     [-8.0, 1.0, 2.0, 4.0]], dtype=np.float16)
    q, sc = orc.quantize_e4m3_rows(rows.view(np.uint16))
    assert q[0].tolist() == [0x7E, 0xF6, 0x6E, 0x00]
    assert sc[0] == np.float32(1 / 224)   # the binary32 nearest 1/224 (not near a tie)
    assert q[1].tolist() == [0, 0, 0, 0] and sc[1] == 1.0
    # inv = 1: 448 -> 0x7E, 1 -> 0x38, -3 = -1.5*2^1 -> 0xC4, 0.25 = 2^-2 -> 0x28
    assert q[2].tolist() == [0x7E, 0x38, 0xC4, 0x28] and sc[2] == 1.0
    # amax 8, inv = 56: -448 -> 0xFE, 56 = 1.75*2^5 -> 0x66, 112 -> 0x6E, 224 -> 0x76
    assert q[3].tolist() == [0xFE, 0x66, 0x6E, 0x76] and sc[3] == np.float32(8 / 448)
    # The multiplier is RN32(448 / amax), not 1 / s: amax = 1.765625 gives
    # 448/amax = 253.7345132..., binary32 253.73451232910156; times v =
    # 1.32421875 that is 336 - 1.3e-6, which rounds (binary32 spacing 3.05e-5
    # there) to exactly 336, the e4m3 tie between 320 and 352: to even 320,
    # 0x7A.  1/s = 253.73452758789062 would give 336.00003 and 0x7B.
    q, sc = orc.quantize_e4m3_rows(np.array([[1.765625, 1.32421875]], dtype=np.float16).view(np.uint16))
    assert q[0].tolist() == [0x7E, 0x7A]


def pin_gemm_e4m3_exact(orc):
    """Tiny random codes and scales: the oracle's f64 result equals the
    exact rational value (Fractions) up to the two final f64 scalings."""
    g = np.random.Generator(np.random.PCG64(32))
    M, N, K = 3, 4, 40
    X8 = g.integers(0, 256, (M, K)).astype(np.uint8)
    W8 = g.integers(0, 256, (N, K)).astype(np.uint8)
    X8[(X8 & 0x7F) == 0x7F] = 0x10   # no NaN codes
    W8[(W8 & 0x7F) == 0x7F] = 0x11
    sx = g.uniform(0.01, 2.0, M).astype(np.float32)
    sw = g.uniform(0.01, 2.0, N).astype(np.float32)

    def frac(c):
        e, m = (c >> 3) & 15, c & 7
        v = Fraction(8 + m) * Fraction(2) ** (e - 10) if e else Fraction(m) * Fraction(2) ** -9
        return -v if c & 0x80 else v
    Y = orc.gemm_e4m3_f64(X8, sx, W8, sw)
    for m in range(M):
        for n in range(N):
            exact = sum(frac(int(X8[m, k])) * frac(int(W8[n, k])) for k in range(K))
            exact *= Fraction(float(sw[n])) * Fraction(float(sx[m]))
            assert abs(Y[m, n] - float(exact)) <= 4e-16 * max(abs(float(exact)), 1e-300), (m, n)
    mi = np.array([0, 2, 1]); ni = np.array([3, 0, 2])
    assert np.array_equal(orc.gemm_e4m3_f64_sampled(X8, sx, W8, sw, mi, ni), Y[mi, ni])


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_") and callable(v)]
