"""Pins that tie the CPU oracle to the pages and to mathematics.

Each function takes an oracle object (``oracle.Oracle``) and raises
AssertionError when the oracle disagrees with something fixed outside the
oracle itself: hand-computed blocks (tests/golden), exact rational
rounding, invariants of the quantiser, the int32 bound, a special case that
reduces to a plain integer matvec, and fp64 brute force over dequantised
elements.  The element decoding used here is written from the page's
format table independently of the oracle's C code.

Source of every fixed fact: page "Legacy-ISA ML Inference Runtime -- Design
Spec", Sec. 4 (Quantization Formats), Sec. 5 (Kernel Interface: row range
[r0, r1), rounding rule) and Sec. 7 (Testing: quantize->dequantize error
<= d/2, zero block handling, clamp to +-127, per-block int32 sums exact).
"""
from __future__ import annotations

import json
import os
from fractions import Fraction

import numpy as np

QK = 32
Q8_0, Q4_0 = 0, 1
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
U = 2.0 ** -24  # unit roundoff of binary32


# ----------------------------------------------------------------------------
# independent helpers
# ----------------------------------------------------------------------------
def f32_from_hex(h: str) -> np.float32:
    return np.array([int(h, 16)], dtype=np.uint32).view(np.float32)[0]


def nearest_f32(fr: Fraction) -> np.float32:
    """The binary32 value nearest to the exact rational ``fr`` (ties to even)."""
    c = np.float32(float(fr))
    cands = [c, np.nextafter(c, np.float32(np.inf)), np.nextafter(c, np.float32(-np.inf))]
    best = None
    for v in cands:
        if not np.isfinite(v):
            continue
        err = abs(Fraction(float(v)) - fr)
        key = (err, int(np.array([v], dtype=np.float32).view(np.uint32)[0]) & 1)
        if best is None or key < best[0]:
            best = (key, v)
    return best[1]


def parse_rational(s: str, amax: np.float32) -> Fraction:
    num, den = s.split("/")
    if num.startswith("hex:"):
        n = Fraction(float(f32_from_hex(num[4:])))
    else:
        n = Fraction(int(num))
    out = n / int(den)
    # the fixture's rational must be amax/127 of its own inputs
    assert out == Fraction(float(amax)) / 127, (s, amax)
    return out


def decode_q4_elements(qbytes: np.ndarray, cols: int) -> np.ndarray:
    """Element values (nibble - 8) of Q4_0 rows, from the format table:
    element e of a block sits in byte e (low nibble) for e < 16 and in byte
    e - 16 (high nibble) for e >= 16."""
    rows = qbytes.shape[0]
    out = np.empty((rows, cols), dtype=np.int64)
    qb = qbytes.reshape(rows, cols // QK, 16).astype(np.int64)
    for e in range(QK):
        if e < 16:
            nib = qb[:, :, e] & 0xF
        else:
            nib = qb[:, :, e - 16] >> 4
        out[:, e::QK] = nib - 8
    return out


def weight_elements(wtype, wq, cols):
    if wtype == Q4_0:
        return decode_q4_elements(wq, cols)
    return wq.astype(np.int64).reshape(wq.shape[0], cols)


def random_block_inputs(rng, nblocks):
    """Blocks with varied magnitude: N(0,1) scaled by 10^U(-30, 30) per block,
    some exact zeros, some repeated maxima."""
    x = rng.standard_normal((nblocks, QK)).astype(np.float32)
    scale = (10.0 ** rng.uniform(-30, 30, size=(nblocks, 1))).astype(np.float32)
    x = (x * scale).astype(np.float32)
    x[rng.random((nblocks, QK)) < 0.05] = 0.0
    dup = rng.random(nblocks) < 0.1
    x[dup, 1] = -x[dup, 0]
    return x


# ----------------------------------------------------------------------------
# pins
# ----------------------------------------------------------------------------
def pin_golden_quantize(O):
    g = json.load(open(os.path.join(GOLDEN, "quantize_q8_blocks.json")))
    for blk in g["blocks"]:
        x = np.zeros(QK, dtype=np.float32)
        for i, h in blk.get("x_hex", {}).items():
            x[int(i)] = f32_from_hex(h)
        if "x_int" in blk:
            x[:] = np.array(blk["x_int"], dtype=np.float32)
        q, d = O.quantize_q8(x)
        if "q_all" in blk:
            want = np.array(blk["q_all"], dtype=np.int8)
        else:
            want = np.zeros(QK, dtype=np.int8)
            for i, v in blk["q"].items():
                want[int(i)] = v
        assert np.array_equal(q, want), (blk["name"], q, want)
        amax = np.max(np.abs(x))
        dwant = nearest_f32(parse_rational(blk["d"], amax))
        assert d[0].view(np.uint32) == np.float32(dwant).view(np.uint32), (blk["name"], d[0], dwant)


def _q4_bytes(spec: str) -> np.ndarray:
    if spec.startswith("byte j = j | ((15 - j) << 4)"):
        return np.array([j | ((15 - j) << 4) for j in range(16)], dtype=np.uint8)
    if spec == "all 0x00":
        return np.zeros(16, dtype=np.uint8)
    raise ValueError(spec)


def _vec(spec: str) -> np.ndarray:
    if spec.startswith("all "):
        return np.full(QK, int(spec[4:]), dtype=np.int8)
    if spec.startswith("qx[e] = e"):
        return np.arange(QK, dtype=np.int8)
    raise ValueError(spec)


def pin_golden_block_dot(O):
    g = json.load(open(os.path.join(GOLDEN, "block_dot.json")))
    for c in g["q4"]:
        s = O.block_sumi(Q4_0, _q4_bytes(c["bytes"]).reshape(1, 16), 1, QK, _vec(c["qx"]))
        assert int(s[0, 0]) == c["sumi"], (c["name"], int(s[0, 0]))
    for c in g["q8"]:
        s = O.block_sumi(Q8_0, _vec(c["w"]).reshape(1, QK), 1, QK, _vec(c["qx"]))
        assert int(s[0, 0]) == c["sumi"], (c["name"], int(s[0, 0]))
    assert 32 * 127 * 127 < 2 ** 31 and 32 * 8 * 127 == 32512


def pin_quantize_invariants(O, nblocks=1 << 15, seed=1):
    """Clamp to [-127, 127] (never -128), the largest |x| maps to +-127, the
    d = 0 rule, d = nearest float32 to amax/127, and the Sec. 7 bound
    |x - q*d| <= d/2 with the slack the float32 id/d rounding allows:
    |x/d - x*id| <= 127*3u and the add before trunc can move a value that
    is within half an ulp (<= 2^-18 below 64) of a tie."""
    rng = np.random.default_rng(seed)
    x = random_block_inputs(rng, nblocks)
    x[:4] = 0.0
    q, d = O.quantize_q8(x.reshape(1, -1))
    q = q.reshape(nblocks, QK).astype(np.int64)
    d = d.reshape(nblocks)
    assert q.min() >= -127 and q.max() <= 127
    amax = np.abs(x).max(axis=1)
    zero = amax == 0
    assert np.all(d[zero] == 0) and np.all(q[zero] == 0)
    # d is the correctly rounded quotient (check a sample exactly)
    for i in rng.choice(nblocks, 256, replace=False):
        assert d[i] == nearest_f32(Fraction(float(amax[i])) / 127)
    normal = amax >= np.float32(2e-36)  # id finite and d a normal number
    am = np.abs(x) == amax[:, None]
    hit = am & normal[:, None]
    assert np.all(np.abs(q[hit]) == 127)
    assert np.all(np.sign(q[hit]) == np.sign(x[hit]))
    xd = x.astype(np.float64)
    err = np.abs(xd - q * d.astype(np.float64)[:, None])
    bound = d.astype(np.float64)[:, None] * (0.5 + 127 * 3 * U + 2.0 ** -18)
    assert np.all(err[normal] <= bound[normal]), float(np.max(err[normal] / bound[normal]))


def pin_bruteforce_fp64(O, seed=2):
    """fp64 brute force over dequantised elements (w_k*dw)*(x_k*dx) on tiny
    matrices against the oracle's float32 y; tolerance = the recursive
    float32 summation bound (nb + 2) u sum_b |t_b| with t_b the exact block
    terms.  Block sums are compared exactly against int64 sums."""
    rng = np.random.default_rng(seed)
    for trial in range(24):
        wtype = (Q4_0, Q8_0)[trial % 2]
        rows = int(rng.integers(1, 9))
        cols = QK * int(rng.integers(1, 5))
        nb = cols // QK
        if wtype == Q4_0:
            wq = rng.integers(0, 256, size=(rows, cols // 2), dtype=np.uint8)
            wd = rng.uniform(1e-3, 1e-2, size=(rows, nb)).astype(np.float32)
        else:
            wq = rng.integers(-127, 128, size=(rows, cols), dtype=np.int8)
            wd = rng.uniform(1e-4, 1e-3, size=(rows, nb)).astype(np.float32)
        xq = rng.integers(-127, 128, size=cols, dtype=np.int8)
        xd = rng.uniform(1e-3, 1e-1, size=nb).astype(np.float32)
        y = O.matvec(wtype, wq, wd, rows, cols, xq, xd)
        sumi = O.block_sumi(wtype, wq, rows, cols, xq)
        we = weight_elements(wtype, wq, cols)
        for r in range(rows):
            exact = 0.0
            absterms = 0.0
            for b in range(nb):
                s = 0
                acc = 0.0
                for j in range(QK):
                    k = b * QK + j
                    s += int(we[r, k]) * int(xq[k])
                    acc += (float(we[r, k]) * float(wd[r, b])) * (float(xq[k]) * float(xd[b]))
                assert int(sumi[r, b]) == s, (trial, r, b)
                exact += acc
                absterms += abs(s * float(wd[r, b]) * float(xd[b]))
            tol = (nb + 2) * U * (1 + 1e-6) * absterms + 1e-300
            assert abs(float(y[r]) - exact) <= tol, (trial, r, float(y[r]), exact, tol)


def pin_unit_scales_integer_matvec(O, seed=3):
    """With every dw = dx = 1 the product is a plain integer matvec of the
    decoded weights, exact in float32 while |y| < 2^24."""
    rng = np.random.default_rng(seed)
    for wtype in (Q4_0, Q8_0):
        rows, cols = 7, 128
        nb = cols // QK
        if wtype == Q4_0:
            wq = rng.integers(0, 256, size=(rows, cols // 2), dtype=np.uint8)
        else:
            wq = rng.integers(-127, 128, size=(rows, cols), dtype=np.int8)
        wd = np.ones((rows, nb), dtype=np.float32)
        xq = rng.integers(-127, 128, size=cols, dtype=np.int8)
        xd = np.ones(nb, dtype=np.float32)
        y = O.matvec(wtype, wq, wd, rows, cols, xq, xd)
        ref = weight_elements(wtype, wq, cols) @ xq.astype(np.int64)
        assert np.array_equal(y.astype(np.int64), ref), (wtype, y, ref)
        assert np.all(np.abs(ref) < 2 ** 24)


def pin_row_range(O, seed=4):
    """Only rows [r0, r1) are written (Sec. 5: matvec processes rows [r0, r1))."""
    rng = np.random.default_rng(seed)
    rows, cols = 10, 64
    wq = rng.integers(0, 256, size=(rows, cols // 2), dtype=np.uint8)
    wd = rng.uniform(1e-3, 1e-2, size=(rows, 2)).astype(np.float32)
    xq = rng.integers(-127, 128, size=cols, dtype=np.int8)
    xd = rng.uniform(1e-3, 1e-1, size=2).astype(np.float32)
    full = O.matvec(Q4_0, wq, wd, rows, cols, xq, xd)
    y = np.full(rows, np.nan, dtype=np.float32)
    O.matvec(Q4_0, wq, wd, rows, cols, xq, xd, r0=3, r1=7, y=y)
    assert np.all(np.isnan(y[:3])) and np.all(np.isnan(y[7:]))
    assert np.array_equal(y[3:7], full[3:7])
    y2 = np.full(rows, 5.0, dtype=np.float32)
    O.matvec(Q4_0, wq, wd, rows, cols, xq, xd, r0=4, r1=4, y=y2)
    assert np.all(y2 == 5.0)


def pin_small_m_rows_independent(O, seed=5):
    """Each of the M activation rows gives exactly the M = 1 product with its
    own scales; output row m starts at Y + m*ldy."""
    rng = np.random.default_rng(seed)
    rows, cols, M, ldy = 9, 96, 4, 12
    nb = cols // QK
    wq = rng.integers(0, 256, size=(rows, cols // 2), dtype=np.uint8)
    wd = rng.uniform(1e-3, 1e-2, size=(rows, nb)).astype(np.float32)
    Xq = rng.integers(-127, 128, size=(M, cols), dtype=np.int8)
    Xd = rng.uniform(1e-3, 1e-1, size=(M, nb)).astype(np.float32)
    Y = np.full((M, ldy), -1.0, dtype=np.float32)
    O.gemm_small_m(Q4_0, wq, wd, rows, cols, Xq, Xd, M, r0=2, r1=9, ldy=ldy, Y=Y)
    for m in range(M):
        y = O.matvec(Q4_0, wq, wd, rows, cols, Xq[m], Xd[m])
        assert np.array_equal(Y[m, 2:9], y[2:9])
        assert np.all(Y[m, :2] == -1.0) and np.all(Y[m, 9:] == -1.0)
        # and brute force of one entry, integer part exact
        we = decode_q4_elements(wq, cols)
        s = [int(np.dot(we[5, b * QK:(b + 1) * QK], Xq[m, b * QK:(b + 1) * QK].astype(np.int64)))
             for b in range(nb)]
        ex = sum(s[b] * float(wd[5, b]) * float(Xd[m, b]) for b in range(nb))
        tol = (nb + 2) * U * 1.01 * sum(abs(s[b] * float(wd[5, b]) * float(Xd[m, b])) for b in range(nb))
        assert abs(float(Y[m, 5]) - ex) <= tol + 1e-300


# ----------------------------------------------------------------------------
# the floating-point steps of a decode layer (Design Spec Sec. 5 and Sec. 6)
# ----------------------------------------------------------------------------
def pin_rmsnorm_closed_form(O):
    """x = (3, 4, 0, 0): the mean square is 25/4; with eps = 11/4 the root is
    exactly 3, so o = w * x / 3 exactly.  Leaving out the mean, putting eps
    outside the root or dropping w all break it."""
    x = np.array([3, 4, 0, 0], np.float32)
    w = np.array([3, 3, 1, 1], np.float32)
    o = O.rmsnorm(x, w, 2.75)
    assert np.array_equal(o, np.array([3, 4, 0, 0], np.float32)), o
    # degree-0 homogeneity without eps: rmsnorm(c x) = rmsnorm(x)
    rng = np.random.default_rng(21)
    x = rng.standard_normal(96).astype(np.float32)
    w = rng.uniform(0.5, 2, 96).astype(np.float32)
    a, b = O.rmsnorm(x, w, 0.0), O.rmsnorm(np.float32(8) * x, w, 0.0)
    assert np.allclose(a, b, rtol=4 * U, atol=0)
    # the root mean square of the normalised vector with unit weights is 1
    o = O.rmsnorm(x, np.ones(96, np.float32), 0.0).astype(np.float64)
    assert abs(np.sqrt(np.mean(o * o)) - 1.0) < 1e-6


def pin_softmax_values(O):
    """exp of (0, ln 2, ln 3) is (1, 2, 3): the result is (1/6, 1/3, 1/2);
    adding 1000 to every input changes nothing (no overflow either)."""
    v = np.array([0.0, np.log(2.0), np.log(3.0)], np.float32)
    y = O.softmax(v).astype(np.float64)
    assert np.allclose(y, [1 / 6, 1 / 3, 1 / 2], rtol=1e-6, atol=0), y
    y2 = O.softmax(v + np.float32(1000)).astype(np.float64)
    assert np.all(np.isfinite(y2)) and np.allclose(y2, [1 / 6, 1 / 3, 1 / 2], rtol=1e-4, atol=0)
    rng = np.random.default_rng(22)
    z = O.softmax(rng.standard_normal(257).astype(np.float32) * 5).astype(np.float64)
    assert abs(z.sum() - 1.0) < 1e-5 and np.all(z > 0)


def pin_silu_mul_values(O):
    """silu(x) = x sigma(x): silu(0) = 0, silu(ln 3) = (3/4) ln 3, and
    silu(x) - silu(-x) = x for every x (sigma(x) + sigma(-x) = 1)."""
    g = np.array([0.0, np.log(3.0)], np.float32)
    y = O.silu_mul(g, np.array([5.0, 2.0], np.float32)).astype(np.float64)
    assert y[0] == 0.0 and abs(y[1] - 2 * 0.75 * float(np.float32(np.log(3.0)))) < 1e-6
    rng = np.random.default_rng(23)
    x = rng.uniform(-6, 6, 200).astype(np.float32)
    one = np.ones(200, np.float32)
    d = O.silu_mul(x, one).astype(np.float64) - O.silu_mul(-x, one).astype(np.float64)
    assert np.allclose(d, x.astype(np.float64), rtol=0, atol=2e-6)


def pin_add_exact(O):
    """y += x is one rounded float32 addition per element."""
    rng = np.random.default_rng(24)
    y = rng.standard_normal(100).astype(np.float32)
    x = rng.standard_normal(100).astype(np.float32)
    assert np.array_equal(O.add(y, x), (y + x).astype(np.float32))


def pin_rope_tables_and_pairs(O):
    """Tables: position 0 is the identity; with head_dim 4 and theta 100 the
    second pair turns at 100^(-1/2) = 0.1 per position.  Rotation: the pairs
    are (2i, 2i+1), each turned by +angle; a q head (1, 0, 0, 1) at position
    1 becomes (cos 1, sin 1, -sin 0.1, cos 0.1)."""
    import math
    c, s = O.rope_tables(4, 4, 100.0)
    assert np.array_equal(c[0], [1, 1]) and np.array_equal(s[0], [0, 0])
    assert abs(float(c[3, 1]) - math.cos(0.3)) < 1e-7 and abs(float(s[3, 1]) - math.sin(0.3)) < 1e-7
    assert abs(float(c[2, 0]) - math.cos(2.0)) < 1e-7
    q = np.array([1, 0, 0, 1, 0.5, -2, 3, 1], np.float32)  # two q heads
    k = np.array([0, 1, 1, 0], np.float32)                   # one k head
    q2, k2 = O.rope(q, k, c[1], s[1], 4, 2, 1)
    want = [math.cos(1), math.sin(1), -math.sin(0.1), math.cos(0.1)]
    assert np.allclose(q2[:4], want, atol=1e-7), q2
    assert np.allclose(k2, [-math.sin(1), math.cos(1), math.cos(0.1), math.sin(0.1)], atol=1e-7), k2
    # each pair keeps its length
    n0 = np.hypot(q[4::2], q[5::2])
    n1 = np.hypot(q2[4::2], q2[5::2])
    assert np.allclose(n0, n1, rtol=1e-6)


def pin_attention_cases(O):
    """One position: o = V_0.  Zero query: uniform weights, o = mean of V.
    Scale: with q . K_0 = 2 and head_dim 4 the score is 2 / 2 = 1, so two
    positions with V = (1, 0) give e / (1 + e).  GQA: with 4 query heads and
    2 KV heads, heads 0, 1 read KV head 0 and heads 2, 3 read KV head 1."""
    import math
    hd, nh, nkv = 4, 4, 2
    rng = np.random.default_rng(25)
    q = rng.standard_normal(nh * hd).astype(np.float32)
    kc = rng.standard_normal((3, nkv * hd)).astype(np.float32)
    vc = rng.standard_normal((3, nkv * hd)).astype(np.float32)
    o = O.attention(q, kc, vc, 1, hd, nh, nkv)
    for h in range(nh):
        g = h // (nh // nkv)
        assert np.array_equal(o[h * hd:(h + 1) * hd], vc[0, g * hd:(g + 1) * hd])
    o = O.attention(np.zeros(nh * hd, np.float32), kc, vc, 3, hd, nh, nkv)
    for h in range(nh):
        g = h // (nh // nkv)
        assert np.allclose(o[h * hd:(h + 1) * hd], vc[:, g * hd:(g + 1) * hd].astype(np.float64).mean(0),
                           rtol=1e-6, atol=1e-7)
    q1 = np.zeros(hd, np.float32); q1[0] = 1
    k2 = np.zeros((2, hd), np.float32); k2[0, 0] = 2
    v2 = np.zeros((2, hd), np.float32); v2[0, :] = 1
    o = O.attention(q1, k2, v2, 2, hd, 1, 1)
    assert np.allclose(o, math.e / (1 + math.e), rtol=1e-6), o
    # distinct constant V per KV head: the mapping shows in every output
    vconst = np.repeat(np.array([[10.0, 20.0]], np.float32), 4, axis=1).reshape(1, -1)
    vconst = np.repeat(vconst, 3, axis=0)
    o = O.attention(q, kc, vconst, 3, hd, nh, nkv)
    assert np.allclose(o.reshape(nh, hd)[:, 0], [10, 10, 20, 20], rtol=1e-6), o


# ----------------------------------------------------------------------------
# Q4_K-style super-blocks (page "SKaiNET-native-kernels", section "Proving an
# optimization is safe before writing it"; the layout reading is the one
# stated in the oracle: q nibbles in the Q4_0 order per 32-element sub-block,
# s = per super-block 8 scales then 8 minima, d and dmin float32 per
# super-block; value = d * s_b * n - dmin * m_b; activations per 256 with
# the Q8_0 rounding rule and int32 sums per 32)
# ----------------------------------------------------------------------------
QKK = 256


def decode_q4k_nibbles(wq: np.ndarray, cols: int) -> np.ndarray:
    """Unsigned nibbles n in [0, 15] of every element, [rows, cols] int64."""
    rows = wq.shape[0]
    qb = wq.reshape(rows, cols // QK, 16).astype(np.int64)
    out = np.empty((rows, cols), dtype=np.int64)
    for e in range(QK):
        out[:, e::QK] = (qb[:, :, e] & 0xF) if e < 16 else (qb[:, :, e - 16] >> 4)
    return out


def q4k_sub_params(ws: np.ndarray, cols: int):
    """Per-sub-block scale s_b and minimum m_b, each [rows, cols/32] int64."""
    rows = ws.shape[0]
    sm = ws.reshape(rows, cols // QKK, 16).astype(np.int64)
    return sm[:, :, :8].reshape(rows, -1), sm[:, :, 8:].reshape(rows, -1)


def random_q4k(rng, rows, cols, smax=63):
    nsb = cols // QKK
    wq = rng.integers(0, 256, size=(rows, cols // 2), dtype=np.uint8)
    ws = rng.integers(0, smax + 1, size=(rows, nsb * 16), dtype=np.uint8)
    wd = rng.uniform(1e-4, 1e-3, size=(rows, nsb)).astype(np.float32)
    wdmin = rng.uniform(1e-4, 1e-3, size=(rows, nsb)).astype(np.float32)
    return wq, ws, wd, wdmin


def pin_q4k_overflow_bound(O):
    """The page's bound is attained and fits int32: all nibbles 15, all
    sub-block scales 63, every activation +127 (or -127) gives |ISUM| =
    8*63*32*127*15 = 30,723,840, about 70x below 2^31 - 1; MSUM with all
    minima 63 is 8*63*(32*127)."""
    cols = QKK
    wq = np.full((1, cols // 2), 0xFF, dtype=np.uint8)
    ws = np.full((1, 16), 63, dtype=np.uint8)
    for sign in (1, -1):
        xq = np.full(cols, 127 * sign, dtype=np.int8)
        xbs = np.full(cols // QK, 32 * 127 * sign, dtype=np.int32)
        isum, msum = O.block_sums_q4k(wq, ws, 1, cols, xq, xbs)
        assert int(isum[0, 0]) == sign * 8 * 63 * 32 * 127 * 15 == sign * 30723840, isum
        assert int(msum[0, 0]) == sign * 8 * 63 * 32 * 127, msum
    assert 30723840 * 69 < 2 ** 31 - 1 < 30723840 * 70


def pin_q4k_bruteforce_fp64(O, seed=21):
    """Integer sums exactly, and y within the float32 rounding bound, against
    fp64 brute force over the dequantised elements (d*s_b*n - dmin*m_b) *
    (dx*q) on tiny matrices."""
    rng = np.random.default_rng(seed)
    for trial in range(12):
        rows = int(rng.integers(1, 6))
        cols = QKK * int(rng.integers(1, 4))
        nsb = cols // QKK
        wq, ws, wd, wdmin = random_q4k(rng, rows, cols)
        x = rng.standard_normal(cols).astype(np.float32)
        xq, xd, xbs = O.quantize_q8k(x)
        y = O.matvec_q4k(wq, ws, wd, wdmin, rows, cols, xq, xd, xbs)
        isum, msum = O.block_sums_q4k(wq, ws, rows, cols, xq, xbs)
        n = decode_q4k_nibbles(wq, cols)
        s_b, m_b = q4k_sub_params(ws, cols)
        qx = xq.astype(np.int64)
        for r in range(rows):
            exact, absterms = 0.0, 0.0
            for B in range(nsb):
                I = M = 0
                acc = 0.0
                for sb in range(B * 8, B * 8 + 8):
                    e = slice(sb * QK, sb * QK + QK)
                    I += int(s_b[r, sb]) * int(np.dot(n[r, e], qx[e]))
                    M += int(m_b[r, sb]) * int(qx[e].sum())
                    for k in range(sb * QK, sb * QK + QK):
                        w = float(wd[r, B]) * float(s_b[r, sb]) * float(n[r, k]) - \
                            float(wdmin[r, B]) * float(m_b[r, sb])
                        acc += w * (float(xd[B]) * float(qx[k]))
                assert int(isum[r, B]) == I and int(msum[r, B]) == M, (trial, r, B)
                exact += acc
                absterms += (abs(I * float(wd[r, B])) + abs(M * float(wdmin[r, B]))) * float(xd[B])
            tol = (nsb + 5) * U * (1 + 1e-6) * absterms + 1e-300
            assert abs(float(y[r]) - exact) <= tol, (trial, r, float(y[r]), exact, tol)


def pin_q4k_special_cases(O, seed=22):
    """d = dx = 1, dmin = 0 and unit scales reduce the product to a plain
    integer matvec of the unsigned nibbles; d = 0, dmin = 1 leaves minus
    the minima-weighted sums of the activation quants."""
    rng = np.random.default_rng(seed)
    rows, cols = 5, 2 * QKK
    nsb = cols // QKK
    wq = rng.integers(0, 256, size=(rows, cols // 2), dtype=np.uint8)
    ws = np.zeros((rows, nsb * 16), dtype=np.uint8)
    ws.reshape(rows, nsb, 16)[:, :, :8] = 1
    ws.reshape(rows, nsb, 16)[:, :, 8:] = rng.integers(0, 64, size=(rows, nsb, 8))
    xq = rng.integers(-127, 128, size=cols, dtype=np.int8)
    xbs = xq.astype(np.int64).reshape(-1, QK).sum(axis=1).astype(np.int32)
    ones = np.ones((rows, nsb), np.float32)
    zeros = np.zeros((rows, nsb), np.float32)
    y = O.matvec_q4k(wq, ws, ones, zeros, rows, cols, xq, np.ones(nsb, np.float32), xbs)
    ref = decode_q4k_nibbles(wq, cols) @ xq.astype(np.int64)
    assert np.array_equal(y.astype(np.int64), ref) and np.all(np.abs(ref) < 2 ** 24), (y, ref)
    y = O.matvec_q4k(wq, ws, zeros, ones, rows, cols, xq, np.ones(nsb, np.float32), xbs)
    _, m_b = q4k_sub_params(ws, cols)
    ref = -(m_b * xbs.astype(np.int64)[None, :]).sum(axis=1)
    assert np.array_equal(y.astype(np.int64), ref), (y, ref)


def pin_q8k_quantizer(O, seed=23):
    """Per-256 quantisation with the Q8_0 rule: where every 32-element
    sub-block holds the 256-block's largest magnitude, the quants and scale
    equal those of the (separately pinned) Q8_0 quantiser; the sub-block
    sums are the integer sums of the quants; an all-zero block gives d = 0."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((3, 2 * QKK)).astype(np.float32)
    for r in range(3):
        for B in range(2):
            blk = x[r, B * QKK:(B + 1) * QKK]
            amax = np.float32(np.abs(blk).max() * 1.5)
            for sb in range(8):
                blk[sb * QK + int(rng.integers(0, QK))] = amax if rng.random() < 0.5 else -amax
    x[2, QKK:] = 0.0
    q, d, bs = O.quantize_q8k(x)
    q0, d0 = O.quantize_q8(x)
    assert np.array_equal(q, q0)
    assert np.array_equal(np.repeat(d, 8, axis=1).view(np.uint32), d0.view(np.uint32))
    assert np.array_equal(bs, q.astype(np.int64).reshape(3, -1, QK).sum(axis=2))
    assert d[2, 1] == 0 and not np.any(q[2, QKK:])
    # generic blocks: one scale per 256, d = max|x| / 127, and every element
    # within d/2 of q*d (the dequantisation bound, plus float32 rounding)
    x = (rng.standard_normal((4, 4 * QKK)) * 10.0 ** rng.uniform(-3, 3, (4, 1))).astype(np.float32)
    q, d, _ = O.quantize_q8k(x)
    blocks = x.reshape(4, -1, QKK)
    amax = np.abs(blocks).max(axis=2)
    assert np.array_equal(d.view(np.uint32), (amax / np.float32(127)).astype(np.float32).view(np.uint32))
    err = np.abs(blocks.astype(np.float64) - q.reshape(4, -1, QKK) * d.astype(np.float64)[:, :, None])
    assert np.all(err <= d.astype(np.float64)[:, :, None] * (0.5 + 127 * 3 * U + 2.0 ** -18))


def pin_q4k_row_range(O, seed=24):
    """Only rows [r0, r1) are written."""
    rng = np.random.default_rng(seed)
    rows, cols = 6, QKK
    wq, ws, wd, wdmin = random_q4k(rng, rows, cols)
    xq, xd, xbs = O.quantize_q8k(rng.standard_normal(cols).astype(np.float32))
    full = O.matvec_q4k(wq, ws, wd, wdmin, rows, cols, xq, xd, xbs)
    y = np.full(rows, 7.0, np.float32)
    O.matvec_q4k(wq, ws, wd, wdmin, rows, cols, xq, xd, xbs, r0=2, r1=5, y=y)
    assert np.array_equal(y[2:5], full[2:5]) and np.all(y[[0, 1, 5]] == 7.0)


# ----------------------------------------------------------------------------
# block length 32 / 128, float32 / binary16 scales, 8-bit weights in the
# packed signed form B' = B - 128 with per-block zero points (page "ONNX
# Runtime", "How we got there", items 3-5)
# ----------------------------------------------------------------------------
def nbits_elements(wq, zp, rows, cols, bits, blk) -> np.ndarray:
    """Weight values w = n - 8 (4-bit: element j of a block in the low
    nibble of byte j, element j + blk/2 in its high nibble) or B' + 128 - zp
    (8-bit), [rows, cols] int64, written from the stated format."""
    nb = cols // blk
    if bits == 4:
        qb = wq.reshape(rows, nb, blk // 2).astype(np.int64)
        w = np.concatenate([qb & 0xF, qb >> 4], axis=2) - 8
        return w.reshape(rows, cols)
    bp = wq.view(np.int8).reshape(rows, nb, blk).astype(np.int64)
    z = np.full((rows, nb), 128, np.int64) if zp is None else zp.reshape(rows, nb).astype(np.int64)
    return (bp + 128 - z[:, :, None]).reshape(rows, cols)


def random_nbits(rng, rows, cols, bits, blk, f16, with_zp):
    nb = cols // blk
    if bits == 4:
        wq = rng.integers(0, 256, size=(rows, cols // 2), dtype=np.uint8)
    else:
        wq = rng.integers(-128, 128, size=(rows, cols), dtype=np.int8)
    sc = rng.uniform(1e-4, 1e-2, size=(rows, nb)).astype(np.float16 if f16 else np.float32)
    zp = rng.integers(0, 256, size=(rows, nb), dtype=np.uint8) if (bits == 8 and with_zp) else None
    return wq, sc, zp


def pin_half_to_float_all_patterns(O):
    """The binary16 decoder against numpy's float16 on every bit pattern."""
    pats = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = pats.view(np.float16).astype(np.float32)
    got = np.array([O.half_to_float(int(p)) for p in range(0, 1 << 16, 1)], dtype=np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def pin_nbits_reduces_to_q4_0_and_q8_0(O, seed=31):
    """Block length 32 with float32 scales: the 4-bit product is the Q4_0
    product (same nibble order), the 8-bit product with every zero point
    128 (or none) is the Q8_0 product of B' (both pinned above)."""
    rng = np.random.default_rng(seed)
    rows, cols = 6, 128
    xq = rng.integers(-127, 128, size=cols, dtype=np.int8)
    xd = rng.uniform(1e-3, 1e-1, size=cols // QK).astype(np.float32)
    wq4 = rng.integers(0, 256, size=(rows, cols // 2), dtype=np.uint8)
    sc = rng.uniform(1e-3, 1e-2, size=(rows, cols // QK)).astype(np.float32)
    assert np.array_equal(O.matvec_nbits(wq4, sc, None, rows, cols, 4, 32, xq, xd).view(np.uint32),
                          O.matvec(Q4_0, wq4, sc, rows, cols, xq, xd).view(np.uint32))
    wq8 = rng.integers(-128, 128, size=(rows, cols), dtype=np.int8)
    wq8[wq8 == -128] = -127    # the Q8_0 range
    ref = O.matvec(Q8_0, wq8, sc, rows, cols, xq, xd)
    for zp in (None, np.full((rows, cols // 32), 128, np.uint8)):
        y = O.matvec_nbits(wq8, sc, zp, rows, cols, 8, 32, xq, xd)
        assert np.array_equal(y.view(np.uint32), ref.view(np.uint32))


def pin_nbits_bruteforce_fp64(O, seed=32):
    """Every combination of bits, block length, scale type and zero points:
    block sums exact against int64 sums of the decoded elements, y within the
    float32 summation bound of fp64 brute force over dequantised elements."""
    rng = np.random.default_rng(seed)
    for bits in (4, 8):
        for blk in (32, 128):
            for f16 in (False, True):
                for with_zp in ((False, True) if bits == 8 else (False,)):
                    rows, cols = int(rng.integers(1, 5)), blk * int(rng.integers(1, 4))
                    nb = cols // blk
                    wq, sc, zp = random_nbits(rng, rows, cols, bits, blk, f16, with_zp)
                    x = rng.standard_normal(cols).astype(np.float32)
                    xq, xd, xbs = O.quantize_blk(x, blk)
                    y = O.matvec_nbits(wq, sc, zp, rows, cols, bits, blk, xq, xd)
                    sumi = O.block_sumi_nbits(wq, zp, rows, cols, bits, blk, xq)
                    w = nbits_elements(wq, zp, rows, cols, bits, blk)
                    s32 = sc.astype(np.float64)
                    for r in range(rows):
                        exact, absterms = 0.0, 0.0
                        for b in range(nb):
                            e = slice(b * blk, (b + 1) * blk)
                            s = int(np.dot(w[r, e], xq[e].astype(np.int64)))
                            assert int(sumi[r, b]) == s, (bits, blk, f16, with_zp, r, b)
                            exact += float(np.sum((w[r, e] * s32[r, b]) * (xq[e].astype(np.float64) * float(xd[b]))))
                            absterms += abs(s * s32[r, b] * float(xd[b]))
                        tol = (nb + 2) * U * (1 + 1e-6) * absterms + 1e-300
                        assert abs(float(y[r]) - exact) <= tol, (bits, blk, f16, r, float(y[r]), exact)


def pin_nbits_signed_offset_and_bound(O, seed=33):
    """8-bit: the signed packing B' = B - 128 with zero point zp gives the
    weight B - zp (checked on B = 0, 128, 255 against zp = 0, 128, 255);
    the largest |sumi| a 128-block can reach, 255*127*128 = 4,145,280, is
    attained exactly and fits int32; the block-128 quantiser matches the
    Q8_0 one where each 32-element part holds the block's largest value."""
    cols, blk = 128, 128
    for B in (0, 128, 255):
        for z in (0, 128, 255):
            wq = np.full((1, cols), B - 128, np.int8)
            xq = np.ones(cols, np.int8)
            s = O.block_sumi_nbits(wq, np.array([[z]], np.uint8), 1, cols, 8, blk, xq)
            assert int(s[0, 0]) == (B - z) * cols, (B, z, s)
    wq = np.full((1, cols), 127, np.int8)          # B = 255
    s = O.block_sumi_nbits(wq, np.array([[0]], np.uint8), 1, cols, 8, blk, np.full(cols, 127, np.int8))
    assert int(s[0, 0]) == 255 * 127 * 128 == 4145280 < 2 ** 31
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(4 * blk).astype(np.float32)
    for b in range(4):
        amax = np.float32(np.abs(x[b * blk:(b + 1) * blk]).max() * 1.25)
        for part in range(4):
            x[b * blk + part * 32 + int(rng.integers(0, 32))] = amax
    q, d, bs = O.quantize_blk(x, blk)
    q0, d0 = O.quantize_q8(x)
    assert np.array_equal(q, q0) and np.array_equal(np.repeat(d, 4).view(np.uint32), d0.view(np.uint32))
    assert np.array_equal(bs, q.astype(np.int64).reshape(4, blk).sum(axis=1))
    xg = (rng.standard_normal(8 * blk) * 10.0 ** rng.uniform(-3, 3)).astype(np.float32)
    q, d, _ = O.quantize_blk(xg, blk)
    amax = np.abs(xg.reshape(-1, blk)).max(axis=1)
    assert np.array_equal(d.view(np.uint32), (amax / np.float32(127)).astype(np.float32).view(np.uint32))
    err = np.abs(xg.reshape(-1, blk).astype(np.float64) - q.reshape(-1, blk) * d.astype(np.float64)[:, None])
    assert np.all(err <= d.astype(np.float64)[:, None] * (0.5 + 127 * 3 * U + 2.0 ** -18))


ALL_PINS = [
    pin_rmsnorm_closed_form,
    pin_softmax_values,
    pin_silu_mul_values,
    pin_add_exact,
    pin_rope_tables_and_pairs,
    pin_attention_cases,
    pin_golden_quantize,
    pin_golden_block_dot,
    pin_quantize_invariants,
    pin_bruteforce_fp64,
    pin_unit_scales_integer_matvec,
    pin_row_range,
    pin_small_m_rows_independent,
    pin_q4k_overflow_bound,
    pin_q4k_bruteforce_fp64,
    pin_q4k_special_cases,
    pin_q8k_quantizer,
    pin_q4k_row_range,
    pin_half_to_float_all_patterns,
    pin_nbits_reduces_to_q4_0_and_q8_0,
    pin_nbits_bruteforce_fp64,
    pin_nbits_signed_offset_and_bound,
]
