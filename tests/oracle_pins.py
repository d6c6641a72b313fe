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


ALL_PINS = [
    pin_golden_quantize,
    pin_golden_block_dot,
    pin_quantize_invariants,
    pin_bruteforce_fp64,
    pin_unit_scales_integer_matvec,
    pin_row_range,
    pin_small_m_rows_independent,
]
