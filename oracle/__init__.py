"""CPU oracle for the block-quantized decode matvec (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product library never does, and this
package imports nothing from the product.

The arithmetic lives in ``mlq_oracle.c`` (plain C11, compiled with
``-O2 -ffp-contract=off`` and no fast-math); this module only builds it with
gcc and marshals numpy arrays through ctypes.  Every definition it follows
is cited in the C file's header (page "Legacy-ISA ML Inference Runtime --
Design Spec", sections 4 and 5).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mlq_oracle.c")
_LIB = os.path.join(_HERE, "libmlq_oracle.so")

Q8_0 = 0
Q4_0 = 1
QK = 32
QKK = 256   # Q4_K-style super-block

_default = None


def build(force: bool = False) -> str:
    """Compile mlq_oracle.c into libmlq_oracle.so (in-tree) with gcc."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    compile_c(_SRC, _LIB)
    return _LIB


def compile_c(src: str, out: str) -> str:
    """gcc -O2 -ffp-contract=off (no fast-math) -shared; atomic replace of ``out``."""
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """ctypes view of one compiled oracle library (the real one, or a
    deliberately broken copy that a test builds to check that the pins
    catch it)."""

    def __init__(self, path: str):
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I = ctypes.c_int
        L.mlqo_quantize_q8.argtypes = [P, P, P, I, I]
        L.mlqo_block_sumi.argtypes = [P, I, P, I, I, P, I, I]
        L.mlqo_matvec.argtypes = [P, I, P, P, I, I, P, P, I, I]
        L.mlqo_gemm_small_m.argtypes = [P, I, I, P, P, I, I, P, P, I, I, I]
        F = ctypes.c_float
        L.mlqo_rmsnorm.argtypes = [P, P, P, I, F]
        L.mlqo_softmax.argtypes = [P, I]
        L.mlqo_silu_mul.argtypes = [P, P, I]
        L.mlqo_add.argtypes = [P, P, I]
        L.mlqo_rope_tables.argtypes = [P, P, I, I, F]
        L.mlqo_rope.argtypes = [P, P, P, P, I, I, I]
        L.mlqo_attention.argtypes = [P, P, P, P, I, I, I, I]
        L.mlqo_quantize_q8k.argtypes = [P, P, P, P, I, I]
        L.mlqo_block_sums_q4k.argtypes = [P, P, P, P, I, I, P, P, I, I]
        L.mlqo_matvec_q4k.argtypes = [P, P, P, P, P, I, I, P, P, P, I, I]
        L.mlqo_half_to_float.argtypes = [ctypes.c_uint16]
        L.mlqo_half_to_float.restype = ctypes.c_float
        L.mlqo_quantize_blk.argtypes = [P, P, P, P, I, I]
        L.mlqo_block_sumi_nbits.argtypes = [P, P, P, I, I, I, I, P, I, I]
        L.mlqo_matvec_nbits.argtypes = [P, P, P, I, P, I, I, I, I, P, P, I, I]
        for f in (L.mlqo_quantize_q8, L.mlqo_block_sumi, L.mlqo_matvec, L.mlqo_gemm_small_m,
                  L.mlqo_rmsnorm, L.mlqo_softmax, L.mlqo_silu_mul, L.mlqo_add, L.mlqo_rope_tables,
                  L.mlqo_rope, L.mlqo_attention, L.mlqo_quantize_q8k, L.mlqo_block_sums_q4k,
                  L.mlqo_matvec_q4k, L.mlqo_quantize_blk, L.mlqo_block_sumi_nbits,
                  L.mlqo_matvec_nbits):
            f.restype = ctypes.c_int
        self.lib = L
        self.path = path

    def quantize_q8(self, x: np.ndarray):
        """Q8_0-quantise x (float32, shape [k] or [m, k]) -> (q int8, d float32)."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        squeeze = x.ndim == 1
        x2 = x.reshape(1, -1) if squeeze else x
        m, k = x2.shape
        q = np.empty((m, k), dtype=np.int8)
        d = np.empty((m, k // QK), dtype=np.float32)
        rc = self.lib.mlqo_quantize_q8(_ptr(q), _ptr(d), _ptr(x2), m, k)
        if rc != 0:
            raise ValueError("oracle quantize_q8: k must be a multiple of 32")
        return (q[0], d[0]) if squeeze else (q, d)

    def block_sumi(self, wtype: int, wq: np.ndarray, rows: int, cols: int, xq: np.ndarray,
                   r0: int = 0, r1: int | None = None) -> np.ndarray:
        """Per-block int32 sums for rows [r0, r1) -> int32 [r1 - r0, cols/32]."""
        r1 = rows if r1 is None else r1
        nb = cols // QK
        out = np.zeros((max(r1 - r0, 0), nb), dtype=np.int32)
        rc = self.lib.mlqo_block_sumi(_ptr(out), wtype, _ptr(np.ascontiguousarray(wq)), rows, cols,
                                      _ptr(np.ascontiguousarray(xq, dtype=np.int8)), r0, r1)
        if rc != 0:
            raise ValueError("oracle block_sumi: bad arguments")
        return out

    def matvec(self, wtype: int, wq: np.ndarray, wd: np.ndarray, rows: int, cols: int,
               xq: np.ndarray, xd: np.ndarray, r0: int = 0, r1: int | None = None,
               y: np.ndarray | None = None) -> np.ndarray:
        """y[r] for r in [r0, r1); other entries of y are left as they are."""
        r1 = rows if r1 is None else r1
        if y is None:
            y = np.zeros(rows, dtype=np.float32)
        rc = self.lib.mlqo_matvec(_ptr(y), wtype, _ptr(np.ascontiguousarray(wq)),
                                  _ptr(np.ascontiguousarray(wd, dtype=np.float32)), rows, cols,
                                  _ptr(np.ascontiguousarray(xq, dtype=np.int8)),
                                  _ptr(np.ascontiguousarray(xd, dtype=np.float32)), r0, r1)
        if rc != 0:
            raise ValueError("oracle matvec: bad arguments")
        return y

    def gemm_small_m(self, wtype: int, wq: np.ndarray, wd: np.ndarray, rows: int, cols: int,
                     Xq: np.ndarray, Xd: np.ndarray, M: int, r0: int = 0, r1: int | None = None,
                     ldy: int | None = None, Y: np.ndarray | None = None) -> np.ndarray:
        """Y[m, r] for m < M and r in [r0, r1); Y is [M, ldy] float32."""
        r1 = rows if r1 is None else r1
        ldy = rows if ldy is None else ldy
        if Y is None:
            Y = np.zeros((M, ldy), dtype=np.float32)
        rc = self.lib.mlqo_gemm_small_m(_ptr(Y), ldy, wtype, _ptr(np.ascontiguousarray(wq)),
                                        _ptr(np.ascontiguousarray(wd, dtype=np.float32)), rows, cols,
                                        _ptr(np.ascontiguousarray(Xq, dtype=np.int8)),
                                        _ptr(np.ascontiguousarray(Xd, dtype=np.float32)), M, r0, r1)
        if rc != 0:
            raise ValueError("oracle gemm_small_m: bad arguments")
        return Y


class _Q4KOps:
    """Q4_K-style super-blocks (page "SKaiNET-native-kernels", "Proving an
    optimization is safe before writing it"); the layout is the one stated
    in mlq_oracle.c."""

    def quantize_q8k(self, x: np.ndarray):
        """x float32 [k] or [m, k] -> (q int8, d float32 per 256, bsums int32 per 32)."""
        x = np.ascontiguousarray(x, dtype=np.float32)
        squeeze = x.ndim == 1
        x2 = x.reshape(1, -1) if squeeze else x
        m, k = x2.shape
        q = np.empty((m, k), dtype=np.int8)
        d = np.empty((m, k // QKK), dtype=np.float32)
        bs = np.empty((m, k // QK), dtype=np.int32)
        _ok(self.lib.mlqo_quantize_q8k(_ptr(q), _ptr(d), _ptr(bs), _ptr(x2), m, k), "quantize_q8k")
        return (q[0], d[0], bs[0]) if squeeze else (q, d, bs)

    def block_sums_q4k(self, wq, ws, rows: int, cols: int, xq, xbs, r0: int = 0,
                       r1: int | None = None):
        """(ISUM, MSUM) int32 [r1 - r0, cols/256] for rows [r0, r1)."""
        r1 = rows if r1 is None else r1
        nsb = cols // QKK
        isum = np.zeros((max(r1 - r0, 0), nsb), dtype=np.int32)
        msum = np.zeros_like(isum)
        _ok(self.lib.mlqo_block_sums_q4k(_ptr(isum), _ptr(msum), _ptr(_u8(wq)), _ptr(_u8(ws)), rows,
                                         cols, _ptr(_i8(xq)), _ptr(_i32(xbs)), r0, r1),
            "block_sums_q4k")
        return isum, msum

    def matvec_q4k(self, wq, ws, wd, wdmin, rows: int, cols: int, xq, xd, xbs, r0: int = 0,
                   r1: int | None = None, y: np.ndarray | None = None) -> np.ndarray:
        """y[r] for r in [r0, r1); other entries of y are left as they are."""
        r1 = rows if r1 is None else r1
        if y is None:
            y = np.zeros(rows, dtype=np.float32)
        _ok(self.lib.mlqo_matvec_q4k(_ptr(y), _ptr(_u8(wq)), _ptr(_u8(ws)), _ptr(_f32(wd)),
                                     _ptr(_f32(wdmin)), rows, cols, _ptr(_i8(xq)), _ptr(_f32(xd)),
                                     _ptr(_i32(xbs)), r0, r1), "matvec_q4k")
        return y


class _NBitsOps:
    """Block length 32 / 128, float32 / binary16 scales, 8-bit weights in
    the packed signed form with per-block zero points (page "ONNX Runtime",
    "How we got there", items 3-5); the layout is the one stated in
    mlq_oracle.c."""

    def half_to_float(self, bits: int) -> float:
        return float(self.lib.mlqo_half_to_float(int(bits) & 0xFFFF))

    def quantize_blk(self, x: np.ndarray, blk: int):
        """x float32 [k] -> (q int8 [k], d float32 [k/blk], bsums int32 [k/blk])."""
        x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1)
        k = x.size
        q = np.empty(k, dtype=np.int8)
        d = np.empty(k // blk, dtype=np.float32)
        bs = np.empty(k // blk, dtype=np.int32)
        _ok(self.lib.mlqo_quantize_blk(_ptr(q), _ptr(d), _ptr(bs), _ptr(x), k, blk), "quantize_blk")
        return q, d, bs

    def block_sumi_nbits(self, wq, zp, rows: int, cols: int, bits: int, blk: int, xq, r0: int = 0,
                         r1: int | None = None) -> np.ndarray:
        r1 = rows if r1 is None else r1
        out = np.zeros((max(r1 - r0, 0), cols // blk), dtype=np.int32)
        zptr = None if zp is None else _ptr(_u8(zp))
        _ok(self.lib.mlqo_block_sumi_nbits(_ptr(out), _ptr(_u8(wq.view(np.uint8))), zptr, rows, cols,
                                           bits, blk, _ptr(_i8(xq)), r0, r1), "block_sumi_nbits")
        return out

    def matvec_nbits(self, wq, scales, zp, rows: int, cols: int, bits: int, blk: int, xq, xd,
                     r0: int = 0, r1: int | None = None, y: np.ndarray | None = None) -> np.ndarray:
        """scales: float32, or float16 (passed as their binary16 bit patterns)."""
        r1 = rows if r1 is None else r1
        if y is None:
            y = np.zeros(rows, dtype=np.float32)
        f16 = scales.dtype == np.float16
        sc = np.ascontiguousarray(scales.view(np.uint16) if f16 else _f32(scales))
        zptr = None if zp is None else _ptr(_u8(zp))
        _ok(self.lib.mlqo_matvec_nbits(_ptr(y), _ptr(_u8(wq.view(np.uint8))), _ptr(sc), 1 if f16 else 0,
                                       zptr, rows, cols, bits, blk, _ptr(_i8(xq)), _ptr(_f32(xd)),
                                       r0, r1), "matvec_nbits")
        return y


def _u8(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.uint8)


def _i8(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int8)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.int32)


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def _ok(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what}: bad arguments")


class _LayerOps:
    """The floating-point steps of a decode layer (Design Spec Sec. 5 and 6);
    each returns new float32 arrays and leaves its inputs unchanged."""

    def rmsnorm(self, x, w, eps: float) -> np.ndarray:
        x, w = _f32(x), _f32(w)
        o = np.empty_like(x)
        _ok(self.lib.mlqo_rmsnorm(_ptr(o), _ptr(x), _ptr(w), x.size, eps), "rmsnorm")
        return o

    def softmax(self, x) -> np.ndarray:
        y = _f32(x).copy()
        _ok(self.lib.mlqo_softmax(_ptr(y), y.size), "softmax")
        return y

    def silu_mul(self, g, u) -> np.ndarray:
        y, u = _f32(g).copy(), _f32(u)
        _ok(self.lib.mlqo_silu_mul(_ptr(y), _ptr(u), y.size), "silu_mul")
        return y

    def add(self, y, x) -> np.ndarray:
        out, x = _f32(y).copy(), _f32(x)
        _ok(self.lib.mlqo_add(_ptr(out), _ptr(x), out.size), "add")
        return out

    def rope_tables(self, max_seq: int, head_dim: int, theta: float):
        c = np.empty((max_seq, head_dim // 2), dtype=np.float32)
        s = np.empty_like(c)
        _ok(self.lib.mlqo_rope_tables(_ptr(c), _ptr(s), max_seq, head_dim, theta), "rope_tables")
        return c, s

    def rope(self, q, k, cos_row, sin_row, head_dim: int, n_heads: int, n_kv_heads: int):
        q2, k2 = _f32(q).copy(), _f32(k).copy()
        _ok(self.lib.mlqo_rope(_ptr(q2), _ptr(k2), _ptr(_f32(cos_row)), _ptr(_f32(sin_row)),
                               head_dim, n_heads, n_kv_heads), "rope")
        return q2, k2

    def attention(self, q, kc, vc, n_pos: int, head_dim: int, n_heads: int, n_kv_heads: int):
        o = np.empty(n_heads * head_dim, dtype=np.float32)
        _ok(self.lib.mlqo_attention(_ptr(o), _ptr(_f32(q)), _ptr(_f32(kc)), _ptr(_f32(vc)), n_pos,
                                    head_dim, n_heads, n_kv_heads), "attention")
        return o


for _name in ("rmsnorm", "softmax", "silu_mul", "add", "rope_tables", "rope", "attention"):
    setattr(Oracle, _name, getattr(_LayerOps, _name))
for _name in ("quantize_q8k", "block_sums_q4k", "matvec_q4k"):
    setattr(Oracle, _name, getattr(_Q4KOps, _name))
for _name in ("half_to_float", "quantize_blk", "block_sumi_nbits", "matvec_nbits"):
    setattr(Oracle, _name, getattr(_NBitsOps, _name))


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def quantize_q8(x):
    return default().quantize_q8(x)


def block_sumi(*a, **k):
    return default().block_sumi(*a, **k)


def matvec(*a, **k):
    return default().matvec(*a, **k)


def gemm_small_m(*a, **k):
    return default().gemm_small_m(*a, **k)


def rmsnorm(*a, **k):
    return default().rmsnorm(*a, **k)


def softmax(*a, **k):
    return default().softmax(*a, **k)


def silu_mul(*a, **k):
    return default().silu_mul(*a, **k)


def add(*a, **k):
    return default().add(*a, **k)


def rope_tables(*a, **k):
    return default().rope_tables(*a, **k)


def rope(*a, **k):
    return default().rope(*a, **k)


def attention(*a, **k):
    return default().attention(*a, **k)


def quantize_q8k(x):
    return default().quantize_q8k(x)


def block_sums_q4k(*a, **k):
    return default().block_sums_q4k(*a, **k)


def matvec_q4k(*a, **k):
    return default().matvec_q4k(*a, **k)


def quantize_blk(*a, **k):
    return default().quantize_blk(*a, **k)


def block_sumi_nbits(*a, **k):
    return default().block_sumi_nbits(*a, **k)


def matvec_nbits(*a, **k):
    return default().matvec_nbits(*a, **k)
