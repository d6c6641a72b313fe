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
        for f in (L.mlqo_quantize_q8, L.mlqo_block_sumi, L.mlqo_matvec, L.mlqo_gemm_small_m):
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
