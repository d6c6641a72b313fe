"""Helpers for the GPU-vs-oracle parity tests.

Bar (page "Legacy-ISA ML Inference Runtime -- Design Spec", Sec. 7): quant
bytes, scales and per-block int32 sums bit-exact; float32 outputs within
1e-5 * sum_b |(float)sumi * dw * dx| per row (the in-order float32 sum of
the oracle and the kernel's reordered sum may each differ from the exact
value by a few ulp of that magnitude).
"""
from __future__ import annotations

import numpy as np
import torch

import block_quantized_decode_gb300 as M
import oracle

DEV = torch.device("cuda:0")
REL = 1e-5


def to_dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def gpu_quantize(x: np.ndarray):
    x2 = np.ascontiguousarray(x.reshape(-1, x.shape[-1]), dtype=np.float32)
    m, k = x2.shape
    q = torch.empty((m, k), dtype=torch.int8, device=DEV)
    d = torch.empty((m, k // 32), dtype=torch.float32, device=DEV)
    M.mlq_quantize_q8(M.QAct(q, d, k, m), to_dev(x2), k)
    return q.cpu().numpy(), d.cpu().numpy()


def assert_quant_equal(gq, gd, oq, od, what=""):
    gq = gq.reshape(oq.shape)
    gd = gd.reshape(od.shape)
    bad = np.argwhere(gq != oq)
    assert bad.size == 0, f"{what}: {len(bad)} quant bytes differ, first at {bad[:3].tolist()}"
    badd = np.argwhere(gd.view(np.uint32) != od.view(np.uint32))
    assert badd.size == 0, f"{what}: {len(badd)} scales differ, first at {badd[:3].tolist()}"


def tol_rows(sumi: np.ndarray, wd_rows: np.ndarray, xd: np.ndarray) -> np.ndarray:
    terms = np.abs(sumi.astype(np.float64) * wd_rows.astype(np.float64)
                   * xd.astype(np.float64)[None, :])
    return REL * terms.sum(axis=1)


def assert_y_close(y_gpu, y_or, tol, what=""):
    err = np.abs(np.asarray(y_gpu, dtype=np.float64) - np.asarray(y_or, dtype=np.float64))
    ok = err <= tol
    if not np.all(ok):
        i = int(np.argmax(err - tol))
        raise AssertionError(f"{what}: {int((~ok).sum())} outputs outside tolerance; worst row {i}: "
                             f"gpu {float(np.asarray(y_gpu)[i])!r} oracle {float(np.asarray(y_or)[i])!r} "
                             f"tol {float(tol[i])!r}")


def weights_dev(wtype, wq, wd, rows, cols):
    return M.QTensor(to_dev(wq.reshape(-1)), to_dev(wd.reshape(-1)), rows, cols, wtype)


def check_matvec(wtype, wq, wd, rows, cols, xq, xd, r0, r1, windows=None, y_gpu=None, what=""):
    """Run (or take) the GPU product over [r0, r1) and compare either every
    row or the given row windows [(a, b), ...] against the oracle."""
    if y_gpu is None:
        W = weights_dev(wtype, wq, wd, rows, cols)
        x = M.QAct(to_dev(xq), to_dev(xd), cols, 1)
        y = torch.full((rows,), float("nan"), dtype=torch.float32, device=DEV)
        f = M.mlq_matvec_q4 if wtype == oracle.Q4_0 else M.mlq_matvec_q8
        f(y, W, x, r0, r1)
        y_gpu = y.cpu().numpy()
        assert np.all(np.isnan(y_gpu[:r0])) and np.all(np.isnan(y_gpu[r1:])), \
            f"{what}: rows outside [r0, r1) were written"
    windows = [(r0, r1)] if windows is None else windows
    nb = cols // 32
    for a, b in windows:
        if b <= a:
            continue
        yo = oracle.matvec(wtype, wq, wd, rows, cols, xq, xd, a, b)
        s = oracle.block_sumi(wtype, wq, rows, cols, xq, a, b)
        tol = tol_rows(s, wd.reshape(rows, nb)[a:b], xd)
        assert_y_close(y_gpu[a:b], yo[a:b], tol, f"{what} rows [{a},{b})")
    return y_gpu


def sample_windows(rows: int, rng, count=6, width=32):
    wins = [(0, min(width, rows)), (max(0, rows - width), rows)]
    for _ in range(count):
        a = int(rng.integers(0, max(1, rows - width)))
        wins.append((a, min(rows, a + width)))
    return wins
