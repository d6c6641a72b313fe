"""The host-side plan of mlq_decode_chain's streaming kernel, on the CPU
(no GPU; fake, aligned device addresses that are never dereferenced):
which phases read their input as Q8_0 from an earlier product, the
per-phase row split over the CTAs, the stage geometry and the shared
memory it needs.  Data flow: page "Legacy-ISA ML Inference Runtime --
Design Spec", Sec. 6 "Forward pass" (a product's output is the next
phase's quantised input)."""
import ctypes

import numpy as np
import pytest

WARPS = 12          # consumer warps of the streaming kernel
CHUNK = 64          # blocks of K a warp holds in registers at most
SMEM_MAX = 227 * 1024


@pytest.fixture(scope="module")
def M():
    from block_quantized_decode_gb300 import build as B
    B.build()
    import block_quantized_decode_gb300 as pkg
    pkg.lib()
    return pkg


class Addr:
    """Bump allocator of fake 256-byte aligned device addresses."""

    def __init__(self):
        self.next = 1 << 32

    def __call__(self, nbytes):
        a = self.next
        self.next += (nbytes + 255) // 256 * 256 + 256
        return a


def plan(M, mats, qtype, num_sms=152, with_xq=True):
    """mats: (rows, cols, input) with input "x" or the index of the product
    whose output it is; consecutive products with the same input form a
    phase.  Returns (info array, phases, products as dicts)."""
    from block_quantized_decode_gb300.binding import _ChainPhase, _ChainProduct, _QTensor
    A = Addr()
    prods, phases = [], []
    for j, (rows, cols, inp) in enumerate(mats):
        qbytes = rows * cols // (2 if qtype == 1 else 1)
        prods.append(dict(rows=rows, cols=cols, inp=inp, q=A(qbytes), d=A(rows * cols // 8), y=A(rows * 4)))
        key = ("x", cols) if inp == "x" else inp   # float inputs of different widths are different vectors
        if phases and phases[-1]["key"] == key:
            phases[-1]["count"] += 1
        else:
            phases.append(dict(inp=inp, key=key, first=j, count=1, n=cols))
    for ph in phases:
        ph["x"] = A(ph["n"] * 4) if ph["inp"] == "x" else prods[ph["inp"]]["y"]
        ph["xq"] = A(ph["n"]) if with_xq else 0
        ph["xd"] = A(ph["n"] // 8) if with_xq else 0
    cph = (_ChainPhase * len(phases))(*[
        _ChainPhase(p["x"], p["n"], p["first"], p["count"], p["xq"] or None, p["xd"] or None) for p in phases])
    cpr = (_ChainProduct * len(prods))(*[
        _ChainProduct(_QTensor(p["q"], p["d"], p["rows"], p["cols"], qtype), p["y"]) for p in prods])
    info = np.zeros(8 + 8 * len(phases) + len(phases) * (num_sms + 1), dtype=np.int32)
    st = M.binding.raw_call("mlq_debug_chain_plan", cph, len(phases), cpr, len(prods), num_sms,
                            info.ctypes.data_as(ctypes.c_void_p), info.size)
    assert st == M.MLQ_OK, M.mlq_status_str(st)
    return info, phases, prods


def check(info, phases, prods, qtype, num_sms=152):
    """Every invariant the kernel relies on; returns the number of hand-offs."""
    assert info[0] == 1
    grid, ring, smem = int(info[1]), int(info[2]), int(info[3])
    np_ = len(phases)
    assert 1 <= grid <= min(num_sms, 160)
    assert ring % 16 == 0 and smem <= SMEM_MAX - 1024 and ring < smem
    handoffs = 0
    cum = np.zeros(grid, dtype=np.float64)
    amax = 0.0
    for p, ph in enumerate(phases):
        C, cblk, G, RW, R, qin, any_out, outmask = (int(v) for v in info[4 + 8 * p: 12 + 8 * p])
        nb = ph["n"] // 32
        rowb = nb * (16 if qtype == 1 else 32) + nb * 4
        assert WARPS % C == 0 and C * G == WARPS and cblk == -(-nb // C) and cblk <= CHUNK
        assert RW in (1, 2, 4) and R == RW * G
        assert R * rowb <= ring // 2, "two stages must fit the ring"
        b = info[4 + 8 * np_ + p * (grid + 1): 4 + 8 * np_ + (p + 1) * (grid + 1)].astype(np.int64)
        total = sum(prods[j]["rows"] for j in range(ph["first"], ph["first"] + ph["count"]))
        assert b[0] == 0 and b[-1] == total and np.all(np.diff(b) >= 0)
        if any_out:
            assert np.all(b % 32 == 0), "rows quantised in-chain go to CTAs in whole 32-row blocks"
            assert all(prods[j]["rows"] % 32 == 0 for j in range(ph["first"], ph["first"] + ph["count"]))
        assert bool(any_out) == (outmask != 0)
        if qin:
            handoffs += 1
            src = [j for j, pr in enumerate(prods) if pr["y"] == ph["x"]]
            assert len(src) == 1 and prods[src[0]]["rows"] == ph["n"] and ph["xq"]
            q = [k for k, pq in enumerate(phases) if pq["first"] <= src[0] < pq["first"] + pq["count"]][0]
            assert q < p and (int(info[4 + 8 * q + 7]) >> (src[0] - phases[q]["first"])) & 1
        # the row split keeps each CTA's streamed bytes even: giving a phase's
        # extra atoms to the lightest CTAs keeps the spread of the bytes
        # streamed so far within the largest atom (in bytes) seen so far
        rows = np.diff(b)
        cum += rows * rowb
        amax = max(amax, (32 if any_out else 1) * rowb)
        assert cum.max() - cum.min() <= amax + 1e-6, (p, cum.max() - cum.min(), amax)
    return handoffs


def llama7b(qtype, layers=8):
    mats = []
    for l in range(layers):
        mats.append((11008, 4096, "x" if l == 0 else 2 * l - 1))
        mats.append((4096, 11008, 2 * l))
    return mats


def test_plan_llama7b_q4_stack(M):
    info, ph, pr = plan(M, llama7b(1), 1)
    assert check(info, ph, pr, 1) == 15          # every phase after the first reads Q8_0 in-chain
    assert int(info[1]) == 152


def test_plan_llama7b_q8_with_lm_head(M):
    mats = llama7b(0) + [(151936, 896, "x")]
    info, ph, pr = plan(M, mats, 0)
    assert check(info, ph, pr, 0) == 15
    lm = len(ph) - 1
    assert int(info[4 + 8 * lm + 5]) == 0          # the lm_head reads the float x


def test_plan_tinyllama_layer(M):
    d, kv, ff = 2048, 256, 5632
    mats = [(d, d, "x"), (kv, d, "x"), (kv, d, "x"), (d, d, 0), (ff, d, 3), (ff, d, 3), (d, ff, 4)]
    info, ph, pr = plan(M, mats, 1)
    assert check(info, ph, pr, 1) == 3
    assert int(info[4 + 7]) == 1                   # only Wq's output (bit 0) of the q|k|v phase is handed on


def test_plan_without_output_buffers_has_no_handoffs(M):
    info, ph, pr = plan(M, llama7b(1, layers=2), 1, with_xq=False)
    assert check(info, ph, pr, 1) == 0


def test_plan_partial_blocks_and_small_grids(M):
    """A phase with a product whose rows are not whole 32-row blocks hands
    nothing on (its reader quantises the floats); few CTAs; tiny shapes."""
    mats = [(512, 16384, "x"), (16384, 512, 0), (128, 16384, 1), (4096, 128, 2), (77, 128, 2),
            (64, 4096, 3)]
    for sms in (152, 7, 1):
        info, ph, pr = plan(M, mats, 1, num_sms=sms)
        assert check(info, ph, pr, 1, num_sms=sms) == 3
        assert int(info[4 + 8 * 4 + 5]) == 0       # the phase reading W4's output quantises it itself
    info, ph, pr = plan(M, [(1001, 128, "x"), (7, 128, "x"), (384, 1024, "x"), (1000, 384, 2)], 0)
    check(info, ph, pr, 0)


def test_plan_declines_rows_wider_than_its_warps(M):
    """K = 40960 needs more than 12 chunks of 64 blocks: the legacy kernel runs it."""
    info, _, _ = plan(M, [(300, 40960, "x")], 0)
    assert info[0] == 0
    info, ph, pr = plan(M, [(300, 20480, "x")], 0)      # 12 chunks of 54 blocks still fit
    check(info, ph, pr, 0)


def test_plan_hook_validation(M):
    from block_quantized_decode_gb300.binding import _ChainPhase, _ChainProduct, _QTensor
    cph = (_ChainPhase * 1)(_ChainPhase(1 << 32, 128, 0, 1, None, None))
    cpr = (_ChainProduct * 1)(_ChainProduct(_QTensor(1 << 33, 1 << 34, 64, 128, 1), 1 << 35))
    info = np.zeros(4, dtype=np.int32)
    call = lambda n, sms=152: M.binding.raw_call("mlq_debug_chain_plan", cph, 1, cpr, 1, sms,
                                                 info.ctypes.data_as(ctypes.c_void_p), n)
    assert call(4) == M.MLQ_E_SHAPE                  # too small for the plan
    assert call(64, sms=0) == M.MLQ_E_SHAPE
    big = np.zeros(4096, dtype=np.int32)
    assert M.binding.raw_call("mlq_debug_chain_plan", cph, 1, cpr, 1, 152,
                              big.ctypes.data_as(ctypes.c_void_p), big.size) == M.MLQ_OK
    assert big[0] == 1
