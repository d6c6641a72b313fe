"""Device-resident workloads driven through the C ABI.

A ``WorkloadRunner`` owns the device buffers of one workload (weights,
activations, Q8_0 activation buffers, outputs) and issues one pass of the
hot path -- quantize each input once, then the Q4_0/Q8_0 products -- as C-ABI
calls on a stream.  torch supplies device memory, pinned host memory, streams
and CUDA graphs; every arithmetic step runs in libmlq's kernels.

Weights can be replicated ``copies`` times so that consecutive passes read
different bytes (inputs larger than L2 between timed passes).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from . import binding as B
from . import inputs as I


@dataclass
class _Mat:
    spec: I.Matvec
    src: str               # input buffer name
    q: list                # per copy: device quant bytes
    d: list                # per copy: device scales
    y: torch.Tensor        # output [m, rows] float32
    host_q: np.ndarray
    host_d: np.ndarray


# Guard bands (canary=True): every output buffer gets GUARD elements of a
# sentinel before and after it; check_canaries() asserts them unchanged, so a
# kernel that writes past the rows or blocks it owns is caught.
GUARD = 64
_SENTINEL_F32 = 0x7FA5A5A5   # a NaN bit pattern no kernel writes
_SENTINEL_I8 = -91           # 0xA5


class WorkloadRunner:
    def __init__(self, wl: I.Workload, copies: int = 1, device: str = "cuda:0",
                 seed_base: int = 0, x_seed_base: int = 1000, canary: bool = False):
        self.wl = wl
        self.canary = canary
        self.m = wl.m
        self.copies = copies
        self.dev = torch.device(device)
        self.mats: list[_Mat] = []
        self.sources: dict[str, int] = {}   # input name -> length K
        self.x_host: dict[str, np.ndarray] = {}
        self.x_pinned: dict[str, torch.Tensor] = {}
        self.fp32: dict[str, torch.Tensor] = {}   # float32 vectors feeding a quantize
        self.qbuf: dict[str, B.QAct] = {}
        # every product's output is a view of one buffer (128-byte aligned
        # offsets), so one copy brings all of them to the host
        g = GUARD if canary else 0
        self.y_offs, tot = [], 0
        for mv in wl.mats:
            tot += g
            self.y_offs.append(tot)
            tot += (self.m * mv.rows + 31) // 32 * 32
        tot += g
        self.y_all = torch.zeros(tot, dtype=torch.float32, device=self.dev)
        if canary:
            self.y_all.view(torch.int32).fill_(_SENTINEL_F32)
        for i, mv in enumerate(wl.mats):
            src = f"x{mv.cols}" if mv.input_of == "x" else mv.input_of
            if mv.input_of == "x" and src not in self.x_host:
                xs = I.activations(self.m, mv.cols, seed=x_seed_base + len(self.x_host))
                self.x_host[src] = xs
                self.x_pinned[src] = torch.from_numpy(xs).pin_memory()
                self.fp32[src] = torch.from_numpy(xs).to(self.dev)
            self.sources.setdefault(src, mv.cols)
            hq, hd = I.weights(mv.wtype, mv.rows, mv.cols, seed=seed_base + i)
            qs, ds = [], []
            for _ in range(copies):
                qs.append(torch.from_numpy(hq.reshape(-1)).to(self.dev))
                ds.append(torch.from_numpy(hd.reshape(-1)).to(self.dev))
            y = self.y_all[self.y_offs[i]: self.y_offs[i] + self.m * mv.rows].view(self.m, mv.rows)
            self.mats.append(_Mat(mv, src, qs, ds, y, hq, hd))
        for m in self.mats:
            self.fp32.setdefault(m.spec.name, m.y)
        self._qguard = {}
        for src, k in self.sources.items():
            if canary:
                qb = torch.full((self.m * k + 2 * 128,), _SENTINEL_I8, dtype=torch.int8, device=self.dev)
                db = torch.empty(self.m * (k // I.QK) + 2 * 32, dtype=torch.float32, device=self.dev)
                db.view(torch.int32).fill_(_SENTINEL_F32)
                q = qb[128:128 + self.m * k].view(self.m, k)
                d = db[32:32 + self.m * (k // I.QK)].view(self.m, k // I.QK)
                self._qguard[src] = (qb, db)
            else:
                q = torch.empty((self.m, k), dtype=torch.int8, device=self.dev)
                d = torch.empty((self.m, k // I.QK), dtype=torch.float32, device=self.dev)
            self.qbuf[src] = B.QAct(q, d, k, self.m)
        self.kernels_per_step = len(self.sources) + len(self.mats)
        self._chain_calls = {}
        self.chain_ws = None

    def check_canaries(self) -> None:
        """With canary=True: every guard band around the outputs (the y
        buffers, the quantised activations and their scales) still holds its
        sentinel; raises AssertionError naming the buffer otherwise."""
        if not self.canary:
            return
        yb = self.y_all.view(torch.int32).cpu().numpy()
        inside = np.zeros(yb.size, dtype=bool)
        for m, off in zip(self.mats, self.y_offs):
            inside[off:off + m.y.numel()] = True
        bad = np.nonzero(~inside & (yb != _SENTINEL_F32))[0]
        assert bad.size == 0, f"y guard band overwritten at {bad[:8].tolist()} (buffer of {yb.size})"
        for src, (qb, db) in self._qguard.items():
            q = qb.cpu().numpy()
            d = db.view(torch.int32).cpu().numpy()
            for name, arr, n, sent in (("q", q, 128, _SENTINEL_I8), ("d", d, 32, _SENTINEL_F32)):
                assert np.all(arr[:n] == sent), f"{src}.{name}: head guard band overwritten"
                assert np.all(arr[arr.size - n:] == sent), f"{src}.{name}: tail guard band overwritten"

    # ---- the whole pass as one chain launch ------------------------------------
    def chain_phases(self):
        """Runs of consecutive products that read the same input."""
        phases = []
        for i, m in enumerate(self.mats):
            if phases and phases[-1][0] == m.src:
                phases[-1][2] += 1
            else:
                phases.append([m.src, i, 1])
        return phases

    def chain_call(self, copy: int = 0):
        if copy not in self._chain_calls:
            if self.m != 1:
                raise ValueError("decode chains are M = 1")
            phases = self.chain_phases()
            if self.chain_ws is None:
                nbytes = B.mlq_chain_workspace_bytes(len(phases))
                self.chain_ws = torch.zeros((nbytes + 3) // 4, dtype=torch.int32, device=self.dev)
            cp = [B.ChainPhase(self.fp32[src], self.sources[src], first, count,
                               self.qbuf[src].q, self.qbuf[src].d) for src, first, count in phases]
            pr = [B.ChainProduct(B.QTensor(m.q[copy], m.d[copy], m.spec.rows, m.spec.cols,
                                           m.spec.wtype), m.y) for m in self.mats]
            self._chain_calls[copy] = B.ChainCall(cp, pr, self.chain_ws)
        return self._chain_calls[copy]

    def fused_calls(self, copy: int = 0, static_weights: bool = True):
        """One mlq_matvec_fused call per phase.  The runner's weights are
        written once at construction, so it passes MLQ_F_STATIC_WEIGHTS."""
        key = ("fused", copy, static_weights)
        if key not in self._chain_calls:
            if self.m != 1:
                raise ValueError("fused phases are M = 1")
            calls = []
            for src, first, count in self.chain_phases():
                pr = [B.ChainProduct(B.QTensor(m.q[copy], m.d[copy], m.spec.rows, m.spec.cols,
                                               m.spec.wtype), m.y)
                      for m in self.mats[first:first + count]]
                calls.append(B.FusedCall(self.fp32[src], self.sources[src], pr,
                                         self.qbuf[src].q, self.qbuf[src].d,
                                         B.MLQ_F_STATIC_WEIGHTS if static_weights else 0))
            self._chain_calls[key] = calls
        return self._chain_calls[key]

    def step_fused(self, copy: int = 0, stream=None, static_weights: bool = True) -> None:
        """One pass as one mlq_matvec_fused launch per phase."""
        for c in self.fused_calls(copy, static_weights):
            c(stream)

    def phase_weight_ranges(self, k: int, copy: int):
        """(tensor, bytes) of every weight array of phase k, copy `copy`."""
        _, first, count = self.chain_phases()[k]
        out = []
        for m in self.mats[first:first + count]:
            out += [(m.q[copy], m.host_q.nbytes), (m.d[copy], m.host_d.nbytes)]
        return out

    def phase_calls(self, copy: int = 0, static_weights: bool = True, prefetch: str = "none",
                    handoff: str = "q8", static_input: bool = True):
        """One mlq_decode_phase call per phase (static_input: the phases that
        read the workload's own float inputs pass MLQ_F_STATIC_INPUT).  handoff
        "q8": a product whose
        output is the input of a later phase also writes it in Q8_0 (into
        that input's buffer), so the later phase starts from quantised bytes
        (the producing phase then splits its rows in whole 32-row blocks);
        "float": every phase reads its input as float32 and quantises it in
        each CTA (rows split freely).  The workload's own float inputs are
        quantised by the phase that reads them.  prefetch: "ahead1" /
        "ahead2" -- each phase hints the weights of the phase one / two later
        into L2 (past the last phase: the next pass, next weight copy);
        "self" -- the same phase's next copy (back-to-back timing of one
        phase); "none"."""
        if handoff not in ("q8", "float"):
            raise ValueError(f"handoff {handoff!r}")
        key = ("phase", copy, static_weights, prefetch, handoff, static_input)
        if key not in self._chain_calls:
            if self.m != 1:
                raise ValueError("decode phases are M = 1")
            phases = self.chain_phases()
            pre = set()   # sources whose producer quantises them
            for src, first, count in phases:
                group = self.mats[first:first + count]
                if handoff == "q8" and all(m.spec.rows % I.QK == 0 for m in group):
                    pre.update(m.spec.name for m in group if m.spec.name in self.sources)
            flags = B.MLQ_F_STATIC_WEIGHTS if static_weights else 0
            calls = []
            nph = len(phases)
            for k, (src, first, count) in enumerate(phases):
                pf = ()
                if prefetch in ("ahead1", "ahead2"):
                    kk = k + (1 if prefetch == "ahead1" else 2)
                    pf = self.phase_weight_ranges(kk % nph, (copy + kk // nph) % self.copies)
                elif prefetch == "self":
                    pf = self.phase_weight_ranges(k, (copy + 1) % self.copies)
                elif prefetch != "none":
                    raise ValueError(f"prefetch {prefetch!r}")
                pr = []
                for m in self.mats[first:first + count]:
                    out = self.qbuf[m.spec.name] if m.spec.name in pre else None
                    pr.append(B.PhaseProduct(
                        B.QTensor(m.q[copy], m.d[copy], m.spec.rows, m.spec.cols, m.spec.wtype),
                        m.y, out.q if out else None, out.d if out else None))
                qa = self.qbuf[src]
                if src in pre:
                    calls.append(B.PhaseCall(self.sources[src], pr, xq=qa.q, xd=qa.d, flags=flags,
                                             prefetch=pf))
                else:
                    # the workload's own inputs are written once (or by a copy
                    # before the step's first launch): MLQ_F_STATIC_INPUT lets the
                    # launch read them before the previous kernel has finished
                    own = src in self.x_host and static_input
                    calls.append(B.PhaseCall(self.sources[src], pr, x=self.fp32[src],
                                             xq_out=qa.q, xd_out=qa.d,
                                             flags=flags | (B.MLQ_F_STATIC_INPUT if own else 0),
                                             prefetch=pf))
            self._chain_calls[key] = calls
        return self._chain_calls[key]

    def step_phase(self, copy: int = 0, stream=None, static_weights: bool = True,
                   prefetch: str = "none", handoff: str = "q8") -> None:
        """One pass as one mlq_decode_phase launch per phase."""
        for c in self.phase_calls(copy, static_weights, prefetch, handoff):
            c(stream)

    def step_chain(self, copy: int = 0, stream=None) -> None:
        """One pass as a single mlq_decode_chain launch."""
        self.chain_call(copy)(stream)

    # ---- sizes ---------------------------------------------------------------
    def weight_bytes(self) -> int:
        return sum(m.host_q.nbytes + m.host_d.nbytes for m in self.mats)

    def ops(self) -> int:
        return sum(2 * self.m * m.spec.rows * m.spec.cols for m in self.mats)

    def h2d_bytes(self) -> int:
        return sum(t.numel() * 4 for t in self.x_pinned.values())

    def d2h_bytes(self) -> int:
        return self.y_all.numel() * 4

    # ---- one pass --------------------------------------------------------------
    def weight_ranges(self, i: int, copy: int = 0):
        m = self.mats[i]
        return [(m.q[copy], m.host_q.nbytes), (m.d[copy], m.host_d.nbytes)]

    def step(self, copy: int = 0, stream=None, before_mat=None, after_mat=None,
             prefetch: str | None = None) -> None:
        """Issue one pass on `stream`: each input is quantised right before
        its first consumer, then each product runs.  before_mat/after_mat
        (optional callables taking the matrix index) let the bench record
        events around the products.  prefetch: None, "all" (hint every
        weight of the pass into L2 first) or "next" (hint the next
        product's weights into L2 before each product)."""
        done = set()
        if prefetch == "all":
            ranges = []
            for i in range(len(self.mats)):
                ranges += self.weight_ranges(i, copy)
            B.mlq_prefetch_l2(ranges, stream)
        elif prefetch == "next" and self.mats:
            B.mlq_prefetch_l2(self.weight_ranges(0, copy), stream)
        for i, m in enumerate(self.mats):
            if prefetch == "next" and i + 1 < len(self.mats):
                B.mlq_prefetch_l2(self.weight_ranges(i + 1, copy), stream)
            if m.src not in done:
                B.mlq_quantize_q8(self.qbuf[m.src], self.fp32[m.src], self.sources[m.src], stream)
                done.add(m.src)
            W = B.QTensor(m.q[copy], m.d[copy], m.spec.rows, m.spec.cols, m.spec.wtype)
            if before_mat is not None:
                before_mat(i)
            if self.m == 1:
                f = B.mlq_matvec_q4 if m.spec.wtype == I.Q4_0 else B.mlq_matvec_q8
                f(m.y, W, self.qbuf[m.src], 0, m.spec.rows, stream)
            else:
                B.mlq_gemm_q4_small_m(m.y, m.spec.rows, W, self.qbuf[m.src], self.m, 0,
                                      m.spec.rows, stream)
            if after_mat is not None:
                after_mat(i)

    def product(self, i: int, copy: int = 0, stream=None) -> None:
        """Only the i-th product (its input must already be quantised)."""
        m = self.mats[i]
        W = B.QTensor(m.q[copy], m.d[copy], m.spec.rows, m.spec.cols, m.spec.wtype)
        if self.m == 1:
            f = B.mlq_matvec_q4 if m.spec.wtype == I.Q4_0 else B.mlq_matvec_q8
            f(m.y, W, self.qbuf[m.src], 0, m.spec.rows, stream)
        else:
            B.mlq_gemm_q4_small_m(m.y, m.spec.rows, W, self.qbuf[m.src], self.m, 0, m.spec.rows,
                                  stream)

    def upload_inputs(self, stream=None) -> None:
        """Host -> device copy of every external input (pinned, async)."""
        with torch.cuda.stream(stream) if stream is not None else _null():
            for src, t in self.x_pinned.items():
                self.fp32[src].copy_(t, non_blocking=True)

    def outputs_to_host(self, host: dict | None = None) -> dict:
        """Every product's output to pinned host memory in one D2H copy (the
        outputs are views of one device buffer); returns {name: host view}."""
        if host is None:
            flat = torch.empty(self.y_all.numel(), dtype=torch.float32).pin_memory()
            host = {"_flat": flat}
            for m, off in zip(self.mats, self.y_offs):
                host[m.spec.name] = flat[off: off + m.y.numel()].view(m.y.shape)
        host["_flat"].copy_(self.y_all, non_blocking=True)
        return host


class _null:
    def __enter__(self):
        return None

    def __exit__(self, *a):
        return False


def phase_groups(mats, max_products: int = 4):
    """Consecutive products (name, rows, cols, input) that read one input,
    at most max_products per group, in pass order: [(input, [names], K)].
    A product that reads another's output starts a new group after it, so
    every group's input exists before the group runs."""
    out = []
    for name, rows, cols, inp in mats:
        if out and out[-1][0] == inp and len(out[-1][1]) < max_products:
            out[-1][1].append(name)
        else:
            out.append((inp, [name], cols))
    return out


class Q4KRunner:
    """Device buffers and one pass of a Q4KWorkload through the C ABI: per
    input, mlq_quantize_q8k, then every mlq_matvec_q4k that reads it."""

    def __init__(self, wl: I.Q4KWorkload, copies: int = 1, device: str = "cuda:0"):
        self.wl = wl
        self.copies = copies
        self.dev = torch.device(device)
        self.host = {}
        self.W = [dict() for _ in range(copies)]
        self.y = {}
        self.src = {}
        for i, (name, rows, cols, inp) in enumerate(wl.mats):
            q, s, d, dmin = I.q4k_weights(rows, cols, seed=wl.seed + i)
            self.host[name] = (q, s, d, dmin, rows, cols)
            for c in range(copies):
                self.W[c][name] = B.Q4KTensor(*(torch.from_numpy(t).to(self.dev) for t in (q, s, d, dmin)),
                                              rows, cols)
            self.y[name] = torch.zeros(rows, dtype=torch.float32, device=self.dev)
            self.src.setdefault(inp, cols)
        x_cols = self.src["x"]
        self.x_host = I.activations(1, x_cols, seed=wl.seed + 1000)[0]
        self.x = torch.from_numpy(self.x_host).to(self.dev)
        self.x_pinned = torch.from_numpy(self.x_host).pin_memory()
        self.act = {}
        for name, k in self.src.items():
            self.act[name] = B.Q8KAct(torch.empty(k, dtype=torch.int8, device=self.dev),
                                      torch.empty(k // I.QKK, dtype=torch.float32, device=self.dev),
                                      torch.empty(k // I.QK, dtype=torch.int32, device=self.dev), k)
        self.launches_per_step = len(self.src) + len(wl.mats)

    def vec(self, name):
        return self.x if name == "x" else self.y[name]

    def step(self, copy: int = 0, stream=None) -> None:
        done = set()
        for name, rows, cols, inp in self.wl.mats:
            if inp not in done:
                B.mlq_quantize_q8k(self.act[inp], self.vec(inp), cols, stream)
                done.add(inp)
            B.mlq_matvec_q4k(self.y[name], self.W[copy][name], self.act[inp], 0, rows, stream)

    def phases(self):
        """The pass's phases (phase_groups); one mlq_q4k_phase launch each."""
        return phase_groups(self.wl.mats)

    def step_phase(self, copy: int = 0, stream=None) -> None:
        """One pass as phases: each launch quantises its float input itself
        (the pass's own input x, written once, as MLQ_F_STATIC_INPUT)."""
        for inp, names, cols in self.phases():
            B.mlq_q4k_phase(self.vec(inp), cols, [(self.W[copy][n], self.y[n]) for n in names], stream,
                            flags=B.MLQ_F_STATIC_INPUT if inp == "x" else 0)

    def product(self, name: str, copy: int = 0, stream=None) -> None:
        rows, inp = self.host[name][4], [m[3] for m in self.wl.mats if m[0] == name][0]
        B.mlq_matvec_q4k(self.y[name], self.W[copy][name], self.act[inp], 0, rows, stream)

    def weight_bytes(self) -> int:
        return sum(q.nbytes + s.nbytes + d.nbytes + dm.nbytes for q, s, d, dm, _, _ in self.host.values())

    def ops(self) -> int:
        return sum(2 * rows * cols for _, rows, cols, _ in self.wl.mats)


class NBitsRunner:
    """Device buffers and one pass of an NBitsWorkload through the C ABI:
    per input mlq_quantize_blk, then every mlq_matvec_nbits that reads it.
    Scale and zero-point rows are padded to 16 bytes (the tensor's strides)."""

    def __init__(self, wl: I.NBitsWorkload, copies: int = 1, device: str = "cuda:0"):
        self.wl = wl
        self.copies = copies
        self.dev = torch.device(device)
        self.host = {}
        self.W = [dict() for _ in range(copies)]
        self.y = {}
        self.src = {}
        t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(self.dev)
        for i, (name, rows, cols, inp) in enumerate(wl.mats):
            q, sc, zp = I.nbits_weights(rows, cols, wl.bits, wl.blk, wl.f16, wl.with_zp, seed=wl.seed + i)
            self.host[name] = (q, sc, zp)
            scp = I.pad_rows(sc)
            zpp = None if zp is None else I.pad_rows(zp)
            for c in range(copies):
                self.W[c][name] = B.NBitsTensor(
                    t(q), t(scp.view(np.uint16) if wl.f16 else scp), None if zpp is None else t(zpp),
                    rows, cols, wl.bits, wl.blk, 1 if wl.f16 else 0, scp.shape[1],
                    0 if zpp is None else zpp.shape[1])
            self.y[name] = torch.zeros(rows, dtype=torch.float32, device=self.dev)
            self.src.setdefault(inp, cols)
        self.x_host = I.activations(1, self.src["x"], seed=wl.seed + 1000)[0]
        self.x = torch.from_numpy(self.x_host).to(self.dev)
        self.x_pinned = torch.from_numpy(self.x_host).pin_memory()
        self.act = {}
        for name, k in self.src.items():
            self.act[name] = B.BlkAct(torch.empty(k, dtype=torch.int8, device=self.dev),
                                      torch.empty(k // wl.blk, dtype=torch.float32, device=self.dev),
                                      torch.empty(k // wl.blk, dtype=torch.int32, device=self.dev), k, wl.blk)
        self.launches_per_step = len(self.src) + len(wl.mats)

    def vec(self, name):
        return self.x if name == "x" else self.y[name]

    def step(self, copy: int = 0, stream=None) -> None:
        done = set()
        for name, rows, cols, inp in self.wl.mats:
            if inp not in done:
                B.mlq_quantize_blk(self.act[inp], self.vec(inp), cols, stream)
                done.add(inp)
            B.mlq_matvec_nbits(self.y[name], self.W[copy][name], self.act[inp], 0, rows, stream)

    def phases(self):
        """The pass's phases (phase_groups); one mlq_nbits_phase launch each."""
        return phase_groups(self.wl.mats)

    def step_phase(self, copy: int = 0, stream=None) -> None:
        """One pass as phases: each launch quantises its float input itself
        (the pass's own input x, written once, as MLQ_F_STATIC_INPUT)."""
        for inp, names, cols in self.phases():
            B.mlq_nbits_phase(self.vec(inp), cols, [(self.W[copy][n], self.y[n]) for n in names], stream,
                              flags=B.MLQ_F_STATIC_INPUT if inp == "x" else 0)

    def product(self, name: str, copy: int = 0, stream=None) -> None:
        rows, inp = [(m[1], m[3]) for m in self.wl.mats if m[0] == name][0]
        B.mlq_matvec_nbits(self.y[name], self.W[copy][name], self.act[inp], 0, rows, stream)

    def weight_bytes(self) -> int:
        return sum(q.nbytes + sc.nbytes + (0 if zp is None else zp.nbytes) for q, sc, zp in self.host.values())

    def ops(self) -> int:
        return sum(2 * rows * cols for _, rows, cols, _ in self.wl.mats)
