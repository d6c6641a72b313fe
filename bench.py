"""Benchmark of the block-quantized decode hot path on GB300.

One step = one pass of the workload's hot path through the C ABI: Q8_0
quantisation of each input vector, then every Q4_0 / Q8_0 product.  The
default workload is the largest single-GPU configuration: the 8-layer
Llama-7B-shaped FFN stack in Q8_0 (16 chained products, 811.6 MB) plus the
Qwen2.5-0.5B-shaped lm_head (151936 x 896 Q8_0, 153.2 MB), M = 1.  The same
line carries, under "also", the Q4_0 stack and the batched M = 4 / M = 16
Q4_0 products, each timed the same way; --workload picks another workload
alone.

Timing: W untimed warm-up steps, then R back-to-back repeats of exactly K
steps, each bracketed by CUDA events on the launching stream, with a barrier
and a device synchronize on both sides; R is chosen so that the region lasts
at least --min-region seconds and ms_per_step is the median over the
repeats.  The steps replay CUDA graphs, and consecutive steps read
different weight copies (together more than 3x the L2 size), so every step
streams its weights from HBM.  Rank 0 prints one JSON line.

Also measured in the same run: the dominant kernel's per-launch duration
(CUDA events captured into an instrumented copy of the graphs), the same
metric end to end (pinned host input -> device, step, outputs -> host),
SM clocks during the timed region, and the CPU oracle on the host cores
(cpu_baseline).  ``--impl reference`` times the oracle alone as the
reference arm.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "M=1 Q4_0/Q8_0 matvec weight GB/s and GOP/s; % of GB300 HBM roofline"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=0,
                   help="timed steps (0 = as many as fill about --seconds of the timed region)")
    p.add_argument("--seconds", type=float, default=1.5)
    p.add_argument("--min-region", type=float, default=1.0,
                   help="the K timed steps are repeated back to back until the timed region "
                        "lasts at least this many seconds (clock samples under load)")
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="llama7b_ffn_q8_lm_head")
    p.add_argument("--no-extras", action="store_true",
                   help="headline workload only (skip the Q4_0 stack and M = 4 / 16 records)")
    p.add_argument("--copies", type=int, default=0, help="weight copies (0 = auto, > 3x L2)")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-graph", action="store_true")
    p.add_argument("--path", choices=["auto", "phase", "fused", "chain", "calls"], default="auto",
                   help="phase: one mlq_decode_phase launch per phase, each phase writing "
                        "the next one's input already quantised; fused: one mlq_matvec_fused "
                        "launch per phase (float inputs); chain: one mlq_decode_chain launch "
                        "per step; calls: one C-ABI call per quantize and product; auto: phase "
                        "for M = 1 (one launch per phase, measured fastest at every size), "
                        "calls for M > 1")
    p.add_argument("--phase-prefetch", choices=["none", "ahead1", "ahead2"], default="none",
                   help="phase path: each phase hints the weights of the phase one / two "
                        "later into L2 once it has read its input")
    p.add_argument("--handoff", choices=["q8", "float"], default="q8",
                   help="phase path: a phase's output reaches the next phase as Q8_0 written by "
                        "the producing launch (q8), or as float32 quantised by every CTA of the "
                        "reading launch (float)")
    p.add_argument("--prefetch", choices=["none", "all", "next"], default="none",
                   help="L2 prefetch of weights through mlq_prefetch_l2: all (whole pass "
                        "first) or next (one product ahead); measured slower in-chain, so off")
    return p.parse_args()


# ----------------------------------------------------------------------------
# distributed plumbing (one process per GPU; no data-path collective)
# ----------------------------------------------------------------------------
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        dist.init_process_group(backend=backend)
        pg = dist
    return world, rank, local, pg


def barrier(pg, device=None):
    if pg is not None:
        if device is not None:
            pg.barrier(device_ids=[device])
        else:
            pg.barrier()


def max_over_ranks(pg, v: float, device=None) -> float:
    if pg is None:
        return v
    import torch
    t = torch.tensor([v], dtype=torch.float64, device=device if device is not None else "cpu")
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------
# host-side helpers
# ----------------------------------------------------------------------------
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except Exception:
        return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self, t0: float | None = None, t1: float | None = None):
        """Median clocks of the samples taken between host times t0 and t1
        (the timed region); if none fell inside it, of all samples taken."""
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        import datetime
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        samples = []
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                samples.append((ts, float(parts[1]), float(parts[2]),
                                {n for n, v in zip(names, parts[5:9]) if v.lower() == "active"}))
            except ValueError:
                continue
        if not samples:
            return None
        inside = [x for x in samples if t0 is not None and t0 <= x[0] <= t1]
        use = inside or samples
        return {"sm_mhz": statistics.median(x[1] for x in use),
                "sm_max_mhz": max(x[2] for x in use),
                "samples": len(use), "window": "timed region" if inside else "whole run",
                "reasons": sorted(set().union(*[x[3] for x in use]))}


def phase_kernel_of(r, num_sms: int):
    """The kernel that streams most of a pass's weight bytes on the phase
    path: phase_kernel when a CTA's share of a phase's rows fits in shared
    memory (about 120 KB with the input), else phase_ring_kernel.  An
    estimate of the library's choice, used to label the roofline only."""
    fit = ring = 0
    for _, first, count in r.chain_phases():
        mats = r.mats[first:first + count]
        rows = sum(m.spec.rows for m in mats)
        nb = mats[0].spec.cols // 32
        rowb = nb * ((16 if mats[0].spec.wtype == 1 else 32) + 4)
        share = -(-rows // max(1, min(num_sms, rows))) + 16  # + uneven 32-row splits
        smem = -(-(nb * 36) // 128) * 128 + share * rowb
        nbytes = sum(m.host_q.nbytes + m.host_d.nbytes for m in mats)
        if smem <= 120 * 1024:
            fit += nbytes
        else:
            ring += nbytes
    return ("phase_kernel", "phase.cu") if fit >= ring else ("phase_ring_kernel", "phase_ring.cu")


def e2e_graph_steps(args, copies: int, stream, body):
    """One end-to-end step per call: a replay of the graph that holds body(c)
    (the H2D copy of the step's inputs from pinned memory, the C-ABI calls,
    the D2H copy of the outputs) for weight copy c = i % copies, or body run
    eagerly with --no-graph.  Every graph is replayed once before it returns."""
    import torch
    graphs = []
    if not args.no_graph:
        for c in range(copies):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                body(c)
            graphs.append(g)

    def step(i):
        if graphs:
            graphs[i % copies].replay()
        else:
            body(i % copies)
    with torch.cuda.stream(stream):
        for i in range(copies):
            step(i)
    stream.synchronize()
    return step


def ncu_traffic(profile: str, sources, bytes_per_launch: float):
    """DRAM bytes per launch of the dominant kernel: the DRAM/algorithmic
    ratio of the committed ncu summary profiles/<profile>.md times the
    algorithmic bytes per launch, if the summary was taken on the current
    kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", f"{profile}.md")
    csrc = os.path.join(ROOT, "block_quantized_decode_gb300", "csrc")
    try:
        text = open(path).read()
        h = hashlib.sha256()
        for f in sources:
            h.update(open(os.path.join(csrc, f), "rb").read())
        sha = h.hexdigest()[:16]
    except OSError:
        return None
    m_sha = re.search(r"source_sha256_16:\s*([0-9a-f]+)", text)
    m_r = re.search(r"dram_over_algorithmic:\s*([0-9.eE+]+)", text)
    if not m_sha or not m_r or m_sha.group(1) != sha:
        return None
    return float(m_r.group(1)) * bytes_per_launch


# ----------------------------------------------------------------------------
# the CPU oracle on the host cores (cpu_baseline and the reference arm)
# ----------------------------------------------------------------------------
class OraclePass:
    """One pass of the workload with the oracle: quantise each input, then
    every product with rows split statically over `threads` host threads
    (the oracle's own [r0, r1) interface; ctypes releases the GIL)."""

    def __init__(self, wl, threads: int):
        import numpy as np
        from concurrent.futures import ThreadPoolExecutor

        import oracle
        from block_quantized_decode_gb300 import inputs as I
        self.np = np
        self.O = oracle
        self.wl = wl
        self.threads = threads
        self.pool = ThreadPoolExecutor(max_workers=threads)
        self.mats = []
        self.x = {}
        for i, mv in enumerate(wl.mats):
            src = f"x{mv.cols}" if mv.input_of == "x" else mv.input_of
            if mv.input_of == "x" and src not in self.x:
                self.x[src] = I.activations(wl.m, mv.cols, seed=1000 + len(self.x))
            q, d = I.weights(mv.wtype, mv.rows, mv.cols, seed=i)
            self.mats.append((mv, src, q, d))
        self.weight_bytes = sum(q.nbytes + d.nbytes for _, _, q, d in self.mats)
        self.ops = sum(2 * wl.m * mv.rows * mv.cols for mv, _, _, _ in self.mats)

    def run(self):
        np, O = self.np, self.O
        fp = dict(self.x)
        qa = {}
        for mv, src, q, d in self.mats:
            if src not in qa:
                qa[src] = O.quantize_q8(fp[src].reshape(self.wl.m, -1))
            xq, xd = qa[src]
            Y = np.zeros((self.wl.m, mv.rows), dtype=np.float32)
            cuts = [mv.rows * t // self.threads for t in range(self.threads + 1)]
            futs = []
            for t in range(self.threads):
                a, b = cuts[t], cuts[t + 1]
                if b > a:
                    futs.append(self.pool.submit(O.gemm_small_m, mv.wtype, q, d, mv.rows, mv.cols,
                                                 xq, xd, self.wl.m, a, b, None, Y))
            for f in futs:
                f.result()
            fp[mv.name] = Y


class OracleLayerPass:
    """One token through one decode layer with the oracle (Design Spec Sec. 6
    forward pass): the same seeded inputs as the GPU layer, the products'
    rows split over `threads` host threads."""

    def __init__(self, shape, threads: int):
        import numpy as np
        from concurrent.futures import ThreadPoolExecutor

        import oracle
        from block_quantized_decode_gb300 import inputs as I
        self.np, self.O, self.s, self.threads = np, oracle, shape, threads
        self.pool = ThreadPoolExecutor(max_workers=threads)
        self.W = {name: I.weights(shape.wtype, rows, cols, shape.seed + i) + (rows, cols)
                  for i, (name, rows, cols) in enumerate(shape.mats())}
        self.att_norm = I.norm_weights(shape.dim, shape.seed + 10)
        self.ffn_norm = I.norm_weights(shape.dim, shape.seed + 11)
        self.kc = np.zeros((shape.pos + 1, shape.kv_dim), np.float32)
        self.vc = np.zeros_like(self.kc)
        self.kc[:shape.pos] = I.kv_history(shape.pos, shape.kv_dim, shape.seed + 12)
        self.vc[:shape.pos] = I.kv_history(shape.pos, shape.kv_dim, shape.seed + 13)
        self.x0 = I.activations(1, shape.dim, shape.seed + 14)[0]
        self.cos, self.sin = oracle.rope_tables(shape.pos + 1, shape.head_dim, shape.rope_theta)
        self.weight_bytes = sum(q.nbytes + d.nbytes for q, d, _, _ in self.W.values())
        self.ops = sum(2 * rows * cols for _, _, rows, cols in self.W.values())

    def _mv(self, name, xq, xd):
        q, d, rows, cols = self.W[name]
        y = self.np.zeros(rows, dtype=self.np.float32)
        cuts = [rows * t // self.threads for t in range(self.threads + 1)]
        futs = [self.pool.submit(self.O.matvec, self.s.wtype, q, d, rows, cols, xq, xd, a, b, y)
                for a, b in zip(cuts, cuts[1:]) if b > a]
        for f in futs:
            f.result()
        return y

    def run(self):
        O, s = self.O, self.s
        x = self.x0.copy()
        h = O.quantize_q8(O.rmsnorm(x, self.att_norm, s.norm_eps))
        q, k, v = (self._mv(n, *h) for n in ("wq", "wk", "wv"))
        q, k = O.rope(q, k, self.cos[s.pos], self.sin[s.pos], s.head_dim, s.n_heads, s.n_kv_heads)
        self.kc[s.pos], self.vc[s.pos] = k, v
        o = O.attention(q, self.kc, self.vc, s.pos + 1, s.head_dim, s.n_heads, s.n_kv_heads)
        x = O.add(x, self._mv("wo", *O.quantize_q8(o)))
        h = O.quantize_q8(O.rmsnorm(x, self.ffn_norm, s.norm_eps))
        g = O.silu_mul(self._mv("w1", *h), self._mv("w3", *h))
        return O.add(x, self._mv("w2", *O.quantize_q8(g)))


class OracleQ4KPass:
    """One pass of a Q4KWorkload with the oracle: quantise each input per
    256, then every product with rows split statically over `threads` host
    threads (the oracle's own [r0, r1) interface)."""

    def __init__(self, wl, threads: int):
        import numpy as np
        from concurrent.futures import ThreadPoolExecutor

        import oracle
        from block_quantized_decode_gb300 import inputs as I
        self.np, self.O, self.wl, self.threads = np, oracle, wl, threads
        self.pool = ThreadPoolExecutor(max_workers=threads)
        self.W = {name: I.q4k_weights(rows, cols, seed=wl.seed + i) + (rows, cols)
                  for i, (name, rows, cols, _) in enumerate(wl.mats)}
        self.x0 = I.activations(1, wl.mats[0][2], seed=wl.seed + 1000)[0]
        self.weight_bytes = sum(q.nbytes + s.nbytes + d.nbytes + dm.nbytes
                                for q, s, d, dm, _, _ in self.W.values())
        self.ops = sum(2 * rows * cols for _, rows, cols, _ in wl.mats)

    def run(self):
        O, np = self.O, self.np
        vecs = {"x": self.x0}
        acts = {}
        for name, rows, cols, inp in self.wl.mats:
            if inp not in acts:
                acts[inp] = O.quantize_q8k(vecs[inp])
            q, s, d, dm, _, _ = self.W[name]
            y = np.zeros(rows, dtype=np.float32)
            cuts = [rows * t // self.threads for t in range(self.threads + 1)]
            futs = [self.pool.submit(O.matvec_q4k, q, s, d, dm, rows, cols, *acts[inp], a, b, y)
                    for a, b in zip(cuts, cuts[1:]) if b > a]
            for f in futs:
                f.result()
            vecs[name] = y
        return vecs


class OracleNBitsPass:
    """One pass of an NBitsWorkload with the oracle (per input the per-block
    quantiser, then every product with rows split over `threads` threads)."""

    def __init__(self, wl, threads: int):
        import numpy as np
        from concurrent.futures import ThreadPoolExecutor

        import oracle
        from block_quantized_decode_gb300 import inputs as I
        self.np, self.O, self.wl, self.threads = np, oracle, wl, threads
        self.pool = ThreadPoolExecutor(max_workers=threads)
        self.W = {name: I.nbits_weights(rows, cols, wl.bits, wl.blk, wl.f16, wl.with_zp, seed=wl.seed + i)
                  for i, (name, rows, cols, _) in enumerate(wl.mats)}
        self.x0 = I.activations(1, wl.mats[0][2], seed=wl.seed + 1000)[0]
        self.weight_bytes = sum(q.nbytes + sc.nbytes + (0 if zp is None else zp.nbytes)
                                for q, sc, zp in self.W.values())
        self.ops = sum(2 * rows * cols for _, rows, cols, _ in wl.mats)

    def run(self):
        O, np, wl = self.O, self.np, self.wl
        vecs = {"x": self.x0}
        acts = {}
        for name, rows, cols, inp in wl.mats:
            if inp not in acts:
                acts[inp] = O.quantize_blk(vecs[inp], wl.blk)
            q, sc, zp = self.W[name]
            xq, xd, _ = acts[inp]
            y = np.zeros(rows, dtype=np.float32)
            cuts = [rows * t // self.threads for t in range(self.threads + 1)]
            futs = [self.pool.submit(O.matvec_nbits, q, sc, zp, rows, cols, wl.bits, wl.blk, xq, xd, a, b, y)
                    for a, b in zip(cuts, cuts[1:]) if b > a]
            for f in futs:
                f.result()
            vecs[name] = y
        return vecs


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def oracle_pass(wl, threads: int):
    from block_quantized_decode_gb300 import inputs as I
    if isinstance(wl, I.LayerShape):
        return OracleLayerPass(wl, threads)
    if isinstance(wl, I.Q4KWorkload):
        return OracleQ4KPass(wl, threads)
    if isinstance(wl, I.NBitsWorkload):
        return OracleNBitsPass(wl, threads)
    return OraclePass(wl, threads)


def time_oracle(wl, seconds: float, threads: int, max_steps: int | None = None):
    op = oracle_pass(wl, threads)
    op.run()  # warm (page-in, thread start)
    n, t0 = 0, time.perf_counter()
    while True:
        op.run()
        n += 1
        el = time.perf_counter() - t0
        if (max_steps is not None and n >= max_steps) or (max_steps is None and el >= seconds):
            break
    return op, n, el


# ----------------------------------------------------------------------------
# the reference arm: the oracle as it stands
# ----------------------------------------------------------------------------
def run_reference(args, wl, world, rank):
    if rank != 0:
        return 0
    from block_quantized_decode_gb300 import inputs as I
    threads = host_cores()
    layer = isinstance(wl, (I.LayerShape, I.Q4KWorkload, I.NBitsWorkload))
    op = oracle_pass(wl, threads)
    warm = max(0, args.warmup)
    for _ in range(warm):
        op.run()
    steps = args.steps if args.steps > 0 else max(3, int(args.seconds / 0.1))
    t0 = time.perf_counter()
    for _ in range(steps):
        op.run()
    el = time.perf_counter() - t0
    v = op.weight_bytes * steps / el / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world,
        "steps": steps, "warmup": warm, "ms_per_step": el / steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int8 dot -> int32, f32 accumulate (CPU oracle)", "data": "synthetic",
        "config": {"workload": wl.name, "M": 1 if layer else wl.m, "weight_bytes_per_step": op.weight_bytes},
        "gops": op.ops * steps / el / 1e9,
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": f"{steps} full passes of {wl.name} after {warm} warm-up passes, "
                                   f"rows split over {threads} threads"},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


MAX_GRAPH_LAUNCHES = 4096
# the size from which the library runs an M = 1 product call as a one-product
# ring phase (matvec.cu)
PHASE_ROUTE_BYTES = 16 << 20


def step_graphs(stream, one_pass, copies, per_step_launches, use_graphs):
    """Graphs for timed runs of whole steps: one graph per weight copy, one
    cycle graph of every copy, and prepare(n), which captures n consecutive
    steps (cycling through the copies from copy 0) as ONE graph, so that
    every step of a timed repeat chains to the next through programmatic
    dependent launch (at most MAX_GRAPH_LAUNCHES kernel launches per graph;
    beyond that, do_steps runs whole cycles).  do_steps(n) runs exactly n
    steps from copy 0.  Returns (prepare, do_steps, run_graphs), the last
    the graphs prepare() captured, by step count."""
    import torch
    graphs, cycle, run_graphs = [], None, {}
    if use_graphs:
        for c in range(copies):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                one_pass(c)
            graphs.append(g)
        cycle = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cycle, stream=stream):
            for c in range(copies):
                one_pass(c)

    def prepare(n):
        if not graphs or n <= 0 or n in run_graphs or n * per_step_launches > MAX_GRAPH_LAUNCHES:
            return
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(n):
                one_pass(i % copies)
        run_graphs[n] = g

    def do_steps(n):
        if n in run_graphs:
            run_graphs[n].replay()
            return
        i = 0
        if cycle is not None:
            while n - i >= copies:
                cycle.replay()
                i += copies
        while i < n:
            if graphs:
                graphs[i % copies].replay()
            else:
                one_pass(i % copies)
            i += 1
    return prepare, do_steps, run_graphs

# ----------------------------------------------------------------------------
# timing helpers shared by every workload kind
# ----------------------------------------------------------------------------
def timed_region(args, stream, do_steps, pg, dev, clocks, prepare=None):
    """W warm-up steps (exactly args.warmup), then the timed region: R
    back-to-back repeats of exactly K steps, each repeat bracketed by CUDA
    events on `stream`, with a barrier and a device synchronize on both sides
    of the region.  K = --steps (or, when 0, as many steps as fill about
    --seconds); R = enough repeats that the region lasts at least
    --min-region seconds, so that the clock sampler sees the GPU under load.
    prepare(n), when given, is called before n steps are first run (outside
    any timing), e.g. to capture them as one CUDA graph.
    Returns (K, R, median ms per step over the repeats (max over ranks),
    [ms per step of each repeat], region seconds, clocks)."""
    import torch
    if prepare is not None:
        prepare(max(0, args.warmup))
        if args.steps > 0:
            prepare(args.steps)
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        a0.record(stream)
        do_steps(max(0, args.warmup))
        a1.record(stream)
    stream.synchronize()
    per = a0.elapsed_time(a1) / 1e3 / max(1, args.warmup) if args.warmup > 0 else None
    if per is None:  # no warm-up asked: one untimed probe step sizes the region
        with torch.cuda.stream(stream):
            a0.record(stream)
            do_steps(1)
            a1.record(stream)
        stream.synchronize()
        per = a0.elapsed_time(a1) / 1e3
    steps = args.steps
    if steps <= 0:
        steps = max(10, int(args.seconds / max(per, 1e-7)))
        steps = int(max_over_ranks(pg, float(steps), dev))
    if prepare is not None:
        prepare(steps)
    reps = max(1, math.ceil(args.min_region / max(steps * per, 1e-7)))
    reps = int(max_over_ranks(pg, float(min(reps, 100000)), dev))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(reps)]
    barrier(pg, dev.index if dev is not None else None)
    torch.cuda.synchronize()
    t_host0 = time.time()
    with torch.cuda.stream(stream):
        for e0, e1 in evs:
            e0.record(stream)
            do_steps(steps)
            e1.record(stream)
    torch.cuda.synchronize()
    t_host1 = time.time()
    barrier(pg, dev.index if dev is not None else None)
    clk = clocks.stop(t_host0, t_host1)
    per_rep = [e0.elapsed_time(e1) / steps for e0, e1 in evs]
    med = statistics.median(per_rep)
    med = max_over_ranks(pg, med, dev)
    return steps, reps, med, per_rep, t_host1 - t_host0, clk


def back_to_back_us(stream, launch, launches: int) -> float:
    """Mean duration of one launch: `launches` back-to-back calls of
    launch(j) captured in one CUDA graph, best of 3 replays, CUDA events on
    the launching stream."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for j in range(launches):
            launch(j)
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    best = None
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            g.replay()
            b.record(stream)
        stream.synchronize()
        t = a.elapsed_time(b) / 1e3 / launches
        best = t if best is None else min(best, t)
    del g
    return best * 1e6


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------
def measure_workload(args, wl, world, local, pg, *, path_arg="auto", with_e2e=True):
    """Time one Workload (M = 1 products or a small-M GEMM pass) through the
    C ABI: returns the fields of its bench record (value, step time,
    roofline of the dominant kernel, end to end, launches)."""
    import torch

    import block_quantized_decode_gb300 as M
    from block_quantized_decode_gb300 import inputs as I
    from block_quantized_decode_gb300.runner import WorkloadRunner

    dev = torch.device("cuda", local)
    props = torch.cuda.get_device_properties(local)
    l2 = getattr(props, "L2_cache_size", 126 * 2 ** 20)
    wbytes = sum((mv.rows * mv.cols // 2 if mv.wtype == I.Q4_0 else mv.rows * mv.cols)
                 + mv.rows * mv.cols // 32 * 4 for mv in wl.mats)
    copies = args.copies or max(2, math.ceil(3 * l2 / wbytes))
    r = WorkloadRunner(wl, copies=copies, device=f"cuda:{local}")
    pf = None if args.prefetch == "none" else args.prefetch
    path = path_arg if path_arg != "auto" else ("phase" if r.m == 1 else "calls")

    def one_pass(c):
        if path == "chain":
            r.step_chain(copy=c)
        elif path == "fused":
            r.step_fused(copy=c)
        elif path == "phase":
            r.step_phase(copy=c, prefetch=args.phase_prefetch, handoff=args.handoff)
        else:
            r.step(copy=c, prefetch=pf)
    assert r.weight_bytes() == wbytes
    stream = torch.cuda.Stream(device=dev)
    clocks = ClockSampler(local)
    clocks.start()

    # Initialisation (not counted as warm-up steps): one eager pass per weight
    # copy (kernel attributes, first-touch of every buffer), then the graphs
    # of step_graphs, so that consecutive steps chain through programmatic
    # dependent launch instead of paying a graph launch each.
    with torch.cuda.stream(stream):
        for c in range(copies):
            one_pass(c)
    stream.synchronize()
    # Each run of n steps (the warm-up, each timed repeat of K steps) as ONE
    # CUDA graph of n consecutive steps cycling through the weight copies,
    # captured before it is timed (step_graphs).
    per_step_launches = (1 if path == "chain" else len(r.chain_phases()) if path in ("fused", "phase")
                         else r.kernels_per_step + {None: 0, "all": 1, "next": len(r.mats)}[pf])
    prepare, do_steps, run_graphs = step_graphs(stream, one_pass, copies, per_step_launches, not args.no_graph)

    steps, reps, ms, per_rep, region_s, clk = timed_region(args, stream, do_steps, pg, dev, clocks,
                                                           prepare=prepare)
    value = world * wbytes / (ms / 1e3) / 1e9
    gops = world * r.ops() / (ms / 1e3) / 1e9

    # ---- the dominant kernel: every phase (or product shape) of the step
    # replayed back to back in its own graph (rotating weight copies, so every
    # launch streams from HBM); achieved = algorithmic weight bytes per launch
    # / mean launch duration, summed over the step's launches.
    peaks, peak_src = measured_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))
    launches = 2 * copies
    qt = "Q4_0" if r.mats[0].spec.wtype == I.Q4_0 else "Q8_0"
    roofline = None
    use_graphs = not args.no_graph
    if use_graphs and path == "chain":
        us = back_to_back_us(stream, lambda j: r.step_chain(copy=j % copies), launches)
        ach = wbytes / (us * 1e-6) / 1e9
        roofline = {"kernel": f"decode_stream_kernel<{qt}>", "bound": "hbm", "achieved": ach,
                    "peak": hbm, "unit": "GB/s", "frac": ach / hbm, "peak_source": peak_src,
                    "traffic": ncu_traffic(f"chain_{wl.name}", ("stream.cu", "phase_common.cuh",
                                                                "mlq_device.cuh"), wbytes),
                    "bytes_per_launch": wbytes, "us_per_launch": us,
                    "method": f"{launches} back-to-back chain launches (one per step) in one CUDA "
                              "graph, best of 3 replays, CUDA events on the launching stream"}
    elif use_graphs and path in ("fused", "phase"):
        def calls_of(c):
            return r.fused_calls(c) if path == "fused" else r.phase_calls(
                c, prefetch="self" if args.phase_prefetch != "none" else "none",
                handoff=args.handoff)
        per_phase, tot_bytes, tot_us = [], 0.0, 0.0
        for k, (src, first, count) in enumerate(r.chain_phases()):
            us = back_to_back_us(stream, lambda j, k=k: calls_of(j % copies)[k](), launches)
            mats = r.mats[first:first + count]
            nbytes = sum(m.host_q.nbytes + m.host_d.nbytes for m in mats)
            per_phase.append({"phase": "+".join(m.spec.name for m in mats),
                              "shape": f"{sum(m.spec.rows for m in mats)}x{mats[0].spec.cols}",
                              "bytes": nbytes, "us_per_launch": us, "GBps": nbytes / us / 1e3})
            tot_bytes += nbytes
            tot_us += us
        ach = tot_bytes / (tot_us * 1e-6) / 1e9
        nph = len(per_phase)
        kname, ksrc = phase_kernel_of(r, props.multi_processor_count)
        roofline = {"kernel": f"{kname}<{qt}>", "bound": "hbm", "achieved": ach,
                    "peak": hbm, "unit": "GB/s", "frac": ach / hbm, "peak_source": peak_src,
                    "traffic": ncu_traffic(f"{ksrc[:-3]}_{wl.name}",
                                           (ksrc, "phase_common.cuh", "mlq_device.cuh"),
                                           tot_bytes / nph),
                    "bytes_per_launch": tot_bytes / nph, "us_per_launch": tot_us / nph,
                    "method": f"{launches} back-to-back launches of each phase in one CUDA graph, "
                              "best of 3 replays, CUDA events on the launching stream; achieved = "
                              "sum of per_phase bytes / sum of per_phase us_per_launch",
                    "per_phase": per_phase}
    elif use_graphs:
        # M = 1 calls of PHASE_ROUTE_BYTES and more run as one-product ring
        # phases inside the library (mlq_matvec_q4 / _q8), smaller ones on
        # the M = 1 kernel
        ring_route = r.m == 1 and all(m.host_q.nbytes + m.host_d.nbytes >= PHASE_ROUTE_BYTES for m in r.mats)
        dominant = (f"phase_ring_kernel<{qt}> (one-product phases)" if ring_route else
                    f"matvec_m1_kernel<{qt}>" if r.m == 1 else
                    "gemm_q4_mma_cluster_kernel" if r.m >= 6 else
                    "gemm_q4_ring_kernel" if r.m <= 4 else "gemm_q4_small_m_dp4a_kernel")
        kernel_src = (("phase_ring.cu", "phase_common.cuh", "mlq_device.cuh") if ring_route else
                      ("matvec.cu", "mlq_device.cuh") if r.m == 1 else
                      ("gemm_mma_cluster.cu", "mma_frag.cuh", "mlq_device.cuh") if r.m >= 6 else
                      ("gemm_ring.cu", "phase_common.cuh", "mlq_device.cuh") if r.m <= 4 else
                      ("gemm_small_m.cu", "mlq_device.cuh"))
        kernel_profile = ("phase_ring" if ring_route else "matvec_q4" if r.m == 1 else
                          "gemm_mma_cluster" if r.m >= 6 else "gemm_ring" if r.m <= 4 else "gemm_small_m")
        shapes = {}
        for i, m in enumerate(r.mats):
            shapes.setdefault((m.spec.wtype, m.spec.rows, m.spec.cols), []).append(i)
        per_shape, tot_bytes, tot_us, nl = [], 0.0, 0.0, 0
        for (wt, rows, cols), idx in shapes.items():
            i0 = idx[0]
            us = back_to_back_us(stream, lambda j, i0=i0: r.product(i0, copy=j % copies), launches)
            m = r.mats[i0]
            nbytes = m.host_q.nbytes + m.host_d.nbytes
            per_shape.append({"shape": f"{rows}x{cols}:{'q4_0' if wt == I.Q4_0 else 'q8_0'}",
                              "per_step": len(idx), "bytes": nbytes, "us_per_launch": us,
                              "GBps": nbytes / us / 1e3})
            tot_bytes += nbytes * len(idx)
            tot_us += us * len(idx)
            nl += len(idx)
        ach = tot_bytes / (tot_us * 1e-6) / 1e9
        roofline = {"kernel": dominant, "bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s",
                    "frac": ach / hbm, "peak_source": peak_src,
                    "traffic": ncu_traffic(f"{kernel_profile}_{wl.name}", kernel_src, tot_bytes / nl),
                    "bytes_per_launch": tot_bytes / nl, "us_per_launch": tot_us / nl,
                    "method": f"{launches} back-to-back launches per shape in one CUDA graph, "
                              "best of 3 replays, CUDA events on the launching stream",
                    "per_shape": per_shape}
        if r.m >= 6:
            # the tensor-core side of the same launches: 2 M N K per product
            flops = sum(2.0 * r.m * r.mats[idx[0]].spec.rows * r.mats[idx[0]].spec.cols * len(idx)
                        for idx in shapes.values())
            tf = flops / (tot_us * 1e-6) / 1e12
            bf16 = peaks.get("bf16_tflops")
            roofline["tensor"] = {"achieved": tf, "unit": "TFLOP/s", "operands": "fp16 mma.sync",
                                  "peak_bf16_dense": bf16, "frac": tf / bf16 if bf16 else None,
                                  "peak_note": "fp16 dense = bf16 dense (same tensor rate); "
                                               "burst peak, the kernel timed alone"}

    # ---- end to end: pinned host input -> step -> outputs to pinned host.
    # A decode loop replays one graph per step: the H2D copy of the inputs,
    # the C-ABI calls and the D2H copy of every output, then one sync.
    e2e = None
    if with_e2e:
        host_out = r.outputs_to_host()
        torch.cuda.synchronize()

        def e2e_body(c):
            r.upload_inputs(stream)
            one_pass(c)
            r.outputs_to_host(host_out)
        e2e_step = e2e_graph_steps(args, copies, stream, e2e_body)
        e2e_steps = max(steps, min(500, steps * reps))
        with torch.cuda.stream(stream):
            t0 = time.perf_counter()
            for i in range(e2e_steps):
                e2e_step(i)
                stream.synchronize()
        e2e_s = time.perf_counter() - t0
        e2e_s = max_over_ranks(pg, e2e_s, dev)
        e2e = {"value": world * wbytes * e2e_steps / e2e_s / 1e9, "unit": UNIT,
               "h2d_bytes_per_step": r.h2d_bytes(), "d2h_bytes_per_step": r.d2h_bytes(),
               "steps": e2e_steps, "how": "wall clock; per step: one graph replay holding the pinned "
                                          "H2D of the inputs, the C-ABI calls and the D2H of every "
                                          "output, then a stream sync"}
    assert M.mlq_last_device_error(stream) == M.MLQ_OK
    per_step = (1 if path == "chain" else len(r.chain_phases()) if path in ("fused", "phase") else
                r.kernels_per_step + {None: 0, "all": 1, "next": len(r.mats)}[pf])
    out = {
        "workload": wl.name, "M": r.m, "path": path, "value": value, "unit": UNIT,
        "ms_per_step": ms, "steps": steps, "repeats": reps,
        "ms_per_step_repeats": {"min": min(per_rep), "max": max(per_rep)},
        "timed_region_s": region_s, "gops": gops, "hbm_frac": value / world / hbm,
        "weight_bytes_per_step": wbytes, "roofline": roofline, "e2e": e2e,
        "gpu_launches_per_step": per_step, "gpu_launches": per_step * steps * reps,
        "clocks": clk,
        "matrices": [f"{m.spec.name}:{m.spec.rows}x{m.spec.cols}:"
                     f"{'q4_0' if m.spec.wtype == I.Q4_0 else 'q8_0'}" for m in r.mats],
        "l2": f"inputs larger than L2: {copies} rotating weight copies "
              f"({copies * wbytes / 1e6:.0f} MB vs L2 {l2 / 1e6:.0f} MB)",
        "graphs": (("one graph of the %d timed steps per repeat" % steps) if steps in run_graphs
                   else False if args.no_graph else "one graph per step or per cycle of steps"),
        "l2_prefetch": (args.phase_prefetch if path == "phase" else pf or "none"),
        "handoff": args.handoff if path == "phase" else None,
    }
    del prepare, do_steps, run_graphs, r
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


# The headline line measures the largest single-GPU configuration (the
# 8-layer Llama-7B FFN stack in Q8_0 plus the Qwen2.5-0.5B lm_head); the
# same line carries the Q4_0 stack and the batched M = 4 / 16 products,
# each timed the same way with its own roofline record.
HEADLINE = "llama7b_ffn_q8_lm_head"
EXTRAS = ("llama7b_ffn_q4", "small_m4", "small_m16")


def run_ours(args, wl, world, rank, local, pg):
    import torch

    import block_quantized_decode_gb300 as M
    from block_quantized_decode_gb300 import inputs as I

    torch.cuda.set_device(local)
    M.mlq_init()
    head = measure_workload(args, wl, world, local, pg, path_arg=args.path, with_e2e=True)
    extras = {}
    if args.workload == HEADLINE and not args.no_extras:
        for name in EXTRAS:
            sub = measure_workload(args, I.WORKLOADS[name](), world, local, pg, with_e2e=False)
            sub.pop("e2e", None)
            extras[name] = sub

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        threads = host_cores()
        op, n, el = time_oracle(wl, args.cpu_seconds, threads)
        cpu = {"value": op.weight_bytes * n / el / 1e9, "unit": UNIT, "cores": threads,
               "kind": "oracle",
               "sample": f"{n} full passes of {wl.name} in {el:.1f} s, rows split over {threads} threads"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world,
            "steps": head["steps"], "warmup": max(0, args.warmup), "ms_per_step": head["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "q4_0/q8_0: int8 dot -> int32, f32 accumulate", "data": "synthetic",
            "config": {"workload": head["workload"], "M": head["M"], "matrices": head["matrices"],
                       "weight_bytes_per_step": head["weight_bytes_per_step"], "l2": head["l2"],
                       "graphs": head["graphs"], "path": head["path"],
                       "l2_prefetch": head["l2_prefetch"],
                       "timing": (f"{head['repeats']} back-to-back repeats of exactly "
                                  f"{head['steps']} steps, each bracketed by CUDA events; "
                                  "ms_per_step is the median over the repeats"),
                       "init": "one eager pass per weight copy and the graph captures, before "
                               "the warm-up steps",
                       "parallelism": f"replicas x{world} (independent decode streams)"},
            "repeats": head["repeats"], "ms_per_step_repeats": head["ms_per_step_repeats"],
            "timed_region_s": head["timed_region_s"],
            "gops": head["gops"], "hbm_frac": head["hbm_frac"],
            "roofline": head["roofline"], "cpu_baseline": cpu, "e2e": head["e2e"],
            "gpu_launches": head["gpu_launches"],
            "gpu_launches_per_step": head["gpu_launches_per_step"],
            "clocks": head["clocks"],
        }
        if extras:
            line["also"] = extras
        print(json.dumps(line), flush=True)
    return 0


def run_layer(args, shape, world, rank, local, pg):
    """A whole decode layer (Design Spec Sec. 6) per step: the ten launches
    of DecodeLayer.step for one token at position shape.pos, captured in a
    CUDA graph per weight copy.  value = weight bytes per step / step time
    (the metric's weight GB/s); the KV-cache bytes the attention reads are
    reported beside it."""
    import torch

    import block_quantized_decode_gb300 as M
    from block_quantized_decode_gb300.layer import DecodeLayer

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    M.mlq_init()
    props = torch.cuda.get_device_properties(local)
    l2 = getattr(props, "L2_cache_size", 126 * 2 ** 20)
    probe = DecodeLayer(shape, copies=1, device=f"cuda:{local}")
    wbytes = probe.weight_bytes()
    copies = args.copies or max(2, math.ceil(3 * l2 / wbytes))
    del probe
    L = DecodeLayer(shape, copies=copies, device=f"cuda:{local}")
    L.x.copy_(torch.from_numpy(L.x_in))
    kvb = L.kv_bytes()
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for c in range(copies):
            L.step(copy=c, stream=stream)
    stream.synchronize()
    prepare, do_steps, run_graphs = step_graphs(stream, lambda c: L.step(copy=c, stream=stream), copies,
                                                L.launches_per_step, not args.no_graph)

    clocks = ClockSampler(local)
    clocks.start()
    steps, reps, ms_step, per_rep, region_s, clk = timed_region(args, stream, do_steps, pg, dev, clocks,
                                                                prepare=prepare)
    warm = max(0, args.warmup)
    ms_max = ms_step * steps  # median over the repeats, max over ranks
    value = world * wbytes * steps / (ms_max / 1e3) / 1e9
    peaks, peak_src = measured_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))

    # ---- per launch: each of the ten launches replayed back to back in its
    # own graph (the products on rotating weight copies), CUDA events
    names = ["rmsnorm_att", "qkv", "rope", "attention", "wo", "add_rmsnorm_ffn", "ffn",
             "silu_mul", "down", "add"]
    per_launch = {}
    for nm in names:
        reps = 2 * copies
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for j in range(reps):
                L.launch(nm, copy=j % copies, stream=stream)
        with torch.cuda.stream(stream):
            g.replay()
        stream.synchronize()
        best = None
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                a.record(stream)
                g.replay()
                b.record(stream)
            stream.synchronize()
            t = a.elapsed_time(b) / 1e3 / reps
            best = t if best is None else min(best, t)
        per_launch[nm] = best * 1e6
        del g
    phase_b = {n: sum(L.host[m][0].nbytes + L.host[m][1].nbytes for m in ms)
               for n, ms in (("qkv", ("wq", "wk", "wv")), ("wo", ("wo",)), ("ffn", ("w1", "w3")),
                             ("down", ("w2",)))}
    ph_us = sum(per_launch[n] for n in phase_b)
    ach = sum(phase_b.values()) / (ph_us * 1e-6) / 1e9
    roofline = {"kernel": "phase_kernel", "bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s",
                "frac": ach / hbm, "peak_source": peak_src,
                "traffic": ncu_traffic("phase_tinyllama1.1b_layer_q4_0",
                                       ("phase.cu", "phase_common.cuh", "mlq_device.cuh"),
                                       sum(phase_b.values()) / 4),
                "bytes_per_launch": sum(phase_b.values()) / 4, "us_per_launch": ph_us / 4,
                "method": "each of the ten launches replayed back to back in its own graph "
                          "(products on rotating weight copies), best of 3, CUDA events",
                "us_per_launch_kind": per_launch}

    # ---- end to end: x from pinned host memory, the step, x back to pinned host
    host_x = torch.empty(shape.dim, dtype=torch.float32).pin_memory()

    def e2e_body(c):
        L.x.copy_(L.x_host, non_blocking=True)
        L.step(copy=c, stream=stream)
        host_x.copy_(L.x, non_blocking=True)
    e2e_step = e2e_graph_steps(args, copies, stream, e2e_body)
    e2e_steps = min(steps, 500)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        t0 = time.perf_counter()
        for i in range(e2e_steps):
            e2e_step(i)
            stream.synchronize()
    e2e_s = max_over_ranks(pg, time.perf_counter() - t0, dev)
    e2e = {"value": world * wbytes * e2e_steps / e2e_s / 1e9, "unit": UNIT,
           "h2d_bytes_per_step": 4 * shape.dim, "d2h_bytes_per_step": 4 * shape.dim,
           "steps": e2e_steps, "how": "wall clock; per step: one graph replay holding the pinned "
                                      "H2D of x, the ten C-ABI calls and the D2H of x, then a "
                                      "stream sync"}
    assert M.mlq_last_device_error(stream) == M.MLQ_OK

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        threads = host_cores()
        op, n, el = time_oracle(shape, args.cpu_seconds, threads)
        cpu = {"value": op.weight_bytes * n / el / 1e9, "unit": UNIT, "cores": threads,
               "kind": "oracle",
               "sample": f"{n} tokens through the layer in {el:.1f} s, product rows split over "
                         f"{threads} threads"}
    if rank == 0:
        ops = sum(2 * rows * cols for _, rows, cols in shape.mats())
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
            "warmup": warm, "ms_per_step": ms_max / steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "q4_0 products: int8 dot -> int32, f32 accumulate; f32 norm, rope, attention",
            "data": "synthetic",
            "config": {"workload": shape.name, "M": 1, "pos": shape.pos,
                       "matrices": [f"{n}:{r}x{c}:q4_0" for n, r, c in shape.mats()],
                       "weight_bytes_per_step": wbytes, "kv_bytes_per_step": kvb,
                       "hbm_frac_with_kv": (wbytes + kvb) * world * steps / (ms_max / 1e3) / 1e9 / hbm,
                       "l2": f"inputs larger than L2: {copies} rotating weight copies "
                             f"({copies * wbytes / 1e6:.0f} MB vs L2 {l2 / 1e6:.0f} MB)",
                       "graphs": (("one graph of the %d timed steps per repeat" % steps) if steps in run_graphs
                                  else False if args.no_graph else "one graph per step or per cycle of steps"),
                       "path": "layer", "parallelism": f"replicas x{world} (independent decode streams)"},
            "gops": world * ops * steps / (ms_max / 1e3) / 1e9, "hbm_frac": value / world / hbm,
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": L.launches_per_step * steps * reps, "repeats": reps,
            "timed_region_s": region_s,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    return 0


def run_q4k(args, wl, world, rank, local, pg):
    """A pass of products on the other weight formats per step: Q4_K-style
    super-blocks (per input one mlq_quantize_q8k, then its mlq_matvec_q4k
    calls) or blocks of 32 / 128 with float16 scales and signed-offset 8-bit
    weights (mlq_quantize_blk, mlq_matvec_nbits), captured in a CUDA graph
    per weight copy.  value = weight bytes (quants and all scale, minimum and
    zero-point bytes) per step / step time."""
    import torch

    import numpy as np

    import block_quantized_decode_gb300 as M
    from block_quantized_decode_gb300 import inputs as I
    from block_quantized_decode_gb300.runner import NBitsRunner, Q4KRunner
    nbits = isinstance(wl, I.NBitsWorkload)
    Q4KRunner = NBitsRunner if nbits else Q4KRunner

    # The runner writes its weights once, before any product: declare them
    # static, so that under programmatic dependent launch each product
    # streams its weights before the previous launch has finished.
    os.environ.setdefault("MLQ_STATIC_WEIGHTS", "1")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    M.mlq_init()
    props = torch.cuda.get_device_properties(local)
    l2 = getattr(props, "L2_cache_size", 126 * 2 ** 20)
    probe = Q4KRunner(wl, copies=1, device=f"cuda:{local}")
    wbytes = probe.weight_bytes()
    del probe
    copies = args.copies or max(2, math.ceil(3 * l2 / wbytes))
    r = Q4KRunner(wl, copies=copies, device=f"cuda:{local}")
    # Both formats run as phases by default (mlq_q4k_phase / mlq_nbits_phase:
    # products sharing an input in one launch that quantises it); --path
    # calls keeps one quantiser launch per input and one launch per product.
    phase = args.path in ("auto", "phase")

    def one_pass(c):
        if phase:
            r.step_phase(copy=c, stream=stream)
        else:
            r.step(copy=c, stream=stream)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for c in range(copies):
            one_pass(c)
    stream.synchronize()
    prepare, do_steps, run_graphs = step_graphs(stream, one_pass, copies,
                                                len(r.phases()) if phase else r.launches_per_step,
                                                not args.no_graph)

    clocks = ClockSampler(local)
    clocks.start()
    steps, reps, ms_step, per_rep, region_s, clk = timed_region(args, stream, do_steps, pg, dev, clocks,
                                                                prepare=prepare)
    warm = max(0, args.warmup)
    ms_max = ms_step * steps  # median over the repeats, max over ranks
    value = world * wbytes * steps / (ms_max / 1e3) / 1e9
    peaks, peak_src = measured_peaks()
    hbm = float(peaks.get("hbm_gbs", FALLBACK_HBM_GBS))

    # ---- the dominant kernel: each product's launches back to back in its
    # own graph over rotating weight copies, CUDA events on the stream
    per_prod, tot_b, tot_s = {}, 0.0, 0.0
    for name, rows, cols, _ in wl.mats:
        reps = 2 * copies
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for j in range(reps):
                r.product(name, copy=j % copies, stream=stream)
        with torch.cuda.stream(stream):
            g.replay()
        stream.synchronize()
        best = None
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(stream):
                a.record(stream)
                g.replay()
                b.record(stream)
            stream.synchronize()
            t = a.elapsed_time(b) / 1e3 / reps
            best = t if best is None else min(best, t)
        del g
        nb = sum(a.nbytes for a in r.host[name] if isinstance(a, np.ndarray))
        per_prod[f"{name}:{rows}x{cols}"] = {"us": best * 1e6, "GBps": nb / best / 1e9}
        tot_b += nb
        tot_s += best
    ach = tot_b / tot_s / 1e9
    nprod = len(wl.mats)
    kname, ksrc = (("matvec_nbits_kernel", "nbits.cu") if nbits else ("matvec_q4k_kernel", "q4k.cu"))
    roofline = {"kernel": kname, "bound": "hbm", "achieved": ach, "peak": hbm,
                "unit": "GB/s", "frac": ach / hbm, "peak_source": peak_src,
                "traffic": ncu_traffic(f"{kname.replace('_kernel', '')}_{wl.name}", (ksrc, "mlq_device.cuh"),
                                       tot_b / nprod),
                "bytes_per_launch": tot_b / nprod, "us_per_launch": tot_s / nprod * 1e6,
                "method": "each product's launches back to back in its own graph over rotating "
                          "weight copies, best of 3, CUDA events on the launching stream",
                "per_product": per_prod}

    # ---- end to end: x from pinned host memory, the step, the last output back
    last = wl.mats[-1][0]
    host_y = torch.empty(r.y[last].numel(), dtype=torch.float32).pin_memory()

    def e2e_body(c):
        r.x.copy_(r.x_pinned, non_blocking=True)
        one_pass(c)
        host_y.copy_(r.y[last], non_blocking=True)
    e2e_step = e2e_graph_steps(args, copies, stream, e2e_body)
    e2e_steps = min(steps, 500)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        t0 = time.perf_counter()
        for i in range(e2e_steps):
            e2e_step(i)
            stream.synchronize()
    e2e_s = max_over_ranks(pg, time.perf_counter() - t0, dev)
    e2e = {"value": world * wbytes * e2e_steps / e2e_s / 1e9, "unit": UNIT,
           "h2d_bytes_per_step": r.x.numel() * 4, "d2h_bytes_per_step": host_y.numel() * 4,
           "steps": e2e_steps, "how": "wall clock; per step: one graph replay holding the pinned "
                                      "H2D of x, the C-ABI calls and the D2H of the last product's "
                                      "output, then a stream sync"}
    assert M.mlq_last_device_error(stream) == M.MLQ_OK

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        threads = host_cores()
        op, n, el = time_oracle(wl, args.cpu_seconds, threads)
        cpu = {"value": op.weight_bytes * n / el / 1e9, "unit": UNIT, "cores": threads,
               "kind": "oracle",
               "sample": f"{n} passes of {wl.name} in {el:.1f} s, product rows split over "
                         f"{threads} threads"}
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": steps,
            "warmup": warm, "ms_per_step": ms_max / steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": (f"{'u4' if wl.bits == 4 else 's8 (B-128)'} x s8 dot -> int32 per block of "
                      f"{wl.blk}, {'f16' if wl.f16 else 'f32'} scales, f32 accumulate" if nbits else
                      "q4_k products: u4 x s8 dot -> int32, sub-block scales folded in int32, "
                      "f32 per super-block"),
            "data": "synthetic",
            "config": {"workload": wl.name, "M": 1,
                       "matrices": [f"{n}:{rw}x{c}:" + (f"{'int4' if wl.bits == 4 else 'int8'}_blk{wl.blk}"
                                                        if nbits else "q4_k") for n, rw, c, _ in wl.mats],
                       "weight_bytes_per_step": wbytes,
                       "l2": f"inputs larger than L2: {copies} rotating weight copies "
                             f"({copies * wbytes / 1e6:.0f} MB vs L2 {l2 / 1e6:.0f} MB)",
                       "graphs": (("one graph of the %d timed steps per repeat" % steps) if steps in run_graphs
                                  else False if args.no_graph else "one graph per step or per cycle of steps"),
                       "path": "phase" if phase else "calls", "static_weights": os.environ.get("MLQ_STATIC_WEIGHTS") == "1",
                       "parallelism": f"replicas x{world} (independent decode streams)"},
            "gops": world * r.ops() * steps / (ms_max / 1e3) / 1e9, "hbm_frac": value / world / hbm,
            "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": (len(r.phases()) if phase else r.launches_per_step) * steps * reps,
            "repeats": reps, "timed_region_s": region_s,
            "clocks": clk,
        }
        print(json.dumps(line), flush=True)
    return 0


def main():
    args = parse_args()
    from block_quantized_decode_gb300 import inputs as I
    known = {**I.WORKLOADS, **I.LAYERS, **I.Q4K_WORKLOADS, **I.NBITS_WORKLOADS}
    if args.workload not in known:
        raise SystemExit(f"unknown workload {args.workload}; choose from {sorted(known)}")
    wl = known[args.workload]()
    world, rank, local, pg = dist_setup(args)
    try:
        if args.impl == "reference":
            return run_reference(args, wl, world, rank)
        if isinstance(wl, I.LayerShape):
            return run_layer(args, wl, world, rank, local, pg)
        if isinstance(wl, (I.Q4KWorkload, I.NBitsWorkload)):
            return run_q4k(args, wl, world, rank, local, pg)
        return run_ours(args, wl, world, rank, local, pg)
    finally:
        if pg is not None:
            pg.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())
