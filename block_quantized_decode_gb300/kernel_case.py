"""Run one libmlq entry point on one shape, for timing and for profilers.

    python -m block_quantized_decode_gb300.kernel_case --op matvec_q4 --rows 4096 --cols 11008

Weights are random device bytes, replicated over enough copies that the
copies together exceed 3x L2; the call is captured ITERS times in one CUDA
graph (one copy per launch) and replayed.  Prints the mean time per launch
from CUDA events and the weight bytes per launch over that time.
"""
from __future__ import annotations

import argparse
import json
import math

import torch

from . import binding as B


def main():
    p = argparse.ArgumentParser()
    p.add_argument("--op", default="matvec_q4",
                   choices=["matvec_q4", "matvec_q8", "gemm_q4", "quantize", "fused", "phase", "chain",
                            "matvec_q4k", "matvec_nbits"])
    p.add_argument("--workload", default="tinyllama_layer",
                   help="for --op fused / phase / chain: the workload whose phases run as "
                        "mlq_matvec_fused / mlq_decode_phase calls, or as one "
                        "mlq_decode_chain call")
    p.add_argument("--rows", type=int, default=4096)
    p.add_argument("--cols", type=int, default=11008)
    p.add_argument("--m", type=int, default=1)
    p.add_argument("--iters", type=int, default=50)
    p.add_argument("--reps", type=int, default=5)
    p.add_argument("--copies", type=int, default=0)
    p.add_argument("--no-graph", action="store_true")
    p.add_argument("--bits", type=int, default=8, help="for --op matvec_nbits: 4 or 8")
    p.add_argument("--blk", type=int, default=32, help="for --op matvec_nbits: 32 or 128")
    p.add_argument("--f16", action="store_true", help="for --op matvec_nbits: float16 scales")
    p.add_argument("--zp", action="store_true", help="for --op matvec_nbits: 8-bit zero points")
    a = p.parse_args()

    dev = torch.device("cuda:0")
    torch.cuda.set_device(0)
    B.mlq_init()
    if a.op in ("fused", "phase", "chain"):
        return fused_case(a)
    if a.op in ("matvec_q4k", "matvec_nbits"):
        return q4k_case(a)
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    rows, cols, m = a.rows, a.cols, a.m
    nb = cols // 32
    q8 = a.op == "matvec_q8"
    qbytes = rows * cols if q8 else rows * cols // 2
    wbytes = qbytes + rows * nb * 4
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    copies = a.copies or max(1, math.ceil(3 * l2 / max(wbytes, 1)))
    copies = min(copies, a.iters)
    Ws = []
    if a.op != "quantize":
        for _ in range(copies):
            q = torch.randint(-128, 128, (qbytes,), dtype=torch.int8, device=dev, generator=g)
            if q8:
                q.clamp_(-127, 127)
            d = torch.rand((rows * nb,), device=dev, generator=g) * 9e-3 + 1e-3
            Ws.append(B.QTensor(q, d, rows, cols, B.MLQ_Q8_0 if q8 else B.MLQ_Q4_0))
    x = torch.randn((m, cols), device=dev, generator=g)
    xa = B.QAct(torch.empty((m, cols), dtype=torch.int8, device=dev),
                torch.empty((m, nb), dtype=torch.float32, device=dev), cols, m)
    B.mlq_quantize_q8(xa, x, cols)
    y = torch.empty((m, rows), dtype=torch.float32, device=dev)

    def call(i):
        if a.op == "quantize":
            B.mlq_quantize_q8(xa, x, cols)
        elif a.op == "gemm_q4":
            B.mlq_gemm_q4_small_m(y, rows, Ws[i % copies], xa, m, 0, rows)
        elif q8:
            B.mlq_matvec_q8(y, Ws[i % copies], xa, 0, rows)
        else:
            B.mlq_matvec_q4(y, Ws[i % copies], xa, 0, rows)

    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for i in range(copies):
            call(i)
    s.synchronize()
    graph = None
    if not a.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            for i in range(a.iters):
                call(i)
    times = []
    for _ in range(a.reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            if graph is not None:
                graph.replay()
            else:
                for i in range(a.iters):
                    call(i)
            e1.record(s)
        s.synchronize()
        times.append(e0.elapsed_time(e1) / a.iters * 1e3)
    assert B.mlq_last_device_error(s) == B.MLQ_OK
    us = min(times)
    moved = wbytes if a.op != "quantize" else m * cols * (4 + 1) + m * nb * 4
    print(json.dumps({"op": a.op, "rows": rows, "cols": cols, "m": m, "copies": copies,
                      "us_per_launch": us, "us_all": times, "bytes_per_launch": moved,
                      "GBps": moved / (us * 1e-6) / 1e9,
                      "gops": 2.0 * m * rows * cols / (us * 1e-6) / 1e9 if a.op != "quantize" else 0.0}))


def q4k_case(a):
    """Back-to-back mlq_matvec_q4k launches over rotating weight copies."""
    from . import inputs as I
    import numpy as np
    rows, cols = a.rows, a.cols
    dev = torch.device("cuda:0")
    tt = lambda t: torch.from_numpy(np.ascontiguousarray(t)).to(dev)
    x = torch.from_numpy(I.activations(1, cols, seed=1)[0]).to(dev)
    if a.op == "matvec_q4k":
        host = I.q4k_weights(rows, cols, seed=0)
        make = lambda: B.Q4KTensor(*(tt(t) for t in host), rows, cols)
        act = B.Q8KAct(torch.empty(cols, dtype=torch.int8, device=dev),
                       torch.empty(cols // 256, dtype=torch.float32, device=dev),
                       torch.empty(cols // 32, dtype=torch.int32, device=dev), cols)
        B.mlq_quantize_q8k(act, x, cols)
        mv = B.mlq_matvec_q4k
    else:
        q, sc, zp = I.nbits_weights(rows, cols, a.bits, a.blk, a.f16, a.zp, seed=0)
        host = (q, sc) + (() if zp is None else (zp,))
        scp, zpp = I.pad_rows(sc), (None if zp is None else I.pad_rows(zp))
        make = lambda: B.NBitsTensor(tt(q), tt(scp.view(np.uint16) if a.f16 else scp),
                                     None if zpp is None else tt(zpp), rows, cols, a.bits, a.blk,
                                     1 if a.f16 else 0, scp.shape[1], 0 if zpp is None else zpp.shape[1])
        act = B.BlkAct(torch.empty(cols, dtype=torch.int8, device=dev),
                       torch.empty(cols // a.blk, dtype=torch.float32, device=dev),
                       torch.empty(cols // a.blk, dtype=torch.int32, device=dev), cols, a.blk)
        B.mlq_quantize_blk(act, x, cols)
        mv = B.mlq_matvec_nbits
    wbytes = sum(t.nbytes for t in host)
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    copies = a.copies or max(1, math.ceil(3 * l2 / wbytes))
    copies = min(copies, a.iters)
    Ws = [make() for _ in range(copies)]
    y = torch.empty(rows, dtype=torch.float32, device=dev)
    s_ = torch.cuda.Stream()
    with torch.cuda.stream(s_):
        for i in range(copies):
            mv(y, Ws[i], act, 0, rows)
    s_.synchronize()
    graph = None
    if not a.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s_):
            for i in range(a.iters):
                mv(y, Ws[i % copies], act, 0, rows)
    times = []
    for _ in range(a.reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s_):
            e0.record(s_)
            if graph is not None:
                graph.replay()
            else:
                for i in range(a.iters):
                    mv(y, Ws[i % copies], act, 0, rows)
            e1.record(s_)
        s_.synchronize()
        times.append(e0.elapsed_time(e1) / a.iters * 1e3)
    assert B.mlq_last_device_error(s_) == B.MLQ_OK
    us = min(times)
    print(json.dumps({"op": a.op, "rows": rows, "cols": cols, "copies": copies, "us_per_launch": us,
                      "us_all": times, "bytes_per_launch": wbytes, "GBps": wbytes / (us * 1e-6) / 1e9,
                      "gops": 2.0 * rows * cols / (us * 1e-6) / 1e9}))


def fused_case(a):
    """One pass of a workload as mlq_matvec_fused (or mlq_decode_phase)
    launches, one per phase, or as one mlq_decode_chain launch."""
    from . import inputs as I
    from .runner import WorkloadRunner
    wl = I.WORKLOADS[a.workload]()
    copies = a.copies or 3
    r = WorkloadRunner(wl, copies=copies)
    step = {"fused": r.step_fused, "phase": r.step_phase, "chain": r.step_chain}[a.op]
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for c in range(copies):
            step(copy=c)
    s.synchronize()
    graph = None
    if not a.no_graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            for i in range(a.iters):
                step(copy=i % copies)
    times = []
    for _ in range(a.reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(s):
            e0.record(s)
            if graph is not None:
                graph.replay()
            else:
                for i in range(a.iters):
                    step(copy=i % copies)
            e1.record(s)
        s.synchronize()
        times.append(e0.elapsed_time(e1) / a.iters * 1e3)
    assert B.mlq_last_device_error(s) == B.MLQ_OK
    us = min(times)
    print(json.dumps({"op": a.op, "workload": wl.name, "copies": copies, "us_per_step": us,
                      "bytes_per_step": r.weight_bytes(), "GBps": r.weight_bytes() / (us * 1e-6) / 1e9}))


if __name__ == "__main__":
    main()
