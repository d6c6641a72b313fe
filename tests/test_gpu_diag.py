"""MLQ_DIAG=1: each entry point reports, once per distinct line, which
kernel ran and how it was laid out.  A child process runs the dispatch
branches -- the shared-memory phase kernel, the ring phase kernel, an M = 1
call on each route, the small-M ring and cluster-MMA kernels -- and the test
reads the lines from its stderr."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_CHILD = r"""
import sys
sys.path.insert(0, sys.argv[1])
import torch
import block_quantized_decode_gb300 as M
from block_quantized_decode_gb300 import inputs as I
from block_quantized_decode_gb300.runner import WorkloadRunner
torch.cuda.set_device(0)
M.mlq_init()
r = WorkloadRunner(I.tinyllama_layer())
r.step_phase(); r.step_phase()          # phase kernel, twice: one line each
r.step()                                # quantize + M = 1 calls (small products)
big = WorkloadRunner(I.Workload("up", 1, [I.Matvec("up", I.Q4_0, 11008, 4096, "x")]))
big.step()                              # an M = 1 call of 28 MB: the phase route
big.step_phase()                        # a float-input ring phase
WorkloadRunner(I.small_m(4)).step()     # small-M ring kernel
WorkloadRunner(I.small_m(16)).step()    # cluster MMA kernel
torch.cuda.synchronize()
assert M.mlq_last_device_error() == M.MLQ_OK
"""


def test_diag_lines_for_each_dispatch_branch():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, MLQ_DIAG="1", PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", _CHILD, ROOT], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    lines = [l for l in r.stderr.splitlines() if l.startswith("mlq diag: ")]
    assert len(lines) == len(set(lines)), "a line was printed twice"

    def has(*parts):
        return any(all(p in l for p in parts) for l in lines)

    assert has("mlq_decode_phase", "phase_kernel<", "phase: products=3", "grid=", "smem=")
    assert has("mlq_decode_phase", "phase_ring_kernel<", "ring: products=1 rows=11008 K=4096",
               "rows/stage=", "slots=")
    assert has("mlq_matvec_q4 rows=11008 cols=4096", "route=phase")
    assert has("mlq_matvec_q4 rows=256 cols=2048", "route=ldg", "matvec_m1_kernel<")
    assert has("mlq_quantize_q8", "quantize_q8_kernel")
    assert has("mlq_gemm_q4_small_m M=4", "gemm_q4_ring_kernel<", "ring: M=4")
    assert has("mlq_gemm_q4_small_m M=16", "gemm_q4_mma_cluster_kernel", "mma_cluster: M=16", "cluster=")


def test_diag_off_by_default():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = {k: v for k, v in os.environ.items() if k != "MLQ_DIAG"}
    env["PYTHONPATH"] = ROOT
    r = subprocess.run([sys.executable, "-c", _CHILD, ROOT], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    assert "mlq diag:" not in r.stderr
