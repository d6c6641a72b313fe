"""The M = 1 products run as one-product decode phases (phase.cu /
phase_ring.cu) where those kernels take the shape, else on one of two
kernels of their own (register-pipelined loads, and a bulk-copy ring); the
dispatcher picks per shape.  Re-run the per-block sum and product parity
tests with each choice forced, in child processes (the choice is read once
per process from MLQ_MATVEC_KERNEL); the small-M, fused and phase kernels
likewise."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.skipif(os.environ.get("MLQ_MATVEC_KERNEL") is not None,
                    reason="already inside a forced-kernel run")
@pytest.mark.parametrize("kernel", ["ldg", "tma", "phase"])
def test_parity_with_forced_kernel(kernel):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, MLQ_MATVEC_KERNEL=kernel, PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "tests/test_gpu_parity.py", "-k", "sumi or matvec or timeout"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]


@pytest.mark.skipif(os.environ.get("MLQ_GEMM_KERNEL") is not None,
                    reason="already inside a forced-kernel run")
@pytest.mark.parametrize("kernel", ["dp4a", "mma", "mma_ldg", "umma", "ring"])
def test_small_m_parity_with_forced_kernel(kernel):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, MLQ_GEMM_KERNEL=kernel, PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "tests/test_gpu_parity.py", "-k", "gemm"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]


@pytest.mark.skipif(os.environ.get("MLQ_MMA_I8") is not None,
                    reason="already inside a forced-form run")
@pytest.mark.parametrize("form", ["0", "1"])
def test_small_m_parity_with_forced_activation_form(form):
    """The cluster MMA kernel holds its activations as fp16 fragments or as
    int8 words converted per stage (per shape); each form forced on every
    small-M case (MLQ_MMA_I8, read once per process)."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, MLQ_MMA_I8=form, PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "tests/test_gpu_parity.py", "-k", "gemm"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]


@pytest.mark.skipif(os.environ.get("MLQ_FUSED_KERNEL") is not None,
                    reason="already inside a forced-kernel run")
@pytest.mark.parametrize("kernel", ["ldg", "phase"])
def test_fused_parity_with_forced_kernel(kernel):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, MLQ_FUSED_KERNEL=kernel, PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "tests/test_gpu_fused.py"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]


@pytest.mark.skipif(os.environ.get("MLQ_PHASE_WARPS") is not None,
                    reason="already inside a forced-width run")
def test_phase_parity_with_narrow_ctas():
    """The phase kernel with 8-warp CTAs (four per SM) instead of 16."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, MLQ_PHASE_WARPS="8", PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "tests/test_gpu_phase.py"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]


@pytest.mark.skipif(os.environ.get("MLQ_PHASE_KERNEL") is not None,
                    reason="already inside a forced-kernel run")
def test_phase_parity_with_ring_kernel():
    """Every phase through the ring kernel (weights streamed through shared
    memory stages), including the shapes the shared-memory kernel takes."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, MLQ_PHASE_KERNEL="ring", PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "tests/test_gpu_phase.py", "tests/test_gpu_fused.py"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]


@pytest.mark.skipif(os.environ.get("MLQ_RING_INPUT") is not None,
                    reason="already inside a forced-input run")
def test_phase_parity_with_ring_input_loads():
    """The ring kernel reads a Q8_0 input by bulk copies; the consumers'
    16-byte loads (the path for an unaligned input) forced on every phase,
    every phase through the ring kernel."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, MLQ_RING_INPUT="ldg", MLQ_PHASE_KERNEL="ring", PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "tests/test_gpu_phase.py", "tests/test_gpu_configs.py"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]


@pytest.mark.skipif(os.environ.get("MLQ_RING_GRID") is not None,
                    reason="already inside a forced-variant run")
def test_phase_parity_with_ring_variants():
    """The ring kernel's measured choices changed together: another grid (and
    so another row split), another L2-hint fraction and stage count (also for
    Q8_0), and the producer waiting for the input to land.  Every phase
    through the ring kernel."""
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, MLQ_PHASE_KERNEL="ring", MLQ_RING_GRID="100", MLQ_RING_HINT_PARTNER="3",
               MLQ_RING_HINT_STAGES="3", MLQ_RING_ISSUE_RELEASE="0", PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "tests/test_gpu_phase.py", "tests/test_gpu_configs.py"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
