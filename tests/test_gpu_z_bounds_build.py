"""The bounds-checking build (MLQ_CHECK_BOUNDS=1: libmlq_checked.so, every
kernel index check records MLQ_E_BOUNDS and skips the access) passes the
core parity suites: the phase, configs, chain and M = 1 / small-M parity
files, run in a child process against that library.  Any index outside its
buffer would show up as MLQ_E_BOUNDS from mlq_last_device_error, which
every one of those tests asserts to be MLQ_OK."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.skipif(os.environ.get("MLQ_CHECK_BOUNDS") == "1", reason="already the checking build")
def test_suites_pass_in_the_bounds_checking_build():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    env = dict(os.environ, MLQ_CHECK_BOUNDS="1", PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "tests/test_gpu_parity.py", "tests/test_gpu_phase.py", "tests/test_gpu_configs.py",
                        "tests/test_gpu_chain.py", "tests/test_gpu_fused.py"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
    assert os.path.exists(os.path.join(ROOT, "block_quantized_decode_gb300", "libmlq_checked.so"))
