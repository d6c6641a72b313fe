"""mlq_decode_chain (a whole decode step in one cooperative launch) against
the oracle: every phase's in-kernel quantisation bit-exact (via xq_out /
xd_out), every product within tolerance, per step on the GPU's own inputs;
the workspace is left zeroed; results are deterministic; graph replay; the
bounded waits report MLQ_E_TIMEOUT and leave the workspace reusable."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from block_quantized_decode_gb300 import inputs as I  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_quantized_decode_gb300 import build as B
    B.build()
    import block_quantized_decode_gb300 as M
    M.mlq_init()
    torch.cuda.set_device(0)
    yield M
    assert M.mlq_last_device_error() == M.MLQ_OK


from tests.test_gpu_configs import run_and_check  # noqa: E402
from block_quantized_decode_gb300.runner import WorkloadRunner  # noqa: E402


def test_chain_tiny():
    run_and_check(I.tiny_q4(), chain=True)


def test_chain_tinyllama_layer():
    run_and_check(I.tinyllama_layer(), chain=True)


def test_chain_tinyllama_layer_graph():
    run_and_check(I.tinyllama_layer(), chain=True, graph=True)


def test_chain_llama7b_ffn_q4():
    run_and_check(I.llama7b_ffn(I.Q4_0), chain=True)


def test_chain_llama7b_ffn_q8_lm_head():
    run_and_check(I.llama7b_ffn_q8_lm_head(), chain=True)


def test_chain_ragged_rows_and_widths():
    """Phases whose row counts do not divide by the CTA count, a product
    with fewer rows than CTAs, two products in one phase, a chained phase,
    widths 128 to 1024."""
    wl = I.Workload("ragged", 1, [
        I.Matvec("a", I.Q4_0, 1001, 128, "x"),
        I.Matvec("b", I.Q4_0, 7, 128, "x"),
        I.Matvec("c", I.Q4_0, 384, 1024, "x"),
        I.Matvec("e", I.Q4_0, 1000, 384, "c"),
        I.Matvec("d", I.Q4_0, 2049, 384, "x"),
    ])
    run_and_check(wl, chain=True)


def test_chain_ragged_q8():
    wl = I.Workload("ragged_q8", 1, [
        I.Matvec("a", I.Q8_0, 999, 256, "x"),
        I.Matvec("b", I.Q8_0, 640, 256, "x"),
        I.Matvec("c", I.Q8_0, 155, 640, "b"),
    ])
    run_and_check(wl, chain=True)


def test_chain_deterministic_and_matches_calls(lib):
    M = lib
    r = WorkloadRunner(I.tinyllama_layer(), copies=1)
    r.step_chain()
    torch.cuda.synchronize()
    first = [m.y.clone() for m in r.mats]
    r.step_chain()
    torch.cuda.synchronize()
    for a, m in zip(first, r.mats):
        assert torch.equal(a, m.y), "chain results differ between two identical calls"
    assert M.mlq_last_device_error() == M.MLQ_OK


def test_chain_timeout_path(lib):
    M = lib
    r = WorkloadRunner(I.tinyllama_layer(), copies=1)
    r.step_chain()
    torch.cuda.synchronize()
    assert M.mlq_last_device_error() == M.MLQ_OK
    try:
        M.mlq_debug_set_wait_limit_ns(0)
        r.step_chain()
        assert M.mlq_last_device_error() == M.MLQ_E_TIMEOUT
    finally:
        M.mlq_debug_set_wait_limit_ns(10 ** 9)
    assert int(r.chain_ws.abs().sum()) == 0, "workspace not zero after a timed-out call"
    for m in r.mats:
        m.y.fill_(float("nan"))
    r.step_chain()
    torch.cuda.synchronize()
    assert M.mlq_last_device_error() == M.MLQ_OK
    assert all(torch.isfinite(m.y).all() for m in r.mats)
