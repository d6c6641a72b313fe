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


@pytest.fixture(params=["stream", "stream_float_inputs", "legacy"], autouse=True)
def chain_kernel(request, monkeypatch):
    """Each chain test runs on the streaming kernel (the default), on the
    streaming kernel with every phase quantising its float input itself
    (no in-chain Q8_0 hand-off), and on the legacy kernel."""
    if request.param == "stream_float_inputs":
        monkeypatch.setenv("MLQ_CHAIN_QIN", "0")
    elif request.param == "legacy":
        monkeypatch.setenv("MLQ_CHAIN_KERNEL", "legacy")
    yield request.param


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


def test_chain_handoffs_and_wide_rows():
    """In-chain Q8_0 hand-offs over several phases in a row (outputs of
    whole 32-row blocks feeding the next phase), a phase with a product whose
    rows are not whole blocks (the phase after it quantises its float input
    itself), the widest rows the streaming kernel holds (K = 16384) and a
    narrow one (K = 128)."""
    wl = I.Workload("handoffs", 1, [
        I.Matvec("a", I.Q4_0, 512, 16384, "x"),
        I.Matvec("b", I.Q4_0, 16384, 512, "a"),
        I.Matvec("c", I.Q4_0, 128, 16384, "b"),
        I.Matvec("d", I.Q4_0, 4096, 128, "c"),
        I.Matvec("e", I.Q4_0, 77, 128, "c"),
        I.Matvec("f", I.Q4_0, 64, 4096, "d"),
    ])
    run_and_check(wl, chain=True)


def test_chain_widest_stream_rows():
    """K = 20480: sixteen K-chunks of 40 blocks, one row per stage."""
    wl = I.Workload("wide", 1, [
        I.Matvec("a", I.Q8_0, 300, 20480, "x"),
        I.Matvec("b", I.Q8_0, 640, 20480, "x"),
    ])
    run_and_check(wl, chain=True)


def test_chain_wider_than_stream_falls_back():
    """K = 40960 is wider than the streaming kernel's warps hold in
    registers: the call still runs (on the legacy kernel) and is correct."""
    wl = I.Workload("wider", 1, [I.Matvec("a", I.Q8_0, 300, 40960, "x")])
    run_and_check(wl, chain=True)


def test_chain_deterministic_and_matches_calls(lib):
    M = lib
    r = WorkloadRunner(I.tinyllama_layer(), copies=1, canary=True)
    r.step_chain()
    torch.cuda.synchronize()
    r.check_canaries()
    first = [m.y.clone() for m in r.mats]
    r.step_chain()
    torch.cuda.synchronize()
    r.check_canaries()
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
