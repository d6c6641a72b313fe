"""mlq_matvec_fused (quantise + grouped products, one launch per phase,
chained under programmatic dependent launch) against the oracle, per step
on the GPU's own inputs: quantisation bit-exact (xq_out / xd_out), every
product within tolerance."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

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


def test_fused_tiny():
    run_and_check(I.tiny_q4(), fused=True)


@pytest.mark.parametrize("static", [True, False], ids=["static_weights", "plain"])
def test_fused_tinyllama_layer(static):
    run_and_check(I.tinyllama_layer(), fused=True, static_weights=static)


def test_fused_tinyllama_layer_graph():
    run_and_check(I.tinyllama_layer(), fused=True, graph=True)


def test_fused_llama7b_ffn_q4():
    run_and_check(I.llama7b_ffn(I.Q4_0), fused=True)


def test_fused_llama7b_ffn_q8_lm_head():
    run_and_check(I.llama7b_ffn_q8_lm_head(), fused=True)


def test_fused_ragged_plain():
    wl = I.Workload("ragged_plain", 1, [
        I.Matvec("a", I.Q4_0, 1001, 128, "x"),
        I.Matvec("b", I.Q4_0, 5, 128, "x"),
        I.Matvec("c", I.Q4_0, 640, 1024, "x"),
    ])
    run_and_check(wl, fused=True, static_weights=False)


def test_fused_ragged():
    wl = I.Workload("ragged", 1, [
        I.Matvec("a", I.Q4_0, 1001, 96, "x"),
        I.Matvec("b", I.Q4_0, 7, 96, "x"),
        I.Matvec("c", I.Q4_0, 0, 96, "x"),
        I.Matvec("d", I.Q4_0, 64, 4128, "x"),
        I.Matvec("e", I.Q4_0, 33, 64, "d"),
        I.Matvec("f", I.Q4_0, 2049, 32, "x"),
    ])
    run_and_check(wl, fused=True)


def test_fused_ragged_q8():
    wl = I.Workload("ragged_q8", 1, [
        I.Matvec("a", I.Q8_0, 999, 160, "x"),
        I.Matvec("b", I.Q8_0, 480, 160, "x"),
        I.Matvec("c", I.Q8_0, 155, 480, "b"),
        I.Matvec("d", I.Q8_0, 3, 65536, "x"),
    ])
    run_and_check(wl, fused=True)
