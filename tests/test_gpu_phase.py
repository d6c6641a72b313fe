"""mlq_decode_phase (one launch per decode phase; a product whose output
feeds a later phase writes it in Q8_0 itself) against the oracle, per step
on the GPU's own inputs: every quantised activation -- written by the
phase that reads a float input, or by the product that produced it -- must
equal the oracle's quantisation of the float vector the GPU stored, byte
for byte; every product within tolerance of the oracle on those bytes.
Shapes cover the shared-memory phase kernel (one to eight K-chunks per
warp, Q4_0 and Q8_0, 32-row output blocks split between CTAs) and the
multi-launch path taken when a CTA's weights do not fit on chip."""
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
from tests import parity as PT  # noqa: E402


def test_phase_tiny():
    run_and_check(I.tiny_q4(), phase=True)


@pytest.mark.parametrize("static", [True, False], ids=["static_weights", "plain"])
def test_phase_tinyllama_layer(static):
    r = run_and_check(I.tinyllama_layer(), phase=True, static_weights=static)
    # the chained inputs really were produced by the products
    calls = r.phase_calls(0, static)
    assert sum(1 for c in calls if c.inp.x is None) == 3


def test_phase_tinyllama_layer_graph():
    run_and_check(I.tinyllama_layer(), phase=True, graph=True)


def test_phase_llama7b_ffn_q4():      # CTA slices too large: multi-launch path
    run_and_check(I.llama7b_ffn(I.Q4_0), phase=True)


def test_phase_llama7b_ffn_q8_lm_head():
    run_and_check(I.llama7b_ffn_q8_lm_head(), phase=True)


def test_phase_chunks_q4():
    # K = 128 .. 16384: 1, 2, 4 and 8 chunks per warp, chunk tails of 38, 43
    # and 44 blocks
    wl = I.Workload("chunks_q4", 1, [
        I.Matvec("a", I.Q4_0, 320, 4096, "x"),
        I.Matvec("b", I.Q4_0, 1024, 320, "a"),
        I.Matvec("c", I.Q4_0, 640, 1024, "b"),
        I.Matvec("d", I.Q4_0, 5632, 640, "c"),
        I.Matvec("e", I.Q4_0, 160, 5632, "d"),
        I.Matvec("f", I.Q4_0, 96, 11008, "x"),
        I.Matvec("g", I.Q4_0, 1000, 16384, "x"),
        I.Matvec("h", I.Q4_0, 608, 9600, "x"),
    ])
    run_and_check(wl, phase=True)


def test_phase_q8_chain():
    wl = I.Workload("q8_chain", 1, [
        I.Matvec("a", I.Q8_0, 768, 256, "x"),
        I.Matvec("b", I.Q8_0, 300, 256, "x"),
        I.Matvec("c", I.Q8_0, 2048, 768, "a"),
        I.Matvec("d", I.Q8_0, 200, 2048, "c"),
        I.Matvec("e", I.Q8_0, 64, 5632, "x"),
    ])
    run_and_check(wl, phase=True)


def test_phase_ragged():
    # rows not multiples of 32 (no producer-side quantisation there), empty
    # products, K with nb % 4 != 0 (multi-launch path), one-block rows
    wl = I.Workload("ragged_phase", 1, [
        I.Matvec("a", I.Q4_0, 1001, 96, "x"),
        I.Matvec("b", I.Q4_0, 7, 96, "x"),
        I.Matvec("c", I.Q4_0, 0, 96, "x"),
        I.Matvec("d", I.Q4_0, 64, 4128, "x"),
        I.Matvec("e", I.Q4_0, 33, 64, "d"),
        I.Matvec("f", I.Q4_0, 2049, 32, "x"),
        I.Matvec("g", I.Q4_0, 32, 128, "x"),
        I.Matvec("h", I.Q4_0, 0, 128, "x"),
        I.Matvec("i", I.Q4_0, 96, 32, "g"),
    ])
    run_and_check(wl, phase=True)


def test_phase_one_block_output_fp32_input():
    # 32 output rows over 32 CTAs: every CTA but the last gets no rows, yet
    # CTA 0 still writes the quantised input
    wl = I.Workload("one_block", 1, [
        I.Matvec("a", I.Q4_0, 32, 2048, "x"),
        I.Matvec("b", I.Q4_0, 64, 32, "a"),
    ])
    run_and_check(wl, phase=True)


def test_phase_direct_api(lib):
    """The entry point called directly: float input with xq_out, a product
    quantising its output next to one that does not, then a second call
    from those Q8_0 bytes; repeated twice (buffers reused)."""
    M = lib
    K, R1, R2 = 2048, 256, 512
    x = I.activations(1, K, seed=99).reshape(-1)
    w1q, w1d = I.weights(I.Q4_0, R1, K, seed=1)
    w2q, w2d = I.weights(I.Q4_0, 96, K, seed=2)
    w3q, w3d = I.weights(I.Q4_0, R2, R1, seed=3)
    dev = PT.DEV
    W1 = PT.weights_dev(I.Q4_0, w1q, w1d, R1, K)
    W2 = PT.weights_dev(I.Q4_0, w2q, w2d, 96, K)
    W3 = PT.weights_dev(I.Q4_0, w3q, w3d, R2, R1)
    xg = PT.to_dev(x)
    xq = torch.empty(K, dtype=torch.int8, device=dev)
    xd = torch.empty(K // 32, dtype=torch.float32, device=dev)
    y1 = torch.empty(R1, device=dev)
    y2 = torch.empty(96, device=dev)
    y1q = torch.empty(R1, dtype=torch.int8, device=dev)
    y1d = torch.empty(R1 // 32, dtype=torch.float32, device=dev)
    y3 = torch.empty(R2, device=dev)
    for _ in range(2):
        for t in (y1, y2, y3, y1d, xd):
            t.fill_(float("nan"))
        y1q.fill_(0)
        M.mlq_decode_phase(K, [M.PhaseProduct(W1, y1, y1q, y1d), M.PhaseProduct(W2, y2)],
                           x=xg, xq_out=xq, xd_out=xd, flags=M.MLQ_F_STATIC_WEIGHTS)
        M.mlq_decode_phase(R1, [M.PhaseProduct(W3, y3)], xq=y1q, xd=y1d,
                           flags=M.MLQ_F_STATIC_WEIGHTS)
        torch.cuda.synchronize()
        assert M.mlq_last_device_error() == M.MLQ_OK
        oq, od = oracle.quantize_q8(x.reshape(1, K))
        PT.assert_quant_equal(xq.cpu().numpy(), xd.cpu().numpy(), oq, od, "x")
        PT.check_matvec(I.Q4_0, w1q, w1d, R1, K, oq[0], od[0], 0, R1, y_gpu=y1.cpu().numpy(), what="y1")
        PT.check_matvec(I.Q4_0, w2q, w2d, 96, K, oq[0], od[0], 0, 96, y_gpu=y2.cpu().numpy(), what="y2")
        o1q, o1d = oracle.quantize_q8(y1.cpu().numpy().reshape(1, R1))
        PT.assert_quant_equal(y1q.cpu().numpy(), y1d.cpu().numpy(), o1q, o1d, "y1 quantised")
        PT.check_matvec(I.Q4_0, w3q, w3d, R2, R1, o1q[0], o1d[0], 0, R2, y_gpu=y3.cpu().numpy(),
                        what="y3")


def test_phase_timeout_reports_status(lib):
    """A bounded wait that gives up (limit 0) is reported, not hung on."""
    M = lib
    K, R = 2048, 512
    wq, wd = I.weights(I.Q4_0, R, K, seed=5)
    W = PT.weights_dev(I.Q4_0, wq, wd, R, K)
    x = PT.to_dev(I.activations(1, K, seed=6).reshape(-1))
    y = torch.empty(R, device=PT.DEV)
    M.mlq_debug_set_wait_limit_ns(0)
    try:
        M.mlq_decode_phase(K, [M.PhaseProduct(W, y)], x=x, flags=M.MLQ_F_STATIC_WEIGHTS)
        assert M.mlq_last_device_error() == M.MLQ_E_TIMEOUT
    finally:
        M.mlq_debug_set_wait_limit_ns(1_000_000_000)
    M.mlq_decode_phase(K, [M.PhaseProduct(W, y)], x=x, flags=M.MLQ_F_STATIC_WEIGHTS)
    assert M.mlq_last_device_error() == M.MLQ_OK
