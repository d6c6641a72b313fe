"""Every workload at its full size, in the launch configuration the bench
times (the same C-ABI calls issued by WorkloadRunner), against the oracle.

Chained stacks are checked per step on the GPU's own inputs: the oracle
quantises the float vector the GPU fed to each quantize (bytes and scales
must match exactly), then recomputes the product from those bytes, so an
upstream difference within tolerance can never be counted downstream.
Products are compared on sampled row windows (first, last and random rows)
where the oracle would take too long for every row.
"""
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


from tests import parity as PT  # noqa: E402
from block_quantized_decode_gb300.runner import WorkloadRunner  # noqa: E402


def run_and_check(wl, full_rows_limit=300_000_000, graph=False, chain=False, fused=False,
                  static_weights=True, phase=False, static_chain=False):
    r = WorkloadRunner(wl, copies=1, canary=True)
    if chain:
        step = r.step_chain
    elif static_chain:  # mlq_decode_chain_static: the chain without a caller workspace
        import block_quantized_decode_gb300 as M
        phases = [M.ChainPhase(r.fp32[src], r.sources[src], first, count, r.qbuf[src].q, r.qbuf[src].d)
                  for src, first, count in r.chain_phases()]
        products = [M.ChainProduct(M.QTensor(m.q[0], m.d[0], m.spec.rows, m.spec.cols, m.spec.wtype), m.y)
                    for m in r.mats]

        def step():
            M.mlq_decode_chain_static(phases, products)
    elif phase:
        def step():
            r.step_phase(static_weights=static_weights)
    elif fused:
        def step():
            r.step_fused(static_weights=static_weights)
    else:
        step = r.step
    if graph:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            step()            # warm-up outside capture (sets kernel attributes)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        for m in r.mats:
            m.y.fill_(float("nan"))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        g.replay()
    else:
        step()
    torch.cuda.synchronize()
    r.check_canaries()   # no write outside the outputs' own rows and blocks
    if chain:
        assert int(r.chain_ws.abs().sum()) == 0, "chain workspace not left zeroed"
    rng = np.random.default_rng(12345)
    checked = set()
    for m in r.mats:
        spec = m.spec
        k = r.sources[m.src]
        xin = r.fp32[m.src].cpu().numpy().reshape(r.m, k)
        gq = r.qbuf[m.src].q.cpu().numpy().reshape(r.m, k)
        gd = r.qbuf[m.src].d.cpu().numpy().reshape(r.m, k // 32)
        if m.src not in checked:
            oq, od = oracle.quantize_q8(xin)
            PT.assert_quant_equal(gq, gd, oq, od, f"{wl.name}: quantize of {m.src}")
            checked.add(m.src)
        y = m.y.cpu().numpy()
        assert np.all(np.isfinite(y)), f"{wl.name}/{spec.name}: non-finite output"
        full = spec.rows * spec.cols <= full_rows_limit // 64
        wins = None if full else PT.sample_windows(spec.rows, rng)
        for mi in range(r.m):
            PT.check_matvec(spec.wtype, m.host_q, m.host_d, spec.rows, spec.cols, gq[mi], gd[mi],
                            0, spec.rows, windows=wins, y_gpu=y[mi], what=f"{wl.name}/{spec.name}[m={mi}]")
    return r


def test_tiny_q4():
    run_and_check(I.tiny_q4())


def test_tinyllama_layer():
    run_and_check(I.tinyllama_layer())


def test_tinyllama_layer_graph_replay():
    run_and_check(I.tinyllama_layer(), graph=True)


def test_llama7b_ffn_q4():
    run_and_check(I.llama7b_ffn(I.Q4_0))


def test_llama7b_ffn_q8_lm_head():
    run_and_check(I.llama7b_ffn_q8_lm_head())


@pytest.mark.parametrize("m", [4, 16])
def test_small_m(m):
    run_and_check(I.small_m(m))
