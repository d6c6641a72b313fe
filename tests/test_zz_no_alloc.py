"""mlq_decode_chain_static -- the decode chain for callers that cannot
allocate device memory once they run (a load-once decode loop, a framework
that owns the allocator, code inside a stream capture).  It takes no
workspace: the library keeps the chain's grid-barrier counters in a fixed
device array of its own.

Called through the C ABI and compared with the existing entry point,
mlq_decode_chain (caller workspace), on the same inputs: the quantised
activations of every phase must be identical and every output within the
suite's tolerance, 1e-5 * sum_b |(float)sumi * dw * dx| per row, on two
calls in a row (the second call reuses the array the first one left).
This file is collected last on purpose."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from block_quantized_decode_gb300 import inputs as I  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def M():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_quantized_decode_gb300 import build as B
    B.build()
    import block_quantized_decode_gb300 as pkg
    torch.cuda.set_device(0)
    pkg.mlq_init()
    return pkg


def _args(M, r):
    phases = [M.ChainPhase(r.fp32[src], r.sources[src], first, count,
                           r.qbuf[src].q, r.qbuf[src].d)
              for src, first, count in r.chain_phases()]
    products = [M.ChainProduct(M.QTensor(m.q[0], m.d[0], m.spec.rows, m.spec.cols, m.spec.wtype),
                               m.y) for m in r.mats]
    return phases, products


def _snapshot(r):
    ys = [m.y.clone() for m in r.mats]
    qs = {src: (b.q.clone(), b.d.clone()) for src, b in r.qbuf.items()}
    return ys, qs


@pytest.mark.parametrize("wl", [I.tinyllama_layer(),
                                I.Workload("q8_chain", 1, [I.Matvec("a", I.Q8_0, 768, 256, "x"),
                                                           I.Matvec("b", I.Q8_0, 300, 768, "a")])],
                         ids=["tinyllama_layer_q4_0", "q8_two_phase"])
def test_static_chain_matches_workspace_chain(M, wl):
    from block_quantized_decode_gb300.runner import WorkloadRunner
    from tests import parity as PT

    r = WorkloadRunner(wl, copies=1, canary=True)
    phases, products = _args(M, r)
    ws = torch.zeros(M.mlq_chain_workspace_bytes(len(phases)) // 4, dtype=torch.int32,
                     device=PT.DEV)
    M.mlq_decode_chain(phases, products, ws)
    assert M.mlq_last_device_error() == M.MLQ_OK
    ref_y, ref_q = _snapshot(r)

    # per-row tolerance from the oracle's exact block sums on these inputs
    tols = []
    for m, y in zip(r.mats, ref_y):
        xq = ref_q[m.src][0].cpu().numpy().reshape(-1)
        xd = ref_q[m.src][1].cpu().numpy().reshape(-1)
        s = oracle.block_sumi(m.spec.wtype, m.host_q, m.spec.rows, m.spec.cols, xq)
        tols.append(PT.tol_rows(s, m.host_d, xd))

    for call in range(2):
        for m in r.mats:
            m.y.fill_(float("nan"))
        for b in r.qbuf.values():
            b.q.fill_(0)
            b.d.fill_(float("nan"))
        M.mlq_decode_chain_static(phases, products)
        assert M.mlq_last_device_error() == M.MLQ_OK, f"call {call}"
        r.check_canaries()
        for src, (q, d) in ref_q.items():
            assert torch.equal(r.qbuf[src].q, q), f"call {call}: quantised {src} differs"
            assert torch.equal(r.qbuf[src].d.view(torch.int32), d.view(torch.int32)), \
                f"call {call}: scales of {src} differ"
        for m, y0, tol in zip(r.mats, ref_y, tols):
            PT.assert_y_close(m.y.cpu().numpy().reshape(-1), y0.cpu().numpy().reshape(-1), tol,
                              f"call {call}: {m.spec.name}")


@pytest.mark.parametrize("wl", [I.tinyllama_layer(), I.llama7b_ffn(I.Q4_0)],
                         ids=["tinyllama_layer_q4_0", "llama7b_ffn8_q4_0"])
def test_static_chain_against_oracle(M, wl):
    """The static chain checked against the oracle directly, per step on the
    GPU's own inputs (quantised activations byte for byte, every product
    within tolerance), on two calls in a row."""
    from tests.test_gpu_configs import run_and_check
    for _ in range(2):
        run_and_check(wl, static_chain=True)
        assert M.mlq_last_device_error() == M.MLQ_OK


def test_static_chain_rejects_too_many_phases(M):
    """25 phases: above MLQ_CHAIN_STATIC_MAX_PHASES, which equals the general
    chain limit MLQ_CHAIN_MAX_PHASES, so this checks the limit the two entry
    points share (the static array itself holds one word more than that)."""
    x = torch.zeros(128, device="cuda:0")
    q = torch.zeros(4 * 64, dtype=torch.uint8, device="cuda:0")
    d = torch.zeros(4 * 4, device="cuda:0")
    y = torch.zeros(4, device="cuda:0")
    prod = M.ChainProduct(M.QTensor(q, d, 4, 128, M.MLQ_Q4_0), y)
    phases = [M.ChainPhase(x, 128, 0, 1)] * 25
    with pytest.raises(M.MlqError) as e:
        M.mlq_decode_chain_static(phases, [prod])
    assert e.value.status == M.MLQ_E_SHAPE
