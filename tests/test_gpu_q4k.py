"""Q4_K-style super-blocks on the GPU against the oracle (page
"SKaiNET-native-kernels", section "Proving an optimization is safe before
writing it"): the per-256 activation quantiser bit-exact (quants, scales,
per-32 sums), the per-super-block int32 sums ISUM / MSUM bit-exact, and y
within 1e-5 * sum_B |term_B| per row, where term_B = ((float)ISUM * d -
(float)MSUM * dmin) * dx is the float32 super-block term (the kernel adds
the terms in another order than the oracle)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from block_quantized_decode_gb300 import inputs as I  # noqa: E402

pytestmark = pytest.mark.gpu
QKK = 256
REL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def M():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_quantized_decode_gb300 import build as B
    B.build()
    import block_quantized_decode_gb300 as pkg
    pkg.mlq_init()
    torch.cuda.set_device(0)
    yield pkg
    assert pkg.mlq_last_device_error() == pkg.MLQ_OK


DEV = torch.device("cuda:0")


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def gpu_q8k(M, x: np.ndarray):
    k = x.size
    q = torch.empty(k, dtype=torch.int8, device=DEV)
    d = torch.empty(k // QKK, dtype=torch.float32, device=DEV)
    bs = torch.empty(k // 32, dtype=torch.int32, device=DEV)
    act = M.Q8KAct(q, d, bs, k)
    M.mlq_quantize_q8k(act, dev(x.astype(np.float32)), k)
    return act


def tensor(M, q, s, d, dmin, rows, cols):
    return M.Q4KTensor(dev(q), dev(s), dev(d), dev(dmin), rows, cols)


def act_from(M, xq, xd, xbs):
    return M.Q8KAct(dev(xq), dev(xd), dev(xbs), xq.size)


def check_q4k(M, q, s, d, dmin, rows, cols, xq, xd, xbs, r0=0, r1=None, what=""):
    """Integer sums bit-exact and y within the bound, rows [r0, r1)."""
    r1 = rows if r1 is None else r1
    nsb = cols // QKK
    W = tensor(M, q, s, d, dmin, rows, cols)
    X = act_from(M, xq, xd, xbs)
    gi = torch.zeros((max(r1 - r0, 1), nsb), dtype=torch.int32, device=DEV)
    gm = torch.zeros_like(gi)
    M.mlq_block_sums_q4k(gi, gm, W, X, r0, r1)
    y = torch.full((rows,), float("nan"), dtype=torch.float32, device=DEV)
    M.mlq_matvec_q4k(y, W, X, r0, r1)
    torch.cuda.synchronize()
    oi, om = oracle.block_sums_q4k(q, s, rows, cols, xq, xbs, r0, r1)
    assert np.array_equal(gi.cpu().numpy()[: r1 - r0], oi), f"{what}: ISUM differs"
    assert np.array_equal(gm.cpu().numpy()[: r1 - r0], om), f"{what}: MSUM differs"
    yo = oracle.matvec_q4k(q, s, d, dmin, rows, cols, xq, xd, xbs, r0, r1)
    yg = y.cpu().numpy()
    t = oi.astype(np.float32) * d[r0:r1]
    u = om.astype(np.float32) * dmin[r0:r1]
    terms = np.abs(((t - u) * xd[None, :]).astype(np.float64)).sum(axis=1)
    err = np.abs(yg[r0:r1].astype(np.float64) - yo[r0:r1].astype(np.float64))
    assert np.all(err <= REL * terms + 1e-30), f"{what}: max err/bound {np.max(err / (REL * terms + 1e-30))}"
    assert np.all(np.isnan(yg[:r0])) and np.all(np.isnan(yg[r1:])), f"{what}: rows outside [r0, r1) written"


@pytest.mark.parametrize("k", [256, 512, 2048, 5632, 11008, 65536])
def test_quantize_q8k_bit_exact(M, k):
    rng = np.random.default_rng(k)
    x = (rng.standard_normal(k) * 10.0 ** rng.uniform(-20, 20, size=k // QKK).repeat(QKK)).astype(np.float32)
    if k >= 2 * QKK:
        x[:QKK] = 0.0                      # an all-zero block: d = 0, quants 0
        x[QKK + 3] = np.float32(1e-40)     # a subnormal
    act = gpu_q8k(M, x)
    torch.cuda.synchronize()
    oq, od, obs = oracle.quantize_q8k(x)
    assert np.array_equal(act.q.cpu().numpy(), oq)
    assert np.array_equal(act.d.cpu().numpy().view(np.uint32), od.view(np.uint32))
    assert np.array_equal(act.bsums.cpu().numpy(), obs)


@pytest.mark.parametrize("rows,cols", [(1, 256), (7, 512), (64, 2048), (333, 2048), (1000, 256),
                                       (300, 5632), (96, 11008), (40, 16384)])
def test_matvec_q4k_parity(M, rows, cols):
    q, s, d, dmin = I.q4k_weights(rows, cols, seed=rows * 7 + cols)
    x = I.activations(1, cols, seed=cols)[0]
    xq, xd, xbs = oracle.quantize_q8k(x)
    check_q4k(M, q, s, d, dmin, rows, cols, xq, xd, xbs, what=f"{rows}x{cols}")


def test_matvec_q4k_row_ranges(M):
    rows, cols = 777, 1024
    q, s, d, dmin = I.q4k_weights(rows, cols, seed=5)
    xq, xd, xbs = oracle.quantize_q8k(I.activations(1, cols, seed=6)[0])
    for r0, r1 in [(0, 1), (13, 14), (5, 700), (640, 777), (100, 100)]:
        if r1 > r0:
            check_q4k(M, q, s, d, dmin, rows, cols, xq, xd, xbs, r0, r1, what=f"[{r0},{r1})")
    W = tensor(M, q, s, d, dmin, rows, cols)
    y = torch.full((rows,), 3.0, dtype=torch.float32, device=DEV)
    M.mlq_matvec_q4k(y, W, act_from(M, xq, xd, xbs), 100, 100)   # empty range: no write
    torch.cuda.synchronize()
    assert bool((y == 3.0).all())


def test_matvec_q4k_overflow_bound(M):
    """The page's worst case on the GPU: nibbles 15, scales 63, minima 63,
    activations +-127 give ISUM = +-8*63*32*127*15 exactly."""
    rows, cols = 4, 4 * QKK
    nsb = cols // QKK
    q = np.full((rows, cols // 2), 0xFF, np.uint8)
    s = np.full((rows, nsb * 16), 63, np.uint8)
    d = np.full((rows, nsb), 1e-3, np.float32)
    dmin = np.full((rows, nsb), 2e-3, np.float32)
    for sign in (1, -1):
        xq = np.full(cols, 127 * sign, np.int8)
        xbs = np.full(cols // 32, 32 * 127 * sign, np.int32)
        xd = np.full(nsb, 0.01, np.float32)
        W = tensor(M, q, s, d, dmin, rows, cols)
        gi = torch.zeros((rows, nsb), dtype=torch.int32, device=DEV)
        gm = torch.zeros_like(gi)
        M.mlq_block_sums_q4k(gi, gm, W, act_from(M, xq, xd, xbs), 0, rows)
        torch.cuda.synchronize()
        assert bool((gi == sign * 30723840).all()) and bool((gm == sign * 8 * 63 * 32 * 127).all())
        check_q4k(M, q, s, d, dmin, rows, cols, xq, xd, xbs, what=f"bound {sign}")


def test_matvec_q4k_full_byte_scales(M):
    """Scales and minima up to 255 (beyond 6 bits) still sum exactly in int32."""
    rng = np.random.default_rng(9)
    rows, cols = 50, 2048
    q, s, d, dmin = I.q4k_weights(rows, cols, seed=9)
    s = rng.integers(0, 256, size=s.shape, dtype=np.uint8)
    xq = rng.choice(np.array([-127, 127], np.int8), size=cols)
    xbs = xq.astype(np.int64).reshape(-1, 32).sum(axis=1).astype(np.int32)
    xd = np.full(cols // QKK, 1e-2, np.float32)
    check_q4k(M, q, s, d, dmin, rows, cols, xq, xd, xbs, what="byte scales")


def test_q4k_tinyllama_layer_shapes_sampled(M):
    """TinyLlama-1.1B projection shapes in Q4_K (the page's model): the GPU
    quantiser's output feeds the product; sampled rows of every product
    against the oracle, the integer sums of whole matrices bit-exact."""
    rng = np.random.default_rng(3)
    for i, (rows, cols) in enumerate([(2048, 2048), (256, 2048), (5632, 2048), (2048, 5632)]):
        q, s, d, dmin = I.q4k_weights(rows, cols, seed=100 + i)
        x = I.activations(1, cols, seed=200 + i)[0]
        act = gpu_q8k(M, x)
        torch.cuda.synchronize()
        xq, xd, xbs = (act.q.cpu().numpy(), act.d.cpu().numpy(), act.bsums.cpu().numpy())
        W = tensor(M, q, s, d, dmin, rows, cols)
        y = torch.empty(rows, dtype=torch.float32, device=DEV)
        M.mlq_matvec_q4k(y, W, act, 0, rows)
        nsb = cols // QKK
        gi = torch.empty((rows, nsb), dtype=torch.int32, device=DEV)
        gm = torch.empty_like(gi)
        M.mlq_block_sums_q4k(gi, gm, W, act, 0, rows)
        torch.cuda.synchronize()
        oi, om = oracle.block_sums_q4k(q, s, rows, cols, xq, xbs)
        assert np.array_equal(gi.cpu().numpy(), oi) and np.array_equal(gm.cpu().numpy(), om)
        yg = y.cpu().numpy()
        for r0 in rng.integers(0, rows - 8, size=4):
            yo = oracle.matvec_q4k(q, s, d, dmin, rows, cols, xq, xd, xbs, int(r0), int(r0) + 8)
            t = (oi[r0:r0 + 8].astype(np.float32) * d[r0:r0 + 8] -
                 om[r0:r0 + 8].astype(np.float32) * dmin[r0:r0 + 8]) * xd[None, :]
            bound = REL * np.abs(t.astype(np.float64)).sum(axis=1)
            assert np.all(np.abs(yg[r0:r0 + 8] - yo[r0:r0 + 8]) <= bound)


def test_q4k_layer_pass_through_runner(M):
    """The bench's Q4_K pass (per input mlq_quantize_q8k, then its products,
    outputs feeding later inputs): every quantised input bit-exact against
    the oracle's quantisation of the GPU's float vector, every product's
    y within the bound on the GPU's own quantised input."""
    from block_quantized_decode_gb300.runner import Q4KRunner
    wl = I.tinyllama_layer_q4k()
    r = Q4KRunner(wl, copies=1)
    r.step()
    torch.cuda.synchronize()
    for name, rows, cols, inp in wl.mats:
        xv = r.vec(inp).cpu().numpy()
        oq, od, obs = oracle.quantize_q8k(xv)
        act = r.act[inp]
        assert np.array_equal(act.q.cpu().numpy(), oq), f"{name}: quantised input differs"
        assert np.array_equal(act.d.cpu().numpy().view(np.uint32), od.view(np.uint32))
        assert np.array_equal(act.bsums.cpu().numpy(), obs)
        q, s, d, dmin, _, _ = r.host[name]
        yo = oracle.matvec_q4k(q, s, d, dmin, rows, cols, oq, od, obs)
        oi, om = oracle.block_sums_q4k(q, s, rows, cols, oq, obs)
        t = (oi.astype(np.float32) * d - om.astype(np.float32) * dmin) * od[None, :]
        bound = REL * np.abs(t.astype(np.float64)).sum(axis=1)
        yg = r.y[name].cpu().numpy()
        assert np.all(np.abs(yg.astype(np.float64) - yo) <= bound), name


@pytest.mark.parametrize("rows,cols", [(1, 256), (77, 2048), (2048, 2048), (300, 5632)])
def test_q4k_phase_single_product_bitwise(M, rows, cols):
    """One product through mlq_q4k_phase (x quantised inside the launch)
    against mlq_quantize_q8k + mlq_matvec_q4k: the same launch geometry and
    the same quantiser arithmetic, so y must be bit-identical; and within
    the bound of the oracle."""
    q, s, d, dmin = I.q4k_weights(rows, cols, seed=rows + cols)
    x = I.activations(1, cols, seed=cols + 3)[0]
    W = tensor(M, q, s, d, dmin, rows, cols)
    xd_ = dev(x.astype(np.float32))
    y1 = torch.full((rows,), float("nan"), dtype=torch.float32, device=DEV)
    y2 = torch.full((rows,), float("nan"), dtype=torch.float32, device=DEV)
    M.mlq_q4k_phase(xd_, cols, [(W, y1)])
    act = gpu_q8k(M, x)
    M.mlq_matvec_q4k(y2, W, act, 0, rows)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2), "the phase and the separate calls differ"
    xq, xdq, xbs = oracle.quantize_q8k(x)
    yo = oracle.matvec_q4k(q, s, d, dmin, rows, cols, xq, xdq, xbs)
    oi, om = oracle.block_sums_q4k(q, s, rows, cols, xq, xbs)
    t = (oi.astype(np.float32) * d - om.astype(np.float32) * dmin) * xdq[None, :]
    bound = REL * np.abs(t.astype(np.float64)).sum(axis=1)
    assert np.all(np.abs(y1.cpu().numpy().astype(np.float64) - yo) <= bound + 1e-30)


@pytest.mark.parametrize("shapes,cols", [([(2048, 2048), (256, 2048), (256, 2048)], 2048),
                                         ([(5632, 2048), (5632, 2048)], 2048),
                                         ([(77, 512), (1, 512), (300, 512), (33, 512)], 512)])
def test_q4k_phase_grouped_vs_oracle(M, shapes, cols):
    """Products sharing one float input in one launch (rows of several
    products in one CTA, stages that stop at product ends): every y within
    the bound of the oracle on the oracle's quantisation of x."""
    x = I.activations(1, cols, seed=len(shapes) + cols)[0]
    xq, xdq, xbs = oracle.quantize_q8k(x)
    prods, host = [], []
    for i, (rows, c) in enumerate(shapes):
        q, s, d, dmin = I.q4k_weights(rows, c, seed=100 + i)
        y = torch.full((rows,), float("nan"), dtype=torch.float32, device=DEV)
        prods.append((tensor(M, q, s, d, dmin, rows, c), y))
        host.append((q, s, d, dmin, rows))
    M.mlq_q4k_phase(dev(x.astype(np.float32)), cols, prods)
    torch.cuda.synchronize()
    for (q, s, d, dmin, rows), (_, y) in zip(host, prods):
        yo = oracle.matvec_q4k(q, s, d, dmin, rows, cols, xq, xdq, xbs)
        oi, om = oracle.block_sums_q4k(q, s, rows, cols, xq, xbs)
        t = (oi.astype(np.float32) * d - om.astype(np.float32) * dmin) * xdq[None, :]
        bound = REL * np.abs(t.astype(np.float64)).sum(axis=1)
        yg = y.cpu().numpy()
        assert np.all(np.isfinite(yg)), f"{rows} rows: not every row written"
        assert np.all(np.abs(yg.astype(np.float64) - yo) <= bound + 1e-30), f"{rows}x{cols}"


def test_q4k_layer_phase_pass_through_runner(M):
    """The bench's Q4_K pass as four phase launches (q|k|v, o, gate|up,
    down): every product's y within the bound of the oracle on the oracle's
    quantisation of the GPU's own float input."""
    from block_quantized_decode_gb300.runner import Q4KRunner
    wl = I.tinyllama_layer_q4k()
    r = Q4KRunner(wl, copies=1)
    assert len(r.phases()) == 4
    r.step_phase()
    torch.cuda.synchronize()
    for name, rows, cols, inp in wl.mats:
        oq, od, obs = oracle.quantize_q8k(r.vec(inp).cpu().numpy())
        q, s, d, dmin, _, _ = r.host[name]
        yo = oracle.matvec_q4k(q, s, d, dmin, rows, cols, oq, od, obs)
        oi, om = oracle.block_sums_q4k(q, s, rows, cols, oq, obs)
        t = (oi.astype(np.float32) * d - om.astype(np.float32) * dmin) * od[None, :]
        bound = REL * np.abs(t.astype(np.float64)).sum(axis=1)
        yg = r.y[name].cpu().numpy()
        assert np.all(np.abs(yg.astype(np.float64) - yo) <= bound), name
