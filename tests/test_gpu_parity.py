"""CUDA path vs the CPU oracle, through the C ABI, on cuda:0.

Quant bytes, scales and per-block sums must be bit-exact; float outputs
within 1e-5 * sum_b |term_b| per row (tests/parity.py).  Shapes span several
tiles/chunks and ragged tails; edge cases: K = 32, a single row, r0 > 0,
empty ranges, all-zero and tiny-amax blocks, M from 1 to 16.
"""
import json
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from tests import oracle_pins as P  # noqa: E402

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


from tests import parity as PT  # noqa: E402  (imports torch / the package)


def rand_q4(rng, rows, cols):
    return (rng.integers(0, 256, size=(rows, cols // 2), dtype=np.uint8),
            rng.uniform(1e-3, 1e-2, size=(rows, cols // 32)).astype(np.float32))


def rand_q8(rng, rows, cols):
    return (rng.integers(-127, 128, size=(rows, cols), dtype=np.int8),
            rng.uniform(1e-4, 1e-3, size=(rows, cols // 32)).astype(np.float32))


def rand_x(rng, m, k):
    return rng.standard_normal((m, k)).astype(np.float32)


# ---------------------------------------------------------------------------
# quantize
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("m,k", [(1, 32), (1, 96), (1, 512), (1, 896), (1, 2048), (1, 11008),
                                 (3, 4128), (16, 4096), (16, 11008), (2, 65536)])
def test_quantize_bit_exact(m, k):
    rng = np.random.default_rng(100 + m * 7 + k)
    x = P.random_block_inputs(rng, m * k // 32).reshape(m, k)
    x[0, :32] = 0.0                                      # a d = 0 block
    if k >= 64:
        x[0, 32:64] = np.float32(1e-38) * rng.standard_normal(32).astype(np.float32)  # id overflows
    gq, gd = PT.gpu_quantize(x)
    oq, od = oracle.quantize_q8(x)
    PT.assert_quant_equal(gq, gd, oq, od, f"quantize {m}x{k}")


def test_quantize_golden_blocks():
    g = json.load(open(os.path.join(P.GOLDEN, "quantize_q8_blocks.json")))
    xs, want = [], []
    for blk in g["blocks"]:
        x = np.zeros(32, dtype=np.float32)
        for i, h in blk.get("x_hex", {}).items():
            x[int(i)] = P.f32_from_hex(h)
        if "x_int" in blk:
            x[:] = np.array(blk["x_int"], dtype=np.float32)
        w = np.zeros(32, dtype=np.int8)
        if "q_all" in blk:
            w[:] = blk["q_all"]
        else:
            for i, v in blk["q"].items():
                w[int(i)] = v
        xs.append(x)
        want.append(w)
    gq, gd = PT.gpu_quantize(np.concatenate(xs).reshape(1, -1))
    assert np.array_equal(gq.reshape(-1, 32), np.stack(want))
    _, od = oracle.quantize_q8(np.concatenate(xs))
    assert np.array_equal(gd.reshape(-1).view(np.uint32), od.view(np.uint32))


# ---------------------------------------------------------------------------
# per-block sums (exact) and the M = 1 products
# ---------------------------------------------------------------------------
SHAPES = [(1, 32), (7, 96), (5, 128), (256, 512), (33, 2048), (17, 4128), (9, 5632),
          (300, 896), (40, 11008), (3, 65536)]


@pytest.mark.parametrize("wtype", [oracle.Q4_0, oracle.Q8_0], ids=["q4", "q8"])
@pytest.mark.parametrize("rows,cols", SHAPES)
def test_block_sumi_exact(lib, wtype, rows, cols):
    M = lib
    rng = np.random.default_rng(rows * 31 + cols + wtype)
    wq, wd = (rand_q4 if wtype == oracle.Q4_0 else rand_q8)(rng, rows, cols)
    xq = rng.integers(-127, 128, size=cols, dtype=np.int8)
    xd = rng.uniform(1e-3, 1e-1, size=cols // 32).astype(np.float32)
    r0 = 1 if rows > 2 else 0
    r1 = rows
    nb = cols // 32
    out = torch.full(((r1 - r0) * nb,), -12345, dtype=torch.int32, device=PT.DEV)
    W = PT.weights_dev(wtype, wq, wd, rows, cols)
    M.mlq_block_sumi(out, W, M.QAct(PT.to_dev(xq), PT.to_dev(xd), cols, 1), r0, r1)
    got = out.cpu().numpy().reshape(r1 - r0, nb)
    want = oracle.block_sumi(wtype, wq, rows, cols, xq, r0, r1)
    assert np.array_equal(got, want)


def test_block_sumi_extremes(lib):
    """All-zero nibbles against qx = -127 (the Q4_0 extreme 32512), Q8_0
    +-127 products (+-516128), and the hand-computed blocks."""
    M = lib
    cols = 128
    wq4 = np.zeros((2, cols // 2), dtype=np.uint8)
    wq4[1, :16] = [j | ((15 - j) << 4) for j in range(16)]
    xq = np.full(cols, -127, dtype=np.int8)
    xq[:32] = np.arange(32)
    wd = np.ones((2, cols // 32), dtype=np.float32)
    out = torch.zeros(2 * 4, dtype=torch.int32, device=PT.DEV)
    M.mlq_block_sumi(out, PT.weights_dev(oracle.Q4_0, wq4, wd, 2, cols),
                     M.QAct(PT.to_dev(xq), PT.to_dev(np.ones(4, np.float32)), cols, 1), 0, 2)
    got = out.cpu().numpy().reshape(2, 4)
    assert got[0, 1] == 32512 and got[1, 0] == -248
    assert np.array_equal(got, oracle.block_sumi(oracle.Q4_0, wq4, 2, cols, xq))
    wq8 = np.full((2, cols), 127, dtype=np.int8)
    wq8[1] = -127
    xq8 = np.full(cols, 127, dtype=np.int8)
    out = torch.zeros(2 * 4, dtype=torch.int32, device=PT.DEV)
    M.mlq_block_sumi(out, PT.weights_dev(oracle.Q8_0, wq8, wd, 2, cols),
                     M.QAct(PT.to_dev(xq8), PT.to_dev(np.ones(4, np.float32)), cols, 1), 0, 2)
    got = out.cpu().numpy().reshape(2, 4)
    assert np.all(got[0] == 516128) and np.all(got[1] == -516128)


@pytest.mark.parametrize("wtype", [oracle.Q4_0, oracle.Q8_0], ids=["q4", "q8"])
@pytest.mark.parametrize("rows,cols", SHAPES + [(2048, 2048), (1000, 4096)])
def test_matvec_parity(wtype, rows, cols):
    rng = np.random.default_rng(rows * 13 + cols * 3 + wtype)
    wq, wd = (rand_q4 if wtype == oracle.Q4_0 else rand_q8)(rng, rows, cols)
    xq, xd = oracle.quantize_q8(rand_x(rng, 1, cols)[0])
    PT.check_matvec(wtype, wq, wd, rows, cols, xq, xd, 0, rows, what=f"{rows}x{cols}")
    if rows >= 5:
        PT.check_matvec(wtype, wq, wd, rows, cols, xq, xd, 2, rows - 3, what=f"{rows}x{cols} sub")


def test_matvec_zero_blocks_and_empty_range(lib):
    M = lib
    rng = np.random.default_rng(7)
    rows, cols = 64, 256
    wq, wd = rand_q4(rng, rows, cols)
    x = rand_x(rng, 1, cols)[0]
    x[:64] = 0.0                       # two d = 0 activation blocks
    xq, xd = oracle.quantize_q8(x)
    assert xd[0] == 0 and xd[1] == 0
    PT.check_matvec(oracle.Q4_0, wq, wd, rows, cols, xq, xd, 0, rows, what="zero blocks")
    y = torch.full((rows,), 3.0, dtype=torch.float32, device=PT.DEV)
    W = PT.weights_dev(oracle.Q4_0, wq, wd, rows, cols)
    M.mlq_matvec_q4(y, W, M.QAct(PT.to_dev(xq), PT.to_dev(xd), cols, 1), 10, 10)
    assert torch.all(y == 3.0)
    W0 = M.QTensor(PT.to_dev(wq.reshape(-1)), PT.to_dev(wd.reshape(-1)), 0, cols, M.MLQ_Q4_0)
    M.mlq_matvec_q4(y, W0, M.QAct(PT.to_dev(xq), PT.to_dev(xd), cols, 1), 0, 0)
    assert torch.all(y == 3.0)


def test_matvec_all_zero_activation(lib):
    """x = 0: every d = 0, every quant 0, y exactly 0."""
    rows, cols = 100, 512
    rng = np.random.default_rng(8)
    wq, wd = rand_q8(rng, rows, cols)
    gq, gd = PT.gpu_quantize(np.zeros((1, cols), np.float32))
    assert not gq.any() and not gd.any()
    y = PT.check_matvec(oracle.Q8_0, wq, wd, rows, cols, gq[0], gd[0], 0, rows)
    assert np.all(y == 0.0)


# ---------------------------------------------------------------------------
# small-M product
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("Mr", [1, 2, 3, 4, 5, 6, 7, 8, 11, 16])
@pytest.mark.parametrize("rows,cols", [(1, 32), (70, 512), (37, 4128), (64, 11008)])
def test_gemm_small_m_parity(lib, Mr, rows, cols):
    M = lib
    rng = np.random.default_rng(Mr * 1000 + rows + cols)
    wq, wd = rand_q4(rng, rows, cols)
    X = rand_x(rng, Mr, cols)
    Xq, Xd = oracle.quantize_q8(X)
    ldy = rows + 3
    r0 = 1 if rows > 1 else 0
    Y = torch.full((Mr, ldy), float("nan"), dtype=torch.float32, device=PT.DEV)
    W = PT.weights_dev(oracle.Q4_0, wq, wd, rows, cols)
    M.mlq_gemm_q4_small_m(Y, ldy, W, M.QAct(PT.to_dev(Xq), PT.to_dev(Xd), cols, Mr), Mr, r0, rows)
    Yg = Y.cpu().numpy()
    assert np.all(np.isnan(Yg[:, :r0])) and np.all(np.isnan(Yg[:, rows:]))
    Yo = oracle.gemm_small_m(oracle.Q4_0, wq, wd, rows, cols, Xq, Xd, Mr, r0, rows, ldy=ldy)
    nb = cols // 32
    for m in range(Mr):
        s = oracle.block_sumi(oracle.Q4_0, wq, rows, cols, Xq[m], r0, rows)
        tol = PT.tol_rows(s, wd[r0:rows], Xd[m])
        PT.assert_y_close(Yg[m, r0:rows], Yo[m, r0:rows], tol, f"M={Mr} row m={m}")
    assert nb > 0


@pytest.mark.parametrize("rows,cols", [(24576, 4096), (8192, 16384)])
def test_gemm_small_m_many_rows(lib, rows, cols):
    """Enough rows that a cluster of the tensor-core kernel takes several
    rounds (more than 160 rows each), at two K-part counts; checked on
    sampled row windows, with an offset row range and a padded ldy."""
    M = lib
    Mr = 16
    rng = np.random.default_rng(rows + cols)
    wq, wd = rand_q4(rng, rows, cols)
    X = rand_x(rng, Mr, cols)
    Xq, Xd = oracle.quantize_q8(X)
    r0, r1, ldy = 5, rows - 3, rows + 7
    Y = torch.full((Mr, ldy), float("nan"), dtype=torch.float32, device=PT.DEV)
    W = PT.weights_dev(oracle.Q4_0, wq, wd, rows, cols)
    M.mlq_gemm_q4_small_m(Y, ldy, W, M.QAct(PT.to_dev(Xq), PT.to_dev(Xd), cols, Mr), Mr, r0, r1)
    Yg = Y.cpu().numpy()
    assert np.all(np.isnan(Yg[:, :r0])) and np.all(np.isnan(Yg[:, r1:]))
    assert np.all(np.isfinite(Yg[:, r0:r1]))
    wins = [(r0, r0 + 32), (r1 - 32, r1)] + [(a, a + 32) for a in rng.integers(r0, r1 - 32, 6)]
    for m in range(Mr):
        PT.check_matvec(oracle.Q4_0, wq, wd, rows, cols, Xq[m], Xd[m], r0, r1, windows=wins,
                        y_gpu=Yg[m], what=f"M=16 {rows}x{cols} row m={m}")


# ---------------------------------------------------------------------------
# bounded device waits
# ---------------------------------------------------------------------------
def test_timeout_path_reports_status(lib):
    """A wait limit of 0 makes the activation-staging wait give up at once:
    the kernel records MLQ_E_TIMEOUT, drains its own copy and returns; the
    next launch with the normal limit is clean."""
    M = lib
    rng = np.random.default_rng(9)
    rows, cols = 64, 512
    wq, wd = rand_q4(rng, rows, cols)
    xq, xd = oracle.quantize_q8(rand_x(rng, 1, cols)[0])
    W = PT.weights_dev(oracle.Q4_0, wq, wd, rows, cols)
    x = M.QAct(PT.to_dev(xq), PT.to_dev(xd), cols, 1)
    y = torch.zeros(rows, dtype=torch.float32, device=PT.DEV)
    assert M.mlq_last_device_error() == M.MLQ_OK
    try:
        M.mlq_debug_set_wait_limit_ns(0)
        M.mlq_matvec_q4(y, W, x, 0, rows)
        assert M.mlq_last_device_error() == M.MLQ_E_TIMEOUT
        assert M.mlq_last_device_error() == M.MLQ_OK   # cleared by the read
    finally:
        M.mlq_debug_set_wait_limit_ns(10 ** 9)
    PT.check_matvec(oracle.Q4_0, wq, wd, rows, cols, xq, xd, 0, rows, what="after timeout")


@pytest.mark.parametrize("Mr", [2, 8, 16])
def test_gemm_small_m_unit_scales_exact(lib, Mr):
    """With every scale 1 the product is a plain integer GEMM of the decoded
    weights; all partial sums are integers below 2^24, so the result must
    be exact: this pins the tensor-core block sums to the int32 definition."""
    M = lib
    rng = np.random.default_rng(50 + Mr)
    rows, cols = 77, 512
    wq = rng.integers(0, 256, size=(rows, cols // 2), dtype=np.uint8)
    wd = np.ones((rows, cols // 32), dtype=np.float32)
    Xq = rng.integers(-127, 128, size=(Mr, cols), dtype=np.int8)
    Xd = np.ones((Mr, cols // 32), dtype=np.float32)
    Y = torch.full((Mr, rows), float("nan"), dtype=torch.float32, device=PT.DEV)
    M.mlq_gemm_q4_small_m(Y, rows, PT.weights_dev(oracle.Q4_0, wq, wd, rows, cols),
                          M.QAct(PT.to_dev(Xq), PT.to_dev(Xd), cols, Mr), Mr, 0, rows)
    want = P.decode_q4_elements(wq, cols) @ Xq.astype(np.int64).T   # [rows, Mr]
    assert np.array_equal(Y.cpu().numpy().astype(np.int64), want.T)


@pytest.mark.skipif(os.environ.get("MLQ_GEMM_KERNEL") != "umma",
                    reason="the tcgen05 small-M kernel's abort path; run by the forced-kernel test")
def test_gemm_small_m_umma_timeout_path(lib):
    """A wait limit of 0 makes the tcgen05 kernel's first wait give up: every
    role leaves its loop, the producer drains its copies, the cluster meets
    once more, the tensor memory is freed, and MLQ_E_TIMEOUT is recorded.
    The next launch with the normal limit is clean and correct."""
    M = lib
    rng = np.random.default_rng(11)
    Mr, rows, cols = 16, 512, 4096
    wq, wd = rand_q4(rng, rows, cols)
    Xq, Xd = oracle.quantize_q8(rand_x(rng, Mr, cols))
    W = PT.weights_dev(oracle.Q4_0, wq, wd, rows, cols)
    X = M.QAct(PT.to_dev(Xq), PT.to_dev(Xd), cols, Mr)
    Y = torch.zeros((Mr, rows), dtype=torch.float32, device=PT.DEV)
    assert M.mlq_last_device_error() == M.MLQ_OK
    try:
        M.mlq_debug_set_wait_limit_ns(0)
        M.mlq_gemm_q4_small_m(Y, rows, W, X, Mr, 0, rows)
        assert M.mlq_last_device_error() == M.MLQ_E_TIMEOUT
        assert M.mlq_last_device_error() == M.MLQ_OK
    finally:
        M.mlq_debug_set_wait_limit_ns(10 ** 9)
    M.mlq_gemm_q4_small_m(Y, rows, W, X, Mr, 0, rows)
    Yg = Y.cpu().numpy()
    for m in (0, 7, 15):
        PT.check_matvec(oracle.Q4_0, wq, wd, rows, cols, Xq[m], Xd[m], 0, rows, y_gpu=Yg[m],
                        what=f"after timeout m={m}")


def test_gemm_small_m_ring_timeout_path(lib):
    """M <= 4 runs the ring kernel: with a wait limit of 0 its consumers give
    up on their first stage and its producer on its first refill; the
    producer drains the copies it issued, MLQ_E_TIMEOUT is recorded, and the
    next launch with the normal limit is clean and correct."""
    if os.environ.get("MLQ_GEMM_KERNEL") not in (None, "ring"):
        pytest.skip("another small-M kernel is forced")
    M = lib
    rng = np.random.default_rng(12)
    Mr, rows, cols = 4, 2048, 4096
    wq, wd = rand_q4(rng, rows, cols)
    Xq, Xd = oracle.quantize_q8(rand_x(rng, Mr, cols))
    W = PT.weights_dev(oracle.Q4_0, wq, wd, rows, cols)
    X = M.QAct(PT.to_dev(Xq), PT.to_dev(Xd), cols, Mr)
    Y = torch.zeros((Mr, rows), dtype=torch.float32, device=PT.DEV)
    assert M.mlq_last_device_error() == M.MLQ_OK
    try:
        M.mlq_debug_set_wait_limit_ns(0)
        M.mlq_gemm_q4_small_m(Y, rows, W, X, Mr, 0, rows)
        assert M.mlq_last_device_error() == M.MLQ_E_TIMEOUT
        assert M.mlq_last_device_error() == M.MLQ_OK
    finally:
        M.mlq_debug_set_wait_limit_ns(10 ** 9)
    M.mlq_gemm_q4_small_m(Y, rows, W, X, Mr, 0, rows)
    Yg = Y.cpu().numpy()
    for m in range(Mr):
        PT.check_matvec(oracle.Q4_0, wq, wd, rows, cols, Xq[m], Xd[m], 0, rows, y_gpu=Yg[m],
                        what=f"after timeout m={m}")
