"""Blocks of 32 or 128 weights, float32 or float16 scales, 4-bit weights
and 8-bit weights in the packed signed form with per-block zero points
(page "ONNX Runtime", "How we got there", items 3-5) on the GPU against the
oracle: the per-block activation quantiser bit-exact (quants, scales, quant
sums), the per-block int32 sums bit-exact, y within 1e-5 * sum_b |term_b|
per row with term_b = ((float)sumi * scale_b) * dx_b."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from block_quantized_decode_gb300 import inputs as I  # noqa: E402

pytestmark = pytest.mark.gpu
REL = 1e-5
DEV = torch.device("cuda:0")


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


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def tensor(M, q, sc, zp, rows, cols, bits, blk):
    scp = I.pad_rows(sc)
    zpp = None if zp is None else I.pad_rows(zp)
    f16 = sc.dtype == np.float16
    return M.NBitsTensor(dev(q), dev(scp.view(np.uint16) if f16 else scp), None if zpp is None else dev(zpp),
                         rows, cols, bits, blk, 1 if f16 else 0, scp.shape[1],
                         0 if zpp is None else zpp.shape[1])


def gpu_quantize_blk(M, x, blk):
    k = x.size
    act = M.BlkAct(torch.empty(k, dtype=torch.int8, device=DEV),
                   torch.empty(k // blk, dtype=torch.float32, device=DEV),
                   torch.empty(k // blk, dtype=torch.int32, device=DEV), k, blk)
    M.mlq_quantize_blk(act, dev(x.astype(np.float32)), k)
    return act


def check(M, q, sc, zp, rows, cols, bits, blk, xq, xd, xbs, r0=0, r1=None, what=""):
    r1 = rows if r1 is None else r1
    nb = cols // blk
    W = tensor(M, q, sc, zp, rows, cols, bits, blk)
    X = M.BlkAct(dev(xq), dev(xd), dev(xbs), cols, blk)
    gs = torch.zeros((max(r1 - r0, 1), nb), dtype=torch.int32, device=DEV)
    M.mlq_block_sumi_nbits(gs, W, X, r0, r1)
    y = torch.full((rows,), float("nan"), dtype=torch.float32, device=DEV)
    M.mlq_matvec_nbits(y, W, X, r0, r1)
    torch.cuda.synchronize()
    os_ = oracle.block_sumi_nbits(q, zp, rows, cols, bits, blk, xq, r0, r1)
    assert np.array_equal(gs.cpu().numpy()[: r1 - r0], os_), f"{what}: sumi differs"
    yo = oracle.matvec_nbits(q, sc, zp, rows, cols, bits, blk, xq, xd, r0, r1)
    scf = sc.astype(np.float32)[r0:r1]
    terms = np.abs(((os_.astype(np.float32) * scf) * xd[None, :]).astype(np.float64)).sum(axis=1)
    yg = y.cpu().numpy()
    err = np.abs(yg[r0:r1].astype(np.float64) - yo[r0:r1].astype(np.float64))
    assert np.all(err <= REL * terms + 1e-30), f"{what}: max err/bound {np.max(err / (REL * terms + 1e-30))}"
    assert np.all(np.isnan(yg[:r0])) and np.all(np.isnan(yg[r1:])), f"{what}: rows outside [r0, r1) written"


@pytest.mark.parametrize("blk", [32, 128])
@pytest.mark.parametrize("k", [128, 896, 4864, 65536])
def test_quantize_blk_bit_exact(M, k, blk):
    rng = np.random.default_rng(k + blk)
    x = (rng.standard_normal(k) * 10.0 ** rng.uniform(-20, 20, size=k // blk).repeat(blk)).astype(np.float32)
    x[:blk] = 0.0
    act = gpu_quantize_blk(M, x, blk)
    torch.cuda.synchronize()
    oq, od, obs = oracle.quantize_blk(x, blk)
    assert np.array_equal(act.q.cpu().numpy(), oq)
    assert np.array_equal(act.d.cpu().numpy().view(np.uint32), od.view(np.uint32))
    assert np.array_equal(act.bsums.cpu().numpy(), obs)


COMBOS = [(bits, blk, f16, zp) for bits in (4, 8) for blk in (32, 128) for f16 in (False, True)
          for zp in ((False, True) if bits == 8 else (False,))]


@pytest.mark.parametrize("bits,blk,f16,with_zp", COMBOS,
                         ids=[f"b{b}_blk{k}_{'f16' if f else 'f32'}{'_zp' if z else ''}" for b, k, f, z in COMBOS])
@pytest.mark.parametrize("rows,cols", [(1, 128), (33, 896), (500, 896), (896, 4864), (40, 16384)])
def test_matvec_nbits_parity(M, bits, blk, f16, with_zp, rows, cols):
    seed = rows * 31 + cols + bits * 7 + blk + int(f16) * 3 + int(with_zp)
    q, sc, zp = I.nbits_weights(rows, cols, bits, blk, f16, with_zp, seed=seed)
    xq, xd, xbs = oracle.quantize_blk(I.activations(1, cols, seed=seed + 1)[0], blk)
    check(M, q, sc, zp, rows, cols, bits, blk, xq, xd, xbs, what=f"{bits}/{blk}/{f16}/{with_zp} {rows}x{cols}")


def test_matvec_nbits_row_ranges_and_extremes(M):
    rows, cols, blk = 300, 1024, 128
    q, sc, zp = I.nbits_weights(rows, cols, 8, blk, True, True, seed=77)
    zp[:, 0] = 0
    zp[:, 1] = 255
    xq = np.full(cols, 127, np.int8)
    xq[blk:2 * blk] = -127
    xd = np.full(cols // blk, 1e-2, np.float32)
    xbs = xq.astype(np.int64).reshape(-1, blk).sum(axis=1).astype(np.int32)
    for r0, r1 in [(0, 300), (7, 8), (150, 299)]:
        check(M, q, sc, zp, rows, cols, 8, blk, xq, xd, xbs, r0, r1, what=f"[{r0},{r1})")
    # the largest |sumi| of a 128-block: B = 255 (B' = 127) against zp = 0 and +-127 activations
    q2 = np.full((2, cols), 127, np.int8)
    z2 = np.zeros((2, cols // blk), np.uint8)
    sc2 = np.full((2, cols // blk), 1e-3, np.float32)
    W = tensor(M, q2, sc2, z2, 2, cols, 8, blk)
    X = M.BlkAct(dev(xq), dev(xd), dev(xbs), cols, blk)
    gs = torch.zeros((2, cols // blk), dtype=torch.int32, device=DEV)
    M.mlq_block_sumi_nbits(gs, W, X, 0, 2)
    torch.cuda.synchronize()
    g = gs.cpu().numpy()
    assert g[0, 0] == 255 * 127 * 128 and g[0, 1] == -255 * 127 * 128


def test_qwen_layer_pass_through_runner(M):
    """The bench's Qwen2.5-0.5B-shaped pass in both forms (4-bit blocks of
    128 with float32 scales; 8-bit signed-offset blocks of 32 with float16
    scales and zero points): every quantised input bit-exact against the
    oracle on the GPU's float vector, every product's y within the bound."""
    from block_quantized_decode_gb300.runner import NBitsRunner
    for wl in (I.qwen_layer_int4_blk128(), I.qwen_layer_int8_sq8()):
        r = NBitsRunner(wl, copies=1)
        r.step()
        torch.cuda.synchronize()
        for name, rows, cols, inp in wl.mats:
            xv = r.vec(inp).cpu().numpy()
            oq, od, obs = oracle.quantize_blk(xv, wl.blk)
            act = r.act[inp]
            assert np.array_equal(act.q.cpu().numpy(), oq), f"{wl.name}/{name}: quantised input differs"
            assert np.array_equal(act.d.cpu().numpy().view(np.uint32), od.view(np.uint32))
            assert np.array_equal(act.bsums.cpu().numpy(), obs)
            q, sc, zp = r.host[name]
            yo = oracle.matvec_nbits(q, sc, zp, rows, cols, wl.bits, wl.blk, oq, od)
            s_ = oracle.block_sumi_nbits(q, zp, rows, cols, wl.bits, wl.blk, oq)
            t = (s_.astype(np.float32) * sc.astype(np.float32)) * od[None, :]
            bound = REL * np.abs(t.astype(np.float64)).sum(axis=1)
            yg = r.y[name].cpu().numpy()
            assert np.all(np.abs(yg.astype(np.float64) - yo) <= bound), f"{wl.name}/{name}"


@pytest.mark.parametrize("bits,blk,f16,with_zp", COMBOS,
                         ids=[f"b{b}_blk{k}_{'f16' if f else 'f32'}{'_zp' if z else ''}" for b, k, f, z in COMBOS])
def test_nbits_phase_single_product_bitwise(M, bits, blk, f16, with_zp):
    """One product through mlq_nbits_phase (x quantised inside the launch)
    against mlq_quantize_blk + mlq_matvec_nbits: the same geometry and the
    same quantiser arithmetic, so y must be bit-identical."""
    rows, cols = 333, 896
    q, sc, zp = I.nbits_weights(rows, cols, bits, blk, f16, with_zp, seed=rows + bits + blk)
    x = I.activations(1, cols, seed=cols + bits)[0]
    W = tensor(M, q, sc, zp, rows, cols, bits, blk)
    y1 = torch.full((rows,), float("nan"), dtype=torch.float32, device=DEV)
    y2 = torch.full((rows,), float("nan"), dtype=torch.float32, device=DEV)
    M.mlq_nbits_phase(dev(x.astype(np.float32)), cols, [(W, y1)])
    M.mlq_matvec_nbits(y2, W, gpu_quantize_blk(M, x, blk), 0, rows)
    torch.cuda.synchronize()
    assert torch.equal(y1, y2), "the phase and the separate calls differ"


@pytest.mark.parametrize("bits,blk,f16,with_zp", [(4, 128, False, False), (8, 32, True, True)])
def test_nbits_phase_grouped_vs_oracle(M, bits, blk, f16, with_zp):
    """Products of one format sharing one float input in one launch: every y
    within the bound of the oracle on the oracle's quantisation of x."""
    cols = 896
    x = I.activations(1, cols, seed=bits * blk)[0]
    xq, xd, xbs = oracle.quantize_blk(x, blk)
    prods, host = [], []
    for i, rows in enumerate((896, 128, 77, 1)):
        q, sc, zp = I.nbits_weights(rows, cols, bits, blk, f16, with_zp, seed=200 + i)
        y = torch.full((rows,), float("nan"), dtype=torch.float32, device=DEV)
        prods.append((tensor(M, q, sc, zp, rows, cols, bits, blk), y))
        host.append((q, sc, zp, rows))
    M.mlq_nbits_phase(dev(x.astype(np.float32)), cols, prods)
    torch.cuda.synchronize()
    for (q, sc, zp, rows), (_, y) in zip(host, prods):
        yo = oracle.matvec_nbits(q, sc, zp, rows, cols, bits, blk, xq, xd)
        s_ = oracle.block_sumi_nbits(q, zp, rows, cols, bits, blk, xq)
        t = (s_.astype(np.float32) * sc.astype(np.float32)) * xd[None, :]
        bound = REL * np.abs(t.astype(np.float64)).sum(axis=1)
        yg = y.cpu().numpy()
        assert np.all(np.isfinite(yg)), f"{rows} rows: not every row written"
        assert np.all(np.abs(yg.astype(np.float64) - yo) <= bound + 1e-30), f"{rows}x{cols}"


def test_qwen_layer_phase_pass_through_runner(M):
    """The Qwen2.5-0.5B-shaped pass in both forms as phase launches (q|k|v,
    o, gate|up, down): every product's y within the bound of the oracle on
    the oracle's quantisation of the GPU's own float input."""
    from block_quantized_decode_gb300.runner import NBitsRunner
    for wl in (I.qwen_layer_int4_blk128(), I.qwen_layer_int8_sq8()):
        r = NBitsRunner(wl, copies=1)
        assert len(r.phases()) == 4
        r.step_phase()
        torch.cuda.synchronize()
        for name, rows, cols, inp in wl.mats:
            oq, od, obs = oracle.quantize_blk(r.vec(inp).cpu().numpy(), wl.blk)
            q, sc, zp = r.host[name]
            yo = oracle.matvec_nbits(q, sc, zp, rows, cols, wl.bits, wl.blk, oq, od)
            s_ = oracle.block_sumi_nbits(q, zp, rows, cols, wl.bits, wl.blk, oq)
            t = (s_.astype(np.float32) * sc.astype(np.float32)) * od[None, :]
            bound = REL * np.abs(t.astype(np.float64)).sum(axis=1)
            yg = r.y[name].cpu().numpy()
            assert np.all(np.abs(yg.astype(np.float64) - yo) <= bound), f"{wl.name}/{name}"
