"""The floating-point steps of a decode layer on the GPU against the oracle
(page "Legacy-ISA ML Inference Runtime -- Design Spec", Sec. 5 kernel
interface and Sec. 6 forward pass; Sec. 7: FP path relative error <= 1e-5).

Float outputs are compared with bounds derived from the arithmetic (written
in each test); every Q8_0 output must be the oracle's quantisation of the
GPU's own float result, bit for bit.  Inputs are seeded N(0, 1) vectors and
U[0.5, 1.5] norm weights, at TinyLlama's sizes and at ragged and maximum
ones.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import oracle  # noqa: E402

pytestmark = pytest.mark.gpu
U = 2.0 ** -24
TINY = np.float32(np.finfo(np.float32).tiny)


@pytest.fixture(scope="module")
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
    return torch.from_numpy(np.ascontiguousarray(a)).to("cuda")


def q8_out(M, n):
    return M.QAct(torch.zeros(n, dtype=torch.int8, device="cuda"),
                  torch.zeros(n // 32, dtype=torch.float32, device="cuda"), n, 1)


def assert_q8_of(M, qa, h_gpu, what):
    q, d = oracle.quantize_q8(h_gpu)
    assert np.array_equal(qa.q.cpu().numpy(), q), f"{what}: quant bytes"
    assert np.array_equal(qa.d.cpu().numpy().view(np.uint32), d.view(np.uint32)), f"{what}: scales"


def assert_rel(got, ref, rel, what, floor=TINY):
    got = got.astype(np.float64)
    ref = ref.astype(np.float64)
    bad = np.abs(got - ref) > rel * np.abs(ref) + floor
    assert not bad.any(), f"{what}: {bad.sum()} elements off, worst at {np.argmax(np.abs(got - ref))}"


@pytest.mark.parametrize("n", [32, 2048, 5632, 65536])
def test_rmsnorm_q8(M, n):
    """Error of the float32 result relative to each element: the sum of
    squares is a pairwise-shaped tree (ceil(log2 n) + 1 roundings), then
    mean, add eps, sqrt, divide and two products: below (log2 n + 8) u,
    under the page's 1e-5."""
    rng = np.random.default_rng(n)
    x = rng.standard_normal(n).astype(np.float32) * np.float32(3)
    w = rng.uniform(0.5, 1.5, n).astype(np.float32)
    o = torch.full((n,), float("nan"), device="cuda")
    oq = q8_out(M, n)
    M.mlq_rmsnorm(o, dev(x), dev(w), n, 1e-5, oq)
    h = o.cpu().numpy()
    ref = oracle.rmsnorm(x, w, 1e-5)
    assert_rel(h, ref, (math.log2(n) + 8) * U, f"rmsnorm n={n}")
    assert 1e-5 > (math.log2(n) + 8) * U
    assert_q8_of(M, oq, h, f"rmsnorm n={n}")
    # Q8 only (no float output), and float only
    oq2 = q8_out(M, n)
    M.mlq_rmsnorm(None, dev(x), dev(w), n, 1e-5, oq2)
    assert np.array_equal(oq2.q.cpu().numpy(), oq.q.cpu().numpy())
    o2 = torch.zeros(n, device="cuda")
    M.mlq_rmsnorm(o2, dev(x), dev(w), n, 1e-5)
    assert np.array_equal(o2.cpu().numpy(), h)


def test_add_rmsnorm(M):
    """x += y is one float32 addition per element (bit-exact), then the
    rmsnorm of the new x."""
    n = 2048
    rng = np.random.default_rng(7)
    x = rng.standard_normal(n).astype(np.float32)
    y = rng.standard_normal(n).astype(np.float32)
    w = rng.uniform(0.5, 1.5, n).astype(np.float32)
    xd = dev(x)
    o = torch.zeros(n, device="cuda")
    oq = q8_out(M, n)
    M.mlq_add_rmsnorm(xd, dev(y), dev(w), n, 1e-6, o, oq)
    xs = (x + y).astype(np.float32)
    assert np.array_equal(xd.cpu().numpy(), xs)
    h = o.cpu().numpy()
    assert_rel(h, oracle.rmsnorm(xs, w, 1e-6), (math.log2(n) + 8) * U, "add_rmsnorm")
    assert_q8_of(M, oq, h, "add_rmsnorm")


@pytest.mark.parametrize("n", [1, 100, 5632])
def test_add(M, n):
    rng = np.random.default_rng(n + 1)
    y = rng.standard_normal(n).astype(np.float32)
    x = rng.standard_normal(n).astype(np.float32)
    yd = dev(y)
    M.mlq_add(yd, dev(x), n)
    assert np.array_equal(yd.cpu().numpy(), oracle.add(y, x))


@pytest.mark.parametrize("n", [1, 7, 2048, 40000])
def test_softmax(M, n):
    """Per element: x - max in float32 is off by up to u |x - max|, which
    exp turns into that relative error; expf is within 2 ulp (4 u); the sum
    is a tree of ceil(log2 n) + 1 roundings; one division; the oracle rounds
    once: relative error below (|x - max| + log2 n + 8) u."""
    rng = np.random.default_rng(n + 2)
    x = (rng.standard_normal(n) * 4).astype(np.float32)
    xd = dev(x)
    M.mlq_softmax(xd, n)
    got = xd.cpu().numpy()
    rel = (np.abs(x.astype(np.float64) - x.max()) + math.log2(max(n, 2)) + 8) * U
    assert_rel(got, oracle.softmax(x), rel, f"softmax n={n}")
    assert abs(got.astype(np.float64).sum() - 1.0) < 1e-5


@pytest.mark.parametrize("n", [64, 5632])
def test_silu_mul_q8(M, n):
    """silu(g) u: expf (2 ulp: 4 u), an add, a division and a product, and
    the oracle's own rounding: relative error below 10 u.  Large |g|
    included: for g < -88 exp(-g) overflows float32 and silu(g) u becomes
    -0 while the exact value is below 1e-35 in magnitude, so an absolute
    floor of 100 FLT_MIN applies."""
    rng = np.random.default_rng(n + 3)
    g = (rng.standard_normal(n) * 4).astype(np.float32)
    g[:4] = [100.0, -100.0, 88.0, -90.0]
    u = rng.standard_normal(n).astype(np.float32)
    gd = dev(g)
    gq = q8_out(M, n)
    M.mlq_silu_mul(gd, dev(u), n, gq)
    got = gd.cpu().numpy()
    assert_rel(got, oracle.silu_mul(g, u), 10 * U, f"silu_mul n={n}", floor=100 * TINY)
    assert_q8_of(M, gq, got, f"silu_mul n={n}")


@pytest.mark.parametrize("max_seq,hd,theta", [(2048, 64, 10000.0), (300, 128, 500000.0), (5, 2, 10.0)])
def test_rope_tables(M, max_seq, hd, theta):
    """Both sides compute in double and round once: equal to within one
    float32 ulp of 1."""
    c = torch.zeros(max_seq * (hd // 2), device="cuda")
    s = torch.zeros_like(c)
    M.mlq_rope_tables(c, s, max_seq, hd, theta)
    rc, rs = oracle.rope_tables(max_seq, hd, theta)
    assert np.abs(c.cpu().numpy() - rc.reshape(-1)).max() <= 2 * U
    assert np.abs(s.cpu().numpy() - rs.reshape(-1)).max() <= 2 * U


@pytest.mark.parametrize("hd,nh,nkv,pos", [(64, 32, 4, 255), (128, 8, 8, 1000), (2, 3, 1, 7)])
def test_rope(M, hd, nh, nkv, pos):
    """Each rotated element is a*c -/+ b*s: two rounded products and one
    rounded add on the GPU (2 u (|a c| + |b s|)) against the oracle's once-
    rounded exact value (u |a c - b s|): below 3 u (|a c| + |b s|), tables
    shared with the oracle."""
    rng = np.random.default_rng(hd + nh + pos)
    c, s = oracle.rope_tables(pos + 1, hd, 10000.0)
    q = rng.standard_normal(nh * hd).astype(np.float32)
    k = rng.standard_normal(nkv * hd).astype(np.float32)
    v = rng.standard_normal(nkv * hd).astype(np.float32)
    rq, rk = oracle.rope(q, k, c[pos], s[pos], hd, nh, nkv)

    def bound(vec):
        # (a, b) -> (a c - b s, a s + b c): each element's own two terms
        a, b = vec[0::2].astype(np.float64), vec[1::2].astype(np.float64)
        cc = np.tile(c[pos].astype(np.float64), len(a) // len(c[pos]))
        ss = np.tile(s[pos].astype(np.float64), len(a) // len(c[pos]))
        e = np.empty(len(vec))
        e[0::2] = 3 * U * (np.abs(a * cc) + np.abs(b * ss)) + TINY
        e[1::2] = 3 * U * (np.abs(a * ss) + np.abs(b * cc)) + TINY
        return e

    qd, kd = dev(q), dev(k)
    M.mlq_rope(qd, kd, dev(c[pos]), dev(s[pos]), hd, nh, nkv)
    assert np.all(np.abs(qd.cpu().numpy().astype(np.float64) - rq) <= bound(q))
    assert np.all(np.abs(kd.cpu().numpy().astype(np.float64) - rk) <= bound(k))
    # the KV-cache form: k left as it is, rotated k and v written to the rows
    qd, kd = dev(q), dev(k)
    ko, vo = torch.zeros(nkv * hd, device="cuda"), torch.zeros(nkv * hd, device="cuda")
    M.mlq_rope(qd, kd, dev(c[pos]), dev(s[pos]), hd, nh, nkv, ko, dev(v), vo)
    assert np.array_equal(kd.cpu().numpy(), k)
    assert np.all(np.abs(ko.cpu().numpy().astype(np.float64) - rk) <= bound(k))
    assert np.array_equal(vo.cpu().numpy(), v)


@pytest.mark.parametrize("n_pos,hd,nh,nkv", [(1, 64, 32, 4), (17, 64, 32, 4), (256, 64, 32, 4),
                                             (2049, 128, 8, 2), (300, 32, 4, 4), (64, 256, 2, 1)])
def test_attention(M, n_pos, hd, nh, nkv):
    """Bound per output element i of head h, derived from the arithmetic:
    each score's dot product carries at most (hd/4 + 2) u of sum |q_j K_tj|
    (four partial sums of hd/4 fused products, added pairwise), plus the
    division by sqrt(hd); a score error e moves each weight by at most 2e
    relative, and
    exp, the sum tree and the normalisation add (log2 n_pos + 8) u; the
    weighted sum of V (8 warps over slices of n_pos / 8 positions, then the
    8 partials in order) adds (n_pos / 8 + 9) u.  So |o - o_ref| <=
    (2 E + (log2 n_pos + n_pos / 8 + 17) u) * sum_t p_t |V_ti|."""
    rng = np.random.default_rng(n_pos * 7 + hd)
    kv_dim = nkv * hd
    q = rng.standard_normal(nh * hd).astype(np.float32)
    kc = rng.standard_normal((n_pos, kv_dim)).astype(np.float32)
    vc = rng.standard_normal((n_pos, kv_dim)).astype(np.float32)
    o = torch.full((nh * hd,), float("nan"), device="cuda")
    oq = q8_out(M, nh * hd) if hd % 32 == 0 else None
    M.mlq_attention(o, dev(q), dev(kc), dev(vc), n_pos, hd, nh, nkv, oq)
    got = o.cpu().numpy()
    assert_attention_close(got, q, kc, vc, n_pos, hd, nh, nkv, "attention")
    if oq is not None:
        assert_q8_of(M, oq, got, "attention")


def assert_attention_close(got, q, kc, vc, n_pos, hd, nh, nkv, what):
    """The bound of test_attention, per output element."""
    ref = oracle.attention(q, kc, vc, n_pos, hd, nh, nkv)
    for h in range(nh):
        g = h // (nh // nkv)
        qh = q[h * hd:(h + 1) * hd].astype(np.float64)
        K = kc[:n_pos, g * hd:(g + 1) * hd].astype(np.float64)
        V = vc[:n_pos, g * hd:(g + 1) * hd].astype(np.float64)
        sabs = np.abs(K * qh).sum(1) / math.sqrt(hd)
        E = (hd / 4 + 8) * U * sabs.max()
        s = K @ qh / math.sqrt(hd)
        p = np.exp(s - s.max())
        p /= p.sum()
        pv = (p[:, None] * np.abs(V)).sum(0)
        tol = (2 * E + (math.log2(max(n_pos, 2)) + n_pos / 8 + 17) * U) * pv + TINY
        err = np.abs(got[h * hd:(h + 1) * hd].astype(np.float64) - ref[h * hd:(h + 1) * hd])
        assert np.all(err <= tol), f"{what} head {h}: worst {err.max()} vs tol {tol[np.argmax(err)]}"


# ---------------------------------------------------------------------------
# a whole decode layer, one token, checked launch by launch
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("pos", [0, 255])
def test_decode_layer_step(M, pos):
    """The TinyLlama-shaped layer of the forward pass (Design Spec Sec. 6)
    for one token at position pos, through the same C-ABI calls the bench
    times.  After every launch its outputs are checked against the oracle
    run on the GPU's own inputs of that launch, so a difference allowed
    upstream is never counted downstream."""
    from block_quantized_decode_gb300 import inputs as I
    from block_quantized_decode_gb300.layer import DecodeLayer
    from tests import parity as PT
    s = I.tinyllama_decode_layer(pos=pos)
    L = DecodeLayer(s)
    L.x.copy_(torch.from_numpy(L.x_in))
    hd, half, dim = s.head_dim, s.head_dim // 2, s.dim
    snap = {}
    cpu = lambda t: t.detach().cpu().numpy().copy()

    def product(name, xq, xd, y):
        q, d, rows, cols = L.host[name]
        PT.check_matvec(s.wtype, q, d, rows, cols, xq, xd, 0, rows, y_gpu=y, what=f"layer {name}")

    def after(stage):
        torch.cuda.synchronize()
        if stage == "rmsnorm_att":
            h = cpu(L.h1)
            assert_rel(h, oracle.rmsnorm(L.x_in, L.att_norm, s.norm_eps), (math.log2(dim) + 8) * U, stage)
            assert_q8_of(M, L.h1q, h, stage)
            snap["h1q"] = (cpu(L.h1q.q), cpu(L.h1q.d))
        elif stage == "qkv":
            xq, xd = snap["h1q"]
            for name, y in (("wq", L.q), ("wk", L.k), ("wv", L.v)):
                product(name, xq, xd, cpu(y))
            snap["q"], snap["k"], snap["v"] = cpu(L.q), cpu(L.k), cpu(L.v)
        elif stage == "rope":
            c, sn = oracle.rope_tables(pos + 1, hd, s.rope_theta)
            assert np.abs(cpu(L.cos)[pos * half:(pos + 1) * half] - c[pos]).max() <= 2 * U
            rq, rk = oracle.rope(snap["q"], snap["k"], cpu(L.cos)[pos * half:(pos + 1) * half],
                                 cpu(L.sin)[pos * half:(pos + 1) * half], hd, s.n_heads, s.n_kv_heads)
            assert np.allclose(cpu(L.q), rq, rtol=0, atol=6 * U * np.abs(snap["q"]).max())
            assert np.allclose(cpu(L.kc[pos]), rk, rtol=0, atol=6 * U * np.abs(snap["k"]).max())
            assert np.array_equal(cpu(L.vc[pos]), snap["v"])
            if pos:
                assert np.array_equal(cpu(L.kc[:pos]), L.k_hist)
        elif stage == "attention":
            o = cpu(L.o)
            assert_attention_close(o, cpu(L.q), cpu(L.kc), cpu(L.vc), pos + 1, hd, s.n_heads,
                                   s.n_kv_heads, stage)
            assert_q8_of(M, L.oq, o, stage)
            snap["oq"] = (cpu(L.oq.q), cpu(L.oq.d))
            snap["x"] = cpu(L.x)
        elif stage == "wo":
            product("wo", *snap["oq"], cpu(L.yo))
            snap["yo"] = cpu(L.yo)
        elif stage == "add_rmsnorm_ffn":
            xm = (snap["x"] + snap["yo"]).astype(np.float32)
            assert np.array_equal(cpu(L.x), xm)
            h = cpu(L.h2)
            assert_rel(h, oracle.rmsnorm(xm, L.ffn_norm, s.norm_eps), (math.log2(dim) + 8) * U, stage)
            assert_q8_of(M, L.h2q, h, stage)
            snap["h2q"] = (cpu(L.h2q.q), cpu(L.h2q.d))
            snap["xm"] = xm
        elif stage == "ffn":
            for name, y in (("w1", L.g), ("w3", L.u)):
                product(name, *snap["h2q"], cpu(y))
            snap["g"], snap["u"] = cpu(L.g), cpu(L.u)
        elif stage == "silu_mul":
            g = cpu(L.g)
            assert_rel(g, oracle.silu_mul(snap["g"], snap["u"]), 10 * U, stage)
            assert_q8_of(M, L.gq, g, stage)
            snap["gq"] = (cpu(L.gq.q), cpu(L.gq.d))
        elif stage == "down":
            product("w2", *snap["gq"], cpu(L.y2))
            snap["y2"] = cpu(L.y2)
        elif stage == "add":
            assert np.array_equal(cpu(L.x), (snap["xm"] + snap["y2"]).astype(np.float32))
        snap.setdefault("stages", []).append(stage)

    L.step(after=after)
    assert snap["stages"] == ["rmsnorm_att", "qkv", "rope", "attention", "wo", "add_rmsnorm_ffn",
                              "ffn", "silu_mul", "down", "add"]
    assert np.all(np.isfinite(cpu(L.x)))
