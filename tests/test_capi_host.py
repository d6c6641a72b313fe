"""The C-ABI library on the host (no GPU needed): it builds for sm_103a,
loads, exports every symbol include/mlq.h declares, and rejects bad
arguments with the documented status before touching the device
(page "Legacy-ISA ML Inference Runtime -- Design Spec", Sec. 6 "Error
handling": a status, never an abort; loader checks K % 32 == 0)."""
import ctypes
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def M():
    from block_quantized_decode_gb300 import build as B
    B.build()
    import block_quantized_decode_gb300 as pkg
    pkg.lib()
    return pkg


def header_symbols():
    src = open(os.path.join(ROOT, "include", "mlq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mlq_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(M):
    declared = header_symbols()
    assert len(declared) >= 9
    out = subprocess.run(["nm", "-D", "--defined-only", M.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (mlq_[a-z0-9_]+)$", out, flags=re.M))
    missing = [s for s in declared if s not in exported]
    assert not missing, missing
    assert sorted(M.EXPORTS) == declared
    for s in declared:
        getattr(M.lib(), s)


def test_status_strings(M):
    names = ["MLQ_OK", "MLQ_E_SHAPE", "MLQ_E_ALIGN", "MLQ_E_TYPE", "MLQ_E_NULL", "MLQ_E_ARCH",
             "MLQ_E_CUDA", "MLQ_E_TIMEOUT", "MLQ_E_BOUNDS"]
    for i, n in enumerate(names):
        assert M.mlq_status_str(i) == n
    assert M.mlq_status_str(99) == "MLQ_E_UNKNOWN"


# fake, 256-byte aligned "device" addresses: validation never dereferences them
A = 1 << 20


def qt(q=A, d=2 * A, rows=64, cols=128, t=1):
    from block_quantized_decode_gb300.binding import _QTensor
    return _QTensor(q, d, rows, cols, t)


def qa(q=3 * A, d=4 * A, n=128, m=1):
    from block_quantized_decode_gb300.binding import _QAct
    return _QAct(q, d, n, m)


def call(M, name, *args):
    return M.binding.raw_call(name, *args)


def mv(M, name="mlq_matvec_q4", y=5 * A, W=None, x=None, r0=0, r1=64):
    W = qt() if W is None else W
    x = qa() if x is None else x
    return call(M, name, y, ctypes.byref(W), ctypes.byref(x), r0, r1, None)


def test_validation_matvec(M):
    assert mv(M, y=None) == M.MLQ_E_NULL
    assert call(M, "mlq_matvec_q4", 5 * A, None, ctypes.byref(qa()), 0, 1, None) == M.MLQ_E_NULL
    assert mv(M, W=qt(q=0)) == M.MLQ_E_NULL
    assert mv(M, x=qa(d=0)) == M.MLQ_E_NULL
    assert mv(M, W=qt(t=0)) == M.MLQ_E_TYPE            # Q8_0 tensor to the Q4_0 entry
    assert mv(M, "mlq_matvec_q8") == M.MLQ_E_TYPE      # Q4_0 tensor to the Q8_0 entry
    assert mv(M, W=qt(t=7)) == M.MLQ_E_TYPE
    assert mv(M, W=qt(cols=100), x=qa(n=100)) == M.MLQ_E_SHAPE   # K % 32 != 0
    assert mv(M, W=qt(cols=0), x=qa(n=0)) == M.MLQ_E_SHAPE
    assert mv(M, W=qt(cols=65568), x=qa(n=65568)) == M.MLQ_E_SHAPE  # > MLQ_MAX_COLS
    assert mv(M, x=qa(n=96)) == M.MLQ_E_SHAPE          # x->n != W->cols
    assert mv(M, x=qa(m=2)) == M.MLQ_E_SHAPE           # M = 1 entry
    assert mv(M, r0=-1) == M.MLQ_E_SHAPE
    assert mv(M, r0=5, r1=4) == M.MLQ_E_SHAPE
    assert mv(M, r1=65) == M.MLQ_E_SHAPE
    assert mv(M, W=qt(q=A + 8)) == M.MLQ_E_ALIGN
    assert mv(M, W=qt(d=2 * A + 4)) == M.MLQ_E_ALIGN
    assert mv(M, x=qa(q=3 * A + 1)) == M.MLQ_E_ALIGN
    assert mv(M, y=5 * A + 2) == M.MLQ_E_ALIGN


def test_validation_quantize(M):
    q = lambda out, x=6 * A, k=128: call(M, "mlq_quantize_q8", ctypes.byref(out), x, k, None)
    assert q(qa(), x=None) == M.MLQ_E_NULL
    assert q(qa(q=0)) == M.MLQ_E_NULL
    assert q(qa(n=96), k=96 + 1) == M.MLQ_E_SHAPE
    assert q(qa(n=128), k=96) == M.MLQ_E_SHAPE
    assert q(qa(m=0)) == M.MLQ_E_SHAPE
    assert q(qa(), x=6 * A + 4) == M.MLQ_E_ALIGN
    assert q(qa(d=4 * A + 8)) == M.MLQ_E_ALIGN


def test_validation_gemm_and_sumi(M):
    def g(Y=5 * A, ldy=64, W=None, X=None, Mrows=4, r0=0, r1=64):
        W = qt() if W is None else W
        X = qa(m=4) if X is None else X
        return call(M, "mlq_gemm_q4_small_m", Y, ldy, ctypes.byref(W), ctypes.byref(X), Mrows,
                    r0, r1, None)
    assert g(Y=None) == M.MLQ_E_NULL
    assert g(W=qt(t=0)) == M.MLQ_E_TYPE
    assert g(Mrows=0, X=qa(m=0)) == M.MLQ_E_SHAPE
    assert g(Mrows=17, X=qa(m=17)) == M.MLQ_E_SHAPE
    assert g(Mrows=4, X=qa(m=3)) == M.MLQ_E_SHAPE
    assert g(ldy=63) == M.MLQ_E_SHAPE
    assert g(Y=5 * A + 1) == M.MLQ_E_ALIGN
    s = lambda **k: call(M, "mlq_block_sumi", k.get("out", 5 * A), ctypes.byref(k.get("W", qt())),
                         ctypes.byref(qa()), 0, 64, None)
    assert s(out=None) == M.MLQ_E_NULL
    assert s(W=qt(t=9)) == M.MLQ_E_TYPE


def _cuda_available():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.mark.skipif(_cuda_available(), reason="checks the no-device path")
def test_valid_call_without_device_is_arch_error(M):
    # the fake addresses above must never reach a real device
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert M.binding.raw_call("mlq_init") == M.MLQ_E_ARCH
    assert mv(M) == M.MLQ_E_ARCH


def test_arch_guard_with_faked_capability():
    """A device that reports another compute capability is refused with
    MLQ_E_ARCH (the library is built for sm_103a only)."""
    code = ("import block_quantized_decode_gb300 as M; import sys; "
            "sys.exit(M.binding.raw_call('mlq_init'))")
    env = dict(os.environ, MLQ_FAKE_CC="9.0", PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "-c", code], env=env, cwd=ROOT, timeout=300)
    assert r.returncode == 5  # MLQ_E_ARCH


def test_debug_wait_limit_hook(M):
    M.mlq_debug_set_wait_limit_ns(10 ** 9)


def test_validation_chain(M):
    from block_quantized_decode_gb300.binding import _ChainPhase, _ChainProduct
    P = _ChainPhase
    R = _ChainProduct

    def run(phases, prods, ws=7 * A, wsb=64):
        pa = (P * max(1, len(phases)))(*phases)
        ra = (R * max(1, len(prods)))(*prods)
        return call(M, "mlq_decode_chain", pa, len(phases), ra, len(prods), ws, wsb, None)

    good_prod = R(qt(cols=256), 5 * A)
    good_phase = P(6 * A, 256, 0, 1, None, None)
    assert M.mlq_chain_workspace_bytes(3) == 16
    assert run([], [good_prod]) == M.MLQ_E_SHAPE
    assert run([good_phase], []) == M.MLQ_E_SHAPE
    assert run([good_phase], [R(qt(cols=96), 5 * A)]) == M.MLQ_E_SHAPE      # not a multiple of 128
    assert run([good_phase], [R(qt(cols=256), None)]) == M.MLQ_E_NULL
    assert run([good_phase, P(6 * A, 256, 0, 2, None, None)], [good_prod]) == M.MLQ_E_SHAPE
    assert run([P(6 * A, 128, 0, 1, None, None)], [good_prod]) == M.MLQ_E_SHAPE  # n != cols
    assert run([good_phase], [good_prod, R(qt(cols=256, t=0), 5 * A)]) == M.MLQ_E_TYPE
    assert run([P(6 * A + 4, 256, 0, 1, None, None)], [good_prod]) == M.MLQ_E_ALIGN
    assert run([P(6 * A, 256, 0, 1, 8 * A, None)], [good_prod]) == M.MLQ_E_NULL
    assert run([good_phase], [good_prod], ws=None) == M.MLQ_E_NULL
    assert run([good_phase], [good_prod], ws=7 * A + 2) == M.MLQ_E_ALIGN
    assert run([good_phase], [good_prod], wsb=4) == M.MLQ_E_SHAPE
    assert run([good_phase] * 25, [good_prod]) == M.MLQ_E_SHAPE


def test_validation_fused(M):
    from block_quantized_decode_gb300.binding import _ChainProduct
    R = _ChainProduct

    def run(prods, x=6 * A, n=256, xq=None, xd=None, flags=0):
        ra = (R * max(1, len(prods)))(*prods)
        return call(M, "mlq_matvec_fused", x, n, ra, len(prods), xq, xd, flags, None)

    good = R(qt(cols=256), 5 * A)
    assert run([good], x=None) == M.MLQ_E_NULL
    assert run([]) == M.MLQ_E_SHAPE
    assert run([good] * 9) == M.MLQ_E_SHAPE
    assert run([good], n=250) == M.MLQ_E_SHAPE
    assert run([R(qt(cols=128), 5 * A)]) == M.MLQ_E_SHAPE
    assert run([good, R(qt(cols=256, t=0), 5 * A)]) == M.MLQ_E_TYPE
    assert run([good], x=6 * A + 4) == M.MLQ_E_ALIGN
    assert run([good], xq=8 * A) == M.MLQ_E_NULL
    assert run([R(qt(cols=256), 5 * A + 1)]) == M.MLQ_E_ALIGN
    assert run([good], flags=2) == M.MLQ_E_SHAPE


def test_validation_phase(M):
    from block_quantized_decode_gb300.binding import _PhaseInput, _PhaseProduct
    R = _PhaseProduct

    def run(prods, x=6 * A, xq=None, xd=None, n=256, xq_out=None, xd_out=None, flags=0,
            inp=True, pf=None, pfb=None, npf=0):
        ra = (R * max(1, len(prods)))(*prods)
        pin = ctypes.byref(_PhaseInput(x, xq, xd, n, xq_out, xd_out)) if inp else None
        return call(M, "mlq_decode_phase", pin, ra, len(prods), pf, pfb, npf, flags, None)

    good = R(qt(cols=256), 5 * A, None, None)
    quant = R(qt(cols=256, rows=64), 5 * A, 9 * A, 10 * A)
    assert run([good], inp=False) == M.MLQ_E_NULL
    assert run([good], x=None) == M.MLQ_E_NULL                        # no input at all
    assert run([good], x=None, xq=8 * A) == M.MLQ_E_NULL              # xq without xd
    assert run([good], xq=8 * A, xd=11 * A) == M.MLQ_E_SHAPE          # two inputs
    assert run([good], x=None, xq=8 * A, xd=11 * A, xq_out=12 * A, xd_out=13 * A) == M.MLQ_E_SHAPE
    assert run([good], xq_out=12 * A) == M.MLQ_E_NULL
    assert run([]) == M.MLQ_E_SHAPE
    assert run([good] * 9) == M.MLQ_E_SHAPE
    assert run([good], n=250) == M.MLQ_E_SHAPE
    assert run([R(qt(cols=128), 5 * A, None, None)]) == M.MLQ_E_SHAPE
    assert run([good, R(qt(cols=256, t=0), 5 * A, None, None)]) == M.MLQ_E_TYPE
    assert run([good], x=6 * A + 4) == M.MLQ_E_ALIGN
    assert run([good], x=None, xq=8 * A + 8, xd=11 * A) == M.MLQ_E_ALIGN
    assert run([R(qt(cols=256), 5 * A, 9 * A, None)]) == M.MLQ_E_NULL  # yq without yd
    assert run([R(qt(cols=256), 5 * A, 9 * A + 4, 10 * A)]) == M.MLQ_E_ALIGN
    assert run([quant, R(qt(cols=256, rows=40), 5 * A, None, None)]) == M.MLQ_E_SHAPE  # 40 % 32
    assert run([R(qt(cols=256, rows=33), 5 * A, 9 * A, 10 * A)]) == M.MLQ_E_SHAPE
    assert run([good], flags=4) == M.MLQ_E_SHAPE                      # unknown flag
    assert run([good], flags=M.MLQ_F_STATIC_INPUT | M.MLQ_F_STATIC_WEIGHTS) == M.MLQ_E_ARCH  # valid
    ptrs = (ctypes.c_void_p * 17)(*([12 * A] * 17))
    sizes = (ctypes.c_size_t * 17)(*([4096] * 17))
    assert run([good], pf=ptrs, pfb=sizes, npf=17) == M.MLQ_E_SHAPE   # > MLQ_PHASE_MAX_PREFETCH
    assert run([good], pf=ptrs, pfb=sizes, npf=-1) == M.MLQ_E_SHAPE
    assert run([good], pf=None, pfb=sizes, npf=2) == M.MLQ_E_NULL
    assert run([good], pf=ptrs, pfb=None, npf=2) == M.MLQ_E_NULL
    nul = (ctypes.c_void_p * 2)(12 * A, None)
    assert run([good], pf=nul, pfb=sizes, npf=2) == M.MLQ_E_NULL      # bytes > 0 at NULL


def test_validation_layer_steps(M):
    """The decode-layer steps reject bad arguments before touching the device."""
    B = ctypes.byref
    x, w, o = 5 * A, 6 * A, 7 * A
    # rmsnorm / add_rmsnorm
    assert call(M, "mlq_rmsnorm", None, x, w, 256, 1e-5, None, None) == M.MLQ_E_NULL   # no output
    assert call(M, "mlq_rmsnorm", o, None, w, 256, 1e-5, None, None) == M.MLQ_E_NULL
    assert call(M, "mlq_rmsnorm", o, x, w, 0, 1e-5, None, None) == M.MLQ_E_SHAPE
    assert call(M, "mlq_rmsnorm", o, x, w, 256, -1.0, None, None) == M.MLQ_E_SHAPE
    assert call(M, "mlq_rmsnorm", o, x, w, 256, float("nan"), None, None) == M.MLQ_E_SHAPE
    assert call(M, "mlq_rmsnorm", o + 2, x, w, 256, 1e-5, None, None) == M.MLQ_E_ALIGN
    assert call(M, "mlq_rmsnorm", o, x, w, 250, 1e-5, B(qa(n=250)), None) == M.MLQ_E_SHAPE  # Q8 needs n % 32
    assert call(M, "mlq_rmsnorm", o, x, w, 256, 1e-5, B(qa(n=128)), None) == M.MLQ_E_SHAPE  # qa->n != n
    assert call(M, "mlq_rmsnorm", o, x, w, 256, 1e-5, B(qa(n=256, m=2)), None) == M.MLQ_E_SHAPE
    assert call(M, "mlq_rmsnorm", o, x, w, 256, 1e-5, B(qa(q=3 * A + 8, n=256)), None) == M.MLQ_E_ALIGN
    assert call(M, "mlq_rmsnorm", o, x, w, 256, 1e-5, B(qa(q=None, n=256)), None) == M.MLQ_E_NULL
    assert call(M, "mlq_add_rmsnorm", x, None, w, 256, 1e-5, o, None, None) == M.MLQ_E_NULL
    assert call(M, "mlq_add_rmsnorm", x, o, w, 256, 1e-5, None, None, None) == M.MLQ_E_NULL
    # add, softmax, silu_mul
    assert call(M, "mlq_add", None, x, 16, None) == M.MLQ_E_NULL
    assert call(M, "mlq_add", o, x, 0, None) == M.MLQ_E_SHAPE
    assert call(M, "mlq_softmax", None, 16, None) == M.MLQ_E_NULL
    assert call(M, "mlq_softmax", o, 70000, None) == M.MLQ_E_SHAPE
    assert call(M, "mlq_silu_mul", o, None, 64, None, None) == M.MLQ_E_NULL
    assert call(M, "mlq_silu_mul", o, x, 64, B(qa(n=32)), None) == M.MLQ_E_SHAPE
    # rope tables and rope
    assert call(M, "mlq_rope_tables", o, None, 16, 64, 1e4, None) == M.MLQ_E_NULL
    assert call(M, "mlq_rope_tables", o, x, 16, 63, 1e4, None) == M.MLQ_E_SHAPE      # odd head_dim
    assert call(M, "mlq_rope_tables", o, x, 0, 64, 1e4, None) == M.MLQ_E_SHAPE
    assert call(M, "mlq_rope_tables", o, x, 16, 64, 0.0, None) == M.MLQ_E_SHAPE
    rope = lambda **k: call(M, "mlq_rope", k.get("q", o), k.get("k", x), k.get("c", w), 8 * A,
                            k.get("hd", 64), k.get("nh", 32), k.get("nkv", 4), k.get("ko", None),
                            k.get("v", None), k.get("vo", None), None)
    assert rope(q=None) == M.MLQ_E_NULL
    assert rope(v=9 * A) == M.MLQ_E_NULL                     # v without v_out
    assert rope(nkv=5) == M.MLQ_E_SHAPE                      # 32 % 5
    assert rope(hd=512) == M.MLQ_E_SHAPE
    assert rope(ko=9 * A + 1) == M.MLQ_E_ALIGN
    # attention
    att = lambda **k: call(M, "mlq_attention", k.get("o", o), k.get("oq", None), x, w, 8 * A,
                           k.get("npos", 17), k.get("hd", 64), k.get("nh", 32), k.get("nkv", 4), None)
    assert att(o=None) == M.MLQ_E_NULL
    assert att(npos=0) == M.MLQ_E_SHAPE
    assert att(npos=40000) == M.MLQ_E_SHAPE
    assert att(nkv=3) == M.MLQ_E_SHAPE
    assert att(hd=48, oq=B(qa(n=48 * 32))) == M.MLQ_E_SHAPE  # Q8 output needs head_dim % 32
    assert att(oq=B(qa(n=1024))) == M.MLQ_E_SHAPE            # n_heads * head_dim = 2048


def test_validation_q4k(M):
    from block_quantized_decode_gb300.binding import _Q4KTensor, _Q8KAct

    def kt(q=A, s_=2 * A, d=7 * A, dmin=8 * A, rows=64, cols=512):
        return _Q4KTensor(q, s_, d, dmin, rows, cols)

    def ka(q=3 * A, d=4 * A, bs=9 * A, n=512):
        return _Q8KAct(q, d, bs, n)

    def mvk(y=5 * A, W=None, x=None, r0=0, r1=64):
        W = kt() if W is None else W
        x = ka() if x is None else x
        return call(M, "mlq_matvec_q4k", y, ctypes.byref(W), ctypes.byref(x), r0, r1, None)

    assert mvk(y=None) == M.MLQ_E_NULL
    assert mvk(W=kt(s_=0)) == M.MLQ_E_NULL
    assert mvk(W=kt(dmin=0)) == M.MLQ_E_NULL
    assert mvk(x=ka(bs=0)) == M.MLQ_E_NULL
    assert mvk(W=kt(cols=384), x=ka(n=384)) == M.MLQ_E_SHAPE       # not whole super-blocks
    assert mvk(W=kt(cols=65792), x=ka(n=65792)) == M.MLQ_E_SHAPE   # > MLQ_MAX_COLS
    assert mvk(x=ka(n=256)) == M.MLQ_E_SHAPE
    assert mvk(r0=3, r1=2) == M.MLQ_E_SHAPE
    assert mvk(r1=65) == M.MLQ_E_SHAPE
    assert mvk(W=kt(q=A + 8)) == M.MLQ_E_ALIGN
    assert mvk(W=kt(s_=2 * A + 4)) == M.MLQ_E_ALIGN
    assert mvk(W=kt(d=7 * A + 2)) == M.MLQ_E_ALIGN
    assert mvk(x=ka(bs=9 * A + 4)) == M.MLQ_E_ALIGN
    assert mvk(y=5 * A + 1) == M.MLQ_E_ALIGN
    sums = lambda i=10 * A, m=11 * A: call(M, "mlq_block_sums_q4k", i, m, ctypes.byref(kt()),
                                           ctypes.byref(ka()), 0, 64, None)
    assert sums(m=None) == M.MLQ_E_NULL
    assert sums(i=10 * A + 2) == M.MLQ_E_ALIGN
    qk = lambda out, x=6 * A, k=512: call(M, "mlq_quantize_q8k", ctypes.byref(out), x, k, None)
    assert qk(ka(), x=None) == M.MLQ_E_NULL
    assert qk(ka(bs=0)) == M.MLQ_E_NULL
    assert qk(ka(n=480), k=480) == M.MLQ_E_SHAPE
    assert qk(ka(n=512), k=256) == M.MLQ_E_SHAPE
    assert qk(ka(), x=6 * A + 4) == M.MLQ_E_ALIGN
    assert qk(ka(d=4 * A + 4)) == M.MLQ_E_ALIGN
    # the Q4_K-style phase: products sharing one float input
    from block_quantized_decode_gb300.binding import _Q4KProduct

    def ph(x=6 * A, k=512, prods=None, n=None, flags=0):
        prods = [_Q4KProduct(kt(), 5 * A)] if prods is None else prods
        arr = (_Q4KProduct * max(1, len(prods)))(*prods)
        return call(M, "mlq_q4k_phase", x, k, arr, len(prods) if n is None else n, flags, None)

    assert ph(x=None) == M.MLQ_E_NULL
    assert ph(flags=M.MLQ_F_STATIC_WEIGHTS) == M.MLQ_E_SHAPE  # only MLQ_F_STATIC_INPUT
    assert ph(flags=4) == M.MLQ_E_SHAPE
    assert ph(prods=[_Q4KProduct(kt(), 0)]) == M.MLQ_E_NULL
    assert ph(prods=[_Q4KProduct(kt(dmin=0), 5 * A)]) == M.MLQ_E_NULL
    assert ph(n=0) == M.MLQ_E_SHAPE
    assert ph(prods=[_Q4KProduct(kt(), 5 * A)] * 5) == M.MLQ_E_SHAPE  # at most 4 products
    assert ph(k=480) == M.MLQ_E_SHAPE
    assert ph(prods=[_Q4KProduct(kt(), 5 * A), _Q4KProduct(kt(cols=768), 12 * A)]) == M.MLQ_E_SHAPE
    assert ph(prods=[_Q4KProduct(kt(rows=-1), 5 * A)]) == M.MLQ_E_SHAPE
    assert ph(x=6 * A + 4) == M.MLQ_E_ALIGN
    assert ph(prods=[_Q4KProduct(kt(q=A + 8), 5 * A)]) == M.MLQ_E_ALIGN
    assert ph(prods=[_Q4KProduct(kt(), 5 * A + 2)]) == M.MLQ_E_ALIGN


def test_validation_nbits(M):
    from block_quantized_decode_gb300.binding import _BlkAct, _NBitsTensor

    def nt(q=A, sc=2 * A, zp=0, rows=64, cols=896, bits=4, blk=128, f16=0, sld=8, zld=0):
        return _NBitsTensor(q, sc, zp or None, rows, cols, bits, blk, f16, sld, zld)

    def ba(q=3 * A, d=4 * A, bs=9 * A, n=896, blk=128):
        return _BlkAct(q, d, bs, n, blk)

    def mvn(y=5 * A, W=None, x=None, r0=0, r1=64):
        W = nt() if W is None else W
        x = ba() if x is None else x
        return call(M, "mlq_matvec_nbits", y, ctypes.byref(W), ctypes.byref(x), r0, r1, None)

    assert mvn(y=None) == M.MLQ_E_NULL
    assert mvn(W=nt(sc=0)) == M.MLQ_E_NULL
    assert mvn(x=ba(bs=0)) == M.MLQ_E_NULL
    assert mvn(W=nt(bits=2)) == M.MLQ_E_TYPE
    assert mvn(W=nt(f16=2)) == M.MLQ_E_TYPE
    assert mvn(W=nt(zp=6 * A, zld=16)) == M.MLQ_E_TYPE                # zero points on 4-bit
    assert mvn(W=nt(blk=64), x=ba(blk=64)) == M.MLQ_E_SHAPE
    assert mvn(W=nt(cols=960), x=ba(n=960)) == M.MLQ_E_SHAPE          # not whole blocks of 128
    assert mvn(x=ba(blk=32)) == M.MLQ_E_SHAPE                         # block lengths differ
    assert mvn(W=nt(sld=6)) == M.MLQ_E_SHAPE                          # stride < 7 blocks
    assert mvn(W=nt(sld=7)) == M.MLQ_E_SHAPE                          # 28-byte rows
    assert mvn(W=nt(bits=8, zp=6 * A, zld=8)) == M.MLQ_E_SHAPE        # zero-point rows not 16 B
    assert mvn(r1=65) == M.MLQ_E_SHAPE
    assert mvn(W=nt(q=A + 8)) == M.MLQ_E_ALIGN
    assert mvn(W=nt(bits=8, zp=6 * A + 4, zld=16)) == M.MLQ_E_ALIGN
    assert mvn(x=ba(d=4 * A + 2)) == M.MLQ_E_ALIGN
    assert call(M, "mlq_block_sumi_nbits", None, ctypes.byref(nt()), ctypes.byref(ba()), 0, 64,
                None) == M.MLQ_E_NULL
    qb = lambda out, x=6 * A, k=896: call(M, "mlq_quantize_blk", ctypes.byref(out), x, k, None)
    assert qb(ba(), x=None) == M.MLQ_E_NULL
    assert qb(ba(blk=64)) == M.MLQ_E_SHAPE
    assert qb(ba(n=960), k=960) == M.MLQ_E_SHAPE
    assert qb(ba(), x=6 * A + 8) == M.MLQ_E_ALIGN
    # the block-length phase: products of one format sharing one float input
    from block_quantized_decode_gb300.binding import _NBitsProduct

    def ph(x=6 * A, k=896, prods=None, n=None, flags=0):
        prods = [_NBitsProduct(nt(), 5 * A)] if prods is None else prods
        arr = (_NBitsProduct * max(1, len(prods)))(*prods)
        return call(M, "mlq_nbits_phase", x, k, arr, len(prods) if n is None else n, flags, None)

    assert ph(x=None) == M.MLQ_E_NULL
    assert ph(flags=M.MLQ_F_STATIC_WEIGHTS) == M.MLQ_E_SHAPE  # only MLQ_F_STATIC_INPUT
    assert ph(flags=4) == M.MLQ_E_SHAPE
    assert ph(prods=[_NBitsProduct(nt(), 0)]) == M.MLQ_E_NULL
    assert ph(prods=[_NBitsProduct(nt(sc=0), 5 * A)]) == M.MLQ_E_NULL
    assert ph(n=0) == M.MLQ_E_SHAPE
    assert ph(prods=[_NBitsProduct(nt(), 5 * A)] * 5) == M.MLQ_E_SHAPE
    assert ph(prods=[_NBitsProduct(nt(bits=2), 5 * A)]) == M.MLQ_E_TYPE
    assert ph(prods=[_NBitsProduct(nt(), 5 * A), _NBitsProduct(nt(f16=1), 12 * A)]) == M.MLQ_E_TYPE
    assert ph(prods=[_NBitsProduct(nt(bits=8), 5 * A),
                     _NBitsProduct(nt(bits=8, zp=6 * A, zld=16), 12 * A)]) == M.MLQ_E_TYPE  # zp all or none
    assert ph(prods=[_NBitsProduct(nt(), 5 * A), _NBitsProduct(nt(cols=1024), 12 * A)]) == M.MLQ_E_SHAPE
    assert ph(k=960, prods=[_NBitsProduct(nt(cols=960), 5 * A)]) == M.MLQ_E_SHAPE
    assert ph(prods=[_NBitsProduct(nt(sld=6), 5 * A)]) == M.MLQ_E_SHAPE
    assert ph(x=6 * A + 4) == M.MLQ_E_ALIGN
    assert ph(prods=[_NBitsProduct(nt(q=A + 8), 5 * A)]) == M.MLQ_E_ALIGN
    assert ph(prods=[_NBitsProduct(nt(), 5 * A + 2)]) == M.MLQ_E_ALIGN
