"""Thin Python binding of libmlq's C ABI (include/mlq.h).

Argument marshalling only: every function here fills the C structs from
torch tensors (or raw integer device addresses) and calls the entry point of
the same name in libmlq.so.  All arithmetic runs in the library's CUDA
kernels; there is no Python or CPU fallback.  A non-MLQ_OK status raises
``MlqError``.  If libmlq.so has not been built, the first call raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

MLQ_OK, MLQ_E_SHAPE, MLQ_E_ALIGN, MLQ_E_TYPE, MLQ_E_NULL, MLQ_E_ARCH, MLQ_E_CUDA, MLQ_E_TIMEOUT, MLQ_E_BOUNDS = range(9)
MLQ_Q8_0 = 0
MLQ_Q4_0 = 1
MLQ_QK = 32
MLQ_MAX_COLS = 65536
MLQ_MAX_M = 16

# MLQ_CHECK_BOUNDS=1 selects the bounds-checking build of the library
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)),
                        "libmlq_checked.so" if os.environ.get("MLQ_CHECK_BOUNDS") == "1" else "libmlq.so")

# every symbol include/mlq.h declares
EXPORTS = (
    "mlq_init", "mlq_quantize_q8", "mlq_matvec_q4", "mlq_matvec_q8",
    "mlq_gemm_q4_small_m", "mlq_block_sumi", "mlq_last_device_error",
    "mlq_debug_set_wait_limit_ns", "mlq_status_str", "mlq_prefetch_l2",
    "mlq_chain_workspace_bytes", "mlq_decode_chain", "mlq_matvec_fused",
    "mlq_decode_chain_static", "mlq_decode_phase",
    "mlq_rmsnorm", "mlq_add_rmsnorm", "mlq_add", "mlq_softmax", "mlq_silu_mul",
    "mlq_rope_tables", "mlq_rope", "mlq_attention",
    "mlq_quantize_q8k", "mlq_matvec_q4k", "mlq_block_sums_q4k", "mlq_q4k_phase", "mlq_nbits_phase",
    "mlq_quantize_blk", "mlq_matvec_nbits", "mlq_block_sumi_nbits",
    "mlq_debug_chain_plan",
)
MLQ_QKK = 256
MLQ_MAX_SEQ = 32768
MLQ_MAX_HEAD_DIM = 256
MLQ_FUSED_MAX_PRODUCTS = 8
MLQ_F_STATIC_WEIGHTS = 1
MLQ_F_STATIC_INPUT = 2
MLQ_CHAIN_MAX_PRODUCTS = 32
MLQ_CHAIN_MAX_PHASES = 24


class MlqError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_name(status)} ({status})")


class _QTensor(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("d", ctypes.c_void_p), ("rows", ctypes.c_int),
                ("cols", ctypes.c_int), ("type", ctypes.c_uint8)]


class _QAct(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("d", ctypes.c_void_p), ("n", ctypes.c_int),
                ("m", ctypes.c_int)]


class _Q4KTensor(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("s", ctypes.c_void_p), ("d", ctypes.c_void_p),
                ("dmin", ctypes.c_void_p), ("rows", ctypes.c_int), ("cols", ctypes.c_int)]


class _Q4KProduct(ctypes.Structure):
    _fields_ = [("W", _Q4KTensor), ("y", ctypes.c_void_p)]


class _Q8KAct(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("d", ctypes.c_void_p), ("bsums", ctypes.c_void_p),
                ("n", ctypes.c_int)]


class _NBitsTensor(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("scales", ctypes.c_void_p), ("zp", ctypes.c_void_p),
                ("rows", ctypes.c_int), ("cols", ctypes.c_int), ("bits", ctypes.c_int),
                ("blk", ctypes.c_int), ("scale_f16", ctypes.c_int), ("scale_ld", ctypes.c_int),
                ("zp_ld", ctypes.c_int)]


class _NBitsProduct(ctypes.Structure):
    _fields_ = [("W", _NBitsTensor), ("y", ctypes.c_void_p)]


class _BlkAct(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("d", ctypes.c_void_p), ("bsums", ctypes.c_void_p),
                ("n", ctypes.c_int), ("blk", ctypes.c_int)]


class _ChainProduct(ctypes.Structure):
    _fields_ = [("W", _QTensor), ("y", ctypes.c_void_p)]


class _ChainPhase(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("n", ctypes.c_int), ("first", ctypes.c_int),
                ("count", ctypes.c_int), ("xq_out", ctypes.c_void_p), ("xd_out", ctypes.c_void_p)]


class _PhaseProduct(ctypes.Structure):
    _fields_ = [("W", _QTensor), ("y", ctypes.c_void_p), ("yq", ctypes.c_void_p),
                ("yd", ctypes.c_void_p)]


class _PhaseInput(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("xq", ctypes.c_void_p), ("xd", ctypes.c_void_p),
                ("n", ctypes.c_int), ("xq_out", ctypes.c_void_p), ("xd_out", ctypes.c_void_p)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libmlq.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_int
        QT, QA = ctypes.POINTER(_QTensor), ctypes.POINTER(_QAct)
        L.mlq_init.argtypes = []
        L.mlq_quantize_q8.argtypes = [QA, P, I, P]
        L.mlq_matvec_q4.argtypes = [P, QT, QA, I, I, P]
        L.mlq_matvec_q8.argtypes = [P, QT, QA, I, I, P]
        L.mlq_gemm_q4_small_m.argtypes = [P, I, QT, QA, I, I, I, P]
        L.mlq_block_sumi.argtypes = [P, QT, QA, I, I, P]
        L.mlq_last_device_error.argtypes = [P]
        L.mlq_debug_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
        L.mlq_prefetch_l2.argtypes = [P, P, I, P]
        L.mlq_chain_workspace_bytes.argtypes = [I]
        L.mlq_chain_workspace_bytes.restype = ctypes.c_size_t
        L.mlq_decode_chain.argtypes = [ctypes.POINTER(_ChainPhase), I, ctypes.POINTER(_ChainProduct),
                                       I, P, ctypes.c_size_t, P]
        L.mlq_decode_chain_static.argtypes = [ctypes.POINTER(_ChainPhase), I,
                                              ctypes.POINTER(_ChainProduct), I, P]
        L.mlq_matvec_fused.argtypes = [P, I, ctypes.POINTER(_ChainProduct), I, P, P,
                                       ctypes.c_uint, P]
        L.mlq_decode_phase.argtypes = [ctypes.POINTER(_PhaseInput), ctypes.POINTER(_PhaseProduct),
                                       I, P, P, I, ctypes.c_uint, P]
        F = ctypes.c_float
        L.mlq_rmsnorm.argtypes = [P, P, P, I, F, QA, P]
        L.mlq_add_rmsnorm.argtypes = [P, P, P, I, F, P, QA, P]
        L.mlq_add.argtypes = [P, P, I, P]
        L.mlq_softmax.argtypes = [P, I, P]
        L.mlq_silu_mul.argtypes = [P, P, I, QA, P]
        L.mlq_rope_tables.argtypes = [P, P, I, I, F, P]
        L.mlq_rope.argtypes = [P, P, P, P, I, I, I, P, P, P, P]
        L.mlq_attention.argtypes = [P, QA, P, P, P, I, I, I, I, P]
        KT, KA = ctypes.POINTER(_Q4KTensor), ctypes.POINTER(_Q8KAct)
        L.mlq_quantize_q8k.argtypes = [KA, P, I, P]
        L.mlq_matvec_q4k.argtypes = [P, KT, KA, I, I, P]
        L.mlq_block_sums_q4k.argtypes = [P, P, KT, KA, I, I, P]
        L.mlq_q4k_phase.argtypes = [P, I, ctypes.POINTER(_Q4KProduct), I, ctypes.c_uint, P]
        NT, BA = ctypes.POINTER(_NBitsTensor), ctypes.POINTER(_BlkAct)
        L.mlq_quantize_blk.argtypes = [BA, P, I, P]
        L.mlq_matvec_nbits.argtypes = [P, NT, BA, I, I, P]
        L.mlq_nbits_phase.argtypes = [P, I, ctypes.POINTER(_NBitsProduct), I, ctypes.c_uint, P]
        L.mlq_block_sumi_nbits.argtypes = [P, NT, BA, I, I, P]
        L.mlq_debug_chain_plan.argtypes = [ctypes.POINTER(_ChainPhase), I, ctypes.POINTER(_ChainProduct),
                                           I, I, P, I]
        L.mlq_status_str.argtypes = [S]
        L.mlq_status_str.restype = ctypes.c_char_p
        for name in EXPORTS:
            if name not in ("mlq_status_str", "mlq_chain_workspace_bytes"):
                getattr(L, name).restype = S
        _lib = L
    return _lib


def status_name(s: int) -> str:
    try:
        return lib().mlq_status_str(s).decode()
    except Exception:  # library not loadable: still name the code
        names = ["MLQ_OK", "MLQ_E_SHAPE", "MLQ_E_ALIGN", "MLQ_E_TYPE", "MLQ_E_NULL",
                 "MLQ_E_ARCH", "MLQ_E_CUDA", "MLQ_E_TIMEOUT", "MLQ_E_BOUNDS"]
        return names[s] if 0 <= s < len(names) else "MLQ_E_UNKNOWN"


def _addr(t) -> int | None:
    """Device address of a torch tensor, or an integer passed through."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        try:
            import torch
            if torch.cuda.is_available():
                return torch.cuda.current_stream().cuda_stream
        except Exception:
            pass
        return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


@dataclass
class QTensor:
    """Weight tensor: q (raw quant bytes) and d (float32 scales) on the device."""
    q: object
    d: object
    rows: int
    cols: int
    type: int

    def c(self) -> _QTensor:
        return _QTensor(_addr(self.q), _addr(self.d), self.rows, self.cols, self.type)


@dataclass
class QAct:
    """Q8_0 activations: m rows of n (q int8, d float32) on the device."""
    q: object
    d: object
    n: int
    m: int = 1

    def c(self) -> _QAct:
        return _QAct(_addr(self.q), _addr(self.d), self.n, self.m)


def _check(s: int, where: str) -> None:
    if s != MLQ_OK:
        raise MlqError(s, where)


def mlq_init() -> None:
    _check(lib().mlq_init(), "mlq_init")


def mlq_quantize_q8(out: QAct, x, k: int, stream=None) -> None:
    co = out.c()
    _check(lib().mlq_quantize_q8(ctypes.byref(co), _addr(x), k, _stream(stream)), "mlq_quantize_q8")


def mlq_matvec_q4(y, W: QTensor, x: QAct, r0: int, r1: int, stream=None) -> None:
    cw, cx = W.c(), x.c()
    _check(lib().mlq_matvec_q4(_addr(y), ctypes.byref(cw), ctypes.byref(cx), r0, r1,
                               _stream(stream)), "mlq_matvec_q4")


def mlq_matvec_q8(y, W: QTensor, x: QAct, r0: int, r1: int, stream=None) -> None:
    cw, cx = W.c(), x.c()
    _check(lib().mlq_matvec_q8(_addr(y), ctypes.byref(cw), ctypes.byref(cx), r0, r1,
                               _stream(stream)), "mlq_matvec_q8")


def mlq_gemm_q4_small_m(Y, ldy: int, W: QTensor, X: QAct, M: int, r0: int, r1: int,
                        stream=None) -> None:
    cw, cx = W.c(), X.c()
    _check(lib().mlq_gemm_q4_small_m(_addr(Y), ldy, ctypes.byref(cw), ctypes.byref(cx), M, r0, r1,
                                     _stream(stream)), "mlq_gemm_q4_small_m")


def mlq_block_sumi(sumi, W: QTensor, x: QAct, r0: int, r1: int, stream=None) -> None:
    cw, cx = W.c(), x.c()
    _check(lib().mlq_block_sumi(_addr(sumi), ctypes.byref(cw), ctypes.byref(cx), r0, r1,
                                _stream(stream)), "mlq_block_sumi")


# ---- Q4_K-style super-blocks ------------------------------------------------
@dataclass
class Q4KTensor:
    """Q4_K-style weights on the device: q nibbles, s (per super-block 8
    sub-block scales then 8 minima), d and dmin (float32 per super-block)."""
    q: object
    s: object
    d: object
    dmin: object
    rows: int
    cols: int

    def c(self) -> _Q4KTensor:
        return _Q4KTensor(_addr(self.q), _addr(self.s), _addr(self.d), _addr(self.dmin), self.rows,
                          self.cols)


@dataclass
class Q8KAct:
    """Activations for Q4_K products: q int8 [n], d float32 [n/256], bsums int32 [n/32]."""
    q: object
    d: object
    bsums: object
    n: int

    def c(self) -> _Q8KAct:
        return _Q8KAct(_addr(self.q), _addr(self.d), _addr(self.bsums), self.n)


def mlq_quantize_q8k(out: Q8KAct, x, k: int, stream=None) -> None:
    co = out.c()
    _check(lib().mlq_quantize_q8k(ctypes.byref(co), _addr(x), k, _stream(stream)), "mlq_quantize_q8k")


def mlq_matvec_q4k(y, W: Q4KTensor, x: Q8KAct, r0: int, r1: int, stream=None) -> None:
    cw, cx = W.c(), x.c()
    _check(lib().mlq_matvec_q4k(_addr(y), ctypes.byref(cw), ctypes.byref(cx), r0, r1,
                                _stream(stream)), "mlq_matvec_q4k")


def mlq_block_sums_q4k(isum, msum, W: Q4KTensor, x: Q8KAct, r0: int, r1: int, stream=None) -> None:
    cw, cx = W.c(), x.c()
    _check(lib().mlq_block_sums_q4k(_addr(isum), _addr(msum), ctypes.byref(cw), ctypes.byref(cx), r0,
                                    r1, _stream(stream)), "mlq_block_sums_q4k")


def mlq_q4k_phase(x, k: int, products, stream=None, flags: int = 0) -> None:
    """products: [(Q4KTensor, y), ...] (1..4) sharing the float input x;
    flags: 0 or MLQ_F_STATIC_INPUT."""
    arr = (_Q4KProduct * len(products))(*[_Q4KProduct(W.c(), _addr(y)) for W, y in products])
    _check(lib().mlq_q4k_phase(_addr(x), k, arr, len(products), flags, _stream(stream)), "mlq_q4k_phase")


# ---- block length 32 / 128, float16 scales, signed-offset 8-bit ------------
@dataclass
class NBitsTensor:
    """Block-quantised weights: q (4-bit nibbles or 8-bit B' = B - 128),
    scales [rows, scale_ld] float32 or float16, optional zero points
    [rows, zp_ld] uint8 (8-bit only)."""
    q: object
    scales: object
    zp: object
    rows: int
    cols: int
    bits: int
    blk: int
    scale_f16: int
    scale_ld: int
    zp_ld: int = 0

    def c(self) -> _NBitsTensor:
        return _NBitsTensor(_addr(self.q), _addr(self.scales), _addr(self.zp), self.rows, self.cols,
                            self.bits, self.blk, self.scale_f16, self.scale_ld, self.zp_ld)


@dataclass
class BlkAct:
    """Activations quantised per blk: q int8 [n], d float32 [n/blk], bsums int32 [n/blk]."""
    q: object
    d: object
    bsums: object
    n: int
    blk: int

    def c(self) -> _BlkAct:
        return _BlkAct(_addr(self.q), _addr(self.d), _addr(self.bsums), self.n, self.blk)


def mlq_quantize_blk(out: BlkAct, x, k: int, stream=None) -> None:
    co = out.c()
    _check(lib().mlq_quantize_blk(ctypes.byref(co), _addr(x), k, _stream(stream)), "mlq_quantize_blk")


def mlq_nbits_phase(x, k: int, products, stream=None, flags: int = 0) -> None:
    """products: [(NBitsTensor, y), ...] (1..4, one format) sharing the float
    input x; flags: 0 or MLQ_F_STATIC_INPUT."""
    arr = (_NBitsProduct * len(products))(*[_NBitsProduct(W.c(), _addr(y)) for W, y in products])
    _check(lib().mlq_nbits_phase(_addr(x), k, arr, len(products), flags, _stream(stream)), "mlq_nbits_phase")


def mlq_matvec_nbits(y, W: NBitsTensor, x: BlkAct, r0: int, r1: int, stream=None) -> None:
    cw, cx = W.c(), x.c()
    _check(lib().mlq_matvec_nbits(_addr(y), ctypes.byref(cw), ctypes.byref(cx), r0, r1,
                                  _stream(stream)), "mlq_matvec_nbits")


def mlq_block_sumi_nbits(sumi, W: NBitsTensor, x: BlkAct, r0: int, r1: int, stream=None) -> None:
    cw, cx = W.c(), x.c()
    _check(lib().mlq_block_sumi_nbits(_addr(sumi), ctypes.byref(cw), ctypes.byref(cx), r0, r1,
                                      _stream(stream)), "mlq_block_sumi_nbits")


# ---- the floating-point steps of a decode layer --------------------------
def _qa_ref(q: "QAct | None"):
    return None if q is None else ctypes.byref(q.c())


def mlq_rmsnorm(o, x, w, n: int, eps: float, oq: "QAct | None" = None, stream=None) -> None:
    _check(lib().mlq_rmsnorm(_addr(o), _addr(x), _addr(w), n, eps, _qa_ref(oq), _stream(stream)),
           "mlq_rmsnorm")


def mlq_add_rmsnorm(x, y, w, n: int, eps: float, o=None, oq: "QAct | None" = None,
                    stream=None) -> None:
    _check(lib().mlq_add_rmsnorm(_addr(x), _addr(y), _addr(w), n, eps, _addr(o), _qa_ref(oq),
                                 _stream(stream)), "mlq_add_rmsnorm")


def mlq_add(y, x, n: int, stream=None) -> None:
    _check(lib().mlq_add(_addr(y), _addr(x), n, _stream(stream)), "mlq_add")


def mlq_softmax(x, n: int, stream=None) -> None:
    _check(lib().mlq_softmax(_addr(x), n, _stream(stream)), "mlq_softmax")


def mlq_silu_mul(g, u, n: int, gq: "QAct | None" = None, stream=None) -> None:
    _check(lib().mlq_silu_mul(_addr(g), _addr(u), n, _qa_ref(gq), _stream(stream)), "mlq_silu_mul")


def mlq_rope_tables(cos_t, sin_t, max_seq: int, head_dim: int, theta: float, stream=None) -> None:
    _check(lib().mlq_rope_tables(_addr(cos_t), _addr(sin_t), max_seq, head_dim, theta,
                                 _stream(stream)), "mlq_rope_tables")


def mlq_rope(q, k, cos_row, sin_row, head_dim: int, n_heads: int, n_kv_heads: int, k_out=None,
             v=None, v_out=None, stream=None) -> None:
    _check(lib().mlq_rope(_addr(q), _addr(k), _addr(cos_row), _addr(sin_row), head_dim, n_heads,
                          n_kv_heads, _addr(k_out), _addr(v), _addr(v_out), _stream(stream)),
           "mlq_rope")


def mlq_attention(o, q, k_cache, v_cache, n_pos: int, head_dim: int, n_heads: int,
                  n_kv_heads: int, oq: "QAct | None" = None, stream=None) -> None:
    _check(lib().mlq_attention(_addr(o), _qa_ref(oq), _addr(q), _addr(k_cache), _addr(v_cache),
                               n_pos, head_dim, n_heads, n_kv_heads, _stream(stream)),
           "mlq_attention")


def mlq_prefetch_l2(ranges, stream=None) -> None:
    """ranges: sequence of (tensor or device address, byte count)."""
    n = len(ranges)
    ptrs = (ctypes.c_void_p * max(n, 1))(*[_addr(p) for p, _ in ranges])
    sizes = (ctypes.c_size_t * max(n, 1))(*[int(b) for _, b in ranges])
    _check(lib().mlq_prefetch_l2(ptrs, sizes, n, _stream(stream)), "mlq_prefetch_l2")


@dataclass
class ChainProduct:
    """One product of a chain: y = W x (x = its phase's quantised input)."""
    W: QTensor
    y: object


@dataclass
class ChainPhase:
    """Quantise x (n float32) and run products[first:first+count]."""
    x: object
    n: int
    first: int
    count: int
    xq_out: object = None
    xd_out: object = None


def mlq_chain_workspace_bytes(nphases: int) -> int:
    return lib().mlq_chain_workspace_bytes(nphases)


class ChainCall:
    """Marshalled arguments of one mlq_decode_chain call (built once, so
    that repeated calls cost one ctypes call each)."""

    def __init__(self, phases, products, workspace, workspace_bytes=None):
        self.ph = (_ChainPhase * len(phases))(*[
            _ChainPhase(_addr(p.x), p.n, p.first, p.count, _addr(p.xq_out), _addr(p.xd_out))
            for p in phases])
        self.pr = (_ChainProduct * len(products))(*[_ChainProduct(p.W.c(), _addr(p.y)) for p in products])
        self.nph, self.npr = len(phases), len(products)
        self.ws = _addr(workspace)
        self.wsb = (workspace.numel() * workspace.element_size() if workspace_bytes is None
                    else workspace_bytes)

    def __call__(self, stream=None) -> None:
        _check(lib().mlq_decode_chain(self.ph, self.nph, self.pr, self.npr, self.ws, self.wsb,
                                      _stream(stream)), "mlq_decode_chain")


class FusedCall:
    """Marshalled arguments of one mlq_matvec_fused call."""

    def __init__(self, x, n, products, xq_out=None, xd_out=None, flags: int = 0):
        self.x, self.n, self.flags = _addr(x), n, flags
        self.pr = (_ChainProduct * len(products))(*[_ChainProduct(p.W.c(), _addr(p.y)) for p in products])
        self.npr = len(products)
        self.xq, self.xd = _addr(xq_out), _addr(xd_out)

    def __call__(self, stream=None) -> None:
        _check(lib().mlq_matvec_fused(self.x, self.n, self.pr, self.npr, self.xq, self.xd,
                                      self.flags, _stream(stream)), "mlq_matvec_fused")


def mlq_matvec_fused(x, n, products, xq_out=None, xd_out=None, flags: int = 0,
                     stream=None) -> None:
    """Quantise x (n float32) and run every product (ChainProduct) of width n."""
    FusedCall(x, n, products, xq_out, xd_out, flags)(stream)


@dataclass
class PhaseProduct:
    """One product of a phase: y = W x, and optionally y in Q8_0 (yq, yd)."""
    W: QTensor
    y: object
    yq: object = None
    yd: object = None


class PhaseCall:
    """Marshalled arguments of one mlq_decode_phase call.  The input is
    float x (quantised in the launch; xq_out / xd_out receive it) or, with
    x None, Q8_0 (xq, xd) -- e.g. the yq / yd of an earlier phase.
    prefetch: (device pointer or tensor, bytes) ranges to hint into L2 once
    the input has been read, e.g. the weights of the phase after next."""

    def __init__(self, n, products, x=None, xq=None, xd=None, xq_out=None, xd_out=None,
                 flags: int = 0, prefetch=()):
        self.inp = _PhaseInput(_addr(x), _addr(xq), _addr(xd), n, _addr(xq_out), _addr(xd_out))
        self.pr = (_PhaseProduct * len(products))(*[
            _PhaseProduct(p.W.c(), _addr(p.y), _addr(p.yq), _addr(p.yd)) for p in products])
        self.npr, self.flags = len(products), flags
        self.npf = len(prefetch)
        self.pf = (ctypes.c_void_p * max(1, self.npf))(*[_addr(p) for p, _ in prefetch])
        self.pfb = (ctypes.c_size_t * max(1, self.npf))(*[int(b) for _, b in prefetch])

    def __call__(self, stream=None) -> None:
        _check(lib().mlq_decode_phase(ctypes.byref(self.inp), self.pr, self.npr, self.pf, self.pfb,
                                      self.npf, self.flags, _stream(stream)), "mlq_decode_phase")


def mlq_decode_phase(n, products, x=None, xq=None, xd=None, xq_out=None, xd_out=None,
                     flags: int = 0, prefetch=(), stream=None) -> None:
    """One phase: every product (PhaseProduct) of width n on one input."""
    PhaseCall(n, products, x, xq, xd, xq_out, xd_out, flags, prefetch)(stream)


def mlq_decode_chain_static(phases, products, stream=None) -> None:
    """mlq_decode_chain without a workspace: for callers that cannot allocate
    device memory (see include/mlq.h).  Calls on one device must not overlap."""
    ph = (_ChainPhase * len(phases))(*[
        _ChainPhase(_addr(p.x), p.n, p.first, p.count, _addr(p.xq_out), _addr(p.xd_out))
        for p in phases])
    pr = (_ChainProduct * len(products))(*[_ChainProduct(p.W.c(), _addr(p.y)) for p in products])
    _check(lib().mlq_decode_chain_static(ph, len(phases), pr, len(products), _stream(stream)),
           "mlq_decode_chain_static")


def mlq_decode_chain(phases, products, workspace, workspace_bytes=None, stream=None) -> None:
    ChainCall(phases, products, workspace, workspace_bytes)(stream)


def mlq_last_device_error(stream=None) -> int:
    """Synchronise the stream and return (not raise) the device status."""
    return lib().mlq_last_device_error(_stream(stream))


def mlq_debug_set_wait_limit_ns(limit_ns: int) -> None:
    _check(lib().mlq_debug_set_wait_limit_ns(limit_ns), "mlq_debug_set_wait_limit_ns")


def mlq_status_str(s: int) -> str:
    return lib().mlq_status_str(s).decode()


def raw_call(name: str, *args) -> int:
    """Call an entry point with already-marshalled arguments and return its
    status (host-side validation tests use this with fake addresses)."""
    return getattr(lib(), name)(*args)
