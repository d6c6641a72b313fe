"""Seeded synthetic inputs shared by the tests and the bench.

This module holds no arithmetic of the method itself: it only draws raw
quant bytes, scales and float activations with numpy's ``default_rng`` and
describes the workload shapes.  Both the CUDA path and the CPU oracle are
fed the same host bytes from here.

Value distributions (stated for every workload):
  * Q4_0 weights: every nibble uniform in 0..15 (so every byte uniform in
    0..255), block scales float32 uniform in [1e-3, 1e-2];
  * Q8_0 weights: int8 uniform in [-127, 127], scales uniform in [1e-4, 1e-3];
  * activations: float32 standard normal.
Shapes follow the pages' workloads (TinyLlama-1.1B layer, Llama-7B FFN
stack, Qwen2.5-0.5B lm_head; see the ONNX Runtime page, "Results first" and
"Synthetic FFN (context)").  No trained weights or datasets are used.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

QK = 32
Q8_0 = 0
Q4_0 = 1


def q4_weights(rows: int, cols: int, seed: int, lo: float = 1e-3, hi: float = 1e-2):
    """(q uint8 [rows, cols/2], d float32 [rows, cols/32]) with random nibbles."""
    assert cols % QK == 0
    rng = np.random.default_rng(seed)
    q = rng.integers(0, 256, size=(rows, cols // 2), dtype=np.uint8)
    d = rng.uniform(lo, hi, size=(rows, cols // QK)).astype(np.float32)
    return q, d


def q8_weights(rows: int, cols: int, seed: int, lo: float = 1e-4, hi: float = 1e-3):
    """(q int8 [rows, cols], d float32 [rows, cols/32]); q uniform in [-127, 127]."""
    assert cols % QK == 0
    rng = np.random.default_rng(seed)
    q = rng.integers(-127, 128, size=(rows, cols), dtype=np.int8)
    d = rng.uniform(lo, hi, size=(rows, cols // QK)).astype(np.float32)
    return q, d


def weights(wtype: int, rows: int, cols: int, seed: int):
    return q4_weights(rows, cols, seed) if wtype == Q4_0 else q8_weights(rows, cols, seed)


QKK = 256


def q4k_weights(rows: int, cols: int, seed: int, lo: float = 1e-4, hi: float = 1e-3):
    """Q4_K-style weights: uniform nibble bytes; per super-block 8 sub-block
    scales and 8 minima uniform in the 6-bit range [0, 63]; d and dmin
    uniform [lo, hi) float32 (so d * s_b spans about the Q4_0 scales'
    range).  Returns (q [rows, cols/2] u8, s [rows, cols/256*16] u8,
    d [rows, cols/256] f32, dmin [rows, cols/256] f32)."""
    assert cols % QKK == 0
    rng = np.random.default_rng(seed)
    nsb = cols // QKK
    q = rng.integers(0, 256, size=(rows, cols // 2), dtype=np.uint8)
    s = rng.integers(0, 64, size=(rows, nsb * 16), dtype=np.uint8)
    d = rng.uniform(lo, hi, size=(rows, nsb)).astype(np.float32)
    dmin = rng.uniform(lo, hi, size=(rows, nsb)).astype(np.float32)
    return q, s, d, dmin


def activations(m: int, k: int, seed: int) -> np.ndarray:
    """float32 [m, k] ~ N(0, 1)."""
    rng = np.random.default_rng(seed)
    return rng.standard_normal(size=(m, k)).astype(np.float32)


# --------------------------------------------------------------------------
# Workload shapes.  ``seed`` of tensor i is base_seed + i (the pages give no
# seeds; the tiny case uses seed 0 as stated).
# --------------------------------------------------------------------------
@dataclass
class Matvec:
    name: str
    wtype: int
    rows: int
    cols: int
    input_of: str = "x"      # which vector feeds it: "x" or the name of a prior output


@dataclass
class Workload:
    name: str
    m: int
    mats: list = field(default_factory=list)
    chained: bool = False
    description: str = ""


def tiny_q4() -> Workload:
    return Workload("tiny_q4_256x512", 1, [Matvec("w", Q4_0, 256, 512)],
                    description="Q4_0 256x512, M=1, seed 0")


def tinyllama_layer() -> Workload:
    """One TinyLlama-1.1B-shaped decode layer, Q4_0, M=1.

    Data flow (steps outside the matvec path are identity): q, k, v all
    read Q8_0(x); Wo reads Q8_0(q); gate and up read Q8_0(o); down reads
    Q8_0(gate)."""
    d, kv, ff = 2048, 256, 5632
    return Workload("tinyllama1.1b_layer_q4_0", 1, [
        Matvec("wq", Q4_0, d, d, "x"),
        Matvec("wk", Q4_0, kv, d, "x"),
        Matvec("wv", Q4_0, kv, d, "x"),
        Matvec("wo", Q4_0, d, d, "wq"),
        Matvec("w_gate", Q4_0, ff, d, "wo"),
        Matvec("w_up", Q4_0, ff, d, "wo"),
        Matvec("w_down", Q4_0, d, ff, "w_gate"),
    ], chained=True, description="TinyLlama-1.1B-shaped layer, Q4_0, M=1")


def llama7b_ffn(wtype: int = Q4_0, layers: int = 8) -> Workload:
    mats = []
    prev = "x"
    for i in range(layers):
        mats.append(Matvec(f"up{i}", wtype, 11008, 4096, prev))
        mats.append(Matvec(f"down{i}", wtype, 4096, 11008, f"up{i}"))
        prev = f"down{i}"
    tag = "q4_0" if wtype == Q4_0 else "q8_0"
    return Workload(f"llama7b_ffn8_{tag}", 1, mats, chained=True,
                    description=f"8-layer Llama-7B FFN stack, {tag.upper()}, M=1, chained")


def qwen_lm_head() -> Workload:
    return Workload("qwen2.5-0.5b_lm_head_q8_0", 1, [Matvec("lm_head", Q8_0, 151936, 896)],
                    description="Qwen2.5-0.5B-shaped lm_head, Q8_0, M=1")


def small_m(m: int) -> Workload:
    return Workload(f"gemm_q4_0_m{m}", m, [Matvec("up", Q4_0, 11008, 4096, "x"),
                                            Matvec("down", Q4_0, 4096, 11008, "x")],
                    description=f"Q4_0 small-M GEMM, M={m}, 11008x4096 and 4096x11008")


def llama7b_ffn_q8_lm_head() -> Workload:
    wl = llama7b_ffn(Q8_0)
    wl.mats.append(Matvec("lm_head", Q8_0, 151936, 896, "x"))
    wl.name = "llama7b_ffn8_q8_0+qwen2.5-0.5b_lm_head"
    wl.description = "8-layer Llama-7B FFN stack Q8_0 (chained) + Qwen2.5-0.5B lm_head Q8_0, M=1"
    return wl


WORKLOADS = {
    "tiny_q4": tiny_q4,
    "tinyllama_layer": tinyllama_layer,
    "llama7b_ffn_q4": lambda: llama7b_ffn(Q4_0),
    "llama7b_ffn_q8_lm_head": llama7b_ffn_q8_lm_head,
    "qwen_lm_head": qwen_lm_head,
    "small_m4": lambda: small_m(4),
    "small_m16": lambda: small_m(16),
}


# --------------------------------------------------------------------------
# A whole decode layer (Design Spec Sec. 6 forward pass) with random weights:
# the seven Q4_0 products of a TinyLlama-1.1B layer, its two rmsnorm weight
# vectors (uniform in [0.5, 1.5]), the RoPE tables (theta 10000) and a KV
# cache whose first `pos` positions hold N(0, 1) values; the token's input x
# is N(0, 1).  Seeds: base + tensor index, as above.
# --------------------------------------------------------------------------
@dataclass
class LayerShape:
    name: str = "tinyllama1.1b_decode_layer_q4_0"
    dim: int = 2048
    n_heads: int = 32
    n_kv_heads: int = 4
    hidden: int = 5632
    max_seq: int = 2048
    pos: int = 255            # the token's position: attention covers pos + 1 positions
    rope_theta: float = 10000.0
    norm_eps: float = 1e-5
    wtype: int = Q4_0
    seed: int = 0

    @property
    def head_dim(self) -> int:
        return self.dim // self.n_heads

    @property
    def kv_dim(self) -> int:
        return self.n_kv_heads * self.head_dim

    def mats(self):
        """(name, rows, cols) of the seven products, in forward-pass order."""
        d, kv, hd = self.dim, self.kv_dim, self.hidden
        return [("wq", d, d), ("wk", kv, d), ("wv", kv, d), ("wo", d, d),
                ("w1", hd, d), ("w3", hd, d), ("w2", d, hd)]


def norm_weights(n: int, seed: int) -> np.ndarray:
    """float32 [n] uniform in [0.5, 1.5]."""
    rng = np.random.default_rng(seed)
    return rng.uniform(0.5, 1.5, size=n).astype(np.float32)


def kv_history(n_pos: int, kv_dim: int, seed: int) -> np.ndarray:
    """float32 [n_pos, kv_dim] ~ N(0, 1): the cached K or V rows of earlier tokens."""
    rng = np.random.default_rng(seed)
    return rng.standard_normal(size=(n_pos, kv_dim)).astype(np.float32)


def tinyllama_decode_layer(pos: int = 255) -> LayerShape:
    return LayerShape(pos=pos)


LAYERS = {
    "tinyllama_decode_layer": tinyllama_decode_layer,
}


# ---- Q4_K-style super-block workloads ---------------------------------------
@dataclass
class Q4KWorkload:
    """M = 1 products on Q4_K-style weights.  mats: (name, rows, cols,
    input) with input "x" (the workload's float input) or the name of an
    earlier product whose output is the input; every input is quantised per
    256 before the first product that reads it."""
    name: str
    mats: list
    seed: int = 0


def tinyllama_layer_q4k() -> Q4KWorkload:
    """The projections of one TinyLlama-1.1B layer in Q4_K (the model the
    page runs as Q4_K_M): Wq 2048x2048, Wk / Wv 256x2048, Wo 2048x2048,
    gate / up 5632x2048, down 2048x5632."""
    d, kv, ff = 2048, 256, 5632
    return Q4KWorkload("tinyllama1.1b_layer_q4k", [
        ("wq", d, d, "x"), ("wk", kv, d, "x"), ("wv", kv, d, "x"),
        ("wo", d, d, "wq"), ("w_gate", ff, d, "wo"), ("w_up", ff, d, "wo"),
        ("w_down", d, ff, "w_gate")])


Q4K_WORKLOADS = {"tinyllama_layer_q4k": tinyllama_layer_q4k}



# ---- block length 32 / 128, float16 scales, signed-offset 8-bit weights ----
def nbits_weights(rows: int, cols: int, bits: int, blk: int, f16: bool, with_zp: bool, seed: int):
    """4-bit: nibble bytes uniform; 8-bit: B' = B - 128 uniform int8; scales
    U[1e-3, 1e-2] (4-bit) or U[1e-4, 1e-3] (8-bit), float32 or float16;
    8-bit zero points uniform in [120, 136] around the usual 128 (None when
    not requested).  Returns (q, scales [rows, cols/blk], zp or None)."""
    rng = np.random.default_rng(seed)
    nb = cols // blk
    if bits == 4:
        q = rng.integers(0, 256, size=(rows, cols // 2), dtype=np.uint8)
        lo, hi = 1e-3, 1e-2
    else:
        q = rng.integers(-128, 128, size=(rows, cols), dtype=np.int8)
        lo, hi = 1e-4, 1e-3
    sc = rng.uniform(lo, hi, size=(rows, nb)).astype(np.float16 if f16 else np.float32)
    zp = rng.integers(120, 137, size=(rows, nb), dtype=np.uint8) if (bits == 8 and with_zp) else None
    return q, sc, zp


def pad_rows(a: np.ndarray, align_bytes: int = 16) -> np.ndarray:
    """Copy of a [rows, n] array with each row padded (zeros) to a multiple of
    align_bytes; the padded row length in elements is the array's width."""
    per = align_bytes // a.itemsize
    ld = (a.shape[1] + per - 1) // per * per
    out = np.zeros((a.shape[0], ld), dtype=a.dtype)
    out[:, :a.shape[1]] = a
    return out


@dataclass
class NBitsWorkload:
    """M = 1 products on blocks of `blk` with `bits`-bit weights; mats as in
    Q4KWorkload; every input is quantised per `blk` before the first
    product that reads it."""
    name: str
    mats: list
    bits: int
    blk: int
    f16: bool
    with_zp: bool
    seed: int = 0


def _qwen_mats():
    d, kv, ff = 896, 128, 4864   # Qwen2.5-0.5B: hidden 896, 2 KV heads of 64, intermediate 4864
    return [("wq", d, d, "x"), ("wk", kv, d, "x"), ("wv", kv, d, "x"), ("wo", d, d, "wq"),
            ("w_gate", ff, d, "wo"), ("w_up", ff, d, "wo"), ("w_down", d, ff, "w_gate")]


def qwen_layer_int4_blk128() -> NBitsWorkload:
    """One Qwen2.5-0.5B layer's projections as AMD's int4 export stores
    them: 4-bit weights in blocks of 128, float32 scales."""
    return NBitsWorkload("qwen2.5-0.5b_layer_int4_blk128", _qwen_mats(), 4, 128, False, False)


def qwen_layer_int8_sq8() -> NBitsWorkload:
    """The same projections as the int8 export in the signed-offset form:
    8-bit weights B' = B - 128 in blocks of 32, float16 scales, per-block
    zero points around 128."""
    return NBitsWorkload("qwen2.5-0.5b_layer_int8_sq8", _qwen_mats(), 8, 32, True, True)


NBITS_WORKLOADS = {"qwen_layer_int4_blk128": qwen_layer_int4_blk128,
                   "qwen_layer_int8_sq8": qwen_layer_int8_sq8}
