"""One decode layer of the forward pass on the GPU, through the C ABI.

Page "Legacy-ISA ML Inference Runtime -- Design Spec", Sec. 6 (Forward pass
per token), for one layer and one token at position ``pos``:

    h = rmsnorm(x); qa = quantize_q8(h)
    q, k, v = matvec(Wq | Wk | Wv, qa); rope(q, k, pos); KV[pos] = k, v
    per head: s = dot(q_h, K_t) / sqrt(hd); softmax(s); o_h = sum_t s_t V_t
    x += matvec(Wo, quantize_q8(o))
    h = rmsnorm(x); qa = quantize_q8(h)
    g = matvec(W1, qa); u = matvec(W3, qa); silu_mul(g, u)
    x += matvec(W2, quantize_q8(g))

Ten launches: every quantisation happens inside the launch that produces
the vector (rmsnorm, attention, silu_mul), the products sharing an input
run as one phase launch (Wq|Wk|Wv, W1|W3), the residual add of the
attention half is fused into the second rmsnorm.  Orchestration only: all
arithmetic runs in libmlq's kernels.
"""
from __future__ import annotations

import numpy as np
import torch

from . import binding as B
from . import inputs as I


class DecodeLayer:
    """Device state of one random-weight layer and the buffers of one token."""

    def __init__(self, shape: I.LayerShape, copies: int = 1, device: str = "cuda"):
        self.s = s = shape
        self.dev = torch.device(device)
        hd = s.head_dim
        assert s.dim % s.n_heads == 0 and s.n_heads % s.n_kv_heads == 0 and hd % 32 == 0
        # weights: `copies` sets (rotated by the bench so every step streams from HBM)
        self.host = {}
        self.W = []
        for c in range(copies):
            ws = {}
            for i, (name, rows, cols) in enumerate(s.mats()):
                q, d = I.weights(s.wtype, rows, cols, s.seed + i)
                if c == 0:
                    self.host[name] = (q, d, rows, cols)
                ws[name] = B.QTensor(self._t(q.reshape(-1)), self._t(d.reshape(-1)), rows, cols, s.wtype)
            self.W.append(ws)
        self.att_norm = I.norm_weights(s.dim, s.seed + 10)
        self.ffn_norm = I.norm_weights(s.dim, s.seed + 11)
        self.k_hist = I.kv_history(s.pos, s.kv_dim, s.seed + 12)
        self.v_hist = I.kv_history(s.pos, s.kv_dim, s.seed + 13)
        self.x_in = I.activations(1, s.dim, s.seed + 14)[0]
        f32 = dict(dtype=torch.float32, device=self.dev)
        self.att_norm_d, self.ffn_norm_d = self._t(self.att_norm), self._t(self.ffn_norm)
        self.cos = torch.zeros(s.max_seq * hd // 2, **f32)
        self.sin = torch.zeros(s.max_seq * hd // 2, **f32)
        B.mlq_rope_tables(self.cos, self.sin, s.max_seq, hd, s.rope_theta)
        self.kc = torch.zeros(s.max_seq, s.kv_dim, **f32)
        self.vc = torch.zeros(s.max_seq, s.kv_dim, **f32)
        self.reset()
        # per-token buffers
        self.x = torch.zeros(s.dim, **f32)
        self.h1 = torch.zeros(s.dim, **f32)
        self.q = torch.zeros(s.dim, **f32)
        self.k = torch.zeros(s.kv_dim, **f32)
        self.v = torch.zeros(s.kv_dim, **f32)
        self.o = torch.zeros(s.dim, **f32)
        self.yo = torch.zeros(s.dim, **f32)
        self.h2 = torch.zeros(s.dim, **f32)
        self.g = torch.zeros(s.hidden, **f32)
        self.u = torch.zeros(s.hidden, **f32)
        self.y2 = torch.zeros(s.dim, **f32)
        self.h1q, self.oq, self.h2q = self._qa(s.dim), self._qa(s.dim), self._qa(s.dim)
        self.gq = self._qa(s.hidden)
        self.x_host = torch.from_numpy(self.x_in).pin_memory() if self.dev.type == "cuda" else None
        self._calls = [self._build(c) for c in range(copies)]

    def _t(self, a) -> torch.Tensor:
        return torch.from_numpy(np.ascontiguousarray(a)).to(self.dev)

    def _qa(self, n):
        return B.QAct(torch.zeros(n, dtype=torch.int8, device=self.dev),
                      torch.zeros(n // 32, dtype=torch.float32, device=self.dev), n, 1)

    def reset(self):
        """The KV cache as before the token: history rows, nothing at pos."""
        s = self.s
        self.kc.zero_()
        self.vc.zero_()
        if s.pos:
            self.kc[:s.pos] = self._t(self.k_hist)
            self.vc[:s.pos] = self._t(self.v_hist)

    def weight_bytes(self) -> int:
        return sum(q.nbytes + d.nbytes for q, d, _, _ in self.host.values())

    def kv_bytes(self) -> int:
        """Cache bytes the attention reads (K and V of pos + 1 positions)."""
        return 2 * (self.s.pos + 1) * self.s.kv_dim * 4

    def _build(self, c):
        s, W = self.s, self.W[c]
        qkv = B.PhaseCall(s.dim, [B.PhaseProduct(W["wq"], self.q), B.PhaseProduct(W["wk"], self.k),
                                  B.PhaseProduct(W["wv"], self.v)], xq=self.h1q.q, xd=self.h1q.d)
        wo = B.PhaseCall(s.dim, [B.PhaseProduct(W["wo"], self.yo)], xq=self.oq.q, xd=self.oq.d)
        ffn = B.PhaseCall(s.dim, [B.PhaseProduct(W["w1"], self.g), B.PhaseProduct(W["w3"], self.u)],
                          xq=self.h2q.q, xd=self.h2q.d)
        down = B.PhaseCall(s.hidden, [B.PhaseProduct(W["w2"], self.y2)], xq=self.gq.q, xd=self.gq.d)
        return qkv, wo, ffn, down

    LAUNCHES = ("rmsnorm_att", "qkv", "rope", "attention", "wo", "add_rmsnorm_ffn", "ffn",
                "silu_mul", "down", "add")
    launches_per_step = len(LAUNCHES)

    def launch(self, name: str, copy: int = 0, stream=None):
        """One of the ten launches of a step (weights of copy `copy`)."""
        s = self.s
        hd, half = s.head_dim, s.head_dim // 2
        qkv, wo, ffn, down = self._calls[copy]
        if name == "rmsnorm_att":
            B.mlq_rmsnorm(self.h1, self.x, self.att_norm_d, s.dim, s.norm_eps, self.h1q, stream)
        elif name == "qkv":
            qkv(stream)
        elif name == "rope":
            B.mlq_rope(self.q, self.k, self.cos[s.pos * half:], self.sin[s.pos * half:], hd,
                       s.n_heads, s.n_kv_heads, self.kc[s.pos], self.v, self.vc[s.pos], stream)
        elif name == "attention":
            B.mlq_attention(self.o, self.q, self.kc, self.vc, s.pos + 1, hd, s.n_heads, s.n_kv_heads,
                            self.oq, stream)
        elif name == "wo":
            wo(stream)
        elif name == "add_rmsnorm_ffn":
            B.mlq_add_rmsnorm(self.x, self.yo, self.ffn_norm_d, s.dim, s.norm_eps, self.h2,
                              self.h2q, stream)
        elif name == "ffn":
            ffn(stream)
        elif name == "silu_mul":
            B.mlq_silu_mul(self.g, self.u, s.hidden, self.gq, stream)
        elif name == "down":
            down(stream)
        elif name == "add":
            B.mlq_add(self.x, self.y2, s.dim, stream)
        else:
            raise ValueError(name)

    def step(self, copy: int = 0, stream=None, after=None):
        """The layer for the token in self.x (updated in place).  after: None,
        or a function called with each launch's name once it is queued (a
        test inspects the buffers there)."""
        for name in self.LAUNCHES:
            self.launch(name, copy, stream)
            if after is not None:
                after(name)
