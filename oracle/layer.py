"""The feature-level draft head in fp64 (oracle side).

Structure (Page A §4.1; Page B "草稿头到底包含什么"; Page C "draft head 的结构和目标函数"):
    x   = [f ; e(t)]              feature of the parent position and the
                                   embedding of the shifted ("advanced") token
    h   = W_fc x + b_fc            FC 2d -> d (Page B writes h = W z + b)
    f^  = DecoderLayer(h)          one decoder layer
    z   = LM_Head(f^)              frozen, shared with the target
    q   = softmax(z / T)

The pages say only "one decoder layer".  Reading (parity unpinned beyond the
parameter counts of Page A §4.3, which this structure reproduces:
2d^2 + 4d^2 + 3dF = 0.236B for the 7B shape, 0.370B for 13B, and with GQA
0.990B for 70B): a LLaMA pre-norm layer --
    a  = RMSNorm(h; g1, eps)                  RMSNorm(x) = x / sqrt(mean(x^2) + eps) * g
    q, k, v = Wq a, Wk a, Wv a;  RoPE (rotate-half, theta) at the row's position
    o  = softmax(q k^T / sqrt(dh)) v          over the draft's own KV (Page B
                                               "Advanced Token": f^_j = D(f_1..f_{j-1}; t_2..t_j))
    h2 = h + Wo o
    f^ = h2 + W_down( SiLU(W_gate b) * (W_up b) ),  b = RMSNorm(h2; g2)
with no final norm: f is the LM-head input (Page B "先固定记号").
"""
from __future__ import annotations

import numpy as np


def to_f64(t) -> np.ndarray:
    """bf16 / fp32 torch tensor or numpy array -> fp64 numpy (exact)."""
    try:
        import torch  # local: only the conversion of shared input tensors
        if isinstance(t, torch.Tensor):
            return t.detach().to("cpu").to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(t, dtype=np.float64)


class DraftWeights:
    """fp64 copies of the draft head's weights, pad columns dropped."""

    def __init__(self, W: dict, dims):
        d, F = dims.d, dims.d_ff
        qd, kvd = dims.n_q_heads * dims.head_dim, dims.n_kv_heads * dims.head_dim
        self.dims = dims
        self.w_fc = to_f64(W["w_fc"])[:, :2 * d]
        self.b_fc = to_f64(W["b_fc"])
        self.g1 = to_f64(W["g1"])
        self.wq = to_f64(W["wq"])[:, :d]
        self.wk = to_f64(W["wk"])[:, :d]
        self.wv = to_f64(W["wv"])[:, :d]
        self.wo = to_f64(W["wo"])[:, :qd]
        self.g2 = to_f64(W["g2"])
        self.w_gate = to_f64(W["w_gate"])[:, :d]
        self.w_up = to_f64(W["w_up"])[:, :d]
        self.w_down = to_f64(W["w_down"])[:, :F]
        self._embed = W["embed"]          # rows converted on demand
        self.w_lm = to_f64(W["w_lm"])[:, :d]
        assert self.wq.shape[0] == qd and self.wk.shape[0] == kvd

    def embed(self, tokens) -> np.ndarray:
        rows = self._embed[np.asarray(tokens, dtype=np.int64)]
        return to_f64(rows)[:, :self.dims.d]


def rmsnorm(x: np.ndarray, g: np.ndarray, eps: float) -> np.ndarray:
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * g


def rope(x: np.ndarray, pos: int, theta: float) -> np.ndarray:
    """Rotate-half RoPE on [H, dh] at integer position pos (reading; unpinned)."""
    dh = x.shape[-1]
    half = dh // 2
    inv_freq = theta ** (-np.arange(half, dtype=np.float64) * 2.0 / dh)
    ang = float(pos) * inv_freq
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def silu(x: np.ndarray) -> np.ndarray:
    return x / (1.0 + np.exp(-x))


def softmax(z: np.ndarray, temperature: float = 1.0) -> np.ndarray:
    s = np.asarray(z, dtype=np.float64) / temperature
    s = s - s.max(axis=-1, keepdims=True)
    e = np.exp(s)
    return e / e.sum(axis=-1, keepdims=True)


def attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float) -> np.ndarray:
    """Multi-head attention of one row.  q [Hq, dh]; K, V [N, Hkv, dh] (GQA:
    query head h reads kv head h // (Hq / Hkv)).  Returns [Hq, dh]."""
    Hq = q.shape[0]
    Hkv = K.shape[1]
    G = Hq // Hkv
    out = np.empty_like(q)
    for h in range(Hq):
        kv = h // G
        s = K[:, kv, :] @ q[h] * scale
        p = softmax(s)
        out[h] = p @ V[:, kv, :]
    return out


def qkv_rows(W, x_norm: np.ndarray, positions, dims):
    """Projections + RoPE for a batch of normalised rows [n, d]."""
    n = x_norm.shape[0]
    q = (x_norm @ W.wq.T).reshape(n, dims.n_q_heads, dims.head_dim)
    k = (x_norm @ W.wk.T).reshape(n, dims.n_kv_heads, dims.head_dim)
    v = (x_norm @ W.wv.T).reshape(n, dims.n_kv_heads, dims.head_dim)
    for i, p in enumerate(positions):
        q[i] = rope(q[i], p, dims.rope_theta)
        k[i] = rope(k[i], p, dims.rope_theta)
    return q, k, v


def fc_rows(W: DraftWeights, feats: np.ndarray, tokens) -> np.ndarray:
    """h = W_fc [f ; e(t)] + b_fc for rows of (parent feature, shifted token)."""
    x = np.concatenate([feats, W.embed(tokens)], axis=1)
    return x @ W.w_fc.T + W.b_fc


def fuse_rows(w_fuse, b_fuse, l, m, h) -> np.ndarray:
    """EAGLE-3's fused feature (Page C "EAGLE-3：放弃 feature prediction，改成
    多层特征融合与 training-time test"): the target's low-, middle- and
    high-layer features concatenated, [l; m; h] (3k), compressed back to k by
    a fully connected layer, g = FC([l; m; h]).  Rows [n, d] each; the FC's
    bias is optional (None), as the page leaves it unstated."""
    d = np.asarray(l).shape[-1]
    W = to_f64(w_fuse)[:, :3 * d]
    x = np.concatenate([to_f64(l), to_f64(m), to_f64(h)], axis=-1)
    g = x @ W.T
    return g if b_fuse is None else g + to_f64(b_fuse)


def finish_rows(W, h: np.ndarray, o: np.ndarray, dims) -> np.ndarray:
    """h2 = h + Wo o;  f^ = h2 + W_down(SiLU(W_gate b) * W_up b), b = RMSNorm(h2)."""
    h2 = h + o.reshape(o.shape[0], -1) @ W.wo.T
    b = rmsnorm(h2, W.g2, dims.rms_eps)
    m = silu(b @ W.w_gate.T) * (b @ W.w_up.T)
    return h2 + m @ W.w_down.T


def lm_head(W: DraftWeights, f_hat: np.ndarray) -> np.ndarray:
    return f_hat @ W.w_lm.T
