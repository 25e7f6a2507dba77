"""A tiny random-init target decoder, used only to pin the oracle's round.

The target model is not part of the method (the method accelerates someone
else's LLM).  This stand-in supplies real features and logits so that the
invariants of the pages can be checked end to end on the CPU:
  * the target chain T -> E -> f -> p = softmax(LM_Head(f)) -> t
    (Page A §3.1; Page B "先固定记号"; Page C "从 token 自回归转向特征自回归"),
    with f the LM-head input (here: the output of the final RMSNorm);
  * tree-masked verification equals running every root-to-node path on its
    own (Page B "Tree Attention 如何一次验证多条路径");
  * greedy acceptance reproduces plain greedy decoding (Page B "Greedy 验证").
Layers use the same LLaMA pre-norm structure as the draft head's layer.
"""
from __future__ import annotations

from typing import List

import numpy as np

from .layer import attend, rmsnorm, rope, silu, to_f64


class TinyTarget:
    def __init__(self, draft_w, tgt: dict, dims):
        self.dims = dims
        self.dw = draft_w                      # shared embedding + LM head
        d, F = dims.d, dims.d_ff
        qd = dims.n_q_heads * dims.head_dim
        self.layers = []
        for lw in tgt["layers"]:
            self.layers.append({
                "g1": to_f64(lw["g1"]), "g2": to_f64(lw["g2"]),
                "wq": to_f64(lw["wq"])[:, :d], "wk": to_f64(lw["wk"])[:, :d],
                "wv": to_f64(lw["wv"])[:, :d], "wo": to_f64(lw["wo"])[:, :qd],
                "w_gate": to_f64(lw["w_gate"])[:, :d], "w_up": to_f64(lw["w_up"])[:, :d],
                "w_down": to_f64(lw["w_down"])[:, :F],
            })
        self.g_final = to_f64(tgt["g_final"])

    def _qkv(self, lw, a, pos):
        D = self.dims
        q = (lw["wq"] @ a).reshape(D.n_q_heads, D.head_dim)
        k = (lw["wk"] @ a).reshape(D.n_kv_heads, D.head_dim)
        v = (lw["wv"] @ a).reshape(D.n_kv_heads, D.head_dim)
        return rope(q, pos, D.rope_theta), rope(k, pos, D.rope_theta), v

    def _mlp(self, lw, x):
        b = rmsnorm(x, lw["g2"], self.dims.rms_eps)
        return lw["w_down"] @ (silu(lw["w_gate"] @ b) * (lw["w_up"] @ b))

    def _logits(self, f):
        return self.dw.w_lm @ f

    def prefill(self, tokens: List[int]):
        """Causal forward over a token sequence at positions 0..n-1.
        Returns features [n, d], logits [n, V], caches: per layer (K, V) [n, Hkv, dh]."""
        D = self.dims
        scale = 1.0 / np.sqrt(D.head_dim)
        x = self.dw.embed(tokens).copy()
        n = len(tokens)
        caches = []
        for lw in self.layers:
            K = np.zeros((n, D.n_kv_heads, D.head_dim))
            V = np.zeros_like(K)
            out = np.empty_like(x)
            for i in range(n):
                a = rmsnorm(x[i], lw["g1"], D.rms_eps)
                q, K[i], V[i] = self._qkv(lw, a, i)
                o = attend(q, K[:i + 1], V[:i + 1], scale)
                h = x[i] + lw["wo"] @ o.reshape(-1)
                out[i] = h + self._mlp(lw, h)
            x = out
            caches.append((K, V))
        f = rmsnorm(x, self.g_final, D.rms_eps)
        return f, f @ self.dw.w_lm.T, caches

    def forward_tree(self, tokens, depth, anc, L, caches):
        """One verification forward over a flattened tree: node s at position
        L + depth[s], attending to the L cached positions and to its ancestors
        (bitmask anc[s]).  Returns features [S, d], logits [S, V] and the tree's
        per-layer (K, V) [S, Hkv, dh]."""
        D = self.dims
        scale = 1.0 / np.sqrt(D.head_dim)
        S = len(tokens)
        x = self.dw.embed(tokens).copy()
        tree_kv = []
        for lw, (Kc, Vc) in zip(self.layers, caches):
            Kt = np.zeros((S, D.n_kv_heads, D.head_dim))
            Vt = np.zeros_like(Kt)
            qs = []
            for s in range(S):
                a = rmsnorm(x[s], lw["g1"], D.rms_eps)
                q, Kt[s], Vt[s] = self._qkv(lw, a, L + depth[s])
                qs.append(q)
            out = np.empty_like(x)
            for s in range(S):
                vis = [j for j in range(S) if (anc[s] >> j) & 1]
                K = np.concatenate([Kc[:L], Kt[vis]])
                V = np.concatenate([Vc[:L], Vt[vis]])
                o = attend(qs[s], K, V, scale)
                h = x[s] + lw["wo"] @ o.reshape(-1)
                out[s] = h + self._mlp(lw, h)
            x = out
            tree_kv.append((Kt, Vt))
        f = rmsnorm(x, self.g_final, D.rms_eps)
        return f, f @ self.dw.w_lm.T, tree_kv

    def greedy_decode(self, tokens: List[int], n_new: int) -> List[int]:
        """Plain greedy decoding (full recompute each step; ties to the lower id)."""
        seq = list(tokens)
        out = []
        for _ in range(n_new):
            _, logits, _ = self.prefill(seq)
            z = logits[-1]
            g = int(np.flatnonzero(z == z.max())[0])
            out.append(g)
            seq.append(g)
        return out
