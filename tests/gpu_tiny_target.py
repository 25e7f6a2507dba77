"""A stand-in for the target model on the GPU, for the decode-loop tests.

The target model is not part of the method: the method accelerates someone
else's LLM.  To run several draft-and-verify rounds in a row, something must
play the target between drafting and acceptance: this module is the tiny
random-init 2-layer decoder of the tiny workload (the same weights the
oracle's TinyTarget reads), written in plain fp32 PyTorch ops on the GPU,
except that its tree-masked attention over the cached prefix runs through
libeagle's eagle_tree_verify_attn (bf16 caches, as the library stores them).
LLaMA pre-norm layers like the draft head's: RMSNorm, rotate-half RoPE,
attention with kv head = h / G, SwiGLU MLP; a final RMSNorm gives the feature
f that the LM head reads.
"""
from __future__ import annotations

import math

import torch

from eagle_feature_level_gb300 import _binding as B


def _rmsnorm(x, g, eps):
    return x * torch.rsqrt((x * x).mean(-1, keepdim=True) + eps) * g


class GpuTinyTarget:
    def __init__(self, w, W, T):
        d, F = w.d, w.d_ff
        self.w = w
        qd = w.n_q_heads * w.head_dim
        f = lambda t, cols: t[:, :cols].float()
        self.embed = f(W["embed"], d)
        self.w_lm = f(W["w_lm"], d)
        self.layers = [dict(g1=lw["g1"].float(), g2=lw["g2"].float(), wq=f(lw["wq"], d), wk=f(lw["wk"], d),
                            wv=f(lw["wv"], d), wo=f(lw["wo"], qd), w_gate=f(lw["w_gate"], d),
                            w_up=f(lw["w_up"], d), w_down=f(lw["w_down"], F)) for lw in T["layers"]]
        self.g_final = T["g_final"].float()
        self.scale = 1.0 / math.sqrt(w.head_dim)

    def _rope(self, x, pos):
        """x [..., H, dh]; pos [...] integer positions."""
        dh = x.shape[-1]
        half = dh // 2
        inv = self.w.rope_theta ** (-torch.arange(half, dtype=torch.float64, device=x.device) * 2.0 / dh)
        ang = pos.to(torch.float64)[..., None] * inv
        c = torch.cos(ang).float().unsqueeze(-2)
        s = torch.sin(ang).float().unsqueeze(-2)
        x1, x2 = x[..., :half], x[..., half:]
        return torch.cat([x1 * c - x2 * s, x2 * c + x1 * s], dim=-1)

    def _qkv(self, lw, x, pos):
        w = self.w
        a = _rmsnorm(x, lw["g1"], w.rms_eps)
        sh = x.shape[:-1]
        q = (a @ lw["wq"].T).view(*sh, w.n_q_heads, w.head_dim)
        k = (a @ lw["wk"].T).view(*sh, w.n_kv_heads, w.head_dim)
        v = (a @ lw["wv"].T).view(*sh, w.n_kv_heads, w.head_dim)
        return self._rope(q, pos), self._rope(k, pos), v

    def _finish(self, lw, x, o):
        h = x + o @ lw["wo"].T
        b = _rmsnorm(h, lw["g2"], self.w.rms_eps)
        return h + (torch.nn.functional.silu(b @ lw["w_gate"].T) * (b @ lw["w_up"].T)) @ lw["w_down"].T

    def prefill(self, tokens):
        """Causal forward over one prompt (positions 0..n-1): features [n, d],
        logits [n, V], per layer (K, V) [n, Hkv, dh] fp32."""
        w = self.w
        n = tokens.numel()
        x = self.embed[tokens.long()]
        pos = torch.arange(n, device=x.device)
        causal = torch.ones(n, n, dtype=torch.bool, device=x.device).tril()
        caches = []
        G = w.n_q_heads // w.n_kv_heads
        for lw in self.layers:
            q, k, v = self._qkv(lw, x, pos)
            kk, vv = k.repeat_interleave(G, dim=1), v.repeat_interleave(G, dim=1)
            s = torch.einsum("ihd,jhd->hij", q, kk) * self.scale
            p = torch.softmax(s.masked_fill(~causal, float("-inf")), dim=-1)
            o = torch.einsum("hij,jhd->ihd", p, vv).reshape(n, -1)
            x = self._finish(lw, x, o)
            caches.append((k, v))
        f = _rmsnorm(x, self.g_final, w.rms_eps)
        return f, f @ self.w_lm.T, caches

    def verify(self, eng, rd):
        """The target forward over the round's flattened tree: every layer's
        tree Q/K/V (bf16) into the round's buffers, attention through
        eagle_tree_verify_attn over that layer's cache, then the round's true
        features and target logits."""
        x = self.embed[rd.t_token.clamp(min=0).long()]
        pos = rd.t_pos.long()
        st, ws = eng.stream(), eng.ws.data_ptr()
        for l, lw in enumerate(self.layers):
            q, k, v = self._qkv(lw, x, pos)
            rd.tree_q.copy_(q.to(torch.bfloat16))
            rd.tree_k[l].copy_(k.to(torch.bfloat16))
            rd.tree_v[l].copy_(v.to(torch.bfloat16))
            prefix = B.eagle_kv(rd.tgt_k[l].data_ptr(), rd.tgt_v[l].data_ptr(), rd.kv_cap, rd.tgt_len.data_ptr())
            B.eagle_tree_verify_attn(eng.ctx, rd.B, rd.tree_q.data_ptr(), rd.tree_k[l].data_ptr(),
                                     rd.tree_v[l].data_ptr(), prefix, rd.tree_c, self.scale, rd.attn_out.data_ptr(),
                                     ws, st)
            x = self._finish(lw, x, rd.attn_out.reshape(*x.shape[:-1], -1))
        f = _rmsnorm(x, self.g_final, self.w.rms_eps)
        rd.f_true.copy_(f)
        rd.target_logits.copy_(f @ self.w_lm.T)
