"""Pins for the oracle's draft head pieces (CPU only).

Components are checked against library routines written independently of the
oracle (torch's rms_norm, silu and scaled_dot_product_attention in fp64),
RoPE against the properties a rotary embedding must have, the head's
matrix inventory against the parameter counts the pages print, and the
composition against structural properties (a plausible wiring mistake --
swapped [f ; e] halves, a dropped residual, a norm on the wrong tensor --
fails one of them).
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import eagle_synth as S
from conftest import golden_lines
from oracle import layer as Lyr
from oracle.metrics import expected_tokens


def test_rmsnorm_matches_torch():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 64))
    g = rng.standard_normal(64)
    want = F.rms_norm(torch.tensor(x), (64,), torch.tensor(g), eps=1e-5).numpy()
    np.testing.assert_allclose(Lyr.rmsnorm(x, g, 1e-5), want, rtol=1e-12, atol=1e-12)


def test_silu_matches_torch():
    x = np.linspace(-30, 30, 101)
    np.testing.assert_allclose(Lyr.silu(x), F.silu(torch.tensor(x)).numpy(), rtol=1e-12, atol=1e-14)


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 2)])
def test_attention_matches_torch_sdpa(hq, hkv):
    rng = np.random.default_rng(1)
    dh, n = 16, 37
    q = rng.standard_normal((hq, dh))
    K = rng.standard_normal((n, hkv, dh))
    V = rng.standard_normal((n, hkv, dh))
    got = Lyr.attend(q, K, V, 1.0 / np.sqrt(dh))
    G = hq // hkv
    kt = torch.tensor(K).permute(1, 0, 2).repeat_interleave(G, 0)   # [hq, n, dh]
    vt = torch.tensor(V).permute(1, 0, 2).repeat_interleave(G, 0)
    want = F.scaled_dot_product_attention(torch.tensor(q)[:, None, :], kt, vt)[:, 0, :]
    np.testing.assert_allclose(got, want.numpy(), rtol=1e-10, atol=1e-12)


def test_softmax_matches_torch():
    rng = np.random.default_rng(2)
    z = rng.standard_normal((3, 100)) * 5
    for T in (1.0, 0.7):
        want = torch.softmax(torch.tensor(z) / T, -1).numpy()
        np.testing.assert_allclose(Lyr.softmax(z, T), want, rtol=1e-12, atol=1e-15)


def test_rope_is_a_relative_rotation():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((2, 16))
    k = rng.standard_normal((2, 16))
    # position 0 is the identity; norms are preserved
    np.testing.assert_allclose(Lyr.rope(q, 0, 1e4), q, atol=0)
    np.testing.assert_allclose(np.linalg.norm(Lyr.rope(q, 77, 1e4), axis=-1),
                               np.linalg.norm(q, axis=-1), rtol=1e-12)
    # the score depends on the position difference only
    s1 = np.sum(Lyr.rope(q, 10, 1e4) * Lyr.rope(k, 3, 1e4), -1)
    s2 = np.sum(Lyr.rope(q, 1010, 1e4) * Lyr.rope(k, 1003, 1e4), -1)
    np.testing.assert_allclose(s1, s2, rtol=1e-9)
    # pairs (i, i + dh/2) rotate together by angle pos * theta^(-2i/dh)
    e = np.zeros((1, 16)); e[0, 1] = 1.0
    r = Lyr.rope(e, 5, 1e4)
    ang = 5 * 1e4 ** (-2.0 / 16)
    np.testing.assert_allclose(r[0, [1, 9]], [np.cos(ang), np.sin(ang)], atol=1e-14)


def test_parameter_counts_of_the_pages():
    """Page A §4.3: the FC + one LLaMA decoder layer reproduce the printed
    trainable-parameter counts (7B 0.24B, 13B 0.37B, 70B 0.99B)."""
    n = 0
    for line in golden_lines("param_counts.txt"):
        left, right = line.split(":")
        _, d, hq, hkv, dh, ff = left.split()
        d, hq, hkv, dh, ff = map(int, (d, hq, hkv, dh, ff))
        fc = 2 * d * d
        attn = d * hq * dh * 2 + d * hkv * dh * 2          # Wq, Wo, Wk, Wv
        mlp = 3 * d * ff
        total = fc + attn + mlp
        assert round(total / 1e9, 2) == float(right), (left, total)
        n += 1
    assert n == 3


def test_workload_shapes_give_the_same_counts():
    for name, want in (("7b_static26", 0.24), ("70b_x16_eagle2", 0.99)):
        w = S.WORKLOADS[name]
        qd, kvd = w.n_q_heads * w.head_dim, w.n_kv_heads * w.head_dim
        shapes = {"w_fc": (w.d, 2 * w.d), "wq": (qd, w.d), "wk": (kvd, w.d), "wv": (kvd, w.d),
                  "wo": (w.d, qd), "w_gate": (w.d_ff, w.d), "w_up": (w.d_ff, w.d),
                  "w_down": (w.d, w.d_ff)}
        assert round(sum(a * b for a, b in shapes.values()) / 1e9, 2) == want


@pytest.fixture(scope="module")
def tiny():
    w = S.WORKLOADS["tiny_fp32"]
    W = S.draft_weights(w, 1000)
    return w, W


def _head(w, W, feat, tok, ctx_k=None, ctx_v=None):
    Wd = Lyr.DraftWeights(W, w)
    h = Lyr.fc_rows(Wd, feat[None], [tok])
    a = Lyr.rmsnorm(h, Wd.g1, w.rms_eps)
    q, k, v = Lyr.qkv_rows(Wd, a, [5], w)
    K = k if ctx_k is None else np.concatenate([ctx_k, k])
    V = v if ctx_v is None else np.concatenate([ctx_v, v])
    o = Lyr.attend(q[0], K, V, 1.0 / np.sqrt(w.head_dim))[None]
    return h, Lyr.finish_rows(Wd, h, o, w)


def test_fc_input_order_is_feature_then_token(tiny):
    w, W = tiny
    W = dict(W)
    W["w_fc"] = W["w_fc"].clone()
    W["w_fc"][:, w.d:] = 0            # kill the embedding half
    f = np.random.default_rng(4).standard_normal(w.d)
    h1, _ = _head(w, W, f, 3)
    h2, _ = _head(w, W, f, 400)
    np.testing.assert_array_equal(h1, h2)
    W["w_fc"] = S.draft_weights(w, 1000)["w_fc"].clone()
    W["w_fc"][:, :w.d] = 0            # kill the feature half
    h3, _ = _head(w, W, f, 3)
    h4, _ = _head(w, W, -f, 3)
    np.testing.assert_array_equal(h3, h4)


def test_residual_paths(tiny):
    w, W = tiny
    W = dict(W)
    for key in ("wo", "w_down"):
        W[key] = torch.zeros_like(W[key])
    f = np.random.default_rng(5).standard_normal(w.d)
    h, f_hat = _head(w, W, f, 7)
    np.testing.assert_array_equal(f_hat, h)      # both residual adds, nothing else
    W2 = dict(tiny[1])
    W2["w_down"] = torch.zeros_like(W2["w_down"])
    h, f_hat = _head(w, W2, f, 7)
    Wd = Lyr.DraftWeights(W2, w)
    assert not np.allclose(f_hat, h)             # attention output does reach f^


def test_norm_gains_scale_their_own_branch(tiny):
    """Scaling g1 by c scales q, k, v (the attention input) but not the FC output;
    scaling g2 by c leaves h2 unchanged."""
    w, W = tiny
    W = dict(W)
    Wd = Lyr.DraftWeights(W, w)
    f = np.random.default_rng(6).standard_normal(w.d)
    h = Lyr.fc_rows(Wd, f[None], [9])
    a = Lyr.rmsnorm(h, Wd.g1, w.rms_eps)
    a2 = Lyr.rmsnorm(h, 2.0 * Wd.g1, w.rms_eps)
    np.testing.assert_allclose(a2, 2.0 * a, rtol=1e-14)
    # rmsnorm is scale invariant in its input
    np.testing.assert_allclose(Lyr.rmsnorm(3.0 * h, Wd.g1, 0.0), Lyr.rmsnorm(h, Wd.g1, 0.0), rtol=1e-12)


def test_expected_tokens_worked_examples():
    n = 0
    for line in golden_lines("expected_tokens.txt"):
        left, right = line.split(":")
        alphas = [float(x) for x in left.split(",")]
        printed = right.strip()
        half_ulp = 0.5 * 10.0 ** -len(printed.split(".")[1])   # the page rounds its answers
        assert abs(expected_tokens(alphas) - float(printed)) <= half_ulp + 1e-12
        n += 1
    assert n == 4


def test_fuse_rows_input_order_is_low_middle_high():
    """g = FC([l; m; h]): each third of the FC's input columns reads its own
    layer's feature, in the order low, middle, high."""
    from oracle.layer import fuse_rows
    w = S.variant("tiny_fp32", name="fuse_pin")
    F = S.fuse_weights(w, 7)
    rng = np.random.default_rng(5)
    l, m, h = (rng.standard_normal((2, w.d)) for _ in range(3))
    d = w.d
    for blk, feat in enumerate((l, m, h)):
        Wb = F["w_fuse"].clone()
        keep = slice(blk * d, (blk + 1) * d)
        mask = torch.zeros_like(Wb)
        mask[:, keep] = 1
        Wb = Wb * mask
        g = fuse_rows(Wb, None, l, m, h)
        # only this block's feature matters: the others can change freely
        others = [np.zeros_like(l) if i != blk else feat for i in range(3)]
        np.testing.assert_array_equal(g, fuse_rows(Wb, None, *others))
        np.testing.assert_allclose(g, feat @ Wb.double().numpy()[:, keep].T, rtol=1e-12, atol=1e-12)
    g0 = fuse_rows(F["w_fuse"], None, l, m, h)
    np.testing.assert_allclose(fuse_rows(F["w_fuse"], F["b_fuse"], l, m, h) - g0,
                               np.broadcast_to(F["b_fuse"].double().numpy(), g0.shape), rtol=0, atol=1e-12)
