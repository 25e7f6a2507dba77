"""The parity harness's follow-the-GPU logic, checked on the CPU.

A stand-in "GPU result" is assembled from an oracle round (its values
rounded to fp32, node values recomputed from the fp32 confidences as the
library stores them).  compare_round must pass it with every request
reaching the commit; a stand-in whose children at one row were swapped (and
whose logits were nudged so that the swap is its own row's choice) must be
reported as exactly one near-tie, with the oracle continuing from the swapped
choice and still comparing every later stage."""
import numpy as np
import pytest
import torch

import eagle_synth as S
from oracle.layer import DraftWeights
from oracle.round import run_round
from tests.gpu_harness import compare_round, run_oracle_round

W_EAGLE2 = S.variant("70b_x16_eagle2", name="follow_eagle2", d=64, n_q_heads=4, n_kv_heads=2, head_dim=16,
                     d_ff=96, vocab=300, batch=3, prefix_len=20, top_k=3, depth=3, top_m=7, weight_std=0.1,
                     temps=(0.0, 1.0, 0.7))
W_STATIC = S.variant("7b_static26", name="follow_static8", d=64, n_q_heads=4, n_kv_heads=4, head_dim=16,
                     d_ff=96, vocab=300, batch=2, prefix_len=20, tree="static8", top_k=3, depth=3, top_m=8,
                     weight_std=0.1, temps=(0.0, 1.0))


class _Swap:
    """Oracle guide that swaps the first two greedy children of one row."""

    def __init__(self, b, e):
        self.b, self.e = b, e

    def children(self, b, e, st):
        if (b, e) == (self.b, self.e):
            t = list(st.child_tok[e])
            return [t[1], t[0]] + t[2:]
        return None

    def frontier(self, b, st, prev, keys):
        return None

    def final(self, b, st, keys):
        return None

    def accept(self, b, tree, result):
        return None


def _standin_gpu(w, seed, guide=None):
    W = S.draft_weights(w, seed)
    inp = S.round_inputs(w, seed)
    ic = {k: (v.detach().clone() if torch.is_tensor(v) else v) for k, v in inp.items()}
    res = run_round(DraftWeights(W, w), w, ic, guide=guide)
    Bn, V, d = w.batch, w.vocab, w.d
    E, K, Sn = S.max_expanded(w), w.top_k, 1 + w.top_m
    Hkv, dh = w.n_kv_heads, w.head_dim
    f32 = lambda *s: torch.zeros(*s, dtype=torch.float32)
    i32 = lambda *s: torch.full(s, -1, dtype=torch.int32)
    g = {"p_token": i32(Bn, E), "p_parent": i32(Bn, E), "p_rank": i32(Bn, E), "p_depth": i32(Bn, E),
         "p_value": torch.zeros(Bn, E, dtype=torch.float64), "c_token": i32(Bn, E, K), "c_prob": f32(Bn, E, K),
         "f_hat": f32(Bn, E, d), "logits": f32(Bn, E, V), "probs": f32(Bn, E, V), "dk_tree": f32(Bn, E, Hkv, dh),
         "t_token": i32(Bn, Sn), "t_parent": i32(Bn, Sn), "t_depth": i32(Bn, Sn), "t_pos": i32(Bn, Sn),
         "t_exp": i32(Bn, Sn), "t_anc": torch.zeros(Bn, Sn, (Sn + 63) // 64, dtype=torch.int64), "t_size": i32(Bn),
         "t_child_slot": i32(Bn, E, K), "attn_out": f32(Bn, Sn, w.n_q_heads, dh),
         "target_logits": f32(Bn, Sn, V), "target_probs": f32(Bn, Sn, V), "target_argmax": i32(Bn, Sn),
         "accept_len": i32(Bn), "path": i32(Bn, w.depth + 1), "final_token": i32(Bn), "last_slot": i32(Bn),
         "f_commit": f32(Bn, w.depth + 1, d), "tok_commit": i32(Bn, w.depth + 2), "f_last_out": f32(Bn, d),
         "t_next_out": i32(Bn), "prefix_len_out": i32(Bn), "draft_len_out": i32(Bn),
         "draft_k": inp["draft_k"].clone(), "draft_v": inp["draft_v"].clone(), "tgt_k_after": inp["tgt_k"].clone()}
    for b, r in enumerate(res):
        st, tr, ex = r["draft"], r["tree"], r["draft"].ex
        n = len(ex.token)
        g["p_token"][b, :n] = torch.tensor(ex.token)
        g["p_parent"][b, :n] = torch.tensor(ex.parent)
        g["p_rank"][b, :n] = torch.tensor(ex.rank)
        g["p_depth"][b, :n] = torch.tensor(ex.depth)
        for e in range(n):
            k = len(st.child_tok[e])
            g["c_token"][b, e, :k] = torch.tensor(st.child_tok[e])
            g["c_prob"][b, e, :k] = torch.tensor(st.child_q[e])
            g["f_hat"][b, e] = torch.from_numpy(st.f_hat[e])
            g["logits"][b, e] = torch.from_numpy(st.z[e])
            g["probs"][b, e] = torch.from_numpy(st.q[e])
            g["dk_tree"][b, e] = torch.from_numpy(st.k_tree[e])
        # node values as the library forms them: fp64 products of fp32 confidences
        g["p_value"][b, 0] = 1.0
        for e in range(1, n):
            g["p_value"][b, e] = float(g["p_value"][b, ex.parent[e]]) * float(g["c_prob"][b, ex.parent[e], ex.rank[e]])
        s = tr.size
        g["t_size"][b] = s
        for name, vals in (("t_token", tr.token), ("t_parent", tr.parent), ("t_depth", tr.depth),
                           ("t_exp", tr.exp)):
            g[name][b, :s] = torch.tensor(vals)
        g["t_pos"][b, :s] = torch.tensor([inp["prefix_len"][b] + dd for dd in tr.depth])
        for w_ in range(g["t_anc"].shape[2]):            # mask words: bits 64 w .. 64 w + 63
            words = [(a >> (64 * w_)) & 0xFFFFFFFFFFFFFFFF for a in tr.anc]
            g["t_anc"][b, :s, w_] = torch.tensor([x - (1 << 64) if x >= (1 << 63) else x for x in words])
        for (e, rr), slot in tr.child_slot.items():
            g["t_child_slot"][b, e, rr] = slot
        g["attn_out"][b, :s] = torch.from_numpy(r["verify_out"])
        g["target_logits"][b, :s] = torch.from_numpy(r["target_logits"])
        if r["target_probs"] is not None:
            g["target_probs"][b, :s] = torch.from_numpy(r["target_probs"])
        a = r["accept_len"]
        g["accept_len"][b] = a
        g["path"][b, :a + 1] = torch.tensor(r["path"])
        g["final_token"][b] = r["final"]
        g["last_slot"][b] = r["path"][-1]
        cm = r["commit"]
        g["f_commit"][b, :a + 1] = torch.from_numpy(cm["f_commit"])
        g["tok_commit"][b, :a + 2] = torch.tensor(cm["tok_commit"])
        g["f_last_out"][b] = torch.from_numpy(cm["f_last"])
        g["t_next_out"][b] = cm["t_next"]
        g["prefix_len_out"][b] = cm["prefix_len"]
        g["draft_len_out"][b] = cm["draft_len"]
        L, Ld = inp["prefix_len"][b], inp["draft_len"][b]
        g["tgt_k_after"][b, L:L + a + 1] = torch.from_numpy(cm["kv_rows_k"]).to(torch.bfloat16)
        g["draft_k"][b, Ld] = torch.from_numpy(cm["draft_root_k"]).to(torch.bfloat16)
    g["status"] = 0
    g["inputs_cpu"] = inp
    g["weights_cpu"] = W
    return g, res


@pytest.mark.parametrize("w", [W_EAGLE2, W_STATIC], ids=lambda w: w.name)
def test_follow_matches_itself(w):
    gpu, _ = _standin_gpu(w, 404)
    ref = run_oracle_round(w, 404, gpu["inputs_cpu"], gpu["weights_cpu"], gpu=gpu)
    rep = compare_round(w, gpu, ref)
    assert rep["ok"], rep["errors"]
    assert rep["reached"] == {b: "commit" for b in range(w.batch)}
    assert rep["near_ties"] == []


def test_follow_continues_after_a_flagged_choice():
    w = W_EAGLE2
    gpu, res = _standin_gpu(w, 404, guide=_Swap(0, 0))
    # make the swap the stand-in's own choice: its logits of the two tokens trade places
    a, c = [int(x) for x in gpu["c_token"][0, 0, :2]]
    z = gpu["logits"][0, 0]
    za, zc = float(z[a]), float(z[c])
    z[a], z[c] = zc, za
    ref = run_oracle_round(w, 404, gpu["inputs_cpu"], gpu["weights_cpu"], gpu=gpu)
    rep = compare_round(w, gpu, ref)
    ties = rep["near_ties"]
    assert len(ties) == 1 and ties[0]["request"] == 0 and ties[0]["stage"] == "children", ties
    assert 0 < ties[0]["margin"] <= ties[0]["bound"]
    # the swapped logits are reported as logit errors, every stage after the swap still compared
    assert rep["reached"] == {b: "commit" for b in range(w.batch)}
    assert [e for e in rep["errors"] if not e.startswith("logits")] == [], rep["errors"]
    assert rep["max_err"]["logits"] == pytest.approx(abs(za - zc), abs=1e-6)   # plus fp32 rounding
    # a row whose choice its own logits do not support is a failure, not a near-tie
    gpu["logits"][0, 0, a], gpu["logits"][0, 0, c] = za, zc
    ref = run_oracle_round(w, 404, gpu["inputs_cpu"], gpu["weights_cpu"], gpu=gpu)
    rep = compare_round(w, gpu, ref)
    assert not rep["ok"] and any("its own row selects" in e for e in rep["errors"]), rep["errors"]
    assert np.isfinite(rep["max_err"]["f_hat"])


def test_flip_measure_matches_brute_force():
    """The expected sampling flips per draw: the measure of uniforms on which
    inverse-CDF draws over two nearby distributions differ."""
    from tests.gpu_harness import _flip_measure
    assert _flip_measure(np.array([0.2, 0.5, 1.0]), np.array([0.21, 0.5, 1.0])) == pytest.approx(0.01)
    assert _flip_measure(np.array([0.2, 0.5, 1.0]), np.array([0.25, 0.45, 1.0])) == pytest.approx(0.1)
    rng = np.random.default_rng(0)
    q = rng.dirichlet(np.ones(50))
    q2 = q * np.exp(rng.normal(0, 0.01, 50))
    ca, cb = np.cumsum(q), np.cumsum(q2 / q2.sum())
    u = rng.random(400000)
    brute = np.mean(np.searchsorted(ca, u, side="right") != np.searchsorted(cb, u, side="right"))
    assert _flip_measure(ca, cb) == pytest.approx(brute, abs=1e-3)
