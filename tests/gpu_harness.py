"""GPU-vs-oracle round harness used by the parity tests and smoke().

run_gpu_round: seeded inputs -> one round through libeagle's C ABI on cuda:0.
run_oracle_round: the same inputs (copied to the host) through the CPU oracle.
compare_round: element-wise comparison.  Discrete results (children, tree,
accept length, path, tokens) must be identical; a mismatch is tolerated only
as a flagged near-tie, when the oracle's own margin for that decision is
below the floating-point tolerance (a logit gap, a sampling CDF margin, or
for EAGLE-2 two node values -- products of draft confidences -- closer than
the confidences' observed error can reorder), and the request's later
comparisons are then skipped.  Floating point: features, logits and attention outputs within
max-abs 1e-4 (fp32 workload) or 2e-2 (bf16 workloads), applied to values in
units of the row's RMS when that exceeds 1 (random draft weights grow the
residual stream layer by layer, to RMS ~10^2 at depth 5 of the 70B shape,
while the bound presumes unit-scale features); probabilities within 1e-3.
"""
from __future__ import annotations

import numpy as np
import torch

import eagle_synth as S
from eagle_feature_level_gb300 import runtime as R
from eagle_feature_level_gb300.workload import make_round, standin

TOL_PROB = 1e-3


def feature_tol(w) -> float:
    return 1e-4 if w.name.startswith("tiny") else 2e-2


GPU_FIELDS = ["p_token", "p_parent", "p_depth", "p_value", "c_token", "c_prob", "f_hat", "logits", "probs",
              "dk_tree", "t_token", "t_parent", "t_depth", "t_pos", "t_exp", "t_anc", "t_size", "attn_out",
              "target_logits", "target_probs", "target_argmax", "accept_len", "path", "final_token", "last_slot",
              "f_commit", "tok_commit", "f_last_out", "t_next_out", "prefix_len_out", "draft_len_out",
              "draft_k", "draft_v"]


def run_gpu_round(w, seed, device="cuda", weights=None, inputs=None):
    W = weights if weights is not None else S.draft_weights(w, seed, device=device)
    inp = inputs if inputs is not None else S.round_inputs(w, seed, device=device)
    eng, rd = make_round(w, inp, device)
    rd.run(eng.weights(W), target_fn=standin(inp))
    torch.cuda.synchronize()
    status = eng.status()
    out = {k: getattr(rd, k).detach().to("cpu") for k in GPU_FIELDS}
    out["tgt_k_after"] = rd.tgt_k[0].detach().to("cpu")
    out["status"] = status
    out["launches"] = R.B.eagle_launch_count(eng.ctx)
    out["inputs_cpu"] = {k: (v.detach().to("cpu") if torch.is_tensor(v) else v) for k, v in inp.items()}
    out["weights_cpu"] = {k: v.detach().to("cpu") for k, v in W.items()}
    eng.close()
    return out


def run_oracle_round(w, seed, inputs_cpu, weights_cpu, requests=None):
    from oracle.layer import DraftWeights
    from oracle.round import run_round
    Wd = DraftWeights(weights_cpu, w)
    return run_round(Wd, w, inputs_cpu, requests=requests)


def _maxerr(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b))) if a.size else 0.0


def _maxerr_scaled(a, b) -> float:
    """max |a - b| in units of max(1, RMS of the oracle row b)."""
    b = np.asarray(b, dtype=np.float64)
    scale = max(1.0, float(np.sqrt(np.mean(b * b)))) if b.size else 1.0
    return _maxerr(a, b) / scale


def _f64(t):
    return t.to(torch.float64).numpy() if torch.is_tensor(t) else np.asarray(t, dtype=np.float64)


def _conf_rel_err(gpu, b, st):
    """Largest relative error of a GPU draft confidence against the oracle's."""
    rho = 0.0
    for e in range(len(st.ex.token)):
        k = len(st.child_tok[e])
        want = np.asarray(st.child_q[e], dtype=np.float64)
        got = np.asarray(gpu["c_prob"][b, e, :k], dtype=np.float64)
        ok = want > 0
        if ok.any():
            rho = max(rho, float(np.max(np.abs(got[ok] - want[ok]) / want[ok])))
    return rho


def _value_tie(gpu, b, st, e_par, tok, v_ref, depth):
    """EAGLE-2 value near-tie: the GPU kept (child `tok` of expanded node
    `e_par`) where the oracle kept a node of value v_ref.  Values are products
    of at most `depth` draft confidences, so two values closer than twice
    depth x (the confidences' observed relative error + fp32 rounding) may
    order either way.  Returns a description, or None."""
    ex = st.ex
    if not 0 <= e_par < len(ex.token):
        return None
    ranks = [r for r, t in enumerate(st.child_tok[e_par]) if t == tok]
    if not ranks:
        return None
    v_gpu = ex.value[e_par] * float(st.child_q[e_par][ranks[0]])
    bound = 2.0 * depth * (_conf_rel_err(gpu, b, st) + 2.0 ** -23) * max(v_gpu, v_ref)
    gap = abs(v_gpu - v_ref)
    if gap <= bound:
        return f"values {v_ref:.9g} vs {v_gpu:.9g} (gap {gap:.2e} <= {bound:.2e})"
    return None


def _rerank_near_tie(gpu, b, st, tr, depth):
    """The final trees first differ at a slot whose two candidates are an
    EAGLE-2 value near-tie (see _value_tie)."""
    size = tr.size
    g_tok = [int(x) for x in gpu["t_token"][b, :size]]
    g_par = [int(x) for x in gpu["t_parent"][b, :size]]
    s = next((j for j in range(size) if (g_tok[j], g_par[j]) != (tr.token[j], tr.parent[j])), None)
    if s is None or s == 0:
        return None
    p = g_par[s]
    if not 0 <= p < s or tr.exp[p] < 0:
        return None
    tie = _value_tie(gpu, b, st, tr.exp[p], g_tok[s], tr.value[s], depth)
    return None if tie is None else f"slot {s}: {tie}"


def compare_round(w, gpu, ref, requests=None):
    """Returns a report dict; report['ok'] is False on any non-near-tie mismatch."""
    from oracle import philox
    from oracle.sampling import quantize
    tol = feature_tol(w)
    reqs = list(range(w.batch)) if requests is None else list(requests)
    rep = {"ok": True, "near_ties": [], "errors": [], "max_err": {}}

    def err(name, val, lim):
        rep["max_err"][name] = max(rep["max_err"].get(name, 0.0), val)
        if not val <= lim:
            rep["ok"] = False
            rep["errors"].append(f"{name}: {val:.3g} > {lim:g}")

    def fail(msg):
        rep["ok"] = False
        rep["errors"].append(msg)

    if gpu["status"] != 0:
        fail(f"device status {gpu['status']}")
    inp = gpu["inputs_cpu"]
    for i, b in enumerate(reqs):
        r = ref[i]
        st, tr = r["draft"], r["tree"]
        ex = st.ex
        temp = float(inp["temps"][b])
        diverged = False
        # draft head outputs, per expanded node in creation order
        for e in range(len(ex.token)):
            if int(gpu["p_token"][b, e]) != ex.token[e] or int(gpu["p_parent"][b, e]) != ex.parent[e]:
                tie = None
                if e > 0 and w.tree == "eagle2":
                    tie = _value_tie(gpu, b, st, int(gpu["p_parent"][b, e]), int(gpu["p_token"][b, e]),
                                     ex.value[e], w.depth)
                if tie is not None:
                    rep["near_ties"].append(f"b{b} frontier e{e}: {tie}")
                else:
                    fail(f"b{b} pool token e{e}: {int(gpu['p_token'][b, e])} vs {ex.token[e]}")
                diverged = True
                break
            err("f_hat", _maxerr_scaled(gpu["f_hat"][b, e], st.f_hat[e]), tol)
            err("logits", _maxerr_scaled(gpu["logits"][b, e], st.z[e]), tol)
            err("probs", _maxerr(gpu["probs"][b, e], st.q[e]), TOL_PROB)
            err("draft_k", _maxerr(gpu["dk_tree"][b, e], st.k_tree[e]), tol)
            k = len(st.child_tok[e])
            g_ch = [int(x) for x in gpu["c_token"][b, e, :k]]
            if g_ch != list(st.child_tok[e]):
                rank = next(j for j in range(k) if g_ch[j] != st.child_tok[e][j])
                a_tok, g_tok = st.child_tok[e][rank], g_ch[rank]
                if temp <= 0:
                    # two logits closer than twice the row's measured logit error
                    # (plus fp32 rounding of the logits themselves) may order either way
                    margin = abs(st.z[e][a_tok] - st.z[e][g_tok]) if g_tok >= 0 else np.inf
                    dz = _maxerr(gpu["logits"][b, e], st.z[e])
                    near = margin <= 2.0 * dz + 2.0 ** -22 * abs(st.z[e][a_tok])
                else:
                    u = philox.uniform_u32(inp["philox_seed"], rank, e, philox.PURPOSE_DRAW, b, inp["round_id"])
                    wq = quantize(st.q[e]).astype(np.float64)
                    for t in st.child_tok[e][:rank]:
                        wq[t] = 0.0
                    cdf = np.cumsum(wq) / wq.sum()
                    margin = float(np.min(np.abs(cdf - u / 2.0 ** 32)))
                    # q = softmax(z / T): a logit error dz moves every CDF point by at
                    # most 2 max|dz| / T (relative to the remaining mass)
                    dz = _maxerr(gpu["logits"][b, e], st.z[e])
                    rem = wq.sum() / max(1.0, float(quantize(st.q[e]).sum()))
                    near = margin < 2.0 * dz / temp / max(rem, 1e-12) + 1e-6
                if near:
                    rep["near_ties"].append(f"b{b} children e{e} rank{rank} margin {margin:.2e}")
                    diverged = True
                    break
                fail(f"b{b} children of e{e}: {g_ch} vs {list(st.child_tok[e])}")
                diverged = True
                break
            err("child_prob", _maxerr(gpu["c_prob"][b, e, :k], st.child_q[e]), TOL_PROB)
        if diverged:
            continue
        # tree
        size = tr.size
        if int(gpu["t_size"][b]) != size:
            fail(f"b{b} tree size {int(gpu['t_size'][b])} vs {size}")
            continue
        tie = _rerank_near_tie(gpu, b, st, tr, w.depth)
        if tie is not None:
            rep["near_ties"].append(f"b{b} rerank {tie}")
            continue
        for name, mine, want in (("token", gpu["t_token"], tr.token), ("parent", gpu["t_parent"], tr.parent),
                                 ("depth", gpu["t_depth"], tr.depth), ("exp", gpu["t_exp"], tr.exp)):
            got = [int(x) for x in mine[b, :size]]
            if got != list(want):
                fail(f"b{b} tree {name}: {got} vs {list(want)}")
                diverged = True
        anc = [int(x) & 0xFFFFFFFFFFFFFFFF for x in gpu["t_anc"][b, :size]]
        if anc != list(tr.anc):
            fail(f"b{b} tree anc differs")
            diverged = True
        pos = [int(x) for x in gpu["t_pos"][b, :size]]
        if pos != [inp["prefix_len"][b] + dd for dd in tr.depth]:
            fail(f"b{b} tree pos differs")
        if diverged:
            continue
        # verification attention, target distribution
        err("verify_out", _maxerr(gpu["attn_out"][b, :size], r["verify_out"]), tol)
        for s_ in range(size):
            err("target_logits", _maxerr_scaled(gpu["target_logits"][b, s_], r["target_logits"][s_]), tol)
        if temp > 0:
            err("target_probs", _maxerr(gpu["target_probs"][b, :size], r["target_probs"]), TOL_PROB)
        # acceptance
        a = int(gpu["accept_len"][b])
        path = [int(x) for x in gpu["path"][b, :a + 1]]
        final = int(gpu["final_token"][b])
        if (a, path, final) != (r["accept_len"], list(r["path"]), r["final"]):
            fail(f"b{b} accept: gpu ({a}, {path}, {final}) vs oracle ({r['accept_len']}, {r['path']}, {r['final']})")
            continue
        # commit
        cm = r["commit"]
        toks = [int(x) for x in gpu["tok_commit"][b, :a + 2]]
        if toks != cm["tok_commit"]:
            fail(f"b{b} tok_commit {toks} vs {cm['tok_commit']}")
        err("f_commit", _maxerr(gpu["f_commit"][b, :a + 1], cm["f_commit"]), 0.0)
        err("f_last", _maxerr(gpu["f_last_out"][b], cm["f_last"]), 0.0)
        if int(gpu["t_next_out"][b]) != cm["t_next"] or int(gpu["prefix_len_out"][b]) != cm["prefix_len"]:
            fail(f"b{b} next-round state differs")
        if int(gpu["draft_len_out"][b]) != cm["draft_len"]:
            fail(f"b{b} draft_len differs")
        L = inp["prefix_len"][b]
        got_kv = _f64(gpu["tgt_k_after"][b, L:L + a + 1])
        err("kv_commit", _maxerr(got_kv, cm["kv_rows_k"]), 0.0)
        Ld = inp["draft_len"][b]
        root_k = np.asarray(cm["draft_root_k"])
        # the cache is bf16: the appended row carries one bf16 rounding (2^-9 relative)
        err("draft_kv_append", _maxerr(_f64(gpu["draft_k"][b, Ld]), root_k),
            tol + 2.0 ** -8 * float(np.max(np.abs(root_k))))
    return rep
