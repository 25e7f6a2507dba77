"""Wiring of the seeded synthetic workloads (eagle_synth) to the runtime:
capacities, dims, loading one round's inputs into a Round, and the
synthetic target's logits.  Marshalling only."""
from __future__ import annotations

import torch

import eagle_synth as S
from eagle_synth.standin import target_logits_from_draft

from . import runtime as R


def limits_for(w):
    if w.tree == "eagle2":
        rows = w.batch * w.top_k
    else:
        plan = R.plan_for(w.tree)
        rows = w.batch * max(plan.layer_rows[l] for l in range(plan.n_layers))
    rows = max(rows, w.batch * w.depth)     # the draft-cache refresh of a whole accepted path
    return dict(max_batch=w.batch, max_rows=rows, max_expanded=S.max_expanded(w), max_children=w.top_k,
                max_tree=1 + w.top_m)


def dims_of(w):
    return dict(d=w.d, n_q_heads=w.n_q_heads, n_kv_heads=w.n_kv_heads, head_dim=w.head_dim, d_ff=w.d_ff,
                vocab=w.vocab, rms_eps=w.rms_eps, rope_theta=w.rope_theta)


def make_round(w, inp, device="cuda"):
    eng = R.Engine(dims_of(w), max_prefix=inp["kv_cap"], device=device, **limits_for(w))
    plan = R.plan_for(w.tree, w.top_k, w.depth, w.top_m)
    rd = R.Round(eng, plan, w.batch, inp["kv_cap"])
    load_round(rd, inp)
    return eng, rd


def load_round(rd, inp):
    dev = rd.eng.device
    L = torch.tensor(inp["prefix_len"], dtype=torch.int32, device=dev)
    rd.t_next.copy_(inp["t_next"])
    rd.f_last.copy_(inp["f_last"])
    rd.pos0.copy_(L)
    rd.temps.copy_(torch.tensor(inp["temps"], dtype=torch.float32, device=dev))
    rd.draft_k.copy_(inp["draft_k"])
    rd.draft_v.copy_(inp["draft_v"])
    rd.draft_len.copy_(torch.tensor(inp["draft_len"], dtype=torch.int32, device=dev))
    rd.tgt_k[0].copy_(inp["tgt_k"])
    rd.tgt_v[0].copy_(inp["tgt_v"])
    rd.tgt_len.copy_(L)
    rd.tree_q.copy_(inp["tree_q"])
    rd.tree_k[0].copy_(inp["tree_k"])
    rd.tree_v[0].copy_(inp["tree_v"])
    rd.f_true.copy_(inp["f_true"])
    rd.set_sampling(inp["philox_seed"], inp["round_id"])


def standin(inp):
    """target_fn for Round.run: the synthetic target's logits for this tree."""
    def fn(rd):
        target_logits_from_draft(rd.logits, rd.t_exp, inp["tgt_noise"], inp["tgt_fresh"], rd.target_logits)
    return fn


def weight_bytes_per_forward(w) -> int:
    """bf16 bytes one draft forward must stream: FC, QKV, O, gate/up, down, LM head."""
    qd, kvd = w.n_q_heads * w.head_dim, w.n_kv_heads * w.head_dim
    params = 2 * w.d * w.d + (qd + 2 * kvd) * w.d + w.d * qd + 3 * w.d * w.d_ff + w.vocab * w.d
    return 2 * params


def gemm_weight_bytes(w):
    """Algorithmic bytes (bf16 weights) of each GEMM class per launch."""
    qd, kvd = w.n_q_heads * w.head_dim, w.n_kv_heads * w.head_dim
    return {"gemm_fc": 2 * 2 * w.d * w.d, "gemm_qkv": 2 * (qd + 2 * kvd) * w.d, "gemm_o": 2 * w.d * qd,
            "gemm_gateup": 2 * 2 * w.d_ff * w.d, "gemm_down": 2 * w.d * w.d_ff, "gemm_lm": 2 * w.vocab * w.d}
