"""Graph replay at discrete tree budgets, against the oracle.

[B] "部署前要确认的兼容边界": graphs are captured per tree shape.  One round
buffer set, sized for the largest budget, holds several EAGLE-2 budgets
(depth, retained nodes); each is captured as two CUDA graphs around the
target model -- (draft, tree, verification attention) and (acceptance,
commit, draft-cache refresh) -- and replayed with the synthetic target run
between them.  Every replayed round is compared with the oracle element by
element (the oracle following the GPU's discrete choices)."""
import pytest
import torch

import eagle_synth as S
from eagle_feature_level_gb300 import runtime as R
from eagle_feature_level_gb300.workload import make_round, standin
from tests.gpu_harness import GPU_FIELDS, compare_round, run_oracle_round

pytestmark = pytest.mark.gpu

BASE = S.variant("70b_x16_eagle2", name="graphs_eagle2_gqa", d=256, n_q_heads=8, n_kv_heads=2, head_dim=32,
                 d_ff=688, vocab=1000, batch=3, prefix_len=100, top_k=4, depth=4, top_m=12, weight_std=0.05)
BUDGETS = [(4, 12), (3, 6), (4, 5)]      # (depth, retained nodes); the first is the buffers' size


def test_budget_graphs_against_the_oracle():
    w = BASE
    seed = 303
    W = S.draft_weights(w, seed, device="cuda")
    inp = S.round_inputs(w, seed, device="cuda")
    eng, rd = make_round(w, inp)
    w_c = eng.weights(W)
    inputs_cpu = {k: (v.detach().to("cpu") if torch.is_tensor(v) else v) for k, v in inp.items()}
    W_cpu = {k: v.cpu() for k, v in W.items()}
    state = {k: getattr(rd, k).clone() for k in ("draft_len", "tgt_len")}
    caches = (rd.draft_k.clone(), rd.draft_v.clone(), rd.tgt_k[0].clone(), rd.tgt_v[0].clone())
    graphs = {}
    for depth, m in BUDGETS:
        rd.set_plan(R.plan_for("eagle2", w.top_k, depth, m))
        rd.run(w_c, target_fn=standin(inp))                # warm-up before capture
        torch.cuda.synchronize()
        graphs[(depth, m)] = rd.capture_segments(w_c, refresh=True)
    for depth, m in BUDGETS:
        # the same round state before every replay (the commit appended rows)
        for k, t in state.items():
            getattr(rd, k).copy_(t)
        for dst, src in zip((rd.draft_k, rd.draft_v, rd.tgt_k[0], rd.tgt_v[0]), caches):
            dst.copy_(src)
        for k in ("f_hat", "logits", "probs", "c_token", "t_token", "attn_out", "accept_len", "path",
                  "final_token", "tok_commit", "f_last_out", "f_commit"):
            getattr(rd, k).zero_()
        rd.set_plan(R.plan_for("eagle2", w.top_k, depth, m))
        pre, post = graphs[(depth, m)]
        pre.replay()
        standin(inp)(rd)                                    # the target, between the two graphs
        post.replay()
        torch.cuda.synchronize()
        gpu = {k: getattr(rd, k).detach().to("cpu") for k in GPU_FIELDS}
        gpu["tgt_k_after"] = rd.tgt_k[0].detach().to("cpu")
        gpu["status"] = eng.status()
        gpu["inputs_cpu"] = inputs_cpu
        wb = S.variant("70b_x16_eagle2", name=f"graphs_d{depth}_m{m}", d=w.d, n_q_heads=w.n_q_heads,
                       n_kv_heads=w.n_kv_heads, head_dim=w.head_dim, d_ff=w.d_ff, vocab=w.vocab, batch=w.batch,
                       prefix_len=w.prefix_len, top_k=w.top_k, depth=depth, top_m=m, weight_std=w.weight_std)
        ref = run_oracle_round(wb, seed, inputs_cpu, W_cpu, gpu=gpu)
        rep = compare_round(wb, gpu, ref)
        assert rep["ok"], ((depth, m), rep["errors"])
        assert rep["reached"] == {b: "commit" for b in range(w.batch)}, ((depth, m), rep["reached"])
        assert all(int(s) == m + 1 for s in rd.t_size.cpu()), (depth, m)
        # the refresh in the second graph appended the accepted path
        a = rd.accept_len.cpu()
        assert rd.draft_len_next.cpu().tolist() == [int(state["draft_len"][b]) + 1 + int(a[b]) for b in range(w.batch)]
    eng.close()
