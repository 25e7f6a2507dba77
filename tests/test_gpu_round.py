"""GPU parity: whole rounds through the C ABI against the oracle, element by
element, on small cases that span several tiles and ragged tails, and on the
full-size workloads (sampled requests)."""
import json

import pytest
import torch

import eagle_synth as S
from tests.gpu_harness import compare_round, run_gpu_round, run_oracle_round

SMALL = {
    "tiny_greedy_static8": S.WORKLOADS["tiny_fp32"],
    "tiny_sampling_static8": S.variant("tiny_fp32", name="tiny_sampling_static8", temps=(1.0,)),
    "tiny_greedy_chain4": S.variant("tiny_fp32", name="tiny_greedy_chain4", tree="chain4", top_k=1, depth=4,
                                    top_m=4),
    "tiny_sampling_chain4": S.variant("tiny_fp32", name="tiny_sampling_chain4", tree="chain4", top_k=1,
                                      depth=4, top_m=4, temps=(1.0,)),
    "small_eagle2_gqa_mixed": S.variant("70b_x16_eagle2", name="small_eagle2_gqa_mixed", d=256, n_q_heads=8,
                                        n_kv_heads=2, head_dim=32, d_ff=688, vocab=1000, batch=3,
                                        prefix_len=100, top_k=4, depth=4, top_m=12, weight_std=0.05),
    "small_static26_dh128": S.variant("7b_static26", name="small_static26_dh128", d=256, n_q_heads=2,
                                      n_kv_heads=2, head_dim=128, d_ff=688, vocab=2000, prefix_len=300,
                                      weight_std=0.05),
    "small_eagle2_ragged_k10": S.variant("13b_x8_eagle2", name="small_eagle2_ragged_k10", d=128, n_q_heads=2,
                                         n_kv_heads=2, head_dim=64, d_ff=344, vocab=3000, batch=4,
                                         prefix_range=(50, 400), weight_std=0.05),
    "small_rows160_two_mma": S.variant("70b_x16_eagle2", name="small_rows160_two_mma", d=128, n_q_heads=4,
                                       n_kv_heads=2, head_dim=32, d_ff=256, vocab=700, prefix_len=64,
                                       weight_std=0.05),
    # 160 activation rows against a 19520-wide MLP: one accumulator fits
    # (2 x 160 columns), gate/up's 305 tiles over 152 CTAs, so CTAs own two
    # whole tiles after their split share and free the accumulator of the
    # first before its epilogue
    "small_mlp_rows160_f19520": S.variant("70b_x16_eagle2", name="small_mlp_rows160_f19520", d=128, n_q_heads=4,
                                          n_kv_heads=2, head_dim=32, d_ff=19520, vocab=1000, prefix_len=64,
                                          temps=(0.0,), depth=3, top_m=20, weight_std=0.05),
    # an odd vocabulary (1001: the selection's unvectorised slice reads, the
    # LM head's row tail) with greedy and sampled requests mixed
    "small_eagle2_v1001_mixed": S.variant("70b_x16_eagle2", name="small_eagle2_v1001_mixed", d=128, n_q_heads=4,
                                          n_kv_heads=2, head_dim=32, d_ff=256, vocab=1001, batch=4,
                                          prefix_len=80, top_k=4, depth=3, top_m=12, weight_std=0.05),
    # trees past 63 nodes (multi-word ancestor masks): EAGLE-2 pools of 73 and
    # 71 expanded slots (two mask words) with trees of 121 and 256 slots (two
    # and four words), and a 120-node static template
    "small_eagle2_m120_k8_d10": S.variant("70b_x16_eagle2", name="small_eagle2_m120_k8_d10", d=128, n_q_heads=4,
                                          n_kv_heads=2, head_dim=32, d_ff=256, vocab=700, batch=2, prefix_len=64,
                                          top_k=8, depth=10, top_m=120, weight_std=0.05),
    "small_eagle2_m255_k10_d8": S.variant("70b_x16_eagle2", name="small_eagle2_m255_k10_d8", d=128, n_q_heads=4,
                                          n_kv_heads=2, head_dim=32, d_ff=256, vocab=1500, batch=2, prefix_len=90,
                                          top_k=10, depth=8, top_m=255, weight_std=0.05),
    "small_ternary4_m120": S.variant("7b_static26", name="small_ternary4_m120", tree="ternary4", top_k=3, depth=4,
                                     top_m=120, d=128, n_q_heads=2, n_kv_heads=2, head_dim=64, d_ff=344, vocab=900,
                                     prefix_len=70, weight_std=0.05),
    # verification with more than 32 query rows per kv head at head_dim 128
    # (the tensor-memory kernel): 164 rows in two row blocks over a
    # five-split prefix (partials merged), and 42 rows for 160 (request, kv
    # head) pairs (one split each, written directly)
    "small_tc_merge_dh128": S.variant("70b_x16_eagle2", name="small_tc_merge_dh128", d=256, n_q_heads=8,
                                      n_kv_heads=2, head_dim=128, d_ff=512, vocab=1000, batch=3, prefix_len=300,
                                      top_k=4, depth=4, top_m=40, weight_std=0.05),
    "small_tc_direct_dh128": S.variant("70b_x16_eagle2", name="small_tc_direct_dh128", d=512, n_q_heads=16,
                                       n_kv_heads=8, head_dim=128, d_ff=512, vocab=500, batch=20, prefix_len=100,
                                       top_k=3, depth=3, top_m=20, weight_std=0.05),
    # the draft layer on the tensor-memory kernel (head_dim 128, 8 or more
    # query rows per kv head): 80 rows per kv head (8 query heads of one kv
    # head, k = 10) over a 700-key prefix with a 60-key partial tile, 248
    # verification rows in two row blocks; and 10 rows per kv head (MHA,
    # k = 10, depth 6: a 51-slot draft tree in two 32-key tiles) over ragged
    # prefixes split one 64-key tile per CTA, 61 verification rows
    "small_ws_g8_k10_dh128": S.variant("70b_x16_eagle2", name="small_ws_g8_k10_dh128", d=256, n_q_heads=8,
                                       n_kv_heads=1, head_dim=128, d_ff=512, vocab=1000, batch=2, prefix_len=700,
                                       top_k=10, depth=4, top_m=30, weight_std=0.05),
    "small_ws_mha_k10_dh128": S.variant("13b_x8_eagle2", name="small_ws_mha_k10_dh128", d=256, n_q_heads=2,
                                        n_kv_heads=2, head_dim=128, d_ff=512, vocab=1500, batch=3,
                                        prefix_range=(50, 900), top_k=10, depth=6, top_m=60, weight_std=0.05),
}


def _check(w, rep, reqs):
    """Every compared request reaches the commit.  Near-ties are logged with
    their margins; each one is within the measured floating-point difference
    of its inputs (else compare_round fails).  Sampling draws: their count
    per request stays within what the measured CDF differences predict (the
    expected count is the sum over draws of the gaps between the two sides'
    CDF boundaries); every other kind of decision: at most one per request.
    The report is printed so the log carries every tensor's plain max-abs
    error."""
    print(w.name, json.dumps({k: rep[k] for k in ("max_err", "max_err_rms", "f_hat_by_depth", "near_ties",
                                                   "expected_flips")}))
    if not rep["ok"]:
        pytest.fail(json.dumps({k: v for k, v in rep.items() if k != "ok"}, indent=1, default=str))
    assert rep["reached"] == {b: "commit" for b in reqs}, rep["reached"]
    draws, other = {}, {}
    for t in rep["near_ties"]:
        kind = draws if (t["stage"] == "children" and " draw" in t["where"]) else other
        kind[t["request"]] = kind.get(t["request"], 0) + 1
    assert all(n <= 1 for n in other.values()), rep["near_ties"]
    for b, n in draws.items():
        mu = rep["expected_flips"].get(b, 0.0)
        assert n <= 2 + 3 * mu + 4 * mu ** 0.5, (b, n, mu, rep["near_ties"])


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(SMALL))
def test_round_parity_small(name):
    w = SMALL[name]
    seed = 77
    gpu = run_gpu_round(w, seed)
    ref = run_oracle_round(w, seed, gpu["inputs_cpu"], gpu["weights_cpu"], gpu=gpu)
    rep = compare_round(w, gpu, ref)
    _check(w, rep, list(range(w.batch)))


FULL = {"7b_static26": None, "7b_eagle2": None, "13b_x8_eagle2": [0, 3, 7], "70b_x16_eagle2": [0, 1]}


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(FULL))
def test_round_parity_full_size(name):
    """Full-size workloads in the bench's launch configuration; the oracle
    recomputes the listed requests (all when None)."""
    w = S.WORKLOADS[name]
    seed = S.WORKLOAD_SEEDS[name]
    gpu = run_gpu_round(w, seed)
    reqs = FULL[name]
    ref = run_oracle_round(w, seed, gpu["inputs_cpu"], gpu["weights_cpu"], requests=reqs, gpu=gpu)
    rep = compare_round(w, gpu, ref, requests=reqs)
    _check(w, rep, list(range(w.batch)) if reqs is None else reqs)


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["small_eagle2_gqa_mixed", "tiny_greedy_static8"])
def test_graph_replay_matches_eager(name):
    """The round captured as one CUDA graph reproduces the eager round bit for
    bit (the kernels are deterministic: fixed-order reductions, no atomics on
    values)."""
    from eagle_feature_level_gb300.workload import make_round, standin
    w = SMALL[name]
    W = S.draft_weights(w, 5, device="cuda")
    inp = S.round_inputs(w, 5, device="cuda")
    eng, rd = make_round(w, inp)
    wc = eng.weights(W)
    rd.run(wc, target_fn=standin(inp))
    torch.cuda.synchronize()
    fields = ["f_hat", "logits", "probs", "c_token", "t_token", "t_anc", "attn_out", "accept_len", "path",
              "final_token", "tok_commit", "f_last_out"]
    eager = {k: getattr(rd, k).clone() for k in fields}
    g = rd.capture(wc)
    for k in fields:
        getattr(rd, k).zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    for k in fields:
        assert torch.equal(getattr(rd, k), eager[k]), k
    assert eng.status() == 0
    eng.close()
