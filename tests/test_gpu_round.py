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
}


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(SMALL))
def test_round_parity_small(name):
    w = SMALL[name]
    seed = 77
    gpu = run_gpu_round(w, seed)
    ref = run_oracle_round(w, seed, gpu["inputs_cpu"], gpu["weights_cpu"])
    rep = compare_round(w, gpu, ref)
    if not rep["ok"]:
        pytest.fail(json.dumps(rep, indent=1))
    # A decision between two candidates closer than the measured fp32 error
    # (two logits 2.8e-8 apart in small_eagle2_ragged_k10; two EAGLE-2 node
    # values 2.4e-6 apart relative in small_rows160_two_mma) is flagged and
    # skips only that request's later stages; at most one request in eight.
    assert len(rep["near_ties"]) <= max(1, w.batch // 8), rep


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
    ref = run_oracle_round(w, seed, gpu["inputs_cpu"], gpu["weights_cpu"], requests=reqs)
    rep = compare_round(w, gpu, ref, requests=reqs)
    if not rep["ok"]:
        pytest.fail(json.dumps(rep, indent=1))
    # sampling at T > 0 over V = 32000 nearly flat draft distributions: a draw can
    # land within the fp32-vs-fp64 CDF difference of a boundary; such draws are
    # flagged (not failed) and the request's later stages are compared only
    # when no flag was raised.  Greedy requests must never flag a child choice.
    greedy = [b for b in (reqs or range(w.batch)) if w.temps_for_batch()[b] <= 0]
    assert not any(f"b{b} children " in t for t in rep["near_ties"] for b in greedy), rep


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
