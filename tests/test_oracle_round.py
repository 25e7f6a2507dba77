"""The oracle's whole round on small variants of the workloads (CPU only):
state consistency after commit (Page B "正确性与状态边界": target KV, drafter
state and committed length agree after verification)."""
import numpy as np
import pytest

import eagle_synth as S
from oracle.layer import DraftWeights
from oracle.round import run_round

SMALL = {
    "eagle2_gqa": S.variant("70b_x16_eagle2", d=128, n_q_heads=8, n_kv_heads=2, head_dim=32,
                            d_ff=344, vocab=700, batch=2, prefix_len=40, top_k=4, depth=4,
                            top_m=12, weight_std=0.05),
    "static26": S.variant("7b_static26", d=128, n_q_heads=4, n_kv_heads=4, head_dim=32,
                          d_ff=344, vocab=600, prefix_len=33, weight_std=0.05),
    "chain4_sampling": S.variant("tiny_fp32", tree="chain4", top_k=1, depth=4, top_m=4,
                                 temps=(1.0,)),
}


@pytest.mark.parametrize("name", list(SMALL))
def test_round_state_is_consistent(name):
    w = SMALL[name]
    seed = 4242
    Wd = DraftWeights(S.draft_weights(w, seed), w)
    inp = S.round_inputs(w, seed)
    res = run_round(Wd, w, inp)
    assert len(res) == w.batch
    for b, r in enumerate(res):
        tr, cm = r["tree"], r["commit"]
        L = inp["prefix_len"][b]
        assert tr.size == 1 + w.top_m
        assert tr.token[0] == int(inp["t_next"][b])
        # path is a root-to-node chain of the tree
        for a, s in zip(r["path"], r["path"][1:]):
            assert tr.parent[s] == a
        assert cm["prefix_len"] == L + 1 + r["accept_len"]
        assert cm["kv_positions"] == list(range(L, L + r["accept_len"] + 1))
        tk = inp["tree_k"][b].to(dtype=__import__("torch").float64).numpy()
        np.testing.assert_array_equal(cm["kv_rows_k"], tk[r["path"]])
        assert cm["tok_commit"][-1] == cm["t_next"] == r["final"]
        assert 0 <= r["final"] < w.vocab
        # q rows are distributions
        for e, q in r["draft"].q.items():
            assert abs(q.sum() - 1.0) < 1e-12


def test_refresh_rows_are_the_draft_layers_kv_of_those_rows():
    """draft_refresh_rows gives, for a row (feature, token, position), the
    K/V the draft step computes for a node with that parent feature, token
    and position: the root row of a round is one."""
    import eagle_synth as S
    from oracle.layer import DraftWeights
    from oracle.round import draft_refresh_rows, draft_tree, numpy_inputs
    w = S.WORKLOADS["tiny_fp32"]
    seed = S.WORKLOAD_SEEDS["tiny_fp32"]
    Wd = DraftWeights(S.draft_weights(w, seed), w)
    inp = numpy_inputs(S.round_inputs(w, seed))
    st, _ = draft_tree(Wd, w, 0, inp)
    k, v = draft_refresh_rows(Wd, w, inp["f_last"][:1], [inp["t_next"][0]], [inp["prefix_len"][0]])
    assert np.array_equal(k[0], st.k_tree[0]) and np.array_equal(v[0], st.v_tree[0])
