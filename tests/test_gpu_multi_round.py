"""Several rounds in a row against the oracle, with non-trivial acceptance.

Each round of the loop (draft, tree, verification, acceptance, commit, the
draft-cache refresh of the accepted path, and the hand-over of the committed
state) is compared with the oracle element by element, the oracle following
the GPU's discrete choices (tests/gpu_harness.py).  Between rounds the state
the GPU hands over is checked against what the round defines ([B] "KV Cache
必须按事务提交"; [A] §6.2 closing remark): the target cache gained exactly
the committed path's K/V rows, the draft cache the root row and the refresh
rows (the oracle's draft-layer K/V of [true feature of p - 1 ; token at p]),
lengths advanced by 1 + accept length, t_next = the final token, f_last = the
last accepted slot's true feature.  The next oracle round then starts from
the GPU's state.  The synthetic target (draft logits + N(0, 0.5^2) noise)
gives acceptance lengths well above zero, so the refresh and the cache
appends carry real rows."""
import numpy as np
import pytest
import torch

import eagle_synth as S
from eagle_feature_level_gb300.workload import make_round
from oracle.layer import DraftWeights
from oracle.round import draft_refresh_rows
from tests.gpu_harness import compare_round, round_on, run_oracle_round

pytestmark = pytest.mark.gpu

ROUNDS = 4
CASES = {
    "static26_greedy": S.variant("7b_static26", name="multi_static26", d=256, n_q_heads=2, n_kv_heads=2,
                                 head_dim=128, d_ff=688, vocab=2000, prefix_len=300, weight_std=0.05),
    "eagle2_gqa_mixed": S.variant("70b_x16_eagle2", name="multi_eagle2_gqa", d=256, n_q_heads=8, n_kv_heads=2,
                                  head_dim=32, d_ff=688, vocab=1000, batch=3, prefix_len=100, top_k=4, depth=4,
                                  top_m=12, weight_std=0.05),
}


def _with_room(inp, extra):
    """Round inputs whose caches have `extra` more rows (zeros)."""
    out = dict(inp)
    for k in ("draft_k", "draft_v", "tgt_k", "tgt_v"):
        t = inp[k]
        out[k] = torch.cat([t, torch.zeros(t.shape[0], extra, *t.shape[2:], dtype=t.dtype, device=t.device)], 1)
    out["kv_cap"] = inp["kv_cap"] + extra
    return out


def _state(rd, base_cpu):
    """Host copy of the round inputs as the GPU holds them now."""
    inp = dict(base_cpu)
    inp["prefix_len"] = [int(x) for x in rd.pos0.cpu()]
    inp["draft_len"] = [int(x) for x in rd.draft_len.cpu()]
    inp["t_next"] = rd.t_next.cpu()
    inp["f_last"] = rd.f_last.cpu()
    for k, t in (("draft_k", rd.draft_k), ("draft_v", rd.draft_v), ("tgt_k", rd.tgt_k[0]), ("tgt_v", rd.tgt_v[0])):
        inp[k] = t.cpu()
    inp["round_id"] = rd.round_id
    return inp


@pytest.mark.parametrize("name", list(CASES))
def test_rounds_in_a_row_against_the_oracle(name):
    w = CASES[name]
    seed = 91
    W = S.draft_weights(w, seed, device="cuda")
    W_cpu = {k: v.cpu() for k, v in W.items()}
    Wd = DraftWeights(W_cpu, w)
    inp = _with_room(S.round_inputs(w, seed, device="cuda"), ROUNDS * (w.depth + 1))
    eng, rd = make_round(w, inp)
    w_c = eng.weights(W)
    base_cpu = {k: (v.detach().to("cpu") if torch.is_tensor(v) else v) for k, v in inp.items()}
    accepted = []
    for r in range(ROUNDS):
        rd.set_sampling(inp["philox_seed"], 7 + r)
        start = _state(rd, base_cpu)
        gpu = round_on(eng, rd, w_c, inp, start)
        ref = run_oracle_round(w, seed, start, W_cpu, gpu=gpu)
        rep = compare_round(w, gpu, ref)
        assert rep["ok"], (r, rep["errors"])
        assert rep["reached"] == {b: "commit" for b in range(w.batch)}, (r, rep["reached"])
        rd.refresh(w_c)
        torch.cuda.synchronize()
        assert eng.status() == 0, r
        for b in range(w.batch):
            a = int(rd.accept_len[b])
            accepted.append(a)
            L, Ld = start["prefix_len"][b], start["draft_len"][b]
            assert int(rd.draft_len_next[b]) == Ld + 1 + a and int(rd.prefix_len_out[b]) == L + 1 + a
            toks = rd.tok_commit[b, :a + 2].tolist()
            fc = rd.f_commit[b, :a + 1].double().cpu().numpy()
            if a:
                kr, vr = draft_refresh_rows(Wd, w, fc[:a], toks[1:a + 1], range(L + 1, L + 1 + a))
                got_k = rd.draft_k[b, Ld + 1:Ld + 1 + a].double().cpu().numpy()
                got_v = rd.draft_v[b, Ld + 1:Ld + 1 + a].double().cpu().numpy()
                assert np.all(np.abs(got_k - kr) <= 2e-2 + 2.0 ** -8 * np.abs(kr)), (r, b)
                assert np.all(np.abs(got_v - vr) <= 2e-2 + 2.0 ** -8 * np.abs(vr)), (r, b)
            # rows past the new lengths are untouched
            assert torch.equal(rd.draft_k[b, Ld + 1 + a:].cpu(), start["draft_k"][b, Ld + 1 + a:]), (r, b)
            assert torch.equal(rd.tgt_k[0][b, L + 1 + a:].cpu(), start["tgt_k"][b, L + 1 + a:]), (r, b)
            assert int(rd.t_next_out[b]) == toks[-1]
            assert torch.equal(rd.f_last_out[b].cpu(), rd.f_commit[b, a].cpu())
        rd.advance()
    assert sum(accepted) > 0, accepted
    print(name, "accept lengths", accepted)
    eng.close()
