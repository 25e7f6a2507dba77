"""Several rounds in a row (the multi-round decode loop) and the draft-cache
refresh, on the GPU.

[B] "KV Cache 必须按事务提交": after a round the target cache holds exactly
the committed path and the drafter continues from the committed path;
[B] "正确性与状态边界": under greedy decoding the tokens EAGLE commits equal
those of plain decoding with the target.  The loop: the tiny workload's
2-layer random-init target (GPU stand-in, tests/gpu_tiny_target.py) fills
both caches from a prompt -- the draft cache through eagle_draft_refresh over
the prompt's true features -- then each round drafts a tree, runs the target
over it, accepts, commits both target layers' K/V, appends the accepted
path's draft K/V (eagle_draft_refresh) and hands the committed state to the
next round.  The oracle's TinyTarget (fp64) is the checker: the committed
sequence must be its greedy decoding of the prompt, token for token, except
where the oracle's own top-two logit gap is within the measured difference
of the two targets' logits (a near-tie, after which the check continues on
the GPU's sequence)."""
import numpy as np
import pytest
import torch

import eagle_synth as S
from eagle_feature_level_gb300 import _binding as B
from eagle_feature_level_gb300 import runtime as R
from eagle_feature_level_gb300.runtime import _p
from eagle_feature_level_gb300.workload import dims_of, limits_for
from oracle.layer import DraftWeights
from oracle.round import draft_refresh_rows
from oracle.target import TinyTarget
from tests.gpu_tiny_target import GpuTinyTarget

pytestmark = pytest.mark.gpu

ROUNDS = 10


def _bf16_bound(ref, tol):
    return tol + 2.0 ** -8 * np.abs(ref)


def _refresh_call(eng, w_c, batch, f_rows, tok_rows, n_act, pos0, k, v, cap, len_in, len_out):
    path_cap = f_rows.shape[1]
    acc = B.eagle_accept_out(_p(n_act), 0, 0, 0, path_cap)
    cm = B.eagle_commit_out(_p(f_rows), _p(tok_rows), 0, 0, 0, 0)
    kv = B.eagle_kv(_p(k), _p(v), cap, _p(len_in))
    B.eagle_draft_refresh(eng.ctx, batch, w_c, acc, cm, _p(pos0), kv, _p(len_out), eng.ws.data_ptr(), eng.stream())


def test_refresh_rows_match_the_oracle():
    """Ragged accept lengths over four requests (0, 1, 3 and the maximum), a
    fifth request whose cache cannot take its rows (nothing written, length
    kept, EAGLE_ERR_CAPACITY): appended rows against the oracle's draft
    layer K/V of the same rows, everything else untouched."""
    w = S.variant("13b_x8_eagle2", name="refresh_small", d=128, n_q_heads=4, n_kv_heads=2, head_dim=32, d_ff=256,
                  vocab=900, batch=5, prefix_len=40, weight_std=0.05)
    seed = 61
    W = S.draft_weights(w, seed, device="cuda")
    dims = dims_of(w)
    Rmax, cap, Bn = 6, 64, 5
    eng = R.Engine(dims, max_batch=Bn, max_rows=Bn * Rmax, max_expanded=4, max_children=4, max_tree=8,
                   max_prefix=cap, device="cuda")
    w_c = eng.weights(W)
    f_rows = S.random_tensor((Bn, Rmax + 1, w.d), seed, "refresh_f").cuda()
    tok_rows = S.random_ints(0, w.vocab, (Bn, Rmax + 2), seed, "refresh_tok").int().cuda()
    n_act = torch.tensor([0, 1, 3, Rmax, 2], dtype=torch.int32, device="cuda")
    pos0 = torch.tensor([40, 17, 55, 3, 60], dtype=torch.int32, device="cuda")
    len_in = torch.tensor([10, 0, 30, 57, cap - 1], dtype=torch.int32, device="cuda")   # request 4: no room for 2
    len_out = torch.full((Bn,), -7, dtype=torch.int32, device="cuda")
    Hkv, dh = w.n_kv_heads, w.head_dim
    k = torch.full((Bn, cap, Hkv, dh), 3.0, dtype=torch.bfloat16, device="cuda")
    v = torch.full_like(k, -3.0)
    _refresh_call(eng, w_c, Bn, f_rows, tok_rows, n_act, pos0, k, v, cap, len_in, len_out)
    torch.cuda.synchronize()
    assert eng.status() == 4                      # EAGLE_ERR_CAPACITY from request 4
    assert len_out.tolist() == [10, 1, 33, 57 + Rmax, cap - 1]
    Wd = DraftWeights({n: t.cpu() for n, t in W.items()}, w)
    fr, tr = f_rows.cpu().double().numpy(), tok_rows.cpu().numpy()
    kc, vc = k.cpu().double().numpy(), v.cpu().double().numpy()
    for b in range(Bn):
        a = int(n_act[b]) if b != 4 else 0
        L0, p0 = int(len_in[b]), int(pos0[b])
        if a:
            kr, vr = draft_refresh_rows(Wd, w, fr[b, :a], tr[b, 1:a + 1], [p0 + i for i in range(1, a + 1)])
            assert np.all(np.abs(kc[b, L0:L0 + a] - kr) <= _bf16_bound(kr, 2e-4)), b
            assert np.all(np.abs(vc[b, L0:L0 + a] - vr) <= _bf16_bound(vr, 2e-4)), b
        untouched = np.ones(cap, dtype=bool)
        untouched[L0:L0 + a] = False
        assert np.all(kc[b, untouched] == 3.0) and np.all(vc[b, untouched] == -3.0), b
    eng.close()


def test_greedy_decode_loop_equals_plain_decoding():
    w = S.WORKLOADS["tiny_fp32"]
    seed = S.WORKLOAD_SEEDS["tiny_fp32"]
    dev = "cuda"
    W = S.draft_weights(w, seed, device=dev)
    T = S.target_weights(w, seed, device=dev)
    tgt = GpuTinyTarget(w, W, T)
    prompt = S.random_ints(0, w.vocab, (32,), seed, "prefix_tokens").to(dev)
    L = prompt.numel()
    cap = L + ROUNDS * (w.depth + 1) + 8
    lim = dict(limits_for(w))
    lim["max_rows"] = max(lim["max_rows"], L)
    eng = R.Engine(dims_of(w), max_prefix=cap, device=dev, **lim)
    plan = R.plan_for(w.tree, w.top_k, w.depth, w.top_m)
    rd = R.Round(eng, plan, 1, cap, n_target_layers=2)
    w_c = eng.weights(W)

    # the prompt: target caches, first token, and the draft cache (a refresh over the prompt)
    f, logits, caches = tgt.prefill(prompt)
    gpu_logits = {L - 1: logits[-1].double().cpu().numpy()}      # position -> GPU target logits there
    for l, (k, v) in enumerate(caches):
        rd.tgt_k[l][0, :L] = k.to(torch.bfloat16)
        rd.tgt_v[l][0, :L] = v.to(torch.bfloat16)
    t_first = int(torch.argmax(logits[-1]))
    rd.t_next.fill_(t_first)
    rd.f_last.copy_(f[-1:])
    rd.pos0.fill_(L)
    rd.tgt_len.fill_(L)
    rd.temps.fill_(0.0)
    f_rows = torch.zeros(1, L, w.d, device=dev)
    f_rows[0, :L - 1] = f[:L - 1]
    tok_rows = torch.zeros(1, L + 1, dtype=torch.int32, device=dev)
    tok_rows[0, :L] = prompt.int()
    zero = torch.zeros(1, dtype=torch.int32, device=dev)
    _refresh_call(eng, w_c, 1, f_rows, tok_rows, torch.tensor([L - 1], dtype=torch.int32, device=dev), zero,
                  rd.draft_k, rd.draft_v, cap, zero.clone(), rd.draft_len)
    torch.cuda.synchronize()
    assert eng.status() == 0 and int(rd.draft_len) == L - 1

    Wd = DraftWeights({n: t.cpu() for n, t in W.items()}, w)
    tiny = TinyTarget(Wd, {"layers": [{n: t.cpu() for n, t in lw.items()} for lw in T["layers"]],
                           "g_final": T["g_final"].cpu()}, w)
    # draft cache of the prompt (positions 1 .. L-1 at rows 0 .. L-2) against the oracle
    kr, vr = draft_refresh_rows(Wd, w, f[:L - 1].cpu().double().numpy(), prompt[1:].cpu().numpy(), range(1, L))
    dk = rd.draft_k[0, :L - 1].cpu().double().numpy()
    assert np.all(np.abs(dk - kr) <= _bf16_bound(kr, 2e-4))

    seq = [int(t) for t in prompt.cpu()] + [t_first]
    accepted = []
    for r in range(ROUNDS):
        rd.set_sampling(seed, r)
        Ld, Lr = int(rd.draft_len), int(rd.pos0)
        rd.draft_and_tree(w_c)
        tgt.verify(eng, rd)
        rd.accept()
        rd.commit()
        rd.refresh(w_c)
        torch.cuda.synchronize()
        assert eng.status() == 0, r
        a = int(rd.accept_len)
        path = rd.path[0, :a + 1].tolist()
        toks = rd.tok_commit[0, :a + 2].tolist()
        assert toks[0] == seq[-1]                  # the root is the token committed last round
        for i, s_ in enumerate(path):
            gpu_logits[Lr + i] = rd.target_logits[0, s_].double().cpu().numpy()
        seq += toks[1:]
        accepted.append(a)
        # lengths advance by the committed path; the draft cache gained the
        # root's row (commit) and the accepted path's rows (refresh), equal to
        # the oracle's draft K/V of [true feature of p - 1 ; token at p]
        assert int(rd.prefix_len_out) == Lr + 1 + a and int(rd.draft_len_next) == Ld + 1 + a
        fc = rd.f_commit[0, :a + 1].double().cpu().numpy()
        f_prev = np.concatenate([rd.f_last.double().cpu().numpy(), fc[:a]])
        kr, _ = draft_refresh_rows(Wd, w, f_prev, toks[:a + 1], range(Lr, Lr + a + 1))
        got = rd.draft_k[0, Ld:Ld + a + 1].double().cpu().numpy()
        assert np.all(np.abs(got - kr) <= _bf16_bound(kr, 2e-4)), r
        rd.advance()
    # the committed tokens against the oracle target, position by position on
    # the GPU's own sequence, then against plain greedy decoding of the prompt
    _, lg, _ = tiny.prefill(seq)
    ties = []
    for j in range(L, len(seq)):
        z = lg[j - 1]
        top = int(np.argmax(z))
        if top != seq[j]:
            dz = np.max(np.abs(gpu_logits[j - 1] - z)) if (j - 1) in gpu_logits else 0.0
            gap = z[top] - z[seq[j]]
            assert gap <= 2 * dz + 1e-6, (j, top, seq[j], gap, dz)
            ties.append((j, gap))
    if not ties:
        assert seq[L:] == tiny.greedy_decode(seq[:L], len(seq) - L)
    print("accept lengths", accepted, "near-ties", ties, "generated", len(seq) - L)
    eng.close()
