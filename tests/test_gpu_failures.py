"""Failure paths on the GPU, injected from the host (no GPU fault, trap or
hang is provoked): non-finite logits and zero-mass distributions set
EAGLE_ERR_NUMERIC in the device status word and the calls still return; a
misaligned pointer is refused with EAGLE_ERR_ALIGN before anything is
launched; a cache that cannot take the accepted path refuses the commit
(EAGLE_ERR_CAPACITY, nothing written for that request), and a prefix length
beyond its cache is read as the cache and reported; a barrier wait that
nothing ends gives up after the device limit with EAGLE_ERR_TIMEOUT."""
import math
import time

import numpy as np
import pytest
import torch

import eagle_synth as S
from eagle_feature_level_gb300 import _binding as B
from eagle_feature_level_gb300.runtime import _p
from eagle_feature_level_gb300.workload import make_round, standin

pytestmark = pytest.mark.gpu

W = S.variant("70b_x16_eagle2", name="failures_small", d=128, n_q_heads=4, n_kv_heads=2, head_dim=32, d_ff=256,
              vocab=700, batch=2, prefix_len=80, top_k=3, depth=3, top_m=6, weight_std=0.05, temps=(0.0, 1.0))
NUMERIC, ALIGN, CAPACITY = 6, 3, 4
TIMEOUT = 7


def _round(seed=31):
    Wt = S.draft_weights(W, seed, device="cuda")
    inp = S.round_inputs(W, seed, device="cuda")
    eng, rd = make_round(W, inp)
    return eng, rd, eng.weights(Wt), inp


@pytest.mark.parametrize("bad", [float("nan"), float("inf")])
def test_nonfinite_target_logits_set_numeric(bad):
    eng, rd, wc, inp = _round()
    rd.draft_and_tree(wc)
    rd.verify()
    standin(inp)(rd)
    rd.target_logits[1, 0, 17] = bad               # the sampling request's root row
    rd.accept()                                    # returns normally
    torch.cuda.synchronize()
    assert eng.status() == NUMERIC
    assert eng.status() == 0                        # reading clears the word
    eng.close()


def test_nonfinite_draft_input_sets_numeric_and_spares_the_other_request():
    eng, rd, wc, inp = _round()
    rd.f_last[0, 3] = float("nan")
    st, ws = eng.stream(), eng.ws.data_ptr()
    B.eagle_tree_expand_rerank(eng.ctx, rd.plan, B.PHASE_ROOT, 0, rd.B, rd.req_c, None, rd.pool_c, None, ws, st)
    B.eagle_draft_step(eng.ctx, rd.plan, 0, rd.B, wc, rd.req_c, rd.draft_kv_c, rd.pool_c, rd.out_c,
                       rd.children_c, rd.sampling_c, ws, st)
    torch.cuda.synchronize()
    assert eng.status() == NUMERIC
    k = rd.plan.top_k
    assert rd.c_token[0, 0, :k].tolist() == [-1] * k            # no mass left to draw from
    ok = rd.c_token[1, 0, :k].tolist()
    assert all(0 <= t < W.vocab for t in ok) and len(set(ok)) == k
    assert torch.isfinite(rd.logits[1, 0]).all()
    eng.close()


def test_zero_mass_target_row_sets_numeric():
    eng, rd, wc, inp = _round()
    rd.run(wc, target_fn=standin(inp))
    torch.cuda.synchronize()
    assert eng.status() == 0
    rd.target_probs[1].zero_()                      # sampling request: no target mass anywhere
    st, ws = eng.stream(), eng.ws.data_ptr()
    B.eagle_accept_from_probs(eng.ctx, rd.plan, rd.B, rd.tree_c, rd.children_c, _p(rd.target_probs),
                              _p(rd.target_argmax), _p(rd.probs), rd.sampling_c, rd.acc_c, ws, st)
    torch.cuda.synchronize()
    assert eng.status() == NUMERIC
    assert int(rd.accept_len[1]) == 0 and int(rd.final_token[1]) == -1   # every candidate rejected, no draw
    eng.close()


def test_misaligned_pointers_refused_before_launch():
    eng, rd, wc, inp = _round()
    before = B.eagle_launch_count(eng.ctx)
    scale = 1.0 / math.sqrt(W.head_dim)
    with pytest.raises(B.EagleError) as e:
        B.eagle_tree_verify_attn(eng.ctx, rd.B, rd.tree_q.data_ptr() + 2, rd.tree_k[0].data_ptr(),
                                 rd.tree_v[0].data_ptr(), rd.prefix_c, rd.tree_c, scale, rd.attn_out.data_ptr(),
                                 eng.ws.data_ptr(), eng.stream())
    assert e.value.code == ALIGN
    with pytest.raises(B.EagleError) as e:          # the workspace must be 256-byte aligned
        B.eagle_tree_verify_attn(eng.ctx, rd.B, rd.tree_q.data_ptr(), rd.tree_k[0].data_ptr(),
                                 rd.tree_v[0].data_ptr(), rd.prefix_c, rd.tree_c, scale, rd.attn_out.data_ptr(),
                                 eng.ws.data_ptr() + 16, eng.stream())
    assert e.value.code == ALIGN
    f_true = rd.f_true.data_ptr() + 4
    with pytest.raises(B.EagleError) as e:
        B.eagle_commit(eng.ctx, rd.B, rd.acc_c, rd.tree_c, f_true, [_p(t) for t in rd.tree_k],
                       [_p(t) for t in rd.tree_v], [_p(t) for t in rd.tgt_k], [_p(t) for t in rd.tgt_v],
                       rd.kv_cap, _p(rd.tgt_len), rd.out_c, rd.draft_kv_c, rd.commit_c, eng.ws.data_ptr(),
                       eng.stream())
    assert e.value.code == ALIGN
    assert B.eagle_launch_count(eng.ctx) == before
    eng.close()


def test_commit_refused_when_a_cache_is_full():
    eng, rd, wc, inp = _round()
    rd.draft_and_tree(wc)
    rd.verify()
    standin(inp)(rd)
    rd.accept()
    torch.cuda.synchronize()
    assert eng.status() == 0
    cap = rd.kv_cap
    rd.tgt_len[0] = cap                             # request 0: target cache full
    rd.draft_len[1] = cap                           # request 1: draft cache full
    k0, dk1 = rd.tgt_k[0].clone(), rd.draft_k.clone()
    rd.commit()
    torch.cuda.synchronize()
    assert eng.status() == CAPACITY
    assert int(rd.prefix_len_out[0]) == cap and int(rd.draft_len_out[1]) == cap
    assert torch.equal(rd.tgt_k[0], k0) and torch.equal(rd.draft_k, dk1)   # nothing written
    # with room again both commit, and the status stays clear
    L = inp["prefix_len"]
    rd.tgt_len.copy_(torch.tensor(L, dtype=torch.int32))
    rd.draft_len.copy_(torch.tensor(inp["draft_len"], dtype=torch.int32))
    rd.commit()
    torch.cuda.synchronize()
    assert eng.status() == 0
    a = rd.accept_len.tolist()
    assert rd.prefix_len_out.tolist() == [L[b] + 1 + a[b] for b in range(rd.B)]
    eng.close()


def test_prefix_longer_than_its_cache_is_read_as_the_cache():
    eng, rd, wc, inp = _round()
    rd.draft_and_tree(wc)
    cap = rd.kv_cap
    rd.tgt_len.fill_(cap)
    rd.verify()
    torch.cuda.synchronize()
    assert eng.status() == 0
    ref = rd.attn_out.clone()
    rd.tgt_len.fill_(cap + 1000)
    rd.attn_out.zero_()
    rd.verify()
    torch.cuda.synchronize()
    assert eng.status() == CAPACITY
    for b in range(rd.B):
        n = int(rd.t_size[b])
        assert torch.equal(rd.attn_out[b, :n], ref[b, :n])
    assert np.isfinite(rd.attn_out.cpu().numpy()).all()
    eng.close()


def test_bounded_wait_gives_up_with_timeout_and_the_context_stays_usable():
    """The kernels' barrier waits are bounded: the self-test's one CTA waits
    on a barrier nothing arrives at, gives up after the 2 s device limit and
    reports EAGLE_ERR_TIMEOUT; the same context then runs a whole round with
    a clean status."""
    eng, rd, wc, inp = _round(seed=71)
    st, ws = eng.stream(), eng.ws.data_ptr()
    torch.cuda.synchronize()
    t0 = time.monotonic()
    B.eagle_wait_selftest(eng.ctx, ws, st)
    torch.cuda.synchronize()
    waited = time.monotonic() - t0
    assert eng.status() == TIMEOUT
    assert 1.5 <= waited <= 30.0, waited
    rd.run(wc, target_fn=standin(inp))
    torch.cuda.synchronize()
    assert eng.status() == 0
    assert (rd.accept_len >= 0).all()
    eng.close()
