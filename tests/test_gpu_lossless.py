"""Invariant (d) on the GPU: the tokens the acceptance walk commits follow
the target distribution ([B] "随机采样验证" and "正确性与状态边界": verify
the output distribution on a small vocabulary; [A] §6.2).

About 10^6 seeded walks through eagle_accept_from_probs on a tiny vocabulary
(V = 6): each request's root has k = 3 children drawn from q_root without
replacement (PyTorch's sampler, independent of both the library and the
oracle), the first of them expanded with 3 children of its own drawn from
q2[x]; the target gives p_root at the root and p2[x] after token x.  The
first committed token must follow p_root -- the law the oracle's exact
rational enumeration of the multi-candidate rule yields -- and, after a
descent into a depth-1 node with token x, the next committed token must
follow p2[x].  With pruning, the last drawn child of each expanded node is
dropped from the tree (it is still tested, and becomes the final token when
accepted).  Checked by chi-square at p > 1e-3."""
import numpy as np
import pytest
import torch
from scipy.stats import chi2, chisquare

from eagle_feature_level_gb300 import _binding as B
from eagle_feature_level_gb300 import runtime as R
from eagle_feature_level_gb300.runtime import _p

pytestmark = pytest.mark.gpu

V, K, BATCH, CALLS = 6, 3, 32768, 32


def _tables():
    rng = np.random.default_rng(20261203)
    d = lambda *s: rng.dirichlet(np.ones(V), size=s).astype(np.float32)
    return d(1)[0], d(1)[0], d(V), d(V), d(1)[0]        # q_root, p_root, q2[x], p2[x], p3


@pytest.mark.parametrize("prune", [False, True], ids=["retained", "pruned"])
def test_committed_tokens_follow_the_target(prune):
    from tests.test_oracle_accept import _exact_multidraft_first_token
    q_root, p_root, q2, p2, p3 = _tables()
    dims = dict(d=64, n_q_heads=4, n_kv_heads=4, head_dim=16, d_ff=64, vocab=V)
    eng = R.Engine(dims, max_batch=BATCH, max_rows=1, max_expanded=2, max_children=K, max_tree=7, max_prefix=1)
    plan = B.eagle_plan_static([-1, -1, -1, 0, 0, 0], [0, 1, 2, 0, 1, 2])
    rd = R.Round(eng, plan, BATCH, kv_cap=1)
    rd.temps.fill_(1.0)
    keep = K - 1 if prune else K
    size = 1 + 2 * keep
    # fixed tree shape: slot 0 root, slots 1..keep its kept children (draw
    # order), slots keep+1 .. 2*keep the kept children of slot 1
    parent = [-1] + [0] * keep + [1] * keep
    rd.t_parent.fill_(-1)
    rd.t_parent[:, :size] = torch.tensor(parent, dtype=torch.int32)
    rd.t_exp.fill_(-1)
    rd.t_exp[:, 0], rd.t_exp[:, 1] = 0, 1
    rd.t_size.fill_(size)
    cs = torch.full((BATCH, rd.E, rd.K), -1, dtype=torch.int32)
    cs[:, 0, :keep] = torch.arange(1, 1 + keep, dtype=torch.int32)
    cs[:, 1, :keep] = torch.arange(1 + keep, 1 + 2 * keep, dtype=torch.int32)
    rd.t_child_slot.copy_(cs)
    g = torch.Generator().manual_seed(7 + prune)
    qr, q2t, p2t = torch.from_numpy(q_root), torch.from_numpy(q2), torch.from_numpy(p2)
    first = np.zeros(V)
    second = np.zeros((V, V))
    for call in range(CALLS):
        d0 = torch.multinomial(qr.expand(BATCH, V), K, replacement=False, generator=g)       # root's draws
        x = d0[:, 0]
        d1 = torch.multinomial(q2t[x], K, replacement=False, generator=g)                    # slot 1's draws
        tok = torch.zeros(BATCH, rd.S, dtype=torch.int32)
        tok[:, 1:1 + keep] = d0[:, :keep].int()
        tok[:, 1 + keep:size] = d1[:, :keep].int()
        rd.t_token.copy_(tok)
        rd.c_token.fill_(-1)
        rd.c_token[:, 0, :K] = d0.int().cuda()
        rd.c_token[:, 1, :K] = d1.int().cuda()
        qrows = torch.zeros(BATCH, rd.E, V)
        qrows[:, 0] = qr
        qrows[:, 1] = q2t[x]
        rd.probs.copy_(qrows)
        prows = torch.zeros(BATCH, rd.S, V)
        prows[:, 0] = torch.from_numpy(p_root)
        prows[:, 1:1 + keep] = p2t[d0[:, :keep]]
        prows[:, 1 + keep:size] = torch.from_numpy(p3)
        rd.target_probs.copy_(prows)
        rd.target_argmax.copy_(prows.argmax(-1).int())
        rd.set_sampling(0x5EED, 1000 + call)
        B.eagle_accept_from_probs(eng.ctx, plan, BATCH, rd.tree_c, rd.children_c, _p(rd.target_probs),
                                  _p(rd.target_argmax), _p(rd.probs), rd.sampling_c, rd.acc_c, eng.ws.data_ptr(),
                                  eng.stream())
        a = rd.accept_len.cpu().numpy()
        path = rd.path.cpu().numpy()
        fin = rd.final_token.cpu().numpy()
        tk = tok.numpy()
        rows = np.arange(BATCH)
        t1 = np.where(a >= 1, tk[rows, path[:, 1].clip(0)], fin)
        np.add.at(first, t1, 1)
        desc = a >= 1
        t2 = np.where(a >= 2, tk[rows, path[:, 2].clip(0)], fin)
        np.add.at(second, (t1[desc], t2[desc]), 1)
    assert eng.status() == 0
    eng.close()
    n = first.sum()
    assert n == BATCH * CALLS
    law = np.array([float(v) for v in _exact_multidraft_first_token([float(v) for v in p_root],
                                                                     [float(v) for v in q_root], K)])
    assert np.allclose(law, p_root / p_root.sum(), atol=1e-12)         # the oracle's enumeration = p_root
    assert chisquare(first, law * n).pvalue > 1e-3, (first / n, law)
    # after a descent into a depth-1 node with token x, the next token follows p2[x]
    stat, dof = 0.0, 0
    for xv in range(V):
        m = second[xv].sum()
        if m < 1000:
            continue
        want = p2[xv] / p2[xv].sum() * m
        stat += float(((second[xv] - want) ** 2 / want).sum())
        dof += V - 1
    assert dof >= 5 * (V - 1)
    assert chi2.sf(stat, dof) > 1e-3, (stat, dof)
