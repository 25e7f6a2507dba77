"""Paged (block-table) target KV on the GPU.

[C] "工程落地时真正要看什么": the authoritative KV of accepted tokens lives in
blocks that the serving system's cache manager allocates (PagedAttention-style
block tables); [B] "KV Cache 必须按事务提交": the commit may land through
block-table remapping as long as the logical state equals that of a target
which generated only the accepted prefix and the correction token.

A paged cache is a pool of blocks plus a per-request table; paging changes
addresses, not arithmetic.  So the verification attention over a paged
prefix must equal the same call over the contiguous cache bit for bit (both
at the same capacity, hence the same prefix split), and the oracle's tree
attention on the logical prefix within the feature bound; the paged commit
must leave, read back through the table, exactly the contiguous commit's
cache.  Pool blocks that no table entry maps hold NaN, so that a stray read
or write shows.  A commit whose rows would land in an unallocated block is
refused for that request (EAGLE_ERR_CAPACITY, nothing of it written); an
unallocated block inside a prefix is reported (EAGLE_ERR_INVALID_ARG)."""
import math

import numpy as np
import pytest
import torch

import eagle_synth as S
from eagle_feature_level_gb300 import _binding as B
from eagle_feature_level_gb300 import runtime as R
from eagle_feature_level_gb300.runtime import _p
from eagle_feature_level_gb300.workload import dims_of, limits_for, load_round, standin
from oracle.verify import tree_attention
from tests.gpu_harness import feature_tol, mask_ints

pytestmark = pytest.mark.gpu

W = S.variant("13b_x8_eagle2", name="paged_small", d=128, n_q_heads=4, n_kv_heads=2, head_dim=64, d_ff=344,
              vocab=1000, batch=4, prefix_range=(50, 400), weight_std=0.05)
# the commit cases run greedy: paging is independent of how tokens are drawn
W_GREEDY = S.variant("13b_x8_eagle2", name="paged_small_greedy", d=128, n_q_heads=4, n_kv_heads=2, head_dim=64,
                     d_ff=344, vocab=1000, batch=4, prefix_range=(50, 400), weight_std=0.05, temps=(0.0,))
# head_dim 128 with 164 query rows per kv head: the tensor-memory kernel,
# whose whole prefix tiles come by TMA (per block when paged, from a block
# size of 8) and the rest by copies
W128 = S.variant("13b_x8_eagle2", name="paged_dh128", d=256, n_q_heads=8, n_kv_heads=2, head_dim=128, d_ff=512,
                 vocab=1000, batch=3, prefix_range=(50, 700), top_k=4, depth=4, top_m=40, weight_std=0.05)
INVALID_ARG, CAPACITY = 1, 4
BF16_NAN = 0x7FC0


def _round(seed, max_prefix=1024, n_target_layers=1, w=W):
    inp = S.round_inputs(w, seed, device="cuda")
    eng = R.Engine(dims_of(w), max_prefix=max_prefix, device="cuda", **limits_for(w))
    plan = R.plan_for(w.tree, w.top_k, w.depth, w.top_m)
    rd = R.Round(eng, plan, w.batch, inp["kv_cap"], n_target_layers=n_target_layers)
    load_round(rd, inp)
    wc = eng.weights(S.draft_weights(w, seed, device="cuda"))
    return eng, rd, wc, inp


def _widen(x, cap):
    """[B][c][Hkv][dh] -> [B][cap][Hkv][dh], the extra rows zero."""
    out = torch.zeros((x.shape[0], cap) + tuple(x.shape[2:]), dtype=x.dtype, device=x.device)
    out[:, :x.shape[1]] = x
    return out


def _paged(kc, vc, bs, seed, lens=None, spare=5):
    """Block pools and a table holding the contiguous caches kc, vc ([B][cap]).
    Blocks are placed in a seeded random order among `spare` extra blocks that
    stay NaN; with `lens`, blocks wholly past lens[b] + 8 rows are left
    unallocated (table -1), as a cache manager that allocates on demand would."""
    Bn, cap = kc.shape[:2]
    per = cap // bs
    n_blocks = Bn * per + spare
    g = torch.Generator().manual_seed(seed)
    perm = torch.randperm(n_blocks, generator=g)
    table = perm[:Bn * per].view(Bn, per).to(torch.int32)
    if lens is not None:
        for b in range(Bn):
            first_free = -(-(int(lens[b]) + 8) // bs)
            table[b, first_free:] = -1
    shape = (n_blocks, bs) + tuple(kc.shape[2:])
    kp = torch.full(shape, 0, dtype=torch.int16, device=kc.device)
    kp.fill_(BF16_NAN)
    kp = kp.view(torch.bfloat16)
    vp = kp.clone()
    for b in range(Bn):
        for j in range(per):
            blk = int(table[b, j])
            if blk >= 0:
                kp[blk] = kc[b, j * bs:(j + 1) * bs]
                vp[blk] = vc[b, j * bs:(j + 1) * bs]
    return kp, vp, table.cuda(), n_blocks


def _gather(pool, table, bs, cap):
    """Pool read back through the table: [B][cap]; rows of unallocated blocks NaN."""
    Bn, per = table.shape
    out = torch.full((Bn, cap) + tuple(pool.shape[2:]), float("nan"), dtype=pool.dtype, device=pool.device)
    for b in range(Bn):
        for j in range(per):
            blk = int(table[b, j])
            if blk >= 0:
                out[b, j * bs:(j + 1) * bs] = pool[blk]
    return out


def _verify(eng, rd, prefix, w=W):
    out = torch.full_like(rd.attn_out, float("nan"))
    B.eagle_tree_verify_attn(eng.ctx, rd.B, _p(rd.tree_q), _p(rd.tree_k[0]), _p(rd.tree_v[0]), prefix, rd.tree_c,
                             1.0 / math.sqrt(w.head_dim), _p(out), eng.ws.data_ptr(), eng.stream())
    return out


@pytest.mark.parametrize("w", [W, W128], ids=["dh64", "dh128"])
@pytest.mark.parametrize("bs", [1, 16, 64, 256])
def test_paged_verify_equals_contiguous_and_oracle(bs, w):
    seed = 1201
    eng, rd, wc, inp = _round(seed, w=w)
    rd.draft_and_tree(wc)
    cap = -(-rd.kv_cap // bs) * bs
    kc, vc = _widen(rd.tgt_k[0], cap), _widen(rd.tgt_v[0], cap)
    want = _verify(eng, rd, B.eagle_kv(_p(kc), _p(vc), cap, _p(rd.tgt_len)), w)
    kp, vp, table, nb = _paged(kc, vc, bs, seed + bs, lens=rd.tgt_len.tolist())
    paging = B.eagle_paging(_p(table), bs, nb)
    got = _verify(eng, rd, B.eagle_kv(_p(kp), _p(vp), cap, _p(rd.tgt_len), paging), w)
    torch.cuda.synchronize()
    assert eng.status() == 0
    sizes = rd.t_size.tolist()
    for b in range(rd.B):
        n = sizes[b]
        assert torch.equal(got[b, :n], want[b, :n]), b
        assert torch.isnan(got[b, n:]).all()               # slots past the tree are not written
        L = int(rd.tgt_len[b])
        anc = mask_ints(rd.t_anc[b, :n])
        f = lambda t: t.double().cpu().numpy()
        ref = tree_attention(f(rd.tree_q[b, :n]), f(rd.tree_k[0][b, :n]), f(rd.tree_v[0][b, :n]),
                             f(rd.tgt_k[0][b, :L]), f(rd.tgt_v[0][b, :L]), anc, 1.0 / math.sqrt(w.head_dim))
        assert np.max(np.abs(f(got[b, :n]) - ref)) <= feature_tol(w), b
    eng.close()


def _commit(eng, rd, kcs, vcs, cap, paging=None):
    B.eagle_commit(eng.ctx, rd.B, rd.acc_c, rd.tree_c, _p(rd.f_true), [_p(t) for t in rd.tree_k],
                   [_p(t) for t in rd.tree_v], [_p(t) for t in kcs], [_p(t) for t in vcs], cap, _p(rd.tgt_len),
                   rd.out_c, rd.draft_kv_c, rd.commit_c, eng.ws.data_ptr(), eng.stream(), target_paging=paging)


def _accepted_round(seed, n_target_layers=2):
    eng, rd, wc, inp = _round(seed, n_target_layers=n_target_layers, w=W_GREEDY)
    for l in range(1, n_target_layers):             # distinct tree rows per target layer
        rd.tree_k[l].copy_(torch.randn_like(rd.tree_k[l], dtype=torch.float32).to(torch.bfloat16))
        rd.tree_v[l].copy_(torch.randn_like(rd.tree_v[l], dtype=torch.float32).to(torch.bfloat16))
        rd.tgt_k[l].copy_(rd.tgt_k[0])
        rd.tgt_v[l].copy_(rd.tgt_v[0])
    rd.draft_and_tree(wc)
    rd.verify()
    standin(inp)(rd)
    rd.accept()
    torch.cuda.synchronize()
    assert eng.status() == 0
    return eng, rd


def test_paged_commit_equals_contiguous():
    seed, bs = 1301, 16
    eng, rd = _accepted_round(seed)
    cap = -(-rd.kv_cap // bs) * bs
    kcs = [_widen(t, cap) for t in rd.tgt_k]
    vcs = [_widen(t, cap) for t in rd.tgt_v]
    kps, vps = [], []
    for k, v in zip(kcs, vcs):                      # the same seed: one table for every layer
        kp, vp, table, nb = _paged(k, v, bs, seed, lens=rd.tgt_len.tolist())
        kps.append(kp)
        vps.append(vp)
    paging = B.eagle_paging(_p(table), bs, nb)
    _commit(eng, rd, kcs, vcs, cap)
    torch.cuda.synchronize()
    assert eng.status() == 0
    len_c = rd.prefix_len_out.clone()
    _commit(eng, rd, kps, vps, cap, paging)
    torch.cuda.synchronize()
    assert eng.status() == 0
    assert torch.equal(rd.prefix_len_out, len_c)
    a = rd.accept_len.tolist()
    for l in range(len(kcs)):
        gk, gv = _gather(kps[l], table, bs, cap), _gather(vps[l], table, bs, cap)
        for b in range(rd.B):
            L = int(rd.tgt_len[b])
            n = L + 1 + a[b]
            assert torch.equal(gk[b, :n], kcs[l][b, :n]) and torch.equal(gv[b, :n], vcs[l][b, :n]), (l, b)
        # the spare blocks no table entry maps are untouched
        mapped = set(int(x) for x in table.flatten().tolist() if x >= 0)
        spare = [i for i in range(nb) if i not in mapped]
        assert torch.isnan(kps[l][spare].float()).all() and torch.isnan(vps[l][spare].float()).all()
    eng.close()


def test_paged_commit_refused_on_unallocated_block():
    seed, bs = 1401, 16
    eng, rd = _accepted_round(seed, n_target_layers=1)
    cap = -(-rd.kv_cap // bs) * bs
    kc, vc = _widen(rd.tgt_k[0], cap), _widen(rd.tgt_v[0], cap)
    kp, vp, table, nb = _paged(kc, vc, bs, seed, lens=rd.tgt_len.tolist())
    L0 = int(rd.tgt_len[0])
    table[0, L0 // bs] = -1                          # request 0: the root's row has no block
    kp0, vp0 = kp.clone(), vp.clone()
    _commit(eng, rd, [kc], [vc], cap)                # contiguous commit of every request
    torch.cuda.synchronize()
    assert eng.status() == 0
    want_len = rd.prefix_len_out.tolist()
    _commit(eng, rd, [kp], [vp], cap, B.eagle_paging(_p(table), bs, nb))
    torch.cuda.synchronize()
    assert eng.status() == CAPACITY
    assert int(rd.prefix_len_out[0]) == L0           # request 0 refused, length kept
    assert rd.prefix_len_out.tolist()[1:] == want_len[1:]
    mine = [int(x) for x in table[0].tolist() if x >= 0]
    assert torch.equal(kp[mine].view(torch.int16), kp0[mine].view(torch.int16))   # nothing of it written
    assert torch.equal(vp[mine].view(torch.int16), vp0[mine].view(torch.int16))
    gk = _gather(kp, table, bs, cap)
    a = rd.accept_len.tolist()
    for b in range(1, rd.B):
        n = int(rd.tgt_len[b]) + 1 + a[b]
        assert torch.equal(gk[b, :n], kc[b, :n]), b
    eng.close()


@pytest.mark.parametrize("w", [W, W128], ids=["dh64", "dh128"])
def test_unallocated_block_inside_prefix_is_reported(w):
    seed, bs = 1501, 16
    eng, rd, wc, inp = _round(seed, w=w)
    rd.draft_and_tree(wc)
    cap = -(-rd.kv_cap // bs) * bs
    kc, vc = _widen(rd.tgt_k[0], cap), _widen(rd.tgt_v[0], cap)
    kp, vp, table, nb = _paged(kc, vc, bs, seed, lens=rd.tgt_len.tolist())
    table[2, 1] = -1                                 # request 2: positions 16..31 lost
    got = _verify(eng, rd, B.eagle_kv(_p(kp), _p(vp), cap, _p(rd.tgt_len), B.eagle_paging(_p(table), bs, nb)), w)
    torch.cuda.synchronize()
    assert eng.status() == INVALID_ARG
    n = int(rd.t_size[2])
    assert torch.isfinite(got[2, :n]).all()           # read as zero rows, no stray access
    eng.close()


def test_paging_arguments_checked_before_launch():
    eng, rd, wc, inp = _round(1601)
    cap = rd.kv_cap
    before = B.eagle_launch_count(eng.ctx)
    table = torch.zeros(rd.B, 64, dtype=torch.int32, device="cuda")
    nondiv = 1
    while cap % nondiv == 0:
        nondiv *= 2
    bad = [B.eagle_paging(_p(table), 3, 10),          # not a power of two
           B.eagle_paging(_p(table), nondiv, 10),     # does not divide the capacity
           B.eagle_paging(_p(table), 1, 0)]          # no blocks
    for pg in bad:
        with pytest.raises(B.EagleError) as e:
            _verify(eng, rd, B.eagle_kv(_p(rd.tgt_k[0]), _p(rd.tgt_v[0]), cap, _p(rd.tgt_len), pg))
        assert e.value.code == INVALID_ARG
    # the draft cache is never paged
    dkv = B.eagle_kv(_p(rd.draft_k), _p(rd.draft_v), cap, _p(rd.draft_len), B.eagle_paging(_p(table), 1, 10))
    with pytest.raises(B.EagleError) as e:
        B.eagle_draft_step(eng.ctx, rd.plan, 0, rd.B, wc, rd.req_c, dkv, rd.pool_c, rd.out_c, rd.children_c,
                           rd.sampling_c, eng.ws.data_ptr(), eng.stream())
    assert e.value.code == INVALID_ARG
    assert B.eagle_launch_count(eng.ctx) == before
    eng.close()
