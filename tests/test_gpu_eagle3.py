"""EAGLE-3 input on the GPU ([C] "EAGLE-3：放弃 feature prediction，改成多层特征融合
与 training-time test"): the target's low, middle and high features of each
position are fused, g = FC([l; m; h]), and g takes the place of the target
feature in the round (the root's f_last and the tree slots' true features).

eagle_fuse_features is compared with the oracle's fuse_rows on ragged row
counts; then a whole EAGLE-2 round driven by fused features (the root's and
every tree slot's) is compared element by element with the oracle, which is
given the same fused inputs."""
import numpy as np
import pytest
import torch

import eagle_synth as S
from eagle_feature_level_gb300 import _binding as B
from eagle_feature_level_gb300.runtime import _p
from eagle_feature_level_gb300.workload import make_round
from oracle.layer import fuse_rows
from tests.gpu_harness import compare_round, round_on, run_oracle_round

pytestmark = pytest.mark.gpu

W3 = S.variant("70b_x16_eagle2", name="eagle3_small", d=256, n_q_heads=8, n_kv_heads=2, head_dim=32, d_ff=688,
               vocab=1000, batch=3, prefix_len=100, top_k=4, depth=4, top_m=12, weight_std=0.05)


def _fuse(eng, F, lmh):
    n = lmh.shape[0]
    g = torch.full((n, lmh.shape[1] // 3), float("nan"), device="cuda")
    B.eagle_fuse_features(eng.ctx, _p(F["w_fuse"]), F["w_fuse"].shape[1], _p(F["b_fuse"]), n, _p(lmh), _p(g),
                          eng.ws.data_ptr(), eng.stream())
    return g


@pytest.mark.parametrize("bias", [True, False], ids=["bias", "no_bias"])
def test_fuse_matches_the_oracle(bias):
    w = W3
    seed = 808
    inp = S.round_inputs(w, seed, device="cuda")
    eng, rd = make_round(w, inp)
    F = S.fuse_weights(w, seed, device="cuda")
    if not bias:
        F = {"w_fuse": F["w_fuse"], "b_fuse": None}
    for n in (1, 7, eng.limits_c.max_rows):
        lmh = S.random_tensor((n, 3 * w.d), seed + n, "eagle3_lmh").cuda()
        g = _fuse(eng, F, lmh)
        torch.cuda.synchronize()
        assert eng.status() == 0
        x = lmh.double().cpu().numpy()
        d = w.d
        want = fuse_rows(F["w_fuse"].cpu(), None if F["b_fuse"] is None else F["b_fuse"].cpu(),
                         x[:, :d], x[:, d:2 * d], x[:, 2 * d:])
        err = np.max(np.abs(g.double().cpu().numpy() - want))
        assert err <= 1e-4 * max(1.0, np.abs(want).max()), (n, err)
    eng.close()


def test_round_driven_by_fused_features():
    w = W3
    seed = 809
    W = S.draft_weights(w, seed, device="cuda")
    inp = S.round_inputs(w, seed, device="cuda")
    F = S.fuse_weights(w, seed, device="cuda")
    eng, rd = make_round(w, inp)
    Bn, Sn, d = w.batch, rd.S, w.d
    # the target's three feature layers of the root's parent position and of every tree slot
    lmh_root = S.random_tensor((Bn, 3 * d), seed, "eagle3_root").cuda()
    lmh_slots = S.random_tensor((Bn * Sn, 3 * d), seed, "eagle3_slots").cuda()
    g_root = _fuse(eng, F, lmh_root)
    g_slots = torch.cat([_fuse(eng, F, lmh_slots[i:i + eng.limits_c.max_rows])
                         for i in range(0, Bn * Sn, eng.limits_c.max_rows)])
    torch.cuda.synchronize()
    rd.f_last.copy_(g_root)
    rd.f_true.copy_(g_slots.view(Bn, Sn, d))
    inp = dict(inp, f_last=rd.f_last, f_true=rd.f_true)
    inputs_cpu = {k: (v.detach().to("cpu") if torch.is_tensor(v) else v) for k, v in inp.items()}
    gpu = round_on(eng, rd, eng.weights(W), inp, inputs_cpu)
    ref = run_oracle_round(w, seed, inputs_cpu, {k: v.cpu() for k, v in W.items()}, gpu=gpu)
    rep = compare_round(w, gpu, ref)
    assert rep["ok"], rep["errors"]
    assert rep["reached"] == {b: "commit" for b in range(Bn)}
    # the next round starts from the fused feature of the last accepted slot
    for b in range(Bn):
        last = int(rd.last_slot[b])
        assert torch.equal(rd.f_last_out[b], rd.f_true[b, last])
    eng.close()
