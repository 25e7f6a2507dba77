"""eagle_tree_verify_attn_noalloc (verify attention with its scratch in the
library's fixed device array) against eagle_tree_verify_attn (scratch in the
caller's workspace) on the same round, two calls in a row.

Collected last (file name) so that it also runs after every other GPU test
in the same process; it sets up all of its own state, so it passes alone in
a fresh process too."""
import math

import pytest
import torch

import eagle_synth as S
from eagle_feature_level_gb300 import _binding as B
from eagle_feature_level_gb300.workload import make_round

pytestmark = pytest.mark.gpu

CASES = {
    # GQA (4 query heads per kv head), ragged tree sizes over 3 requests
    "small_eagle2_gqa": S.variant("70b_x16_eagle2", name="noalloc_small_eagle2_gqa", d=256, n_q_heads=8,
                                  n_kv_heads=2, head_dim=32, d_ff=688, vocab=1000, batch=3, prefix_len=100,
                                  top_k=4, depth=4, top_m=12, weight_std=0.05),
    # the bench's shape: 32 heads of 128, prefix 1024, static 26-node tree
    "7b_static26": S.WORKLOADS["7b_static26"],
    # head_dim 128 with 164 query rows per kv head (the tensor-memory kernel),
    # ragged prefixes over several splits
    "tc_gqa_dh128": S.variant("13b_x8_eagle2", name="noalloc_tc_gqa_dh128", d=256, n_q_heads=8, n_kv_heads=2,
                              head_dim=128, d_ff=512, vocab=1000, batch=3, prefix_range=(50, 700), top_k=4,
                              depth=4, top_m=40, weight_std=0.05),
}

# Same kernel, same split count, same merge order: the two entry points are
# expected to agree to the last bit; the bound leaves room only for that.
TOL = 1e-6


def _drafted_round(w, seed):
    W = S.draft_weights(w, seed, device="cuda")
    inp = S.round_inputs(w, seed, device="cuda")
    eng, rd = make_round(w, inp)
    rd.draft_and_tree(eng.weights(W))
    return eng, rd


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_matches_workspace_entry(name):
    w = CASES[name]
    seed = 4242
    eng, rd = _drafted_round(w, seed)
    rd.verify()                                   # workspace entry point -> rd.attn_out
    torch.cuda.synchronize()
    ref = rd.attn_out.clone()
    sizes = rd.t_size.cpu().tolist()
    scale = 1.0 / math.sqrt(w.head_dim)
    out = torch.empty_like(rd.attn_out)
    for call in range(2):
        out.fill_(float("nan"))
        B.eagle_tree_verify_attn_noalloc(eng.ctx, rd.B, rd.tree_q.data_ptr(), rd.tree_k[0].data_ptr(),
                                         rd.tree_v[0].data_ptr(), rd.prefix_c, rd.tree_c, scale, out.data_ptr(),
                                         eng.stream())
        torch.cuda.synchronize()
        assert B.eagle_read_device_status(eng.ctx, eng.ws.data_ptr(), eng.stream()) == 0
        for b, n in enumerate(sizes):
            assert 1 <= n <= out.shape[1]
            got, want = out[b, :n], ref[b, :n]
            assert torch.isfinite(got).all(), (name, call, b)
            err = (got - want).abs().max().item()
            assert err <= TOL, (name, call, b, err)
            # slots past the tree are not written
            assert torch.isnan(out[b, n:]).all(), (name, call, b)


def test_noalloc_rejects_oversize():
    """64 query heads of 128 over 16 requests with 61-slot trees need ~66 MB
    of partials, beyond the fixed 32 MiB array: EAGLE_ERR_CAPACITY and the
    output untouched (nothing launched)."""
    w = S.variant("70b_x16_eagle2", name="noalloc_oversize", d=256, d_ff=512, vocab=1000, prefix_len=256)
    seed = 4243
    inp = S.round_inputs(w, seed, device="cuda")
    eng, rd = make_round(w, inp)
    out = torch.full_like(rd.attn_out, float("nan"))
    with pytest.raises(B.EagleError) as ei:
        B.eagle_tree_verify_attn_noalloc(eng.ctx, rd.B, rd.tree_q.data_ptr(), rd.tree_k[0].data_ptr(),
                                         rd.tree_v[0].data_ptr(), rd.prefix_c, rd.tree_c, 1.0 / math.sqrt(128),
                                         out.data_ptr(), eng.stream())
    assert ei.value.code == 4                     # EAGLE_ERR_CAPACITY
    torch.cuda.synchronize()
    assert torch.isnan(out).all()


def test_first_call_refused_on_a_capturing_stream():
    """The first call in a CUDA context sets the array up (zeroing and a
    stream synchronisation, which a capture does not allow): on a capturing
    stream it returns EAGLE_ERR_INVALID_ARG without touching the stream, so
    the caller's capture stays valid.  Runs in a fresh process, where no call
    has set the array up yet."""
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    script = r"""
import math, sys, torch
sys.path.insert(0, %r)
import eagle_synth as S
from eagle_feature_level_gb300 import _binding as B
from eagle_feature_level_gb300.workload import make_round
w = S.variant("70b_x16_eagle2", name="noalloc_capture", d=256, n_q_heads=8, n_kv_heads=2, head_dim=32, d_ff=688,
              vocab=1000, batch=2, prefix_len=64, top_k=4, depth=3, top_m=8, weight_std=0.05)
inp = S.round_inputs(w, 4245, device="cuda")
eng, rd = make_round(w, inp)
torch.cuda.synchronize()
g = torch.cuda.CUDAGraph()
code = 0
with torch.cuda.graph(g):
    try:
        B.eagle_tree_verify_attn_noalloc(eng.ctx, rd.B, rd.tree_q.data_ptr(), rd.tree_k[0].data_ptr(),
                                         rd.tree_v[0].data_ptr(), rd.prefix_c, rd.tree_c, 1.0 / math.sqrt(32),
                                         rd.attn_out.data_ptr(), eng.stream())
    except B.EagleError as e:
        code = e.code
torch.cuda.synchronize()
print("CODE", code)
""" % root
    r = subprocess.run([sys.executable, "-c", script], capture_output=True, text=True, timeout=600)
    assert "CODE 1" in r.stdout, (r.stdout[-2000:], r.stderr[-2000:])
