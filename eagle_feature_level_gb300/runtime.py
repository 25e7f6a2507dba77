"""Round buffers and call sequencing over the C ABI.

PyTorch supplies device memory and the stream; every step runs in libeagle's
kernels through the binding.  A `Round` owns the caller-side buffers of one
draft-and-verify round for a fixed batch and shape, builds the ABI structs
once, and issues the calls in order: ROOT, then per draft layer
(FRONTIER, eagle_draft_step), FINAL, eagle_tree_verify_attn, eagle_accept,
eagle_commit.  Nothing here reads device data back.
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional

import numpy as np
import torch

from . import _binding as B


def _p(t: Optional[torch.Tensor]) -> int:
    return 0 if t is None else t.data_ptr()


def _u16(t: torch.Tensor) -> torch.Tensor:
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t


# Static tree layouts (rank paths below the root, listed by depth).  The pages
# give no layout, only "3 forwards -> 10-token tree" and "deeper and wider on
# likely branches"; these are this library's own.
STATIC_TEMPLATES = {
    "chain4": [(0,), (0, 0), (0, 0, 0), (0, 0, 0, 0)],
    "static8": [(0,), (1,), (2,), (0, 0), (0, 1), (1, 0), (0, 0, 0), (0, 0, 1)],
    "static26": [
        (0,), (1,), (2,), (3,),
        (0, 0), (0, 1), (0, 2), (0, 3), (1, 0), (1, 1), (2, 0), (3, 0),
        (0, 0, 0), (0, 0, 1), (0, 0, 2), (0, 1, 0), (0, 1, 1), (1, 0, 0), (2, 0, 0),
        (0, 0, 0, 0), (0, 0, 0, 1), (0, 0, 1, 0), (0, 1, 0, 0), (1, 0, 0, 0),
        (0, 0, 0, 0, 0), (0, 0, 0, 0, 1),
    ],
    # complete ternary tree, depths 1..4 (120 nodes, 40 of them expanded)
    "ternary4": [tuple(int(c) for c in np.base_repr(i, 3).zfill(n)) for n in range(1, 5) for i in range(3 ** n)],
}


def plan_for(tree: str, top_k: int = 0, depth: int = 0, top_m: int = 0) -> B.eagle_plan:
    """EAGLE-2 plan, or the static plan of a named template."""
    if tree == "eagle2":
        return B.eagle_plan_eagle2(top_k, depth, top_m)
    paths = STATIC_TEMPLATES[tree]
    index = {p: i for i, p in enumerate(paths)}
    parents = [index[p[:-1]] if len(p) > 1 else -1 for p in paths]
    ranks = [p[-1] for p in paths]
    return B.eagle_plan_static(parents, ranks)


class Engine:
    """A library context and its workspace on one device."""

    def __init__(self, dims: Dict[str, float], max_batch: int, max_rows: int, max_expanded: int,
                 max_children: int, max_tree: int, max_prefix: int, device="cuda"):
        self.device = torch.device(device)
        self.dims_c = B.eagle_dims(int(dims["d"]), int(dims["n_q_heads"]), int(dims["n_kv_heads"]),
                                   int(dims["head_dim"]), int(dims["d_ff"]), int(dims["vocab"]),
                                   float(dims.get("rms_eps", 1e-5)), float(dims.get("rope_theta", 10000.0)))
        self.limits_c = B.eagle_limits(max_batch, max_rows, max_expanded, max_children, max_tree, max_prefix)
        self.ctx, ws_bytes = B.eagle_create(self.dims_c, self.limits_c)
        self.ws = torch.empty(ws_bytes, dtype=torch.uint8, device=self.device)
        assert self.ws.data_ptr() % 256 == 0
        self.dims = dict(dims)
        B.eagle_workspace_init(self.ctx, self.ws.data_ptr(), self.stream())

    def stream(self) -> int:
        return torch.cuda.current_stream(self.device).cuda_stream

    def status(self) -> int:
        return B.eagle_read_device_status(self.ctx, self.ws.data_ptr(), self.stream())

    def close(self):
        if self.ctx:
            B.eagle_destroy(self.ctx)
            self.ctx = None

    def weights(self, W: Dict[str, torch.Tensor]) -> B.eagle_draft_weights:
        """The ABI struct of the draft weights W.  The struct holds raw device
        pointers, so it keeps a reference to W: the tensors live as long as
        the struct does."""
        ld = lambda t: t.shape[1]
        w_c = B.eagle_draft_weights(
            _p(W["w_fc"]), ld(W["w_fc"]), _p(W["b_fc"]), _p(W["g1"]), _p(W["wq"]), ld(W["wq"]), _p(W["wk"]),
            ld(W["wk"]), _p(W["wv"]), ld(W["wv"]), _p(W["wo"]), ld(W["wo"]), _p(W["g2"]), _p(W["w_gate"]),
            ld(W["w_gate"]), _p(W["w_up"]), ld(W["w_up"]), _p(W["w_down"]), ld(W["w_down"]), _p(W["embed"]),
            ld(W["embed"]), _p(W["w_lm"]), ld(W["w_lm"]))
        w_c.tensors = dict(W)
        return w_c


def mask_words(n: int) -> int:
    """64-bit words per slot of an ancestor mask over n slots (EAGLE_MASK_WORDS)."""
    return (n + 63) // 64


def _packed(specs, device):
    """One zeroed device allocation holding several tensors at 256-byte
    aligned offsets: a host buffer of the same layout moves all of them in
    one copy.  specs: [(shape, dtype)]; returns (flat uint8 tensor, views)."""
    offs, total = [], 0
    for shape, dtype in specs:
        n = math.prod(shape) * torch.empty((), dtype=dtype).element_size()
        offs.append((total, n))
        total += (n + 255) // 256 * 256
    flat = torch.zeros(max(total, 256), dtype=torch.uint8, device=device)
    views = [flat[o:o + n].view(dtype).view(shape) for (o, n), (shape, dtype) in zip(offs, specs)]
    return flat, views


class Round:
    """Caller-side buffers and ABI structs of one round (batch B, plan fixed)."""

    def __init__(self, eng: Engine, plan: B.eagle_plan, batch: int, kv_cap: int, n_target_layers: int = 1):
        self.eng, self.plan, self.B = eng, plan, batch
        d, V = eng.dims["d"], eng.dims["vocab"]
        Hq, Hkv, dh = eng.dims["n_q_heads"], eng.dims["n_kv_heads"], eng.dims["head_dim"]
        E, K, S = eng.limits_c.max_expanded, eng.limits_c.max_children, eng.limits_c.max_tree
        self.E, self.K, self.S = E, K, S
        self.kv_cap = kv_cap
        self.path_cap = plan.depth + 1
        dev = eng.device
        i32 = dict(dtype=torch.int32, device=dev)
        f32 = dict(dtype=torch.float32, device=dev)
        bf = dict(dtype=torch.bfloat16, device=dev)
        z = torch.zeros
        # What a round takes from the host (request state, the target's
        # verification-layer inputs and outputs) and gives back (acceptance
        # and commit results) sits in one allocation each way: `io_in` and
        # `io_out`, one copy per direction and round.
        self.io_in, (self.t_next, self.f_last, self.pos0, self.temps, self.target_logits, self.f_true,
                     self.tree_q, tree_k0, tree_v0) = _packed(
            [((batch,), torch.int32), ((batch, d), torch.float32), ((batch,), torch.int32),
             ((batch,), torch.float32), ((batch, S, V), torch.float32), ((batch, S, d), torch.float32),
             ((batch, S, Hq, dh), torch.bfloat16), ((batch, S, Hkv, dh), torch.bfloat16),
             ((batch, S, Hkv, dh), torch.bfloat16)], dev)
        self.io_out, (self.accept_len, self.path, self.final_token, self.tok_commit, self.f_last_out,
                      self.prefix_len_out) = _packed(
            [((batch,), torch.int32), ((batch, self.path_cap), torch.int32), ((batch,), torch.int32),
             ((batch, self.path_cap + 1), torch.int32), ((batch, d), torch.float32), ((batch,), torch.int32)],
            dev)
        self.draft_k = z(batch, kv_cap, Hkv, dh, **bf)
        self.draft_v = z(batch, kv_cap, Hkv, dh, **bf)
        self.draft_len = z(batch, **i32)
        # pool, children, draft outputs
        self.p_token = z(batch, E, **i32)
        self.p_parent = z(batch, E, **i32)
        self.p_rank = z(batch, E, **i32)
        self.p_depth = z(batch, E, **i32)
        self.p_value = z(batch, E, dtype=torch.float64, device=dev)
        self.p_anc = z(batch, E, mask_words(E), dtype=torch.int64, device=dev)
        self.p_child_exp = z(batch, E, K, **i32)
        self.c_token = z(batch, E, K, **i32)
        self.c_prob = z(batch, E, K, **f32)
        self.f_hat = z(batch, E, d, **f32)
        self.logits = z(batch, E, V, **f32)
        self.probs = z(batch, E, V, **f32)
        self.dk_tree = z(batch, E, Hkv, dh, **f32)
        self.dv_tree = z(batch, E, Hkv, dh, **f32)
        # tree
        self.t_token = z(batch, S, **i32)
        self.t_parent = z(batch, S, **i32)
        self.t_depth = z(batch, S, **i32)
        self.t_pos = z(batch, S, **i32)
        self.t_exp = z(batch, S, **i32)
        self.t_anc = z(batch, S, mask_words(S), dtype=torch.int64, device=dev)
        self.t_child_slot = z(batch, E, K, **i32)
        self.t_size = z(batch, **i32)
        # verification layer(s) and the target's outputs
        self.n_layers = n_target_layers
        self.tree_k = [tree_k0] + [z(batch, S, Hkv, dh, **bf) for _ in range(n_target_layers - 1)]
        self.tree_v = [tree_v0] + [z(batch, S, Hkv, dh, **bf) for _ in range(n_target_layers - 1)]
        self.tgt_k = [z(batch, kv_cap, Hkv, dh, **bf) for _ in range(n_target_layers)]
        self.tgt_v = [z(batch, kv_cap, Hkv, dh, **bf) for _ in range(n_target_layers)]
        self.tgt_len = z(batch, **i32)
        self.attn_out = z(batch, S, Hq, dh, **f32)
        self.target_probs = z(batch, S, V, **f32)
        self.target_argmax = z(batch, S, **i32)
        # accept + commit outputs
        self.last_slot = z(batch, **i32)
        self.f_commit = z(batch, self.path_cap, d, **f32)
        self.t_next_out = z(batch, **i32)
        self.draft_len_out = z(batch, **i32)
        self.draft_len_next = z(batch, **i32)    # after the draft-cache refresh
        self.seed, self.round_id = 0, 0
        self._structs()

    def _structs(self):
        self.req_c = B.eagle_requests(_p(self.t_next), _p(self.f_last), _p(self.pos0))
        self.draft_kv_c = B.eagle_kv(_p(self.draft_k), _p(self.draft_v), self.kv_cap, _p(self.draft_len))
        self.pool_c = B.eagle_pool(_p(self.p_token), _p(self.p_parent), _p(self.p_rank), _p(self.p_depth),
                                   _p(self.p_value), _p(self.p_anc), _p(self.p_child_exp))
        self.children_c = B.eagle_children(_p(self.c_token), _p(self.c_prob))
        self.out_c = B.eagle_draft_out(_p(self.f_hat), _p(self.logits), _p(self.probs), _p(self.dk_tree),
                                       _p(self.dv_tree))
        self.tree_c = B.eagle_tree(_p(self.t_token), _p(self.t_parent), _p(self.t_depth), _p(self.t_pos),
                                   _p(self.t_exp), _p(self.t_anc), _p(self.t_child_slot), _p(self.t_size),
                                   self.S)
        self.prefix_c = B.eagle_kv(_p(self.tgt_k[0]), _p(self.tgt_v[0]), self.kv_cap, _p(self.tgt_len))
        self.acc_c = B.eagle_accept_out(_p(self.accept_len), _p(self.path), _p(self.final_token),
                                        _p(self.last_slot), self.path_cap)
        self.commit_c = B.eagle_commit_out(_p(self.f_commit), _p(self.tok_commit), _p(self.f_last_out),
                                           _p(self.t_next_out), _p(self.prefix_len_out), _p(self.draft_len_out))
        self.sampling_c = B.eagle_sampling(_p(self.temps), self.seed, self.round_id)

    def set_sampling(self, seed: int, round_id: int):
        self.seed, self.round_id = int(seed) & 0xFFFFFFFF, int(round_id) & 0xFFFFFFFF
        self.sampling_c = B.eagle_sampling(_p(self.temps), self.seed, self.round_id)

    # ---- the calls ------------------------------------------------------------
    def draft_and_tree(self, w_c: B.eagle_draft_weights):
        e, st, ws = self.eng, self.eng.stream(), self.eng.ws.data_ptr()
        B.eagle_tree_expand_rerank(e.ctx, self.plan, B.PHASE_ROOT, 0, self.B, self.req_c, None, self.pool_c,
                                   None, ws, st)
        for layer in range(self.plan.n_layers):
            if layer >= 1:
                B.eagle_tree_expand_rerank(e.ctx, self.plan, B.PHASE_FRONTIER, layer, self.B, self.req_c,
                                           self.children_c, self.pool_c, None, ws, st)
            B.eagle_draft_step(e.ctx, self.plan, layer, self.B, w_c, self.req_c, self.draft_kv_c, self.pool_c,
                               self.out_c, self.children_c, self.sampling_c, ws, st)
        B.eagle_tree_expand_rerank(e.ctx, self.plan, B.PHASE_FINAL, 0, self.B, self.req_c, self.children_c,
                                   self.pool_c, self.tree_c, ws, st)

    def verify(self):
        e = self.eng
        scale = 1.0 / math.sqrt(e.dims["head_dim"])
        B.eagle_tree_verify_attn(e.ctx, self.B, _p(self.tree_q), _p(self.tree_k[0]), _p(self.tree_v[0]),
                                 self.prefix_c, self.tree_c, scale, _p(self.attn_out), e.ws.data_ptr(),
                                 e.stream())

    def accept(self):
        e = self.eng
        B.eagle_accept(e.ctx, self.plan, self.B, self.tree_c, self.children_c, _p(self.target_logits),
                       _p(self.probs), self.sampling_c, _p(self.target_probs), _p(self.target_argmax), self.acc_c,
                       e.ws.data_ptr(), e.stream())

    def commit(self):
        e = self.eng
        B.eagle_commit(e.ctx, self.B, self.acc_c, self.tree_c, _p(self.f_true),
                       [_p(t) for t in self.tree_k], [_p(t) for t in self.tree_v],
                       [_p(t) for t in self.tgt_k], [_p(t) for t in self.tgt_v], self.kv_cap, _p(self.tgt_len),
                       self.out_c, self.draft_kv_c, self.commit_c, e.ws.data_ptr(), e.stream())

    def refresh(self, w_c: B.eagle_draft_weights):
        """Append the draft layer's K/V of the accepted path (from the
        committed true features) after the root row commit appended:
        draft_len_next = draft_len_out + accept_len."""
        e = self.eng
        kv = B.eagle_kv(_p(self.draft_k), _p(self.draft_v), self.kv_cap, _p(self.draft_len_out))
        B.eagle_draft_refresh(e.ctx, self.B, w_c, self.acc_c, self.commit_c, _p(self.pos0), kv,
                              _p(self.draft_len_next), e.ws.data_ptr(), e.stream())

    def advance(self):
        """Make the committed state the next round's input by exchanging
        buffers (nothing is copied): t_next <- final token, f_last <- the
        last accepted slot's true feature, root position and target cache
        length <- the new prefix length, draft cache length <- the length
        after the refresh."""
        self.t_next, self.t_next_out = self.t_next_out, self.t_next
        self.f_last, self.f_last_out = self.f_last_out, self.f_last
        self.pos0, self.prefix_len_out = self.prefix_len_out, self.pos0
        self.tgt_len = self.pos0                 # both equal the prefix length
        self.draft_len, self.draft_len_next = self.draft_len_next, self.draft_len
        self._structs()

    def set_plan(self, plan: B.eagle_plan):
        """Switch to another tree budget whose shapes fit this round's buffers
        (depth, retained nodes, expanded slots, children per node)."""
        if (plan.depth + 1 > self.path_cap or plan.top_m + 1 > self.S or plan.n_expanded > self.E
                or plan.top_k > self.K):
            raise ValueError("plan does not fit the round's buffers")
        self.plan = plan

    def capture_segments(self, w_c: B.eagle_draft_weights, refresh: bool = False):
        """The round as two CUDA graphs around the target model: (draft,
        tree, verification attention) and (acceptance, commit[, refresh]).
        A server replays the first, runs its target over the tree, then the
        second.  Run the round eagerly once first."""
        pre, post = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(pre):
            self.draft_and_tree(w_c)
            self.verify()
        with torch.cuda.graph(post):
            self.accept()
            self.commit()
            if refresh:
                self.refresh(w_c)
        return pre, post

    def capture(self, w_c: B.eagle_draft_weights) -> "torch.cuda.CUDAGraph":
        """Capture one whole round (target logits already in place) as a CUDA
        graph; replaying it re-issues the same kernels with no host work.
        Run the round eagerly once before the first capture."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.run(w_c)
        return g

    def run(self, w_c: B.eagle_draft_weights, target_fn=None):
        """One whole round.  `target_fn(round)` stands in for the target model
        between drafting and acceptance (fills target_logits)."""
        self.draft_and_tree(w_c)
        self.verify()
        if target_fn is not None:
            target_fn(self)
        self.accept()
        self.commit()
