"""Seeded synthetic inputs for one EAGLE/EAGLE-2 draft-and-verify round.

This module holds workload shapes and random-number draws only: no step of
the method's arithmetic lives here.  Both the CUDA path and the CPU oracle
take their inputs from it, so they see identical bytes.

Distributions follow the workload descriptions:
  * draft weights, bias, token embedding and LM head ~ N(0, std) with
    std = 0.02 (7B/13B/70B shapes) or 1/sqrt(d) = 0.125 (tiny shape); the
    second argument of N(., .) is read as the standard deviation;
  * "LM-head logits are rescaled to unit std": the constant
    s = 1/(std*sqrt(d)) is folded into the LM head at generation time (fp32,
    then rounded to bf16), so logits of N(0,1) features have unit std;
  * RMSNorm gains (trained weights the workloads do not state) are drawn as
    1 + N(0, 0.1) so that a misplaced gain shows up in parity;
  * features f ~ N(0,1); prefix KV entries ~ N(0,1) (stored post-RoPE);
  * the synthetic target: logits of an expanded tree node are the draft
    logits of that node plus N(0, 0.5^2) noise; a retained node that was
    never expanded gets N(0,1) logits.  Both noise tensors come from here.
Every weight matrix is row-major [out, in] with a row pitch ``ld`` equal to
``in`` rounded up to a multiple of 8 elements (16 bytes); pad columns are 0.
"""
from __future__ import annotations

import dataclasses
import hashlib
from typing import Dict, List, Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    d: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    d_ff: int
    vocab: int
    batch: int
    prefix_len: Optional[int]          # fixed prefix length, or None for ragged
    prefix_range: Optional[tuple]      # (lo, hi) inclusive for ragged lengths
    tree: str                          # "eagle2" or a static template name
    temps: tuple                       # per-request temperature pattern (0 = greedy)
    top_k: int                         # children drawn per expanded node
    depth: int                         # tree depth (layers below the root)
    top_m: int                         # retained nodes (excl. root)
    weight_std: float
    rescale_lm: bool
    rms_eps: float = 1e-5
    rope_theta: float = 10000.0

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    def temps_for_batch(self) -> List[float]:
        return [float(self.temps[b % len(self.temps)]) for b in range(self.batch)]


# The five workloads.  Static templates (rank paths) live in the oracle and
# the library; their node counts are fixed by name: chain4 -> 4, static8 -> 8,
# static26 -> 26.
WORKLOADS: Dict[str, Workload] = {
    "tiny_fp32": Workload("tiny_fp32", d=64, n_q_heads=4, n_kv_heads=4, head_dim=16,
                          d_ff=172, vocab=512, batch=1, prefix_len=32, prefix_range=None,
                          tree="static8", temps=(0.0,), top_k=3, depth=3, top_m=8,
                          weight_std=0.125, rescale_lm=False),
    "7b_static26": Workload("7b_static26", d=4096, n_q_heads=32, n_kv_heads=32, head_dim=128,
                            d_ff=11008, vocab=32000, batch=1, prefix_len=1024, prefix_range=None,
                            tree="static26", temps=(0.0,), top_k=4, depth=5, top_m=26,
                            weight_std=0.02, rescale_lm=True),
    "7b_eagle2": Workload("7b_eagle2", d=4096, n_q_heads=32, n_kv_heads=32, head_dim=128,
                          d_ff=11008, vocab=32000, batch=1, prefix_len=2048, prefix_range=None,
                          tree="eagle2", temps=(1.0,), top_k=10, depth=6, top_m=60,
                          weight_std=0.02, rescale_lm=True),
    "13b_x8_eagle2": Workload("13b_x8_eagle2", d=5120, n_q_heads=40, n_kv_heads=40, head_dim=128,
                              d_ff=13824, vocab=32000, batch=8, prefix_len=None,
                              prefix_range=(512, 4096), tree="eagle2", temps=(1.0,), top_k=10,
                              depth=6, top_m=60, weight_std=0.02, rescale_lm=True),
    "70b_x16_eagle2": Workload("70b_x16_eagle2", d=8192, n_q_heads=64, n_kv_heads=8, head_dim=128,
                               d_ff=28672, vocab=32000, batch=16, prefix_len=8192, prefix_range=None,
                               tree="eagle2", temps=(0.0, 0.7), top_k=10, depth=6, top_m=60,
                               weight_std=0.02, rescale_lm=True),
}

# Seeds: 1000 + position of the workload in the list above.
WORKLOAD_SEEDS = {name: 1000 + i for i, name in enumerate(WORKLOADS)}


def variant(base: str, **changes) -> Workload:
    """A workload with some fields replaced (small parity cases, tiny chains)."""
    w = WORKLOADS[base]
    fields = dataclasses.asdict(w)
    fields.update(changes)
    return Workload(**fields)


def ld_of(n: int) -> int:
    return (n + 7) // 8 * 8


def _sub_seed(seed: int, name: str) -> int:
    h = hashlib.sha256(f"{seed}:{name}".encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _randn(shape, seed: int, name: str, device) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(_sub_seed(seed, name))
    return torch.randn(*shape, generator=g, device=device, dtype=torch.float32)


def _randint(lo: int, hi: int, shape, seed: int, name: str, device) -> torch.Tensor:
    g = torch.Generator(device=device)
    g.manual_seed(_sub_seed(seed, name))
    return torch.randint(lo, hi, shape, generator=g, device=device, dtype=torch.int64)


def _bf16_matrix(out_f: int, in_f: int, std: float, seed: int, name: str, device,
                 scale: float = 1.0) -> torch.Tensor:
    """[out, ld(in)] bf16 with zero pad columns; values N(0, std) * scale."""
    w = _randn((out_f, in_f), seed, name, device) * std
    if scale != 1.0:
        w = w * scale
    ld = ld_of(in_f)
    if ld != in_f:
        w = torch.nn.functional.pad(w, (0, ld - in_f))
    return w.to(torch.bfloat16).contiguous()


def draft_weights(w: Workload, seed: int, device="cpu") -> Dict[str, torch.Tensor]:
    d, F, V = w.d, w.d_ff, w.vocab
    qd, kvd = w.n_q_heads * w.head_dim, w.n_kv_heads * w.head_dim
    std = w.weight_std
    lm_scale = 1.0 / (std * d ** 0.5) if w.rescale_lm else 1.0
    W = {
        "w_fc": _bf16_matrix(d, 2 * d, std, seed, "w_fc", device),
        "b_fc": (_randn((d,), seed, "b_fc", device) * std).contiguous(),
        "g1": (1.0 + 0.1 * _randn((d,), seed, "g1", device)).contiguous(),
        "wq": _bf16_matrix(qd, d, std, seed, "wq", device),
        "wk": _bf16_matrix(kvd, d, std, seed, "wk", device),
        "wv": _bf16_matrix(kvd, d, std, seed, "wv", device),
        "wo": _bf16_matrix(d, qd, std, seed, "wo", device),
        "g2": (1.0 + 0.1 * _randn((d,), seed, "g2", device)).contiguous(),
        "w_gate": _bf16_matrix(F, d, std, seed, "w_gate", device),
        "w_up": _bf16_matrix(F, d, std, seed, "w_up", device),
        "w_down": _bf16_matrix(d, F, std, seed, "w_down", device),
        "embed": _bf16_matrix(V, d, std, seed, "embed", device),
        "w_lm": _bf16_matrix(V, d, std, seed, "w_lm", device, scale=lm_scale),
    }
    return W


def prefix_lengths(w: Workload, seed: int) -> List[int]:
    if w.prefix_len is not None:
        return [w.prefix_len] * w.batch
    lo, hi = w.prefix_range
    t = _randint(lo, hi + 1, (w.batch,), seed, "prefix_len", "cpu")
    return [int(x) for x in t]


def max_tree_slots(w: Workload) -> int:
    return 1 + w.top_m


def max_expanded(w: Workload) -> int:
    """Expanded-node slots per request (root + every frontier row)."""
    if w.tree == "eagle2":
        return 1 + w.top_k * (w.depth - 1)
    # static templates: fixed by name
    return {"chain4": 4, "static8": 4, "static26": 14, "ternary4": 40}[w.tree]


def round_inputs(w: Workload, seed: int, device="cpu") -> Dict[str, object]:
    """Per-round request state and the synthetic target's tensors."""
    B, d, V = w.batch, w.d, w.vocab
    Hkv, Hq, dh = w.n_kv_heads, w.n_q_heads, w.head_dim
    L = prefix_lengths(w, seed)
    Lcap = max(L) + w.depth + 2
    S = max_tree_slots(w)
    out: Dict[str, object] = {
        "prefix_len": L,                      # root (t_next) sits at position L[b]
        "draft_len": list(L),                 # rows in the draft's own prefix KV
        "kv_cap": Lcap,
        "f_last": _randn((B, d), seed, "f_last", device),
        "t_next": _randint(0, V, (B,), seed, "t_next", device).to(torch.int32),
        "temps": w.temps_for_batch(),
        "philox_seed": int(_sub_seed(seed, "philox") & 0xFFFFFFFF),
        "round_id": 7,
        # draft layer's own prefix KV, [B][Lcap][Hkv][dh]
        "draft_k": _randn((B, Lcap, Hkv, dh), seed, "draft_k", device).to(torch.bfloat16),
        "draft_v": _randn((B, Lcap, Hkv, dh), seed, "draft_v", device).to(torch.bfloat16),
        # one target layer for verification: prefix KV and the tree's Q/K/V
        "tgt_k": _randn((B, Lcap, Hkv, dh), seed, "tgt_k", device).to(torch.bfloat16),
        "tgt_v": _randn((B, Lcap, Hkv, dh), seed, "tgt_v", device).to(torch.bfloat16),
        "tree_q": _randn((B, S, Hq, dh), seed, "tree_q", device).to(torch.bfloat16),
        "tree_k": _randn((B, S, Hkv, dh), seed, "tree_k", device).to(torch.bfloat16),
        "tree_v": _randn((B, S, Hkv, dh), seed, "tree_v", device).to(torch.bfloat16),
        # synthetic target: noise added to draft logits / logits of unexpanded nodes
        "tgt_noise": _randn((B, S, V), seed, "tgt_noise", device) * 0.5,
        "tgt_fresh": _randn((B, S, V), seed, "tgt_fresh", device),
        # true features of the tree nodes (the target forward's output)
        "f_true": _randn((B, S, d), seed, "f_true", device),
    }
    return out


def fuse_weights(w: Workload, seed: int, device="cpu") -> Dict[str, torch.Tensor]:
    """EAGLE-3 feature fusion FC (3d -> d): weights and bias N(0, std)."""
    return {"w_fuse": _bf16_matrix(w.d, 3 * w.d, w.weight_std, seed, "w_fuse", device),
            "b_fuse": (_randn((w.d,), seed, "b_fuse", device) * w.weight_std).contiguous()}


def random_probs(rows: int, V: int, seed: int, name: str, sigma: float = 1.0,
                 device="cpu") -> torch.Tensor:
    """fp32 random probability rows for stage tests: log-normal weights
    exp(sigma * N(0,1)) divided by their sum.  A random draw of a probability
    vector, handed verbatim to both sides; rows need not sum to exactly 1."""
    w = torch.exp(_randn((rows, V), seed, name, device) * sigma)
    return (w / w.sum(dim=-1, keepdim=True)).to(torch.float32).contiguous()


def random_logits(rows: int, V: int, seed: int, name: str, device="cpu") -> torch.Tensor:
    return _randn((rows, V), seed, name, device).contiguous()


def random_tensor(shape, seed: int, name: str, device="cpu", std: float = 1.0) -> torch.Tensor:
    return (_randn(tuple(shape), seed, name, device) * std).contiguous()


def random_ints(lo: int, hi: int, shape, seed: int, name: str, device="cpu") -> torch.Tensor:
    return _randint(lo, hi, tuple(shape), seed, name, device)


def target_weights(w: Workload, seed: int, n_layers: int = 2, device="cpu") -> Dict[str, object]:
    """Random-init target decoder layers (the tiny workload's 2-layer target).
    The embedding and LM head are the draft's shared ones (draft_weights)."""
    d, F = w.d, w.d_ff
    qd, kvd = w.n_q_heads * w.head_dim, w.n_kv_heads * w.head_dim
    std = w.weight_std
    layers = []
    for l in range(n_layers):
        p = f"tgt{l}_"
        layers.append({
            "g1": (1.0 + 0.1 * _randn((d,), seed, p + "g1", device)),
            "wq": _bf16_matrix(qd, d, std, seed, p + "wq", device),
            "wk": _bf16_matrix(kvd, d, std, seed, p + "wk", device),
            "wv": _bf16_matrix(kvd, d, std, seed, p + "wv", device),
            "wo": _bf16_matrix(d, qd, std, seed, p + "wo", device),
            "g2": (1.0 + 0.1 * _randn((d,), seed, p + "g2", device)),
            "w_gate": _bf16_matrix(F, d, std, seed, p + "w_gate", device),
            "w_up": _bf16_matrix(F, d, std, seed, p + "w_up", device),
            "w_down": _bf16_matrix(d, F, std, seed, p + "w_down", device),
        })
    return {"layers": layers, "g_final": 1.0 + 0.1 * _randn((d,), seed, "tgt_gf", device)}
