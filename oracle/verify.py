"""Tree-masked verification attention and acceptance (oracle side).

Attention (Page B "Tree Attention 如何一次验证多条路径"; Page A §6.2, §12 item 5):
the tree's nodes are flattened into one verification batch; node u attends
to the committed prefix and to tree node v iff v is an ancestor of u or v = u
(M_uv = 0, else -inf), at position id = prefix length + depth.

Greedy acceptance (Page B "Greedy 验证"): start at the root; take the target
argmax g at the current node; if a child of the node carries g, accept it and
continue there; otherwise commit g as the correction token and stop; at a
node with no children, g is the bonus token.  Ties: lowest token id.

Sampling acceptance (Page A §6.2, Page B "随机采样验证", Page C
"为什么普通草稿模型不够理想"; recursive multi-candidate verification after
SpecInfer, Page A §15 item 3): candidate x drawn from q is accepted with
probability min(1, p(x)/q(x)); on rejection the target distribution becomes
the residual norm(max(0, p - q)) and the next candidate is tried.  The
candidates of a node are its k drawn children, taken in draw order; since
they were drawn without replacement, candidate i was drawn from q with the
earlier candidates removed (Q_i), which is the proposal each test must use
(Page B "随机采样验证": construction and verification must match).  A
candidate that was drawn but pruned by the rerank is still tested; if it is
accepted it becomes the round's final token.  When every candidate is
rejected, or the node has no candidates, the final token is one draw from
the current residual.

Integer form of the test with weights P (target / residual) and Q_i:
    accept  iff  u32 * Q_i[x] * sum(P)  <  P[x] * sum(Q_i) * 2^32
i.e. r < p(x)/q(x) with r = u32 / 2^32 (strict, so p(x) = 0 never accepts).
Residual after rejecting x:  P <- max(0, P * sum(Q_i) - Q_i * sum(P)), then
shifted right by the smallest amount that brings max(P) below 2^40.
"""
from __future__ import annotations

import numpy as np

from . import philox
from .layer import attend
from .sampling import QBITS, argmax_low_id, draw_one, quantize


def tree_attention(q, k_tree, v_tree, k_prefix, v_prefix, anc, scale):
    """q [S, Hq, dh]; k/v_tree [S, Hkv, dh]; k/v_prefix [L, Hkv, dh]; anc [S]
    bitmasks over tree slots.  Returns O [S, Hq, dh]."""
    S = q.shape[0]
    out = np.empty_like(q)
    for i in range(S):
        vis = [j for j in range(S) if (anc[i] >> j) & 1]
        K = np.concatenate([k_prefix, k_tree[vis]], axis=0)
        V = np.concatenate([v_prefix, v_tree[vis]], axis=0)
        out[i] = attend(q[i], K, V, scale)
    return out


def accept_greedy(tree, target_logits):
    """Returns (accept_len, path slots incl. root, final token)."""
    u, path = 0, [0]
    while True:
        g = argmax_low_id(target_logits[u])
        nxt = [c for c in tree.children(u) if tree.token[c] == g]
        if nxt:
            u = nxt[0]
            path.append(u)
            continue
        return len(path) - 1, path, g


def _bitlen(x: int) -> int:
    return int(x).bit_length()


def accept_sampling(tree, p_rows, q_rows, child_tok, request, seed, round_id, margins=None):
    """Recursive multi-candidate rejection sampling on the flattened tree.

    p_rows[s]: target probabilities at tree slot s; q_rows[e]: draft
    probabilities of expanded node e; child_tok[e]: drawn children in draw
    order.  Returns (accept_len, path, final token).  If ``margins`` is a
    list, each decision appends how far it was from going the other way,
    relative: |r Q ΣP - P ΣQ 2^32| / (P ΣQ 2^32) for a test, and the distance
    of r from the nearest CDF boundary for the final draw."""
    u, path = 0, [0]
    while True:
        P = [int(w) for w in quantize(p_rows[u])]
        e = tree.exp[u]
        descended = False
        if e >= 0:
            Wq = [int(w) for w in quantize(q_rows[e])]
            sum_q = sum(Wq)
            taken = []
            for i, x in enumerate(child_tok[e]):
                if x < 0:
                    break
                sum_qi = sum_q - sum(Wq[t] for t in taken)
                sum_p = sum(P)
                r = philox.uniform_u32(seed, i, u, philox.PURPOSE_ACCEPT, request, round_id)
                if margins is not None:
                    rhs = P[x] * sum_qi * (1 << 32)
                    margins.append(abs(r * Wq[x] * sum_p - rhs) / rhs if rhs else float("inf"))
                if r * Wq[x] * sum_p < P[x] * sum_qi * (1 << 32):
                    slot = tree.child_slot.get((e, i), -1)
                    if slot < 0:
                        return len(path) - 1, path, int(x)
                    u = slot
                    path.append(u)
                    descended = True
                    break
                qi = [0 if v in taken else Wq[v] for v in range(len(Wq))]
                res = [max(0, P[v] * sum_qi - qi[v] * sum_p) for v in range(len(P))]
                shift = max(0, _bitlen(max(res)) - QBITS)
                P = [w >> shift for w in res]
                taken.append(int(x))
        if descended:
            continue
        r = philox.uniform_u32(seed, 0, u, philox.PURPOSE_FINAL, request, round_id)
        if margins is not None:
            total = sum(P)
            cum = np.cumsum(np.array(P, dtype=np.float64)) / max(total, 1)
            margins.append(float(np.min(np.abs(cum - r / 2.0 ** 32))) if total else float("inf"))
        return len(path) - 1, path, draw_one(np.array(P, dtype=np.int64), r)


def residual_exact(P, Q):
    """The unshifted residual of one rejection, as Python ints (for pins)."""
    P = [int(a) for a in P]
    Q = [int(b) for b in Q]
    sp, sq = sum(P), sum(Q)
    return [max(0, a * sq - b * sp) for a, b in zip(P, Q)]
