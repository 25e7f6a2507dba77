"""Exact integer sampling and the greedy child order (oracle side).

The pages require draws from the draft distribution q (Page A §4.1 and §6.1:
t ~ q = LM_Head(f)), an accept test r <= min(1, p/q) with a resample from
norm(max(0, p - q)) on rejection (Page A §6.2; Page B "随机采样验证";
Page C "为什么普通草稿模型不够理想"), and for greedy decoding the target
argmax (Page B "Greedy 验证").  They fix no arithmetic for these steps; our
specification makes every sampling decision exact integer arithmetic so
that two independent implementations that see the same fp32 probabilities
make the same decision:

  * a probability vector pi becomes weights W[v] = floor(pi_v * 2^40)
    (a power-of-two scale, exact for any float input);
  * one draw with a uniform u32: t = (u32 * S) >> 32 with S = sum(W); the
    draw is the smallest v whose inclusive prefix sum exceeds t;
  * k draws without replacement: each draw zeroes the drawn weight and
    draws again from what remains (the sequential definition);
  * greedy children: the k largest logits, ties to the lower token id.
"""
from __future__ import annotations

import numpy as np

QBITS = 40
MAX_VOCAB = 1 << 15          # keeps S < 2^55 and every accept-test product < 2^128


def quantize(probs) -> np.ndarray:
    """W[v] = floor(pi_v * 2^40) as int64 (exact: pi in [0, 1])."""
    p = np.asarray(probs, dtype=np.float64)
    assert p.ndim == 1 and p.size <= MAX_VOCAB
    assert np.all(p >= 0.0) and np.all(p <= 1.0)
    return np.floor(p * float(1 << QBITS)).astype(np.int64)


def draw_one(weights, u32: int) -> int:
    """Inverse-CDF draw on integer weights; -1 if the weights are all zero."""
    w = np.asarray(weights, dtype=np.int64)
    total = int(w.sum())
    if total == 0:
        return -1
    t = (int(u32) * total) >> 32
    cum = np.cumsum(w)
    return int(np.searchsorted(cum, t, side="right"))


def draws_without_replacement(weights, u32s) -> list:
    """Draw len(u32s) distinct indices; stops early (fills -1) when mass runs out."""
    w = np.array(weights, dtype=np.int64)
    out = []
    for u in u32s:
        v = draw_one(w, u)
        out.append(v)
        if v < 0:
            continue
        w[v] = 0
    return out


def greedy_top_k(z, k: int) -> list:
    """Indices of the k largest entries, ordered by (value desc, index asc)."""
    z = np.asarray(z, dtype=np.float64)
    order = np.lexsort((np.arange(z.size), -z))
    return [int(v) for v in order[:k]]


def argmax_low_id(z) -> int:
    z = np.asarray(z, dtype=np.float64)
    return int(np.flatnonzero(z == z.max())[0])
