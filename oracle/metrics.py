"""Expected tokens per round from an acceptance profile (oracle side).

Page A §8 and exercise 2: with per-position acceptance rates alpha_1..alpha_K
of a chain draft, the expected number of tokens one verification yields is
    E[N] = 1 + sum_{i=1..K} prod_{j<=i} alpha_j
(the leading 1 is the token the target always contributes).
"""
from __future__ import annotations


def expected_tokens(alphas) -> float:
    total, run = 1.0, 1.0
    for a in alphas:
        run *= float(a)
        total += run
    return total
