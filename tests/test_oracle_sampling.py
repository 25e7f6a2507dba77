"""Pins for the oracle's random stream and integer sampling rules (CPU only)."""
from fractions import Fraction

import numpy as np
import pytest

from conftest import golden_lines
from oracle import philox
from oracle.sampling import (QBITS, argmax_low_id, draw_one, draws_without_replacement,
                             greedy_top_k, quantize)


def test_philox_known_answers():
    n = 0
    for line in golden_lines("philox_kat.txt"):
        vals = [int(x, 16) for x in line.split()]
        ctr, key, want = vals[:4], vals[4:6], tuple(vals[6:])
        assert philox.philox4x32_10(ctr, key) == want
        n += 1
    assert n == 3


def test_philox_stream_fields_are_distinct():
    # every field of the counter changes the output
    base = philox.uniform_u32(5, 1, 2, 1, 3, 4)
    assert len({base,
                philox.uniform_u32(6, 1, 2, 1, 3, 4), philox.uniform_u32(5, 0, 2, 1, 3, 4),
                philox.uniform_u32(5, 1, 3, 1, 3, 4), philox.uniform_u32(5, 1, 2, 2, 3, 4),
                philox.uniform_u32(5, 1, 2, 1, 4, 4), philox.uniform_u32(5, 1, 2, 1, 3, 5)}) == 7


def test_quantize_is_exact_floor():
    rng = np.random.default_rng(0)
    p = rng.random(1000).astype(np.float32)
    w = quantize(p)
    for pi, wi in zip(p[:200], w[:200]):
        exact = Fraction(float(pi)) * (1 << QBITS)
        assert wi == int(exact) and wi <= exact < wi + 1
    assert quantize(np.array([1.0]))[0] == 1 << QBITS
    assert quantize(np.array([0.0]))[0] == 0


def _draw_by_rationals(weights, u32):
    """Textbook inverse CDF on exact rationals: smallest v with CDF(v) > u."""
    total = sum(int(x) for x in weights)
    u = Fraction(int(u32), 1 << 32)
    acc = Fraction(0)
    for v, x in enumerate(weights):
        acc += Fraction(int(x), total)
        # t = floor(u * S) compared with integer prefix sums is the same as
        # comparing floor(u*S) < C_v, i.e. u*S < C_v rounded to the integer grid
        if int(u * total) < acc * total:
            return v
    raise AssertionError


def test_single_draw_matches_inverse_cdf():
    rng = np.random.default_rng(1)
    for trial in range(20):
        V = int(rng.integers(1, 40))
        w = rng.integers(0, 1 << 40, V).astype(np.int64)
        w[rng.random(V) < 0.3] = 0
        if w.sum() == 0:
            w[0] = 1
        for u in [0, (1 << 32) - 1] + [int(x) for x in rng.integers(0, 1 << 32, 50)]:
            v = draw_one(w, u)
            assert v == _draw_by_rationals(w, u)
            assert w[v] > 0          # never draws a zero-weight entry


def test_single_draw_frequencies_are_exact():
    # Count, exactly, the u32 values that select each entry: ceil(C_v 2^32 / S) - ceil(C_{v-1} 2^32 / S)
    w = np.array([3, 0, 5, 1 << 20, 7], dtype=np.int64)
    S = int(w.sum())
    cum = np.concatenate([[0], np.cumsum(w)])
    bounds = [-(-int(c) * (1 << 32) // S) for c in cum]
    for v in range(len(w)):
        lo, hi = bounds[v], bounds[v + 1]
        if hi > lo:
            assert draw_one(w, lo) == v and draw_one(w, hi - 1) == v
        count = hi - lo
        assert abs(count - w[v] * (1 << 32) / S) <= 1


def test_draws_without_replacement_equal_adjusted_prefix_search():
    """Zeroing drawn entries and redrawing equals searching the prefix sums with
    the drawn weights subtracted (the form a parallel implementation uses)."""
    rng = np.random.default_rng(2)
    for trial in range(30):
        V = int(rng.integers(2, 60))
        w = rng.integers(0, 1 << 38, V).astype(np.int64)
        us = [int(x) for x in rng.integers(0, 1 << 32, min(V, 8))]
        got = draws_without_replacement(w, us)
        cum = np.cumsum(w)
        taken, remaining = [], int(w.sum())
        for u in us:
            if remaining == 0:
                assert got[len(taken)] == -1
                taken.append(-1)
                continue
            t = (u * remaining) >> 32
            lo, hi = 0, V - 1
            while lo < hi:
                mid = (lo + hi) // 2
                adj = int(cum[mid]) - sum(int(w[x]) for x in taken if 0 <= x <= mid)
                if adj > t:
                    hi = mid
                else:
                    lo = mid + 1
            assert got[len(taken)] == lo
            taken.append(lo)
            remaining -= int(w[lo])
        assert len(set(x for x in got if x >= 0)) == len([x for x in got if x >= 0])


def test_draws_stop_when_mass_runs_out():
    w = np.array([0, 5, 0, 9], dtype=np.int64)
    got = draws_without_replacement(w, [1, 2 ** 31, 3, 4])
    assert sorted(got[:2]) == [1, 3] and got[2:] == [-1, -1]


def test_greedy_top_k_is_a_total_order_sort():
    rng = np.random.default_rng(3)
    z = rng.standard_normal(500)
    z[10] = z[20] = z[30] = 5.0                  # forced ties go to the lower id
    top = greedy_top_k(z, 7)
    want = sorted(range(500), key=lambda v: (-z[v], v))[:7]
    assert top == want and top[:3] == [10, 20, 30]
    assert argmax_low_id(z) == 10


def test_first_draw_distribution_chi2():
    """k = 1 draws with the Philox stream follow the weights (chi-square)."""
    from scipy.stats import chisquare
    p = np.array([0.05, 0.4, 0.25, 0.3])
    w = quantize(p)
    counts = np.zeros(4)
    for i in range(20000):
        counts[draw_one(w, philox.uniform_u32(11, i, 0, 0, 0, 0))] += 1
    assert chisquare(counts, p * counts.sum()).pvalue > 1e-3
