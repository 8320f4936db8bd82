"""Pins of the oracle's row allocation (CPU only).

The pages fix the constraints (L³: Large Lookup Layers, gist.science, Technical Summary >
Information-Theoretic Embedding Allocation: at least 1 and at most k rows per token, a
budget of v rows, more rows for frequent tokens). The frequency rule itself is this
library's reading; it is pinned here by hand-worked cases, an exact rational solution of
the water-filling, and brute force over all integer vectors on tiny inputs.
"""
import itertools
import json
import os
from fractions import Fraction

import numpy as np
import pytest

import l3_workloads as W
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _cases():
    with open(os.path.join(GOLDEN, "hand_worked_allocation.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_hand_worked_allocation(case):
    a = oracle.allocate(case["freq"], case["v"], case["n_min"], case["n_max"], case["power"])
    np.testing.assert_allclose(a.target, case["target"], rtol=1e-15)
    assert a.n.tolist() == case["n"]
    assert a.offs.tolist() == case["offs"]


@pytest.mark.parametrize("cid", sorted(W.PRESETS))
def test_preset_allocation_invariants(cid):
    p = W.PRESETS[cid]
    a = oracle.allocate(W.zipf_freq(p.vocab), p.v, 1, p.k_max, p.power)
    assert a.n.sum() == p.v and a.offs[-1] == p.v and a.offs[0] == 0
    assert a.n.min() >= 1 and a.n.max() <= p.k_max
    assert np.all(np.diff(a.n) <= 0), "more frequent ids never get fewer rows"
    assert np.all(np.abs(a.n - a.target) < 1.0)
    # heavy tail: the most frequent id is at the cap
    assert a.n[0] == p.k_max


def _exact_water_fill(w, v, lo, hi):
    """Exact rational targets: try every (capped prefix, floored suffix) of the sorted weights."""
    N = len(w)
    order = sorted(range(N), key=lambda i: -w[i])
    for h in range(N + 1):
        for l in range(N - h + 1):
            free = order[h:N - l]
            H, L = order[:h], order[N - l:]
            if not free:
                if hi * h + lo * l == v:
                    r = [Fraction(hi) if i in H else Fraction(lo) for i in range(N)]
                    return r
                continue
            c = Fraction(v - hi * h - lo * l) / sum(w[i] for i in free)
            ok = all(c * w[i] >= hi for i in H) and all(c * w[i] <= lo for i in L) and \
                all(lo <= c * w[i] <= hi for i in free)
            if ok:
                return [Fraction(hi) if i in H else Fraction(lo) if i in L else c * w[i] for i in range(N)]
    raise AssertionError("no consistent active set")


@pytest.mark.parametrize("seed", range(25))
def test_water_filling_matches_exact_rational_solution(seed):
    rng = np.random.default_rng(seed)
    N = int(rng.integers(2, 9))
    num = rng.integers(1, 40, size=N)
    den = rng.integers(1, 9, size=N)
    w = [Fraction(int(a), int(b)) for a, b in zip(num, den)]
    lo, hi = 1, int(rng.integers(2, 12))
    v = int(rng.integers(N * lo, N * hi + 1))
    a = oracle.allocate([float(x) for x in w], v, lo, hi, 1.0)
    exact = _exact_water_fill(w, v, lo, hi)
    np.testing.assert_allclose(a.target, [float(x) for x in exact], rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("seed", range(40))
def test_rounding_minimises_squared_error_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    N = int(rng.integers(1, 6))
    lo, hi = 1, int(rng.integers(1, 6))
    v = int(rng.integers(N * lo, min(N * hi, 20) + 1)) if N * lo <= min(N * hi, 20) else N * lo
    freq = rng.uniform(0.1, 10.0, size=N)
    a = oracle.allocate(freq, v, lo, hi, float(rng.choice([0.5, 0.7, 1.0])))
    r = a.target
    best, best_vecs = None, []
    for n in itertools.product(range(lo, hi + 1), repeat=N):
        if sum(n) != v:
            continue
        err = sum((ni - ri) ** 2 for ni, ri in zip(n, r))
        if best is None or err < best - 1e-12:
            best, best_vecs = err, [n]
        elif abs(err - best) <= 1e-12:
            best_vecs.append(n)
    assert tuple(a.n.tolist()) in best_vecs
    # among tied optima the lower ids get the extra rows: lexicographically largest
    assert tuple(a.n.tolist()) == max(best_vecs)


def test_infeasible_and_bad_arguments_raise():
    with pytest.raises(ValueError):
        oracle.allocate([1.0, 1.0], 5, 1, 2, 1.0)
    with pytest.raises(ValueError):
        oracle.allocate([1.0, 1.0], 1, 1, 2, 1.0)
    with pytest.raises(ValueError):
        oracle.allocate([1.0, 0.0], 3, 1, 2, 1.0)


def test_extreme_budgets_hit_the_bounds():
    f = W.zipf_freq(10)
    assert oracle.allocate(f, 10, 1, 7, 0.7).n.tolist() == [1] * 10
    assert oracle.allocate(f, 70, 1, 7, 0.7).n.tolist() == [7] * 10
