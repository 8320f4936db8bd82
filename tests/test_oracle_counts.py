"""Pins of the oracle's token-stream counting and the allocation taken from counts.

The pages ("Information-Theoretic Embedding Allocation", gist.science explainer) tie each
token's rows to how often it occurs. The pins: counts by brute force on tiny streams;
counts sum to the stream length; a stream in which every id occurs equally often gives
the even allocation; counts proportional to a pmf give the pmf's own allocation (the
rule is scale-free); more frequent ids never get fewer rows; unseen ids get the fewest rows.
"""
import numpy as np
import pytest

import l3_workloads as W
import oracle


@pytest.mark.parametrize("seed", range(5))
def test_counts_match_brute_force(seed):
    rng = np.random.default_rng(seed)
    vocab = int(rng.integers(1, 40))
    ids = rng.integers(0, vocab, int(rng.integers(0, 200)))
    got = oracle.count_ids(ids, vocab)
    want = [sum(1 for i in ids.tolist() if i == t) for t in range(vocab)]
    assert got.dtype == np.int64 and got.tolist() == want
    assert int(got.sum()) == len(ids)


def test_count_rejects_ids_out_of_range():
    with pytest.raises(ValueError):
        oracle.count_ids([0, 3, 4], 4)
    with pytest.raises(ValueError):
        oracle.count_ids([-1], 4)
    assert oracle.count_ids([], 3).tolist() == [0, 0, 0]


def test_equal_counts_give_the_even_allocation():
    vocab, v = 64, 64 * 5
    counts = oracle.count_ids(np.tile(np.arange(vocab), 7), vocab)
    al = oracle.allocate_from_counts(counts, v, 1, 16, 0.7, 1.0)
    assert np.all(al.n == 5)


def test_counts_proportional_to_a_pmf_reproduce_its_allocation():
    # freq_t = c * (t+1)^-1.1 scaled to integers exactly: allocate is scale-free, so with
    # no smoothing the counts give the closed-form allocation of the pmf
    vocab = 256
    f = W.zipf_freq(vocab)
    counts = np.array([round(1e6 * x) for x in f], dtype=np.int64)
    from_counts = oracle.allocate_from_counts(counts, 1024, 1, 16, 1.0, 0.0)
    from_pmf = oracle.allocate(counts.astype(np.float64), 1024, 1, 16, 1.0)
    assert np.array_equal(from_counts.offs, from_pmf.offs)
    # and close to the unrounded pmf's own allocation (counts differ by rounding only)
    exact = oracle.allocate(f, 1024, 1, 16, 1.0)
    assert np.abs(from_counts.n - exact.n).max() <= 1


def test_allocation_from_counts_is_monotone_and_unseen_ids_get_fewest():
    rng = np.random.default_rng(3)
    vocab = 500
    ids = W.sample_ids(vocab, 20000, rng)
    counts = oracle.count_ids(ids, vocab)
    al = oracle.allocate_from_counts(counts, 8000, 1, 64, 0.7, 1.0)
    assert al.n.sum() == 8000 and al.n.min() >= 1 and al.n.max() <= 64
    order = np.argsort(-counts, kind="stable")
    assert np.all(np.diff(al.n[order]) <= 0)  # more occurrences, at least as many rows
    assert (counts == 0).any() and np.all(al.n[counts == 0] == al.n.min())  # fewest rows
