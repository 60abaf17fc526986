"""Pins of the Top-P and minimum-frequency selections (VocabTrim, section 3:
the trimmed vocabulary may be chosen by Top-P or by a minimum frequency in
the calibration data instead of Top-K)."""
import numpy as np
import pytest

import oracle
import synthetic


def test_hand_worked_counts():
    # counts by id: 5, 0, 9, 5, 1  -> ranking 2, 0, 3, 4, 1 (ties to the lower id)
    c = np.array([5, 0, 9, 5, 1])
    assert oracle.ranking(c).tolist() == [2, 0, 3, 4, 1]
    # total 20: P = 0.45 needs 9 (< 9.0? no: 9 >= 9.0) -> K = 1
    assert oracle.top_p(c, 0.45)[1] == 1
    assert oracle.top_p(c, 0.46)[1] == 2     # 9 < 9.2 <= 14
    assert oracle.top_p(c, 0.70)[1] == 2     # 14 >= 14.0
    assert oracle.top_p(c, 0.71)[1] == 3     # 19 >= 14.2
    assert oracle.top_p(c, 1.0)[1] == 4      # every counted id, not the zero
    assert oracle.min_count(c, 5)[1] == 3
    assert oracle.min_count(c, 6)[1] == 1
    assert oracle.min_count(c, 0)[1] == 5
    assert oracle.min_count(c, 1)[1] == 4


def test_empty_stream():
    c = np.zeros(7, np.int64)
    assert oracle.top_p(c, 0.5)[1] == 0
    assert oracle.min_count(c, 1)[1] == 0
    assert oracle.ranking(c).tolist() == list(range(7))


def test_p_out_of_range():
    for P in (0.0, -0.1, 1.5):
        with pytest.raises(ValueError):
            oracle.top_p(np.ones(3), P)


def test_brute_force_on_random_counts():
    g = synthetic.rng(5, 0)
    for trial in range(200):
        V = int(g.integers(1, 40))
        c = g.integers(0, 6, V)
        P = float(g.uniform(0.01, 1.0))
        order, K = oracle.top_p(c, P)
        total = c.sum()
        # the ranking is Python's sort on (-count, id)
        assert order.tolist() == sorted(range(V), key=lambda t: (-c[t], t))
        if total == 0:
            assert K == 0
            continue
        prefix = np.cumsum(c[order])
        # K is the first prefix length reaching P * total
        assert prefix[K - 1] >= P * total
        assert K == 1 or prefix[K - 2] < P * total
        f = int(g.integers(0, 7))
        order2, K2 = oracle.min_count(c, f)
        assert K2 == sum(1 for t in range(V) if c[t] >= f)
        assert all(c[t] >= f for t in order2[:K2]) and all(c[t] < f for t in order2[K2:])


def test_selections_agree_with_top_k():
    ids = synthetic.zipf_ids(200_000, 3000, seed=9)
    c = oracle.token_histogram(ids, 3000)
    for P in (0.5, 0.9, 0.99):
        order, K = oracle.top_p(c, P)
        assert np.array_equal(order[:K], oracle.top_k(c, K))
    order, K = oracle.min_count(c, 20)
    assert np.array_equal(order[:K], oracle.top_k(c, K))
