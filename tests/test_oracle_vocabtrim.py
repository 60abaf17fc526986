"""Pins for the oracle's calibration, trimming and drafting step.

Expected values come from hand-worked fixtures (golden/histogram_topk.json),
brute force with independent Python routines (collections.Counter, sorted,
exact rational arithmetic), closed forms of softmax, and the head sizes that
VocabTrim's Tables 1-3 quote for the Llama-3 vocabulary (128256 ids).
"""
import collections
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
from scipy import stats

import oracle
import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _cases():
    with open(os.path.join(GOLDEN, "histogram_topk.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _cases())
def test_golden_histogram_topk_trim(case):
    c = oracle.token_histogram(np.array(case["ids"], dtype=np.int32), case["V"])
    assert list(c) == case["counts"]
    t = oracle.top_k(c, case["K"])
    assert list(t) == case["topk"]
    W = np.arange(case["V"] * 3, dtype=np.uint16).reshape(case["V"], 3)
    W_trim, trim_ids, inv_map = oracle.trim_head(W, t)
    assert list(trim_ids) == case["trim_ids"]
    assert list(inv_map) == case["inv_map"]
    assert np.array_equal(W_trim, W[case["trim_ids"]])


def test_histogram_brute_force():
    g = synthetic.rng(21, 0)
    for V, N in [(1, 10), (7, 1000), (300, 5000)]:
        ids = g.integers(0, V, N).astype(np.int32)
        c = oracle.token_histogram(ids, V)
        ref = collections.Counter(int(x) for x in ids)
        assert all(c[t] == ref.get(t, 0) for t in range(V))
        assert c.sum() == N                      # conservation
    assert oracle.token_histogram(np.zeros(0, np.int32), 4).tolist() == [0, 0, 0, 0]


def test_histogram_rejects_out_of_range():
    with pytest.raises(oracle.BadInput):
        oracle.token_histogram(np.array([0, 5], np.int32), 5)
    with pytest.raises(oracle.BadInput):
        oracle.token_histogram(np.array([-1], np.int32), 5)


def test_topk_brute_force_with_ties():
    g = synthetic.rng(22, 0)
    for V, K, hi in [(50, 10, 4), (200, 200, 3), (1000, 137, 20), (5, 1, 1)]:
        c = g.integers(0, hi, V)
        t = oracle.top_k(c, K)
        ref = sorted(range(V), key=lambda i: (-int(c[i]), i))[:K]
        assert list(t) == ref


def test_topk_rejects_bad_k():
    with pytest.raises(ValueError):
        oracle.top_k(np.ones(4), 0)
    with pytest.raises(ValueError):
        oracle.top_k(np.ones(4), 5)


def test_trim_properties():
    g = synthetic.rng(23, 0)
    V, H, K = 500, 24, 77
    W = g.integers(0, 65535, (V, H)).astype(np.uint16)
    topk = g.permutation(V)[:K].astype(np.int32)
    W_trim, trim_ids, inv_map = oracle.trim_head(W, topk)
    assert np.all(np.diff(trim_ids) > 0)
    assert set(trim_ids.tolist()) == set(topk.tolist())
    for j, tok in enumerate(trim_ids):
        assert inv_map[tok] == j
        assert np.array_equal(W_trim[j], W[tok])          # bit for bit
    assert int((inv_map >= 0).sum()) == K


def test_trim_rejects_duplicates_and_range():
    W = np.zeros((5, 2), np.uint16)
    with pytest.raises(oracle.BadInput):
        oracle.trim_head(W, np.array([1, 1], np.int32))
    with pytest.raises(oracle.BadInput):
        oracle.trim_head(W, np.array([5], np.int32))


def test_head_sizes_match_vocabtrim_tables():
    # LM-head sizes quoted for the Llama-3 vocabulary: 394.0M (H=3072),
    # 525.3M (H=4096), 131.3M (H=1024); a trimmed head of ~32.9K ids gives
    # 101.3M at H=3072.  The trimmed head has K*H parameters.
    V = 128256
    for H, quoted in [(3072, 394.0), (4096, 525.3), (1024, 131.3)]:
        W = np.zeros((V, 1), np.uint16)
        W_trim, _, _ = oracle.trim_head(W, np.arange(V, dtype=np.int32))
        assert round(W_trim.shape[0] * H / 1e6, 1) == quoted
    W = np.zeros((V, 1), np.uint16)
    W_trim, _, _ = oracle.trim_head(W, np.arange(32976, dtype=np.int32))
    assert round(W_trim.shape[0] * 3072 / 1e6, 1) == 101.3


def _bf16(x):
    return synthetic.to_bf16_bits(np.asarray(x, dtype=np.float32))


def test_draft_logits_exact_rational():
    g = synthetic.rng(24, 0)
    B, K, H = 3, 5, 7
    h = _bf16(g.standard_normal((B, H)))
    W = _bf16(g.standard_normal((K, H)))
    z = oracle.draft_logits(h, W, 1.0)
    hf = oracle.bf16_to_f64(h)
    Wf = oracle.bf16_to_f64(W)
    for b in range(B):
        for j in range(K):
            exact = sum(Fraction(float(hf[b, k])) * Fraction(float(Wf[j, k])) for k in range(H))
            assert z[b, j] == float(exact)          # bf16 products sum exactly in fp64


def test_draft_logits_one_hot_hidden():
    g = synthetic.rng(25, 0)
    K, H = 9, 6
    W = _bf16(g.standard_normal((K, H)))
    h = np.zeros((H, H), np.float32)
    h[np.arange(H), np.arange(H)] = 1.0
    z = oracle.draft_logits(_bf16(h), W, 0.5)
    assert np.array_equal(z, oracle.bf16_to_f64(W).T / 0.5)


def test_draft_step_two_token_softmax_and_sampling():
    # z = (0, ln 3) -> q = (1/4, 3/4); the draw is A for u < 1/4, B otherwise
    h = _bf16(np.array([[1.0]]))
    W = np.array([[0.0], [math.log(3.0)]])
    # store ln 3 exactly as a bf16 value and compare with its softmax
    Wb = _bf16(W)
    z1 = float(oracle.bf16_to_f64(Wb)[1, 0])
    want = [1 / (1 + math.exp(z1)), math.exp(z1) / (1 + math.exp(z1))]
    for u, tok in [(0.0, 10), (want[0] - 1e-6, 10), (want[0] + 1e-6, 20), (0.99, 20)]:
        r = oracle.draft_step(h, Wb, np.array([10, 20], np.int32), np.array([u]), 1.0)
        assert r["q"][0] == pytest.approx(want, abs=1e-15)
        assert int(r["tokens"][0]) == tok


def test_draft_step_trimmed_equals_masked_full_head():
    # restricting the head to the trimmed rows equals the full-vocab softmax
    # with q set to zero off the trimmed set and renormalised, and sampling in
    # ascending id order makes the drawn id identical
    g = synthetic.rng(26, 0)
    V, H, K, B = 40, 8, 13, 6
    W = _bf16(g.standard_normal((V, H)))
    h = _bf16(g.standard_normal((B, H)))
    topk = g.permutation(V)[:K].astype(np.int32)
    W_trim, trim_ids, _ = oracle.trim_head(W, topk)
    u = synthetic.uniforms(26, 1, B)
    full = oracle.draft_step(h, W, np.arange(V, dtype=np.int32), u, 0.8)
    trim = oracle.draft_step(h, W_trim, trim_ids, u, 0.8)
    masked = full["q"][:, trim_ids]
    masked = masked / masked.sum(axis=1, keepdims=True)
    assert trim["q"] == pytest.approx(masked, rel=1e-12)
    assert trim["q"].sum(axis=1) == pytest.approx(np.ones(B), abs=1e-12)
    for b in range(B):
        w = np.zeros(V)
        w[trim_ids] = full["q"][b, trim_ids]
        cdf = np.cumsum(w) / w.sum()
        assert int(trim["tokens"][b]) == int(np.argmax(cdf > u[b]))


def test_draft_step_frequencies_chi_square():
    g = synthetic.rng(27, 0)
    K, H = 12, 4
    W = _bf16(g.standard_normal((K, H)))
    h1 = _bf16(g.standard_normal((1, H)))
    N = 20_000
    h = np.repeat(h1, N, axis=0)
    u = synthetic.uniforms(27, 1, N)
    r = oracle.draft_step(h, W, np.arange(K, dtype=np.int32), u, 1.0)
    counts = np.bincount(r["tokens"], minlength=K)
    qv = r["q"][0]
    assert stats.chisquare(counts, qv * N).pvalue > 1e-3
