"""Pins for the oracle's inverse-CDF sampler, softmax and acceptance pieces.

The facts checked here come from the pages or from plain arithmetic, never
from the oracle itself:
* the glossary's two-token table fixes a(A)=0.75, a(B)=1 and a residual that
  puts all mass on B;
* softmax of logits (0, ln 3) is (1/4, 3/4), and at T = 1/2 it is (1/10, 9/10);
* a strict inverse CDF over weights (1, 1, 2) has edges at 1/4 and 1/2.
"""
import json
import math
import os

import numpy as np
import pytest
from scipy import stats

import oracle
import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _two_token():
    with open(os.path.join(GOLDEN, "two_token.json")) as f:
        return json.load(f)


def test_acceptance_matches_two_token_table():
    g = _two_token()
    for px, qx, want in zip(g["p"], g["q"], g["acceptance_given_proposal"]):
        assert oracle.acceptance_probability(px, qx) == pytest.approx(want, abs=1e-15)
    # accepted mass q(x) a(x) and its total
    acc = [qx * oracle.acceptance_probability(px, qx) for px, qx in zip(g["p"], g["q"])]
    assert acc == pytest.approx(g["accepted_mass"], abs=1e-15)
    assert sum(acc) == pytest.approx(g["accepted_total"], abs=1e-15)


def test_residual_matches_two_token_table():
    g = _two_token()
    w = oracle.residual_weights(g["p"], g["q"])
    assert (w / w.sum()) == pytest.approx(g["residual"], abs=1e-12)
    # the residual draw returns B for every uniform, including u = 0
    for u in [0.0, 1e-9, 0.3, 0.5, 0.999999]:
        assert oracle.inverse_cdf(w, u).index == 1


def test_acceptance_rejects_zero_draft_mass():
    with pytest.raises(oracle.BadInput):
        oracle.acceptance_probability(0.5, 0.0)


def test_softmax_closed_forms():
    p = oracle.softmax([0.0, math.log(3.0)], 1.0)
    assert p == pytest.approx([0.25, 0.75], abs=1e-15)
    p = oracle.softmax([0.0, math.log(3.0)], 0.5)
    assert p == pytest.approx([0.1, 0.9], abs=1e-15)
    # shift invariance on large logits (no overflow)
    p = oracle.softmax([1000.0, 1000.0 + math.log(3.0)], 1.0)
    assert p == pytest.approx([0.25, 0.75], abs=1e-12)


def test_inverse_cdf_edges_are_strict():
    w = [1.0, 1.0, 2.0]
    cases = [(0.0, 0), (0.2499999, 0), (0.25, 1), (0.4999999, 1), (0.5, 2), (0.9999999, 2)]
    for u, want in cases:
        assert oracle.inverse_cdf(w, u).index == want, u


def test_inverse_cdf_skips_zero_weight_bins():
    assert oracle.inverse_cdf([0.0, 1.0], 0.0).index == 1
    assert oracle.inverse_cdf([0.0, 0.0, 3.0, 0.0, 1.0], 0.74).index == 2
    assert oracle.inverse_cdf([0.0, 0.0, 3.0, 0.0, 1.0], 0.75).index == 4


def test_inverse_cdf_fallback_is_last_positive():
    r = oracle.inverse_cdf([1.0, 1.0, 0.0, 0.0], 1.0)
    assert r.fallback and r.index == 1 and r.margin == 0.0


def test_inverse_cdf_margin():
    r = oracle.inverse_cdf([1.0, 1.0, 2.0], 0.3)
    assert r.index == 1
    assert r.margin == pytest.approx(0.05, abs=1e-15)


def test_inverse_cdf_frequencies_chi_square():
    # sampler sanity check shaped like the nightly-build page's 200k-draw test
    g = synthetic.rng(123, 0)
    p = g.dirichlet(np.ones(18))
    u = synthetic.uniforms(123, 1, 200_000)
    counts = np.zeros(18, dtype=np.int64)
    for x in u[:200_000]:
        counts[oracle.inverse_cdf(p, float(x)).index] += 1
    chi2, pval = stats.chisquare(counts, p * counts.sum())
    assert pval > 1e-3
    assert np.abs(counts / counts.sum() - p).max() < 0.005
