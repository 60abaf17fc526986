"""Comparison rules between the CUDA library and the CPU oracle.

* integers decided without floating point (histograms, Top-K ids, copied
  weights, the drafted prefix): bit-exact;
* logits: |gpu - ref| <= 1e-3 * max(|ref|, rms(row));
* probabilities: |gpu - ref| <= 1e-3 * |ref| + 1e-7;
* decisions taken by comparing a uniform with a floating-point quantity (an
  accept test, an inverse-CDF draw): identical unless the oracle's uniform
  lies within 1e-5 of the decision boundary (the oracle's fp64 value).
  Excluded cases are counted and returned.
"""
from __future__ import annotations

import numpy as np

BOUNDARY = 1e-5
PROB_RTOL = 1e-3
PROB_ATOL = 1e-7


def assert_probs_close(gpu, ref, what="probabilities"):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    err = np.abs(gpu - ref)
    lim = PROB_RTOL * np.abs(ref) + PROB_ATOL
    bad = ~(err <= lim)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} out of tolerance, first at {tuple(i)}: "
                             f"gpu={gpu[tuple(i)]!r} ref={ref[tuple(i)]!r}")


def assert_logits_close(gpu, ref, what="logits"):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = np.sqrt(np.mean(ref ** 2, axis=-1, keepdims=True))
    lim = 1e-3 * np.maximum(np.abs(ref), rms)
    bad = ~(np.abs(gpu - ref) <= lim)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} out of tolerance, first at {tuple(i)}: "
                             f"gpu={gpu[tuple(i)]!r} ref={ref[tuple(i)]!r}")


def draw_is_valid(weights, u, index, tol=BOUNDARY):
    """For a draw excluded as a boundary case: the chosen bin must lie within
    ``tol`` of the uniform in the oracle's fp64 CDF, and have positive weight."""
    w = np.asarray(weights, dtype=np.float64)
    if not (0 <= index < w.size) or not w[index] > 0:
        return False
    cdf = np.cumsum(w) / w.sum()
    lo = cdf[index - 1] if index > 0 else 0.0
    hi = cdf[index]
    return lo - tol <= float(u) < hi + tol


def compare_verify(tokens, n_acc, accept_prob, ref, boundary=BOUNDARY, draw_weights=None):
    """Compare vt_verify outputs with oracle.verify's VerifyResult.

    ``draw_weights(b, n)`` (optional) returns the oracle's fp64 weights of the
    final draw of sequence b; with it, boundary draws are checked for
    validity instead of skipped.
    Returns dict(compared=..., excluded_seq=..., excluded_draw=...).
    """
    tokens = np.asarray(tokens)
    n_acc = np.asarray(n_acc)
    B, R = tokens.shape
    gamma = R - 1
    stats = dict(compared=0, excluded_seq=0, excluded_draw=0)
    for b in range(B):
        n_ref = int(ref.num_accepted[b])
        tested = min(n_ref, gamma - 1) + 1
        margins = ref.accept_margin[b, :tested]
        if np.nanmin(margins) <= boundary:
            stats["excluded_seq"] += 1
            continue
        assert int(n_acc[b]) == n_ref, f"seq {b}: accepted {int(n_acc[b])} vs oracle {n_ref}"
        assert np.array_equal(tokens[b, :n_ref], ref.tokens[b, :n_ref]), f"seq {b}: prefix"
        assert np.all(tokens[b, n_ref + 1:] == -1), f"seq {b}: padding"
        if accept_prob is not None:
            assert_probs_close(np.asarray(accept_prob)[b, :tested], ref.accept_prob[b, :tested],
                               f"accept prob seq {b}")
            assert np.all(np.isnan(np.asarray(accept_prob)[b, tested:])), f"seq {b}: NaN tail"
        if ref.draw_margin[b] <= boundary:
            stats["excluded_draw"] += 1
            if draw_weights is not None:
                w, u = draw_weights(b, n_ref)
                assert draw_is_valid(w, u, int(tokens[b, n_ref])), (
                    f"seq {b}: boundary draw {int(tokens[b, n_ref])} not within tolerance")
        else:
            assert int(tokens[b, n_ref]) == int(ref.tokens[b, n_ref]), (
                f"seq {b}: drawn token {int(tokens[b, n_ref])} vs oracle {int(ref.tokens[b, n_ref])}"
                f" (n={n_ref}, margin={ref.draw_margin[b]:.3g})")
        stats["compared"] += 1
    return stats
