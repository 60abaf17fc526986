"""Inverse-CDF draw of one categorical sample from one explicit uniform.

The toy sampler on "A rejection rule keeps speculative decoding's output
exact" (section "A target and a draft small enough to print in full") walks
the distribution in a fixed order, accumulates probability, and returns the
first token whose running total passes the uniform, with a floating-point
fallback to the last token.  Two readings are fixed here:

* the comparison is strict (first index whose CDF is *greater than* u), so a
  zero-probability token can never be drawn, even at u = 0; the page's
  "<=" form would return a zero-weight first token when u = 0.0, which would
  break the glossary's two-token example (its residual must always return B);
* the fallback (u at or above the computed total through rounding) returns
  the last index with positive weight, not the last index overall.

Weights need not be normalised: the CDF is divided by their fp64 sum.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass
class InverseCdfResult:
    index: int            # chosen index
    margin: float         # distance of u from the nearest edge of the chosen bin
    fallback: bool        # True when no CDF value exceeded u (rounding)


def inverse_cdf(weights, u: float) -> InverseCdfResult:
    """Smallest j with CDF_j > u, CDF_j = sum_{i<=j} w_i / sum_i w_i (fp64).

    ``weights`` are non-negative; at least one must be positive.
    """
    w = np.asarray(weights, dtype=np.float64)
    if w.ndim != 1 or w.size == 0:
        raise ValueError("weights must be a non-empty vector")
    if np.any(w < 0) or not np.all(np.isfinite(w)):
        raise ValueError("weights must be finite and non-negative")
    total = w.sum()
    if not total > 0:
        raise ValueError("weights sum to zero")
    cdf = np.cumsum(w) / total
    u = float(u)
    j = int(np.searchsorted(cdf, u, side="right"))
    if j >= w.size:
        pos = np.nonzero(w > 0)[0]
        # u sits at the very top of the CDF: always a boundary case
        return InverseCdfResult(int(pos[-1]), 0.0, True)
    lower = cdf[j - 1] if j > 0 else 0.0
    margin = min(u - lower, cdf[j] - u)
    return InverseCdfResult(j, float(margin), False)
