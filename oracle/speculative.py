"""Speculative verification by modified rejection sampling (fp64 oracle).

Sources:
* "Speculative decoding" (SelfMadeQuant glossary), "Why a rejection needs a
  special draw": a proposal x ~ q is accepted with probability
  a(x) = min(1, p(x)/q(x)); on rejection the replacement is drawn from
  r(x) = max(p(x)-q(x), 0) / sum_y max(p(y)-q(y), 0).  Section "Distributional
  exactness has conditions": temperature and vocabulary filtering must be
  reflected in the p and q used for correction.
* "A rejection rule keeps speculative decoding's output exact", section
  "Extending the rule from one token to a drafted run": the target scores all
  gamma+1 positions; the accept test walks left to right and stops at the
  first rejection; the replacement at a rejection uses the rejected
  position's own p and q; if all gamma drafts survive, a bonus token is drawn
  from the target's distribution at position gamma.

Readings where the pages leave a step open:
* accept iff u < a(x) (the toy uses "<="; both accept with probability
  exactly a(x) for a continuous uniform);
* the drafter's q is zero outside the trimmed vocabulary (VocabTrim eq. (1)),
  so q_i(x) = q[b, i, inv_map[x]] for trimmed x and 0 otherwise;
* a drafted token with q(x) <= 0 is invalid input (the glossary: the ratio is
  only needed for proposed tokens, so its denominator is positive);
* a rejection whose residual mass is exactly zero cannot happen in exact
  arithmetic (a rejection needs q(x) > p(x), hence some p(y) > q(y)); if
  rounding produces it, the draw falls back to p at that position and the
  event is flagged;
* every categorical draw is the strict inverse CDF of ``sampling.py`` in
  ascending token-id order.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from .sampling import inverse_cdf
from .vocabtrim import BadInput, bf16_to_f64


def softmax(logits_row, temperature: float = 1.0) -> np.ndarray:
    """p = softmax(l / T) in fp64 over one row."""
    l = np.asarray(logits_row, dtype=np.float64) / float(temperature)
    if not np.all(np.isfinite(l)):
        raise BadInput("non-finite target logits")
    e = np.exp(l - l.max())
    return e / e.sum()


def acceptance_probability(p_x: float, q_x: float) -> float:
    """a(x) = min(1, p(x)/q(x)) for a proposed token (q(x) > 0)."""
    if not q_x > 0:
        raise BadInput("draft probability of a proposed token must be positive")
    return min(1.0, float(p_x) / float(q_x))


def residual_weights(p, q) -> np.ndarray:
    """Unnormalised residual max(p - q, 0) over the whole vocabulary."""
    return np.maximum(np.asarray(p, dtype=np.float64) - np.asarray(q, dtype=np.float64), 0.0)


@dataclass
class VerifyResult:
    tokens: np.ndarray            # [B, gamma+1] int32, -1 padded
    num_accepted: np.ndarray      # [B] int32
    accept_prob: np.ndarray       # [B, gamma] fp64, a(x) at each drafted token
    accept_margin: np.ndarray     # [B, gamma] |u - a|, nan where not tested
    draw_margin: np.ndarray       # [B] distance of the final draw's u to a bin edge
    draw_fallback: np.ndarray     # [B] bool: inverse-CDF fell back (rounding)
    zero_residual: np.ndarray     # [B] bool: residual mass was zero at a reject
    row_max: np.ndarray = field(default=None)   # [B, gamma+1] max of l/T
    row_sum: np.ndarray = field(default=None)   # [B, gamma+1] sum exp(l/T - max)


def _decode_logits(logits, dtype: str) -> np.ndarray:
    if dtype == "bf16":
        return bf16_to_f64(logits)
    return np.asarray(logits, dtype=np.float64)


def verify(logits, q, inv_map, draft_tokens, u_accept, u_resample,
           temperature: float = 1.0, logits_dtype: str = "f32") -> VerifyResult:
    """Verify a batch of drafted blocks.

    logits       [B, gamma+1, V] target logits (fp32/fp64 values, or bf16 bits
                 with logits_dtype="bf16")
    q            [B, gamma, K] drafter probabilities over the trimmed vocabulary
    inv_map      [V] target id -> trimmed index, -1 if not trimmed
    draft_tokens [B, gamma] drafted target ids
    u_accept     [B, gamma] and u_resample [B, gamma+1] explicit uniforms
    """
    T = float(temperature)
    if not (np.isfinite(T) and T > 0):
        raise ValueError("temperature must be finite and > 0")
    L = _decode_logits(logits, logits_dtype)
    B, R, V = L.shape
    gamma = R - 1
    q = np.asarray(q, dtype=np.float64)
    K = q.shape[2]
    inv_map = np.asarray(inv_map, dtype=np.int64)
    draft = np.asarray(draft_tokens, dtype=np.int64)
    u_acc = np.asarray(u_accept, dtype=np.float64)
    u_res = np.asarray(u_resample, dtype=np.float64)
    if q.shape != (B, gamma, K) or draft.shape != (B, gamma):
        raise ValueError("shape mismatch")

    tokens = np.full((B, R), -1, dtype=np.int32)
    n_acc = np.zeros(B, dtype=np.int32)
    a_out = np.full((B, gamma), np.nan)
    a_margin = np.full((B, gamma), np.nan)
    d_margin = np.zeros(B)
    d_fallback = np.zeros(B, dtype=bool)
    zero_res = np.zeros(B, dtype=bool)
    row_max = np.empty((B, R))
    row_sum = np.empty((B, R))

    for b in range(B):
        # target distributions at every scored position, p_i = softmax(l_i / T)
        p_rows = []
        for i in range(R):
            l = L[b, i] / T
            if not np.all(np.isfinite(l)):
                raise BadInput("non-finite target logits")
            row_max[b, i] = l.max()
            e = np.exp(l - row_max[b, i])
            row_sum[b, i] = e.sum()
            p_rows.append(e / row_sum[b, i])

        def q_full(i):
            # drafter distribution of position i over the full vocabulary
            out = np.zeros(V)
            present = inv_map >= 0
            out[present] = q[b, i, inv_map[present]]
            return out

        # left-to-right accept test, stop at the first rejection
        n = 0
        for i in range(gamma):
            x = int(draft[b, i])
            if not 0 <= x < V:
                raise BadInput("drafted token outside [0, V)")
            k = int(inv_map[x])
            if k < 0:
                raise BadInput("drafted token is not in the trimmed vocabulary")
            a = acceptance_probability(p_rows[i][x], q[b, i, k])
            a_out[b, i] = a
            a_margin[b, i] = abs(u_acc[b, i] - a)
            if u_acc[b, i] < a:
                n = i + 1
            else:
                break

        if n == gamma:
            # whole draft accepted: bonus draw from p at position gamma
            r = inverse_cdf(p_rows[gamma], u_res[b, gamma])
        else:
            w = residual_weights(p_rows[n], q_full(n))
            if w.sum() > 0:
                r = inverse_cdf(w, u_res[b, n])
            else:
                zero_res[b] = True
                r = inverse_cdf(p_rows[n], u_res[b, n])
        tokens[b, :n] = draft[b, :n]
        tokens[b, n] = r.index
        n_acc[b] = n
        d_margin[b] = r.margin
        d_fallback[b] = r.fallback

    return VerifyResult(tokens, n_acc, a_out, a_margin, d_margin, d_fallback,
                        zero_res, row_max, row_sum)
