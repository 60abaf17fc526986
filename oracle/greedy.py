"""Greedy (temperature 0) drafting and verification (fp64 oracle).

Sources:
* "VocabTrim: Vocabulary Pruning for Efficient Speculative Decoding in LLMs",
  section 4 (experimental setup): the target decodes greedily, so a drafted
  token is accepted only if it equals the target's own choice, which keeps
  the generation lossless.
* the same paper, Appendix C.1, Algorithm 2: the drafter proposes k tokens
  through the trimmed head and the index mapper T_{d->t}; the target scores
  them; left to right, a token "consistent with P_t" is appended, and at the
  first inconsistent one the target's own token is generated instead and the
  block ends.

Readings where the pages leave a step open:
* greedy choice = the highest logit, ties to the lower id (the lower trimmed
  index for the drafter, which is the lower target id because trim_ids are
  ascending);
* the drafter's distribution at temperature 0 is the limit of softmax(z/T):
  one-hot at its greedy choice (the limit is uniform over tied maxima; the
  one-hot at the lower index is the greedy choice that reading fixes);
* when all gamma drafted tokens are consistent, the target's greedy token at
  position gamma is appended (the bonus of the stochastic rule; Algorithm 2
  as printed stops without it), so a block always emits n + 1 tokens;
* the acceptance "probability" reported per position is 1 for an accepted
  token and 0 for the rejected one.

Test infrastructure only; see the package docstring.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from .speculative import _decode_logits
from .vocabtrim import BadInput, bf16_to_f64


@dataclass
class GreedyResult:
    tokens: np.ndarray        # [B, gamma+1] int32, -1 padded
    num_accepted: np.ndarray  # [B] int32
    accept: np.ndarray        # [B, gamma] 1 accepted, 0 rejected, nan not tested
    choice: np.ndarray        # [B, gamma+1] the target's greedy token at each position
    gap: np.ndarray           # [B, gamma+1] top-2 gap of each target row


def argmax_lowest(row) -> int:
    """Index of the largest value, the lowest index among ties."""
    r = np.asarray(row, dtype=np.float64)
    if not np.all(np.isfinite(r)):
        raise BadInput("non-finite values in an argmax")
    m = r.max()
    return int(np.flatnonzero(r == m)[0])


def top2_gap(row) -> float:
    """Largest value minus the second largest (0 with a tie); inf for one value."""
    r = np.sort(np.asarray(row, dtype=np.float64))
    return float(r[-1] - r[-2]) if r.size > 1 else float("inf")


def draft_step_greedy(hidden_bits, W_trim_bits, trim_ids):
    """One greedy drafting step through the trimmed head (Algorithm 2).

    z = hidden @ W_trim^T in fp64; j* = argmax_lowest(z[b]); token =
    trim_ids[j*]; q[b] = one-hot at j*.  Returns dict(tokens, index, q,
    logits, gap) where gap is the top-2 gap of z[b] (near ties are where an
    fp32 projection may legitimately choose the other index).
    """
    h = bf16_to_f64(hidden_bits)
    W = bf16_to_f64(W_trim_bits)
    z = h @ W.T
    if not np.all(np.isfinite(z)):
        raise BadInput("non-finite drafter logits")
    B, K = z.shape
    trim_ids = np.asarray(trim_ids, dtype=np.int32)
    index = np.array([argmax_lowest(z[b]) for b in range(B)], dtype=np.int64)
    q = np.zeros((B, K))
    q[np.arange(B), index] = 1.0
    gap = np.array([top2_gap(z[b]) for b in range(B)])
    return dict(tokens=trim_ids[index], index=index, q=q, logits=z, gap=gap)


def verify_greedy(logits, draft_tokens, logits_dtype: str = "f32") -> GreedyResult:
    """Greedy verification of a batch of drafted blocks.

    logits       [B, gamma+1, V] target logits (fp32/fp64 values, or bf16 bits
                 with logits_dtype="bf16")
    draft_tokens [B, gamma] drafted target ids

    Position i accepts x_i iff x_i = argmax_lowest(l[b, i]); n = the first
    position that does not; the emitted block is x_0..x_{n-1} followed by
    argmax_lowest(l[b, n]) (n = gamma: the bonus position).
    """
    L = _decode_logits(logits, logits_dtype)
    B, R, V = L.shape
    gamma = R - 1
    draft = np.asarray(draft_tokens, dtype=np.int64)
    if draft.shape != (B, gamma):
        raise ValueError("shape mismatch")
    tokens = np.full((B, R), -1, dtype=np.int32)
    n_acc = np.zeros(B, dtype=np.int32)
    a_out = np.full((B, gamma), np.nan)
    choice = np.empty((B, R), dtype=np.int64)
    gap = np.empty((B, R))
    for b in range(B):
        for i in range(R):
            choice[b, i] = argmax_lowest(L[b, i])
            gap[b, i] = top2_gap(L[b, i])
        n = 0
        for i in range(gamma):
            x = int(draft[b, i])
            if not 0 <= x < V:
                raise BadInput("drafted token outside [0, V)")
            ok = x == choice[b, i]
            a_out[b, i] = 1.0 if ok else 0.0
            if ok:
                n = i + 1
            else:
                break
        tokens[b, :n] = draft[b, :n]
        tokens[b, n] = choice[b, n]
        n_acc[b] = n
    return GreedyResult(tokens, n_acc, a_out, choice, gap)
