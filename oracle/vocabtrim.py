"""VocabTrim calibration, trimmed LM head and drafting step (fp64 oracle).

Source: "VocabTrim: Vocabulary Pruning for Efficient Speculative Decoding in
LLMs" (arXiv 2506.22694).

* ``token_histogram``  - Algorithm 1, "Count Token Frequencies": a counter
  c in N^|V| starts at zero and is incremented once per token occurrence.
* ``top_k``            - eq. (1), Top-K(c, k): the k ids with the largest
  counts.  The page does not order ties; the lower id wins (reading fixed for
  the calibration workload), and the result is ranked (count desc, id asc).
* ``top_p`` / ``min_count`` - section 3 notes the trimmed vocabulary may also
  be chosen by Top-P or by a minimum frequency in the calibration data; the
  page defines neither, so: the smallest ranked prefix holding at least a
  fraction P of the calibration tokens, and every id counted at least f
  times.
* ``trim_head``        - eq. (1), W^Trim = W[Top-K(c,k), :], with the rows
  kept in ascending id order (the page fixes no order), plus the token index
  mapper T_{d->t} of Algorithm 2 (trimmed index -> target id, here
  ``trim_ids``) and its inverse (target id -> trimmed index or -1).
* ``draft_logits`` / ``draft_step`` - Algorithm 2's drafting lines: the
  trimmed head produces logits over the trimmed vocabulary only, a sample is
  drawn from their softmax, and the sample is mapped back to a target id.
  Temperature divides the logits (the glossary page: temperature must be
  reflected in the distributions used for correction).

Everything is fp64 on inputs converted exactly from bf16 / fp32.
"""
from __future__ import annotations

import numpy as np

from .sampling import inverse_cdf


class BadInput(ValueError):
    """Input data the method cannot accept (out-of-range id, zero draft mass
    at a drafted token, non-finite values)."""


def bf16_to_f64(bits) -> np.ndarray:
    """Exact decode of bfloat16 bit patterns (uint16) to float64."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def token_histogram(ids, V: int) -> np.ndarray:
    """c[t] = number of occurrences of id t in ``ids`` (Algorithm 1).

    Raises BadInput for an id outside [0, V).  Returns int64 counts [V].
    """
    ids = np.asarray(ids)
    if ids.size and (ids.min() < 0 or ids.max() >= V):
        raise BadInput("token id outside [0, V)")
    return np.bincount(ids.astype(np.int64), minlength=V).astype(np.int64)


def top_k(counts, K: int) -> np.ndarray:
    """Top-K(c, K) of eq. (1): ids ranked by (count descending, id ascending)."""
    c = np.asarray(counts, dtype=np.int64)
    V = c.size
    if not 1 <= K <= V:
        raise ValueError("need 1 <= K <= V")
    ids = np.arange(V, dtype=np.int64)
    # lexsort: last key is primary -> sort by -count, then by id
    order = np.lexsort((ids, -c))
    return order[:K].astype(np.int32)


def ranking(counts) -> np.ndarray:
    """All V ids ranked by (count descending, id ascending)."""
    c = np.asarray(counts, dtype=np.int64)
    return top_k(c, c.size)


def top_p(counts, P: float):
    """Top-P selection (section 3: the trimmed vocabulary may be chosen by
    Top-P instead of Top-K).  Reading: the smallest K such that the K
    highest-ranked ids cover at least a fraction P of the calibration tokens,
    sum of their counts >= P * sum(c), compared in fp64.  P in (0, 1]; no
    calibration tokens gives K = 0.  Returns (ranked ids [V], K)."""
    P = float(P)
    if not 0.0 < P <= 1.0:
        raise ValueError("need 0 < P <= 1")
    c = np.asarray(counts, dtype=np.int64)
    order = ranking(c)
    total = int(c.sum())
    if total == 0:
        return order, 0
    run = 0
    for k, t in enumerate(order):
        run += int(c[t])
        if run >= P * total:
            return order, k + 1
    return order, int(np.count_nonzero(c))  # not reached: run ends at total


def min_count(counts, f: int):
    """Minimum-frequency selection (section 3): every id seen at least f
    times in the calibration stream.  Returns (ranked ids [V], K) with K =
    #{t : c[t] >= f}; the selected ids are the first K of the ranking."""
    c = np.asarray(counts, dtype=np.int64)
    return ranking(c), int(np.count_nonzero(c >= int(f)))


def trim_head(W_bits, topk_ids):
    """W^Trim = W[Top-K, :] (eq. (1)) and the index mapper of Algorithm 2.

    ``W_bits``: bf16 bit patterns [V, H].  ``topk_ids``: K distinct ids.
    Returns (W_trim bits [K, H], trim_ids [K] ascending, inv_map [V] int32
    with inv_map[trim_ids[j]] = j and -1 elsewhere).  Rows are copied bit
    for bit.
    """
    W = np.asarray(W_bits, dtype=np.uint16)
    V = W.shape[0]
    t = np.asarray(topk_ids, dtype=np.int64)
    if t.size == 0 or t.min() < 0 or t.max() >= V:
        raise BadInput("top-K id outside [0, V)")
    if np.unique(t).size != t.size:
        raise BadInput("duplicate top-K id")
    trim_ids = np.sort(t).astype(np.int32)
    W_trim = W[trim_ids].copy()
    inv_map = np.full(V, -1, dtype=np.int32)
    for j, tok in enumerate(trim_ids):
        inv_map[tok] = j
    return W_trim, trim_ids, inv_map


def draft_logits(hidden_bits, W_trim_bits, temperature: float) -> np.ndarray:
    """z[b, j] = (sum_h h[b,h] W_trim[j,h]) / T in fp64 (the trimmed head)."""
    T = float(temperature)
    if not (np.isfinite(T) and T > 0):
        raise ValueError("temperature must be finite and > 0")
    h = bf16_to_f64(hidden_bits)
    W = bf16_to_f64(W_trim_bits)
    return (h @ W.T) / T


def draft_step(hidden_bits, W_trim_bits, trim_ids, uniforms, temperature: float):
    """One drafting step through the trimmed head (Algorithm 2).

    For each row b: z = draft_logits, q = softmax(z) over the trimmed
    vocabulary, j* = inverse_cdf(q, u_b) in ascending trimmed index (that is,
    ascending target id), token = trim_ids[j*].

    Returns dict(q [B,K] fp64, tokens [B] int32, index [B], margin [B],
    logits [B,K] fp64).
    """
    z = draft_logits(hidden_bits, W_trim_bits, temperature)
    if not np.all(np.isfinite(z)):
        raise BadInput("non-finite drafter logits")
    B, K = z.shape
    u = np.asarray(uniforms, dtype=np.float64).reshape(B)
    trim_ids = np.asarray(trim_ids, dtype=np.int32)
    q = np.empty_like(z)
    tokens = np.empty(B, dtype=np.int32)
    index = np.empty(B, dtype=np.int64)
    margin = np.empty(B, dtype=np.float64)
    for b in range(B):
        m = z[b].max()
        e = np.exp(z[b] - m)
        q[b] = e / e.sum()
        r = inverse_cdf(q[b], u[b])
        index[b] = r.index
        margin[b] = r.margin
        tokens[b] = trim_ids[r.index]
    return dict(q=q, tokens=tokens, index=index, margin=margin, logits=z)
