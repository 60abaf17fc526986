"""Greedy verification of a draft tree, and the drafter's top-k candidates
(fp64 oracle).

Sources: "VocabTrim: Vocabulary Pruning for Efficient Speculative Decoding
in LLMs", section 4.1 ("Draft Tree": a tree of depth 3, top-K 8, at most 32
tokens, drafted, built and verified as in EAGLE-2) with the greedy target of
section 4 (a token is accepted only if it equals the target's choice), and
Algorithm 2 (accept the consistent prefix, replace the first inconsistent
token by the target's).

Readings where the pages leave a step open:
* a tree holds N drafted nodes in topological order: node i carries a
  target id tokens[i] and a parent parent[i] in {-1} or [0, i), -1 meaning
  the context; the target scores N + 1 positions: row 0 after the context,
  row i + 1 after node i;
* node i is accepted iff its parent is accepted (the context always is) and
  tokens[i] is the target's greedy choice at its parent's row; the emitted
  block is the token path from the context to the deepest accepted node
  (ties to the lower node index) followed by the target's choice at that
  node's row -- for a chain (parent[i] = i - 1) this is exactly the greedy
  block of ``greedy.verify_greedy``;
* the drafter's top-k at one position are its k highest trimmed logits,
  ties to the lower trimmed index, each with its log-probability
  log softmax(z / T); how a tree is grown from them (EAGLE-2's expansion and
  re-ranking) is the caller's policy and not restated here.

Test infrastructure only; see the package docstring.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from .greedy import argmax_lowest
from .speculative import _decode_logits
from .vocabtrim import BadInput, bf16_to_f64


@dataclass
class TreeResult:
    tokens: np.ndarray        # [B, N+1] the emitted block, -1 padded
    num_accepted: np.ndarray  # [B] accepted drafted tokens (path length)
    path: np.ndarray          # [B, N] node indices of the accepted path, -1 padded
    choice: np.ndarray        # [B, N+1] the target's greedy choice at every row


def verify_tree_greedy(logits, parent, tokens, logits_dtype: str = "f32") -> TreeResult:
    """Greedy verification of B draft trees of N nodes.

    logits [B, N+1, V] (row 0: after the context, row i+1: after node i),
    parent [B, N] (or [N], shared) in {-1} or [0, i), tokens [B, N] target ids.
    """
    L = _decode_logits(logits, logits_dtype)
    B, R, V = L.shape
    N = R - 1
    parent = np.asarray(parent, dtype=np.int64)
    if parent.ndim == 1:
        parent = np.broadcast_to(parent, (B, N))
    tokens = np.asarray(tokens, dtype=np.int64)
    if parent.shape != (B, N) or tokens.shape != (B, N):
        raise ValueError("shape mismatch")
    out = np.full((B, R), -1, dtype=np.int32)
    n_acc = np.zeros(B, dtype=np.int32)
    path = np.full((B, N), -1, dtype=np.int32)
    choice = np.empty((B, R), dtype=np.int64)
    for b in range(B):
        for r in range(R):
            choice[b, r] = argmax_lowest(L[b, r])
        accepted = np.zeros(N, dtype=bool)
        depth = np.zeros(N, dtype=np.int64)
        for i in range(N):
            p = int(parent[b, i])
            if not -1 <= p < i:
                raise BadInput("a parent must precede its node")
            if not 0 <= tokens[b, i] < V:
                raise BadInput("drafted token outside [0, V)")
            parent_ok = True if p < 0 else bool(accepted[p])
            accepted[i] = parent_ok and tokens[b, i] == choice[b, p + 1]
            depth[i] = 1 if p < 0 else depth[p] + 1
        best, best_depth = -1, 0
        for i in range(N):
            if accepted[i] and depth[i] > best_depth:
                best, best_depth = i, int(depth[i])
        nodes = []
        i = best
        while i >= 0:
            nodes.append(i)
            i = int(parent[b, i])
        nodes.reverse()
        for k, i in enumerate(nodes):
            out[b, k] = tokens[b, i]
            path[b, k] = i
        out[b, len(nodes)] = choice[b, best + 1]
        n_acc[b] = len(nodes)
    return TreeResult(out, n_acc, path, choice)


def draft_topk(hidden_bits, W_trim_bits, trim_ids, k: int, temperature: float = 1.0):
    """The drafter's k best candidates at one position, per row b.

    z = hidden @ W_trim^T (fp64); the k highest z (ties to the lower trimmed
    index) in descending order; their target ids and log q = log softmax(z/T).
    Returns dict(index [B,k], ids [B,k], logq [B,k], logits [B,K]).
    """
    T = float(temperature)
    if not (np.isfinite(T) and T > 0):
        raise ValueError("temperature must be finite and > 0")
    h = bf16_to_f64(hidden_bits)
    W = bf16_to_f64(W_trim_bits)
    z = h @ W.T
    if not np.all(np.isfinite(z)):
        raise BadInput("non-finite drafter logits")
    B, K = z.shape
    if not 1 <= k <= K:
        raise ValueError("need 1 <= k <= K")
    trim_ids = np.asarray(trim_ids, dtype=np.int32)
    index = np.empty((B, k), dtype=np.int64)
    logq = np.empty((B, k))
    for b in range(B):
        order = sorted(range(K), key=lambda j: (-z[b, j], j))[:k]
        index[b] = order
        s = z[b] / T
        m = s.max()
        lse = m + np.log(np.exp(s - m).sum())
        logq[b] = s[order] - lse
    return dict(index=index, ids=trim_ids[index], logq=logq, logits=z)
