"""Exact integration of a verify routine over its explicit uniforms.

Verification is a deterministic function of (drafts, u_accept, u_resample).
For one sequence with a fixed draft, the accept test at position i is a step
function of u_accept[i] (accepted below a threshold), and the final draw is a
non-decreasing step function of u_resample[n] (an inverse CDF).  Locating the
steps by bisection on the black box and measuring the pieces gives the exact
output distribution (to the bisection width, 2^-50), without restating any
formula of the routine under test.
"""
from __future__ import annotations

import itertools

import numpy as np

_ITERS = 50
_TOP = 1.0 - 2.0 ** -53   # largest double below 1


def _call(verify, logits, q, inv_map, draft, u_acc, u_res, T):
    r = verify(logits[None], q[None], inv_map, draft[None], u_acc[None], u_res[None], T)
    n = int(r.num_accepted[0])
    return n, tuple(int(t) for t in r.tokens[0, : n + 1])


def _threshold(fn):
    """sup{u in [0,1): fn(u)} for a predicate true on [0, theta)."""
    if not fn(0.0):
        return 0.0
    if fn(_TOP):
        return 1.0
    lo, hi = 0.0, _TOP
    for _ in range(_ITERS):
        mid = 0.5 * (lo + hi)
        if fn(mid):
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def _step_measure(fn, lo=0.0, hi=_TOP, vlo=None, vhi=None, out=None, depth=0):
    """Measure of each value of a non-decreasing step function on [0, 1)."""
    if out is None:
        out = {}
    if vlo is None:
        vlo = fn(lo)
    if vhi is None:
        vhi = fn(hi)
    if vlo == vhi:
        out[vlo] = out.get(vlo, 0.0) + (hi - lo)
        return out
    if depth >= _ITERS:
        mid = 0.5 * (lo + hi)
        out[vlo] = out.get(vlo, 0.0) + (mid - lo)
        out[vhi] = out.get(vhi, 0.0) + (hi - mid)
        return out
    mid = 0.5 * (lo + hi)
    vm = fn(mid)
    _step_measure(fn, lo, mid, vlo, vm, out, depth + 1)
    _step_measure(fn, mid, hi, vm, vhi, out, depth + 1)
    return out


def block_distribution(verify, logits, q, inv_map, draft, T=1.0):
    """Exact distribution of verify's output tuple for one fixed draft.

    logits [gamma+1, V], q [gamma, K], inv_map [V], draft [gamma].
    Returns {output tuple: probability} over u ~ U[0,1)^(2 gamma + 1).
    """
    gamma = draft.shape[0]
    u_acc = np.zeros(gamma)
    u_res = np.zeros(gamma + 1)
    thetas = []
    for i in range(gamma):
        def acc(u, i=i):
            ua = np.zeros(gamma)
            ua[i] = u
            n, _ = _call(verify, logits, q, inv_map, draft, ua, u_res, T)
            return n >= i + 1
        thetas.append(_threshold(acc))
    dist = {}
    reach = 1.0
    for k in range(gamma + 1):
        if k < gamma:
            pk = reach * (1.0 - thetas[k])
        else:
            pk = reach
        if pk > 0:
            ua = np.zeros(gamma)
            if k < gamma:
                ua[k] = 0.5 * (thetas[k] + 1.0)

            def draw(u, ua=ua, k=k):
                ur = np.zeros(gamma + 1)
                ur[k] = u
                n, toks = _call(verify, logits, q, inv_map, draft, ua, ur, T)
                assert n == k
                return toks
            for toks, meas in _step_measure(draw).items():
                dist[toks] = dist.get(toks, 0.0) + pk * meas
        if k < gamma:
            reach *= thetas[k]
    return dist


def markov_block_distribution(verify, p_tab, q_tab, ctx, gamma, T=1.0,
                              logit_fn=np.log):
    """Exact block output distribution for the toy Markov setting.

    p_tab [C, V], q_tab [C, V]: rows indexed by context (0 = BOS, t+1 after
    token t).  The draft is enumerated over V^gamma sequences with weight
    prod q(x_i | c_i); logits at position i are logit_fn(p(. | c_i)).
    """
    V = p_tab.shape[1]
    inv_map = np.arange(V, dtype=np.int32)
    dist = {}
    for draft in itertools.product(range(V), repeat=gamma):
        ctxs = [ctx] + [d + 1 for d in draft]
        w = 1.0
        for i in range(gamma):
            w *= q_tab[ctxs[i], draft[i]]
        if w == 0:
            continue
        logits = np.stack([logit_fn(p_tab[c]) for c in ctxs])
        q = np.stack([q_tab[c] for c in ctxs[:gamma]])
        d = block_distribution(verify, logits, q, inv_map, np.array(draft), T)
        for toks, pr in d.items():
            dist[toks] = dist.get(toks, 0.0) + w * pr
    return dist
