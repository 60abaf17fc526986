"""Pins for the oracle's block verification (modified rejection sampling).

What fixes the expected values:
* the glossary's two-token worked example (golden/two_token.json): final
  mass (0.6, 0.4) with the residual, (0.72, 0.28) with a naive redraw;
* the exactness theorem on the nightly-build page: each emitted token is
  distributed as the target p, and a chained stream follows the target chain
  (checked by exact integration over the uniforms and by chi-square);
* beta = sum_x min(p(x), q(x)) is the probability that a position survives,
  and with constant beta the block length has mean (1-beta^(gamma+1))/(1-beta)
  (Leviathan et al. eq. 1 as quoted on the nightly-build page).
"""
import json
import math
import os

import numpy as np
import pytest
from scipy import stats

import oracle
import oracle.speculative as spec
import synthetic
from exact import block_distribution, markov_block_distribution

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _two_token():
    with open(os.path.join(GOLDEN, "two_token.json")) as f:
        return json.load(f)


def _two_token_final(verify):
    g = _two_token()
    p = np.array(g["p"])
    q = np.array(g["q"])
    logits = np.log(np.stack([p, p]))
    inv_map = np.arange(2, dtype=np.int32)
    first = np.zeros(2)
    rej = 0.0
    for x in range(2):
        d = block_distribution(verify, logits, q[None], inv_map, np.array([x]))
        for toks, pr in d.items():
            first[toks[0]] += q[x] * pr
            if len(toks) == 1:
                rej += q[x] * pr
    return g, first, rej


def test_two_token_example_exact():
    g, first, rej = _two_token_final(oracle.verify)
    assert first == pytest.approx(g["final"], abs=1e-12)
    assert rej == pytest.approx(g["rejection_probability"], abs=1e-12)


def test_two_token_naive_redraw_negative_control(monkeypatch):
    # plant the biased rule (redraw from the unadjusted target) in the oracle
    monkeypatch.setattr(spec, "residual_weights", lambda p, q: np.asarray(p, dtype=np.float64))
    g, first, _ = _two_token_final(oracle.verify)
    assert first == pytest.approx(g["naive_redraw_final"], abs=1e-12)


def test_two_token_spot_checks():
    g = _two_token()
    p = np.array(g["p"])
    q = np.array(g["q"])
    logits = np.log(np.stack([p, p]))[None]
    inv_map = np.arange(2, dtype=np.int32)
    for u, want_n in [(0.74, 1), (0.76, 0)]:
        r = oracle.verify(logits, q[None, None], inv_map, np.array([[0]]),
                          np.array([[u]]), np.array([[0.0, 0.0]]))
        assert int(r.num_accepted[0]) == want_n
        if want_n == 0:
            assert list(r.tokens[0]) == [1, -1]   # residual returns B
    # proposal B is always accepted (a = 1)
    r = oracle.verify(logits, q[None, None], inv_map, np.array([[1]]),
                      np.array([[0.999999]]), np.array([[0.0, 0.0]]))
    assert int(r.num_accepted[0]) == 1
    assert r.accept_prob[0, 0] == pytest.approx(1.0)


def _exact_first_and_pairs(p_tab, q_tab, gamma, T=1.0, logit_fn=np.log, ctxs=None):
    C, V = p_tab.shape
    blocks = {}
    for c in (range(C) if ctxs is None else ctxs):
        blocks[c] = markov_block_distribution(oracle.verify, p_tab, q_tab, c, gamma, T, logit_fn)
    return blocks


def _first_marginal(block, V):
    m = np.zeros(V)
    for toks, pr in block.items():
        m[toks[0]] += pr
    return m


def test_exactness_small_vocab_gamma2():
    # V=3, gamma=2: every emitted token and every emitted pair follows p
    g = synthetic.rng(5, 0)
    V = 3
    p_tab = g.dirichlet(np.ones(V), size=V + 1)
    q_tab = g.dirichlet(np.ones(V), size=V + 1)
    blocks = _exact_first_and_pairs(p_tab, q_tab, 2)
    for c in range(V + 1):
        total = sum(blocks[c].values())
        assert total == pytest.approx(1.0, abs=1e-12)
        assert _first_marginal(blocks[c], V) == pytest.approx(p_tab[c], abs=1e-12)
    # stream joint of the first two tokens from BOS composes across a block
    # boundary when the block emits a single token
    joint = np.zeros((V, V))
    for toks, pr in blocks[0].items():
        if len(toks) >= 2:
            joint[toks[0], toks[1]] += pr
        else:
            joint[toks[0]] += pr * _first_marginal(blocks[toks[0] + 1], V)
    want = p_tab[0][:, None] * p_tab[1:]
    assert joint == pytest.approx(want, abs=1e-12)


def test_exactness_with_temperature():
    # p = softmax(l / T): the output follows the tempered target
    g = synthetic.rng(6, 0)
    V, T = 3, 0.7
    l_tab = g.standard_normal((V + 1, V)) * 2.0
    q_tab = g.dirichlet(np.ones(V), size=V + 1)
    blocks = _exact_first_and_pairs(np.exp(l_tab), q_tab, 1, T=T, logit_fn=np.log, ctxs=[0, 2])
    for c in [0, 2]:
        e = [math.exp(x / T) for x in l_tab[c]]
        want = [x / sum(e) for x in e]
        assert _first_marginal(blocks[c], V) == pytest.approx(want, abs=1e-12)


def test_exactness_toy_vocab_gamma1():
    # V=18 toy tables: the emitted token follows p(.|ctx) exactly
    p_tab, _, q_tab = synthetic.toy_tables()
    V = p_tab.shape[1]
    for c in [0, 7]:
        d = markov_block_distribution(oracle.verify, p_tab, q_tab, c, 1)
        assert _first_marginal(d, V) == pytest.approx(p_tab[c], abs=1e-12)


def test_acceptance_rate_is_overlap():
    # P(first position survives) = beta = sum min(p, q)
    g = synthetic.rng(7, 0)
    V = 4
    p_tab = g.dirichlet(np.ones(V), size=V + 1)
    q_tab = g.dirichlet(np.ones(V), size=V + 1)
    for c in range(V + 1):
        d = markov_block_distribution(oracle.verify, p_tab, q_tab, c, 1)
        survive = sum(pr for toks, pr in d.items() if len(toks) == 2)
        beta = sum(min(a, b) for a, b in zip(p_tab[c], q_tab[c]))
        assert survive == pytest.approx(beta, abs=1e-12)


def test_expected_tokens_closed_form_constant_beta():
    # identical rows in every context make beta constant; then
    # E[#tokens per block] = (1 - beta^(gamma+1)) / (1 - beta)
    g = synthetic.rng(8, 0)
    V, gamma = 3, 3
    p_row = g.dirichlet(np.ones(V))
    q_row = g.dirichlet(np.ones(V))
    p_tab = np.tile(p_row, (V + 1, 1))
    q_tab = np.tile(q_row, (V + 1, 1))
    d = markov_block_distribution(oracle.verify, p_tab, q_tab, 0, gamma)
    mean = sum(len(toks) * pr for toks, pr in d.items())
    beta = float(np.minimum(p_row, q_row).sum())
    assert mean == pytest.approx((1 - beta ** (gamma + 1)) / (1 - beta), abs=1e-11)


def test_identical_distributions_accept_everything():
    # glossary: if the two distributions coincide every proposal is accepted
    g = synthetic.rng(9, 0)
    V, gamma = 5, 4
    p = g.dirichlet(np.ones(V))
    logits = np.log(np.tile(p, (1, gamma + 1, 1)))
    q = np.tile(p, (1, gamma, 1))
    r = oracle.verify(logits, q, np.arange(V), np.array([[0, 1, 2, 3]]),
                      np.full((1, gamma), 0.999), np.full((1, gamma + 1), 0.5))
    assert int(r.num_accepted[0]) == gamma


def test_bad_inputs_raise():
    V = 4
    logits = np.zeros((1, 2, V))
    q = np.array([[[0.5, 0.5, 0.0]]])
    inv = np.array([0, 1, 2, -1], dtype=np.int32)
    u1, u2 = np.zeros((1, 1)), np.zeros((1, 2))
    with pytest.raises(oracle.BadInput):      # q(x) = 0 at a drafted token
        oracle.verify(logits, q, inv, np.array([[2]]), u1, u2)
    with pytest.raises(oracle.BadInput):      # drafted token not trimmed
        oracle.verify(logits, q, inv, np.array([[3]]), u1, u2)
    with pytest.raises(oracle.BadInput):      # out of range
        oracle.verify(logits, q, inv, np.array([[4]]), u1, u2)
    bad = logits.copy()
    bad[0, 1, 2] = np.nan
    with pytest.raises(oracle.BadInput):      # non-finite logits
        oracle.verify(bad, q, inv, np.array([[0]]), u1, u2)


def _toy_chain(steps, gamma=4, seed=11):
    """Run the toy chain through the oracle: returns transition counts."""
    p_tab, _, q_tab = synthetic.toy_tables()
    V = p_tab.shape[1]
    g = synthetic.rng(seed, 0)
    ua = synthetic.uniforms(seed, 1, (steps, gamma))
    ur = synthetic.uniforms(seed, 2, (steps, gamma + 1))
    logp = np.log(p_tab)
    inv_map = np.arange(V, dtype=np.int32)
    counts = np.zeros((V + 1, V), dtype=np.int64)
    ctx = 0
    for s in range(steps):
        draft = synthetic.toy_drafts(g, q_tab, ctx, gamma)
        ctxs = [ctx] + [int(d) + 1 for d in draft]
        logits = logp[ctxs][None]
        q = q_tab[ctxs[:gamma]][None]
        r = oracle.verify(logits, q, inv_map, draft[None], ua[s:s + 1], ur[s:s + 1])
        n = int(r.num_accepted[0])
        for t in r.tokens[0, : n + 1]:
            counts[ctx, t] += 1
            ctx = int(t) + 1
    return counts, p_tab


def _chi2_pvalue(counts, p_tab):
    stat, dof = 0.0, 0
    for c in range(counts.shape[0]):
        n = counts[c].sum()
        if n == 0:
            continue
        e = n * p_tab[c]
        stat += float(((counts[c] - e) ** 2 / e).sum())
        dof += counts.shape[1] - 1
    return stats.chi2.sf(stat, dof)


def test_toy_chain_chi_square():
    counts, p_tab = _toy_chain(20_000)
    assert _chi2_pvalue(counts, p_tab) > 1e-3


def test_toy_chain_chi_square_rejects_naive_redraw(monkeypatch):
    monkeypatch.setattr(spec, "residual_weights", lambda p, q: np.asarray(p, dtype=np.float64))
    counts, p_tab = _toy_chain(20_000)
    assert _chi2_pvalue(counts, p_tab) < 1e-6


def test_toy_expectations_match_enumeration():
    # bench.toy_expectations (beta per context and the expected tokens per
    # block of the Markov toy) against the exact block distribution obtained by
    # enumerating every draft and integrating oracle.verify over its uniforms
    import bench
    for V, gamma, seed in [(3, 2, 5), (4, 3, 6)]:
        p_tab, _, q_tab = synthetic.toy_tables(V=V, w=0.4, seed=seed)
        beta, etok = bench.toy_expectations(p_tab, q_tab, gamma)
        for c in range(V + 1):
            d1 = markov_block_distribution(oracle.verify, p_tab, q_tab, c, 1)
            acc1 = sum(pr for toks, pr in d1.items() if len(toks) == 2)
            assert beta[c] == pytest.approx(acc1, abs=1e-12)
            d = markov_block_distribution(oracle.verify, p_tab, q_tab, c, gamma)
            assert etok[c] == pytest.approx(sum(pr * len(t) for t, pr in d.items()), abs=1e-12)
