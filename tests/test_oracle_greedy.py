"""Pins of the greedy (temperature 0) oracle.

* VocabTrim, section 4: with a greedily decoding target a drafted token is
  accepted only if it equals the target's own choice, which keeps the
  generation lossless -- chained greedy speculative decoding must emit
  exactly the target's own greedy stream, whatever the drafter proposes.
* Algorithm 2 (Appendix C.1): left to right, the first inconsistent token
  is replaced by the target's token and the block ends.
* the limit of the stochastic rule: at a vanishing temperature p and q are
  one-hot, so the (independently pinned) stochastic verify must agree with
  the greedy one for any uniforms in (0, 1).
"""
import numpy as np
import pytest

import oracle
import synthetic


def _bf16_exact(a):
    # small integers and halves are exact in bf16: keep the top 16 bits
    return (np.asarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)


# ------------------------------------------------------------------ argmax
def test_argmax_ties_go_to_the_lower_index():
    assert oracle.argmax_lowest([1.0, 3.0, 3.0, 2.0]) == 1
    assert oracle.argmax_lowest([7.0]) == 0
    assert oracle.argmax_lowest([-2.0, -2.0, -5.0]) == 0
    assert oracle.argmax_lowest([0.0, -1.0, 0.5, 0.5]) == 2


def test_argmax_matches_numpy_on_distinct_values():
    g = synthetic.rng(123, 0)
    for _ in range(50):
        x = g.permutation(1000).astype(np.float64) * 0.5 - 100
        assert oracle.argmax_lowest(x) == int(np.argmax(x))


def test_top2_gap():
    assert oracle.top2_gap([1.0, 4.0, 2.5]) == 1.5
    assert oracle.top2_gap([3.0, 3.0]) == 0.0


def test_argmax_rejects_non_finite():
    with pytest.raises(oracle.BadInput):
        oracle.argmax_lowest([0.0, np.nan])


# ----------------------------------------------------------------- drafting
def test_draft_greedy_exact_dot_products():
    # z = h . W_trim[j] by hand: h = (1, 2); rows (1,0), (0,1), (1,1), (2,-1)
    h = _bf16_exact([[1.0, 2.0], [1.0, 1.0]])
    W = _bf16_exact([[1, 0], [0, 1], [1, 1], [2, -1]])
    trim_ids = np.array([5, 9, 12, 40], np.int32)
    d = oracle.draft_step_greedy(h, W, trim_ids)
    assert np.array_equal(d["logits"], [[1, 2, 3, 0], [1, 1, 2, 1]])
    assert list(d["index"]) == [2, 2] and list(d["tokens"]) == [12, 12]
    assert np.array_equal(d["q"], [[0, 0, 1, 0], [0, 0, 1, 0]])
    # a tie between trimmed rows 0 and 1 goes to row 0 (the lower target id)
    d = oracle.draft_step_greedy(_bf16_exact([[1.0, 1.0]]), _bf16_exact([[2, 0], [0, 2], [1, 0]]),
                                 trim_ids[:3])
    assert list(d["index"]) == [0] and list(d["tokens"]) == [5] and d["gap"][0] == 0.0


def test_draft_greedy_is_the_vanishing_temperature_draw():
    g = synthetic.rng(7, 0)
    B, H, K = 6, 8, 50
    h = _bf16_exact(g.integers(-3, 4, (B, H)))
    W = _bf16_exact(g.integers(-3, 4, (K, H)))
    trim_ids = np.sort(g.choice(1000, K, replace=False)).astype(np.int32)
    d = oracle.draft_step_greedy(h, W, trim_ids)
    keep = d["gap"] >= 1.0  # integer logits: a unit gap makes the limit one-hot
    assert keep.any()
    for u in [1e-6, 0.3, 0.999999]:
        s = oracle.draft_step(h, W, trim_ids, np.full(B, u, np.float32), 1e-3)
        assert np.array_equal(s["tokens"][keep], d["tokens"][keep])


# ------------------------------------------------------------ verification
def test_verify_greedy_hand_worked_blocks():
    # V = 4, gamma = 3; target choices per position: 2, 0, 3, 1
    l = np.array([[0, 1, 5, 2], [4, 1, 1, 0], [0, 0, 1, 3], [0, 2, 1, 1]], np.float32)
    L = np.stack([l, l, l, l])
    drafts = np.array([[2, 0, 3], [2, 0, 1], [1, 0, 3], [2, 3, 3]], np.int32)
    r = oracle.verify_greedy(L, drafts)
    assert list(r.num_accepted) == [3, 2, 0, 1]
    assert r.tokens.tolist() == [[2, 0, 3, 1], [2, 0, 3, -1], [2, -1, -1, -1], [2, 0, -1, -1]]
    assert np.array_equal(r.accept[1], [1, 1, 0]) and np.isnan(r.accept[2, 1:]).all()
    assert r.choice[0].tolist() == [2, 0, 3, 1]


def test_verify_greedy_tie_in_the_target_row():
    L = np.array([[[3, 3, 1], [0, 5, 5]]], np.float32)  # gamma = 1
    assert oracle.verify_greedy(L, np.array([[1]], np.int32)).tokens.tolist() == [[0, -1]]
    assert oracle.verify_greedy(L, np.array([[0]], np.int32)).tokens.tolist() == [[0, 1]]


def test_verify_greedy_bf16_logits():
    l = np.array([[[0.5, 2.0, -1.0], [1.0, 0.0, 3.0]]], np.float32)
    r = oracle.verify_greedy(_bf16_exact(l).reshape(1, 2, 3), np.array([[1]], np.int32),
                             logits_dtype="bf16")
    assert r.tokens.tolist() == [[1, 2]]


def test_verify_greedy_rejects_out_of_range_drafts():
    with pytest.raises(oracle.BadInput):
        oracle.verify_greedy(np.zeros((1, 2, 3), np.float32), np.array([[3]], np.int32))


@pytest.mark.parametrize("gamma", [1, 4])
@pytest.mark.parametrize("drafter", ["greedy", "sampled"])
def test_greedy_speculative_decoding_is_lossless(gamma, drafter):
    # toy target p(. | previous token) over 18 tokens, toy drafter q_w; the
    # emitted stream must equal the target's own greedy stream token by token
    p, _, q_w = synthetic.toy_tables()
    V = p.shape[1]
    g = synthetic.rng(31, gamma)
    n_tokens = 3000
    ref, c = [], 0
    for _ in range(n_tokens):
        t = oracle.argmax_lowest(np.log(p[c]))
        ref.append(t)
        c = t + 1
    out, c, blocks, accepted = [], 0, 0, 0
    while len(out) < n_tokens:
        if drafter == "greedy":
            x, cc = [], c
            for _ in range(gamma):
                x.append(oracle.argmax_lowest(q_w[cc]))
                cc = x[-1] + 1
            x = np.array(x, np.int32)
        else:
            x = synthetic.toy_drafts(g, q_w, c, gamma)
        ctx = [c] + [int(t) + 1 for t in x]
        L = np.log(p[ctx])[None].astype(np.float64)
        r = oracle.verify_greedy(L, x[None])
        n = int(r.num_accepted[0])
        emitted = r.tokens[0, : n + 1].tolist()
        out.extend(emitted)
        c = emitted[-1] + 1
        blocks += 1
        accepted += n
    assert out[:n_tokens] == ref
    assert blocks < n_tokens  # some drafted tokens were accepted
    assert 0 <= accepted <= blocks * gamma


def test_verify_greedy_is_the_vanishing_temperature_limit():
    # distinct logits (gaps >= 0.5), one-hot q at the drafted token: the
    # stochastic rule at T = 1e-3 must give the greedy block for any uniforms
    g = synthetic.rng(77, 0)
    B, gamma, V = 40, 5, 30
    L = np.stack([np.stack([g.permutation(V) * 0.5 for _ in range(gamma + 1)]) for _ in range(B)])
    choice = L.argmax(axis=2)
    # drafts: the target's choice for a random prefix, then something else
    drafts = choice[:, :gamma].copy()
    cut = g.integers(0, gamma + 1, B)
    for b in range(B):
        if cut[b] < gamma:
            drafts[b, cut[b]] = (choice[b, cut[b]] + 1 + g.integers(0, V - 1)) % V
    inv_map = np.arange(V, dtype=np.int32)
    q = np.zeros((B, gamma, V))
    for b in range(B):
        q[b, np.arange(gamma), drafts[b]] = 1.0
    gr = oracle.verify_greedy(L.astype(np.float32), drafts)
    assert np.array_equal(gr.num_accepted, np.minimum(cut, gamma))
    for seed in range(3):
        u_a = synthetic.uniforms(seed, 1, (B, gamma)).astype(np.float64)
        u_r = synthetic.uniforms(seed, 2, (B, gamma + 1)).astype(np.float64)
        u_a = np.clip(u_a, 1e-7, None)
        u_r = np.clip(u_r, 1e-7, None)
        st = oracle.verify(L, q, inv_map, drafts, u_a, u_r, temperature=1e-3)
        assert np.array_equal(st.num_accepted, gr.num_accepted)
        assert np.array_equal(st.tokens, gr.tokens)
