"""Pins of the draft-tree oracle (oracle/tree.py).

* a chain is a tree: verify_tree_greedy on parent[i] = i - 1 must equal the
  (independently pinned) linear greedy verification;
* the deepest accepted path can be no shorter than what any root-to-leaf
  chain of the tree would accept on its own (brute force over the chains),
  and no longer;
* lossless: tree speculative decoding on the toy tables, with trees grown
  from the toy drafter's top-2 at each node, emits exactly the target's own
  greedy stream (VocabTrim section 4: greedy target, lossless);
* the drafter's top-k are the k best trimmed logits in order, with
  exp(log q) equal to the pinned draft_step's q.
"""
import numpy as np
import pytest

import oracle
from oracle.tree import draft_topk, verify_tree_greedy
import synthetic


def _bf16_exact(a):
    return (np.asarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def test_a_chain_is_the_linear_greedy_block():
    g = synthetic.rng(3, 0)
    B, N, V = 30, 6, 50
    L = np.stack([np.stack([g.permutation(V) * 0.25 for _ in range(N + 1)]) for _ in range(B)])
    choice = L.argmax(axis=2)
    draft = g.integers(0, V, (B, N))
    cut = g.integers(0, N + 1, B)
    for b in range(B):
        draft[b, :cut[b]] = choice[b, :cut[b]]
    chain = np.arange(-1, N - 1)
    t = verify_tree_greedy(L, chain, draft)
    r = oracle.verify_greedy(L.astype(np.float32), draft.astype(np.int32))
    assert np.array_equal(t.tokens, r.tokens)
    assert np.array_equal(t.num_accepted, r.num_accepted)
    for b in range(B):
        assert t.path[b, :t.num_accepted[b]].tolist() == list(range(t.num_accepted[b]))


def test_hand_worked_tree():
    # context -> node 0 (token 3) and node 1 (token 5); node 0 -> node 2
    # (token 1); node 1 -> node 3 (token 2).  Target choices by row:
    # row 0 (context): 5, row 1 (after node 0): 1, row 2 (after node 1): 2,
    # row 3 (after node 2): 0, row 4 (after node 3): 4
    V = 6
    L = np.full((1, 5, V), -1.0)
    for r, c in enumerate([5, 1, 2, 0, 4]):
        L[0, r, c] = 1.0
    parent = [-1, -1, 0, 1]
    tokens = [[3, 5, 1, 2]]
    t = verify_tree_greedy(L, parent, tokens)
    # node 0 fails (3 != 5); node 1 accepted; node 3 accepted (2 == choice of row 2)
    assert t.num_accepted.tolist() == [2]
    assert t.path[0, :2].tolist() == [1, 3]
    assert t.tokens[0].tolist() == [5, 2, 4, -1, -1]


def test_equal_depth_goes_to_the_lower_node():
    # siblings 0 and 1 carry the same token: both are accepted at depth 1;
    # the lower node wins, so the bonus comes from row 1, not row 2
    V = 4
    L = np.full((1, 3, V), 0.0)
    L[0, 0, 2] = 1.0      # context: 2
    L[0, 1, 3] = 1.0      # after node 0: 3
    L[0, 2, 1] = 1.0      # after node 1: 1
    t = verify_tree_greedy(L, [-1, -1], [[2, 2]])
    assert t.path[0].tolist() == [0, -1] and t.tokens[0].tolist() == [2, 3, -1]


def test_deepest_path_matches_the_best_chain():
    g = synthetic.rng(4, 0)
    for trial in range(300):
        N, V = int(g.integers(1, 12)), 4
        parent = [-1] + [int(g.integers(-1, i)) for i in range(1, N)]
        L = g.integers(0, 3, (1, N + 1, V)).astype(np.float64)   # small ints: many ties
        tokens = g.integers(0, V, (1, N))
        t = verify_tree_greedy(L, parent, tokens)
        # every root-to-node chain verified on its own
        best = 0
        for leaf in range(N):
            chain = []
            i = leaf
            while i >= 0:
                chain.append(i)
                i = parent[i]
            chain.reverse()
            rows = [0] + [c + 1 for c in chain]
            Lc = L[:, rows, :]
            r = oracle.verify_greedy(Lc.astype(np.float32), tokens[:, chain].astype(np.int32))
            best = max(best, int(r.num_accepted[0]))
        assert t.num_accepted[0] == best
        # the emitted path is a chain of accepted nodes ending in the target's choice
        k = t.num_accepted[0]
        nodes = t.path[0, :k].tolist()
        for a, b_ in zip([-1] + nodes, nodes):
            assert parent[b_] == a
        last_row = nodes[-1] + 1 if nodes else 0
        assert t.tokens[0, k] == t.choice[0, last_row]


@pytest.mark.parametrize("width", [1, 2, 3])
def test_tree_speculative_decoding_is_lossless(width):
    p, _, q_w = synthetic.toy_tables()
    n_tokens, depth = 2000, 3
    ref, c = [], 0
    for _ in range(n_tokens):
        t = oracle.argmax_lowest(np.log(p[c]))
        ref.append(t)
        c = t + 1
    out, c, blocks = [], 0, 0
    while len(out) < n_tokens:
        # grow a tree: every node of depth < 3 takes the toy drafter's `width` best
        parent, tokens, ctx = [], [], []
        frontier = [(-1, c)]
        for _ in range(depth):
            nxt = []
            for node, cc in frontier:
                for t in np.argsort(-q_w[cc], kind="stable")[:width]:
                    parent.append(node)
                    tokens.append(int(t))
                    ctx.append(int(t) + 1)
                    nxt.append((len(tokens) - 1, int(t) + 1))
            frontier = nxt
        rows = [c] + ctx
        L = np.log(p[rows])[None]
        r = verify_tree_greedy(L, np.array(parent), np.array([tokens]))
        n = int(r.num_accepted[0])
        emitted = r.tokens[0, :n + 1].tolist()
        out.extend(emitted)
        c = emitted[-1] + 1
        blocks += 1
    assert out[:n_tokens] == ref
    assert blocks < n_tokens


def test_draft_topk_exact_and_consistent_with_the_softmax():
    h = _bf16_exact([[1.0, 2.0]])
    W = _bf16_exact([[1, 0], [0, 1], [1, 1], [2, -1], [0, 1]])   # z = 1, 2, 3, 0, 2
    trim_ids = np.array([4, 8, 15, 16, 23], np.int32)
    d = draft_topk(h, W, trim_ids, 3)
    assert d["index"].tolist() == [[2, 1, 4]]          # tie 2 = 2 goes to index 1 first
    assert d["ids"].tolist() == [[15, 8, 23]]
    g = synthetic.rng(8, 0)
    h = synthetic.normal_bf16(g, (5, 32), 1.0)
    W = synthetic.normal_bf16(g, (300, 32), 0.3)
    trim_ids = np.arange(300, dtype=np.int32)
    for T in (1.0, 0.7):
        d = draft_topk(h, W, trim_ids, 8, T)
        s = oracle.draft_step(h, W, trim_ids, np.zeros(5, np.float32), T)
        for b in range(5):
            assert np.allclose(np.exp(d["logq"][b]), s["q"][b, d["index"][b]], rtol=1e-12)
            assert (np.diff(d["logits"][b, d["index"][b]]) <= 0).all()
    one = draft_topk(h, W, trim_ids, 1)
    assert np.array_equal(one["index"][:, 0], oracle.draft_step_greedy(h, W, trim_ids)["index"])
