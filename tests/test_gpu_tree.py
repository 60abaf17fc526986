"""Draft trees on the GPU (through the C ABI) against oracle/tree.py:
greedy tree verification bit-exact, the drafter's top-k exact on integer
inputs and within the logit tolerance at full size, and one EAGLE-style
tree (depth 3, top-8 expansion of the best nodes, 32 tokens) grown with
vt_draft_topk and verified with vt_verify_tree."""
import numpy as np
import pytest

import oracle
from oracle.tree import draft_topk, verify_tree_greedy
import synthetic

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def vt():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import drafter_sampling_gb300 as m
    from drafter_sampling_gb300 import build
    build.build()
    m.lib()
    return m


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _bf16_exact(a):
    return (np.asarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _random_tree(g, N):
    return np.array([-1] + [int(g.integers(-1, i)) for i in range(1, N)], np.int32)


def _tree_inputs(B, N, V, seed, dtype="f32", shared=False, ties=False):
    g = synthetic.rng(seed, 70)
    if ties:
        logits = g.integers(-2, 3, (B, N + 1, V)).astype(np.float32)
    else:
        logits = (g.standard_normal((B, N + 1, V), dtype=np.float32) * 2)
    if dtype == "bf16":
        logits = _bf16_exact(logits)
        vals = oracle.bf16_to_f64(logits)
    else:
        vals = logits.astype(np.float64)
    parent = _random_tree(g, N) if shared else np.stack([_random_tree(g, N) for _ in range(B)])
    tokens = g.integers(0, V, (B, N)).astype(np.int32)
    # make a random subset of nodes agree with the target at their parent's row
    for b in range(B):
        par = parent if shared else parent[b]
        for i in range(N):
            if g.random() < 0.6:
                tokens[b, i] = int(np.argmax(vals[b, par[i] + 1]))
    return logits, parent, tokens


def _run(vt, logits, parent, tokens, dtype):
    t = _dev(logits.view(np.int16) if dtype == "bf16" else logits)
    if dtype == "bf16":
        t = t.view(torch.bfloat16)
    out, n, path, st = vt.vt_verify_tree(t, _dev(parent), _dev(tokens))
    torch.cuda.synchronize()
    return out.cpu().numpy(), n.cpu().numpy(), path.cpu().numpy(), int(st.item())


@pytest.mark.parametrize("B,N,V,dtype,shared,ties", [
    (8, 32, 20011, "f32", True, False),        # one 32-node tree for all sequences
    (6, 60, 128256, "bf16", False, False),     # per-sequence trees, a 128K vocabulary
    (16, 7, 3000, "f32", False, True),         # integer logits: ties
    (3, 255, 1000, "f32", False, False),       # the largest tree
])
def test_tree_verify_bit_exact(vt, B, N, V, dtype, shared, ties):
    logits, parent, tokens = _tree_inputs(B, N, V, seed=B + N + V, dtype=dtype, shared=shared,
                                          ties=ties)
    out, n, path, st = _run(vt, logits, parent, tokens, dtype)
    assert st == 0
    ref = verify_tree_greedy(logits, parent, tokens, logits_dtype=dtype)
    assert np.array_equal(n, ref.num_accepted)
    assert np.array_equal(out, ref.tokens)
    assert np.array_equal(path, ref.path)
    assert ref.num_accepted.max() >= 1


def test_a_chain_tree_equals_linear_greedy_verify(vt):
    B, N, V = 8, 6, 9000
    logits, _, tokens = _tree_inputs(B, N, V, seed=5, shared=True)
    chain = np.arange(-1, N - 1, dtype=np.int32)
    out, n, _, st = _run(vt, logits, chain, tokens, "f32")
    o2, n2, _, st2 = vt.vt_verify(_dev(logits), None, None, _dev(tokens), None, None, 0.0)
    torch.cuda.synchronize()
    assert st == 0 and int(st2.item()) == 0
    assert np.array_equal(out, o2.cpu().numpy()) and np.array_equal(n, n2.cpu().numpy())


def test_tree_flags(vt):
    logits, parent, tokens = _tree_inputs(4, 5, 500, seed=6)
    parent[1, 3] = 3          # a node that is its own parent
    tokens[2, 0] = 500        # out of range
    logits[3, 0, 9] = np.inf
    out, n, path, st = _run(vt, logits, parent, tokens, "f32")
    assert st & vt.VT_DEV_BAD_DRAFT and st & vt.VT_DEV_NONFINITE
    for b in (1, 2, 3):
        assert (out[b] == -1).all() and n[b] == 0
    ref = verify_tree_greedy(logits[:1], parent[:1], tokens[:1])
    assert np.array_equal(out[:1], ref.tokens)


def test_sampling_trees_are_unsupported(vt):
    logits, parent, tokens = _tree_inputs(1, 3, 100, seed=7)
    with pytest.raises(vt.VtError):
        t = _dev(logits)
        vt.vt_verify_tree(t, _dev(parent), _dev(tokens), temperature=1.0)


# ------------------------------------------------------------------ top-k
@pytest.mark.parametrize("B,H,K,k", [
    (5, 64, 1000, 8), (16, 96, 4096, 32), (1, 32, 40, 1),
    (4, 64, 9000, 5),        # three CTAs per row
    (3, 64, 70001, 12),      # eight CTAs per row, several passes, a ragged tail
    (2, 32, 40000, 32),      # the longest lists
])
def test_topk_integer_inputs_exact(vt, B, H, K, k):
    g = synthetic.rng(B + K, 71)
    hidden = _bf16_exact(g.integers(-2, 3, (B, H)))
    W = _bf16_exact(g.integers(-2, 3, (K, H)))
    trim_ids = np.sort(g.permutation(3 * K)[:K]).astype(np.int32)
    ids, logq, st = vt.vt_draft_topk(_dev(hidden.view(np.int16)), _dev(W.view(np.int16)),
                                     _dev(trim_ids), k, 0.8)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = draft_topk(hidden, W, trim_ids, k, 0.8)
    assert np.array_equal(ids.cpu().numpy(), ref["ids"])
    err = np.abs(logq.cpu().numpy() - ref["logq"])
    assert (err <= 1e-3 * np.maximum(1.0, np.abs(ref["logq"]))).all()


def test_topk_full_size(vt):
    g = synthetic.rng(2, 72)
    B, H, K, k = 16, 2048, 32768, 8
    hidden = synthetic.normal_bf16(g, (B, H), 1.0)
    W = synthetic.normal_bf16(g, (K, H), 0.02)
    trim_ids = np.sort(g.permutation(128256)[:K]).astype(np.int32)
    ids, logq, st = vt.vt_draft_topk(_dev(hidden.view(np.int16)), _dev(W.view(np.int16)),
                                     _dev(trim_ids), k, 1.0)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = draft_topk(hidden, W, trim_ids, k + 4, 1.0)
    z = ref["logits"]
    pos = {int(t): j for j, t in enumerate(trim_ids)}
    ids = ids.cpu().numpy()
    for b in range(B):
        tol = 1e-3 * max(np.abs(z[b]).max(), np.sqrt((z[b] ** 2).mean()))
        got = [pos[int(t)] for t in ids[b]]
        # every pick lies within tolerance of the oracle's value at that rank,
        # and the picks are distinct and in descending order of z
        assert len(set(got)) == k
        for r, j in enumerate(got):
            assert abs(z[b, j] - z[b, ref["index"][b, r]]) <= 2 * tol, (b, r)
        exact = [r for r in range(k) if z[b, ref["index"][b, r]] - z[b, ref["index"][b, r + 1]] > 2 * tol
                 and (r == 0 or z[b, ref["index"][b, r - 1]] - z[b, ref["index"][b, r]] > 2 * tol)]
        for r in exact:
            assert got[r] == ref["index"][b, r], (b, r)


def test_an_eagle_style_tree_end_to_end(vt):
    # depth 3: expand the context with top-8, then the best 4 nodes of each
    # depth with top-4, keeping at most 32 nodes; verify on target logits that
    # agree with one branch
    g = synthetic.rng(3, 73)
    B, H, K, V = 4, 128, 2048, 6000
    W = synthetic.normal_bf16(g, (K, H), 0.1)
    trim_ids = np.sort(g.permutation(V)[:K]).astype(np.int32)
    d_W, d_ids = _dev(W.view(np.int16)), _dev(trim_ids)
    parent, tokens, score = [[] for _ in range(B)], [[] for _ in range(B)], [[] for _ in range(B)]
    frontier = [[(-1, 0.0)] for _ in range(B)]
    for depth, width in [(1, 8), (2, 4), (3, 4)]:
        for b in range(B):
            frontier[b] = sorted(frontier[b], key=lambda x: -x[1])[: (1 if depth == 1 else 4)]
        nxt = [[] for _ in range(B)]
        for slot in range(max(len(f) for f in frontier)):
            hidden = synthetic.normal_bf16(g, (B, H), 1.0)
            ids, logq, st = vt.vt_draft_topk(_dev(hidden.view(np.int16)), d_W, d_ids, width, 1.0)
            ids, logq = ids.cpu().numpy(), logq.cpu().numpy()
            for b in range(B):
                if slot >= len(frontier[b]):
                    continue
                node, sc = frontier[b][slot]
                for r in range(width):
                    if len(tokens[b]) >= 32:
                        break
                    parent[b].append(node)
                    tokens[b].append(int(ids[b, r]))
                    score[b].append(sc + float(logq[b, r]))
                    nxt[b].append((len(tokens[b]) - 1, score[b][-1]))
        frontier = nxt
    N = min(len(t) for t in tokens)
    par = np.array([p[:N] for p in parent], np.int32)
    tok = np.array([t[:N] for t in tokens], np.int32)
    logits = g.standard_normal((B, N + 1, V)).astype(np.float32)
    for b in range(B):           # the target agrees with node path 0 -> child -> grandchild
        i = 0
        logits[b, 0, tok[b, 0]] = 50.0
        kids = [j for j in range(N) if par[b, j] == i]
        if kids:
            logits[b, i + 1, tok[b, kids[0]]] = 50.0
    out, n, path, st = _run(vt, logits, par, tok, "f32")
    assert st == 0
    ref = verify_tree_greedy(logits, par, tok)
    assert np.array_equal(out, ref.tokens) and np.array_equal(n, ref.num_accepted)
    assert (n >= 1).all()


def test_topk_non_finite_row_is_flagged(vt):
    # a NaN hidden state makes row 1's logits non-finite: its picks are -1
    # with NaN log q and the status flags it; the other rows are unaffected
    g = synthetic.rng(9, 74)
    B, H, K, k = 3, 64, 3000, 8
    hidden = synthetic.normal_bf16(g, (B, H), 1.0).copy()
    hidden[1, 5] = 0x7FC0                      # bf16 NaN
    W = synthetic.normal_bf16(g, (K, H), 0.1)
    trim_ids = np.sort(g.permutation(2 * K)[:K]).astype(np.int32)
    ids, logq, st = vt.vt_draft_topk(_dev(hidden.view(np.int16)), _dev(W.view(np.int16)),
                                     _dev(trim_ids), k, 1.0)
    torch.cuda.synchronize()
    assert int(st.item()) & vt.VT_DEV_NONFINITE
    ids, logq = ids.cpu().numpy(), logq.cpu().numpy()
    assert (ids[1] == -1).all() and np.isnan(logq[1]).all()
    keep = [0, 2]
    ref = draft_topk(hidden[keep], W, trim_ids, k, 1.0)
    assert np.array_equal(ids[keep], ref["ids"])
    err = np.abs(logq[keep] - ref["logq"])
    assert (err <= 1e-3 * np.maximum(1.0, np.abs(ref["logq"]))).all()
