"""Greedy (temperature 0) drafting and verification through the C ABI
against the oracle (oracle/greedy.py).

Verification compares the logits exactly as given, so its outputs must be
bit-identical to the oracle's.  Drafting decides an argmax over fp32
projections: rows whose oracle top-2 gap is within the logit tolerance may
pick either near-maximal index; the GPU's pick must then be one of them.
"""
import numpy as np
import pytest

import oracle
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


def _bf(a):
    return _dev(np.ascontiguousarray(a).view(np.int16))


def _bf16_exact(a):
    return (np.asarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)


# ------------------------------------------------------------------ drafting
def _check_greedy_draft(vt, hidden, W, trim_ids, exact_inputs=False):
    B, K = hidden.shape[0], W.shape[0]
    q, tok, st = vt.vt_draft_step(_bf(hidden), _bf(W), _dev(trim_ids), None, 0.0)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    q, tok = q.cpu().numpy(), tok.cpu().numpy()
    ref = oracle.draft_step_greedy(hidden, W, trim_ids)
    z = ref["logits"]
    exact = 0
    for b in range(B):
        j = int(np.flatnonzero(q[b])[0]) if q[b].any() else -1
        assert q[b].sum() == 1.0 and q[b, j] == 1.0, b          # one-hot
        assert tok[b] == trim_ids[j], b
        tol = 1e-3 * max(abs(z[b]).max(), np.sqrt((z[b] ** 2).mean()))
        if exact_inputs or ref["gap"][b] > tol:
            # exact projections (integer inputs) must also break ties the same way
            assert j == ref["index"][b], (b, j, ref["index"][b], ref["gap"][b])
            exact += 1
        else:
            assert z[b, j] >= z[b].max() - tol, (b, j)        # a near-maximal index
    return exact


@pytest.mark.parametrize("B,H,K", [(1, 64, 128), (5, 200, 1000), (16, 2048, 4096),
                                   (33, 96, 777), (64, 512, 2000),
                                   (100, 520, 3001),     # two 128-row tiles per CTA
                                   (256, 128, 1300),     # padded batch 256
                                   (200, 96, 12345),     # three passes per finalize CTA
                                   (300, 64, 2000)])     # B > 256: the CUDA-core projection
def test_greedy_draft_integer_inputs_bit_exact(vt, B, H, K):
    # small integers: fp32 accumulation is exact, so the argmax is too
    g = synthetic.rng(B + H + K, 3)
    hidden = _bf16_exact(g.integers(-2, 3, (B, H)))
    W = _bf16_exact(g.integers(-2, 3, (K, H)))
    W[K // 2] = W[K // 3]                     # duplicated rows: a tie at the lower index
    trim_ids = np.sort(g.permutation(3 * K)[:K]).astype(np.int32)
    assert _check_greedy_draft(vt, hidden, W, trim_ids, exact_inputs=True) == B


def test_greedy_draft_ties_go_to_the_lower_index(vt):
    # every row of W equal: every index ties, index 0 wins
    B, H, K = 4, 64, 3000
    hidden = _bf16_exact(np.ones((B, H)))
    W = _bf16_exact(np.ones((K, H)))
    trim_ids = np.arange(K, dtype=np.int32) * 2
    q, tok, st = vt.vt_draft_step(_bf(hidden), _bf(W), _dev(trim_ids), None, 0.0)
    torch.cuda.synchronize()
    assert tok.cpu().tolist() == [0] * B
    assert (q.cpu().numpy()[:, 0] == 1).all() and q.cpu().numpy()[:, 1:].sum() == 0


@pytest.mark.parametrize("B", [1, 16, 64])
def test_greedy_draft_full_size(vt, B):
    # the drafting workload: hidden N(0,1), W_trim N(0,0.02) [32768, 2048]
    g = synthetic.rng(B, 44)
    hidden = synthetic.normal_bf16(g, (B, 2048), 1.0)
    W = synthetic.normal_bf16(g, (32768, 2048), 0.02)
    trim_ids = np.sort(g.permutation(128256)[:32768]).astype(np.int32)
    assert _check_greedy_draft(vt, hidden, W, trim_ids) >= B - 1


def test_greedy_draft_cuda_core_path(vt):
    # H not a multiple of 8: the CUDA-core projection
    g = synthetic.rng(5, 45)
    hidden = synthetic.normal_bf16(g, (7, 300), 1.0)
    W = synthetic.normal_bf16(g, (5000, 300), 0.02)
    trim_ids = np.arange(5000, dtype=np.int32)
    assert _check_greedy_draft(vt, hidden, W, trim_ids) >= 6


def test_greedy_draft_non_finite_sets_status(vt):
    g = synthetic.rng(6, 46)
    hidden = synthetic.normal_bf16(g, (3, 64), 1.0)
    hidden[1, 5] = 0x7fc0                     # NaN
    W = synthetic.normal_bf16(g, (500, 64), 0.02)
    q, tok, st = vt.vt_draft_step(_bf(hidden), _bf(W), _dev(np.arange(500, dtype=np.int32)),
                                  None, 0.0)
    torch.cuda.synchronize()
    assert int(st.item()) & vt.VT_DEV_NONFINITE
    assert int(tok[1].item()) == -1 and int(tok[0].item()) >= 0


# -------------------------------------------------------------- verification
def _greedy_inputs(B, gamma, V, dtype, seed, ties=False):
    g = synthetic.rng(seed, 47)
    if ties:
        logits = g.integers(-3, 4, (B, gamma + 1, V)).astype(np.float32)
    else:
        vi = synthetic.verify_inputs(B=B, gamma=gamma, V=V, K=min(V, 4096), seed=seed)
        logits = vi["logits"].astype(np.float32)
    if dtype == "bf16":
        logits = _bf16_exact(logits)
        vals = oracle.bf16_to_f64(logits)
    else:
        vals = logits.astype(np.float64)
    choice = np.array([[oracle.argmax_lowest(vals[b, i]) for i in range(gamma + 1)]
                       for b in range(B)])
    # drafts: the target's choice for a random prefix, then a mismatch
    draft = g.integers(0, V, (B, gamma)).astype(np.int32)
    cut = g.integers(0, gamma + 1, B)
    for b in range(B):
        draft[b, :cut[b]] = choice[b, :cut[b]]
        if cut[b] < gamma and draft[b, cut[b]] == choice[b, cut[b]]:
            draft[b, cut[b]] = (choice[b, cut[b]] + 1) % V
    return logits, draft, cut


def _run_greedy_verify(vt, logits, draft, dtype, noalloc=False):
    t = _dev(logits.view(np.int16) if dtype == "bf16" else logits)
    if dtype == "bf16":
        t = t.view(torch.bfloat16)
    if not noalloc:
        out, n, acc, st = vt.vt_verify(t, None, None, _dev(draft), None, None, 0.0)
    else:
        from drafter_sampling_gb300 import _lib
        B, R, V = logits.shape
        out = torch.empty((B, R), dtype=torch.int32, device="cuda")
        n = torch.empty(B, dtype=torch.int32, device="cuda")
        acc = torch.empty((B, R - 1), dtype=torch.float32, device="cuda")
        st = torch.empty(1, dtype=torch.int32, device="cuda")
        d = _dev(draft)
        rc = vt.lib().vt_verify_noalloc(t.data_ptr(), 1 if dtype == "bf16" else 0, B, R - 1, V,
                                        None, None, 1, d.data_ptr(), None, None, 0.0,
                                        out.data_ptr(), n.data_ptr(), acc.data_ptr(),
                                        st.data_ptr(), None)
        _lib.check("vt_verify_noalloc", rc)
    torch.cuda.synchronize()
    return out.cpu().numpy(), n.cpu().numpy(), acc.cpu().numpy(), int(st.item())


def _assert_greedy_equal(out, n, acc, ref):
    assert np.array_equal(n, ref.num_accepted)
    assert np.array_equal(out, ref.tokens)
    tested = ~np.isnan(ref.accept)
    assert np.array_equal(acc[tested], ref.accept[tested])
    assert np.isnan(acc[~tested]).all()


@pytest.mark.parametrize("B,gamma,V,dtype,ties", [
    (4, 3, 1000, "f32", False),
    (9, 6, 20011, "bf16", False),           # ragged V, bf16
    (16, 6, 128256, "f32", False),          # the batched-verify workload's sizes
    (6, 64, 3001, "f32", False),            # the largest gamma
    (8, 4, 5000, "f32", True),              # integer logits: ties everywhere
    (5, 2, 4099, "bf16", True),
])
def test_greedy_verify_bit_exact(vt, B, gamma, V, dtype, ties):
    logits, draft, cut = _greedy_inputs(B, gamma, V, dtype, seed=B * V + gamma, ties=ties)
    out, n, acc, st = _run_greedy_verify(vt, logits, draft, dtype)
    assert st == 0
    ref = oracle.verify_greedy(logits, draft, logits_dtype=dtype)
    assert np.array_equal(ref.num_accepted, np.minimum(cut, gamma))
    _assert_greedy_equal(out, n, acc, ref)


def test_greedy_verify_noalloc(vt):
    logits, draft, _ = _greedy_inputs(7, 5, 9000, "f32", seed=3)
    out, n, acc, st = _run_greedy_verify(vt, logits, draft, "f32", noalloc=True)
    assert st == 0
    _assert_greedy_equal(out, n, acc, oracle.verify_greedy(logits, draft))


def test_greedy_verify_large_batch_sampled(vt):
    # B=256, gamma=8, V=152064 bf16 logits; the oracle checks 24 sequences
    B, gamma, V = 256, 8, 152064
    g = synthetic.rng(11, 48)
    logits = _bf16_exact(g.standard_normal((B, gamma + 1, V), dtype=np.float32) * 2)
    draft = g.integers(0, V, (B, gamma)).astype(np.int32)
    cut = g.integers(0, gamma + 1, B)
    for b in range(B):
        for i in range(cut[b]):
            draft[b, i] = oracle.argmax_lowest(oracle.bf16_to_f64(logits[b, i]))
    out, n, acc, st = _run_greedy_verify(vt, logits, draft, "bf16")
    assert st == 0
    for b in synthetic.rng(12, 49).choice(B, 24, replace=False):
        ref = oracle.verify_greedy(logits[b:b + 1], draft[b:b + 1], logits_dtype="bf16")
        _assert_greedy_equal(out[b:b + 1], n[b:b + 1], acc[b:b + 1], ref)


def test_greedy_verify_flags(vt):
    logits, draft, _ = _greedy_inputs(3, 4, 2000, "f32", seed=9)
    # sequence 0: a NaN logit; sequence 1: the first drafted token out of range
    logits[0, 2, 17] = np.nan
    draft[1, 0] = 2000
    out, n, acc, st = _run_greedy_verify(vt, logits, draft, "f32")
    assert st & vt.VT_DEV_NONFINITE and st & vt.VT_DEV_BAD_DRAFT
    assert (out[0] == -1).all() and (out[1] == -1).all() and n[0] == 0 and n[1] == 0
    ref = oracle.verify_greedy(logits[2:], draft[2:])
    _assert_greedy_equal(out[2:], n[2:], acc[2:], ref)


def test_greedy_block_drafter_to_verify(vt):
    # the drafter's greedy tokens verified against logits that agree with
    # them for a prefix: draft -> verify through the library only
    B, H, K, V, gamma = 8, 256, 2048, 6000, 4
    g = synthetic.rng(13, 50)
    trim_ids = np.sort(g.permutation(V)[:K]).astype(np.int32)
    W = synthetic.normal_bf16(g, (K, H), 0.05)
    q_all = torch.empty((B, gamma, K), dtype=torch.float32, device="cuda")
    tok_all = torch.empty((B, gamma), dtype=torch.int32, device="cuda")
    for j in range(gamma):
        hidden = synthetic.normal_bf16(g, (B, H), 1.0)
        vt.vt_draft_step(_bf(hidden), _bf(W), _dev(trim_ids), None, 0.0, q=q_all[:, j, :],
                         tokens=tok_all[:, j])
    torch.cuda.synchronize()
    draft = tok_all.cpu().numpy()
    logits = g.normal(0, 1, (B, gamma + 1, V)).astype(np.float32)
    cut = g.integers(0, gamma + 1, B)
    for b in range(B):
        for i in range(cut[b]):
            logits[b, i, draft[b, i]] = 100.0      # the target agrees up to the cut
    out, n, acc, st = _run_greedy_verify(vt, logits, draft, "f32")
    assert st == 0
    assert np.array_equal(n, cut)
    _assert_greedy_equal(out, n, acc, oracle.verify_greedy(logits, draft))
