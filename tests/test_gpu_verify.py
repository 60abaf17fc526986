"""vt_verify (CUDA, through the C ABI) against the CPU oracle."""
import json
import os

import numpy as np
import pytest

import oracle
import synthetic
from parity import compare_verify

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


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


def _logits_tensor(d):
    if d["logits_dtype"] == "bf16":
        return _dev(d["logits"].view(np.int16))
    return _dev(d["logits"])


def _run(vt, d, T=1.0, ws=None):
    toks, n, acc, st = vt.vt_verify(_logits_tensor(d), _dev(d["q"]), _dev(d["inv_map"]),
                                    _dev(d["draft"]), _dev(d["u_accept"]),
                                    _dev(d["u_resample"]), T, workspace=ws)
    torch.cuda.synchronize()
    return toks.cpu().numpy(), n.cpu().numpy(), acc.cpu().numpy(), int(st.item())


def _oracle(d, T=1.0):
    return oracle.verify(d["logits"], d["q"], d["inv_map"], d["draft"], d["u_accept"],
                         d["u_resample"], T, logits_dtype=d["logits_dtype"])


def _weights(d, T=1.0):
    """Oracle fp64 weights of the final draw of sequence b at position n."""
    def f(b, n):
        l = d["logits"][b, n]
        l = oracle.bf16_to_f64(l) if d["logits_dtype"] == "bf16" else l
        p = oracle.softmax(l, T)
        gamma = d["q"].shape[1]
        if n == gamma:
            return p, d["u_resample"][b, n]
        qf = np.zeros_like(p)
        present = d["inv_map"] >= 0
        qf[present] = d["q"][b, n, d["inv_map"][present]]
        return oracle.residual_weights(p, qf), d["u_resample"][b, n]
    return f


def test_two_token_example(vt):
    with open(os.path.join(GOLDEN, "two_token.json")) as f:
        g = json.load(f)
    p = np.array(g["p"])
    d = dict(logits=np.log(np.stack([p, p]))[None].astype(np.float32), logits_dtype="f32",
             q=np.array(g["q"], np.float32)[None, None], inv_map=np.arange(2, dtype=np.int32))
    for x, ua, want_n in [(0, 0.74, 1), (0, 0.76, 0), (1, 0.999, 1)]:
        for ur in [0.0, 0.3, 0.9999]:
            d.update(draft=np.array([[x]], np.int32), u_accept=np.array([[ua]], np.float32),
                     u_resample=np.array([[ur, ur]], np.float32))
            toks, n, acc, st = _run(vt, d)
            assert st == 0
            assert int(n[0]) == want_n
            assert acc[0, 0] == pytest.approx(g["acceptance_given_proposal"][x], rel=1e-5)
            if want_n == 0:
                assert list(toks[0]) == [1, -1]      # the residual always returns B
            else:
                assert toks[0, 0] == x


CASES = [
    # B, gamma, V, K, dtype, T, noise
    (3, 3, 5000, 700, "f32", 1.0, 1.0),
    (5, 4, 1003, 97, "f32", 0.7, 1.0),       # V not a multiple of 4: scalar loads
    (4, 2, 4104, 512, "bf16", 0.7, 1.0),
    (2, 5, 777, 777, "bf16", 1.3, 1.0),      # K = V, ragged V
    (1, 1, 64, 1, "f32", 1.0, 1.0),          # K = 1: q is one-hot
    (6, 3, 9000, 9000, "f32", 1.0, 0.0),     # q = p on the full vocabulary
    (8, 6, 20000, 3000, "f32", 1.0, 0.05),   # high acceptance: bonus draws
    (3, 64, 2048, 256, "bf16", 1.0, 0.3),    # the largest gamma
    (2, 2, 262144, 5000, "f32", 1.0, 1.0),   # a large vocabulary: 128 residual tiles
    (2, 3, 200003, 3000, "bf16", 0.9, 1.0),  # a large ragged vocabulary
    (1, 1, 1 << 22, 4096, "f32", 1.0, 1.0),  # the largest vocabulary: 2048 residual tiles
    (40, 3, 50000, 4000, "f32", 1.0, 1.0),   # two residual tiles per finish CTA, one left over
    (300, 3, 70001, 3000, "bf16", 0.8, 0.3),  # 18 and 17 tiles per finish CTA, ragged V
]


@pytest.mark.parametrize("B,gamma,V,K,dt,T,noise", CASES)
def test_parity_small(vt, B, gamma, V, K, dt, T, noise):
    totals = dict(compared=0, excluded_seq=0, excluded_draw=0)
    for seed in range(3):
        d = synthetic.verify_inputs(B=B, gamma=gamma, V=V, K=K, seed=100 + seed,
                                    logits_dtype=dt, noise_std=noise)
        toks, n, acc, st = _run(vt, d, T)
        assert st == 0
        ref = _oracle(d, T)
        s = compare_verify(toks, n, acc, ref, draw_weights=_weights(d, T))
        for k in totals:
            totals[k] += s[k]
    assert totals["compared"] >= 3 * B - 1, totals


def test_parity_batched_verify_full_size(vt):
    # B=16, gamma=6, V=128256, K=32768, fp32 logits (the metric's workload)
    for seed in [1, 2, 3]:
        d = synthetic.verify_inputs(seed=seed)
        toks, n, acc, st = _run(vt, d)
        assert st == 0
        ref = _oracle(d)
        s = compare_verify(toks, n, acc, ref, draw_weights=_weights(d))
        assert s["compared"] >= 15, s


def test_parity_large_batch_bf16_full_size(vt):
    # B=256, gamma=8, V=152064, K=38016, bf16 logits, T=0.7
    d = synthetic.verify_inputs(B=256, gamma=8, V=152064, K=38016, seed=1,
                                logits_dtype="bf16")
    toks, n, acc, st = _run(vt, d, 0.7)
    assert st == 0
    ref = _oracle(d, 0.7)
    s = compare_verify(toks, n, acc, ref, draw_weights=_weights(d, 0.7))
    assert s["compared"] >= 250, s


def test_repeat_calls_same_workspace_are_identical(vt):
    d = synthetic.verify_inputs(B=5, gamma=4, V=30000, K=4000, seed=9)
    ws = torch.empty(vt.workspace_bytes("verify", B=5, gamma=4, V=30000, K=4000),
                     dtype=torch.uint8, device="cuda")
    first = _run(vt, d, ws=ws)
    for _ in range(3):
        again = _run(vt, d, ws=ws)
        assert np.array_equal(first[0], again[0]) and np.array_equal(first[1], again[1])


def test_bad_inputs_set_device_status(vt):
    d = synthetic.verify_inputs(B=4, gamma=3, V=3000, K=300, seed=4)
    # sequence 1: a drafted token outside the trimmed vocabulary
    absent = int(np.nonzero(d["inv_map"] < 0)[0][0])
    d["draft"][1, 0] = absent
    toks, n, acc, st = _run(vt, d)
    assert st & vt.VT_DEV_BAD_DRAFT
    assert int(n[1]) == 0 and np.all(toks[1] == -1)
    # the other sequences are still verified
    ref_d = dict(d)
    ref_d["draft"] = d["draft"].copy()
    keep = [0, 2, 3]
    sub = {k: (v[keep] if isinstance(v, np.ndarray) and v.ndim >= 2 and v.shape[0] == 4 else v)
           for k, v in ref_d.items()}
    ref = _oracle(sub)
    compare_verify(toks[keep], n[keep], acc[keep], ref)
    # q(x) = 0 at a drafted token, and a drafted id out of range
    d2 = synthetic.verify_inputs(B=2, gamma=2, V=3000, K=300, seed=5)
    d2["q"][0, 0, d2["inv_map"][d2["draft"][0, 0]]] = 0.0
    d2["draft"][1, 0] = 3000
    toks, n, acc, st = _run(vt, d2)
    assert st & vt.VT_DEV_BAD_DRAFT
    assert np.all(toks == -1)
    # a NaN logit makes the normaliser non-finite
    d3 = synthetic.verify_inputs(B=2, gamma=2, V=3000, K=300, seed=6)
    d3["logits"][1, 2, 17] = np.nan
    toks, n, acc, st = _run(vt, d3)
    assert st & vt.VT_DEV_NONFINITE
    assert np.all(toks[1] == -1)


def test_toy_chain_exact_and_chi_square(vt):
    """200k chained blocks of the toy (V=18, gamma=4, w=0.5) through the GPU:
    per-block parity with the oracle on the first 20k blocks, a chi-square
    test of every emitted transition against the target chain p, and the
    empirical tokens per block (tau) and acceptance rate (alpha) within 4
    sigma of their exact expectations over the visited contexts."""
    import bench
    from scipy import stats
    steps, gamma, parity_steps = 200_000, 4, 20_000
    p_tab, _, q_tab = synthetic.toy_tables()
    V = p_tab.shape[1]
    logp32 = np.log(p_tab).astype(np.float32)
    q32 = q_tab.astype(np.float32)
    g = synthetic.rng(31, 0)
    ua = synthetic.uniforms(31, 1, (steps, gamma))
    ur = synthetic.uniforms(31, 2, (steps, gamma + 1))
    inv_map = torch.arange(V, dtype=torch.int32, device="cuda")
    logits_t = torch.empty((1, gamma + 1, V), dtype=torch.float32, device="cuda")
    q_t = torch.empty((1, gamma, V), dtype=torch.float32, device="cuda")
    draft_t = torch.empty((1, gamma), dtype=torch.int32, device="cuda")
    ua_t = torch.from_numpy(ua).cuda()
    ur_t = torch.from_numpy(ur).cuda()
    logp_d = torch.from_numpy(logp32).cuda()
    q_d = torch.from_numpy(q32).cuda()
    ws = torch.empty(vt.workspace_bytes("verify", B=1, gamma=gamma, V=V, K=V),
                     dtype=torch.uint8, device="cuda")
    out_t = torch.empty((1, gamma + 1), dtype=torch.int32, device="cuda")
    n_t = torch.empty(1, dtype=torch.int32, device="cuda")
    st_t = torch.empty(1, dtype=torch.int32, device="cuda")
    rec_ctx = np.empty(parity_steps, np.int64)
    rec_draft = np.empty((parity_steps, gamma), np.int32)
    rec_tok = np.empty((parity_steps, gamma + 1), np.int32)
    rec_n = np.empty(parity_steps, np.int32)
    counts = np.zeros((V + 1, V), np.int64)
    beta, etok = bench.toy_expectations(p_tab, q_tab, gamma)
    ns = np.empty(steps, np.int64)
    e_tok = np.empty(steps)
    b_sum = b_var = 0.0
    tested = 0
    ctx = 0
    status = 0
    for s in range(steps):
        draft = synthetic.toy_drafts(g, q_tab, ctx, gamma)
        ctxs = torch.tensor([ctx] + [int(x) + 1 for x in draft], device="cuda")
        logits_t[0].copy_(logp_d[ctxs])
        q_t[0].copy_(q_d[ctxs[:gamma]])
        draft_t[0].copy_(torch.from_numpy(draft))
        vt.vt_verify(logits_t, q_t, inv_map, draft_t, ua_t[s:s + 1], ur_t[s:s + 1], 1.0,
                     out_tokens=out_t, out_num_accepted=n_t, dev_status=st_t, workspace=ws,
                     want_accept_prob=False)
        res = torch.cat([out_t[0], n_t, st_t]).cpu().numpy()
        toks = res[: gamma + 1]
        n = int(res[gamma + 1])
        status |= int(res[gamma + 2])
        ns[s] = n
        e_tok[s] = etok[ctx]
        t = min(n + 1, gamma)
        bb = beta[np.array([ctx] + [int(x) + 1 for x in draft[: t - 1]])]
        b_sum += float(bb.sum())
        b_var += float((bb * (1 - bb)).sum())
        tested += t
        if s < parity_steps:
            rec_ctx[s] = ctx
            rec_draft[s] = draft
            rec_tok[s] = toks
            rec_n[s] = n
        for t in toks[: n + 1]:
            counts[ctx, t] += 1
            ctx = int(t) + 1
    assert status == 0
    # parity on the recorded blocks (the oracle replays each block)
    ctxs = np.concatenate([rec_ctx[:, None], rec_draft.astype(np.int64) + 1], axis=1)
    ref = oracle.verify(logp32[ctxs], q32[ctxs[:, :gamma]], np.arange(V), rec_draft,
                        ua[:parity_steps], ur[:parity_steps], 1.0)
    st = compare_verify(rec_tok, rec_n, None, ref)
    assert st["compared"] >= parity_steps - 10, st
    # chi-square of all transitions against p
    stat, dof = 0.0, 0
    for c in range(V + 1):
        tot = counts[c].sum()
        if tot == 0:
            continue
        e = tot * p_tab[c]
        stat += float(((counts[c] - e) ** 2 / e).sum())
        dof += V - 1
    assert stats.chi2.sf(stat, dof) > 1e-3
    # tau and alpha against the exact expectations of the rule
    tau, tau_exact = (ns + 1).mean(), e_tok.mean()
    assert abs(tau - tau_exact) <= 4 * np.std(ns + 1 - e_tok) / np.sqrt(steps)
    alpha, alpha_exact = ns.sum() / tested, b_sum / tested
    assert abs(alpha - alpha_exact) <= 4 * np.sqrt(b_var) / tested


def test_parity_largest_batch(vt):
    # B = 65535 sequences (the largest grid the entry point takes), gamma = 1,
    # V = 64: a seeded base set of 1024 sequences repeated; every sequence is
    # compared with the oracle's result for its base sequence
    import dataclasses
    base = synthetic.verify_inputs(B=1024, gamma=1, V=64, K=16, seed=7)
    B = 65535
    reps = -(-B // 1024)
    d = dict(base)
    for k in ("logits", "q", "draft", "u_accept", "u_resample"):
        d[k] = np.ascontiguousarray(np.concatenate([base[k]] * reps)[:B])
    toks, n, acc, st = _run(vt, d)
    assert st == 0
    ref = _oracle(base)
    tiled = {}
    for f in dataclasses.fields(ref):
        v = getattr(ref, f.name)
        tiled[f.name] = np.concatenate([v] * reps)[:B] if isinstance(v, np.ndarray) else v
    ref_big = dataclasses.replace(ref, **tiled)
    s = compare_verify(toks, n, acc, ref_big, draw_weights=_weights(d))
    assert s["compared"] >= B - 64 * reps, s
