"""Seeded random shapes through the C ABI against the oracle: drafting
(sampling and greedy, both projection engines, every finalize pass split)
and verification (every finish tile split, fp32 and bf16 logits).

Each case draws its shape from a fixed seed, so a failure names a shape
that can be rerun.  Tokens are compared exactly away from a CDF boundary
and validated against the oracle's fp64 CDF inside the 1e-5 band, as in
the other parity tests.
"""
import numpy as np
import pytest

import oracle
import synthetic
from parity import BOUNDARY, assert_probs_close, compare_verify, draw_is_valid

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


def _draft_shape(seed):
    g = synthetic.rng(seed, 70)
    B = int(g.choice([1, 2, 3, 7, 16, 31, 64, 100, 129, 200, 256, 300]))
    # H a multiple of 8 takes the tensor cores (B <= 256), otherwise CUDA cores
    H = int(g.choice([8, 64, 136, 512, 1000, 1030, 2048]))
    K = int(g.integers(1, 20_000))
    T = float(g.choice([0.0, 0.1, 0.3, 0.7, 1.3]))
    return B, H, K, T


@pytest.mark.parametrize("seed", range(48))
def test_draft_step_random_shapes(vt, seed):
    B, H, K, T = _draft_shape(seed)
    g = synthetic.rng(seed, 71)
    hidden = synthetic.normal_bf16(g, (B, H), 1.0)
    W = synthetic.normal_bf16(g, (K, H), 0.05)
    trim_ids = np.sort(g.permutation(3 * K + 7)[:K]).astype(np.int32)
    u = synthetic.uniforms(seed, 72, B)
    q, tok, st = vt.vt_draft_step(_bf(hidden), _bf(W), _dev(trim_ids),
                                  None if T == 0.0 else _dev(u), T)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, (B, H, K, T)
    q, tok = q.cpu().numpy(), tok.cpu().numpy()
    if T == 0.0:
        ref = oracle.draft_step_greedy(hidden, W, trim_ids)
        z = ref["logits"]
        for b in range(B):
            j = int(np.flatnonzero(q[b])[0]) if q[b].any() else -1
            assert q[b].sum() == 1.0 and q[b, j] == 1.0, (B, H, K, b)
            assert tok[b] == trim_ids[j], (B, H, K, b)
            tol = 1e-3 * max(abs(z[b]).max(), np.sqrt((z[b] ** 2).mean()))
            if ref["gap"][b] > tol:
                assert j == ref["index"][b], (B, H, K, b, j, ref["index"][b])
            else:
                assert z[b, j] >= z[b].max() - tol, (B, H, K, b)
        return
    ref = oracle.draft_step(hidden, W, trim_ids, u, T)
    assert_probs_close(q, ref["q"], f"q B={B} H={H} K={K} T={T}")
    pos = {int(t): j for j, t in enumerate(trim_ids)}
    for b in range(B):
        if ref["margin"][b] > BOUNDARY:
            assert tok[b] == ref["tokens"][b], (B, H, K, T, b, tok[b], ref["tokens"][b])
        else:
            assert int(tok[b]) in pos, (B, H, K, T, b)
            assert draw_is_valid(ref["q"][b], u[b], pos[int(tok[b])]), (B, H, K, T, b)


def _verify_shape(seed):
    g = synthetic.rng(seed, 73)
    B = int(g.choice([1, 2, 5, 16, 40, 64, 100]))
    gamma = int(g.integers(1, 9))
    V = int(g.integers(2, 60_000))
    K = int(g.integers(1, V + 1))
    dt = str(g.choice(["f32", "bf16"]))
    T = float(g.choice([0.5, 0.9, 1.0, 1.4]))
    noise = float(g.choice([0.05, 0.3, 1.0]))
    return B, gamma, V, K, dt, T, noise


def _weights(d, T):
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


@pytest.mark.parametrize("seed", range(48))
def test_verify_random_shapes(vt, seed):
    B, gamma, V, K, dt, T, noise = _verify_shape(seed)
    d = synthetic.verify_inputs(B=B, gamma=gamma, V=V, K=K, seed=500 + seed,
                                logits_dtype=dt, noise_std=noise)
    L = _dev(d["logits"].view(np.int16)) if dt == "bf16" else _dev(d["logits"])
    toks, n, acc, st = vt.vt_verify(L, _dev(d["q"]), _dev(d["inv_map"]), _dev(d["draft"]),
                                    _dev(d["u_accept"]), _dev(d["u_resample"]), T)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, (B, gamma, V, K, dt, T)
    ref = oracle.verify(d["logits"], d["q"], d["inv_map"], d["draft"], d["u_accept"],
                        d["u_resample"], T, logits_dtype=dt)
    compare_verify(toks.cpu().numpy(), n.cpu().numpy(), acc.cpu().numpy(), ref,
                   draw_weights=_weights(d, T))
