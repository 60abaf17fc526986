"""The speculative block as a CUDA graph (vt_block_graph_*): a replay gives
bit-for-bit what the same vt_draft_step / vt_verify calls give when made
directly, a replay matches the oracle's block (drafting and verification) on
the same generator inputs, it reads the input buffers live, and the greedy
block works the same way."""
import numpy as np
import pytest

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


def _inputs(B, gamma, H, K, V, seed, dtype="f32"):
    vi = synthetic.verify_inputs(B=B, gamma=gamma, V=V, K=K, seed=seed, logits_dtype=dtype)
    g = synthetic.rng(seed, 60)
    W = synthetic.normal_bf16(g, (K, H), 0.02)
    hidden = synthetic.hidden_states((gamma, B, H), seed=seed)
    logits = _dev(vi["logits"].view(np.int16) if dtype == "bf16" else vi["logits"])
    if dtype == "bf16":
        logits = logits.view(torch.bfloat16)
    trim_ids = np.sort(np.flatnonzero(vi["inv_map"] >= 0)).astype(np.int32)
    return dict(hidden=_dev(hidden.view(np.int16)), W_trim=_dev(W.view(np.int16)),
                trim_ids=_dev(trim_ids), inv_map=_dev(vi["inv_map"]), logits=logits,
                u_draft=_dev(synthetic.uniforms(seed, 61, (gamma, B))),
                u_accept=_dev(vi["u_accept"]), u_resample=_dev(vi["u_resample"]))


def _direct(vt, x, T):
    gamma, B, _ = x["hidden"].shape
    K = x["W_trim"].shape[0]
    q = torch.empty((B, gamma, K), dtype=torch.float32, device="cuda")
    tok = torch.empty((B, gamma), dtype=torch.int32, device="cuda")
    st_d = torch.zeros(gamma, dtype=torch.int32, device="cuda")
    for j in range(gamma):
        vt.vt_draft_step(x["hidden"][j], x["W_trim"], x["trim_ids"],
                         x["u_draft"][j] if T > 0 else None, T, q=q[:, j, :], tokens=tok[:, j],
                         dev_status=st_d[j:j + 1])
    out, n, acc, st_v = vt.vt_verify(x["logits"], q, x["inv_map"], tok,
                                     x["u_accept"] if T > 0 else None,
                                     x["u_resample"] if T > 0 else None, T)
    torch.cuda.synchronize()
    return q, tok, out, n, acc, int(st_d.max().item()), int(st_v.item())


def _graph(vt, x, T):
    return vt.BlockGraph(x["hidden"], x["W_trim"], x["trim_ids"], x["inv_map"], x["logits"],
                         u_draft=x["u_draft"] if T > 0 else None,
                         u_accept=x["u_accept"] if T > 0 else None,
                         u_resample=x["u_resample"] if T > 0 else None, temperature=T)


def _same(a, b):
    return torch.equal(a, b) if a.dtype != torch.float32 else \
        torch.equal(a.nan_to_num(-7.0), b.nan_to_num(-7.0))


@pytest.mark.parametrize("B,gamma,H,K,V,T,dtype", [
    (16, 6, 2048, 32768, 128256, 1.0, "f32"),   # the block of the bench step
    (4, 3, 512, 3000, 20011, 0.7, "bf16"),
    (8, 4, 256, 2048, 9000, 0.0, "f32"),        # the greedy block
])
def test_graph_replay_equals_direct_calls(vt, B, gamma, H, K, V, T, dtype):
    x = _inputs(B, gamma, H, K, V, seed=B + gamma + V, dtype=dtype)
    ref = _direct(vt, x, T)
    g = _graph(vt, x, T)
    for _ in range(2):                         # replays are repeatable
        g.launch()
        torch.cuda.synchronize()
        got = (g.q, g.draft_tokens, g.out_tokens, g.out_num_accepted, g.out_accept_prob)
        for a, b in zip(got, ref[:5]):
            assert _same(a, b)
        assert int(g.dev_status[0].item()) == ref[5] and int(g.dev_status[1].item()) == ref[6]
    g.close()


def test_graph_reads_inputs_live(vt):
    x = _inputs(6, 4, 256, 1024, 5000, seed=4)
    g = _graph(vt, x, 1.0)
    g.launch()
    torch.cuda.synchronize()
    # every accept uniform at 1: every drafted token is rejected at position 0
    x["u_accept"].fill_(1.0)
    g.launch()
    torch.cuda.synchronize()
    assert (g.out_num_accepted == 0).all()
    assert (g.out_tokens[:, 1:] == -1).all()
    # and the graph's result equals a direct run on the changed inputs
    ref = _direct(vt, x, 1.0)
    assert torch.equal(g.out_tokens, ref[2])
    g.close()


def test_drafting_flags_of_every_step_are_kept(vt):
    # a NaN hidden state in step 1 (of 3): the drafting status word keeps its
    # flag although steps 2 and 3 are clean
    x = _inputs(4, 3, 256, 1024, 4000, seed=5)
    h = x["hidden"].clone()
    h[1, 2, 7] = 0x7fc0
    x["hidden"] = h
    g = _graph(vt, x, 1.0)
    g.launch()
    torch.cuda.synchronize()
    assert int(g.dev_status[0].item()) & vt.VT_DEV_NONFINITE
    g.close()


def test_hidden_states_written_just_before_a_replay_are_read(vt):
    # the projections of a replay stage the hidden states before their
    # dependency wait: a kernel that rewrites them right before the launch, on
    # the same stream and with no synchronisation between, must still be seen
    x = _inputs(8, 3, 256, 1024, 4000, seed=6)
    g = _graph(vt, x, 1.0)
    g.launch()
    torch.cuda.synchronize()
    first = g.draft_tokens.clone()
    fresh = _dev(synthetic.hidden_states(tuple(x["hidden"].shape), seed=77).view(np.int16))
    big = torch.empty(1 << 26, dtype=torch.float32, device="cuda")
    for _ in range(3):
        big.mul_(1.0)                          # keep the stream busy before the rewrite
    x["hidden"].copy_(fresh)
    g.launch()
    torch.cuda.synchronize()
    ref = _direct(vt, x, 1.0)
    assert _same(g.q, ref[0]) and torch.equal(g.draft_tokens, ref[1])
    assert torch.equal(g.out_tokens, ref[2])
    assert not torch.equal(g.draft_tokens, first)
    g.close()


def _oracle_block(x, T, dtype):
    """The block on the oracle: each drafting step from the same hidden
    states, trimmed head and uniforms, then the verification of the GPU's
    drafted tokens (equal to the oracle's wherever a draw is not a boundary
    case, and then checked as a valid draw) with the oracle's own q."""
    import oracle
    h = x["hidden"].cpu().numpy().view(np.uint16)
    W = x["W_trim"].cpu().numpy().view(np.uint16)
    trim_ids = x["trim_ids"].cpu().numpy()
    u = x["u_draft"].cpu().numpy()
    gamma, B, _ = h.shape
    steps = [oracle.draft_step(h[j], W, trim_ids, u[j], T) for j in range(gamma)]
    logits = x["logits"].cpu()
    logits = logits.view(torch.int16).numpy().view(np.uint16) if dtype == "bf16" else logits.numpy()
    return steps, logits


@pytest.mark.parametrize("B,gamma,H,K,V,T,dtype", [
    (16, 6, 2048, 32768, 128256, 1.0, "f32"),   # the block of the bench step
    (8, 4, 1024, 6000, 40000, 0.7, "bf16"),     # bf16 target logits, T = 0.7
])
def test_graph_replay_against_the_oracle(vt, B, gamma, H, K, V, T, dtype):
    # one replay of the captured block (VocabTrim Appendix C.1, Algorithm 2:
    # draft gamma tokens, then score and verify them) against the oracle run
    # on the same generator inputs
    import oracle
    from parity import BOUNDARY, assert_probs_close, compare_verify, draw_is_valid
    x = _inputs(B, gamma, H, K, V, seed=3 * B + gamma, dtype=dtype)
    g = _graph(vt, x, T)
    g.launch()
    torch.cuda.synchronize()
    assert int(g.dev_status[0].item()) == 0 and int(g.dev_status[1].item()) == 0
    steps, logits = _oracle_block(x, T, dtype)
    q = g.q.cpu().numpy()
    tok = g.draft_tokens.cpu().numpy()
    trim_ids = x["trim_ids"].cpu().numpy()
    pos = {int(t): j for j, t in enumerate(trim_ids)}
    compared = 0
    for j, ref in enumerate(steps):
        assert_probs_close(q[:, j, :], ref["q"], f"q of drafting step {j}")
        for b in range(B):
            if ref["margin"][b] > BOUNDARY:
                assert tok[b, j] == ref["tokens"][b], (j, b)
                compared += 1
            else:
                assert draw_is_valid(ref["q"][b], x["u_draft"][j, b].item(), pos[int(tok[b, j])])
    assert compared >= (B * gamma) // 3
    q_ref = np.stack([s["q"] for s in steps], axis=1)
    ref = oracle.verify(logits, q_ref, x["inv_map"].cpu().numpy(), tok,
                        x["u_accept"].cpu().numpy(), x["u_resample"].cpu().numpy(), T,
                        logits_dtype=dtype)

    im = x["inv_map"].cpu().numpy()

    def weights(b, n):
        l = oracle.bf16_to_f64(logits[b, n]) if dtype == "bf16" else logits[b, n]
        p = oracle.softmax(l, T)
        if n < gamma:
            qf = np.zeros(V)
            qf[im >= 0] = q_ref[b, n, im[im >= 0]]
            p = oracle.residual_weights(p, qf)
        return p, float(x["u_resample"][b, n].item())

    stats = compare_verify(g.out_tokens.cpu().numpy(), g.out_num_accepted.cpu().numpy(),
                           g.out_accept_prob.cpu().numpy(), ref, draw_weights=weights)
    assert stats["compared"] + stats["excluded_seq"] == B
    assert stats["compared"] >= B // 2
    g.close()
