"""vt_draft_logits / vt_draft_step (CUDA, through the C ABI) against the oracle."""
import numpy as np
import pytest

import oracle
import synthetic
from parity import BOUNDARY, assert_logits_close, assert_probs_close, draw_is_valid

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


def _head(B, H, K, V=None, seed=0, w_std=0.02):
    V = V or max(K, 2 * K)
    g = synthetic.rng(seed, 40)
    hidden = synthetic.normal_bf16(g, (B, H), 1.0)
    W = synthetic.normal_bf16(g, (K, H), w_std)
    trim_ids = np.sort(g.permutation(V)[:K]).astype(np.int32)
    u = synthetic.uniforms(seed, 41, B)
    return hidden, W, trim_ids, u


def _check_step(vt, hidden, W, trim_ids, u, T):
    B = hidden.shape[0]
    q, tok, st = vt.vt_draft_step(_bf(hidden), _bf(W), _dev(trim_ids), _dev(u), T)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = oracle.draft_step(hidden, W, trim_ids, u, T)
    assert_probs_close(q.cpu().numpy(), ref["q"], "q")
    tok = tok.cpu().numpy()
    checked = 0
    pos = {int(t): j for j, t in enumerate(trim_ids)}
    for b in range(B):
        if ref["margin"][b] > BOUNDARY:
            assert tok[b] == ref["tokens"][b], (b, tok[b], ref["tokens"][b], ref["margin"][b])
            checked += 1
        else:
            # boundary case: the GPU's draw must sit in a bin within 1e-5 of u
            assert int(tok[b]) in pos, (b, tok[b])
            assert draw_is_valid(ref["q"][b], u[b], pos[int(tok[b])]), (b, tok[b])
    return checked


SHAPES = [
    # B, H, K, T
    (1, 64, 100, 1.0),
    (3, 136, 1001, 0.7),     # K not a multiple of 4, H % 32 != 0
    (5, 100, 777, 1.0),      # H % 8 != 0: scalar loads
    (16, 2048, 4096, 1.0),
    (17, 256, 3000, 1.3),    # two batch tiles
    (64, 512, 2000, 1.0),    # four batch tiles
    (100, 520, 3001, 0.8),   # padded batch 128: two 128-row tiles per CTA, odd tile count
    (2, 8, 1, 1.0),          # K = 1
    (2, 65536, 64, 1.0),     # the largest hidden size
    (40, 2048, 9000, 0.1),   # finalize CTAs of four 1024-id passes, the last CTA one ragged pass
    (200, 1024, 12345, 0.1),  # padded batch 256: two warp groups in the epilogue, six passes
                             # per finalize CTA, a tile pair whose second tile is past K
    (300, 128, 3000, 0.1),   # B > 256: the CUDA-core projection, three passes per finalize CTA
]


@pytest.mark.parametrize("B,H,K,T", SHAPES)
def test_draft_logits_parity(vt, B, H, K, T):
    hidden, W, _, _ = _head(B, H, K, seed=B + H + K)
    z = vt.vt_draft_logits(_bf(hidden), _bf(W), T)
    torch.cuda.synchronize()
    assert_logits_close(z.cpu().numpy(), oracle.draft_logits(hidden, W, T))


@pytest.mark.parametrize("B,H,K,T", SHAPES)
def test_draft_step_parity(vt, B, H, K, T):
    hidden, W, trim_ids, u = _head(B, H, K, seed=7 * B + H + K)
    checked = _check_step(vt, hidden, W, trim_ids, u, T)
    # draws whose uniform lies within the boundary band are validated, not compared
    assert checked >= B - max(1, B // 10)


@pytest.mark.parametrize("B", [1, 8, 16, 64])
def test_draft_step_trimmed_head_full_size(vt, B):
    # hidden [B,2048] N(0,1), W_trim [32768,2048] N(0,0.02), T = 1
    g = synthetic.rng(50 + B, 0)
    hidden = synthetic.normal_bf16(g, (B, 2048), 1.0)
    W = synthetic.normal_bf16(g, (32768, 2048), 0.02)
    perm = synthetic.rank_permutation(128256)
    _, trim_ids, _ = synthetic.trimmed_set(128256, 32768, perm)
    u = synthetic.uniforms(50 + B, 1, B)
    checked = _check_step(vt, hidden, W, trim_ids, u, 1.0)
    # q's bins here are about 1/32768 = 3e-5 wide against a boundary band 2e-5
    # wide, so about half the draws are compared exactly (on these seeds:
    # 1 of 1, 5 of 8, 9 of 16, 33 of 64); the rest are checked as valid draws
    assert checked >= max(1, B // 2)


def test_draft_step_large_batch_full_size(vt):
    # the large-batch configuration: B=256, H=4096, K=38016 trimmed ids of
    # V=152064, W_trim N(0,0.02), hidden N(0,1), T = 0.7 (one tcgen05 tile of
    # 256 batch columns per 128 rows of W_trim)
    B, H, V, K = 256, 4096, 152064, 38016
    g = synthetic.rng(90, 0)
    hidden = synthetic.normal_bf16(g, (B, H), 1.0)
    W = synthetic.normal_bf16(g, (K, H), 0.02)
    perm = synthetic.rank_permutation(V)
    _, trim_ids, _ = synthetic.trimmed_set(V, K, perm)
    u = synthetic.uniforms(90, 1, B)
    checked = _check_step(vt, hidden, W, trim_ids, u, 0.7)
    # with 38016 ids at T = 0.7 most bins are narrower than the 1e-5 boundary
    # band, so many draws are checked as valid draws rather than compared
    assert checked >= B // 2


def test_full_vocab_head_and_trimmed_consistency(vt):
    # the full-vocabulary head (K = V, identity map) against the oracle, and
    # the trimmed head equal to the full one restricted and renormalised
    V, H, B, K = 128256, 2048, 8, 32768
    g = synthetic.rng(60, 0)
    hidden = synthetic.normal_bf16(g, (B, H), 1.0)
    W = synthetic.normal_bf16(g, (V, H), 0.02)
    u = synthetic.uniforms(60, 1, B)
    ident = np.arange(V, dtype=np.int32)
    checked = _check_step(vt, hidden, W, ident, u, 1.0)
    # bins of about 1/128256 = 7.8e-6 against a band 2e-5 wide: about a third
    # of the draws are compared exactly (3 of 8 on this seed)
    assert checked >= B // 4
    perm = synthetic.rank_permutation(V)
    _, trim_ids, _ = synthetic.trimmed_set(V, K, perm)
    qf, _, _ = vt.vt_draft_step(_bf(hidden), _bf(W), _dev(ident), _dev(u), 1.0)
    qt, _, _ = vt.vt_draft_step(_bf(hidden), _bf(W[trim_ids]), _dev(trim_ids), _dev(u), 1.0)
    torch.cuda.synchronize()
    masked = qf.cpu().numpy()[:, trim_ids].astype(np.float64)
    masked /= masked.sum(axis=1, keepdims=True)
    assert_probs_close(qt.cpu().numpy(), masked, "trimmed vs restricted full head")


def test_q_and_tokens_written_into_a_position_of_block_tensors(vt):
    B, H, K, gamma, pos = 4, 64, 500, 5, 2
    hidden, W, trim_ids, u = _head(B, H, K, seed=3)
    q_all = torch.full((B, gamma, K), -5.0, dtype=torch.float32, device="cuda")
    t_all = torch.full((B, gamma), -5, dtype=torch.int32, device="cuda")
    vt.vt_draft_step(_bf(hidden), _bf(W), _dev(trim_ids), _dev(u), 1.0, q=q_all[:, pos, :],
                     tokens=t_all[:, pos])
    torch.cuda.synchronize()
    ref = oracle.draft_step(hidden, W, trim_ids, u, 1.0)
    qa = q_all.cpu().numpy()
    assert_probs_close(qa[:, pos, :], ref["q"], "q slice")
    assert np.all(np.delete(qa, pos, axis=1) == -5.0)
    ta = t_all.cpu().numpy()
    for b in range(B):
        if ref["margin"][b] > BOUNDARY:
            assert ta[b, pos] == ref["tokens"][b]
    assert np.all(np.delete(ta, pos, axis=1) == -5)


def test_one_hot_hidden_gives_exact_logits(vt):
    # toy drafter: one-hot hidden rows select columns of W exactly
    K, H = 18, 32
    g = synthetic.rng(70, 0)
    W = synthetic.normal_bf16(g, (K, H), 1.0)
    hidden = np.zeros((H, H), np.float32)
    hidden[np.arange(H), np.arange(H)] = 1.0
    hb = synthetic.to_bf16_bits(hidden)
    z = vt.vt_draft_logits(_bf(hb), _bf(W), 1.0)
    torch.cuda.synchronize()
    assert np.array_equal(z.cpu().numpy().astype(np.float64), oracle.bf16_to_f64(W).T)


def test_non_finite_hidden_sets_status(vt):
    B, H, K = 3, 64, 300
    hidden, W, trim_ids, u = _head(B, H, K, seed=9)
    hidden = hidden.copy()
    hidden[1, 5] = 0x7FC0                      # bf16 NaN
    q, tok, st = vt.vt_draft_step(_bf(hidden), _bf(W), _dev(trim_ids), _dev(u), 1.0)
    torch.cuda.synchronize()
    assert int(st.item()) & vt.VT_DEV_NONFINITE
    assert int(tok[1].item()) == -1


def test_draft_step_sampling_frequencies(vt):
    # many identical rows: draw frequencies follow q (chi-square)
    from scipy import stats
    B, H, K = 4096, 64, 40
    g = synthetic.rng(80, 0)
    h1 = synthetic.normal_bf16(g, (1, H), 1.0)
    W = synthetic.normal_bf16(g, (K, H), 0.3)
    hidden = np.repeat(h1, B, axis=0)
    trim_ids = np.arange(K, dtype=np.int32)
    counts = np.zeros(K)
    for rep in range(5):
        u = synthetic.uniforms(80, 1 + rep, B)
        q, tok, st = vt.vt_draft_step(_bf(hidden), _bf(W), _dev(trim_ids), _dev(u), 1.0)
        torch.cuda.synchronize()
        counts += np.bincount(tok.cpu().numpy(), minlength=K)
    ref = oracle.draft_step(h1, W, trim_ids, np.array([0.5]), 1.0)["q"][0]
    assert stats.chisquare(counts, ref * counts.sum()).pvalue > 1e-3
