"""Top-P and minimum-frequency vocabulary selection (CUDA, through the C ABI)
against the oracle: counts, the full ranking and K bit-exact."""
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


def _top_p(vt, ids, V, P):
    c, r, k, st = vt.vt_calibrate_top_p(_dev(ids), V, P)
    torch.cuda.synchronize()
    return c.cpu().numpy().view(np.uint32).astype(np.int64), r.cpu().numpy(), int(k.item()), \
        int(st.item())


def _min_count(vt, ids, V, f):
    c, r, k, st = vt.vt_calibrate_min_count(_dev(ids), V, f)
    torch.cuda.synchronize()
    return c.cpu().numpy().view(np.uint32).astype(np.int64), r.cpu().numpy(), int(k.item()), \
        int(st.item())


def test_hand_worked_counts(vt):
    ids = np.repeat(np.arange(5, dtype=np.int32), [5, 0, 9, 5, 1])
    ids = ids[synthetic.rng(1, 0).permutation(ids.size)]
    for P, K in [(0.45, 1), (0.46, 2), (0.70, 2), (0.71, 3), (1.0, 4)]:
        c, r, k, st = _top_p(vt, ids, 5, P)
        assert st == 0 and r.tolist() == [2, 0, 3, 4, 1] and k == K, (P, k)
    for f, K in [(5, 3), (6, 1), (0, 5), (1, 4)]:
        assert _min_count(vt, ids, 5, f)[2] == K, f


@pytest.mark.parametrize("V,N,s", [(3001, 100_003, 1.1), (70_000, 1_000_001, 1.1),
                                   (20_000, 300_000, 0.7)])
def test_top_p_and_min_count_bit_exact(vt, V, N, s):
    ids = synthetic.zipf_ids(N, V, s=s, seed=V + N)
    ref_c = oracle.token_histogram(ids, V)
    ref_r = oracle.ranking(ref_c)
    for P in [0.01, 0.5, 0.9, 0.99, 0.999999, 1.0]:
        c, r, k, st = _top_p(vt, ids, V, P)
        assert st == 0
        assert np.array_equal(c, ref_c) and np.array_equal(r, ref_r)
        assert k == oracle.top_p(ref_c, P)[1], P
    for f in [0, 1, 2, 10, 1000, 10 ** 9]:
        c, r, k, st = _min_count(vt, ids, V, f)
        assert st == 0 and np.array_equal(r, ref_r)
        assert k == oracle.min_count(ref_c, f)[1], f


def test_threshold_exactly_on_a_prefix(vt):
    # counts 4, 3, 2, 1 (total 10): P = 0.7 is reached exactly by 4 + 3
    ids = np.repeat(np.arange(4, dtype=np.int32), [4, 3, 2, 1])
    assert _top_p(vt, ids, 4, 0.7)[2] == oracle.top_p([4, 3, 2, 1], 0.7)[1] == 2
    assert _top_p(vt, ids, 4, 0.7000001)[2] == 3


def test_heavy_ties_and_empty_stream(vt):
    g = synthetic.rng(92, 0)
    V = 40_000
    target = g.integers(0, 4, V)
    ids = np.repeat(np.arange(V, dtype=np.int32), target)
    ids = ids[g.permutation(ids.size)]
    ref_r = oracle.ranking(target)
    for P in [0.3, 0.75]:
        c, r, k, st = _top_p(vt, ids, V, P)
        assert np.array_equal(r, ref_r) and k == oracle.top_p(target, P)[1]
    c, r, k, st = _top_p(vt, np.zeros(0, np.int32), 50, 0.5)
    assert st == 0 and k == 0 and r.tolist() == list(range(50))
    assert _min_count(vt, np.zeros(0, np.int32), 50, 0)[2] == 50


def test_selection_full_size_then_trim(vt):
    # 50M Zipf(1.1) ids over V=128256; the Top-P selection feeds the trim
    V, N = 128256, 50_000_000
    ids = synthetic.zipf_ids(N, V, s=1.1, seed=synthetic.SEED_CALIB)
    ref_c = oracle.token_histogram(ids, V)
    d_ids = _dev(ids)
    for P in [0.8, 0.95]:
        c, r, k, st = vt.vt_calibrate_top_p(d_ids, V, P)
        torch.cuda.synchronize()
        K = int(k.item())
        assert int(st.item()) == 0 and K == oracle.top_p(ref_c, P)[1]
        assert np.array_equal(r.cpu().numpy()[:K], oracle.top_k(ref_c, K))
        W = synthetic.head_weights(V, 8, seed=3)
        Wt, ti, im, st2 = vt.vt_trim_head(_dev(W.view(np.int16)), r[:K].contiguous())
        torch.cuda.synchronize()
        assert int(st2.item()) == 0 and np.array_equal(ti.cpu().numpy(),
                                                      np.sort(oracle.top_k(ref_c, K)))
