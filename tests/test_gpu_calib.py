"""vt_calibrate_topk / vt_trim_head (CUDA, through the C ABI) against the
oracle: bit-exact counts, ranked ids, trimmed rows and maps."""
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


def _calib(vt, ids, V, K):
    c, t, st = vt.vt_calibrate_topk(_dev(ids), V, K)
    torch.cuda.synchronize()
    return c.cpu().numpy().view(np.uint32), t.cpu().numpy(), int(st.item())


@pytest.mark.parametrize("V,N,K,s", [
    (3001, 100_003, 257, 1.1),
    (3001, 100_003, 3001, 1.1),     # K = V: a full ranking
    (1000, 50_000, 1, 0.5),         # K = 1
    (70_000, 1_000_001, 5000, 1.1),
    (17, 9, 5, 1.1),                # many zero counts (ties at 0)
    (300_000, 2_100_000, 20_000, 1.1),  # counts need 22 bits: three sort passes, 74 tiles
    (600_000, 1_000_003, 4096, 1.0),    # V beyond the shared-memory hot-id table
    (1 << 22, 2_000_000, 4096, 1.05),   # the largest vocabulary the sort takes
])
def test_histogram_and_topk_bit_exact(vt, V, N, K, s):
    ids = synthetic.zipf_ids(N, V, s=s, seed=V + N)
    c, t, st = _calib(vt, ids, V, K)
    assert st == 0
    ref_c = oracle.token_histogram(ids, V)
    assert np.array_equal(c.astype(np.int64), ref_c)
    assert np.array_equal(t, oracle.top_k(ref_c, K))


def test_heavy_ties(vt):
    # 600 ids, counts drawn from {0,1,2,3}: ties everywhere, lower id wins
    g = synthetic.rng(90, 0)
    V = 600
    target = g.integers(0, 4, V)
    ids = np.repeat(np.arange(V, dtype=np.int32), target)
    ids = ids[g.permutation(ids.size)]
    for K in [1, 100, 599, 600]:
        c, t, st = _calib(vt, ids, V, K)
        assert np.array_equal(c.astype(np.int64), target)
        assert np.array_equal(t, oracle.top_k(target, K))


def test_heavy_ties_many_tiles(vt):
    # 40000 ids over twenty sort tiles, counts in {0,..,5}: equal counts span tiles
    g = synthetic.rng(91, 0)
    V = 40_000
    target = g.integers(0, 6, V)
    ids = np.repeat(np.arange(V, dtype=np.int32), target)
    ids = ids[g.permutation(ids.size)]
    for K in [1, 8191, 8192, 8193, 39_999]:
        c, t, st = _calib(vt, ids, V, K)
        assert st == 0
        assert np.array_equal(c.astype(np.int64), target)
        assert np.array_equal(t, oracle.top_k(target, K))


def test_vocabulary_above_sort_limit_is_unsupported(vt):
    ids = torch.zeros(4, dtype=torch.int32, device="cuda")
    with pytest.raises(vt.VtError):
        vt.vt_calibrate_topk(ids, (1 << 22) + 1, 10)


def test_empty_stream(vt):
    c, t, st = _calib(vt, np.zeros(0, np.int32), 50, 7)
    assert st == 0 and not c.any()
    assert list(t) == list(range(7))


def test_out_of_range_ids_flagged_and_skipped(vt):
    ids = np.array([1, 2, -1, 2, 50, 3, 2], np.int32)
    c, t, st = _calib(vt, ids, 50, 3)
    assert st & vt.VT_DEV_BAD_ID
    good = ids[(ids >= 0) & (ids < 50)]
    assert np.array_equal(c.astype(np.int64), np.bincount(good, minlength=50))
    assert list(t) == [2, 1, 3]


def test_unaligned_id_stream(vt):
    # a view starting one element in: scalar loads
    ids = synthetic.zipf_ids(10_007, 999, seed=5)
    full = _dev(ids)
    view = full[1:]
    c, t, st = vt.vt_calibrate_topk(view, 999, 50)
    torch.cuda.synchronize()
    ref_c = oracle.token_histogram(ids[1:], 999)
    assert np.array_equal(c.cpu().numpy().view(np.uint32).astype(np.int64), ref_c)
    assert np.array_equal(t.cpu().numpy(), oracle.top_k(ref_c, 50))


def test_calibration_full_size(vt):
    # 50M Zipf(1.1) ids over V=128256; K in {8192, 16384, 32768, 65536}
    V, N = 128256, 50_000_000
    ids = synthetic.zipf_ids(N, V, s=1.1, seed=synthetic.SEED_CALIB)
    ref_c = oracle.token_histogram(ids, V)
    d_ids = _dev(ids)
    for K in [8192, 16384, 32768, 65536]:
        c, t, st = vt.vt_calibrate_topk(d_ids, V, K)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert np.array_equal(c.cpu().numpy().view(np.uint32).astype(np.int64), ref_c)
        assert np.array_equal(t.cpu().numpy(), oracle.top_k(ref_c, K))


@pytest.mark.parametrize("V,H,K", [(500, 24, 77), (1000, 13, 999), (64, 8, 64), (300, 3072, 1),
                                   (70_001, 16, 40_000),       # K above one index-kernel batch
                                   ((1 << 20) + 37, 8, 5000),   # V above the one-CTA index mapper
                                   (1 << 22, 8, 3000)])         # the largest vocabulary
def test_trim_head_bit_exact(vt, V, H, K):
    g = synthetic.rng(V + H + K, 0)
    W = g.integers(0, 65535, (V, H)).astype(np.uint16)
    topk = g.permutation(V)[:K].astype(np.int32)
    Wt, ti, im, st = vt.vt_trim_head(_dev(W.view(np.int16)), _dev(topk))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rW, rti, rim = oracle.trim_head(W, topk)
    assert np.array_equal(Wt.cpu().numpy().view(np.uint16), rW)
    assert np.array_equal(ti.cpu().numpy(), rti)
    assert np.array_equal(im.cpu().numpy(), rim)


def test_trim_head_full_size(vt):
    # W [128256, 3072] bf16 N(0,0.02); trim to the calibrated top-K
    V, H = 128256, 3072
    W = synthetic.head_weights(V, H, seed=synthetic.SEED_CALIB)
    ids = synthetic.zipf_ids(5_000_000, V, s=1.1, seed=synthetic.SEED_CALIB)
    d_W = _dev(W.view(np.int16))
    _, topk, _ = vt.vt_calibrate_topk(_dev(ids), V, 65536)
    topk_h = topk.cpu().numpy()
    for K in [8192, 16384, 32768, 65536]:
        Wt, ti, im, st = vt.vt_trim_head(d_W, topk[:K].contiguous())
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        rW, rti, rim = oracle.trim_head(W, topk_h[:K])
        assert np.array_equal(ti.cpu().numpy(), rti)
        assert np.array_equal(im.cpu().numpy(), rim)
        # every trimmed row, bit for bit, at every K
        assert np.array_equal(Wt.cpu().numpy().view(np.uint16), rW), K
        del Wt


def test_trim_head_flags_duplicates_and_range(vt):
    W = np.arange(40, dtype=np.uint16).reshape(10, 4)
    Wt, ti, im, st = vt.vt_trim_head(_dev(W.view(np.int16)), _dev(np.array([1, 3, 3], np.int32)))
    torch.cuda.synchronize()
    assert int(st.item()) & vt.VT_DEV_DUPLICATE_ID
    # the distinct ids are kept in id order, the missing slot is -1
    assert list(ti.cpu().numpy()) == [1, 3, -1]
    expect = np.full(10, -1, np.int32)
    expect[1], expect[3] = 0, 1
    assert np.array_equal(im.cpu().numpy(), expect)
    assert np.array_equal(Wt.cpu().numpy().view(np.uint16)[:2], W[[1, 3]])
    for bad in ([1, 10], [-2, 4]):
        _, ti, _, st = vt.vt_trim_head(_dev(W.view(np.int16)), _dev(np.array(bad, np.int32)))
        torch.cuda.synchronize()
        assert int(st.item()) & vt.VT_DEV_BAD_ID
        assert sorted(ti.cpu().numpy().tolist()) == [-1, [b for b in bad if 0 <= b < 10][0]]
