"""Failure detection on the GPU without a fault: the bounded device waits of
the library, run through vt_selftest_wait on an mbarrier or a flag that
nothing completes, give up after their limit, report VT_DEV_TIMEOUT in the
status word, and leave the context usable (a calibration run afterwards is
still bit-exact against the oracle)."""
import numpy as np
import pytest

import oracle
import synthetic

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

VT_DEV_TIMEOUT = 32


@pytest.fixture(scope="module")
def vt():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import drafter_sampling_gb300 as m
    from drafter_sampling_gb300 import build
    build.build()
    m.lib()
    return m


def _status(vt, which, limit, flag=None):
    st = vt.vt_selftest_wait(which, limit, flag=flag)
    torch.cuda.synchronize()
    return int(st.item())


@pytest.mark.parametrize("limit", [1, 1000, 1 << 16])
def test_mbarrier_wait_that_nothing_completes_gives_up(vt, limit):
    assert _status(vt, 0, limit) == VT_DEV_TIMEOUT


@pytest.mark.parametrize("limit", [1, 1000, 1 << 16])
def test_flag_poll_that_nothing_publishes_gives_up(vt, limit):
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    flag[0] = 0x7fffffff  # every bit but the published one
    assert _status(vt, 2, limit, flag) == VT_DEV_TIMEOUT


def test_completed_waits_report_nothing(vt):
    assert _status(vt, 1, 1000) == 0
    flag = torch.tensor([-(1 << 31) + 5], dtype=torch.int32, device="cuda")  # bit 31 set
    assert _status(vt, 2, 1000, flag) == 0


def test_status_bits_accumulate_and_are_the_only_write(vt):
    st = torch.full((1,), 4, dtype=torch.int32, device="cuda")  # a bit set earlier
    vt.vt_selftest_wait(0, 100, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 4 | VT_DEV_TIMEOUT


def test_context_usable_after_waits_gave_up(vt):
    for which in (0, 2):
        flag = torch.zeros(1, dtype=torch.int32, device="cuda") if which == 2 else None
        assert _status(vt, which, 5000, flag) == VT_DEV_TIMEOUT
    V, N, K = 3001, 100_003, 257
    ids = synthetic.zipf_ids(N, V, s=1.1, seed=7)
    c, t, st = vt.vt_calibrate_topk(torch.from_numpy(ids).cuda(), V, K)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = oracle.token_histogram(ids, V)
    assert np.array_equal(c.cpu().numpy().view(np.uint32).astype(np.int64), ref)
    assert np.array_equal(t.cpu().numpy(), oracle.top_k(ref, K))
