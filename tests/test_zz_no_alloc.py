"""vt_verify_noalloc: verification for callers that cannot allocate device
memory (a plug-in inside a runtime that owns all device memory, C code with no
device allocator, a loop that must not risk cudaMalloc's device-wide
synchronisation).  Its scratch is a static array inside libvt, so the only
things a caller passes are inputs and outputs.

The entry point is called through the C ABI and compared with vt_verify on
the same inputs, on two calls in a row (the second call runs on the scratch
the first one left behind).  This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

import synthetic

torch = pytest.importorskip("torch")


def _lib():
    from drafter_sampling_gb300 import _lib as L
    from drafter_sampling_gb300 import build
    build.build()
    return L, L.load()


def test_noalloc_rejects_problems_beyond_its_static_scratch():
    L, lib = _lib()
    fake = ctypes.c_void_p(256)
    # 4096 sequences x 65 positions need far more than the static 2 MiB
    st = lib.vt_verify_noalloc(fake, L.VT_F32, 4096, 64, 1000, fake, fake, 10, fake, fake,
                               fake, 1.0, fake, fake, None, fake, None)
    assert st == L.VT_ERR_SCRATCH_LIMIT
    assert lib.vt_verify_workspace_bytes(4096, 64, 1000, 10) > L.VT_VERIFY_NOALLOC_SCRATCH_BYTES
    # the two workloads below fit
    assert lib.vt_verify_workspace_bytes(16, 6, 128256, 32768) <= L.VT_VERIFY_NOALLOC_SCRATCH_BYTES
    assert lib.vt_verify_workspace_bytes(256, 8, 152064, 38016) <= L.VT_VERIFY_NOALLOC_SCRATCH_BYTES


@pytest.mark.gpu
@pytest.mark.parametrize("B,gamma,V,K,dt,T", [
    (16, 6, 128256, 32768, "f32", 1.0),
    (5, 4, 1003, 97, "bf16", 0.7),
])
def test_noalloc_matches_vt_verify_on_two_calls(B, gamma, V, K, dt, T):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import drafter_sampling_gb300 as vt
    from parity import assert_probs_close
    L, lib = _lib()
    d = synthetic.verify_inputs(B=B, gamma=gamma, V=V, K=K, seed=21, logits_dtype=dt)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    logits = dev(d["logits"].view(np.int16) if dt == "bf16" else d["logits"])
    q, inv_map, draft = dev(d["q"]), dev(d["inv_map"]), dev(d["draft"])
    ua, ur = dev(d["u_accept"]), dev(d["u_resample"])

    ref_tok, ref_n, ref_acc, ref_st = vt.vt_verify(logits, q, inv_map, draft, ua, ur, T)
    torch.cuda.synchronize()
    assert int(ref_st.item()) == 0

    R = gamma + 1
    dtype_code = L.VT_BF16 if dt == "bf16" else L.VT_F32
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        tok = torch.full((B, R), -7, dtype=torch.int32, device="cuda")
        n = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        acc = torch.zeros((B, gamma), dtype=torch.float32, device="cuda")
        st = torch.full((1,), -7, dtype=torch.int32, device="cuda")
        rc = lib.vt_verify_noalloc(logits.data_ptr(), dtype_code, B, gamma, V, q.data_ptr(),
                                   inv_map.data_ptr(), K, draft.data_ptr(), ua.data_ptr(),
                                   ur.data_ptr(), T, tok.data_ptr(), n.data_ptr(),
                                   acc.data_ptr(), st.data_ptr(), stream)
        assert rc == L.VT_OK, (call, rc)
        torch.cuda.synchronize()
        assert int(st.item()) == 0, call
        assert torch.equal(tok, ref_tok), call
        assert torch.equal(n, ref_n), call
        a, r = acc.cpu().numpy(), ref_acc.cpu().numpy()
        assert np.array_equal(np.isnan(a), np.isnan(r)), call
        m = ~np.isnan(r)
        assert_probs_close(a[m], r[m], f"accept prob, call {call}")
