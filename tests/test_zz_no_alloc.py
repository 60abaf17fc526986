"""vt_verify_noalloc: verification for callers that cannot allocate device
memory (a plug-in inside a runtime that owns all device memory, C code with no
device allocator, a loop that must not risk cudaMalloc's device-wide
synchronisation).  Its scratch is a static array inside libvt, so the only
things a caller passes are inputs and outputs.

The entry point is called through the C ABI and compared with vt_verify on
the same inputs: on two calls in a row (the second call runs on the scratch
the first one left behind), on a sequence of different shapes on one stream,
and from a second context that the test creates on the same device (each
context has its own copy of the static array).  This file is collected last
on purpose.
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


def _inputs(B, gamma, V, K, dt, seed):
    d = synthetic.verify_inputs(B=B, gamma=gamma, V=V, K=K, seed=seed, logits_dtype=dt)
    logits = d["logits"].view(np.int16) if dt == "bf16" else d["logits"]
    return {"logits": np.ascontiguousarray(logits), "q": d["q"], "inv_map": d["inv_map"],
            "draft": d["draft"], "ua": d["u_accept"], "ur": d["u_resample"]}


def _reference(h, T):
    """vt_verify (caller-provided workspace) on the same inputs."""
    import drafter_sampling_gb300 as vt
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    tok, n, acc, st = vt.vt_verify(dev(h["logits"]), dev(h["q"]), dev(h["inv_map"]),
                                   dev(h["draft"]), dev(h["ua"]), dev(h["ur"]), T)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return tok.cpu().numpy(), n.cpu().numpy(), acc.cpu().numpy()


def _compare(got, ref, what):
    from parity import assert_probs_close
    tok, n, acc = got
    rtok, rn, racc = ref
    assert np.array_equal(tok, rtok), what
    assert np.array_equal(n, rn), what
    assert np.array_equal(np.isnan(acc), np.isnan(racc)), what
    m = ~np.isnan(racc)
    assert_probs_close(acc[m], racc[m], f"accept prob, {what}")


def _noalloc_torch(L, lib, h, B, gamma, V, K, dt, T):
    """One vt_verify_noalloc call on torch-owned buffers, on torch's stream."""
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    logits, q, inv_map, draft = dev(h["logits"]), dev(h["q"]), dev(h["inv_map"]), dev(h["draft"])
    ua, ur = dev(h["ua"]), dev(h["ur"])
    R = gamma + 1
    tok = torch.full((B, R), -7, dtype=torch.int32, device="cuda")
    n = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    acc = torch.zeros((B, gamma), dtype=torch.float32, device="cuda")
    st = torch.full((1,), -7, dtype=torch.int32, device="cuda")
    code = L.VT_BF16 if dt == "bf16" else L.VT_F32
    rc = lib.vt_verify_noalloc(logits.data_ptr(), code, B, gamma, V, q.data_ptr(),
                               inv_map.data_ptr(), K, draft.data_ptr(), ua.data_ptr(),
                               ur.data_ptr(), T, tok.data_ptr(), n.data_ptr(), acc.data_ptr(),
                               st.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == L.VT_OK, rc
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return tok.cpu().numpy(), n.cpu().numpy(), acc.cpu().numpy()


def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


@pytest.mark.gpu
@pytest.mark.parametrize("B,gamma,V,K,dt,T", [
    (16, 6, 128256, 32768, "f32", 1.0),
    (5, 4, 1003, 97, "bf16", 0.7),
])
def test_noalloc_matches_vt_verify_on_two_calls(B, gamma, V, K, dt, T):
    _need_gpu()
    L, lib = _lib()
    h = _inputs(B, gamma, V, K, dt, 21)
    ref = _reference(h, T)
    for call in range(2):
        _compare(_noalloc_torch(L, lib, h, B, gamma, V, K, dt, T), ref, f"call {call}")


@pytest.mark.gpu
def test_noalloc_shape_sequence_on_one_stream():
    # a large problem, a small one in another dtype, then the large one
    # again: each call must clear what it relies on, whatever the last left
    _need_gpu()
    L, lib = _lib()
    shapes = [(16, 6, 128256, 32768, "f32", 1.0, 31), (5, 4, 1003, 97, "bf16", 0.7, 32),
              (3, 2, 4096, 512, "f32", 1.3, 33), (16, 6, 128256, 32768, "f32", 1.0, 34)]
    for B, gamma, V, K, dt, T, seed in shapes:
        h = _inputs(B, gamma, V, K, dt, seed)
        ref = _reference(h, T)
        _compare(_noalloc_torch(L, lib, h, B, gamma, V, K, dt, T), ref, (B, gamma, V, dt))


class _Driver:
    """The few driver-API calls the second-context test needs (ctypes)."""

    def __init__(self):
        self.cu = ctypes.CDLL("libcuda.so.1")

    def ok(self, rc, what):
        assert rc == 0, f"{what} failed with CUresult {rc}"

    def alloc_copy(self, arr):
        ptr = ctypes.c_uint64(0)
        self.ok(self.cu.cuMemAlloc_v2(ctypes.byref(ptr), ctypes.c_size_t(max(arr.nbytes, 16))),
                "cuMemAlloc")
        if arr.nbytes:
            self.ok(self.cu.cuMemcpyHtoD_v2(ptr, arr.ctypes.data_as(ctypes.c_void_p),
                                            ctypes.c_size_t(arr.nbytes)), "cuMemcpyHtoD")
        return ptr

    def read(self, ptr, arr):
        self.ok(self.cu.cuMemcpyDtoH_v2(arr.ctypes.data_as(ctypes.c_void_p), ptr,
                                        ctypes.c_size_t(arr.nbytes)), "cuMemcpyDtoH")
        return arr


@pytest.mark.gpu
def test_noalloc_from_a_second_context_on_the_same_device():
    # A caller that creates and makes current a context of its own (driver
    # API) gets that context's copy of the static scratch: the call before
    # and the call after, in torch's primary context, agree with vt_verify too.
    _need_gpu()
    L, lib = _lib()
    B, gamma, V, K, dt, T = 4, 3, 4096, 512, "f32", 1.0
    h = _inputs(B, gamma, V, K, dt, 41)
    ref = _reference(h, T)
    _compare(_noalloc_torch(L, lib, h, B, gamma, V, K, dt, T), ref, "primary context, before")

    drv = _Driver()
    dev = ctypes.c_int(0)
    drv.ok(drv.cu.cuDeviceGet(ctypes.byref(dev), torch.cuda.current_device()), "cuDeviceGet")
    ctx = ctypes.c_void_p(0)
    drv.ok(drv.cu.cuCtxCreate_v2(ctypes.byref(ctx), 0, dev), "cuCtxCreate")
    ptrs = []
    try:
        # no torch call while this context is current: torch would use it too
        args = {k: drv.alloc_copy(np.ascontiguousarray(v)) for k, v in h.items()}
        ptrs += list(args.values())
        R = gamma + 1
        out = {"tok": np.full((B, R), -7, np.int32), "n": np.full(B, -7, np.int32),
               "acc": np.zeros((B, gamma), np.float32), "st": np.full(1, -7, np.int32)}
        dptr = {k: drv.alloc_copy(v) for k, v in out.items()}
        ptrs += list(dptr.values())
        rc = lib.vt_verify_noalloc(args["logits"].value, L.VT_F32, B, gamma, V, args["q"].value,
                                   args["inv_map"].value, K, args["draft"].value,
                                   args["ua"].value, args["ur"].value, T, dptr["tok"].value,
                                   dptr["n"].value, dptr["acc"].value, dptr["st"].value, None)
        assert rc == L.VT_OK, rc
        drv.ok(drv.cu.cuCtxSynchronize(), "cuCtxSynchronize")
        got = {k: drv.read(dptr[k], v.copy()) for k, v in out.items()}
    finally:
        for p in ptrs:
            drv.cu.cuMemFree_v2(p)
        popped = ctypes.c_void_p(0)
        drv.ok(drv.cu.cuCtxPopCurrent_v2(ctypes.byref(popped)), "cuCtxPopCurrent")
        drv.ok(drv.cu.cuCtxDestroy_v2(ctx), "cuCtxDestroy")
    assert int(got["st"][0]) == 0
    _compare((got["tok"], got["n"], got["acc"]), ref, "second context")

    _compare(_noalloc_torch(L, lib, h, B, gamma, V, K, dt, T), ref, "primary context, after")
