"""ctypes view of libvt.so, the C ABI declared in include/vt.h.

Loading fails loudly when the library has not been built: there is no
fallback implementation anywhere in this package.
"""
from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libvt.so")

VT_OK = 0
VT_ERR_INVALID_ARG = -1
VT_ERR_UNSUPPORTED = -2
VT_ERR_CUDA = -3
VT_ERR_BAD_INPUT = -4
VT_ERR_WORKSPACE = -5
VT_ERR_SCRATCH_LIMIT = -6
VT_VERIFY_NOALLOC_SCRATCH_BYTES = 2 << 20

VT_F32 = 0
VT_BF16 = 1

VT_DEV_BAD_ID = 1
VT_DEV_DUPLICATE_ID = 2
VT_DEV_BAD_DRAFT = 4
VT_DEV_NONFINITE = 8
VT_DEV_ZERO_RESIDUAL = 16
VT_DEV_TIMEOUT = 32

_p = C.c_void_p
_i32 = C.c_int32
_i64 = C.c_int64
_f32 = C.c_float
_sz = C.c_size_t

# name -> (restype, argtypes); mirrors include/vt.h
class BlockDesc(C.Structure):
    """vt_block_desc of include/vt.h, field for field."""
    _fields_ = [("B", C.c_int32), ("H", C.c_int32), ("K", C.c_int32), ("V", C.c_int32),
                ("gamma", C.c_int32), ("logits_dtype", C.c_int32), ("temperature", C.c_float),
                ("hidden", C.c_void_p), ("W_trim", C.c_void_p), ("trim_ids", C.c_void_p),
                ("inv_map", C.c_void_p), ("u_draft", C.c_void_p), ("target_logits", C.c_void_p),
                ("u_accept", C.c_void_p), ("u_resample", C.c_void_p), ("q", C.c_void_p),
                ("draft_tokens", C.c_void_p), ("out_tokens", C.c_void_p),
                ("out_num_accepted", C.c_void_p), ("out_accept_prob", C.c_void_p),
                ("dev_status", C.c_void_p), ("workspace", C.c_void_p),
                ("workspace_bytes", C.c_size_t)]


SIGNATURES = {
    "vt_status_string": (C.c_char_p, [C.c_int]),
    "vt_abi_version": (C.c_int, []),
    "vt_selftest_wait": (C.c_int, [_i32, C.c_uint32, _p, _p, _p]),
    "vt_calibrate_topk_workspace_bytes": (_sz, [_i64, _i32, _i32]),
    "vt_calibrate_topk": (C.c_int, [_p, _i64, _i32, _i32, _p, _p, _p, _p, _sz, _p]),
    "vt_calibrate_select_workspace_bytes": (_sz, [_i64, _i32]),
    "vt_calibrate_top_p": (C.c_int, [_p, _i64, _i32, C.c_double, _p, _p, _p, _p, _p, _sz, _p]),
    "vt_calibrate_min_count": (C.c_int, [_p, _i64, _i32, C.c_uint32, _p, _p, _p, _p, _p, _sz,
                                         _p]),
    "vt_trim_head_workspace_bytes": (_sz, [_i32, _i32]),
    "vt_trim_head": (C.c_int, [_p, _i32, _i32, _p, _i32, _p, _p, _p, _p, _p, _sz, _p]),
    "vt_draft_workspace_bytes": (_sz, [_i32, _i32, _i32]),
    "vt_draft_logits": (C.c_int, [_p, _i32, _i32, _p, _i32, _f32, _p, _i64, _p, _sz, _p]),
    "vt_draft_step": (C.c_int, [_p, _i32, _i32, _p, _p, _i32, _p, _f32, _p, _i64, _p, _i64,
                                _p, _p, _sz, _p]),
    "vt_draft_topk_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32]),
    "vt_draft_topk": (C.c_int, [_p, _i32, _i32, _p, _p, _i32, _i32, _f32, _p, _p, _p, _p, _sz,
                                _p]),
    "vt_verify_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32]),
    "vt_verify": (C.c_int, [_p, _i32, _i32, _i32, _i32, _p, _p, _i32, _p, _p, _p, _f32, _p,
                            _p, _p, _p, _p, _sz, _p]),
    "vt_verify_noalloc": (C.c_int, [_p, _i32, _i32, _i32, _i32, _p, _p, _i32, _p, _p, _p, _f32,
                                    _p, _p, _p, _p, _p]),
    "vt_verify_tree_workspace_bytes": (_sz, [_i32, _i32, _i32]),
    "vt_verify_tree": (C.c_int, [_p, _i32, _i32, _i32, _i32, _p, _i64, _p, _f32, _p, _p, _p, _p,
                                 _p, _sz, _p]),
    "vt_block_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32, _i32]),
    "vt_block_graph_create": (C.c_int, [C.POINTER(BlockDesc), C.POINTER(C.c_void_p)]),
    "vt_block_graph_launch": (C.c_int, [_p, _p]),
    "vt_block_graph_destroy": (C.c_int, [_p]),
}


class VtError(RuntimeError):
    def __init__(self, fn: str, status: int, text: str):
        super().__init__(f"{fn} failed: {text} ({status})")
        self.status = status


_LIB = None


def load(path: str = LIB_PATH):
    """Load libvt.so once and attach the C signatures."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it with drafter_sampling_gb300.build.build() "
            "(or __graft_entry__.build()); there is no CPU fallback")
    lib = C.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def check(fn: str, status: int) -> None:
    if status != VT_OK:
        text = load().vt_status_string(status).decode()
        raise VtError(fn, status, text)
