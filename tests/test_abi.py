"""The C-ABI library builds, loads without a GPU, and exports every entry
point include/vt.h declares.  Only calls that touch no device are made."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "vt.h")


@pytest.fixture(scope="module")
def lib():
    from drafter_sampling_gb300 import build
    build.build()
    from drafter_sampling_gb300 import _lib
    return _lib.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(vt_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = _declared_functions()
    for want in ["vt_calibrate_topk", "vt_trim_head", "vt_draft_logits", "vt_draft_step",
                 "vt_verify"]:
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name


def test_binding_signatures_cover_header():
    from drafter_sampling_gb300 import _lib
    assert set(_declared_functions()) == set(_lib.SIGNATURES)


def test_status_strings_and_version(lib):
    assert lib.vt_abi_version() >= 100
    for code in [0, -1, -2, -3, -4, -5, 12345]:
        assert isinstance(lib.vt_status_string(code), bytes)


def test_workspace_queries(lib):
    assert lib.vt_verify_workspace_bytes(16, 6, 128256, 32768) > 0
    assert lib.vt_verify_workspace_bytes(0, 6, 10, 10) == 0
    assert lib.vt_draft_workspace_bytes(16, 2048, 32768) > 0
    assert lib.vt_calibrate_topk_workspace_bytes(1000, 128256, 32768) > 0
    assert lib.vt_calibrate_topk_workspace_bytes(1000, (1 << 22) + 1, 10) == 0


def test_host_argument_checks_need_no_gpu(lib):
    from drafter_sampling_gb300 import _lib
    # null pointers and bad sizes are rejected before any CUDA call
    st = lib.vt_verify(None, 0, 1, 1, 10, None, None, 5, None, None, None, 1.0,
                       None, None, None, None, None, 0, None)
    assert st == _lib.VT_ERR_INVALID_ARG
    fake = ctypes.c_void_p(256)
    st = lib.vt_verify(fake, 0, 1, 1, 10, fake, fake, 5, fake, fake, fake, -1.0,
                       fake, fake, None, fake, fake, 1 << 20, None)
    assert st == _lib.VT_ERR_INVALID_ARG          # temperature < 0
    st = lib.vt_verify(fake, 0, 1, 1, 10, fake, fake, 5, fake, fake, fake, float("nan"),
                       fake, fake, None, fake, fake, 1 << 20, None)
    assert st == _lib.VT_ERR_INVALID_ARG          # temperature not finite
    st = lib.vt_verify(fake, 0, 1, 1, 10, fake, fake, 5, fake, fake, fake, 1.0,
                       fake, fake, None, fake, None, 0, None)
    assert st == _lib.VT_ERR_WORKSPACE            # sampling needs q and uniforms: given
    st = lib.vt_verify(fake, 0, 1, 1, 10, None, None, 5, fake, None, None, 1.0,
                       fake, fake, None, fake, fake, 1 << 20, None)
    assert st == _lib.VT_ERR_INVALID_ARG          # sampling without q / uniforms
    st = lib.vt_verify(fake, 0, 1, 1, 10, None, None, 5, fake, None, None, 0.0,
                       fake, fake, None, fake, None, 0, None)
    assert st == _lib.VT_ERR_WORKSPACE            # greedy: q and uniforms not needed
    st = lib.vt_verify(fake, 0, 1, 1, 10, fake, fake, 11, fake, fake, fake, 1.0,
                       fake, fake, None, fake, fake, 1 << 20, None)
    assert st == _lib.VT_ERR_INVALID_ARG          # K > V
    st = lib.vt_verify(fake, 0, 1, 1, 10, fake, fake, 5, fake, fake, fake, 1.0,
                       fake, fake, None, fake, None, 0, None)
    assert st == _lib.VT_ERR_WORKSPACE            # no workspace
    st = lib.vt_verify(fake, 7, 1, 1, 10, fake, fake, 5, fake, fake, fake, 1.0,
                       fake, fake, None, fake, fake, 1 << 20, None)
    assert st == _lib.VT_ERR_INVALID_ARG          # unknown dtype


def test_draft_argument_checks_need_no_gpu(lib):
    from drafter_sampling_gb300 import _lib
    fake = ctypes.c_void_p(256)
    # vt_draft_logits needs T > 0; vt_draft_step also accepts T == 0 (greedy)
    st = lib.vt_draft_logits(fake, 2, 8, fake, 16, 0.0, fake, 16, fake, 1 << 20, None)
    assert st == _lib.VT_ERR_INVALID_ARG
    st = lib.vt_draft_step(fake, 2, 8, fake, fake, 16, fake, -1.0, fake, 16, fake, 1, fake,
                           fake, 1 << 20, None)
    assert st == _lib.VT_ERR_INVALID_ARG
    st = lib.vt_draft_step(fake, 2, 8, fake, fake, 16, None, 1.0, fake, 16, fake, 1, fake,
                           fake, 1 << 20, None)
    assert st == _lib.VT_ERR_INVALID_ARG          # sampling needs uniforms
    st = lib.vt_draft_step(fake, 2, 8, fake, fake, 16, None, 0.0, fake, 16, fake, 1, fake,
                           None, 0, None)
    assert st == _lib.VT_ERR_WORKSPACE            # greedy: uniforms not needed


def test_selection_argument_checks_need_no_gpu(lib):
    from drafter_sampling_gb300 import _lib
    fake = ctypes.c_void_p(256)
    assert lib.vt_calibrate_select_workspace_bytes(1000, 128256) > \
        lib.vt_calibrate_topk_workspace_bytes(1000, 128256, 10)
    assert lib.vt_calibrate_select_workspace_bytes(1000, (1 << 22) + 1) == 0
    for P in (0.0, -0.5, 1.5, float("nan")):
        st = lib.vt_calibrate_top_p(fake, 10, 100, P, fake, fake, fake, fake, fake, 1 << 24, None)
        assert st == _lib.VT_ERR_INVALID_ARG, P
    st = lib.vt_calibrate_top_p(fake, 10, 100, 0.5, fake, fake, None, fake, fake, 1 << 24, None)
    assert st == _lib.VT_ERR_INVALID_ARG          # no k_out
    st = lib.vt_calibrate_min_count(fake, 10, 100, 3, fake, fake, fake, fake, fake, 16, None)
    assert st == _lib.VT_ERR_WORKSPACE            # workspace too small


def test_block_descriptor_layout_matches_the_header(tmp_path):
    # the ctypes mirror of vt_block_desc must have the C layout, field for field
    import shutil
    import subprocess
    from drafter_sampling_gb300 import _lib
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    fields = [f for f, _ in _lib.BlockDesc._fields_]
    src = tmp_path / "layout.c"
    src.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "vt.h"\nint main(void) {\n'
                   '  printf("%zu\\n", sizeof(vt_block_desc));\n' +
                   "".join(f'  printf("%zu\\n", offsetof(vt_block_desc, {f}));\n' for f in fields) +
                   "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.check_call([cc, "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    got = [int(x) for x in subprocess.check_output([str(exe)]).split()]
    assert got[0] == ctypes.sizeof(_lib.BlockDesc)
    assert got[1:] == [getattr(_lib.BlockDesc, f).offset for f in fields]


def test_block_graph_argument_checks_need_no_gpu(lib):
    from drafter_sampling_gb300 import _lib
    h = ctypes.c_void_p()
    assert lib.vt_block_graph_create(None, ctypes.byref(h)) == _lib.VT_ERR_INVALID_ARG
    d = _lib.BlockDesc()  # all zero: bad sizes
    assert lib.vt_block_graph_create(ctypes.byref(d), ctypes.byref(h)) == _lib.VT_ERR_INVALID_ARG
    assert lib.vt_block_graph_launch(None, None) == _lib.VT_ERR_INVALID_ARG
    assert lib.vt_block_graph_destroy(None) == _lib.VT_OK
    assert lib.vt_block_workspace_bytes(16, 2048, 32768, 128256, 6) >= \
        lib.vt_verify_workspace_bytes(16, 6, 128256, 32768)


def test_tree_and_topk_argument_checks_need_no_gpu(lib):
    from drafter_sampling_gb300 import _lib
    fake = ctypes.c_void_p(256)
    # the drafter's top-k: 1 <= k <= 32 and k <= K, T > 0
    assert lib.vt_draft_topk_workspace_bytes(16, 2048, 32768, 8) > \
        lib.vt_draft_workspace_bytes(16, 2048, 32768)
    for B, K, k in [(16, 32768, 0), (16, 32768, 33), (16, 4, 5), (0, 100, 1)]:
        assert lib.vt_draft_topk_workspace_bytes(B, 64, K, k) == 0, (B, K, k)
    for K, k, T in [(100, 0, 1.0), (100, 33, 1.0), (4, 5, 1.0), (100, 8, 0.0),
                    (100, 8, float("inf"))]:
        st = lib.vt_draft_topk(fake, 2, 64, fake, fake, K, k, T, fake, fake, fake, fake,
                               1 << 24, None)
        assert st == _lib.VT_ERR_INVALID_ARG, (K, k, T)
    st = lib.vt_draft_topk(fake, 2, 64, fake, None, 100, 8, 1.0, fake, fake, fake, fake,
                           1 << 24, None)
    assert st == _lib.VT_ERR_INVALID_ARG          # no trim_ids
    st = lib.vt_draft_topk(fake, 2, 64, fake, fake, 100, 8, 1.0, fake, fake, fake, fake, 16,
                           None)
    assert st == _lib.VT_ERR_WORKSPACE            # workspace too small
    # greedy tree verification: N <= 255 nodes, T == 0 only
    assert lib.vt_verify_tree_workspace_bytes(16, 32, 128256) > 0
    st = lib.vt_verify_tree(fake, _lib.VT_F32, 2, 256, 1000, fake, 0, fake, 0.0, fake, fake,
                            fake, fake, fake, 1 << 24, None)
    assert st == _lib.VT_ERR_INVALID_ARG          # too many nodes
    st = lib.vt_verify_tree(fake, _lib.VT_F32, 2, 8, 1000, fake, 4, fake, 0.0, fake, fake,
                            fake, fake, fake, 1 << 24, None)
    assert st == _lib.VT_ERR_INVALID_ARG          # parent stride shorter than a tree
    st = lib.vt_verify_tree(fake, _lib.VT_F32, 2, 8, 1000, fake, 0, fake, 0.7, fake, fake,
                            fake, fake, fake, 1 << 24, None)
    assert st == _lib.VT_ERR_UNSUPPORTED          # sampling trees
    st = lib.vt_verify_tree(fake, _lib.VT_F32, 2, 8, 1000, fake, 0, fake, 0.0, fake, fake,
                            fake, fake, fake, 16, None)
    assert st == _lib.VT_ERR_WORKSPACE


def test_selftest_wait_arguments_need_no_gpu(lib):
    from drafter_sampling_gb300 import _lib
    fake = ctypes.c_void_p(256)
    bad = _lib.VT_ERR_INVALID_ARG
    assert lib.vt_selftest_wait(3, 10, None, fake, None) == bad         # unknown wait
    assert lib.vt_selftest_wait(-1, 10, None, fake, None) == bad
    assert lib.vt_selftest_wait(0, 0, None, fake, None) == bad          # limit 0
    assert lib.vt_selftest_wait(0, (1 << 20) + 1, None, fake, None) == bad
    assert lib.vt_selftest_wait(2, 10, None, fake, None) == bad         # flag missing
    assert lib.vt_selftest_wait(0, 10, None, None, None) == bad         # no status word


def test_noalloc_checks_arguments_before_its_scratch_limit(lib):
    from drafter_sampling_gb300 import _lib
    fake = ctypes.c_void_p(256)
    bad = _lib.VT_ERR_INVALID_ARG
    # out-of-range arguments report what vt_verify reports, not the scratch limit
    for B, gamma, V, K, dt, T in [(70000, 6, 1000, 10, _lib.VT_F32, 1.0),
                                  (16, 65, 1000, 10, _lib.VT_F32, 1.0),
                                  (16, 6, (1 << 22) + 1, 10, _lib.VT_F32, 1.0),
                                  (16, 6, 1000, 1001, _lib.VT_F32, 1.0),
                                  (16, 6, 1000, 10, 7, 1.0),
                                  (16, 6, 1000, 10, _lib.VT_F32, -1.0),
                                  (16, 6, 1000, 10, _lib.VT_F32, float("nan"))]:
        args = (fake, dt, B, gamma, V, fake, fake, K, fake, fake, fake, T, fake, fake, None,
                fake, None)
        assert lib.vt_verify_noalloc(*args) == bad, (B, gamma, V, K, dt, T)
        assert lib.vt_verify(*args[:-1], fake, 1 << 30, None) == bad, (B, gamma, V, K, dt, T)
    # a missing pointer too
    st = lib.vt_verify_noalloc(fake, _lib.VT_F32, 16, 6, 1000, None, fake, 10, fake, fake, fake,
                               1.0, fake, fake, None, fake, None)
    assert st == bad
