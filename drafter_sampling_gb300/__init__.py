"""drafter_sampling_gb300: VocabTrim drafting and speculative verification on
one GB300 GPU (sm_103a).

Thin Python binding over libvt.so (include/vt.h).  Each function below has
the name of the C entry point it calls and only marshals arguments: it checks
tensor devices, dtypes and shapes, allocates outputs and workspace with
PyTorch, and passes raw device pointers and the current CUDA stream.  Every
step of the computation runs in the library's CUDA kernels.

bf16 tensors may be passed as torch.bfloat16 or as int16/uint16 bit patterns.
"""
from __future__ import annotations

from . import _lib
from ._lib import (VT_BF16, VT_DEV_BAD_DRAFT, VT_DEV_BAD_ID,  # noqa: F401
                   VT_DEV_DUPLICATE_ID, VT_DEV_NONFINITE, VT_DEV_TIMEOUT,
                   VT_DEV_ZERO_RESIDUAL, VT_F32,
                   VtError)

__all__ = ["vt_selftest_wait", "vt_calibrate_topk", "vt_calibrate_top_p", "vt_calibrate_min_count", "vt_trim_head",
           "vt_draft_logits", "vt_draft_step", "vt_draft_topk", "vt_verify", "vt_verify_tree",
           "BlockGraph",
           "workspace_bytes",
           "VtError", "lib"]


def lib():
    """The loaded ctypes library (raises if libvt.so is not built)."""
    return _lib.load()


_TORCH = None
_RAW_STREAM = None  # torch's raw current-stream getter, or False where it has none
_BF16 = None


def _torch():
    global _TORCH
    if _TORCH is None:
        import torch
        _TORCH = torch
    return _TORCH


def _stream_ptr(stream):
    """The cudaStream_t of `stream`, or of the current device's current
    stream (read without building a torch.cuda.Stream object, which costs a
    few microseconds of host time per call)."""
    global _RAW_STREAM
    torch = _torch()
    if stream is not None:
        return stream.cuda_stream
    if _RAW_STREAM is None:
        _RAW_STREAM = getattr(torch._C, "_cuda_getCurrentRawStream", False)
    if _RAW_STREAM:
        return _RAW_STREAM(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


def _dev(t, name, dtypes, dim=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype not in dtypes:
        raise TypeError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dim is not None and t.dim() != dim:
        raise ValueError(f"{name} must have {dim} dimensions, got {t.dim()}")
    return t


def _bf16_dtypes():
    global _BF16
    if _BF16 is None:
        torch = _torch()
        _BF16 = (torch.bfloat16, torch.int16, torch.uint16)
    return _BF16


def _ws(nbytes, device):
    torch = _torch()
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def workspace_bytes(kind: str, **kw) -> int:
    L = lib()
    if kind == "calibrate":
        return L.vt_calibrate_topk_workspace_bytes(kw["n"], kw["V"], kw["K"])
    if kind == "select":
        return L.vt_calibrate_select_workspace_bytes(kw["n"], kw["V"])
    if kind == "trim":
        return L.vt_trim_head_workspace_bytes(kw["V"], kw["K"])
    if kind == "draft":
        return L.vt_draft_workspace_bytes(kw["B"], kw["H"], kw["K"])
    if kind == "verify":
        return L.vt_verify_workspace_bytes(kw["B"], kw["gamma"], kw["V"], kw["K"])
    raise ValueError(kind)


def vt_calibrate_topk(ids, V: int, K: int, counts=None, topk_ids=None, dev_status=None,
                      workspace=None, stream=None):
    """Token histogram and Top-K (count desc, id asc) of int32 ids.

    Returns (counts uint32-as-int32 [V], topk_ids int32 [K], dev_status int32 [1]).
    """
    torch = _torch()
    _dev(ids, "ids", (torch.int32,), 1)
    dev = ids.device
    n = ids.numel()
    if counts is None:
        counts = torch.empty(V, dtype=torch.int32, device=dev)
    if topk_ids is None:
        topk_ids = torch.empty(K, dtype=torch.int32, device=dev)
    if dev_status is None:
        dev_status = torch.empty(1, dtype=torch.int32, device=dev)
    _dev(counts, "counts", (torch.int32, torch.uint32), 1)
    _dev(topk_ids, "topk_ids", (torch.int32,), 1)
    if counts.numel() != V or topk_ids.numel() != K:
        raise ValueError("counts must have V elements and topk_ids K elements")
    L = lib()
    if workspace is None:
        workspace = _ws(L.vt_calibrate_topk_workspace_bytes(n, V, K), dev)
    st = L.vt_calibrate_topk(ids.data_ptr(), n, V, K, counts.data_ptr(), topk_ids.data_ptr(),
                             dev_status.data_ptr(), workspace.data_ptr(), workspace.numel(),
                             _stream_ptr(stream))
    _lib.check("vt_calibrate_topk", st)
    return counts, topk_ids, dev_status


def _calibrate_select(fn: str, ids, V: int, param, counts, ranked_ids, k_out, dev_status,
                      workspace, stream):
    torch = _torch()
    _dev(ids, "ids", (torch.int32,), 1)
    dev = ids.device
    n = ids.numel()
    if counts is None:
        counts = torch.empty(V, dtype=torch.int32, device=dev)
    if ranked_ids is None:
        ranked_ids = torch.empty(V, dtype=torch.int32, device=dev)
    if k_out is None:
        k_out = torch.empty(1, dtype=torch.int32, device=dev)
    if dev_status is None:
        dev_status = torch.empty(1, dtype=torch.int32, device=dev)
    _dev(counts, "counts", (torch.int32, torch.uint32), 1)
    _dev(ranked_ids, "ranked_ids", (torch.int32,), 1)
    if counts.numel() != V or ranked_ids.numel() != V:
        raise ValueError("counts and ranked_ids must have V elements")
    L = lib()
    if workspace is None:
        workspace = _ws(L.vt_calibrate_select_workspace_bytes(n, V), dev)
    st = getattr(L, fn)(ids.data_ptr(), n, V, param, counts.data_ptr(), ranked_ids.data_ptr(),
                        k_out.data_ptr(), dev_status.data_ptr(), workspace.data_ptr(),
                        workspace.numel(), _stream_ptr(stream))
    _lib.check(fn, st)
    return counts, ranked_ids, k_out, dev_status


def vt_calibrate_top_p(ids, V: int, P: float, counts=None, ranked_ids=None, k_out=None,
                       dev_status=None, workspace=None, stream=None):
    """Token histogram, full ranking, and K = the smallest ranked prefix whose
    counts reach P of the calibration tokens.  Returns (counts [V], ranked_ids
    [V], k_out int32 [1] on the device, dev_status [1])."""
    return _calibrate_select("vt_calibrate_top_p", ids, V, float(P), counts, ranked_ids, k_out,
                             dev_status, workspace, stream)


def vt_calibrate_min_count(ids, V: int, min_count: int, counts=None, ranked_ids=None, k_out=None,
                           dev_status=None, workspace=None, stream=None):
    """Token histogram, full ranking, and K = the number of ids counted at
    least min_count times.  Returns (counts, ranked_ids, k_out, dev_status)."""
    return _calibrate_select("vt_calibrate_min_count", ids, V, int(min_count), counts,
                             ranked_ids, k_out, dev_status, workspace, stream)


def vt_trim_head(W, topk_ids, W_trim=None, trim_ids=None, inv_map=None, dev_status=None,
                 workspace=None, stream=None):
    """W_trim = W[sorted(topk_ids)], trim_ids (ascending) and inv_map.

    Returns (W_trim [K,H] same dtype as W, trim_ids int32 [K], inv_map int32 [V], dev_status).
    """
    torch = _torch()
    _dev(W, "W", _bf16_dtypes(), 2)
    _dev(topk_ids, "topk_ids", (torch.int32,), 1)
    V, H = W.shape
    K = topk_ids.numel()
    dev = W.device
    if W_trim is None:
        W_trim = torch.empty((K, H), dtype=W.dtype, device=dev)
    if trim_ids is None:
        trim_ids = torch.empty(K, dtype=torch.int32, device=dev)
    if inv_map is None:
        inv_map = torch.empty(V, dtype=torch.int32, device=dev)
    if dev_status is None:
        dev_status = torch.empty(1, dtype=torch.int32, device=dev)
    _dev(W_trim, "W_trim", _bf16_dtypes(), 2)
    if tuple(W_trim.shape) != (K, H) or trim_ids.numel() != K or inv_map.numel() != V:
        raise ValueError("output shapes do not match (K, H), K and V")
    L = lib()
    if workspace is None:
        workspace = _ws(L.vt_trim_head_workspace_bytes(V, K), dev)
    st = L.vt_trim_head(W.data_ptr(), V, H, topk_ids.data_ptr(), K, W_trim.data_ptr(),
                        trim_ids.data_ptr(), inv_map.data_ptr(), dev_status.data_ptr(),
                        workspace.data_ptr(), workspace.numel(), _stream_ptr(stream))
    _lib.check("vt_trim_head", st)
    return W_trim, trim_ids, inv_map, dev_status


def vt_draft_logits(hidden, W_trim, temperature: float = 1.0, logits=None, workspace=None,
                    stream=None):
    """logits [B, K] fp32 = hidden @ W_trim^T / T."""
    torch = _torch()
    _dev(hidden, "hidden", _bf16_dtypes(), 2)
    _dev(W_trim, "W_trim", _bf16_dtypes(), 2)
    B, H = hidden.shape
    K, H2 = W_trim.shape
    if H2 != H:
        raise ValueError("hidden and W_trim disagree on H")
    if logits is None:
        logits = torch.empty((B, K), dtype=torch.float32, device=hidden.device)
    if logits.dim() != 2 or logits.shape[0] != B or logits.stride(1) != 1 or logits.shape[1] < K:
        raise ValueError("logits must be [B, >=K] with unit inner stride")
    L = lib()
    if workspace is None:
        workspace = _ws(L.vt_draft_workspace_bytes(B, H, K), hidden.device)
    st = L.vt_draft_logits(hidden.data_ptr(), B, H, W_trim.data_ptr(), K, float(temperature),
                           logits.data_ptr(), logits.stride(0), workspace.data_ptr(),
                           workspace.numel(), _stream_ptr(stream))
    _lib.check("vt_draft_logits", st)
    return logits


def vt_draft_step(hidden, W_trim, trim_ids, uniforms, temperature: float = 1.0, q=None,
                  tokens=None, dev_status=None, workspace=None, stream=None):
    """One drafting step; returns (q [B, K] view, tokens int32 [B] view, dev_status).

    ``q`` may be a strided view such as q_all[:, pos, :] of a contiguous
    [B, gamma, K] tensor (unit inner stride), and ``tokens`` a strided view
    such as tok_all[:, pos] of a [B, gamma] tensor.  temperature == 0 drafts
    greedily (q one-hot); ``uniforms`` may then be None.
    """
    torch = _torch()
    greedy = float(temperature) == 0.0
    _dev(hidden, "hidden", _bf16_dtypes(), 2)
    _dev(W_trim, "W_trim", _bf16_dtypes(), 2)
    _dev(trim_ids, "trim_ids", (torch.int32,), 1)
    if uniforms is not None or not greedy:
        _dev(uniforms, "uniforms", (torch.float32,), 1)
    B, H = hidden.shape
    K = W_trim.shape[0]
    dev = hidden.device
    if q is None:
        q = torch.empty((B, K), dtype=torch.float32, device=dev)
    if q.dim() != 2 or q.shape[0] != B or q.shape[1] != K or q.stride(1) != 1:
        raise ValueError("q must be [B, K] with unit inner stride")
    if tokens is None:
        tokens = torch.empty(B, dtype=torch.int32, device=dev)
    if tokens.dim() != 1 or tokens.shape[0] != B or tokens.dtype != torch.int32:
        raise ValueError("tokens must be an int32 vector of B entries (any stride)")
    if dev_status is None:
        dev_status = torch.empty(1, dtype=torch.int32, device=dev)
    if (uniforms is not None and uniforms.numel() != B) or trim_ids.numel() != K:
        raise ValueError("uniforms must have B and trim_ids K elements")
    L = lib()
    if workspace is None:
        workspace = _ws(L.vt_draft_workspace_bytes(B, H, K), dev)
    st = L.vt_draft_step(hidden.data_ptr(), B, H, W_trim.data_ptr(), trim_ids.data_ptr(), K,
                         uniforms.data_ptr() if uniforms is not None else None,
                         float(temperature), q.data_ptr(), q.stride(0),
                         tokens.data_ptr(), tokens.stride(0), dev_status.data_ptr(),
                         workspace.data_ptr(), workspace.numel(), _stream_ptr(stream))
    _lib.check("vt_draft_step", st)
    return q, tokens, dev_status


def vt_verify(target_logits, q, inv_map, draft_tokens, u_accept, u_resample,
              temperature: float = 1.0, out_tokens=None, out_num_accepted=None,
              out_accept_prob=None, dev_status=None, workspace=None, stream=None,
              want_accept_prob: bool = True):
    """Modified rejection sampling over a batch of drafted blocks.

    target_logits [B, gamma+1, V] float32 or bf16; q [B, gamma, K] float32.
    temperature == 0 verifies greedily (a drafted token is kept iff it is the
    target's highest logit); q, inv_map and the uniforms may then be None.
    Returns (out_tokens [B, gamma+1], out_num_accepted [B], out_accept_prob
    [B, gamma] or None, dev_status [1]).
    """
    torch = _torch()
    if target_logits.dtype == torch.float32:
        dt = VT_F32
    elif target_logits.dtype in _bf16_dtypes():
        dt = VT_BF16
    else:
        raise TypeError("target_logits must be float32 or bf16")
    greedy = float(temperature) == 0.0
    _dev(target_logits, "target_logits", (target_logits.dtype,), 3)
    _dev(draft_tokens, "draft_tokens", (torch.int32,), 2)
    B, R, V = target_logits.shape
    gamma = R - 1
    if tuple(draft_tokens.shape) != (B, gamma):
        raise ValueError("draft_tokens shape does not match target_logits")
    # the sampling rule needs all four; the greedy one reads none (any given
    # one is still checked)
    if not greedy or q is not None:
        _dev(q, "q", (torch.float32,), 3)
        if tuple(q.shape[:2]) != (B, gamma):
            raise ValueError("q shape does not match target_logits")
    if not greedy or inv_map is not None:
        _dev(inv_map, "inv_map", (torch.int32,), 1)
        if inv_map.numel() != V:
            raise ValueError("inv_map must have V entries")
    if not greedy or u_accept is not None:
        _dev(u_accept, "u_accept", (torch.float32,), 2)
        if tuple(u_accept.shape) != (B, gamma):
            raise ValueError("u_accept must be [B, gamma]")
    if not greedy or u_resample is not None:
        _dev(u_resample, "u_resample", (torch.float32,), 2)
        if tuple(u_resample.shape) != (B, R):
            raise ValueError("u_resample must be [B, gamma+1]")
    K = q.shape[2] if q is not None else 1
    ptr = lambda x: x.data_ptr() if x is not None else None
    dev = target_logits.device
    if out_tokens is None:
        out_tokens = torch.empty((B, R), dtype=torch.int32, device=dev)
    if out_num_accepted is None:
        out_num_accepted = torch.empty(B, dtype=torch.int32, device=dev)
    if out_accept_prob is None and want_accept_prob:
        out_accept_prob = torch.empty((B, gamma), dtype=torch.float32, device=dev)
    if dev_status is None:
        dev_status = torch.empty(1, dtype=torch.int32, device=dev)
    L = lib()
    if workspace is None:
        workspace = _ws(L.vt_verify_workspace_bytes(B, gamma, V, K), dev)
    st = L.vt_verify(target_logits.data_ptr(), dt, B, gamma, V, ptr(q), ptr(inv_map),
                     K, draft_tokens.data_ptr(), ptr(u_accept), ptr(u_resample),
                     float(temperature), out_tokens.data_ptr(), out_num_accepted.data_ptr(),
                     out_accept_prob.data_ptr() if out_accept_prob is not None else None,
                     dev_status.data_ptr(), workspace.data_ptr(), workspace.numel(),
                     _stream_ptr(stream))
    _lib.check("vt_verify", st)
    return out_tokens, out_num_accepted, out_accept_prob, dev_status


def vt_draft_topk(hidden, W_trim, trim_ids, k: int, temperature: float = 1.0, out_ids=None,
                  out_logq=None, dev_status=None, workspace=None, stream=None):
    """The drafter's k best trimmed candidates per row (target ids, best
    first) with log q.  Returns (out_ids int32 [B, k], out_logq [B, k],
    dev_status [1])."""
    torch = _torch()
    _dev(hidden, "hidden", _bf16_dtypes(), 2)
    _dev(W_trim, "W_trim", _bf16_dtypes(), 2)
    _dev(trim_ids, "trim_ids", (torch.int32,), 1)
    B, H = hidden.shape
    K = W_trim.shape[0]
    dev = hidden.device
    if out_ids is None:
        out_ids = torch.empty((B, k), dtype=torch.int32, device=dev)
    if out_logq is None:
        out_logq = torch.empty((B, k), dtype=torch.float32, device=dev)
    if dev_status is None:
        dev_status = torch.empty(1, dtype=torch.int32, device=dev)
    L = lib()
    if workspace is None:
        workspace = _ws(L.vt_draft_topk_workspace_bytes(B, H, K, k), dev)
    st = L.vt_draft_topk(hidden.data_ptr(), B, H, W_trim.data_ptr(), trim_ids.data_ptr(), K, k,
                         float(temperature), out_ids.data_ptr(), out_logq.data_ptr(),
                         dev_status.data_ptr(), workspace.data_ptr(), workspace.numel(),
                         _stream_ptr(stream))
    _lib.check("vt_draft_topk", st)
    return out_ids, out_logq, dev_status


def vt_verify_tree(target_logits, parent, tokens, temperature: float = 0.0, out_tokens=None,
                   out_num_accepted=None, out_path=None, dev_status=None, workspace=None,
                   stream=None, want_path: bool = True):
    """Greedy verification of draft trees: target_logits [B, N+1, V] (row 0
    after the context, row i+1 after node i), parent int32 [B, N] or [N]
    (shared tree; -1 = the context), tokens int32 [B, N].  Returns
    (out_tokens [B, N+1], out_num_accepted [B], out_path [B, N] or None,
    dev_status [1])."""
    torch = _torch()
    if target_logits.dtype == torch.float32:
        dt = VT_F32
    elif target_logits.dtype in _bf16_dtypes():
        dt = VT_BF16
    else:
        raise TypeError("target_logits must be float32 or bf16")
    _dev(target_logits, "target_logits", (target_logits.dtype,), 3)
    _dev(tokens, "tokens", (torch.int32,), 2)
    _dev(parent, "parent", (torch.int32,), None)
    B, R, V = target_logits.shape
    N = R - 1
    if tuple(tokens.shape) != (B, N):
        raise ValueError("tokens must be [B, N] with N + 1 = target_logits.shape[1]")
    if parent.dim() == 1 and parent.numel() == N:
        pstride = 0
    elif parent.dim() == 2 and tuple(parent.shape) == (B, N):
        pstride = N
    else:
        raise ValueError("parent must be [N] or [B, N]")
    dev = target_logits.device
    if out_tokens is None:
        out_tokens = torch.empty((B, R), dtype=torch.int32, device=dev)
    if out_num_accepted is None:
        out_num_accepted = torch.empty(B, dtype=torch.int32, device=dev)
    if out_path is None and want_path:
        out_path = torch.empty((B, N), dtype=torch.int32, device=dev)
    if dev_status is None:
        dev_status = torch.empty(1, dtype=torch.int32, device=dev)
    L = lib()
    if workspace is None:
        workspace = _ws(L.vt_verify_tree_workspace_bytes(B, N, V), dev)
    st = L.vt_verify_tree(target_logits.data_ptr(), dt, B, N, V, parent.data_ptr(), pstride,
                          tokens.data_ptr(), float(temperature), out_tokens.data_ptr(),
                          out_num_accepted.data_ptr(),
                          out_path.data_ptr() if out_path is not None else None,
                          dev_status.data_ptr(), workspace.data_ptr(), workspace.numel(),
                          _stream_ptr(stream))
    _lib.check("vt_verify_tree", st)
    return out_tokens, out_num_accepted, out_path, dev_status


def vt_selftest_wait(which: int, limit: int, flag=None, dev_status=None, stream=None):
    """Runs one of the library's bounded device waits on an object that
    nothing completes (which 0: an mbarrier; 1: the same after one arrival,
    the control; 2: a published flag, int32 [1] on the device) for at most
    `limit` polls.  VT_DEV_TIMEOUT is OR-ed into dev_status (int32 [1],
    zeroed here when not given) when the wait gives up."""
    torch = _torch()
    if dev_status is None:
        dev = flag.device if flag is not None else torch.device("cuda", torch.cuda.current_device())
        dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
    _dev(dev_status, "dev_status", (torch.int32,), 1)
    if flag is not None:
        _dev(flag, "flag", (torch.int32, torch.uint32), 1)
    st = lib().vt_selftest_wait(int(which), int(limit),
                                flag.data_ptr() if flag is not None else None,
                                dev_status.data_ptr(), _stream_ptr(stream))
    _lib.check("vt_selftest_wait", st)
    return dev_status


class BlockGraph:
    """One speculative block (gamma drafting steps + verification) captured
    as a CUDA graph by vt_block_graph_create and replayed by launch().

    The tensors are fixed at capture and kept alive by this object; a replay
    reads what they hold when it runs.  Outputs (q, draft_tokens,
    out_tokens, out_num_accepted, out_accept_prob, dev_status [2]) are
    attributes.  temperature == 0 captures the greedy block (u_draft,
    u_accept and u_resample may then be None)."""

    def __init__(self, hidden, W_trim, trim_ids, inv_map, target_logits, u_draft=None,
                 u_accept=None, u_resample=None, temperature: float = 1.0,
                 want_accept_prob: bool = True):
        torch = _torch()
        greedy = float(temperature) == 0.0
        _dev(hidden, "hidden", _bf16_dtypes(), 3)
        _dev(W_trim, "W_trim", _bf16_dtypes(), 2)
        _dev(trim_ids, "trim_ids", (torch.int32,), 1)
        _dev(inv_map, "inv_map", (torch.int32,), 1)
        if target_logits.dtype == torch.float32:
            dt = VT_F32
        elif target_logits.dtype in _bf16_dtypes():
            dt = VT_BF16
        else:
            raise TypeError("target_logits must be float32 or bf16")
        _dev(target_logits, "target_logits", (target_logits.dtype,), 3)
        gamma, B, H = hidden.shape
        K = W_trim.shape[0]
        V = target_logits.shape[2]
        if tuple(target_logits.shape[:2]) != (B, gamma + 1) or inv_map.numel() != V:
            raise ValueError("target_logits must be [B, gamma+1, V] and inv_map [V]")
        for name, x, shape in (("u_draft", u_draft, (gamma, B)), ("u_accept", u_accept, (B, gamma)),
                               ("u_resample", u_resample, (B, gamma + 1))):
            if x is None:
                if not greedy:
                    raise ValueError(f"{name} is needed unless temperature == 0")
                continue
            _dev(x, name, (torch.float32,), 2)
            if tuple(x.shape) != shape:
                raise ValueError(f"{name} must be {shape}")
        dev = hidden.device
        self.q = torch.empty((B, gamma, K), dtype=torch.float32, device=dev)
        self.draft_tokens = torch.empty((B, gamma), dtype=torch.int32, device=dev)
        self.out_tokens = torch.empty((B, gamma + 1), dtype=torch.int32, device=dev)
        self.out_num_accepted = torch.empty(B, dtype=torch.int32, device=dev)
        self.out_accept_prob = (torch.empty((B, gamma), dtype=torch.float32, device=dev)
                                if want_accept_prob else None)
        self.dev_status = torch.zeros(2, dtype=torch.int32, device=dev)
        L = lib()
        self.workspace = _ws(L.vt_block_workspace_bytes(B, H, K, V, gamma), dev)
        self._keep = (hidden, W_trim, trim_ids, inv_map, target_logits, u_draft, u_accept,
                      u_resample)
        ptr = lambda x: x.data_ptr() if x is not None else None
        d = _lib.BlockDesc(B, H, K, V, gamma, dt, float(temperature), ptr(hidden), ptr(W_trim),
                           ptr(trim_ids), ptr(inv_map), ptr(u_draft), ptr(target_logits),
                           ptr(u_accept), ptr(u_resample), ptr(self.q), ptr(self.draft_tokens),
                           ptr(self.out_tokens), ptr(self.out_num_accepted),
                           ptr(self.out_accept_prob), ptr(self.dev_status),
                           ptr(self.workspace), self.workspace.numel())
        import ctypes
        h = ctypes.c_void_p()
        _lib.check("vt_block_graph_create", L.vt_block_graph_create(ctypes.byref(d), ctypes.byref(h)))
        self._handle = h

    def launch(self, stream=None):
        _lib.check("vt_block_graph_launch",
                   lib().vt_block_graph_launch(self._handle, _stream_ptr(stream)))

    def close(self):
        if getattr(self, "_handle", None):
            lib().vt_block_graph_destroy(self._handle)
            self._handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
