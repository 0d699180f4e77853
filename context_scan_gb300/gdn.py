"""Thin ctypes binding of the C ABI in include/gdn.h (argument marshalling only).

Every function here takes torch tensors that already live on the GPU, checks nothing
beyond what marshalling needs, passes raw device pointers plus the current CUDA stream to
``libgdn.so`` and raises ``GdnError`` on a non-OK status. All validation and all compute
happen in the library's CUDA kernels; there is no fallback of any kind. If ``libgdn.so``
has not been built, loading raises.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libgdn.so")

GDN_DTYPE_F32, GDN_DTYPE_BF16 = 0, 1
STATUS = {0: "GDN_OK", 1: "GDN_ERR_INVALID_ARG", 2: "GDN_ERR_UNSUPPORTED_SHAPE",
          3: "GDN_ERR_UNSUPPORTED_DTYPE", 4: "GDN_ERR_MISALIGNED", 5: "GDN_ERR_WORKSPACE",
          6: "GDN_ERR_CUDA", 7: "GDN_ERR_TIMEOUT", 8: "GDN_ERR_DEVICE"}
EXPORTED = ("gdn_workspace_bytes", "gdn_segmented_pieces", "gdn_segmented_plan", "gdn_chunk_fwd",
            "gdn_segment_summary", "gdn_summary_scan", "gdn_segment_fwd", "gdn_segmented_fwd",
            "gdn_segmented_fwd_timed", "gdn_segmented_fwd_noalloc",
            "gdn_varlen_workspace_bytes", "gdn_varlen_fwd", "gdn_varlen_fwd_timed",
            "gdn_state_grad_summary", "gdn_state_grad_scan", "gdn_chunk_bwd_workspace_bytes",
            "gdn_chunk_bwd", "gdn_chunk_bwd_timed", "gdn_status_string", "gdn_check_device_error", "gdn_selftest_wait_timeout")


class GdnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)} "
                         f"({lib().gdn_status_string(status).decode()})")


class Problem(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("H", ctypes.c_int),
                ("K", ctypes.c_int), ("V", ctypes.c_int), ("chunk", ctypes.c_int),
                ("in_dtype", ctypes.c_int), ("out_dtype", ctypes.c_int),
                ("decay_first", ctypes.c_int), ("gate_k", ctypes.c_int)]


_lib = None
_P = ctypes.c_void_p


def lib():
    """Load libgdn.so (raises OSError if it is missing: build it with __graft_entry__.build)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise OSError(f"libgdn.so not built ({LIB_PATH}); run __graft_entry__.build()")
        L = ctypes.CDLL(LIB_PATH)
        pp = ctypes.POINTER(Problem)
        L.gdn_workspace_bytes.argtypes = [pp, ctypes.c_int]
        L.gdn_workspace_bytes.restype = ctypes.c_size_t
        L.gdn_segmented_pieces.argtypes = [pp, ctypes.c_int]
        L.gdn_segmented_pieces.restype = ctypes.c_int
        L.gdn_segmented_plan.argtypes = [pp, ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                                         ctypes.POINTER(ctypes.c_int)]
        L.gdn_segmented_plan.restype = ctypes.c_int
        L.gdn_segment_fwd.argtypes = [pp, ctypes.c_int] + [_P] * 9 + [ctypes.c_size_t, _P]
        L.gdn_chunk_fwd.argtypes = [pp] + [_P] * 9 + [ctypes.c_size_t, _P]
        L.gdn_segment_summary.argtypes = [pp, ctypes.c_int] + [_P] * 7 + [ctypes.c_size_t, _P]
        L.gdn_summary_scan.argtypes = [pp, ctypes.c_int] + [_P] * 5
        L.gdn_segmented_fwd.argtypes = [pp, ctypes.c_int] + [_P] * 10 + [ctypes.c_size_t, _P]
        L.gdn_segmented_fwd_timed.argtypes = ([pp, ctypes.c_int] + [_P] * 10 +
                                              [ctypes.c_size_t, _P, _P])
        L.gdn_segmented_fwd_noalloc.argtypes = [pp, ctypes.c_int] + [_P] * 10
        L.gdn_varlen_workspace_bytes.argtypes = [pp, ctypes.c_int]
        L.gdn_varlen_workspace_bytes.restype = ctypes.c_size_t
        L.gdn_varlen_fwd.argtypes = [pp, ctypes.c_int] + [_P] * 10 + [ctypes.c_size_t, _P]
        L.gdn_varlen_fwd_timed.argtypes = ([pp, ctypes.c_int] + [_P] * 10 +
                                           [ctypes.c_size_t, _P, _P])
        L.gdn_state_grad_summary.argtypes = [pp, ctypes.c_int] + [_P] * 8
        L.gdn_state_grad_scan.argtypes = [pp, ctypes.c_int] + [_P] * 5
        L.gdn_chunk_bwd_workspace_bytes.argtypes = [pp, ctypes.c_int]
        L.gdn_chunk_bwd_workspace_bytes.restype = ctypes.c_size_t
        L.gdn_chunk_bwd.argtypes = [pp, ctypes.c_int] + [_P] * 15 + [ctypes.c_size_t, _P]
        L.gdn_chunk_bwd_timed.argtypes = L.gdn_chunk_bwd.argtypes + [_P]
        L.gdn_status_string.argtypes = [ctypes.c_int]
        L.gdn_status_string.restype = ctypes.c_char_p
        L.gdn_check_device_error.argtypes = [_P, _P, ctypes.POINTER(ctypes.c_uint)]
        L.gdn_selftest_wait_timeout.argtypes = [_P, ctypes.c_longlong, _P]
        for fn in ("gdn_chunk_fwd", "gdn_segment_summary", "gdn_summary_scan", "gdn_segment_fwd",
                   "gdn_segmented_fwd", "gdn_segmented_fwd_timed", "gdn_segmented_fwd_noalloc",
                   "gdn_varlen_fwd", "gdn_varlen_fwd_timed", "gdn_check_device_error",
                   "gdn_selftest_wait_timeout", "gdn_state_grad_summary", "gdn_state_grad_scan",
                   "gdn_chunk_bwd", "gdn_chunk_bwd_timed"):
            getattr(L, fn).restype = ctypes.c_int
        _lib = L
    return _lib


def _dtype_code(t) -> int:
    import torch
    if t.dtype == torch.float32:
        return GDN_DTYPE_F32
    if t.dtype == torch.bfloat16:
        return GDN_DTYPE_BF16
    return 99   # the library rejects it with GDN_ERR_UNSUPPORTED_DTYPE


def problem(q_or_k, v, o=None, chunk: int = 64, decay_first: bool = False, g=None) -> Problem:
    """The problem description of these tensors; g (optional) sets gate_k when it carries
    one gate per key channel ([B, T, H, K])."""
    B, T, H, K = q_or_k.shape
    V = v.shape[-1]
    out = GDN_DTYPE_F32 if o is None else _dtype_code(o)
    gate_k = int(g is not None and g.dim() == 4)
    return Problem(B, T, H, K, V, chunk, _dtype_code(q_or_k), out, int(decay_first), gate_k)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else stream


def _check(status: int, where: str):
    if status != 0:
        raise GdnError(status, where)


def workspace_bytes(prob: Problem, nseg: int = 1) -> int:
    return int(lib().gdn_workspace_bytes(ctypes.byref(prob), nseg))


def segmented_pieces(prob: Problem, nseg: int = 1) -> int:
    """Pieces per sequence the segmented forward uses on the current device (0: invalid)."""
    return int(lib().gdn_segmented_pieces(ctypes.byref(prob), nseg))


def segmented_plan(prob: Problem, nseg: int = 1):
    """(P, chunks of piece 0, chunks of each later piece) of the segmented forward's piece plan
    on the current device ((0, 0, 0): invalid)."""
    first, rest = ctypes.c_int(0), ctypes.c_int(0)
    P = lib().gdn_segmented_plan(ctypes.byref(prob), nseg, ctypes.byref(first), ctypes.byref(rest))
    return int(P), int(first.value), int(rest.value)


def alloc_workspace(prob: Problem, nseg: int = 1, device="cuda"):
    """A zeroed workspace tensor of the size the library asks for (torch owns the memory)."""
    import torch
    n = workspace_bytes(prob, nseg)
    if n == 0:
        raise GdnError(2, "gdn_workspace_bytes")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def gdn_chunk_fwd(q, k, v, g, beta, h0, o, h_final, workspace, stream=None, prob=None):
    prob = prob or problem(k, v, o, g=g)
    _check(lib().gdn_chunk_fwd(ctypes.byref(prob), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                               _ptr(beta), _ptr(h0), _ptr(o), _ptr(h_final), _ptr(workspace),
                               workspace.numel() if workspace is not None else 0,
                               _stream(stream)), "gdn_chunk_fwd")


def gdn_segment_summary(k, v, g, beta, M, S, nseg, workspace, stream=None, prob=None):
    prob = prob or problem(k, v, g=g)
    _check(lib().gdn_segment_summary(ctypes.byref(prob), nseg, _ptr(k), _ptr(v), _ptr(g),
                                     _ptr(beta), _ptr(M), _ptr(S), _ptr(workspace),
                                     workspace.numel() if workspace is not None else 0,
                                     _stream(stream)), "gdn_segment_summary")


def gdn_summary_scan(M, S, h0, H_in, stream=None, prob=None):
    nseg, B, H, K, V = H_in.shape
    prob = prob or Problem(B, 0, H, K, V, 64, GDN_DTYPE_F32, GDN_DTYPE_F32)
    _check(lib().gdn_summary_scan(ctypes.byref(prob), nseg, _ptr(M), _ptr(S), _ptr(h0),
                                  _ptr(H_in), _stream(stream)), "gdn_summary_scan")


def gdn_segment_fwd(q, k, v, g, beta, H_in, o, h_final, nseg, workspace, stream=None,
                    prob=None):
    """The chunked forward of each of nseg segments from H_in[s] (None: zero states);
    workspace sized by workspace_bytes(prob, 1)."""
    prob = prob or problem(k, v, o, g=g)
    _check(lib().gdn_segment_fwd(ctypes.byref(prob), nseg, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                 _ptr(beta), _ptr(H_in), _ptr(o), _ptr(h_final), _ptr(workspace),
                                 workspace.numel() if workspace is not None else 0,
                                 _stream(stream)), "gdn_segment_fwd")


def gdn_segmented_fwd(q, k, v, g, beta, h0, o, h_final, nseg, workspace, H_in=None,
                      stream=None, prob=None):
    prob = prob or problem(k, v, o, g=g)
    _check(lib().gdn_segmented_fwd(ctypes.byref(prob), nseg, _ptr(q), _ptr(k), _ptr(v),
                                   _ptr(g), _ptr(beta), _ptr(h0), _ptr(o), _ptr(h_final),
                                   _ptr(H_in), _ptr(workspace),
                                   workspace.numel() if workspace is not None else 0,
                                   _stream(stream)), "gdn_segmented_fwd")


def gdn_segmented_fwd_timed(q, k, v, g, beta, h0, o, h_final, nseg, workspace, events,
                            H_in=None, stream=None, prob=None):
    """gdn_segmented_fwd recording five torch.cuda.Event (enable_timing=True) around its
    four stages: before the WY factors, before the first phase (piece 0's forward beside the
    piece summaries), before the scan, before the second phase (the forward of pieces
    1..P-1), after it."""
    prob = prob or problem(k, v, o, g=g)
    if len(events) != 5:
        raise ValueError("gdn_segmented_fwd_timed takes five events")
    arr = (_P * 5)(*[e.cuda_event for e in events])
    _check(lib().gdn_segmented_fwd_timed(ctypes.byref(prob), nseg, _ptr(q), _ptr(k), _ptr(v),
                                         _ptr(g), _ptr(beta), _ptr(h0), _ptr(o),
                                         _ptr(h_final), _ptr(H_in), _ptr(workspace),
                                         workspace.numel() if workspace is not None else 0,
                                         _stream(stream), arr), "gdn_segmented_fwd_timed")


def gdn_segmented_fwd_noalloc(q, k, v, g, beta, h0, o, h_final, nseg, device_error=None,
                              stream=None, prob=None):
    """gdn_segmented_fwd with the library's fixed scratch array instead of a workspace.
    device_error: optional int32/uint32 CUDA tensor of >= 2 elements that receives the
    call's device error word {code, detail}."""
    prob = prob or problem(k, v, o, g=g)
    _check(lib().gdn_segmented_fwd_noalloc(ctypes.byref(prob), nseg, _ptr(q), _ptr(k), _ptr(v),
                                           _ptr(g), _ptr(beta), _ptr(h0), _ptr(o),
                                           _ptr(h_final), _ptr(device_error), _stream(stream)),
           "gdn_segmented_fwd_noalloc")


def varlen_workspace_bytes(prob: Problem, nseq: int) -> int:
    return int(lib().gdn_varlen_workspace_bytes(ctypes.byref(prob), nseq))


def alloc_varlen_workspace(prob: Problem, nseq: int, device="cuda"):
    """A zeroed workspace tensor for gdn_varlen_fwd (torch owns the memory)."""
    import torch
    n = varlen_workspace_bytes(prob, nseq)
    if n == 0:
        raise GdnError(2, "gdn_varlen_workspace_bytes")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def gdn_varlen_fwd(q, k, v, g, beta, h0, o, h_final, cu_seqlens, workspace, stream=None,
                   prob=None):
    """Packed variable-length forward: q, k, v, g, beta, o hold [1, T, H, *] tokens of
    nseq = len(cu_seqlens) - 1 sequences; cu_seqlens is an int32 CUDA tensor; h0 and h_final
    are [nseq, H, K, V] fp32 (or None)."""
    prob = prob or problem(k, v, o, g=g)
    nseq = int(cu_seqlens.numel()) - 1
    _check(lib().gdn_varlen_fwd(ctypes.byref(prob), nseq, _ptr(cu_seqlens), _ptr(q), _ptr(k),
                                _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(o), _ptr(h_final),
                                _ptr(workspace), workspace.numel() if workspace is not None else 0,
                                _stream(stream)), "gdn_varlen_fwd")


def gdn_varlen_fwd_timed(q, k, v, g, beta, h0, o, h_final, cu_seqlens, workspace, events,
                         stream=None, prob=None):
    """gdn_varlen_fwd recording five torch.cuda.Event (enable_timing=True): before the length
    check, the plan and the WY factors; before the first phase (the whole forward when no
    sequence is cut); before the scan; before the second phase; after it."""
    prob = prob or problem(k, v, o, g=g)
    if len(events) != 5:
        raise ValueError("gdn_varlen_fwd_timed takes five events")
    arr = (_P * 5)(*[e.cuda_event for e in events])
    nseq = int(cu_seqlens.numel()) - 1
    _check(lib().gdn_varlen_fwd_timed(ctypes.byref(prob), nseq, _ptr(cu_seqlens), _ptr(q),
                                      _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(h0), _ptr(o),
                                      _ptr(h_final), _ptr(workspace),
                                      workspace.numel() if workspace is not None else 0,
                                      _stream(stream), arr), "gdn_varlen_fwd_timed")


def gdn_state_grad_summary(q, k, g, beta, dO, dS, nseg, dH_end=None, stream=None, prob=None):
    """Per-segment state gradients: dS [nseg,B,H,K,V] fp32 receives the gradient on the state
    entering each segment of its outputs' loss (sum dO . o) plus <dH_end[s], state leaving
    it> (dH_end None = 0). dO carries the output dtype (fp32 or bf16)."""
    prob = prob or problem(k, dO, dO, g=g)   # a [B,T,H,K] g sets gate_k: rejected below
    _check(lib().gdn_state_grad_summary(ctypes.byref(prob), nseg, _ptr(q), _ptr(k), _ptr(g),
                                        _ptr(beta), _ptr(dO), _ptr(dH_end), _ptr(dS),
                                        _stream(stream)), "gdn_state_grad_summary")


def gdn_state_grad_scan(M, dS, dht, dH_in, stream=None, prob=None):
    """Reverse scan: dH_in[s] = M[s]^T dH_in[s+1] + dS[s] with dH_in[nseg] = dht (None = 0)."""
    nseg, B, H, K, V = dH_in.shape
    prob = prob or Problem(B, 0, H, K, V, 64, GDN_DTYPE_F32, GDN_DTYPE_F32)
    _check(lib().gdn_state_grad_scan(ctypes.byref(prob), nseg, _ptr(M), _ptr(dS), _ptr(dht),
                                     _ptr(dH_in), _stream(stream)), "gdn_state_grad_scan")


def chunk_bwd_workspace_bytes(prob: Problem, nseg: int = 1) -> int:
    return int(lib().gdn_chunk_bwd_workspace_bytes(ctypes.byref(prob), nseg))


def alloc_bwd_workspace(prob: Problem, nseg: int = 1, device="cuda"):
    """A zeroed workspace tensor for gdn_chunk_bwd (torch owns the memory)."""
    import torch
    n = chunk_bwd_workspace_bytes(prob, nseg)
    if n == 0:
        raise GdnError(2, "gdn_chunk_bwd_workspace_bytes")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def gdn_chunk_bwd(q, k, v, g, beta, h0, dO, dht, dq, dk, dv, dg, dbeta, dh0, nseg, workspace,
                  stream=None, prob=None):
    """The backward: fp32 gradients dq, dk [B,T,H,K], dv [B,T,H,V], dg, dbeta [B,T,H] and dh0
    [B,H,K,V] (None skips it) of sum(dO . o) + <dht, h_final>; dO has the output dtype, dht
    (fp32, or None) the state's shape."""
    prob = prob or problem(k, v, dO, g=g)
    _check(lib().gdn_chunk_bwd(ctypes.byref(prob), nseg, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                               _ptr(beta), _ptr(h0), _ptr(dO), _ptr(dht), _ptr(dq), _ptr(dk),
                               _ptr(dv), _ptr(dg), _ptr(dbeta), _ptr(dh0), _ptr(workspace),
                               workspace.numel() if workspace is not None else 0,
                               _stream(stream)), "gdn_chunk_bwd")


def gdn_chunk_bwd_timed(q, k, v, g, beta, h0, dO, dht, dq, dk, dv, dg, dbeta, dh0, nseg,
                        workspace, events, stream=None, prob=None):
    """gdn_chunk_bwd with six torch.cuda.Event markers recorded between its steps."""
    if len(events) != 6:
        raise ValueError("gdn_chunk_bwd_timed takes six events")
    prob = prob or problem(k, v, dO, g=g)
    arr = (_P * 6)(*[e.cuda_event for e in events])
    _check(lib().gdn_chunk_bwd_timed(ctypes.byref(prob), nseg, _ptr(q), _ptr(k), _ptr(v),
                                     _ptr(g), _ptr(beta), _ptr(h0), _ptr(dO), _ptr(dht),
                                     _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dg), _ptr(dbeta),
                                     _ptr(dh0), _ptr(workspace),
                                     workspace.numel() if workspace is not None else 0,
                                     _stream(stream), arr), "gdn_chunk_bwd_timed")


def gdn_selftest_wait_timeout(workspace, limit_cycles, stream=None):
    """Launches the bounded-wait self-test (a wait that runs out after limit_cycles SM cycles
    and records GDN_ERR_TIMEOUT in the workspace's error word); read it with
    gdn_check_device_error."""
    _check(lib().gdn_selftest_wait_timeout(_ptr(workspace), int(limit_cycles), _stream(stream)),
           "gdn_selftest_wait_timeout")


def gdn_check_device_error(workspace, stream=None):
    """Synchronises, returns (status, detail) from the workspace's device error word."""
    detail = ctypes.c_uint(0)
    st = lib().gdn_check_device_error(_ptr(workspace), _stream(stream), ctypes.byref(detail))
    return int(st), int(detail.value)
