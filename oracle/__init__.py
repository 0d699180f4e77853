"""fp64 CPU oracle for the gated delta rule -- TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package. The CUDA library never uses it and it never uses the CUDA library:
the two share no code. Inputs come from the seeded generator module, which both sides use.

The arithmetic lives in ``oracle.c`` (plain C, fp64, one thread per (b, h, column block)).
This file only compiles it on first use and marshals numpy arrays in and out.

What each function computes (pages cited by title and section):
  recurrence      -- the per-token recurrence of "RFC: HyperParallel Linear Attention
                     Context Parallel", section 2.1: residual_t = beta_t (v_t - k_t @ H),
                     H <- exp(g_t) H + outer(k_t, residual_t), o_t = q_t @ H.
  summary         -- the per-segment affine summary H_out = M @ H_in + S (RFC 2.2), built
                     token by token in rank-1 form from M = I, S = 0.
  compose / scan  -- M = M1 @ M0, S = M1 @ S0 + S1 (RFC 2.2; "Context Parallelism in ART",
                     section 08 "Then parallelize across GPUs"), scanned exclusively in
                     segment order from h0.
  varlen_recurrence -- packed variable-length sequences ("KDA Chunk Backward -- TPU/Pallas
                     Kernel Design", section 3.8): each sequence of the packed token axis
                     runs the recurrence alone from its own initial state.
  kda_recurrence / kda_summary -- per-channel gates ("KDA Chunk Backward -- TPU/Pallas Kernel
                     Design", section 1.2): g is [B,T,H,K] and the state decays row by row,
                     diag(exp(g_t)); written apart from the scalar-gate functions, which
                     it must reproduce when every channel carries the same gate.
  backward        -- the gradients of L = sum_t do_t . o_t + <dht, h_final> with respect to
                     q, k, v, g, beta and h0 (RFC section 6.4.3, the reverse flow ending in
                     dQ/dK/dV/dg/dbeta; "KDA Chunk Backward -- TPU/Pallas Kernel Design",
                     section 1), token by token backwards over recomputed states.
  state_grad_summary -- dS_local of each segment (RFC 6.4.3): the gradient reaching the
                     state entering the segment from its own outputs, rank-1 per token.
  state_grad_scan -- dH_in[s] = M[s]^T dH_in[s+1] + dS[s] from dH_in[nseg] = dht (RFC 6.4.3).
  chunked_bwd.chunked_backward -- (module oracle/chunked_bwd.py, numpy) the same gradients in the
                     chunk form a chunked GPU backward computes; used only to pin
                     chunked == per-token and to expose the chunk intermediates.
  chunked_fwd / chunked_summary -- the chunk equations of "Context Parallelism in ART",
                     section 08 "First parallelize within a GPU", restated for the RFC's
                     un-decayed read; used only to pin chunked == per-token.

Pins: every function here is checked against closed forms, brute force on tiny inputs and
invariants in tests/test_oracle.py (no function is "parity unpinned").
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "liboracle.so")


def build(force: bool = False) -> str:
    os.makedirs(_LIB_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.oracle_recurrence.argtypes = [_I] * 6 + [_P] * 9 + [_I, _I, _I]
        lib.oracle_summary.argtypes = [_I] * 6 + [_P] * 6 + [_I, _I]
        lib.oracle_compose.argtypes = [_I, _I] + [_P] * 6
        lib.oracle_scan.argtypes = [_I] * 4 + [_P] * 4
        lib.oracle_chunked_fwd.argtypes = [_I] * 6 + [_P] * 8 + [_I, _I]
        lib.oracle_chunked_summary.argtypes = [_I] * 7 + [_P] * 6 + [_I, _I]
        lib.oracle_kda_recurrence.argtypes = [_I] * 6 + [_P] * 9 + [_I, _I, _I]
        lib.oracle_kda_summary.argtypes = [_I] * 6 + [_P] * 6 + [_I, _I]
        lib.oracle_backward.argtypes = [_I] * 5 + [_P] * 14 + [_I, _I]
        lib.oracle_state_grad_summary.argtypes = [_I] * 6 + [_P] * 7 + [_I, _I]
        lib.oracle_state_grad_scan.argtypes = [_I] * 4 + [_P] * 4
        lib.oracle_num_threads.argtypes = [_I]
        lib.oracle_num_threads.restype = _I
        for fn in ("oracle_recurrence", "oracle_summary", "oracle_compose", "oracle_scan",
                   "oracle_chunked_fwd", "oracle_chunked_summary", "oracle_kda_recurrence",
                   "oracle_kda_summary", "oracle_backward", "oracle_state_grad_summary",
                   "oracle_state_grad_scan"):
            getattr(lib, fn).restype = None
        _lib = lib
    return _lib


def _f32(x):
    if x is None:
        return None
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


def _f64(x):
    if x is None:
        return None
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data


def num_threads(nthreads: int = 0) -> int:
    return _load().oracle_num_threads(nthreads)


def recurrence(q, k, v, g, beta, h0=None, seg_len: int = 0, col_block: int = 0,
               nthreads: int = 0, want_o: bool = True, decay_first: bool = False):
    """Per-token recurrence. Returns (o [B,T,H,V], h_final [B,H,K,V], H_in or None).

    If seg_len > 0, H_in [T//seg_len, B, H, K, V] holds the state entering each segment.
    decay_first reads exp(g_t) H_{t-1} (the other reading) instead of H_{t-1}.
    """
    q, k, v, g, beta, h0 = map(_f32, (q, k, v, g, beta, h0))
    B, T, H, K = k.shape
    V = v.shape[-1]
    o = np.empty((B, T, H, V), np.float64) if want_o else None
    hf = np.empty((B, H, K, V), np.float64)
    H_in = np.empty((T // seg_len, B, H, K, V), np.float64) if seg_len > 0 else None
    _load().oracle_recurrence(B, T, H, K, V, seg_len, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                              _ptr(beta), _ptr(h0), _ptr(o), _ptr(hf), _ptr(H_in), col_block,
                              nthreads, int(decay_first))
    return o, hf, H_in


def kda_recurrence(q, k, v, g, beta, h0=None, seg_len: int = 0, col_block: int = 0,
                   nthreads: int = 0, want_o: bool = True, decay_first: bool = False):
    """Per-token recurrence with per-channel gates g [B,T,H,K]. Returns (o [B,T,H,V],
    h_final [B,H,K,V], H_in [T//seg_len,B,H,K,V] or None)."""
    q, k, v, g, beta, h0 = map(_f32, (q, k, v, g, beta, h0))
    B, T, H, K = k.shape
    V = v.shape[-1]
    assert g.shape == (B, T, H, K)
    o = np.empty((B, T, H, V), np.float64) if want_o else None
    hf = np.empty((B, H, K, V), np.float64)
    H_in = np.empty((T // seg_len, B, H, K, V), np.float64) if seg_len > 0 else None
    _load().oracle_kda_recurrence(B, T, H, K, V, seg_len, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                  _ptr(beta), _ptr(h0), _ptr(o), _ptr(hf), _ptr(H_in),
                                  col_block, nthreads, int(decay_first))
    return o, hf, H_in


def kda_summary(k, v, g, beta, nseg: int, nthreads: int = 0, decay_first: bool = False):
    """Per-segment summaries (M [nseg,B,H,K,K], S [nseg,B,H,K,V]) with per-channel gates."""
    k, v, g, beta = map(_f32, (k, v, g, beta))
    B, T, H, K = k.shape
    V = v.shape[-1]
    assert g.shape == (B, T, H, K) and T % nseg == 0
    M = np.empty((nseg, B, H, K, K), np.float64)
    S = np.empty((nseg, B, H, K, V), np.float64)
    _load().oracle_kda_summary(B, T, H, K, V, nseg, _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                               _ptr(M), _ptr(S), nthreads, int(decay_first))
    return M, S


def varlen_recurrence(q, k, v, g, beta, cu_seqlens, h0=None, nthreads: int = 0,
                      decay_first: bool = False):
    """Packed sequences: q, k, v, g, beta hold [1, T, H, *]; sequence s is tokens
    cu_seqlens[s] .. cu_seqlens[s+1]-1 and starts from h0[s] (zero when h0 is None); no state
    passes between sequences. Returns (o [1,T,H,V], h_final [nseq,H,K,V])."""
    cu = [int(c) for c in cu_seqlens]
    nseq = len(cu) - 1
    B, T, H, K = np.shape(k)
    V = np.shape(v)[-1]
    assert B == 1 and cu[0] == 0 and cu[-1] == T and all(a <= b for a, b in zip(cu, cu[1:]))
    o = np.zeros((1, T, H, V), np.float64)
    hf = np.empty((nseq, H, K, V), np.float64)
    for s in range(nseq):
        a, b = cu[s], cu[s + 1]
        h0_s = None if h0 is None else np.asarray(h0)[s:s + 1]
        rec = kda_recurrence if np.ndim(g) == 4 else recurrence
        o_s, hf_s, _ = rec(*(np.asarray(x)[:, a:b] for x in (q, k, v, g, beta)), h0_s,
                           nthreads=nthreads, decay_first=decay_first)
        o[:, a:b] = o_s
        hf[s] = hf_s[0]
    return o, hf


def summary(k, v, g, beta, nseg: int, nthreads: int = 0, decay_first: bool = False):
    """Per-segment summaries (M [nseg,B,H,K,K], S [nseg,B,H,K,V]), rank-1 token updates."""
    k, v, g, beta = map(_f32, (k, v, g, beta))
    B, T, H, K = k.shape
    V = v.shape[-1]
    assert T % nseg == 0
    M = np.empty((nseg, B, H, K, K), np.float64)
    S = np.empty((nseg, B, H, K, V), np.float64)
    _load().oracle_summary(B, T, H, K, V, nseg, _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                           _ptr(M), _ptr(S), nthreads, int(decay_first))
    return M, S


def compose(M1, S1, M0, S0):
    """(M0,S0) then (M1,S1): returns (M1 @ M0, M1 @ S0 + S1) for one head."""
    M1, S1, M0, S0 = map(_f64, (M1, S1, M0, S0))
    K, V = S1.shape
    M = np.empty((K, K), np.float64)
    S = np.empty((K, V), np.float64)
    _load().oracle_compose(K, V, _ptr(M1), _ptr(S1), _ptr(M0), _ptr(S0), _ptr(M), _ptr(S))
    return M, S


def scan(M, S, h0=None):
    """Exclusive in-order scan: H_in[0] = h0, H_in[s] = M[s-1] @ H_in[s-1] + S[s-1].

    M [nseg, B, H, K, K], S [nseg, B, H, K, V], h0 [B, H, K, V] or None (zero).
    """
    M, S, h0 = _f64(M), _f64(S), _f64(h0)
    nseg, B, H, K, V = S.shape
    H_in = np.empty((nseg, B, H, K, V), np.float64)
    _load().oracle_scan(nseg, B * H, K, V, _ptr(M), _ptr(S), _ptr(h0), _ptr(H_in))
    return H_in


def chunked_fwd(q, k, v, g, beta, h0=None, chunk: int = 64, nthreads: int = 0,
                decay_first: bool = False):
    q, k, v, g, beta, h0 = map(_f32, (q, k, v, g, beta, h0))
    B, T, H, K = k.shape
    V = v.shape[-1]
    o = np.empty((B, T, H, V), np.float64)
    hf = np.empty((B, H, K, V), np.float64)
    _load().oracle_chunked_fwd(B, T, H, K, V, chunk, _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                               _ptr(beta), _ptr(h0), _ptr(o), _ptr(hf), nthreads,
                               int(decay_first))
    return o, hf


def chunked_summary(k, v, g, beta, nseg: int, chunk: int = 64, nthreads: int = 0,
                    decay_first: bool = False):
    k, v, g, beta = map(_f32, (k, v, g, beta))
    B, T, H, K = k.shape
    V = v.shape[-1]
    assert T % nseg == 0
    M = np.empty((nseg, B, H, K, K), np.float64)
    S = np.empty((nseg, B, H, K, V), np.float64)
    _load().oracle_chunked_summary(B, T, H, K, V, chunk, nseg, _ptr(k), _ptr(v), _ptr(g),
                                   _ptr(beta), _ptr(M), _ptr(S), nthreads, int(decay_first))
    return M, S


def backward(q, k, v, g, beta, dO, h0=None, dht=None, nthreads: int = 0,
             decay_first: bool = False):
    """Gradients of L = sum_t do_t . o_t + <dht, h_final> (dht None = 0).

    Returns (dq [B,T,H,K], dk [B,T,H,K], dv [B,T,H,V], dg [B,T,H], dbeta [B,T,H],
    dh0 [B,H,K,V]), all fp64.
    """
    q, k, v, g, beta, h0, dO, dht = map(_f32, (q, k, v, g, beta, h0, dO, dht))
    B, T, H, K = k.shape
    V = v.shape[-1]
    dq = np.empty((B, T, H, K), np.float64)
    dk = np.empty((B, T, H, K), np.float64)
    dv = np.empty((B, T, H, V), np.float64)
    dg = np.empty((B, T, H), np.float64)
    db = np.empty((B, T, H), np.float64)
    dh0 = np.empty((B, H, K, V), np.float64)
    _load().oracle_backward(B, T, H, K, V, _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta),
                            _ptr(h0), _ptr(dO), _ptr(dht), _ptr(dq), _ptr(dk), _ptr(dv),
                            _ptr(dg), _ptr(db), _ptr(dh0), nthreads, int(decay_first))
    return dq, dk, dv, dg, db, dh0


def state_grad_summary(q, k, g, beta, dO, nseg: int, dH_end=None, nthreads: int = 0,
                       decay_first: bool = False):
    """dS [nseg,B,H,K,V]: the gradient on the state entering each segment from that
    segment's outputs, plus dH_end[s] (the gradient on the state leaving it; None = 0)
    carried back through the segment."""
    q, k, g, beta, dO = map(_f32, (q, k, g, beta, dO))
    dH_end = _f64(dH_end)
    B, T, H, K = k.shape
    V = dO.shape[-1]
    assert T % nseg == 0
    dS = np.empty((nseg, B, H, K, V), np.float64)
    _load().oracle_state_grad_summary(B, T, H, K, V, nseg, _ptr(q), _ptr(k), _ptr(g),
                                      _ptr(beta), _ptr(dO), _ptr(dH_end), _ptr(dS), nthreads,
                                      int(decay_first))
    return dS


def state_grad_scan(M, dS, dht=None):
    """Reverse scan: dH_in[s] = M[s]^T dH_in[s+1] + dS[s], dH_in[nseg] = dht (None = 0).

    M [nseg,B,H,K,K], dS [nseg,B,H,K,V], dht [B,H,K,V]. Returns dH_in [nseg,B,H,K,V].
    """
    M, dS, dht = _f64(M), _f64(dS), _f64(dht)
    nseg, B, H, K, V = dS.shape
    dH_in = np.empty((nseg, B, H, K, V), np.float64)
    _load().oracle_state_grad_scan(nseg, B * H, K, V, _ptr(M), _ptr(dS), _ptr(dht), _ptr(dH_in))
    return dH_in
