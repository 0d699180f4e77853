"""The C-ABI library loads, exports every entry point include/gdn.h declares, and its host
validation rejects bad problems before touching a GPU (no compute call runs here)."""
import ctypes
import os
import re
import subprocess

import pytest

from context_scan_gb300 import _build, gdn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    _build.build_cuda()
    return gdn.lib()


def declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"GDN_API\s+[\w\s\*]+?\b(gdn_\w+)\s*\(", text))
    return names


def test_exports_every_declared_symbol(L):
    declared = declared_symbols()
    assert {"gdn_chunk_fwd", "gdn_segment_summary", "gdn_summary_scan",
            "gdn_segmented_fwd"} <= declared
    out = subprocess.run(["nm", "-D", "--defined-only", gdn.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (gdn_\w+)", out))
    assert declared <= exported, declared - exported
    for name in declared:
        assert hasattr(L, name)
    assert set(gdn.EXPORTED) <= declared


def test_binding_arity_matches_header(L):
    text = "".join(open(os.path.join(ROOT, "include", f)).read()
                   for f in os.listdir(os.path.join(ROOT, "include")) if f.endswith(".h"))
    for m in re.finditer(r"GDN_API\s+[\w\s\*]+?\b(gdn_\w+)\s*\(([^)]*)\)", text):
        name, params = m.group(1), m.group(2)
        n = 0 if params.strip() in ("", "void") else params.count(",") + 1
        assert len(getattr(L, name).argtypes) == n, (name, n)


def test_library_is_sm103a_only():
    flags = " ".join(_build.NVCC_FLAGS)
    assert "arch=compute_103a,code=sm_103a" in flags
    assert flags.count("-gencode") == 1


def P(**kw):
    d = dict(B=1, T=128, H=2, K=128, V=128, chunk=64, in_dtype=1, out_dtype=0)
    d.update(kw)
    return gdn.Problem(**{k: d[k] for k in ("B", "T", "H", "K", "V", "chunk", "in_dtype",
                                             "out_dtype", "decay_first", "gate_k") if k in d})


def test_workspace_bytes_and_status_strings(L):
    p = P(B=2, T=32768, H=32)
    # bf16, K = V = 128: the error word and a WY tile pair of 10 KiB per chunk of each head
    # (the two 64 x 64 bf16 factors without their zero blocks above the diagonal)
    wy = 64 * (32768 // 64) * 10240
    assert L.gdn_workspace_bytes(ctypes.byref(p), 1) == 256 + wy
    # without a current device the planner keeps one piece per segment
    assert L.gdn_segmented_pieces(ctypes.byref(p), 1) == 1
    assert L.gdn_segmented_pieces(ctypes.byref(p), 4) == 4
    assert L.gdn_segmented_pieces(ctypes.byref(P(T=100)), 1) == 0
    n4 = L.gdn_workspace_bytes(ctypes.byref(p), 4)
    # plus, for P = 4 pieces of 64 heads in fp32: M and S of the piece summaries and the state
    # entering each piece
    assert n4 == 256 + wy + 4 * 64 * 128 * 128 * 4 * (1 + 1 + 1)
    # two pieces need no summaries, only the state entering each piece
    n2 = L.gdn_workspace_bytes(ctypes.byref(p), 2)
    assert n2 == 256 + wy + 2 * 64 * 128 * 128 * 4
    # the CUDA-core shapes need no WY tiles
    assert L.gdn_workspace_bytes(ctypes.byref(P(B=2, T=32768, H=32, in_dtype=0)), 1) == 256
    assert L.gdn_workspace_bytes(ctypes.byref(P(B=2, T=32768, H=32, K=64, V=64)), 1) == 256
    assert L.gdn_workspace_bytes(ctypes.byref(P(K=96, V=96)), 1) == 0
    assert L.gdn_workspace_bytes(ctypes.byref(P(T=100)), 1) == 0
    assert L.gdn_workspace_bytes(ctypes.byref(P(T=128)), 4) == 0   # 128 % (64*4) != 0
    for code in range(9):
        assert L.gdn_status_string(code)
    assert L.gdn_status_string(0) == b"ok"


@pytest.mark.parametrize("prob,nseg,expect", [
    (dict(chunk=32), 1, 2),
    (dict(K=128, V=64), 1, 2),
    (dict(K=256, V=256), 1, 2),
    (dict(T=100), 1, 2),
    (dict(T=192), 2, 2),
    (dict(B=0), 1, 1),
    (dict(T=-64), 1, 1),
    (dict(in_dtype=7), 1, 3),
    (dict(out_dtype=5), 1, 3),
    (dict(), 0, 1),
])
def test_validation_rejects_before_launch(L, prob, nseg, expect):
    p = P(**prob)
    # all pointers NULL: every rejection here happens before pointers are examined or used
    st = L.gdn_segmented_fwd(ctypes.byref(p), nseg, *([None] * 10), 0, None)
    assert st == expect, gdn.STATUS.get(st)


def test_null_pointers_and_missing_workspace_rejected(L):
    p = P()
    st = L.gdn_chunk_fwd(ctypes.byref(p), *([None] * 9), 0, None)
    assert st == 1  # q/k/v/g/beta/o missing
    st = L.gdn_segment_summary(ctypes.byref(p), 1, *([None] * 7), 0, None)
    assert st == 1  # M/S missing
    st = L.gdn_summary_scan(ctypes.byref(p), 2, None, None, None, None, None)
    assert st == 1
    st = L.gdn_check_device_error(None, None, None)
    assert st == 5


def test_varlen_workspace_and_validation(L):
    # packed sequences: B == 1, any T; the WY tiles of at most T/64 + nseq chunks per head,
    # then two int32 arrays of nseq + 1 (each region 256-byte aligned)
    p = P(B=1, T=7300, H=16)
    wy = 16 * (7300 // 64 + 5) * 10240

    def rup(n):
        return (n + 255) // 256 * 256

    def pieces(nseq, H):
        # the piece plan (tcgen05 shapes): three tables of 8-int entries (nseq, e_max, e_max),
        # eight counts, four ints per sequence, then fp32 states, M and S for e_max = 256 / H
        # pieces past the first ones
        e = max(1, 256 // H)
        return (rup(32 * nseq) + 2 * rup(32 * e) + rup(32) + rup(16 * nseq) +
                3 * rup(4 * e * H * 128 * 128))

    assert L.gdn_varlen_workspace_bytes(ctypes.byref(p), 5) == 256 + wy + 256 + 256 + pieces(5, 16)
    assert L.gdn_varlen_workspace_bytes(ctypes.byref(P(B=1, T=7300, H=16, in_dtype=0)), 5) == 768
    assert L.gdn_varlen_workspace_bytes(ctypes.byref(P(B=1, T=0)), 1) == (256 + 2 * 10240 + 512 +
                                                                          pieces(1, 2))
    assert L.gdn_varlen_workspace_bytes(ctypes.byref(P(B=2, T=7300)), 5) == 0   # B must be 1
    assert L.gdn_varlen_workspace_bytes(ctypes.byref(p), 0) == 0
    assert L.gdn_varlen_workspace_bytes(ctypes.byref(P(B=1, K=96, V=96)), 1) == 0
    # rejections before any pointer is used
    assert L.gdn_varlen_fwd(ctypes.byref(P(B=2)), 1, *([None] * 10), 0, None) == 1
    assert L.gdn_varlen_fwd(ctypes.byref(P(B=1, chunk=32)), 1, *([None] * 10), 0, None) == 2
    assert L.gdn_varlen_fwd(ctypes.byref(P(B=1)), 1, *([None] * 10), 0, None) == 1   # no cu_seqlens


def test_state_grad_validation(L):
    # the backward's state-gradient entry points reject bad problems before any launch
    S, C = L.gdn_state_grad_summary, L.gdn_state_grad_scan
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: every case fails validation first
    odd = ctypes.c_void_p((1 << 20) + 8)
    args = [fake] * 5 + [None, fake, None]
    assert S(ctypes.byref(P(T=100)), 1, *args) == 2
    assert S(ctypes.byref(P(T=128)), 4, *args) == 2               # T % (64 nseg)
    assert S(ctypes.byref(P(K=96, V=96)), 1, *args) == 2
    assert S(ctypes.byref(P(gate_k=1)), 1, *args) == 2            # per-channel gates
    assert S(ctypes.byref(P(in_dtype=4)), 1, *args) == 3
    assert S(ctypes.byref(P()), 0, *args) == 1
    assert S(ctypes.byref(P()), 1, *([fake] * 5), None, None, None) == 1      # no dS
    assert S(ctypes.byref(P()), 1, None, *([fake] * 4), None, fake, None) == 1   # no q
    assert S(ctypes.byref(P()), 1, *([fake] * 4), odd, None, fake, None) == 4    # dO misaligned
    assert C(ctypes.byref(P()), 2, None, fake, None, fake, None) == 1            # no M
    assert C(ctypes.byref(P(K=64, V=128)), 2, fake, fake, None, fake, None) == 2
    assert C(ctypes.byref(P()), 0, fake, fake, None, fake, None) == 1
    assert C(ctypes.byref(P()), 2, fake, fake, odd, fake, None) == 4             # dht misaligned


def test_state_grad_binding_rejects_per_channel_gates(L):
    # the binding describes g's layout to the library: per-channel gates [B,T,H,K] are
    # refused (GDN_ERR_UNSUPPORTED_SHAPE) before any pointer is used, never read as [B,T,H]
    import torch
    B, T, H, K = 1, 64, 2, 64
    q = torch.zeros((B, T, H, K))
    g4 = torch.zeros((B, T, H, K))
    beta = torch.zeros((B, T, H))
    dO = torch.zeros((B, T, H, K))
    dS = torch.zeros((1, B, H, K, K))
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_state_grad_summary(q, q, g4, beta, dO, dS, 1, stream=0)
    assert e.value.status == 2
