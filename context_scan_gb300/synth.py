"""Seeded synthetic inputs for the gated delta rule.

This module draws inputs and nothing else: it holds none of the recurrence's arithmetic.
Both the CUDA path's harness and the fp64 oracle's tests take their inputs from here, so
both sides see bit-identical values.

Distributions follow the workloads described on the pages (head dim 128, chunk 64,
BF16 q/k/v/beta as in "RFC: HyperParallel Linear Attention Context Parallel", section 8):
q and k are N(0,1) draws L2-normalised per (token, head) -- the normalisation the
surrounding GDN layer applies before the recurrence (RFC, section 6.4.2
"forward_prepare: Q/K norm") -- v ~ N(0,1), g = log(sigmoid(N(mu, sd))) (a natural-log
decay, so exp(g) is in (0, 1)), beta = sigmoid(N(mu, sd)), h0 ~ N(0, sd) in fp32.
N(mu, sd) takes sd as the standard deviation.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csrc", "synth.c")
_LIB_DIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIB_DIR, "libgdn_synth.so")

TENSOR_IDS = {"q": 1, "k": 2, "v": 3, "g": 4, "beta": 5, "h0": 6, "dO": 7, "dht": 8}
KIND_NORMAL, KIND_UNIT, KIND_LOGSIGMOID, KIND_SIGMOID = 0, 1, 2, 3


def build_synth(force: bool = False) -> str:
    """Compile the generator's shared library (gcc, host code only)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                               _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build_synth())
        lib.synth_fill.restype = ctypes.c_int
        lib.synth_fill.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_long, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_double,
                                   ctypes.c_int, ctypes.c_void_p, ctypes.c_int]
        _lib = lib
    return _lib


def fill(seed: int, name: str, shape, kind: int, mu: float = 0.0, sd: float = 1.0,
         bf16: bool = False, group: int = 0, nthreads: int = 0) -> np.ndarray:
    """Draw one tensor. Row = product of all dims but the last two for 4-d tensors
    ([B,T,H,K] -> rows of H*K); for [B,T,H] and [B,H,K,V] see the callers."""
    out = np.empty(shape, dtype=np.float32)
    if out.size == 0:
        return out
    n_rows = int(np.prod(shape[:2])) if len(shape) >= 2 else 1
    row_len = int(out.size // max(n_rows, 1))
    rc = _load().synth_fill(ctypes.c_uint64(seed & 0xFFFFFFFFFFFFFFFF), TENSOR_IDS[name], n_rows,
                            row_len, group, kind, mu, sd, 1 if bf16 else 0,
                            out.ctypes.data, nthreads)
    if rc != 0:
        raise ValueError(f"synth_fill rejected its arguments for {name} {shape}")
    return out


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: shapes, storage dtype and the input distributions."""
    name: str
    B: int
    H: int
    T: int
    K: int
    V: int
    nseg: int
    in_dtype: str              # "f32" or "bf16": storage type of q, k, v, g, beta
    g_mu: float
    g_sd: float
    beta_mu: float
    beta_sd: float
    h0_sd: float | None        # None: h0 = 0 (no initial state passed)
    seed: int
    per_sequence_seed: int | None = None   # if set, batch b uses seed per_sequence_seed + b
    # packed variable-length sequences: B == 1, T == sum(seq_lens), one initial state per
    # sequence (h0 is [len(seq_lens), H, K, V])
    seq_lens: tuple | None = None
    # one gate per key channel (g is [B, T, H, K], each entry log(sigmoid(N(g_mu, g_sd))))
    gate_k: bool = False
    chunk: int = 64
    notes: str = field(default="", compare=False)

    @property
    def seg_len(self) -> int:
        return self.T // self.nseg

    @property
    def tokens(self) -> int:
        return self.B * self.T


WORKLOADS = {
    w.name: w for w in [
        Workload("tiny_f32_k64_cp4", B=1, H=2, T=256, K=64, V=64, nseg=4, in_dtype="f32",
                 g_mu=2, g_sd=1, beta_mu=0, beta_sd=1, h0_sd=0.1, seed=0x6D6E0000,
                 notes="fp32 throughout; oracle finishes in well under a second"),
        Workload("single_seg_h16_t8k", B=1, H=16, T=8192, K=128, V=128, nseg=1, in_dtype="bf16",
                 g_mu=2, g_sd=1, beta_mu=0, beta_sd=1, h0_sd=None, seed=0x6D6E0001),
        Workload("cp4_b2_h32_t32k", B=2, H=32, T=32768, K=128, V=128, nseg=4, in_dtype="bf16",
                 g_mu=2, g_sd=1, beta_mu=0, beta_sd=1, h0_sd=0.1, seed=0x6D6E0002,
                 notes="the headline workload"),
        Workload("cp16_h16_t128k", B=1, H=16, T=131072, K=128, V=128, nseg=16, in_dtype="bf16",
                 g_mu=4, g_sd=1, beta_mu=0, beta_sd=1, h0_sd=None, seed=0x6D6E0003),
        Workload("cp2_b16_h32_t4k", B=16, H=32, T=4096, K=128, V=128, nseg=2, in_dtype="bf16",
                 g_mu=1, g_sd=2, beta_mu=0, beta_sd=2, h0_sd=0.1, seed=0x6D6E0004,
                 per_sequence_seed=0x6D6E0400),
        Workload("slow_decay_h4_t1k_cp16", B=1, H=4, T=1024, K=128, V=128, nseg=16,
                 in_dtype="bf16", g_mu=6, g_sd=1, beta_mu=-2, beta_sd=1, h0_sd=0.1,
                 seed=0x6D6E0005,
                 notes="summary M stays O(0.1-1): exercises the compose path numerically"),
        Workload("kda_h16_t8k", B=1, H=16, T=8192, K=128, V=128, nseg=1, in_dtype="bf16",
                 g_mu=3, g_sd=1, beta_mu=0, beta_sd=1, h0_sd=0.1, seed=0x6D6E0007, gate_k=True,
                 notes="per-channel gates at the shape of the KDA design page's measurements"),
        Workload("varlen5_h16_t7300", B=1, H=16, T=7300, K=128, V=128, nseg=1, in_dtype="bf16",
                 g_mu=2, g_sd=1, beta_mu=0, beta_sd=1, h0_sd=0.1, seed=0x6D6E0006,
                 seq_lens=(1800, 1500, 2000, 1200, 800),
                 notes="five packed sequences of the lengths the KDA design page measures"),
        Workload("varlen8_h16_t32k", B=1, H=16, T=32640, K=128, V=128, nseg=1, in_dtype="bf16",
                 g_mu=2, g_sd=1, beta_mu=0, beta_sd=1, h0_sd=0.1, seed=0x6D6E0008,
                 seq_lens=(16384, 8192, 4096, 2048, 1024, 512, 256, 128),
                 notes="a packed batch whose longest sequence (16K) sets the time unless it is "
                       "cut into pieces; halving lengths as in a length-bucketed batch"),
    ]
}


def cu_seqlens(w: Workload) -> np.ndarray:
    """Sequence starts of a packed workload: [0, l0, l0+l1, ..., T] as int32."""
    if w.seq_lens is None:
        raise ValueError(f"{w.name} is not a packed variable-length workload")
    return np.concatenate([[0], np.cumsum(w.seq_lens)]).astype(np.int32)


def scaled(w: Workload, **changes) -> Workload:
    """A copy of a workload with some fields changed (e.g. a shorter T for a CPU test)."""
    d = {f: getattr(w, f) for f in w.__dataclass_fields__}
    d.update(changes)
    return Workload(**d)


def make_inputs(w: Workload, nthreads: int = 0) -> dict:
    """Draw q, k, v, g, beta (and h0 if the workload has one) as float32 numpy arrays.

    With in_dtype == "bf16" every value is exactly representable in bf16, so converting
    the arrays to bf16 loses nothing. h0 is always fp32 (the state is fp32).
    """
    bf16 = w.in_dtype == "bf16"
    if w.seq_lens is not None and (w.B != 1 or sum(w.seq_lens) != w.T or min(w.seq_lens) < 0):
        raise ValueError(f"{w.name}: packed sequences need B == 1 and T == sum(seq_lens)")
    n_states = len(w.seq_lens) if w.seq_lens is not None else None
    seeds = ([w.per_sequence_seed + b for b in range(w.B)] if w.per_sequence_seed is not None
             else [w.seed])
    per_b = w.per_sequence_seed is not None
    Bd = 1 if per_b else w.B
    parts = {n: [] for n in ("q", "k", "v", "g", "beta", "h0")}
    for s in seeds:
        parts["q"].append(fill(s, "q", (Bd, w.T, w.H, w.K), KIND_UNIT, bf16=bf16, group=w.K,
                               nthreads=nthreads))
        parts["k"].append(fill(s, "k", (Bd, w.T, w.H, w.K), KIND_UNIT, bf16=bf16, group=w.K,
                               nthreads=nthreads))
        parts["v"].append(fill(s, "v", (Bd, w.T, w.H, w.V), KIND_NORMAL, 0.0, 1.0, bf16=bf16,
                               nthreads=nthreads))
        gshape = (Bd, w.T, w.H, w.K) if w.gate_k else (Bd, w.T, w.H)
        parts["g"].append(fill(s, "g", gshape, KIND_LOGSIGMOID, w.g_mu, w.g_sd,
                               bf16=bf16, nthreads=nthreads))
        parts["beta"].append(fill(s, "beta", (Bd, w.T, w.H), KIND_SIGMOID, w.beta_mu, w.beta_sd,
                                  bf16=bf16, nthreads=nthreads))
        if w.h0_sd is not None:
            parts["h0"].append(fill(s, "h0", (n_states or Bd, w.H, w.K, w.V), KIND_NORMAL, 0.0,
                                    w.h0_sd, bf16=False, nthreads=nthreads))
    out = {n: (np.concatenate(p, axis=0) if len(p) > 1 else p[0]) for n, p in parts.items() if p}
    if w.h0_sd is None:
        out["h0"] = None
    return out


def make_grads(w: Workload, bf16_out: bool = False, dht_sd=None, nthreads: int = 0) -> dict:
    """The backward's incoming gradients for workload w: dO [B,T,H,V] ~ N(0, 1) (rounded to
    bf16 when the output is bf16) and, when dht_sd is given, dht [B,H,K,V] ~ N(0, dht_sd)
    (fp32, like the state); drawn from the workload's seed with their own tensor ids."""
    dO = fill(w.seed, "dO", (w.B, w.T, w.H, w.V), KIND_NORMAL, 0.0, 1.0, bf16=bf16_out,
              nthreads=nthreads)
    dht = None
    if dht_sd is not None:
        dht = fill(w.seed, "dht", (w.B, w.H, w.K, w.V), KIND_NORMAL, 0.0, dht_sd, bf16=False,
                   nthreads=nthreads)
    return {"dO": dO, "dht": dht}
