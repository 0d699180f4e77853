"""Shared helpers of the GPU parity tests: upload seeded inputs, call the C ABI through the
binding, run the oracle on the same inputs, and the tolerance metric.

Tolerance metric (per tensor): max_i |x_gpu - x_ref| / sqrt(mean(x_ref^2)).
Bars: 1e-4 for fp32 inputs; 2e-2 for bf16 inputs (fp32 outputs).
"""
import json
import os

import numpy as np
import torch

import oracle
from context_scan_gb300 import gdn, synth

TOL_F32 = 1e-4
TOL_BF16 = 2e-2


# When GDN_ERR_LOG names a file, every measured error is appended to it as one JSON line
# (the test, an optional label, the value), so a run records the margin to each bar.
ERR_LOG = os.environ.get("GDN_ERR_LOG")


def record(value, label=None):
    if ERR_LOG:
        test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
        with open(ERR_LOG, "a") as f:
            f.write(json.dumps({"test": test, "label": label, "err": value}) + "\n")
    return value


def rel_err(x, ref, label=None):
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    scale = np.sqrt(np.mean(ref * ref)) if ref.size else 0.0
    if ref.size == 0:
        return 0.0
    return record(float(np.max(np.abs(x - ref)) / max(scale, 1e-30)), label)


def tol_for(w):
    return TOL_F32 if w.in_dtype == "f32" else TOL_BF16


def upload(x, w, device="cuda"):
    dt = torch.bfloat16 if w.in_dtype == "bf16" else torch.float32
    d = {}
    for n in ("q", "k", "v", "g", "beta"):
        d[n] = torch.from_numpy(x[n]).to(device).to(dt).contiguous()
    d["h0"] = None if x["h0"] is None else torch.from_numpy(x["h0"]).to(device).contiguous()
    return d


def run_segmented(w, d, nseg=None, out_dtype=torch.float32, want_hin=True, decay_first=False):
    nseg = nseg or w.nseg
    B, T, H, K = d["k"].shape
    V = d["v"].shape[-1]
    o = torch.empty((B, T, H, V), dtype=out_dtype, device="cuda")
    hf = torch.empty((B, H, K, V), dtype=torch.float32, device="cuda")
    hin = torch.empty((nseg, B, H, K, V), dtype=torch.float32, device="cuda") if want_hin else None
    prob = gdn.problem(d["k"], d["v"], o, decay_first=decay_first, g=d["g"])
    ws = gdn.alloc_workspace(prob, nseg)
    gdn.gdn_segmented_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], o, hf, nseg, ws,
                          H_in=hin, prob=prob)
    torch.cuda.synchronize()
    st, detail = gdn.gdn_check_device_error(ws)
    assert st == 0, (st, detail)
    return o, hf, hin


def run_summary(w, d, nseg=None, decay_first=False):
    nseg = nseg or w.nseg
    B, T, H, K = d["k"].shape
    V = d["v"].shape[-1]
    M = torch.empty((nseg, B, H, K, K), dtype=torch.float32, device="cuda")
    S = torch.empty((nseg, B, H, K, V), dtype=torch.float32, device="cuda")
    prob = gdn.problem(d["k"], d["v"], decay_first=decay_first, g=d["g"])
    ws = gdn.alloc_workspace(prob, 1)
    gdn.gdn_segment_summary(d["k"], d["v"], d["g"], d["beta"], M, S, nseg, ws, prob=prob)
    torch.cuda.synchronize()
    assert gdn.gdn_check_device_error(ws)[0] == 0
    return M, S


def np64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def head_slice(x, b, h):
    """Inputs of one (b, h) head as a B=1, H=1 problem."""
    out = {}
    for n in ("q", "k", "v"):
        out[n] = x[n][b:b + 1, :, h:h + 1, :]
    for n in ("g", "beta"):
        out[n] = x[n][b:b + 1, :, h:h + 1]
    out["h0"] = None if x["h0"] is None else x["h0"][b:b + 1, h:h + 1]
    return out


def oracle_ref(x, seg_len, nthreads=0, col_block=0, decay_first=False):
    return oracle.recurrence(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                             seg_len=seg_len, nthreads=nthreads, col_block=col_block,
                             decay_first=decay_first)
