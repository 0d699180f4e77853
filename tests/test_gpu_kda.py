"""GPU parity of per-channel gates ("KDA Chunk Backward -- TPU/Pallas Kernel Design", section
1.2: g is [B,T,H,K] and the state decays row by row): every entry point through the C ABI
with gate_k set, against the fp64 oracle's kda_recurrence / kda_summary on the same seeded
inputs, element by element. These problems run the fp32 CUDA-core chains for every dtype.

Bars (per tensor, max|err| / RMS(ref)): 1e-4 for fp32 inputs, 2e-2 for bf16 inputs.
"""
import numpy as np
import pytest
import torch

import oracle
from context_scan_gb300 import gdn, synth
from gpu_util import TOL_BF16, TOL_F32, np64, rel_err, upload

pytestmark = pytest.mark.gpu

BASE = synth.WORKLOADS["kda_h16_t8k"]
CASES = {
    "f32_k64_cp4": synth.scaled(BASE, H=2, T=512, K=64, V=64, nseg=4, in_dtype="f32", seed=0x6D6E0701),
    "bf16_k128_cp4": synth.scaled(BASE, B=2, H=2, T=1024, nseg=4, seed=0x6D6E0702),
    "bf16_k128_single": synth.scaled(BASE, H=3, T=640, seed=0x6D6E0703),
    "f32_k64_fast_decay": synth.scaled(BASE, H=2, T=256, K=64, V=64, nseg=2, in_dtype="f32",
                                       g_mu=-1, g_sd=2, seed=0x6D6E0704),
    # bf16 runs the sub-block normalised tensor-core chains: gates of about -6 per token spread
    # every 16-token block past the factored form's limit (the blocks' exact path), and
    # gates of N(-4, 1.5) before the log-sigmoid leave about half the blocks on each path
    "bf16_k128_steep": synth.scaled(BASE, H=2, T=512, nseg=2, g_mu=-6, g_sd=1, seed=0x6D6E0705),
    "bf16_k128_mixed": synth.scaled(BASE, H=2, T=512, nseg=2, g_mu=-4, g_sd=1.5, seed=0x6D6E0706),
    "bf16_k64_cp2": synth.scaled(BASE, H=2, T=512, K=64, V=64, nseg=2, seed=0x6D6E0707),
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from context_scan_gb300 import _build
    _build.build_cuda()
    gdn.lib()


def tol(w):
    return TOL_F32 if w.in_dtype == "f32" else TOL_BF16


def run(w, x, decay_first=False):
    d = upload(x, w)
    B, T, H, K = d["k"].shape
    o = torch.full((B, T, H, w.V), float("nan"), device="cuda")
    hf = torch.full((B, H, K, w.V), float("nan"), device="cuda")
    hin = torch.empty((w.nseg, B, H, K, w.V), device="cuda")
    prob = gdn.problem(d["k"], d["v"], o, decay_first=decay_first, g=d["g"])
    assert prob.gate_k == 1
    ws = gdn.alloc_workspace(prob, w.nseg)
    gdn.gdn_segmented_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], o, hf, w.nseg, ws,
                          H_in=hin, prob=prob)
    torch.cuda.synchronize()
    st, detail = gdn.gdn_check_device_error(ws)
    assert st == 0, (st, detail)
    return o, hf, hin, d


@pytest.mark.parametrize("decay_first", [False, True])
@pytest.mark.parametrize("name", list(CASES))
def test_segmented_matches_oracle(name, decay_first):
    w = CASES[name]
    x = synth.make_inputs(w)
    o, hf, hin, _ = run(w, x, decay_first)
    o_ref, hf_ref, hin_ref = oracle.kda_recurrence(x["q"], x["k"], x["v"], x["g"], x["beta"],
                                                   x["h0"], seg_len=w.seg_len,
                                                   decay_first=decay_first)
    assert torch.isfinite(o).all()
    assert rel_err(np64(o), o_ref) <= tol(w), "o"
    assert rel_err(np64(hf), hf_ref) <= tol(w), "h_final"
    assert rel_err(np64(hin), hin_ref) <= tol(w), "H_in"


@pytest.mark.parametrize("decay_first", [False, True])
def test_summary_matches_oracle(decay_first):
    w = CASES["bf16_k128_cp4"]
    x = synth.make_inputs(w)
    d = upload(x, w)
    B, T, H, K = d["k"].shape
    M = torch.empty((w.nseg, B, H, K, K), device="cuda")
    S = torch.empty((w.nseg, B, H, K, w.V), device="cuda")
    prob = gdn.problem(d["k"], d["v"], decay_first=decay_first, g=d["g"])
    ws = gdn.alloc_workspace(prob, 1)
    gdn.gdn_segment_summary(d["k"], d["v"], d["g"], d["beta"], M, S, w.nseg, ws, prob=prob)
    torch.cuda.synchronize()
    assert gdn.gdn_check_device_error(ws)[0] == 0
    M_ref, S_ref = oracle.kda_summary(x["k"], x["v"], x["g"], x["beta"], w.nseg,
                                      decay_first=decay_first)
    # M is compared on its own scale with an absolute floor (it decays towards zero)
    scale = max(np.sqrt(np.mean(M_ref ** 2)), 1e-12)
    assert np.max(np.abs(np64(M) - M_ref)) / scale <= TOL_BF16
    assert rel_err(np64(S), S_ref) <= TOL_BF16


def test_equal_channels_match_the_scalar_gate():
    # every channel carrying the token's scalar gate gives the scalar-gate result (both
    # through the same fp32 kernels)
    w = synth.scaled(CASES["f32_k64_cp4"], gate_k=False)
    x = synth.make_inputs(w)
    d = upload(x, w)
    gk = d["g"][..., None].expand(*d["g"].shape, w.K).contiguous()
    B, T, H, K = d["k"].shape
    outs = []
    for g in (d["g"], gk):
        o = torch.empty((B, T, H, w.V), device="cuda")
        hf = torch.empty((B, H, K, w.V), device="cuda")
        prob = gdn.problem(d["k"], d["v"], o, g=g)
        ws = gdn.alloc_workspace(prob, w.nseg)
        gdn.gdn_segmented_fwd(d["q"], d["k"], d["v"], g, d["beta"], d["h0"], o, hf, w.nseg, ws,
                              prob=prob)
        torch.cuda.synchronize()
        outs.append((np64(o), np64(hf)))
    assert rel_err(outs[1][0], outs[0][0]) <= 1e-5
    assert rel_err(outs[1][1], outs[0][1]) <= 1e-5


def test_packed_sequences_match_oracle():
    w = synth.scaled(CASES["bf16_k128_single"], T=450, seq_lens=(1, 63, 64, 65, 0, 130, 0, 127),
                     seed=0x6D6E0705)
    x = synth.make_inputs(w)
    d = upload(x, w)
    cu = torch.from_numpy(synth.cu_seqlens(w)).cuda()
    nseq = len(w.seq_lens)
    o = torch.full((1, w.T, w.H, w.V), float("nan"), device="cuda")
    hf = torch.empty((nseq, w.H, w.K, w.V), device="cuda")
    prob = gdn.problem(d["k"], d["v"], o, g=d["g"])
    ws = gdn.alloc_varlen_workspace(prob, nseq)
    gdn.gdn_varlen_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], o, hf, cu, ws, prob=prob)
    torch.cuda.synchronize()
    assert gdn.gdn_check_device_error(ws)[0] == 0
    o_ref, hf_ref = oracle.varlen_recurrence(x["q"], x["k"], x["v"], x["g"], x["beta"],
                                             synth.cu_seqlens(w), x["h0"])
    assert torch.isfinite(o).all()
    assert rel_err(np64(o), o_ref) <= TOL_BF16
    assert rel_err(np64(hf), hf_ref) <= TOL_BF16


def test_deterministic():
    w = CASES["bf16_k128_cp4"]
    x = synth.make_inputs(w)
    o1, hf1, _, _ = run(w, x)
    o2, hf2, _, _ = run(w, x)
    assert torch.equal(o1, o2) and torch.equal(hf1, hf2)


def test_full_size_sampled_heads():
    # the KDA design page's shape (H = 16, T = 8192, K = V = 128, bf16), sampled heads
    w = BASE
    x = synth.make_inputs(w)
    o, hf, _, _ = run(w, x)
    assert torch.isfinite(o).all() and torch.isfinite(hf).all()
    for h in (0, 9):
        xs = {n: x[n][:, :, h:h + 1] for n in ("q", "k", "v", "g", "beta")}
        o_ref, hf_ref, _ = oracle.kda_recurrence(xs["q"], xs["k"], xs["v"], xs["g"], xs["beta"],
                                                 x["h0"][:, h:h + 1], col_block=16)
        assert rel_err(np64(o[:, :, h:h + 1]), o_ref) <= TOL_BF16, h
        assert rel_err(np64(hf[:, h:h + 1]), hf_ref) <= TOL_BF16, h
