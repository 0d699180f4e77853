"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the same seeded
inputs, element by element; plus edge cases, determinism, guard bands and error paths.

Bars (written here, per tensor, max|err| / RMS(ref)): 1e-4 for fp32 inputs, 2e-2 for bf16
inputs with fp32 outputs.
"""
import numpy as np
import pytest
import torch

import oracle
from context_scan_gb300 import gdn, synth
from gpu_util import (TOL_BF16, TOL_F32, head_slice, np64, oracle_ref, record, rel_err,
                      run_segmented, run_summary, tol_for, upload)

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS

# small versions of every workload: several chunks per segment, several heads, fast oracle
SMALL = {
    "tiny_f32_k64_cp4": W["tiny_f32_k64_cp4"],
    "single_seg_small": synth.scaled(W["single_seg_h16_t8k"], H=3, T=1024),
    "cp4_small": synth.scaled(W["cp4_b2_h32_t32k"], B=2, H=3, T=1024),
    "cp16_small": synth.scaled(W["cp16_h16_t128k"], H=2, T=2048),
    "cp2_batched_small": synth.scaled(W["cp2_b16_h32_t4k"], B=3, H=2, T=512),
    "slow_decay_h4_t1k_cp16": W["slow_decay_h4_t1k_cp16"],
    "bf16_k64_cp4": synth.scaled(W["cp4_b2_h32_t32k"], B=1, H=3, T=512, K=64, V=64),
    "one_chunk_segments": synth.scaled(W["cp4_b2_h32_t32k"], B=1, H=2, T=512, nseg=8),
    # few chains on many SMs: pieces whose starts are not segment starts (P = 6 pieces of 8
    # chunks for 4 segments of 12 on 152 SMs), so the forwards write the states entering the
    # segments as they pass them
    "uneven_pieces_cp4": synth.scaled(W["cp4_b2_h32_t32k"], B=1, H=2, T=3072),
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from context_scan_gb300 import _build
    _build.build_cuda()
    gdn.lib()


@pytest.mark.parametrize("name", list(SMALL))
def test_segmented_matches_oracle(name):
    w = SMALL[name]
    x = synth.make_inputs(w)
    o_ref, hf_ref, hin_ref = oracle_ref(x, w.seg_len)
    d = upload(x, w)
    o, hf, hin = run_segmented(w, d)
    tol = tol_for(w)
    e_o = rel_err(np64(o), o_ref, label="o")
    e_h = rel_err(np64(hf), hf_ref, label="h_final")
    e_in = rel_err(np64(hin), hin_ref, label="H_in")
    assert e_o <= tol, (name, "o", e_o)
    assert e_h <= tol, (name, "h_final", e_h)
    assert e_in <= tol, (name, "H_in", e_in)


@pytest.mark.parametrize("name", ["tiny_f32_k64_cp4", "cp4_small", "single_seg_small",
                                  "slow_decay_h4_t1k_cp16", "bf16_k64_cp4", "uneven_pieces_cp4"])
def test_decayed_read_matches_oracle(name):
    # the other reading of the token update (the read sees the decayed state): through the
    # WY tiles on the tensor-core path and the in-chain solve on the CUDA-core path
    w = SMALL[name]
    x = synth.make_inputs(w)
    o_ref, hf_ref, hin_ref = oracle_ref(x, w.seg_len, decay_first=True)
    d = upload(x, w)
    o, hf, hin = run_segmented(w, d, decay_first=True)
    tol = tol_for(w)
    e_o = rel_err(np64(o), o_ref, label="o")
    e_h = rel_err(np64(hf), hf_ref, label="h_final")
    e_in = rel_err(np64(hin), hin_ref, label="H_in")
    assert e_o <= tol, ("o", e_o)
    assert e_h <= tol, ("h_final", e_h)
    assert e_in <= tol, ("H_in", e_in)
    # the flag is honoured: the result is much closer to this reading than to the default one
    o_def, _, _ = oracle_ref(x, w.seg_len)
    assert rel_err(np64(o), o_def) > 2 * rel_err(np64(o), o_ref)
    if w.nseg > 1:
        M_ref, S_ref = oracle.summary(x["k"], x["v"], x["g"], x["beta"], w.nseg, decay_first=True)
        M, S = run_summary(w, d, decay_first=True)
        M, S = np64(M), np64(S)
        m_scale = max(float(np.sqrt(np.mean(M_ref ** 2))), 1e-12)
        assert float(np.max(np.abs(M - M_ref))) / m_scale <= tol
        assert rel_err(S, S_ref) <= tol


@pytest.mark.parametrize("name", ["tiny_f32_k64_cp4", "cp4_small", "slow_decay_h4_t1k_cp16",
                                  "bf16_k64_cp4"])
def test_summary_matches_oracle(name):
    w = SMALL[name]
    x = synth.make_inputs(w)
    M_ref, S_ref = oracle.summary(x["k"], x["v"], x["g"], x["beta"], w.nseg)
    d = upload(x, w)
    M, S = run_summary(w, d)
    tol = tol_for(w)
    M, S = np64(M), np64(S)
    # M shrinks like exp(cumulative gate): over long segments it is ~1e-20 or underflows.
    # Its error matters through M @ H_in (H_in, S are O(1)), so the scale has a floor of
    # 1e-12: an error below 1e-12 * tol in M is below 1e-10 of the state it feeds.
    m_scale = max(float(np.sqrt(np.mean(M_ref ** 2))), 1e-12)
    m_err = record(float(np.max(np.abs(M - M_ref))) / m_scale, "M")
    assert m_err <= tol, ("M", m_err)
    s_err = rel_err(S, S_ref, label="S")
    assert s_err <= tol, ("S", s_err)


@pytest.mark.parametrize("name", ["tiny_f32_k64_cp4", "cp4_small"])
def test_chunk_fwd_matches_oracle(name):
    w = SMALL[name]
    x = synth.make_inputs(w)
    o_ref, hf_ref, _ = oracle_ref(x, 0)
    d = upload(x, w)
    B, T, H, K = d["k"].shape
    o = torch.empty((B, T, H, w.V), device="cuda")
    hf = torch.empty((B, H, K, w.V), device="cuda")
    prob = gdn.problem(d["k"], d["v"], o)
    ws = gdn.alloc_workspace(prob, 1)
    gdn.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], o, hf, ws, prob=prob)
    torch.cuda.synchronize()
    assert rel_err(np64(o), o_ref) <= tol_for(w)
    assert rel_err(np64(hf), hf_ref) <= tol_for(w)


def test_summary_scan_matches_oracle_compose():
    rng = np.random.default_rng(3)
    nseg, B, H, K = 5, 2, 3, 128
    M = (rng.standard_normal((nseg, B, H, K, K)) * 0.05).astype(np.float32)
    S = rng.standard_normal((nseg, B, H, K, K)).astype(np.float32)
    h0 = rng.standard_normal((B, H, K, K)).astype(np.float32)
    ref = oracle.scan(M, S, h0)
    H_in = torch.empty((nseg, B, H, K, K), device="cuda")
    gdn.gdn_summary_scan(torch.from_numpy(M).cuda(), torch.from_numpy(S).cuda(),
                         torch.from_numpy(h0).cuda(), H_in)
    torch.cuda.synchronize()
    assert rel_err(np64(H_in), ref) <= 1e-5


def test_bf16_output():
    w = SMALL["cp4_small"]
    x = synth.make_inputs(w)
    o_ref, hf_ref, _ = oracle_ref(x, w.seg_len)
    o, hf, _ = run_segmented(w, upload(x, w), out_dtype=torch.bfloat16)
    # bf16 storage of o alone costs up to 2^-9 |o|, a few 1e-3 of RMS: bar 3e-2
    assert rel_err(np64(o), o_ref) <= 3e-2
    assert rel_err(np64(hf), hf_ref) <= TOL_BF16


def test_segment_count_does_not_change_results():
    """Emulated context parallelism: nseg in {1, 2, 4, 16} all give the single-pass answer."""
    w = synth.scaled(W["cp4_b2_h32_t32k"], B=1, H=2, T=1024, g_mu=5.0)
    x = synth.make_inputs(w)
    o_ref, hf_ref, _ = oracle_ref(x, 0)
    d = upload(x, w)
    for nseg in (1, 2, 4, 16):
        o, hf, _ = run_segmented(w, d, nseg=nseg)
        assert rel_err(np64(o), o_ref) <= TOL_BF16, nseg
        assert rel_err(np64(hf), hf_ref) <= TOL_BF16, nseg


def test_continuation_through_h_final():
    w = synth.scaled(W["cp4_b2_h32_t32k"], B=1, H=2, T=1024, nseg=1)
    x = synth.make_inputs(w)
    d = upload(x, w)
    o_all, hf_all, _ = run_segmented(w, d)
    half = {n: (t[:, :512].contiguous() if t is not None and n != "h0" else t)
            for n, t in d.items()}
    rest = {n: (t[:, 512:].contiguous() if t is not None and n != "h0" else t)
            for n, t in d.items()}
    o1, h1, _ = run_segmented(w, half)
    rest["h0"] = h1
    o2, h2, _ = run_segmented(w, rest)
    # each half against the oracle: the first half from h0, the second from the oracle's own
    # state after token 511 (so a GPU error in h1 is not carried into the second check)
    xa = {n: (v[:, :512] if v is not None and n != "h0" else v) for n, v in x.items()}
    oa_ref, ha_ref, _ = oracle_ref(xa, 0)
    xb = {n: (v[:, 512:] if v is not None and n != "h0" else v) for n, v in x.items()}
    xb["h0"] = ha_ref.astype(np.float32)
    ob_ref, hb_ref, _ = oracle_ref(xb, 0)
    assert rel_err(np64(o1), oa_ref, label="o first half") <= TOL_BF16
    assert rel_err(np64(h1), ha_ref, label="h first half") <= TOL_BF16
    assert rel_err(np64(o2), ob_ref, label="o second half") <= TOL_BF16
    assert rel_err(np64(h2), hb_ref, label="h second half") <= TOL_BF16
    # The tensor-core chains keep the state as sigma * H_s with sigma a running product of
    # the chunk decays; a continuation restarts sigma at 1, so its tf32 operands round
    # differently from the uninterrupted run's. Each run is within the parity bar of the
    # oracle (checked above); between themselves they agree to rounding noise (~2e-3 of the
    # RMS in o, ~2e-4 in the state).
    assert rel_err(np64(torch.cat([o1, o2], 1)), np64(o_all)) <= 1e-2
    assert rel_err(np64(h2), np64(hf_all)) <= 1e-3


def test_empty_sequence_and_zero_state():
    w = synth.scaled(W["cp4_b2_h32_t32k"], B=2, H=3, T=0, nseg=4)
    K = V = 128
    d = {n: torch.empty((2, 0, 3, K), dtype=torch.bfloat16, device="cuda") for n in ("q", "k", "v")}
    d["g"] = torch.empty((2, 0, 3), dtype=torch.bfloat16, device="cuda")
    d["beta"] = torch.empty((2, 0, 3), dtype=torch.bfloat16, device="cuda")
    h0 = torch.randn((2, 3, K, V), device="cuda")
    d["h0"] = h0
    o, hf, hin = run_segmented(w, d)
    assert torch.equal(hf, h0)
    for s in range(4):
        assert torch.equal(hin[s], h0)
    d["h0"] = None
    o, hf, hin = run_segmented(w, d)
    assert torch.count_nonzero(hf) == 0
    M, S = run_summary(w, d)
    eye = torch.eye(K, device="cuda").expand_as(M)
    assert torch.equal(M, eye) and torch.count_nonzero(S) == 0


def test_deterministic_and_guard_bands():
    w = SMALL["cp4_small"]
    x = synth.make_inputs(w)
    d = upload(x, w)
    B, T, H, K = d["k"].shape
    n_o = B * T * H * w.V
    pad = 4096
    buf = torch.full((n_o + 2 * pad,), float("nan"), device="cuda")
    o = buf[pad:pad + n_o].view(B, T, H, w.V)
    hbuf = torch.full((B * H * K * w.V + 2 * pad,), 7.0, device="cuda")
    hf = hbuf[pad:pad + B * H * K * w.V].view(B, H, K, w.V)
    prob = gdn.problem(d["k"], d["v"], o)
    ws = gdn.alloc_workspace(prob, w.nseg)
    outs = []
    for _ in range(3):
        gdn.gdn_segmented_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], o, hf,
                              w.nseg, ws, prob=prob)
        torch.cuda.synchronize()
        outs.append((o.clone(), hf.clone()))
    assert torch.isnan(buf[:pad]).all() and torch.isnan(buf[pad + n_o:]).all()
    assert (hbuf[:pad] == 7.0).all() and (hbuf[pad + B * H * K * w.V:] == 7.0).all()
    assert torch.isfinite(o).all()
    for a, b in outs[1:]:
        assert torch.equal(a, outs[0][0]) and torch.equal(b, outs[0][1])


def test_error_paths_launch_nothing():
    w = SMALL["cp4_small"]
    x = synth.make_inputs(w)
    d = upload(x, w)
    B, T, H, K = d["k"].shape
    o = torch.full((B, T, H, w.V), 3.0, device="cuda")
    hf = torch.empty((B, H, K, w.V), device="cuda")
    prob = gdn.problem(d["k"], d["v"], o)
    ws = gdn.alloc_workspace(prob, w.nseg)
    # workspace too small
    small = ws[:256]
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_segmented_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], o, hf,
                              w.nseg, small, prob=prob)
    assert e.value.status == 5
    # misaligned output pointer (a real allocation, offset by 4 bytes)
    flat = torch.empty(B * T * H * w.V + 4, device="cuda")
    o_mis = flat[1:1 + B * T * H * w.V].view(B, T, H, w.V)
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_segmented_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], o_mis, hf,
                              w.nseg, ws, prob=prob)
    assert e.value.status == 4
    # unsupported dtype (fp16)
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_segmented_fwd(d["q"].half(), d["k"].half(), d["v"].half(), d["g"].half(),
                              d["beta"].half(), d["h0"], o, hf, w.nseg, ws)
    assert e.value.status == 3
    # T not divisible by 64 * nseg
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_segmented_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], o, hf,
                              3, ws, prob=prob)
    assert e.value.status == 2
    torch.cuda.synchronize()
    assert (o == 3.0).all()   # nothing ran
    assert gdn.gdn_check_device_error(ws)[0] == 0


# --------------------------------------------------------------------------------------
# full sizes, in the launch configuration the benchmark times, checked on sampled heads
# --------------------------------------------------------------------------------------
FULL = ["single_seg_h16_t8k", "cp4_b2_h32_t32k", "cp16_h16_t128k", "cp2_b16_h32_t4k"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled_heads(name):
    w = W[name]
    x = synth.make_inputs(w)
    d = upload(x, w)
    o, hf, hin = run_segmented(w, d)
    assert torch.isfinite(o).all() and torch.isfinite(hf).all()
    heads = [(0, 0), (w.B - 1, w.H - 1)]
    if w.B * w.H > 4:
        heads.append((w.B // 2, w.H // 3))
    for b, h in heads:
        xs = head_slice(x, b, h)
        o_ref, hf_ref, hin_ref = oracle_ref(xs, w.seg_len, col_block=16)
        assert rel_err(np64(o[b:b + 1, :, h:h + 1]), o_ref, label=f"o {b},{h}") <= TOL_BF16, (b, h)
        assert rel_err(np64(hf[b:b + 1, h:h + 1]), hf_ref, label=f"h_final {b},{h}") <= TOL_BF16, (b, h)
        assert rel_err(np64(hin[:, b:b + 1, h:h + 1]), hin_ref, label=f"H_in {b},{h}") <= TOL_BF16, (b, h)


def test_last_piece_wy_tiles_beside_the_first_phase():
    # the schedule the headline runs, at a quarter of its length: the first phase leaves SMs
    # idle, so the last piece's WY tiles are formed there by a grid that takes chunks from a
    # counter while the chains run. Checked on sampled heads against the oracle, with the state
    # entering every segment, and bit for bit from one call to the next (the order in which the
    # chunks are taken varies; each tile does not)
    import bench
    w = synth.scaled(W["cp4_b2_h32_t32k"], T=8192)
    pc = gdn.Problem(w.B, w.T, w.H, 128, 128, 64, gdn.GDN_DTYPE_BF16, gdn.GDN_DTYPE_F32)
    plan = gdn.segmented_plan(pc, w.nseg)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert bench.wy_tail_beside(w, plan, sms), (plan, sms)
    x = synth.make_inputs(w)
    d = upload(x, w)
    runs = [run_segmented(w, d) for _ in range(2)]
    for a, b in zip(runs[0], runs[1]):
        assert torch.equal(a, b)
    o, hf, hin = runs[0]
    for b, h in ((0, 0), (0, w.H - 1), (1, w.H // 2), (w.B - 1, w.H - 1)):
        xs = head_slice(x, b, h)
        o_ref, hf_ref, hin_ref = oracle_ref(xs, w.seg_len, col_block=16)
        assert rel_err(np64(o[b:b + 1, :, h:h + 1]), o_ref, label=f"o {b},{h}") <= TOL_BF16, (b, h)
        assert rel_err(np64(hf[b:b + 1, h:h + 1]), hf_ref, label=f"h_final {b},{h}") <= TOL_BF16, (b, h)
        assert rel_err(np64(hin[:, b:b + 1, h:h + 1]), hin_ref, label=f"H_in {b},{h}") <= TOL_BF16, (b, h)


def test_uneven_pieces_h_in_guard_bands_bf16_and_determinism():
    # few chains on many SMs: the sequences are cut into unequal pieces whose starts are not
    # segment starts, and the forward chains write H_in as they pass the segment starts. Each
    # segment's slot is written exactly once (NaN guard bands around H_in stay NaN), repeated
    # calls agree bit for bit, and bf16 output keeps its bar.
    # the first length whose plan has a first piece of its own length, P not a multiple of
    # nseg (the plan depends on the device's SM count, so it is asked for, not assumed)
    w = None
    for T in (2816, 3328, 3840, 4352, 4096):
        cand = synth.scaled(SMALL["uneven_pieces_cp4"], T=T)
        pc = gdn.Problem(cand.B, T, cand.H, 128, 128, 64, gdn.GDN_DTYPE_BF16, gdn.GDN_DTYPE_F32)
        P, first, rest = gdn.segmented_plan(pc, cand.nseg)
        if first != rest and P % cand.nseg != 0:
            w = cand
            break
    assert w is not None, "no length here gets an unequal piece plan"
    x = synth.make_inputs(w)
    o_ref, hf_ref, hin_ref = oracle_ref(x, w.seg_len)
    d = upload(x, w)
    B, T, H, K = d["k"].shape
    o = torch.empty((B, T, H, w.V), dtype=torch.float32, device="cuda")
    hf = torch.empty((B, H, K, w.V), dtype=torch.float32, device="cuda")
    prob = gdn.problem(d["k"], d["v"], o)
    P = gdn.segmented_pieces(prob, w.nseg)
    assert P not in {w.nseg * m for m in (1, 2, 4, 8)}, P   # not an equal-piece plan
    n_in = w.nseg * B * H * K * w.V
    pad = 4096
    hbuf = torch.full((n_in + 2 * pad,), float("nan"), device="cuda")
    hin = hbuf[pad:pad + n_in].view(w.nseg, B, H, K, w.V)
    ws = gdn.alloc_workspace(prob, w.nseg)
    outs = []
    for _ in range(3):
        gdn.gdn_segmented_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], o, hf,
                              w.nseg, ws, H_in=hin, prob=prob)
        torch.cuda.synchronize()
        st, detail = gdn.gdn_check_device_error(ws)
        assert st == 0, (st, detail)
        outs.append((o.clone(), hf.clone(), hin.clone()))
    assert torch.isnan(hbuf[:pad]).all() and torch.isnan(hbuf[pad + n_in:]).all()
    assert torch.isfinite(hin).all()
    for a, b, c in outs[1:]:
        assert torch.equal(a, outs[0][0]) and torch.equal(b, outs[0][1]) and torch.equal(c, outs[0][2])
    assert rel_err(np64(o), o_ref) <= TOL_BF16
    assert rel_err(np64(hf), hf_ref) <= TOL_BF16
    assert rel_err(np64(hin), hin_ref) <= TOL_BF16
    o16, hf16, _ = run_segmented(w, d, out_dtype=torch.bfloat16)
    assert rel_err(np64(o16), o_ref) <= 3e-2
    assert rel_err(np64(hf16), hf_ref) <= TOL_BF16


def test_bounded_wait_runs_out_and_the_context_stays_usable():
    # the failure path of every kernel wait, made to happen on the host's terms: one CTA waits
    # on a barrier that nothing arrives at, with a ~1 ms limit. The wait gives up, the error word
    # says GDN_ERR_TIMEOUT with the self-test's tag, reading it clears it, and the next call on
    # the same context and workspace runs normally.
    w = SMALL["cp4_small"]
    x = synth.make_inputs(w)
    d = upload(x, w)
    prob = gdn.problem(d["k"], d["v"])
    ws = gdn.alloc_workspace(prob, w.nseg)
    gdn.gdn_selftest_wait_timeout(ws, 2_000_000)
    st, detail = gdn.gdn_check_device_error(ws)
    assert (st, detail) == (7, 0x5E)
    assert gdn.gdn_check_device_error(ws) == (0, 0)
    with pytest.raises(gdn.GdnError):
        gdn.gdn_selftest_wait_timeout(ws, 0)
    o_ref, hf_ref, hin_ref = oracle_ref(x, w.seg_len)
    o, hf, hin = run_segmented(w, d)
    assert rel_err(np64(o), o_ref) <= tol_for(w)
    assert rel_err(np64(hf), hf_ref) <= tol_for(w)


@pytest.mark.parametrize("name", ["tiny_f32_k64_cp4", "cp4_small", "cp16_small", "bf16_k64_cp4",
                                  "slow_decay_h4_t1k_cp16"])
def test_literal_cp_flow_matches_oracle(name):
    # The pages' flow composed from three public calls: every emulated rank's summary
    # (gdn_segment_summary), the in-order apply (gdn_summary_scan), then every rank's local
    # forward from its H_in (gdn_segment_fwd) -- RFC section 6.4.1 / 6.5
    w = SMALL[name]
    x = synth.make_inputs(w)
    o_ref, hf_ref, hin_ref = oracle_ref(x, w.seg_len)
    d = upload(x, w)
    M, S = run_summary(w, d)
    B, T, H, K = d["k"].shape
    hin = torch.empty((w.nseg, B, H, K, w.V), device="cuda")
    gdn.gdn_summary_scan(M, S, d["h0"], hin)
    o = torch.empty((B, T, H, w.V), device="cuda")
    hf = torch.empty((B, H, K, w.V), device="cuda")
    prob = gdn.problem(d["k"], d["v"], o)
    ws = gdn.alloc_workspace(prob, 1)
    gdn.gdn_segment_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], hin, o, hf, w.nseg, ws,
                        prob=prob)
    torch.cuda.synchronize()
    assert gdn.gdn_check_device_error(ws)[0] == 0
    tol = tol_for(w)
    assert rel_err(np64(hin), hin_ref, label="H_in") <= tol
    assert rel_err(np64(o), o_ref, label="o") <= tol
    assert rel_err(np64(hf), hf_ref, label="h_final") <= tol


def test_segment_fwd_edge_cases():
    # no H_in: every segment starts from zero (each segment equals a fresh gdn_chunk_fwd of
    # its own tokens); T = 0: h_final is the last segment's H_in
    w = synth.scaled(W["cp4_b2_h32_t32k"], B=1, H=2, T=512, nseg=2, h0_sd=None)
    x = synth.make_inputs(w)
    d = upload(x, w)
    o = torch.empty((1, 512, 2, 128), device="cuda")
    hf = torch.empty((1, 2, 128, 128), device="cuda")
    prob = gdn.problem(d["k"], d["v"], o)
    ws = gdn.alloc_workspace(prob, 1)
    gdn.gdn_segment_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], None, o, hf, 2, ws,
                        prob=prob)
    torch.cuda.synchronize()
    xb = {n: (v[:, 256:] if v is not None else v) for n, v in x.items()}
    ob_ref, hb_ref, _ = oracle_ref(xb, 0)
    assert rel_err(np64(o[:, 256:]), ob_ref) <= TOL_BF16
    assert rel_err(np64(hf), hb_ref) <= TOL_BF16
    e = {n: torch.empty((1, 0, 2, 128), dtype=torch.bfloat16, device="cuda") for n in ("q", "k", "v")}
    e["g"] = torch.empty((1, 0, 2), dtype=torch.bfloat16, device="cuda")
    e["beta"] = torch.empty((1, 0, 2), dtype=torch.bfloat16, device="cuda")
    hin = torch.randn((3, 1, 2, 128, 128), device="cuda")
    p0 = gdn.problem(e["k"], e["v"], o)
    gdn.gdn_segment_fwd(e["q"], e["k"], e["v"], e["g"], e["beta"], hin, o, hf, 3,
                        gdn.alloc_workspace(p0, 1), prob=p0)
    torch.cuda.synchronize()
    assert torch.equal(hf, hin[2])
