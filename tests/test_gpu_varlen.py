"""GPU parity of the packed variable-length forward ("KDA Chunk Backward -- TPU/Pallas Kernel
Design", section 3.8): gdn_varlen_fwd through the C ABI against the fp64 oracle's
per-sequence recurrence on the same seeded inputs, element by element.

Bars (per tensor, max|err| / RMS(ref)): 1e-4 for fp32 inputs, 2e-2 for bf16 inputs.
Lengths cover sequences shorter than a chunk, exactly one chunk, one token over, empty
sequences first, inside and last, starts that are not multiples of 64, and a total below one
chunk (which runs the CUDA-core kernels).
"""
import numpy as np
import pytest
import torch

import oracle
from context_scan_gb300 import gdn, synth
from gpu_util import TOL_BF16, TOL_F32, np64, rel_err
from plan_rule import expected_plan

pytestmark = pytest.mark.gpu

BASE = synth.WORKLOADS["varlen5_h16_t7300"]


def packed(lens, H=2, K=128, in_dtype="bf16", h0=True, seed=None, **kw):
    lens = tuple(int(n) for n in lens)
    return synth.scaled(BASE, H=H, K=K, V=K, T=sum(lens), seq_lens=lens, in_dtype=in_dtype,
                        h0_sd=0.1 if h0 else None, seed=seed or BASE.seed + sum(lens), **kw)


CASES = {
    "five_scaled": packed((180, 150, 200, 120, 80)),
    "edge_lengths": packed((1, 63, 64, 65, 0, 130, 0, 127)),
    "empty_first_and_last": packed((0, 100, 0, 257, 0)),
    "one_sequence": packed((640,)),
    "below_one_chunk": packed((10, 20, 0, 3)),
    "f32_k64": packed((70, 0, 129, 5), K=64, in_dtype="f32"),
    "bf16_k64": packed((70, 200, 1), K=64),
    "no_initial_state": packed((65, 190), h0=False),
    # long enough for the device plan to cut them into pieces (gdn_varlen.cu): the first into
    # eight of 8 chunks (six scan steps), a ragged last chunk in a cut sequence
    "cut_long_first": packed((4096, 100, 300, 64), H=4),
    "cut_ragged": packed((3000, 37, 700), H=2),
    "cut_no_initial_state": packed((3200, 900), H=3, h0=False),
    # at H = 16 (nine entries of 16 chains per phase on 152 SMs): the first sequence in five
    # pieces, the next two in two (no summary), two whole ones moved to the second phase, an
    # empty one last
    "cut_moved_whole": packed((5000, 1200, 1100, 1000, 900, 800, 700, 0), H=16),
}
CUT = ("cut_long_first", "cut_ragged", "cut_no_initial_state", "cut_moved_whole")
# planned (T of two 8-chunk pieces or more, every chain in one wave) but too short for a cut to
# pay: the longest is 18 chunks, the best cut that fits 31 chunk times
PLANNED_UNCUT = packed((1100, 900, 1000))


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from context_scan_gb300 import _build
    _build.build_cuda()
    gdn.lib()


def run_varlen(w, x, decay_first=False, out_dtype=torch.float32, cu=None, keep_ws=None):
    dt = torch.bfloat16 if w.in_dtype == "bf16" else torch.float32
    d = {n: torch.from_numpy(x[n]).cuda().to(dt).contiguous() for n in ("q", "k", "v", "g", "beta")}
    h0 = None if x["h0"] is None else torch.from_numpy(x["h0"]).cuda().contiguous()
    cu = synth.cu_seqlens(w) if cu is None else np.asarray(cu, np.int32)
    nseq = len(cu) - 1
    # NaN-filled outputs: a token or state the call fails to write shows up
    o = torch.full((1, w.T, w.H, w.V), float("nan"), dtype=out_dtype, device="cuda")
    hf = torch.full((nseq, w.H, w.K, w.V), float("nan"), device="cuda")
    cu_d = torch.from_numpy(cu).cuda()
    prob = gdn.problem(d["k"], d["v"], o, decay_first=decay_first)
    ws = gdn.alloc_varlen_workspace(prob, nseq)
    gdn.gdn_varlen_fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], h0, o, hf, cu_d, ws, prob=prob)
    torch.cuda.synchronize()
    st, detail = gdn.gdn_check_device_error(ws)
    if keep_ws is not None:
        keep_ws.append(ws)
    return o, hf, st, detail


def reference(w, x, decay_first=False):
    return oracle.varlen_recurrence(x["q"], x["k"], x["v"], x["g"], x["beta"],
                                    synth.cu_seqlens(w), x["h0"], decay_first=decay_first)


@pytest.mark.parametrize("name", list(CASES))
def test_varlen_matches_oracle(name):
    w = CASES[name]
    x = synth.make_inputs(w)
    o, hf, st, detail = run_varlen(w, x)
    assert st == 0, (st, detail)
    o_ref, hf_ref = reference(w, x)
    tol = TOL_F32 if w.in_dtype == "f32" else TOL_BF16
    assert torch.isfinite(o).all() and torch.isfinite(hf).all()
    assert rel_err(np64(o), o_ref) <= tol
    assert rel_err(np64(hf), hf_ref) <= tol
    # every sequence on its own scale too (a short one drowns in the others' RMS)
    cu = synth.cu_seqlens(w)
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        if b > a:
            assert rel_err(np64(o[:, a:b]), o_ref[:, a:b]) <= tol, s
        if x["h0"] is not None or b > a:
            assert rel_err(np64(hf[s]), hf_ref[s]) <= tol, s
        else:
            assert not hf[s].any(), s   # empty sequence from a zero state


@pytest.mark.parametrize("name", ["five_scaled", "edge_lengths", "f32_k64", "cut_long_first"])
def test_varlen_decayed_read(name):
    w = CASES[name]
    x = synth.make_inputs(w)
    o, hf, st, _ = run_varlen(w, x, decay_first=True)
    assert st == 0
    o_ref, hf_ref = reference(w, x, decay_first=True)
    tol = TOL_F32 if w.in_dtype == "f32" else TOL_BF16
    assert rel_err(np64(o), o_ref) <= tol
    assert rel_err(np64(hf), hf_ref) <= tol


@pytest.mark.parametrize("name", ["five_scaled", "cut_ragged"])
def test_varlen_bf16_output(name):
    w = CASES[name]
    x = synth.make_inputs(w)
    o, hf, st, _ = run_varlen(w, x, out_dtype=torch.bfloat16)
    assert st == 0 and o.dtype == torch.bfloat16
    o_ref, hf_ref = reference(w, x)
    # bf16 storage of o alone costs up to 2^-9 |o|, a few 1e-3 of RMS: bar 3e-2
    assert rel_err(np64(o), o_ref) <= 3e-2
    assert rel_err(np64(hf), hf_ref) <= TOL_BF16


def test_varlen_all_empty():
    w = packed((0, 0, 0))
    x = synth.make_inputs(w)
    o, hf, st, _ = run_varlen(w, x)
    assert st == 0 and o.numel() == 0
    assert torch.equal(hf.cpu(), torch.from_numpy(x["h0"]))


@pytest.mark.parametrize("cu", [[0, 100, 60, 257], [0, 100, 200, 250], [5, 100, 200, 257]])
def test_varlen_bad_lengths_are_reported(cu):
    # a device array that is not 0 .. T non-decreasing is caught on the device before any
    # chain reads it: the error word says GDN_ERR_INVALID_ARG, every sequence is treated as
    # empty (h_final = h0) and o is left as it was
    w = packed((100, 100, 57))
    x = synth.make_inputs(w)
    o, hf, st, _ = run_varlen(w, x, cu=cu)
    assert st == 1
    assert torch.isnan(o).all()
    assert torch.equal(hf.cpu(), torch.from_numpy(x["h0"]))
    # and a call with the right lengths works
    o, hf, st, _ = run_varlen(w, x)
    assert st == 0 and torch.isfinite(o).all()


@pytest.mark.parametrize("name", ["edge_lengths", "cut_long_first"])
def test_varlen_deterministic(name):
    w = CASES[name]
    x = synth.make_inputs(w)
    o1, hf1, _, _ = run_varlen(w, x)
    o2, hf2, _, _ = run_varlen(w, x)
    assert torch.equal(o1, o2) and torch.equal(hf1, hf2)


def test_varlen_full_size_sampled_heads():
    # the KDA design page's packed lengths at H = 16, K = V = 128, checked on sampled heads
    w = BASE
    x = synth.make_inputs(w)
    o, hf, st, _ = run_varlen(w, x)
    assert st == 0
    assert torch.isfinite(o).all() and torch.isfinite(hf).all()
    cu = synth.cu_seqlens(w)
    for h in (0, 7, 15):
        xs = {n: x[n][:, :, h:h + 1] for n in ("q", "k", "v", "g", "beta")}
        o_ref, hf_ref = oracle.varlen_recurrence(xs["q"], xs["k"], xs["v"], xs["g"], xs["beta"],
                                                 cu, x["h0"][:, h:h + 1])
        assert rel_err(np64(o[:, :, h:h + 1]), o_ref) <= TOL_BF16, h
        assert rel_err(np64(hf[:, h:h + 1]), hf_ref) <= TOL_BF16, h


def test_varlen_cut_timed_matches_plain():
    # with the long sequence cut, the timed entry point (five stage events between the plan's
    # launches) gives the plain call's results bit for bit
    w = CASES["cut_long_first"]
    x = synth.make_inputs(w)
    o, hf, _, _ = run_varlen(w, x)
    dt = torch.bfloat16
    d = {n: torch.from_numpy(x[n]).cuda().to(dt).contiguous() for n in ("q", "k", "v", "g", "beta")}
    h0 = torch.from_numpy(x["h0"]).cuda().contiguous()
    cu = torch.from_numpy(synth.cu_seqlens(w)).cuda()
    nseq = len(w.seq_lens)
    o2 = torch.full_like(o, float("nan"))
    hf2 = torch.full_like(hf, float("nan"))
    prob = gdn.problem(d["k"], d["v"], o2)
    ws = gdn.alloc_varlen_workspace(prob, nseq)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    gdn.gdn_varlen_fwd_timed(d["q"], d["k"], d["v"], d["g"], d["beta"], h0, o2, hf2, cu, ws, ev,
                             prob=prob)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(hf, hf2)
    assert gdn.gdn_check_device_error(ws)[0] == 0


def test_varlen_cut_full_size_sampled_heads():
    # a packed batch whose 16K-token sequence is cut into pieces (H = 16, K = V = 128), checked
    # on sampled heads against the oracle's per-sequence recurrence
    w = synth.WORKLOADS["varlen8_h16_t32k"]
    x = synth.make_inputs(w)
    o, hf, st, _ = run_varlen(w, x)
    assert st == 0
    assert torch.isfinite(o).all() and torch.isfinite(hf).all()
    cu = synth.cu_seqlens(w)
    for h in (0, 9):
        xs = {n: x[n][:, :, h:h + 1] for n in ("q", "k", "v", "g", "beta")}
        o_ref, hf_ref = oracle.varlen_recurrence(xs["q"], xs["k"], xs["v"], xs["g"], xs["beta"],
                                                 cu, x["h0"][:, h:h + 1])
        assert rel_err(np64(o[:, :, h:h + 1]), o_ref, label=f"o {h}") <= TOL_BF16, h
        assert rel_err(np64(hf[:, h:h + 1]), hf_ref, label=f"h_final {h}") <= TOL_BF16, h
        a, b = int(cu[0]), int(cu[1])   # the cut sequence on its own scale
        assert rel_err(np64(o[:, a:b, h:h + 1]), o_ref[:, a:b]) <= TOL_BF16, h


@pytest.mark.parametrize("name", CUT + ("planned_uncut",))
def test_varlen_plan_in_workspace(name):
    # the plan the call made, read from its workspace (the layout gdn_api.cu gives it: header,
    # WY tiles, two int arrays of nseq + 1, then the tables of nseq, e_max and e_max 8-int
    # entries, eight counts, four ints per sequence, each region 256-byte aligned), against
    # the rule restated above: the
    # cut cases are cut as their comments say, and a batch too short to pay is not
    w = PLANNED_UNCUT if name == "planned_uncut" else CASES[name]
    x = synth.make_inputs(w)
    kept = []
    _, _, st, _ = run_varlen(w, x, keep_ws=kept)
    assert st == 0
    ws = kept[0]
    nseq, H = len(w.seq_lens), w.H
    sms = min(torch.cuda.get_device_properties(0).multi_processor_count, 256)
    e_max = max(1, 256 // H)

    def rup(b):
        return (b + 255) // 256 * 256

    off = 256 + rup(H * (w.T // 64 + nseq) * 10240) + 2 * rup(4 * (nseq + 1))
    off += rup(32 * nseq) + 2 * rup(32 * e_max)
    words = ws[off:off + rup(32) + 16 * nseq].cpu().view(torch.int32).numpy()
    # (each region 256-byte aligned: the counts take 64 words)
    counts, seqinfo = words[:5].tolist(), words[64:64 + 3 * nseq].reshape(nseq, 3)
    want_counts, want_k = expected_plan(w.seq_lens, H, sms)
    assert counts == want_counts, (counts, want_counts)
    assert seqinfo[:, 0].tolist() == want_k
    if name == "cut_long_first":
        assert counts[3] == 8 and want_k[0] == 8   # eight pieces of 8 chunks: six scan steps
    if name == "cut_moved_whole" and sms == 152:
        assert want_k == [5, 2, 2, 1, 1, 1, 1, 1] and counts[2] == 8   # 6 pieces + 2 whole
    if name == "planned_uncut":
        assert counts[2] == 0 and counts[4] == 0 and want_k == [1, 1, 1]   # nothing cut
        o, hf, _, _ = run_varlen(w, x)   # and the whole sequences are right
        o_ref, hf_ref = reference(w, x)
        assert rel_err(np64(o), o_ref) <= TOL_BF16 and rel_err(np64(hf), hf_ref) <= TOL_BF16
