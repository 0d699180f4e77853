"""GPU parity of the backward's state-gradient path ("RFC: HyperParallel Linear Attention
Context Parallel", section 6.4.3): per-segment state-gradient summaries dS and the reverse
scan dH_in[s] = M[s]^T dH_in[s+1] + dS[s], through the C ABI, against the fp64 oracle on
the same seeded inputs and incoming gradients.

Bars (per tensor, max|err| / RMS(ref)): 1e-4 for fp32 inputs and 1e-2 for bf16 inputs.
Both sides read the same values (bf16 inputs arrive already rounded, dO is drawn in the
dtype it is stored in). With fp32 inputs the kernel runs fp32 products on the CUDA cores, and
the bar covers fp32 sums of at most 128-term products per chunk carried through up to 128
chunks of decays that are all at most 1. With bf16 inputs the products run on the tensor
cores with tf32 operands (rounded to nearest, 2^-11 of each operand at most): a chunk's
contribution passes about five such roundings in series (dR, A^T dR, the update), measured at
up to 4.1e-3 (wide gates; 2.7e-3 at full size); the bar is half the forward's bar for bf16
inputs. Where a result also passes through the segment summaries M computed on the GPU, it
takes the forward's bar for bf16 inputs, 2e-2, which is the bar M itself is held to.
"""
import numpy as np
import pytest
import torch

import oracle
from context_scan_gb300 import gdn, synth
from gpu_util import head_slice, np64, rel_err, run_summary, upload

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS
TOL = {"f32": 1e-4, "bf16": 1e-2}
TOL_WITH_M = {"f32": 1e-4, "bf16": 2e-2}

SMALL = {
    "tiny_f32_k64_cp4": W["tiny_f32_k64_cp4"],
    "single_seg_small": synth.scaled(W["single_seg_h16_t8k"], H=3, T=1024),
    "cp4_small": synth.scaled(W["cp4_b2_h32_t32k"], B=2, H=3, T=1024),
    "cp16_small": synth.scaled(W["cp16_h16_t128k"], H=2, T=2048),
    "bf16_k64_cp4": synth.scaled(W["cp4_b2_h32_t32k"], B=1, H=3, T=512, K=64, V=64),
    "one_chunk_segments": synth.scaled(W["cp4_b2_h32_t32k"], B=1, H=2, T=512, nseg=8),
    "wide_gates_cp2": synth.scaled(W["cp2_b16_h32_t4k"], B=2, H=2, T=1024),
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from context_scan_gb300 import _build
    _build.build_cuda()
    gdn.lib()


def _dev(a, dtype=torch.float32):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda().to(dtype)


def run_state_grad(d, dO, nseg, dH_end=None, decay_first=False):
    B, T, H, K = d["k"].shape
    V = dO.shape[-1]
    dS = torch.full((nseg, B, H, K, V), float("nan"), device="cuda")
    prob = gdn.problem(d["k"], dO, dO, decay_first=decay_first)
    gdn.gdn_state_grad_summary(d["q"], d["k"], d["g"], d["beta"], dO, dS, nseg, dH_end, prob=prob)
    torch.cuda.synchronize()
    return dS


def run_scan(M, dS, dht):
    dH_in = torch.full_like(dS, float("nan"))
    gdn.gdn_state_grad_scan(M, dS, dht, dH_in)
    torch.cuda.synchronize()
    return dH_in


@pytest.mark.parametrize("decay_first", [False, True])
@pytest.mark.parametrize("with_end", [False, True])
@pytest.mark.parametrize("name", list(SMALL))
def test_state_grad_summary_matches_oracle(name, with_end, decay_first):
    w = SMALL[name]
    if decay_first and name in ("one_chunk_segments", "wide_gates_cp2"):
        pytest.skip("the decayed read is covered by the other workloads")
    x = synth.make_inputs(w)
    gr = synth.make_grads(w, dht_sd=0.5)
    rng = np.random.default_rng(0x5D)
    dH_end = rng.standard_normal((w.nseg, w.B, w.H, w.K, w.V)).astype(np.float32) if with_end else None
    ref = oracle.state_grad_summary(x["q"], x["k"], x["g"], x["beta"], gr["dO"], w.nseg,
                                    dH_end, decay_first=decay_first)
    d = upload(x, w)
    dS = run_state_grad(d, _dev(gr["dO"]), w.nseg, _dev(dH_end), decay_first=decay_first)
    err = rel_err(np64(dS), ref)
    assert err <= TOL[w.in_dtype], (name, err)
    if decay_first:   # the flag is honoured
        other = oracle.state_grad_summary(x["q"], x["k"], x["g"], x["beta"], gr["dO"], w.nseg,
                                          dH_end)
        assert rel_err(np64(dS), other) > 10 * err


def test_bf16_output_gradient():
    # dO carries the output's dtype: a bf16 dO is read as bf16
    w = SMALL["cp4_small"]
    x = synth.make_inputs(w)
    gr = synth.make_grads(w, bf16_out=True)
    ref = oracle.state_grad_summary(x["q"], x["k"], x["g"], x["beta"], gr["dO"], w.nseg)
    d = upload(x, w)
    dS = run_state_grad(d, _dev(gr["dO"], torch.bfloat16), w.nseg)
    assert rel_err(np64(dS), ref) <= TOL["bf16"]


@pytest.mark.parametrize("with_dht", [False, True])
@pytest.mark.parametrize("name", ["tiny_f32_k64_cp4", "cp16_small", "cp4_small"])
def test_state_grad_scan_matches_oracle(name, with_dht):
    # the scan alone, on the oracle's own M and dS (uploaded in fp32)
    w = SMALL[name]
    x = synth.make_inputs(w)
    gr = synth.make_grads(w, dht_sd=0.5 if with_dht else None)
    M, _ = oracle.summary(x["k"], x["v"], x["g"], x["beta"], w.nseg)
    dS = oracle.state_grad_summary(x["q"], x["k"], x["g"], x["beta"], gr["dO"], w.nseg)
    M32, dS32 = M.astype(np.float32), dS.astype(np.float32)
    ref = oracle.state_grad_scan(M32, dS32, gr["dht"])
    dH_in = run_scan(_dev(M32), _dev(dS32), _dev(gr["dht"]))
    assert rel_err(np64(dH_in), ref) <= 1e-5


@pytest.mark.parametrize("decay_first", [False, True])
@pytest.mark.parametrize("name", ["tiny_f32_k64_cp4", "cp4_small", "cp16_small"])
def test_segmented_state_gradient_is_dh0(name, decay_first):
    # the whole GPU route -- M from the segment summaries, dS per segment, the reverse scan --
    # against the oracle's per-token backward: dH_in[0] is dh0, and dH_in[s] is the state
    # gradient at every segment start
    w = SMALL[name]
    x = synth.make_inputs(w)
    gr = synth.make_grads(w, dht_sd=0.5)
    d = upload(x, w)
    M, _ = run_summary(w, d, decay_first=decay_first)
    dS = run_state_grad(d, _dev(gr["dO"]), w.nseg, decay_first=decay_first)
    dH_in = run_scan(M, dS, _dev(gr["dht"]))
    dh0_ref = oracle.backward(x["q"], x["k"], x["v"], x["g"], x["beta"], gr["dO"], x["h0"],
                              gr["dht"], decay_first=decay_first)[5]
    tol = TOL_WITH_M[w.in_dtype]
    assert rel_err(np64(dH_in[0]), dh0_ref) <= tol
    M_ref, _ = oracle.summary(x["k"], x["v"], x["g"], x["beta"], w.nseg, decay_first=decay_first)
    dS_ref = oracle.state_grad_summary(x["q"], x["k"], x["g"], x["beta"], gr["dO"], w.nseg,
                                       decay_first=decay_first)
    assert rel_err(np64(dH_in), oracle.state_grad_scan(M_ref, dS_ref, gr["dht"])) <= tol
    # one segment carrying dht through it gives dh0 directly
    dS1 = run_state_grad(d, _dev(gr["dO"]), 1, _dev(gr["dht"][None]), decay_first=decay_first)
    assert rel_err(np64(dS1[0]), dh0_ref) <= TOL[w.in_dtype]


def test_empty_sequence_and_determinism():
    w = SMALL["cp4_small"]
    x = synth.make_inputs(w)
    gr = synth.make_grads(w, dht_sd=0.5)
    d = upload(x, w)
    # T == 0: nothing to walk back through, dS = dH_end (or zero)
    e = {n: t[:, :0].contiguous() for n, t in d.items() if n != "h0"}
    dO0 = torch.empty((w.B, 0, w.H, w.V), device="cuda")
    end = torch.randn((2, w.B, w.H, w.K, w.V), device="cuda")
    assert torch.equal(run_state_grad(e, dO0, 2, end), end)
    assert torch.count_nonzero(run_state_grad(e, dO0, 2)) == 0
    # the same call twice gives the same bits
    a = run_state_grad(d, _dev(gr["dO"]), w.nseg)
    b = run_state_grad(d, _dev(gr["dO"]), w.nseg)
    assert torch.equal(a, b)


# full size, sampled heads: the launch the benchmark's backward leg times
@pytest.mark.parametrize("name", ["cp4_b2_h32_t32k"])
def test_full_size_sampled_heads(name):
    w = W[name]
    x = synth.make_inputs(w)
    gr = synth.make_grads(w, dht_sd=0.5)
    d = upload(x, w)
    dO = _dev(gr["dO"])
    dS = run_state_grad(d, dO, w.nseg)
    assert torch.isfinite(dS).all()
    M, _ = run_summary(w, d)
    dH_in = run_scan(M, dS, _dev(gr["dht"]))
    assert torch.isfinite(dH_in).all()
    for b, h in [(0, 0), (w.B - 1, w.H - 1), (w.B // 2, w.H // 3)]:
        xs = head_slice(x, b, h)
        dOs = np.ascontiguousarray(gr["dO"][b:b + 1, :, h:h + 1])
        ref = oracle.state_grad_summary(xs["q"], xs["k"], xs["g"], xs["beta"], dOs, w.nseg)
        assert rel_err(np64(dS[:, b:b + 1, h:h + 1]), ref) <= TOL["bf16"], (b, h)
        Ms, _ = oracle.summary(xs["k"], xs["v"], xs["g"], xs["beta"], w.nseg)
        ref_in = oracle.state_grad_scan(Ms, ref, gr["dht"][b:b + 1, h:h + 1])
        assert rel_err(np64(dH_in[:, b:b + 1, h:h + 1]), ref_in) <= TOL_WITH_M["bf16"], (b, h)
