"""GPU parity of the whole backward ("RFC: HyperParallel Linear Attention Context Parallel",
section 6.4.3: state gradients at the chunk boundaries, then "backward_state +
backward_finish" to dQ, dK, dV, dg, dbeta): gdn_chunk_bwd through the C ABI against the
fp64 per-token oracle backward on the same seeded inputs and incoming gradients.

Bars (per tensor, max|err| / RMS(ref)): 1e-4 for fp32 inputs, 2e-2 for bf16 inputs. Both
sides read the same rounded inputs. With fp32 inputs every step runs in fp32 on the CUDA
cores (measured: at most 1.5e-5), and the bar covers fp32 sums of products over a chunk plus
the per-token gate gradients' cancellations (dg is a reverse cumulative sum of terms that
largely cancel). With bf16 inputs at K = V = 128 the states the gradients start from are
recomputed by the tensor-core forward, whose states are within the forward's bar of the
oracle's, and the bar is the forward's (measured: at most 5e-3, slow decay).
"""
import numpy as np
import pytest
import torch

import oracle
from context_scan_gb300 import gdn, synth
from gpu_util import np64, rel_err, upload

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS
TOL = {"f32": 1e-4, "bf16": 2e-2}
NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dh0")

SMALL = {
    "tiny_f32_k64_cp4": W["tiny_f32_k64_cp4"],
    "f32_k128_cp2": synth.scaled(W["cp4_b2_h32_t32k"], B=1, H=2, T=256, nseg=2,
                                 in_dtype="f32"),
    "bf16_k64_cp4": synth.scaled(W["cp4_b2_h32_t32k"], B=1, H=3, T=512, K=64, V=64),
    "cp4_small": synth.scaled(W["cp4_b2_h32_t32k"], B=2, H=2, T=1024),
    "slow_decay_h4_t1k_cp16": W["slow_decay_h4_t1k_cp16"],
    "wide_gates_cp2": synth.scaled(W["cp2_b16_h32_t4k"], B=2, H=2, T=512),
}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from context_scan_gb300 import _build
    _build.build_cuda()
    gdn.lib()


def run_bwd(w, d, dO, dht, nseg=None, decay_first=False, want_dh0=True):
    nseg = nseg or w.nseg
    B, T, H, K = d["k"].shape
    V = d["v"].shape[-1]
    out = {n: torch.full((B, T, H, K), float("nan"), device="cuda") for n in ("dq", "dk")}
    out["dv"] = torch.full((B, T, H, V), float("nan"), device="cuda")
    out["dg"] = torch.full((B, T, H), float("nan"), device="cuda")
    out["dbeta"] = torch.full((B, T, H), float("nan"), device="cuda")
    out["dh0"] = torch.full((B, H, K, V), float("nan"), device="cuda") if want_dh0 else None
    prob = gdn.problem(d["k"], d["v"], dO, decay_first=decay_first, g=d["g"])
    ws = gdn.alloc_bwd_workspace(prob, nseg)
    gdn.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], dO, dht, out["dq"],
                      out["dk"], out["dv"], out["dg"], out["dbeta"], out["dh0"], nseg, ws,
                      prob=prob)
    torch.cuda.synchronize()
    st, detail = gdn.gdn_check_device_error(ws)
    assert st == 0, (st, detail)
    return out


def grads(w, with_dht=True, bf16_out=False):
    gr = synth.make_grads(w, bf16_out=bf16_out, dht_sd=0.5 if with_dht else None)
    dO = torch.from_numpy(gr["dO"]).cuda()
    if bf16_out:
        dO = dO.to(torch.bfloat16)
    dht = None if gr["dht"] is None else torch.from_numpy(gr["dht"]).cuda()
    return gr, dO, dht


def check(w, x, gr, out, decay_first=False, tol=None):
    ref = oracle.backward(x["q"], x["k"], x["v"], x["g"], x["beta"], gr["dO"], x["h0"],
                          gr["dht"], decay_first=decay_first)
    tol = tol or TOL[w.in_dtype]
    for name, r in zip(NAMES, ref):
        if out[name] is None:
            continue
        e = rel_err(np64(out[name]), r, label=name)
        assert e <= tol, (name, e)


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("decay_first", [False, True])
def test_backward_matches_oracle(name, decay_first):
    w = SMALL[name]
    x = synth.make_inputs(w)
    d = upload(x, w)
    gr, dO, dht = grads(w)
    out = run_bwd(w, d, dO, dht, decay_first=decay_first)
    check(w, x, gr, out, decay_first=decay_first)


def test_backward_without_dht_or_h0_and_bf16_do():
    w = synth.scaled(SMALL["cp4_small"], h0_sd=None)
    x = synth.make_inputs(w)
    d = upload(x, w)
    gr, dO, dht = grads(w, with_dht=False, bf16_out=True)
    out = run_bwd(w, d, dO, dht, want_dh0=False)
    check(w, x, gr, out)


def test_backward_does_not_depend_on_the_segment_count():
    w = SMALL["cp4_small"]
    x = synth.make_inputs(w)
    d = upload(x, w)
    gr, dO, dht = grads(w)
    outs = [run_bwd(w, d, dO, dht, nseg=n) for n in (1, 2, 4, 16)]
    for o in outs[1:]:
        for name in NAMES:
            # different segment counts round differently (tf32 forward states, fp32 sums in
            # another order): the same bar as against the oracle
            assert rel_err(np64(o[name]), np64(outs[0][name])) <= TOL["bf16"], name
    check(w, x, gr, outs[2])


def test_backward_empty_sequence():
    w = synth.scaled(SMALL["cp4_small"], T=0)
    K = V = 128
    d = {n: torch.empty((2, 0, 2, K), dtype=torch.bfloat16, device="cuda") for n in ("q", "k", "v")}
    d["g"] = torch.empty((2, 0, 2), dtype=torch.bfloat16, device="cuda")
    d["beta"] = torch.empty((2, 0, 2), dtype=torch.bfloat16, device="cuda")
    d["h0"] = None
    dO = torch.empty((2, 0, 2, V), device="cuda")
    dht = torch.randn((2, 2, K, V), device="cuda")
    out = run_bwd(w, d, dO, dht, nseg=4)
    assert torch.equal(out["dh0"], dht)


def test_backward_rejects_per_channel_gates_and_bad_workspace():
    w = SMALL["cp4_small"]
    x = synth.make_inputs(w)
    d = upload(x, w)
    gr, dO, dht = grads(w)
    B, T, H, K = d["k"].shape
    prob = gdn.problem(d["k"], d["v"], dO)
    ws = gdn.alloc_bwd_workspace(prob, 4)
    out = [torch.empty((B, T, H, K), device="cuda") for _ in range(3)] + \
          [torch.empty((B, T, H), device="cuda") for _ in range(2)]
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], dO, dht, *out,
                          None, 4, ws[:1024], prob=prob)
    assert e.value.status == 5
    gk = torch.zeros((B, T, H, K), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(gdn.GdnError) as e:
        gdn.gdn_chunk_bwd(d["q"], d["k"], d["v"], gk, d["beta"], d["h0"], dO, dht, *out, None,
                          4, ws)
    assert e.value.status == 2


@pytest.mark.parametrize("name", ["cp4_b2_h32_t32k"])
def test_backward_full_size_sampled_heads(name):
    # the bench workload at full size, in the launch configuration bench.py times; two heads
    # checked against the per-token oracle run on those heads alone
    w = W[name]
    x = synth.make_inputs(w)
    d = upload(x, w)
    gr, dO, dht = grads(w)
    out = run_bwd(w, d, dO, dht)
    for n in NAMES:
        assert torch.isfinite(out[n]).all(), n
    for b, h in ((0, 0), (w.B - 1, w.H - 1)):
        xs = {n: np.ascontiguousarray(x[n][b:b + 1, :, h:h + 1]) for n in ("q", "k", "v")}
        xs.update({n: np.ascontiguousarray(x[n][b:b + 1, :, h:h + 1]) for n in ("g", "beta")})
        h0 = x["h0"][b:b + 1, h:h + 1]
        ref = oracle.backward(xs["q"], xs["k"], xs["v"], xs["g"], xs["beta"],
                              np.ascontiguousarray(gr["dO"][b:b + 1, :, h:h + 1]), h0,
                              gr["dht"][b:b + 1, h:h + 1])
        for n, r in zip(NAMES, ref):
            o = out[n]
            got = o[b:b + 1, h:h + 1] if n == "dh0" else o[b:b + 1, :, h:h + 1]
            assert rel_err(np64(got), r, label=f"{n} {b},{h}") <= TOL["bf16"], (n, b, h)


def test_timed_variant_matches_and_records_its_events():
    w = SMALL["cp4_small"]
    x = synth.make_inputs(w)
    d = upload(x, w)
    gr, dO, dht = grads(w)
    ref = run_bwd(w, d, dO, dht)
    B, T, H, K = d["k"].shape
    out = [torch.empty_like(ref[n]) for n in NAMES]
    prob = gdn.problem(d["k"], d["v"], dO, g=d["g"])
    ws = gdn.alloc_bwd_workspace(prob, w.nseg)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    for e in ev:
        e.record()
    gdn.gdn_chunk_bwd_timed(d["q"], d["k"], d["v"], d["g"], d["beta"], d["h0"], dO, dht, *out,
                            w.nseg, ws, ev, prob=prob)
    torch.cuda.synchronize()
    for n, o in zip(NAMES, out):
        assert torch.equal(o, ref[n]), n
    times = [ev[i].elapsed_time(ev[i + 1]) for i in range(5)]
    assert all(t >= 0 for t in times) and sum(times) > 0
