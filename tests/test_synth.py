"""The seeded input generator: deterministic, thread-count independent, and shaped like
the described workloads (unit-norm q/k rows, bf16-representable values, gates in range)."""
import numpy as np

from context_scan_gb300 import synth


def test_thread_count_does_not_change_draws():
    w = synth.scaled(synth.WORKLOADS["cp4_b2_h32_t32k"], B=1, T=256, H=4)
    a = synth.make_inputs(w, nthreads=1)
    b = synth.make_inputs(w, nthreads=7)
    for name in ("q", "k", "v", "g", "beta", "h0"):
        assert np.array_equal(a[name], b[name]), name


def test_distributions_and_rounding():
    w = synth.scaled(synth.WORKLOADS["cp4_b2_h32_t32k"], B=1, T=512, H=8)
    x = synth.make_inputs(w)
    for name in ("q", "k"):
        n = np.linalg.norm(x[name].astype(np.float64), axis=-1)
        assert np.max(np.abs(n - 1.0)) < 2e-2          # unit norm up to bf16 rounding
    for name in ("q", "k", "v", "g", "beta"):
        a = x[name]
        bits = a.view(np.uint32)
        assert np.all(bits & 0xFFFF == 0), f"{name} is not bf16-representable"
    v = x["v"].astype(np.float64)
    assert abs(v.mean()) < 0.02 and abs(v.std() - 1.0) < 0.02
    assert np.all(x["g"] < 0) and np.all(x["beta"] > 0) and np.all(x["beta"] < 1)
    # g = log(sigmoid(N(2,1))): mean decay exp(g) near 0.85
    assert 0.8 < np.exp(x["g"].astype(np.float64)).mean() < 0.9
    assert abs(x["h0"].std() - 0.1) < 0.005


def test_per_sequence_seeds_and_fp32_workload():
    w = synth.scaled(synth.WORKLOADS["cp2_b16_h32_t4k"], B=3, T=128, H=2)
    x = synth.make_inputs(w)
    w1 = synth.scaled(w, B=1, per_sequence_seed=None, seed=w.per_sequence_seed + 2)
    y = synth.make_inputs(w1)
    assert np.array_equal(x["v"][2:3], y["v"])
    t = synth.make_inputs(synth.WORKLOADS["tiny_f32_k64_cp4"])
    assert t["q"].shape == (1, 256, 2, 64) and t["h0"].shape == (1, 2, 64, 64)
    assert np.any(t["v"].view(np.uint32) & 0xFFFF)     # fp32 inputs are not rounded
