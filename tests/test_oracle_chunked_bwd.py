"""Pin: the chunk-form backward (oracle/chunked_bwd.py) equals the per-token backward of the
oracle (itself pinned by finite differences in test_oracle_backward.py) for every gradient,
both readings of the token update, chunk sizes 1, 4 and 64, ragged last chunks and wide gates.

Pages cited by title and section: "Context Parallelism in ART", section 08 ("First
parallelize within a GPU", the chunk equations); "RFC: HyperParallel Linear Attention Context
Parallel", sections 2.1 and 6.4.3 (the token update and the reverse flow).
"""
import numpy as np
import pytest

import oracle
from oracle import chunked_bwd
from context_scan_gb300 import synth

NAMES = ("dq", "dk", "dv", "dg", "dbeta", "dh0")


def _inputs(T, K, V, seed, g_mu=1.0, g_sd=1.0, H=2):
    w = synth.Workload("pin", B=1, H=H, T=T, K=K, V=V, nseg=1, in_dtype="f32", g_mu=g_mu,
                       g_sd=g_sd, beta_mu=0.0, beta_sd=1.0, h0_sd=0.1, seed=seed)
    x = synth.make_inputs(w, nthreads=2)
    rng = np.random.default_rng(seed)
    dO = rng.standard_normal((1, T, H, V)).astype(np.float32)
    dht = rng.standard_normal((1, H, K, V)).astype(np.float32)
    return x, dO, dht


def _check(x, dO, dht, chunk, decay_first, tol=1e-12):
    ref = oracle.backward(x["q"], x["k"], x["v"], x["g"], x["beta"], dO, x["h0"], dht,
                          decay_first=decay_first)
    got = chunked_bwd.chunked_backward(x["q"], x["k"], x["v"], x["g"], x["beta"], dO, x["h0"],
                                       dht, chunk=chunk, decay_first=decay_first)
    for name, a, b in zip(NAMES, got, ref):
        scale = max(float(np.sqrt(np.mean(b * b))), 1e-30)
        assert float(np.max(np.abs(a - b))) / scale <= tol, (name, chunk, decay_first)


@pytest.mark.parametrize("decay_first", [False, True])
@pytest.mark.parametrize("chunk,T,K,V", [(1, 9, 3, 2), (4, 22, 5, 4), (64, 150, 8, 6),
                                          (64, 128, 4, 7)])
def test_chunked_backward_equals_per_token(chunk, T, K, V, decay_first):
    x, dO, dht = _inputs(T, K, V, seed=T + K)
    _check(x, dO, dht, chunk, decay_first)


@pytest.mark.parametrize("decay_first", [False, True])
def test_chunked_backward_wide_gates(decay_first):
    # gates as wide as the batched workload's (log sigmoid of N(1, 2)): every exponent is a
    # difference of cumulative gates that is never positive, so nothing overflows
    x, dO, dht = _inputs(200, 6, 5, seed=3, g_mu=1.0, g_sd=2.0)
    assert float(np.min(x["g"])) < -3.0
    _check(x, dO, dht, 64, decay_first, tol=1e-11)


def test_chunked_backward_without_initial_state_or_final_gradient():
    x, dO, _ = _inputs(70, 4, 4, seed=8)
    x = dict(x, h0=None)
    _check(x, dO, None, 64, False)
