"""Pins for the oracle's backward functions, against the forward oracle rather than against
themselves: central finite differences of the loss for every input element, and exact
adjoint identities (the outputs and the final state are affine in any state they start
from, so <gradient, X> equals the change in the loss when X is added to that state).

Pages cited by title and section:
  "RFC: HyperParallel Linear Attention Context Parallel", section 6.4.3 (the reverse flow:
  state-gradient summary dS_local, dH_in = M^T dH_out + dS_local, then dQ/dK/dV/dg/dbeta);
  "KDA Chunk Backward -- TPU/Pallas Kernel Design", section 1 (the gradients of the
  backward pass, dh0 and the final-state gradient dht included).
"""
import numpy as np
import pytest

import oracle
from context_scan_gb300 import synth


def rand_inputs(B, T, H, K, V, seed, g_mu=2.0, g_sd=1.0):
    w = synth.Workload("pin", B=B, H=H, T=T, K=K, V=V, nseg=1, in_dtype="f32", g_mu=g_mu,
                       g_sd=g_sd, beta_mu=0.0, beta_sd=1.0, h0_sd=0.1, seed=seed)
    return synth.make_inputs(w, nthreads=2)


def loss(q, k, v, g, beta, h0, dO, dht, decay_first):
    o, hf, _ = oracle.recurrence(q, k, v, g, beta, h0, decay_first=decay_first)
    val = float(np.sum(o * dO.astype(np.float64)))
    if dht is not None:
        val += float(np.sum(hf * dht.astype(np.float64)))
    return val


@pytest.mark.parametrize("decay_first", [False, True])
@pytest.mark.parametrize("with_dht", [False, True])
def test_backward_matches_central_differences(decay_first, with_dht):
    B, T, H, K, V = 1, 7, 2, 3, 2
    x = rand_inputs(B, T, H, K, V, seed=0x5EED + 2 * decay_first + with_dht, g_mu=0.5)
    rng = np.random.default_rng(11)
    dO = rng.standard_normal((B, T, H, V)).astype(np.float32)
    dht = rng.standard_normal((B, H, K, V)).astype(np.float32) if with_dht else None
    args = {n: np.array(x[n], np.float32) for n in ("q", "k", "v", "g", "beta", "h0")}
    dq, dk, dv, dg, db, dh0 = oracle.backward(args["q"], args["k"], args["v"], args["g"],
                                              args["beta"], dO, args["h0"], dht,
                                              decay_first=decay_first)
    grads = {"q": dq, "k": dk, "v": dv, "g": dg, "beta": db, "h0": dh0}
    for name, grad in grads.items():
        base = args[name]
        fd = np.empty(base.shape, np.float64)
        for idx in np.ndindex(base.shape):
            step = 1e-3 * max(1.0, abs(float(base[idx])))
            hi, lo = base.copy(), base.copy()
            hi[idx] = np.float32(float(base[idx]) + step)
            lo[idx] = np.float32(float(base[idx]) - step)
            a = dict(args, **{name: hi})
            b = dict(args, **{name: lo})
            f_hi = loss(a["q"], a["k"], a["v"], a["g"], a["beta"], a["h0"], dO, dht, decay_first)
            f_lo = loss(b["q"], b["k"], b["v"], b["g"], b["beta"], b["h0"], dO, dht, decay_first)
            fd[idx] = (f_hi - f_lo) / (float(hi[idx]) - float(lo[idx]))
        scale = max(1.0, float(np.max(np.abs(fd))))
        err = float(np.max(np.abs(grad - fd)))
        assert err <= 2e-5 * scale, (name, err, scale)


def test_backward_sees_the_reading():
    # the two readings give different gradients on the same inputs (the pin above would
    # pass trivially if the flag were ignored on both sides)
    x = rand_inputs(1, 9, 1, 3, 2, seed=77, g_mu=0.0)
    dO = np.random.default_rng(3).standard_normal((1, 9, 1, 2)).astype(np.float32)
    a = oracle.backward(x["q"], x["k"], x["v"], x["g"], x["beta"], dO, x["h0"])
    b = oracle.backward(x["q"], x["k"], x["v"], x["g"], x["beta"], dO, x["h0"], decay_first=True)
    assert np.max(np.abs(a[1] - b[1])) > 1e-3 and np.max(np.abs(a[3] - b[3])) > 1e-3


def _segment(x, a, b):
    return [np.ascontiguousarray(np.asarray(x[n])[:, a:b]) for n in ("q", "k", "v", "g", "beta")]


@pytest.mark.parametrize("decay_first", [False, True])
@pytest.mark.parametrize("with_end", [False, True])
def test_state_grad_summary_adjoint(decay_first, with_end):
    # <dS[s], X> = sum over the segment's tokens of do_t . (o_t(X) - o_t(0))
    #              + <dH_end[s], h_end(X) - h_end(0)>, exactly (the map is affine in X)
    B, H, K, V, nseg, L = 2, 2, 5, 4, 3, 6
    T = nseg * L
    x = rand_inputs(B, T, H, K, V, seed=0xAD + decay_first, g_mu=1.0)
    rng = np.random.default_rng(5 + with_end)
    dO = rng.standard_normal((B, T, H, V)).astype(np.float32)
    dH_end = rng.standard_normal((nseg, B, H, K, V)) if with_end else None
    dS = oracle.state_grad_summary(x["q"], x["k"], x["g"], x["beta"], dO, nseg, dH_end,
                                   decay_first=decay_first)
    for s in range(nseg):
        X = rng.standard_normal((B, H, K, V)).astype(np.float32)
        q, k, v, g, beta = _segment(x, s * L, (s + 1) * L)
        o1, h1, _ = oracle.recurrence(q, k, v, g, beta, X, decay_first=decay_first)
        o0, h0, _ = oracle.recurrence(q, k, v, g, beta, None, decay_first=decay_first)
        d = dO[:, s * L:(s + 1) * L].astype(np.float64)
        for b in range(B):
            for h in range(H):
                lhs = float(np.sum(dS[s, b, h] * X[b, h]))
                rhs = float(np.sum(d[b, :, h] * (o1[b, :, h] - o0[b, :, h])))
                if with_end:
                    rhs += float(np.sum(dH_end[s, b, h] * (h1[b, h] - h0[b, h])))
                assert abs(lhs - rhs) <= 1e-10 * max(1.0, abs(rhs)), (s, b, h, lhs, rhs)


@pytest.mark.parametrize("decay_first", [False, True])
def test_state_grad_scan_adjoint(decay_first):
    # dH_in[s] is the gradient of the whole loss on the state entering segment s: adding X
    # there changes the loss by <dH_in[s], X> exactly. A scan that applied M instead of
    # M^T, ran forwards, or dropped dht or dS fails this.
    B, H, K, V, nseg, L = 1, 3, 4, 3, 4, 5
    T = nseg * L
    x = rand_inputs(B, T, H, K, V, seed=0xBEE + decay_first, g_mu=1.0)
    rng = np.random.default_rng(9)
    dO = rng.standard_normal((B, T, H, V)).astype(np.float32)
    dht = rng.standard_normal((B, H, K, V))
    M, _ = oracle.summary(x["k"], x["v"], x["g"], x["beta"], nseg, decay_first=decay_first)
    assert np.max(np.abs(M - np.swapaxes(M, -1, -2))) > 1e-3   # M is not symmetric
    dS = oracle.state_grad_summary(x["q"], x["k"], x["g"], x["beta"], dO, nseg,
                                   decay_first=decay_first)
    dH_in = oracle.state_grad_scan(M, dS, dht)
    for s in range(nseg):
        X = rng.standard_normal((B, H, K, V)).astype(np.float32)
        q, k, v, g, beta = _segment(x, s * L, T)
        o1, h1, _ = oracle.recurrence(q, k, v, g, beta, X, decay_first=decay_first)
        o0, h0, _ = oracle.recurrence(q, k, v, g, beta, None, decay_first=decay_first)
        d = dO[:, s * L:].astype(np.float64)
        for h in range(H):
            lhs = float(np.sum(dH_in[s, 0, h] * X[0, h]))
            rhs = float(np.sum(d[0, :, h] * (o1[0, :, h] - o0[0, :, h])) +
                        np.sum(dht[0, h] * (h1[0, h] - h0[0, h])))
            assert abs(lhs - rhs) <= 1e-10 * max(1.0, abs(rhs)), (s, h, lhs, rhs)


@pytest.mark.parametrize("decay_first", [False, True])
def test_segmented_state_gradient_is_dh0(decay_first):
    # the segment-parallel route (per-segment dS, then the reverse scan) ends in the dh0 of
    # the per-token backward, for any segmentation
    B, H, K, V, T = 2, 2, 6, 5, 24
    x = rand_inputs(B, T, H, K, V, seed=0xD0 + decay_first, g_mu=1.5)
    rng = np.random.default_rng(21)
    dO = rng.standard_normal((B, T, H, V)).astype(np.float32)
    dht = rng.standard_normal((B, H, K, V)).astype(np.float32)
    dh0 = oracle.backward(x["q"], x["k"], x["v"], x["g"], x["beta"], dO, x["h0"], dht,
                          decay_first=decay_first)[5]
    for nseg in (1, 2, 3, 8):
        M, _ = oracle.summary(x["k"], x["v"], x["g"], x["beta"], nseg, decay_first=decay_first)
        dS = oracle.state_grad_summary(x["q"], x["k"], x["g"], x["beta"], dO, nseg,
                                       decay_first=decay_first)
        dH_in = oracle.state_grad_scan(M, dS, dht)
        assert np.max(np.abs(dH_in[0] - dh0)) <= 1e-11 * max(1.0, float(np.max(np.abs(dh0))))
    # one segment carrying dht through it is the same thing
    dS1 = oracle.state_grad_summary(x["q"], x["k"], x["g"], x["beta"], dO, 1, dht[None],
                                    decay_first=decay_first)
    assert np.max(np.abs(dS1[0] - dh0)) <= 1e-11 * max(1.0, float(np.max(np.abs(dh0))))


def test_scalar_state_closed_form():
    # K = V = 1, one token, un-decayed read: h1 = a h0 + k beta (v - k h0), o = q h1,
    # L = do o + dht h1 = (do q + dht) h1.
    q, k, v, g, beta, h0, do, dht = 0.75, -1.25, 0.5, -0.5, 0.625, 0.375, 1.5, -0.25
    a = np.exp(g)
    r = beta * (v - k * h0)
    h1 = a * h0 + k * r
    w = do * q + dht
    f4 = lambda t: np.full((1, 1, 1, 1), t, np.float32)
    f3 = lambda t: np.full((1, 1, 1), t, np.float32)
    out = oracle.backward(f4(q), f4(k), f4(v), f3(g), f3(beta), f4(do), f4(h0), f4(dht))
    dq, dk, dv, dg, db, dh0 = (float(np.ravel(t)[0]) for t in out)
    assert dq == pytest.approx(do * h1, abs=1e-14)
    assert dv == pytest.approx(w * k * beta, abs=1e-14)
    assert db == pytest.approx(w * k * (v - k * h0), abs=1e-14)
    assert dk == pytest.approx(w * (r - beta * k * h0), abs=1e-14)
    assert dg == pytest.approx(w * a * h0, abs=1e-14)
    assert dh0 == pytest.approx(w * (a - beta * k * k), abs=1e-14)
