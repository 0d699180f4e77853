"""Pins for the fp64 oracle: each check compares it with something other than itself --
hand-worked values, brute-force products of per-token transition matrices, closed forms
and algebraic invariants -- so that a dropped term, a wrong sign or index, a transposed
operand or the other decay reading fails at least one of them.

Pages cited by title and section:
  "RFC: HyperParallel Linear Attention Context Parallel", sections 2.1 and 2.2;
  "Context Parallelism in ART", section 08 ("First parallelize within a GPU",
  "Then parallelize across GPUs").
"""
import json
import os

import numpy as np
import pytest

import oracle
from context_scan_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked_k2v2.json")


def rel_err(x, ref):
    x, ref = np.asarray(x, np.float64), np.asarray(ref, np.float64)
    scale = np.sqrt(np.mean(ref * ref))
    return float(np.max(np.abs(x - ref)) / max(scale, 1e-300))


def rand_inputs(B, T, H, K, V, seed, g_mu=2.0, g_sd=1.0, beta_mu=0.0, beta_sd=1.0, h0=True):
    w = synth.Workload("pin", B=B, H=H, T=T, K=K, V=V, nseg=1, in_dtype="f32", g_mu=g_mu,
                       g_sd=g_sd, beta_mu=beta_mu, beta_sd=beta_sd,
                       h0_sd=0.1 if h0 else None, seed=seed)
    return synth.make_inputs(w, nthreads=2)


# --------------------------------------------------------------------------------------
# hand-worked example (tests/golden): pins orientation (k@H, q@H), the un-decayed read,
# and the summary's M and S
# --------------------------------------------------------------------------------------
@pytest.mark.parametrize("case", [0, 1, 2])
def test_hand_worked_example(case):
    d = json.load(open(GOLDEN))
    c = d["cases"][case]
    df = c.get("reading") == "decay_first"
    tok = d["tokens"]
    q = np.array(tok["q"], np.float32).reshape(1, 3, 1, 2)
    k = np.array(tok["k"], np.float32).reshape(1, 3, 1, 2)
    v = np.array(tok["v"], np.float32).reshape(1, 3, 1, 2)
    beta = np.array(tok["beta"], np.float32).reshape(1, 3, 1)
    g = np.array(c["g"], np.float32).reshape(1, 3, 1)
    h0 = np.array(c["h0"], np.float32).reshape(1, 1, 2, 2)
    tol = c["tol"]
    o, hf, _ = oracle.recurrence(q, k, v, g, beta, h0, decay_first=df)
    assert np.max(np.abs(o[0, :, 0] - np.array(c["o"]))) <= tol
    assert np.max(np.abs(hf[0, 0] - np.array(c["h_final"]))) <= tol
    M, S = oracle.summary(k, v, g, beta, nseg=1, decay_first=df)
    assert np.max(np.abs(M[0, 0, 0] - np.array(c["M"]))) <= tol
    assert np.max(np.abs(S[0, 0, 0] - np.array(c["S"]))) <= tol
    for chunk in (1, 2, 3):
        oc, hc = oracle.chunked_fwd(q, k, v, g, beta, h0, chunk=chunk, decay_first=df)
        assert np.max(np.abs(oc[0, :, 0] - np.array(c["o"]))) <= 10 * tol
        assert np.max(np.abs(hc[0, 0] - np.array(c["h_final"]))) <= 10 * tol
        Mc, Sc = oracle.chunked_summary(k, v, g, beta, nseg=1, chunk=chunk, decay_first=df)
        assert np.max(np.abs(Mc[0, 0, 0] - np.array(c["M"]))) <= 10 * tol
        assert np.max(np.abs(Sc[0, 0, 0] - np.array(c["S"]))) <= 10 * tol


# --------------------------------------------------------------------------------------
# c2: chunked == per-token (the chunk equations are an exact rewrite of the recurrence)
# --------------------------------------------------------------------------------------
@pytest.mark.parametrize("K,V,chunk,T", [(4, 4, 1, 32), (8, 4, 4, 64), (4, 8, 64, 192),
                                         (64, 64, 64, 256), (16, 8, 64, 100), (128, 128, 64, 128)])
def test_chunked_equals_per_token(K, V, chunk, T):
    x = rand_inputs(2, T, 2, K, V, seed=1000 + K * 7 + V + chunk)
    o, hf, _ = oracle.recurrence(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    oc, hc = oracle.chunked_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], chunk=chunk)
    assert rel_err(oc, o) <= 1e-12
    assert rel_err(hc, hf) <= 1e-12


@pytest.mark.parametrize("K,V,chunk,T", [(4, 4, 1, 32), (8, 4, 4, 64), (16, 8, 64, 100),
                                         (64, 64, 64, 256)])
def test_chunked_equals_per_token_decayed_read(K, V, chunk, T):
    # the other reading of the token update: G_i replaces Gx_i in P and Kr
    x = rand_inputs(2, T, 2, K, V, seed=2000 + K * 7 + V + chunk, g_mu=0.5)
    o, hf, _ = oracle.recurrence(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                                 decay_first=True)
    oc, hc = oracle.chunked_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], chunk=chunk,
                                decay_first=True)
    assert rel_err(oc, o) <= 1e-12
    assert rel_err(hc, hf) <= 1e-12
    # and the two readings really differ on these inputs
    o0, _, _ = oracle.recurrence(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    assert rel_err(o0, o) > 1e-3


def test_chunked_equals_per_token_wide_gates():
    # gates spread wide enough that the cumulative decay inside one chunk falls far below
    # exp(-88): only exponent differences are ever formed, so nothing overflows
    x = rand_inputs(1, 256, 2, 16, 16, seed=77, g_mu=-3.0, g_sd=2.0, beta_sd=2.0)
    o, hf, _ = oracle.recurrence(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    oc, hc = oracle.chunked_fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], chunk=64)
    assert np.all(np.isfinite(oc))
    assert rel_err(oc, o) <= 1e-12
    assert rel_err(hc, hf) <= 1e-12


# --------------------------------------------------------------------------------------
# c3: summary == brute-force product of per-token transitions on tiny inputs
#     M = T_L ... T_1,  T_t = exp(g_t) I - beta_t k_t k_t^T
#     S = sum_t (T_L ... T_{t+1}) beta_t k_t v_t^T
# --------------------------------------------------------------------------------------
def brute_summary(k, v, g, beta, decay_first=False):
    """k [L,K], v [L,V], g [L], beta [L] (float64) -> (M, S) by explicit matrices. With
    decay_first the transitions are exp(g_t) (I - beta_t k_t k_t^T)."""
    L, K = k.shape
    V = v.shape[1]
    if decay_first:
        Ts = [np.exp(g[t]) * (np.eye(K) - beta[t] * np.outer(k[t], k[t])) for t in range(L)]
    else:
        Ts = [np.exp(g[t]) * np.eye(K) - beta[t] * np.outer(k[t], k[t]) for t in range(L)]
    M = np.eye(K)
    for t in range(L):
        M = Ts[t] @ M
    S = np.zeros((K, V))
    for t in range(L):
        P = np.eye(K)
        for u in range(t + 1, L):
            P = Ts[u] @ P
        S += P @ (beta[t] * np.outer(k[t], v[t]))
    return M, S


@pytest.mark.parametrize("decay_first", [False, True])
@pytest.mark.parametrize("K,V,L", [(3, 2, 5), (8, 8, 16), (5, 7, 12), (8, 3, 1)])
def test_summary_brute_force(K, V, L, decay_first):
    x = rand_inputs(1, L, 1, K, V, seed=300 + K + V + L, g_mu=1.0)
    k, v = x["k"][0, :, 0].astype(np.float64), x["v"][0, :, 0].astype(np.float64)
    g, beta = x["g"][0, :, 0].astype(np.float64), x["beta"][0, :, 0].astype(np.float64)
    Mb, Sb = brute_summary(k, v, g, beta, decay_first)
    M, S = oracle.summary(x["k"], x["v"], x["g"], x["beta"], nseg=1, decay_first=decay_first)
    assert np.max(np.abs(M[0, 0, 0] - Mb)) <= 1e-13
    assert np.max(np.abs(S[0, 0, 0] - Sb)) <= 1e-13 * max(1.0, np.max(np.abs(Sb)))
    for chunk in (1, 4, 64):
        Mc, Sc = oracle.chunked_summary(x["k"], x["v"], x["g"], x["beta"], nseg=1, chunk=chunk,
                                        decay_first=decay_first)
        assert np.max(np.abs(Mc[0, 0, 0] - Mb)) <= 1e-12
        assert np.max(np.abs(Sc[0, 0, 0] - Sb)) <= 1e-12 * max(1.0, np.max(np.abs(Sb)))


def test_summary_is_affine_map_of_the_recurrence():
    """H_out(H0) = M H0 + S for H0 = 0 and for every unit basis matrix E_ij."""
    K, V, T = 4, 3, 24
    x = rand_inputs(1, T, 1, K, V, seed=41)
    M, S = oracle.summary(x["k"], x["v"], x["g"], x["beta"], nseg=1)
    M, S = M[0, 0, 0], S[0, 0, 0]
    _, h_zero, _ = oracle.recurrence(x["q"], x["k"], x["v"], x["g"], x["beta"], None)
    assert np.max(np.abs(h_zero[0, 0] - S)) <= 1e-13
    for i in range(K):
        for j in range(V):
            E = np.zeros((1, 1, K, V), np.float32)
            E[0, 0, i, j] = 1.0
            _, h, _ = oracle.recurrence(x["q"], x["k"], x["v"], x["g"], x["beta"], E)
            assert np.max(np.abs(h[0, 0] - (M @ E[0, 0] + S))) <= 1e-13


# --------------------------------------------------------------------------------------
# c4: compose is associative, not commutative; three-fold closed form; composing the
#     summaries of any segmentation reproduces the full recurrence; the scan gives the
#     state entering every segment
# --------------------------------------------------------------------------------------
def _rand_summary(rng, K, V):
    return rng.standard_normal((K, K)) * 0.5, rng.standard_normal((K, V))


def test_compose_associative_not_commutative_closed_form():
    rng = np.random.default_rng(5)
    K, V = 6, 4
    a, b, c = (_rand_summary(rng, K, V) for _ in range(3))
    ab = oracle.compose(*b, *a)           # a then b
    ab_c = oracle.compose(*c, *ab)        # (a then b) then c
    bc = oracle.compose(*c, *b)
    a_bc = oracle.compose(*bc, *a)        # a then (b then c)
    assert np.max(np.abs(ab_c[0] - a_bc[0])) <= 1e-13
    assert np.max(np.abs(ab_c[1] - a_bc[1])) <= 1e-13
    ba = oracle.compose(*a, *b)
    assert np.max(np.abs(ba[0] - ab[0])) > 1e-3     # order matters
    # three-fold closed form: M_c M_b M_a H + M_c M_b E_a + M_c E_b + E_c
    Ma, Ea = a
    Mb, Eb = b
    Mc, Ec = c
    H = rng.standard_normal((K, V))
    closed = Mc @ Mb @ Ma @ H + Mc @ Mb @ Ea + Mc @ Eb + Ec
    assert np.max(np.abs(ab_c[0] @ H + ab_c[1] - closed)) <= 1e-12


@pytest.mark.parametrize("cuts", [[1, 2, 3, 10, 11, 30], [17], [0], [5, 6, 7, 8, 9, 31]])
def test_composition_reproduces_recurrence_any_segmentation(cuts):
    K, V, T = 5, 4, 32
    x = rand_inputs(1, T, 1, K, V, seed=99, g_mu=3.0)
    _, hf, _ = oracle.recurrence(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    bounds = [0] + [c for c in cuts if 0 < c < T] + [T]
    Mt, St = np.eye(K), np.zeros((K, V))
    for lo, hi in zip(bounds[:-1], bounds[1:]):
        sl = slice(lo, hi)
        M, S = oracle.summary(x["k"][:, sl], x["v"][:, sl], x["g"][:, sl], x["beta"][:, sl], 1)
        Mt, St = oracle.compose(M[0, 0, 0], S[0, 0, 0], Mt, St)
    h_comp = Mt @ x["h0"][0, 0].astype(np.float64) + St
    assert np.max(np.abs(h_comp - hf[0, 0])) <= 1e-12


def test_scan_gives_state_entering_each_segment():
    K, V, T, nseg = 6, 5, 96, 6
    x = rand_inputs(2, T, 3, K, V, seed=123, g_mu=3.0)
    _, hf, H_in_ref = oracle.recurrence(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                                        seg_len=T // nseg)
    M, S = oracle.summary(x["k"], x["v"], x["g"], x["beta"], nseg)
    H_in = oracle.scan(M, S, x["h0"])
    assert np.max(np.abs(H_in - H_in_ref)) <= 1e-12
    last = np.einsum("bhij,bhjv->bhiv", M[-1], H_in[-1]) + S[-1]
    assert np.max(np.abs(last - hf)) <= 1e-12
    # the chunked summary agrees with the token-by-token one
    Mc, Sc = oracle.chunked_summary(x["k"], x["v"], x["g"], x["beta"], nseg, chunk=4)
    assert np.max(np.abs(Mc - M)) <= 1e-12
    assert np.max(np.abs(Sc - S)) <= 1e-12


# --------------------------------------------------------------------------------------
# c5: with one-token chunks the chunk summary is exactly the per-token transition
# --------------------------------------------------------------------------------------
def test_single_token_chunk_summary_is_transition():
    K, V = 7, 3
    x = rand_inputs(1, 1, 1, K, V, seed=8)
    k = x["k"][0, 0, 0].astype(np.float64)
    v = x["v"][0, 0, 0].astype(np.float64)
    g, b = float(x["g"][0, 0, 0]), float(x["beta"][0, 0, 0])
    M, S = oracle.chunked_summary(x["k"], x["v"], x["g"], x["beta"], nseg=1, chunk=1)
    assert np.max(np.abs(M[0, 0, 0] - (np.exp(g) * np.eye(K) - b * np.outer(k, k)))) <= 1e-15
    assert np.max(np.abs(S[0, 0, 0] - b * np.outer(k, v))) <= 1e-15


# --------------------------------------------------------------------------------------
# c6 - c9: special cases with closed forms
# --------------------------------------------------------------------------------------
def test_no_decay_no_write_keeps_state_exactly():
    K, V, T = 8, 6, 40
    x = rand_inputs(1, T, 2, K, V, seed=3)
    g = np.zeros_like(x["g"])
    beta = np.zeros_like(x["beta"])
    o, hf, _ = oracle.recurrence(x["q"], x["k"], x["v"], g, beta, x["h0"])
    assert np.array_equal(hf, x["h0"].astype(np.float64))
    ref = np.einsum("bthk,bhkv->bthv", x["q"].astype(np.float64), x["h0"].astype(np.float64))
    assert np.max(np.abs(o - ref)) <= 1e-14
    oc, hc = oracle.chunked_fwd(x["q"], x["k"], x["v"], g, beta, x["h0"], chunk=16)
    assert np.max(np.abs(hc - x["h0"])) <= 1e-14


def test_pure_decay():
    K, V, T = 8, 6, 50
    x = rand_inputs(1, T, 2, K, V, seed=4)
    beta = np.zeros_like(x["beta"])
    o, hf, _ = oracle.recurrence(x["q"], x["k"], x["v"], x["g"], beta, x["h0"])
    G = np.cumsum(x["g"].astype(np.float64), axis=1)             # [B,T,H]
    h0 = x["h0"].astype(np.float64)
    ref = np.exp(G)[..., None] * np.einsum("bthk,bhkv->bthv", x["q"].astype(np.float64), h0)
    assert rel_err(o, ref) <= 1e-12
    assert rel_err(hf, np.exp(G[:, -1])[..., None, None] * h0) <= 1e-12


def test_delta_rule_stores_value_along_unit_key():
    """g = 0, beta = 1, |k| = 1: after token t the state maps k_t to v_t exactly; read it
    back through the output by setting q_t = k_t."""
    K, V, T = 16, 8, 30
    x = rand_inputs(1, T, 2, K, V, seed=6)
    k = x["k"].astype(np.float64)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    k = k.astype(np.float32)
    g = np.zeros_like(x["g"])
    beta = np.ones_like(x["beta"])
    o, _, _ = oracle.recurrence(k, k, x["v"], g, beta, x["h0"])
    kn = np.linalg.norm(k.astype(np.float64), axis=-1)            # |k| = 1 to fp32 rounding
    assert np.max(np.abs(kn - 1)) < 1e-6
    assert np.max(np.abs(o - x["v"])) <= 1e-5


def test_orthonormal_keys_closed_form():
    """g = 0, beta = 1, orthonormal keys k_1..k_n: H_n = (I - sum k_i k_i^T) H0 + sum k_i v_i^T
    regardless of order. Signed unit vectors are exactly orthonormal in fp32."""
    K, V, n = 8, 5, 6
    rng = np.random.default_rng(11)
    perm = rng.permutation(K)[:n]
    sign = rng.choice([-1.0, 1.0], size=n)
    k = np.zeros((1, n, 1, K), np.float32)
    for i in range(n):
        k[0, i, 0, perm[i]] = sign[i]
    v = rng.standard_normal((1, n, 1, V)).astype(np.float32)
    h0 = rng.standard_normal((1, 1, K, V)).astype(np.float32)
    q = rng.standard_normal((1, n, 1, K)).astype(np.float32)
    g = np.zeros((1, n, 1), np.float32)
    beta = np.ones((1, n, 1), np.float32)
    _, hf, _ = oracle.recurrence(q, k, v, g, beta, h0)
    kk = k[0, :, 0].astype(np.float64)
    ref = (np.eye(K) - kk.T @ kk) @ h0[0, 0] + kk.T @ v[0, :, 0]
    assert np.max(np.abs(hf[0, 0] - ref)) <= 1e-14
    # a rotated orthonormal basis (fp32-rounded, so approximately orthonormal)
    Q, _ = np.linalg.qr(rng.standard_normal((K, K)))
    k2 = Q[:, :n].T.astype(np.float32).reshape(1, n, 1, K)
    _, hf2, _ = oracle.recurrence(q, k2, v, g, beta, h0)
    kk2 = k2[0, :, 0].astype(np.float64)
    ref2 = (np.eye(K) - kk2.T @ kk2) @ h0[0, 0] + kk2.T @ v[0, :, 0]
    assert np.max(np.abs(hf2[0, 0] - ref2)) <= 1e-5


# --------------------------------------------------------------------------------------
# c10: continuation (the state is the only thing carried between two calls)
# --------------------------------------------------------------------------------------
def test_continuation():
    K, V, T = 16, 16, 128
    x = rand_inputs(1, T, 2, K, V, seed=10)
    o, hf, _ = oracle.recurrence(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    a, b = slice(0, T // 2), slice(T // 2, T)
    o1, h1, _ = oracle.recurrence(x["q"][:, a], x["k"][:, a], x["v"][:, a], x["g"][:, a],
                                  x["beta"][:, a], x["h0"])
    # the hand-off state passes through fp32 (the oracle's state input type)
    o2, h2, _ = oracle.recurrence(x["q"][:, b], x["k"][:, b], x["v"][:, b], x["g"][:, b],
                                  x["beta"][:, b], h1.astype(np.float32))
    assert np.max(np.abs(o1 - o[:, a])) == 0.0
    assert rel_err(o2, o[:, b]) <= 1e-6
    assert rel_err(h2, hf) <= 1e-6


def test_column_blocks_and_threads_do_not_change_results():
    K, V, T = 16, 24, 64
    x = rand_inputs(2, T, 3, K, V, seed=12)
    o1, h1, _ = oracle.recurrence(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                                  nthreads=1)
    o2, h2, _ = oracle.recurrence(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"],
                                  col_block=5, nthreads=4)
    assert np.array_equal(o1, o2) and np.array_equal(h1, h2)


# --------------------------------------------------------------------------------------
# packed variable-length sequences ("KDA Chunk Backward -- TPU/Pallas Kernel Design",
# section 3.8): every sequence runs alone from its own initial state
# --------------------------------------------------------------------------------------
def _golden_tokens(d, c):
    tok = d["tokens"]
    arr = {n: np.array(tok[n], np.float32) for n in ("q", "k", "v", "beta")}
    arr["g"] = np.array(c["g"], np.float32)
    return arr


def test_varlen_hand_worked_packed():
    # the two default-reading hand-worked cases packed one after the other, with an empty
    # sequence between them: outputs and final states are the hand-worked values, and the
    # empty sequence hands back its initial state
    d = json.load(open(GOLDEN))
    c0, c1 = d["cases"][0], d["cases"][1]
    a0, a1 = _golden_tokens(d, c0), _golden_tokens(d, c1)
    pack = {n: np.concatenate([a0[n], a1[n]]) for n in a0}
    q, k, v = (pack[n].reshape(1, 6, 1, 2) for n in ("q", "k", "v"))
    g, beta = pack["g"].reshape(1, 6, 1), pack["beta"].reshape(1, 6, 1)
    h_mid = np.array([[7.0, -1.0], [0.5, 3.0]], np.float32)
    h0 = np.stack([np.array(c0["h0"], np.float32), h_mid,
                   np.array(c1["h0"], np.float32)]).reshape(3, 1, 2, 2)
    o, hf = oracle.varlen_recurrence(q, k, v, g, beta, [0, 3, 3, 6], h0)
    tol = max(c0["tol"], c1["tol"])
    assert np.max(np.abs(o[0, :3, 0] - np.array(c0["o"]))) <= tol
    assert np.max(np.abs(o[0, 3:, 0] - np.array(c1["o"]))) <= tol
    assert np.max(np.abs(hf[0, 0] - np.array(c0["h_final"]))) <= tol
    assert np.array_equal(hf[1, 0], h_mid.astype(np.float64))
    assert np.max(np.abs(hf[2, 0] - np.array(c1["h_final"]))) <= tol


def test_varlen_split_is_a_continuation():
    # one sequence cut in two at an unaligned token, the second part started from the
    # first part's final state, equals the unsplit sequence
    x = rand_inputs(1, 300, 2, 8, 4, seed=4242)
    o, hf, _ = oracle.recurrence(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"])
    h0 = np.concatenate([x["h0"], np.zeros_like(x["h0"])])
    _, hf1 = oracle.varlen_recurrence(x["q"], x["k"], x["v"], x["g"], x["beta"], [0, 97, 300], h0)
    h0[1] = hf1[0]
    o2, hf2 = oracle.varlen_recurrence(x["q"], x["k"], x["v"], x["g"], x["beta"], [0, 97, 300], h0)
    assert np.array_equal(o2[:, :97], o[:, :97])
    # the handed-over state is rounded to fp32 (initial states are fp32 inputs)
    assert rel_err(o2, o) <= 1e-6
    assert rel_err(hf2[1], hf[0]) <= 1e-6


def test_varlen_sequences_are_independent():
    x = rand_inputs(1, 200, 2, 8, 8, seed=4343, h0=False)
    cu = [0, 64, 129, 200]
    o, hf = oracle.varlen_recurrence(x["q"], x["k"], x["v"], x["g"], x["beta"], cu)
    y = {n: x[n].copy() for n in ("q", "k", "v", "g", "beta")}
    for n in y:
        y[n][:, 64:129] = y[n][:, 64:129][:, ::-1]   # change only the middle sequence
    o2, hf2 = oracle.varlen_recurrence(y["q"], y["k"], y["v"], y["g"], y["beta"], cu)
    assert np.array_equal(o2[:, :64], o[:, :64]) and np.array_equal(o2[:, 129:], o[:, 129:])
    assert np.array_equal(hf2[[0, 2]], hf[[0, 2]])
    assert not np.allclose(o2[:, 64:129], o[:, 64:129])


# --------------------------------------------------------------------------------------
# per-channel gates ("KDA Chunk Backward -- TPU/Pallas Kernel Design", section 1.2): the
# state decays row by row by exp(g_t), g_t in R^K
# --------------------------------------------------------------------------------------
GOLDEN_KDA = os.path.join(os.path.dirname(__file__), "golden", "hand_worked_kda_k2v2.json")


def kda_inputs(B, T, H, K, V, seed, g_mu=2.0, g_sd=1.0, h0=True):
    x = rand_inputs(B, T, H, K, V, seed, g_mu=g_mu, g_sd=g_sd, h0=h0)
    gk = synth.fill(seed + 77, "g", (B, T, H, K), synth.KIND_LOGSIGMOID, g_mu, g_sd)
    return x, gk


@pytest.mark.parametrize("case", [0, 1])
def test_kda_hand_worked(case):
    d = json.load(open(GOLDEN_KDA))
    c = d["cases"][case]
    tok = d["tokens"]
    q, k, v = (np.array(tok[n], np.float32).reshape(1, 2, 1, 2) for n in ("q", "k", "v"))
    beta = np.array(tok["beta"], np.float32).reshape(1, 2, 1)
    g = np.array(tok["g"], np.float32).reshape(1, 2, 1, 2)
    h0 = np.array(d["h0"], np.float32).reshape(1, 1, 2, 2)
    df = c["decay_first"]
    o, hf, _ = oracle.kda_recurrence(q, k, v, g, beta, h0, decay_first=df)
    assert np.max(np.abs(o[0, :, 0] - np.array(c["o"]))) <= c["tol"]
    assert np.max(np.abs(hf[0, 0] - np.array(c["h_final"]))) <= c["tol"]
    M, S = oracle.kda_summary(k, v, g, beta, nseg=1, decay_first=df)
    assert np.max(np.abs(M[0, 0, 0] - np.array(c["M"]))) <= c["tol"]
    assert np.max(np.abs(S[0, 0, 0] - np.array(c["S"]))) <= c["tol"]


@pytest.mark.parametrize("decay_first", [False, True])
def test_kda_equal_channels_is_the_scalar_gate(decay_first):
    # every channel carrying the token's scalar gate reproduces the scalar-gate oracle,
    # which is separate code
    x = rand_inputs(2, 96, 2, 8, 4, seed=5151, g_mu=0.5)
    gk = np.repeat(x["g"][..., None], 8, axis=-1)
    o, hf, hin = oracle.recurrence(x["q"], x["k"], x["v"], x["g"], x["beta"], x["h0"], seg_len=32,
                                   decay_first=decay_first)
    ok, hk, hink = oracle.kda_recurrence(x["q"], x["k"], x["v"], gk, x["beta"], x["h0"],
                                         seg_len=32, decay_first=decay_first)
    assert rel_err(ok, o) <= 1e-12 and rel_err(hk, hf) <= 1e-12 and rel_err(hink, hin) <= 1e-12
    M, S = oracle.summary(x["k"], x["v"], x["g"], x["beta"], nseg=3, decay_first=decay_first)
    Mk, Sk = oracle.kda_summary(x["k"], x["v"], gk, x["beta"], nseg=3, decay_first=decay_first)
    assert rel_err(Mk, M) <= 1e-12 and rel_err(Sk, S) <= 1e-12


@pytest.mark.parametrize("decay_first", [False, True])
def test_kda_summary_is_the_product_of_token_transitions(decay_first):
    # brute force on a tiny head: M = T_L ... T_1 with T_t = diag(a_t) - beta_t k_t k_t^T
    # (read before the decay) or (I - beta_t k_t k_t^T) diag(a_t) (decayed read); S is the
    # state reached from zero; and H_out = M H_in + S for a random H_in
    x, gk = kda_inputs(1, 7, 1, 3, 2, seed=5252, g_mu=0.0, g_sd=1.5)
    M, S = oracle.kda_summary(x["k"], x["v"], gk, x["beta"], nseg=1, decay_first=decay_first)
    k, v, b, a = (x["k"][0, :, 0].astype(np.float64), x["v"][0, :, 0].astype(np.float64),
                  x["beta"][0, :, 0].astype(np.float64), np.exp(gk[0, :, 0].astype(np.float64)))
    Mb, Sb = np.eye(3), np.zeros((3, 2))
    for t in range(7):
        P = np.eye(3) - b[t] * np.outer(k[t], k[t])
        Tt = P @ np.diag(a[t]) if decay_first else np.diag(a[t]) - b[t] * np.outer(k[t], k[t])
        Mb = Tt @ Mb
        Sb = Tt @ Sb + b[t] * np.outer(k[t], v[t])
    assert rel_err(M[0, 0, 0], Mb) <= 1e-12 and rel_err(S[0, 0, 0], Sb) <= 1e-12
    _, hf, _ = oracle.kda_recurrence(x["q"], x["k"], x["v"], gk, x["beta"], x["h0"],
                                     decay_first=decay_first)
    assert rel_err(hf[0, 0], Mb @ x["h0"][0, 0].astype(np.float64) + Sb) <= 1e-12


def test_kda_segment_states_are_the_scan_of_the_summaries():
    x, gk = kda_inputs(2, 128, 2, 8, 8, seed=5353, g_mu=1.0)
    _, hf, hin = oracle.kda_recurrence(x["q"], x["k"], x["v"], gk, x["beta"], x["h0"], seg_len=32)
    M, S = oracle.kda_summary(x["k"], x["v"], gk, x["beta"], nseg=4)
    H_in = oracle.scan(M, S, x["h0"])
    assert rel_err(H_in, hin) <= 1e-10
    Mall, Sall = oracle.kda_summary(x["k"], x["v"], gk, x["beta"], nseg=1)
    h_end = np.einsum("bhij,bhjv->bhiv", Mall[0], x["h0"].astype(np.float64)) + Sall[0]
    assert rel_err(h_end, hf) <= 1e-10
