"""Chunk-form backward of the gated delta rule, fp64 numpy -- TEST INFRASTRUCTURE.

Only the tests may import this module (like the rest of ``oracle/``); the CUDA library never
uses it. It restates the backward in the chunk equations that a chunked GPU backward
computes, so that "chunked backward == per-token backward" can be pinned on the CPU and the
chunk intermediates inspected. The per-token backward in ``oracle.c`` is the definition; this
module is checked against it.

Forward of one chunk of n tokens ("Context Parallelism in ART", section 08, "First
parallelize within a GPU", with the read of "RFC: HyperParallel Linear Attention Context
Parallel", section 2.1; G the inclusive cumulative gate in the chunk, Gx = G - g the read
side, or G for the decayed read):
    P[i,j] = exp(Gx_i - G_j) k_i.k_j (j < i),  A = (I + diag(beta) P)^{-1}
    Kr_i = exp(Gx_i) k_i,  U = A diag(beta) V,  W = A diag(beta) Kr,  R = U - W H
    C[i,j] = exp(G_i - G_j) q_i.k_j (j <= i),  Qd_i = exp(G_i) q_i,  O = Qd H + C R
    Kd_j = exp(G_n - G_j) k_j,  H' = exp(G_n) H + Kd^T R
Backward of the chunk, given dO and D' = dL/dH' (the reverse flow of the RFC's section 6.4.3;
every line is the vector-Jacobian product of one line above, last line first):
    dR = Kd D' + C^T dO                   dH = exp(G_n) D' + Qd^T dO - W^T dR
    dC = dO R^T (j <= i)   dQd = dO H^T   dKd = R D'^T   dexp(G_n) = <D', H>
    dU = dR,  dW = -dR H^T
    X = A^T dU:  dv_i = beta_i X_i,  dbeta_i += X_i . v_i
    Y = A^T dW:  dKr_i = beta_i Y_i,  dbeta_i += Y_i . Kr_i
    dA = dU (diag(beta) V)^T + dW (diag(beta) Kr)^T,  dL = -A^T dA A^T (j < i)
    dbeta_i += sum_j dL_ij P_ij,  dP = diag(beta) dL
and the gate, key and query terms of P, C, Qd, Kd, Kr, exp(G_n), summed into dG and dGx, then
dg = reverse cumulative sum of dG (minus dGx for the read before the decay).
"""
from __future__ import annotations

import numpy as np


def _chunk_forward(q, k, v, g, beta, H, decay_first):
    n = k.shape[0]
    G = np.cumsum(g)
    Gx = G if decay_first else G - g
    lower = np.tril(np.ones((n, n), bool), -1)
    lower_eq = np.tril(np.ones((n, n), bool))
    EP = np.where(lower, np.exp(np.where(lower, Gx[:, None] - G[None, :], 0.0)), 0.0)
    P = EP * (k @ k.T)
    A = np.linalg.inv(np.eye(n) + beta[:, None] * P)
    Kr = np.exp(Gx)[:, None] * k
    U = A @ (beta[:, None] * v)
    W = A @ (beta[:, None] * Kr)
    R = U - W @ H
    EC = np.where(lower_eq, np.exp(np.where(lower_eq, G[:, None] - G[None, :], 0.0)), 0.0)
    C = EC * (q @ k.T)
    Qd = np.exp(G)[:, None] * q
    O = Qd @ H + C @ R
    Kd = np.exp(G[-1] - G)[:, None] * k
    Hn = np.exp(G[-1]) * H + Kd.T @ R
    return dict(G=G, Gx=Gx, EP=EP, P=P, A=A, Kr=Kr, U=U, W=W, R=R, EC=EC, C=C, Qd=Qd, O=O,
                Kd=Kd, H=H, Hn=Hn)


def _chunk_backward(q, k, v, g, beta, f, dO, Dn, decay_first):
    """Gradients of one chunk: returns (dq, dk, dv, dg, dbeta, dH)."""
    G, Gx, H = f["G"], f["Gx"], f["H"]
    A, P, C, R, W, Kr, Qd, Kd = (f[x] for x in ("A", "P", "C", "R", "W", "Kr", "Qd", "Kd"))
    eGn = np.exp(G[-1])
    dR = Kd @ Dn + C.T @ dO
    dH = eGn * Dn + Qd.T @ dO - W.T @ dR
    dC = np.tril(dO @ R.T)
    dQd = dO @ H.T
    dKd = R @ Dn.T
    d_eGn = float(np.sum(Dn * H))
    dU, dW = dR, -dR @ H.T
    X, Y = A.T @ dU, A.T @ dW
    dv = beta[:, None] * X
    dKr = beta[:, None] * Y
    dbeta = np.sum(X * v, axis=1) + np.sum(Y * Kr, axis=1)
    dA = dU @ (beta[:, None] * v).T + dW @ (beta[:, None] * Kr).T
    dL = np.tril(-A.T @ dA @ A.T, -1)
    dbeta += np.sum(dL * P, axis=1)
    dP = beta[:, None] * dL

    dG = np.zeros_like(G)
    dGx = np.zeros_like(G)
    # P = EP * (k k^T): keys on both sides, the decay exp(Gx_i - G_j)
    S = dP * f["EP"]
    dk = S @ k + S.T @ k
    t = dP * P
    dGx += t.sum(axis=1)
    dG -= t.sum(axis=0)
    # C = EC * (q k^T): exp(G_i - G_j)
    S = dC * f["EC"]
    dq = S @ k
    dk += S.T @ q
    t = dC * C
    dG += t.sum(axis=1) - t.sum(axis=0)
    # Qd = exp(G) q
    dq += np.exp(G)[:, None] * dQd
    dG += np.sum(dQd * Qd, axis=1)
    # Kd = exp(G_n - G) k
    dk += np.exp(G[-1] - G)[:, None] * dKd
    t = np.sum(dKd * Kd, axis=1)
    dGn = float(t.sum()) + eGn * d_eGn
    dG -= t
    # Kr = exp(Gx) k
    dk += np.exp(Gx)[:, None] * dKr
    dGx += np.sum(dKr * Kr, axis=1)
    dG[-1] += dGn
    # Gx = G - g (read before the decay) or G (decayed read); G = cumsum(g)
    dG += dGx
    dg = np.cumsum(dG[::-1])[::-1].copy()
    if not decay_first:
        dg -= dGx
    return dq, dk, dv, dg, dbeta, dH


def chunked_backward(q, k, v, g, beta, dO, h0=None, dht=None, chunk: int = 64,
                     decay_first: bool = False):
    """Gradients of L = sum_t dO_t . o_t + <dht, h_final> in chunk form.

    Same arguments and returns as ``oracle.backward``: (dq, dk, dv, dg, dbeta, dh0), fp64.
    The last chunk of a sequence may be shorter than ``chunk``.
    """
    q, k, v, g, beta, dO = (np.asarray(x, np.float64) for x in (q, k, v, g, beta, dO))
    B, T, Hh, K = k.shape
    V = v.shape[-1]
    out = [np.zeros((B, T, Hh, K)), np.zeros((B, T, Hh, K)), np.zeros((B, T, Hh, V)),
           np.zeros((B, T, Hh)), np.zeros((B, T, Hh)), np.zeros((B, Hh, K, V))]
    starts = list(range(0, T, chunk))
    for b in range(B):
        for h in range(Hh):
            H = np.zeros((K, V)) if h0 is None else np.asarray(h0, np.float64)[b, h].copy()
            fwd = []
            for t0 in starts:
                s = slice(t0, min(t0 + chunk, T))
                f = _chunk_forward(q[b, s, h], k[b, s, h], v[b, s, h], g[b, s, h],
                                   beta[b, s, h], H, decay_first)
                fwd.append(f)
                H = f["Hn"]
            D = np.zeros((K, V)) if dht is None else np.asarray(dht, np.float64)[b, h].copy()
            for t0, f in zip(reversed(starts), reversed(fwd)):
                s = slice(t0, min(t0 + chunk, T))
                dq, dk, dv, dg, db, D = _chunk_backward(q[b, s, h], k[b, s, h], v[b, s, h],
                                                        g[b, s, h], beta[b, s, h], f,
                                                        dO[b, s, h], D, decay_first)
                out[0][b, s, h], out[1][b, s, h], out[2][b, s, h] = dq, dk, dv
                out[3][b, s, h], out[4][b, s, h] = dg, db
            out[5][b, h] = D
    return tuple(out)
