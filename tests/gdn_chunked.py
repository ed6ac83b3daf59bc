"""The gated delta rule in chunked form (numpy, fp64): a second, independent derivation
of Gated-DeltaNet replay used to pin the token-by-token oracle (both must agree), and
the formulation the GPU kernels follow.  Test infrastructure.

Within a chunk of C tokens entering with state S0 (d_v x d_k), with G_t the running sum
of the log-decays g inside the chunk, gamma_t = exp(G_t), Gam[t, i] = exp(G_t - G_i) for
i <= t and lam_i = gamma_C / gamma_i, the recurrence
    S_t = exp(g_t) S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T,   o_t = S_t (scale q_t)
unrolls to (Yang, Kautz & Hatamizadeh, "Gated Delta Networks", ICLR 2025, chunkwise form):
    Ms  = (K K^T) * Gam, strictly lower;   A = diag(beta) Ms;   T = (I + A)^-1
    Y   = V - diag(gamma) K S0^T;          U = T diag(beta) Y
    O   = diag(gamma) Q' S0^T + ((Q' K^T) * Gam, lower incl.) U,    Q' = scale Q
    S_C = gamma_C S0 + U^T diag(lam) K
The backward is the adjoint of these steps (chunks in reverse order, the state's
gradient carried from chunk to chunk).
"""
from __future__ import annotations

import numpy as np


def _chunk_consts(g, C):
    G = np.cumsum(g)
    gam = np.exp(G)
    Gam = np.exp(G[:, None] - G[None, :]) * np.tril(np.ones((C, C)))
    lam = np.exp(G[-1] - G)
    return G, gam, Gam, lam


def fwd(state0, q, k, v, g, beta, scale, C=4):
    """o [R][H][dv], final state [H][dv][dk]."""
    R, H, dk = q.shape
    dv = v.shape[2]
    o = np.zeros((R, H, dv))
    s_out = np.zeros((H, dv, dk))
    for h in range(H):
        S = state0[h].astype(np.float64).copy()
        for c0 in range(0, R, C):
            c1 = min(R, c0 + C)
            n = c1 - c0
            Q = scale * q[c0:c1, h].astype(np.float64)
            K = k[c0:c1, h].astype(np.float64)
            V = v[c0:c1, h].astype(np.float64)
            b = beta[c0:c1, h]
            G, gam, Gam, lam = _chunk_consts(g[c0:c1, h], n)
            Ms = (K @ K.T) * Gam * np.tril(np.ones((n, n)), -1)
            T = np.linalg.inv(np.eye(n) + b[:, None] * Ms)
            Y = V - gam[:, None] * (K @ S.T)
            U = T @ (b[:, None] * Y)
            P = (Q @ K.T) * Gam
            o[c0:c1, h] = gam[:, None] * (Q @ S.T) + P @ U
            S = gam[-1] * S + U.T @ (lam[:, None] * K)
        s_out[h] = S
    return o, s_out


def bwd(state0, q, k, v, g, beta, scale, d_o, C=4):
    """dq, dk, dv, dg, dbeta and the gradient reaching state0, for the loss <d_o, o>."""
    R, H, dk = q.shape
    dv = v.shape[2]
    dq = np.zeros((R, H, dk))
    dkk = np.zeros((R, H, dk))
    dvv = np.zeros((R, H, dv))
    dg = np.zeros((R, H))
    dbeta = np.zeros((R, H))
    ds0 = np.zeros((H, dv, dk))
    chunks = [(c0, min(R, c0 + C)) for c0 in range(0, R, C)]
    for h in range(H):
        # forward again, keeping each chunk's entering state
        S = state0[h].astype(np.float64).copy()
        starts = []
        for c0, c1 in chunks:
            starts.append(S.copy())
            n = c1 - c0
            K = k[c0:c1, h].astype(np.float64)
            V = v[c0:c1, h].astype(np.float64)
            b = beta[c0:c1, h]
            G, gam, Gam, lam = _chunk_consts(g[c0:c1, h], n)
            Ms = (K @ K.T) * Gam * np.tril(np.ones((n, n)), -1)
            T = np.linalg.inv(np.eye(n) + b[:, None] * Ms)
            U = T @ (b[:, None] * (V - gam[:, None] * (K @ S.T)))
            S = gam[-1] * S + U.T @ (lam[:, None] * K)
        dS = np.zeros((dv, dk))          # gradient of the state leaving the chunk
        for (c0, c1), S0 in reversed(list(zip(chunks, starts))):
            n = c1 - c0
            Q = scale * q[c0:c1, h].astype(np.float64)
            K = k[c0:c1, h].astype(np.float64)
            V = v[c0:c1, h].astype(np.float64)
            dO = d_o[c0:c1, h].astype(np.float64)
            b = beta[c0:c1, h]
            G, gam, Gam, lam = _chunk_consts(g[c0:c1, h], n)
            strict = np.tril(np.ones((n, n)), -1)
            incl = np.tril(np.ones((n, n)))
            KK = K @ K.T
            Ms = KK * Gam * strict
            T = np.linalg.inv(np.eye(n) + b[:, None] * Ms)
            Y = V - gam[:, None] * (K @ S0.T)
            U = T @ (b[:, None] * Y)
            QK = Q @ K.T
            P = QK * Gam
            dG = np.zeros(n)
            # S_C = gamma_C S0 + U^T diag(lam) K
            dS0 = gam[-1] * dS
            dU = lam[:, None] * (K @ dS.T)
            dK = lam[:, None] * (U @ dS)
            dlam = np.einsum("ia,ia->i", U, K @ dS.T)
            dG[-1] += gam[-1] * np.sum(dS * S0) + np.sum(dlam * lam)
            dG -= dlam * lam
            # O = diag(gamma) Q S0^T + P U
            dQ = gam[:, None] * (dO @ S0)
            dS0 += (gam[:, None] * dO).T @ Q
            dG += gam * np.einsum("ta,ta->t", dO, Q @ S0.T)
            dP = (dO @ U.T) * incl
            dU += P.T @ dO
            D1 = dP * P
            dG += D1.sum(1) - D1.sum(0)
            dQ += (dP * Gam) @ K
            dK += (dP * Gam).T @ Q
            # U = T Z, Z = diag(beta) Y, T = (I + diag(beta) Ms)^-1
            dZ = T.T @ dU
            dA = -(dZ @ U.T) * strict
            dY = b[:, None] * dZ
            db = np.einsum("ta,ta->t", dZ, Y) + (dA * Ms).sum(1)
            dMs = b[:, None] * dA
            D2 = dMs * Ms
            dG += D2.sum(1) - D2.sum(0)
            dKK = dMs * Gam
            dK += (dKK + dKK.T) @ K
            # Y = V - diag(gamma) K S0^T
            dV = dY
            dK -= gam[:, None] * (dY @ S0)
            dS0 -= (gam[:, None] * dY).T @ K
            dG -= gam * np.einsum("ta,ta->t", dY, K @ S0.T)
            dq[c0:c1, h] = scale * dQ
            dkk[c0:c1, h] = dK
            dvv[c0:c1, h] = dV
            dbeta[c0:c1, h] = db
            dg[c0:c1, h] = np.cumsum(dG[::-1])[::-1]   # g_j enters every G_t with t >= j
            dS = dS0
        ds0[h] = dS
    return dq, dkk, dvv, dg, dbeta, ds0
