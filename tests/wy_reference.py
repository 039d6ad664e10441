"""Independent fp64 restatements used only to pin the oracle.

* ``chunked_wy``: the chunkwise WY form of the gated delta rule, written as
  plain dense matrices per chunk (gated_deltaproduct test.py: decay-masked
  KK^T, unit-lower-triangular inverse, w/u recompute, state scan, output).
  The WY identity is exact algebra, so it must agree with the token loop for
  every chunk size.
* ``brute_force``: the state after T steps as explicit products of the dense
  per-token transition matrices M_t = e^{g_t}(I - beta_t k_t k_t^T).

Neither shares code with the oracle or with the CUDA path.
"""
from __future__ import annotations

import numpy as np


def chunked_wy(q, k, v, beta, g, S0=None, C=64, scale=1.0):
    q, k, v, beta, g = (np.asarray(a, np.float64) for a in (q, k, v, beta, g))
    B, H, T, Dk = q.shape
    Dv = v.shape[-1]
    o = np.zeros((B, H, T, Dv))
    S_out = np.zeros((B, H, Dk, Dv))
    for b in range(B):
        for h in range(H):
            S = np.zeros((Dk, Dv)) if S0 is None else np.array(S0[b, h], np.float64)
            for c0 in range(0, T, C):
                sl = slice(c0, min(c0 + C, T))
                K, V, Q = k[b, h, sl], v[b, h, sl], q[b, h, sl]
                bb, gam = beta[b, h, sl], np.cumsum(g[b, h, sl])
                L = K.shape[0]
                diff = gam[:, None] - gam[None, :]
                strict = np.tril(np.ones((L, L)), -1)
                A = bb[:, None] * np.exp(diff * strict) * (K @ K.T) * strict
                Tm = np.linalg.inv(np.eye(L) + A)
                W = Tm @ ((bb * np.exp(gam))[:, None] * K)
                U = Tm @ (bb[:, None] * V)
                Dl = U - W @ S
                incl = np.tril(np.ones((L, L)))
                P = (Q @ K.T) * np.exp(diff * incl) * incl
                o[b, h, sl] = scale * (np.exp(gam)[:, None] * (Q @ S) + P @ Dl)
                S = np.exp(gam[-1]) * S + (K * np.exp(gam[-1] - gam)[:, None]).T @ Dl
            S_out[b, h] = S
    return o, S_out


def transition(kt, bt, gt):
    Dk = kt.shape[0]
    return np.exp(gt) * (np.eye(Dk) - bt * np.outer(kt, kt))


def brute_force(q, k, v, beta, g, S0=None, scale=1.0):
    """o_t and S_T from explicit products of the per-token transitions."""
    q, k, v, beta, g = (np.asarray(a, np.float64) for a in (q, k, v, beta, g))
    B, H, T, Dk = q.shape
    Dv = v.shape[-1]
    o = np.zeros((B, H, T, Dv))
    S_out = np.zeros((B, H, Dk, Dv))
    for b in range(B):
        for h in range(H):
            Ms = [transition(k[b, h, t], beta[b, h, t], g[b, h, t]) for t in range(T)]
            s0 = np.zeros((Dk, Dv)) if S0 is None else np.asarray(S0[b, h], np.float64)
            for t in range(T):
                # S_t = (M_t ... M_0) S0 + sum_{i<=t} (M_t ... M_{i+1}) b_i k_i v_i^T
                prod = np.eye(Dk)
                St = np.zeros((Dk, Dv))
                for i in range(t, -1, -1):
                    St += prod @ (beta[b, h, i] * np.outer(k[b, h, i], v[b, h, i]))
                    prod = prod @ Ms[i]
                St += prod @ s0
                o[b, h, t] = scale * (St.T @ q[b, h, t])
                if t == T - 1:
                    S_out[b, h] = St
    return o, S_out


def brute_force_deltaproduct(q, k, v, beta, g, S0=None, scale=1.0):
    """DeltaProduct by dense products: per token the map
    S -> H_{r-1}(...H_0(e^{g} S)...) with H_j(S) = (I - b_j k_j k_j^T) S + b_j k_j v_j^T,
    composed as an affine map (F, G) with S -> F S + G."""
    q, k, v, beta, g = (np.asarray(a, np.float64) for a in (q, k, v, beta, g))
    B, H, T, r, Dk = k.shape
    Dv = v.shape[-1]
    o = np.zeros((B, H, T, Dv))
    S_out = np.zeros((B, H, Dk, Dv))
    for b in range(B):
        for h in range(H):
            s0 = np.zeros((Dk, Dv)) if S0 is None else np.asarray(S0[b, h], np.float64)
            F_tot, G_tot = np.eye(Dk), np.zeros((Dk, Dv))
            for t in range(T):
                F, G = np.exp(g[b, h, t]) * np.eye(Dk), np.zeros((Dk, Dv))
                for j in range(r):
                    kk = k[b, h, t, j]
                    Hj = np.eye(Dk) - beta[b, h, t, j] * np.outer(kk, kk)
                    F, G = Hj @ F, Hj @ G + beta[b, h, t, j] * np.outer(kk, v[b, h, t, j])
                F_tot, G_tot = F @ F_tot, F @ G_tot + G
                St = F_tot @ s0 + G_tot
                o[b, h, t] = scale * (St.T @ q[b, h, t])
            S_out[b, h] = F_tot @ s0 + G_tot
    return o, S_out
