"""Pure numpy fp64 restatement of the oracle, token by token.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Written separately from
``gdn_oracle.c`` so that a slip in one of the two shows up as a disagreement
on small cases.  Loops over tokens in Python: keep T small.
"""
from __future__ import annotations

import numpy as np


def _unit(x):
    n = np.sqrt((x * x).sum(-1, keepdims=True))
    return x / np.maximum(n, 1e-12)


def gdn_fwd(q, k, v, beta, g, initial_state=None, scale=1.0, l2norm=False):
    """S_t = e^{g_t}(I - b_t k_t k_t^T)S_{t-1} + b_t k_t v_t^T ; o_t = scale S_t^T q_t."""
    q, k, v, beta, g = (np.asarray(a, np.float64) for a in (q, k, v, beta, g))
    B, H, T, Dk = q.shape
    Dv = v.shape[-1]
    if l2norm:
        q, k = _unit(q), _unit(k)
    o = np.zeros((B, H, T, Dv))
    S_all = np.zeros((B, H, Dk, Dv))
    for b in range(B):
        for h in range(H):
            S = np.zeros((Dk, Dv)) if initial_state is None else np.array(initial_state[b, h], np.float64)
            for t in range(T):
                kt = k[b, h, t]
                M = np.exp(g[b, h, t]) * (np.eye(Dk) - beta[b, h, t] * np.outer(kt, kt))
                S = M @ S + beta[b, h, t] * np.outer(kt, v[b, h, t])
                o[b, h, t] = scale * (S.T @ q[b, h, t])
            S_all[b, h] = S
    return o, S_all


def deltaproduct_fwd(q, k, v, beta, g, initial_state=None, scale=1.0, l2norm=False):
    """Decay once per token, then r corrections (I - b k k^T) S + b k v^T in order."""
    q, k, v, beta, g = (np.asarray(a, np.float64) for a in (q, k, v, beta, g))
    B, H, T, r, Dk = k.shape
    Dv = v.shape[-1]
    if l2norm:
        q, k = _unit(q), _unit(k)
    o = np.zeros((B, H, T, Dv))
    S_all = np.zeros((B, H, Dk, Dv))
    for b in range(B):
        for h in range(H):
            S = np.zeros((Dk, Dv)) if initial_state is None else np.array(initial_state[b, h], np.float64)
            for t in range(T):
                S = np.exp(g[b, h, t]) * S
                for j in range(r):
                    kt = k[b, h, t, j]
                    S = S - beta[b, h, t, j] * np.outer(kt, kt @ S) + beta[b, h, t, j] * np.outer(kt, v[b, h, t, j])
                o[b, h, t] = scale * (S.T @ q[b, h, t])
            S_all[b, h] = S
    return o, S_all


def masked_deltaproduct_fwd(q, k, v, beta, g, mask, initial_state=None, scale=1.0, l2norm=False):
    """Block-masked DeltaProduct: the state is r row blocks of Dk/r key rows;
    per token the decay once, then sub-row i reads sum_j mask[i][j] of the
    blocks' predictions and writes block i; all sub-rows from the same state."""
    q, k, v, beta, g, mask = (np.asarray(a, np.float64) for a in (q, k, v, beta, g, mask))
    B, H, T, Dk = q.shape
    Dv = v.shape[-1]
    r = mask.shape[0]
    dk = Dk // r
    if l2norm:
        q, k = _unit(q), _unit(k)
    o = np.zeros((B, H, T, Dv))
    S_all = np.zeros((B, H, Dk, Dv))
    for b in range(B):
        for h in range(H):
            S = np.zeros((Dk, Dv)) if initial_state is None else np.array(initial_state[b, h], np.float64)
            for t in range(T):
                S = np.exp(g[b, h, t]) * S
                kb = k[b, h, t].reshape(r, dk)
                z = np.stack([kb[j] @ S[j * dk:(j + 1) * dk] for j in range(r)])  # [r, Dv]
                d = beta[b, h, t] * (v[b, h, t][None, :] - mask @ z)
                for i in range(r):
                    S[i * dk:(i + 1) * dk] += np.outer(kb[i], d[i])
                o[b, h, t] = scale * (S.T @ q[b, h, t])
            S_all[b, h] = S
    return o, S_all


def cam_scan_fwd(q, k, v, beta, decay, initial_state=None, scale=1.0, reverse=False, l2norm=False):
    """Frame-level scan: per frame S <- d_f S, then the joint update
    S <- S + K_f^T diag(beta_f) (V_f - K_f S), and o = scale S^T q after it.
    reverse: frames last to first, frame f reading frames f+1.. only."""
    q, k, v, beta, decay = (np.asarray(a, np.float64) for a in (q, k, v, beta, decay))
    B, H, N, Dk = q.shape
    Dv = v.shape[-1]
    F = decay.shape[-1]
    S_len = N // F
    if l2norm:
        q, k = _unit(q), _unit(k)
    o = np.zeros((B, H, N, Dv))
    S_all = np.zeros((B, H, Dk, Dv))
    for b in range(B):
        for h in range(H):
            S = np.zeros((Dk, Dv)) if initial_state is None else np.array(initial_state[b, h], np.float64)
            order = range(F - 1, -1, -1) if reverse else range(F)
            for f in order:
                take = f + 1 if reverse else f  # frame whose keys enter before frame f reads
                if take < F:
                    sl = slice(take * S_len, (take + 1) * S_len)
                    Kf, Vf, bf = k[b, h, sl], v[b, h, sl], beta[b, h, sl]
                    S = decay[b, h, take] * S
                    S = S + Kf.T @ (bf[:, None] * (Vf - Kf @ S))
                ql = slice(f * S_len, (f + 1) * S_len)
                o[b, h, ql] = scale * (q[b, h, ql] @ S)
            S_all[b, h] = S
    return o, S_all


def rope_tables(N, D_half, base=10000.0):
    """Interleaved cos/sin tables: cos[n,2i]=cos[n,2i+1]=cos th, sin[n,2i]=-sin th,
    sin[n,2i+1]=sin th, th = n * base^(-2i/D_half)."""
    i = np.arange(D_half // 2, dtype=np.float64)
    th = np.arange(N, dtype=np.float64)[:, None] * base ** (-2.0 * i / D_half)[None, :]
    cos = np.repeat(np.cos(th), 2, axis=-1)
    sin = np.stack([-np.sin(th), np.sin(th)], axis=-1).reshape(N, D_half)
    return cos, sin


def cam_prep_fwd(q_raw, k_raw, v_raw, proj_q, proj_kv, q_norm_w=None, k_norm_w=None,
                 rope_cos=None, rope_sin=None, rope_base=10000.0, k_scale=0.5, eps=1e-6):
    q_raw, k_raw, v_raw = (np.asarray(a, np.float64) for a in (q_raw, k_raw, v_raw))
    B, N, H, D = q_raw.shape
    C, Dh = H * D, D // 2
    wq = np.ones(C) if q_norm_w is None else np.asarray(q_norm_w, np.float64)
    wk = np.ones(C) if k_norm_w is None else np.asarray(k_norm_w, np.float64)
    if rope_cos is None:
        rope_cos, rope_sin = rope_tables(N, Dh, rope_base)
    cs = np.asarray(rope_cos, np.float64)[None, :, None, :]
    sn = np.asarray(rope_sin, np.float64)[None, :, None, :]
    iq = 1.0 / np.sqrt((q_raw ** 2).sum((-1, -2)) / C + eps)
    ik = 1.0 / np.sqrt((k_raw ** 2).sum((-1, -2)) / C + eps)
    qn = np.maximum(q_raw * iq[..., None, None] * wq.reshape(H, D), 0.0)
    kn = np.maximum(k_raw * ik[..., None, None] * wk.reshape(H, D), 0.0) * k_scale
    vn = v_raw
    pre = (kn ** 2).sum(-1)
    Pq = np.asarray(proj_q, np.float64)
    Pk = np.asarray(proj_kv, np.float64)

    def project(x, P):
        xg = x[..., :Dh].reshape(B, N, H, Dh // 4, 4)
        return np.einsum("bnij,bnhgj->bnhgi", P, xg).reshape(B, N, H, Dh)

    def rotate(x):
        xs = x[..., Dh:]
        swapped = xs.reshape(B, N, H, Dh // 2, 2)[..., ::-1].reshape(B, N, H, Dh)
        return xs * cs + swapped * sn

    outs = []
    for x, P in ((qn, Pq), (kn, Pk), (vn, Pk)):
        y = np.concatenate([project(x, P), rotate(x)], axis=-1)
        outs.append(y)
    post = (outs[1] ** 2).sum(-1)
    q_out, k_out, v_out = (np.ascontiguousarray(y.transpose(0, 2, 1, 3)) for y in outs)
    return q_out, k_out, v_out, pre.transpose(0, 2, 1).copy(), post.transpose(0, 2, 1).copy()
