"""Pins for the fp64 block-masked DeltaProduct oracle (gated_deltaproduct
test.py: the mask_ij coupling in `gated_chunk_scaled_dot_kkt_fwd_kernel` and
`gated_fwd_recompute_w_u_kernel`, the per-slice state update of
`gated_chunk_delta_rule_fwd_kernel_h`, the sum over r in
`gated_chunk_fwd_o_fn`), each against something other than the oracle: the
pinned GDN oracle (all-ones mask; identity mask as r GDNs on the key slices),
the dense transition-matrix form, and the page's chunked form with its
mask-coupled A, for several chunk sizes."""
import numpy as np
import pytest

import oracle
from oracle import mirror


def inputs(B=1, H=2, T=11, Dk=8, Dv=5, r=2, seed=0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, H, T, Dk))
    k = rng.standard_normal((B, H, T, Dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, H, T, Dv))
    beta = rng.random((B, H, T))
    g = -rng.random((B, H, T)) / 4
    mask = rng.standard_normal((r, r)) * 0.5 + np.eye(r)
    s0 = rng.standard_normal((B, H, Dk, Dv))
    return q, k, v, beta, g, mask, s0


def test_c_matches_numpy_mirror():
    q, k, v, beta, g, mask, s0 = inputs(B=2, T=9, Dk=12, r=3, seed=1)
    a = oracle.masked_deltaproduct_fwd(q, k, v, beta, g, mask, s0, scale=0.6)
    b = mirror.masked_deltaproduct_fwd(q, k, v, beta, g, mask, s0, scale=0.6)
    assert np.max(np.abs(a[0] - b[0])) < 1e-12 and np.max(np.abs(a[1] - b[1])) < 1e-12


@pytest.mark.parametrize("r", [1, 2, 4])
def test_all_ones_mask_is_gdn(r):
    """Every sub-row reads the full key, so the r corrections together are one
    GDN correction: the all-ones mask gives the GDN recurrence exactly."""
    q, k, v, beta, g, _, s0 = inputs(T=13, Dk=8, r=r, seed=2)
    a = oracle.masked_deltaproduct_fwd(q, k, v, beta, g, np.ones((r, r)), s0)
    b = oracle.gdn_fwd(q, k, v, beta, g, s0)
    assert np.max(np.abs(a[0] - b[0])) < 1e-12 and np.max(np.abs(a[1] - b[1])) < 1e-12


def test_identity_mask_is_r_gdns_on_the_key_slices():
    """mask = I decouples the slices: r independent GDNs with keys, queries and
    state rows restricted to slice i, sharing v, beta and g; outputs add up."""
    r, Dk = 2, 8
    q, k, v, beta, g, _, s0 = inputs(T=10, Dk=Dk, r=r, seed=3)
    a = oracle.masked_deltaproduct_fwd(q, k, v, beta, g, np.eye(r), s0)
    dk = Dk // r
    o = 0.0
    for i in range(r):
        sl = slice(i * dk, (i + 1) * dk)
        oi, si = oracle.gdn_fwd(q[..., sl], k[..., sl], v, beta, g, s0[:, :, sl])
        o = o + oi
        assert np.max(np.abs(a[1][:, :, sl] - si)) < 1e-12
    assert np.max(np.abs(a[0] - o)) < 1e-12


def test_dense_transition_matrices():
    """S_t = e^{g_t} (I - beta_t (k_t k_t^T) o M) S_{t-1} + beta_t k_t v_t^T with
    M the mask expanded to Dk/r x Dk/r blocks (o: elementwise product)."""
    r, Dk = 2, 8
    q, k, v, beta, g, mask, s0 = inputs(T=9, Dk=Dk, r=r, seed=4)
    M = np.kron(mask, np.ones((Dk // r, Dk // r)))
    o, sf = oracle.masked_deltaproduct_fwd(q, k, v, beta, g, mask, s0, scale=0.9)
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            S = s0[b, h].copy()
            for t in range(q.shape[2]):
                kt = k[b, h, t]
                S = np.exp(g[b, h, t]) * (np.eye(Dk) - beta[b, h, t] * np.outer(kt, kt) * M) @ S \
                    + beta[b, h, t] * np.outer(kt, v[b, h, t])
                assert np.max(np.abs(o[b, h, t] - 0.9 * S.T @ q[b, h, t])) < 1e-12
            assert np.max(np.abs(sf[b, h] - S)) < 1e-12


def chunked(q, k, v, beta, g, mask, s0, C):
    """The page's chunk algorithm for this variant, as plain matrices: rows
    (t, i) of a chunk of C tokens, A[(t,i),(s,j)] = beta_t e^{G_t - G_s}
    mask[i][j] (k_t,(j) . k_s,(j)) for s < t (zero within a token),
    T = (I + A)^-1, W = T diag(beta e^G) [k_t (.) m_i], U = T diag(beta) [v_t],
    Delta = U - W S, outputs with the slice-wise q.k scores (s <= t) summed
    over r, and the slice-i state rows updated by Delta_(s,i)."""
    B, H, T_, Dk = q.shape
    r = mask.shape[0]
    dk = Dk // r
    o = np.zeros((B, H, T_, v.shape[-1]))
    fin = np.zeros_like(s0)
    for b in range(B):
        for h in range(H):
            S = s0[b, h].copy()
            for c0 in range(0, T_, C):
                n = min(C, T_ - c0)
                kk, qq, vv = k[b, h, c0:c0 + n], q[b, h, c0:c0 + n], v[b, h, c0:c0 + n]
                bb, G = beta[b, h, c0:c0 + n], np.cumsum(g[b, h, c0:c0 + n])
                ks = kk.reshape(n, r, dk)
                P = np.einsum("tjd,sjd->tsj", ks, ks)           # slice-wise k.k
                A = np.zeros((n, r, n, r))
                for t in range(n):
                    for s in range(t):
                        A[t, :, s, :] = bb[t] * np.exp(G[t] - G[s]) * mask * P[t, s][None, :]
                A = A.reshape(n * r, n * r)
                Tm = np.linalg.inv(np.eye(n * r) + A)
                read = (ks[:, None, :, :] * mask[None, :, :, None]).reshape(n, r, Dk)  # k_t (.) m_i
                W = Tm @ (np.repeat(bb * np.exp(G), r)[:, None] * read.reshape(n * r, Dk))
                U = Tm @ (np.repeat(bb, r)[:, None] * np.repeat(vv, r, axis=0))
                Dl = (U - W @ S).reshape(n, r, -1)
                qs = qq.reshape(n, r, dk)
                Pq = np.einsum("tjd,sjd->tsj", qs, ks)
                for t in range(n):
                    intra = sum(np.exp(G[t] - G[s]) * Pq[t, s, j] * Dl[s, j] for s in range(t + 1) for j in range(r))
                    o[b, h, c0 + t] = np.exp(G[t]) * (qq[t] @ S) + intra
                Snew = np.exp(G[-1]) * S
                for j in range(r):
                    Snew[j * dk:(j + 1) * dk] += sum(np.exp(G[-1] - G[s]) * np.outer(ks[s, j], Dl[s, j])
                                                     for s in range(n))
                S = Snew
            fin[b, h] = S
    return o, fin


@pytest.mark.parametrize("C", [1, 3, 4, 16])
def test_page_chunk_form_matches_the_token_recurrence(C):
    q, k, v, beta, g, mask, s0 = inputs(T=11, Dk=8, r=2, seed=5)
    a = oracle.masked_deltaproduct_fwd(q, k, v, beta, g, mask, s0)
    b = chunked(q, k, v, beta, g, mask, s0, C)
    assert np.max(np.abs(a[0] - b[0])) < 1e-10 and np.max(np.abs(a[1] - b[1])) < 1e-10


def test_pins_catch_planted_mistakes():
    """Writing with the read key (a plain expanded-row DeltaProduct with keys
    k (.) m_i), or updating the sub-rows one after the other, both differ from
    the dense form the pin above checks."""
    r, Dk = 2, 8
    q, k, v, beta, g, mask, s0 = inputs(T=8, Dk=Dk, r=r, seed=6)
    ref, _ = oracle.masked_deltaproduct_fwd(q, k, v, beta, g, mask, s0)
    dk = Dk // r
    read = (k.reshape(*k.shape[:3], r, dk)[..., None, :, :] * mask[:, :, None]).reshape(*k.shape[:3], r, Dk)
    wrong, _ = oracle.deltaproduct_fwd(q, read, np.repeat(v[:, :, :, None], r, 3),
                                       np.repeat(beta[..., None], r, -1), g, s0)
    assert np.max(np.abs(wrong - ref)) > 1e-3
    # sequential sub-rows: each reads the state after the previous sub-row
    seq = np.zeros_like(ref)
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            S = s0[b, h].copy()
            for t in range(q.shape[2]):
                S = np.exp(g[b, h, t]) * S
                kb = k[b, h, t].reshape(r, dk)
                for i in range(r):
                    z = np.stack([kb[j] @ S[j * dk:(j + 1) * dk] for j in range(r)])
                    S[i * dk:(i + 1) * dk] += np.outer(kb[i], beta[b, h, t] * (v[b, h, t] - mask[i] @ z))
                seq[b, h, t] = S.T @ q[b, h, t]
    assert np.max(np.abs(seq - ref)) > 1e-3
