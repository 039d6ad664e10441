"""Pins for the fp64 oracle: facts fixed by the definition and by mathematics,
checked against something other than the oracle itself.

GDN:    S_t = e^{g_t}(I - b_t k_t k_t^T)S_{t-1} + b_t k_t v_t^T,  o_t = S_t^T q_t
        (gated_deltaproduct test.py, state-scan / output kernels;
         fused_cam_gdn.py, ``_cam_scan_kernel``).
Every case uses Dk != Dv so that a transposed state or operand cannot pass.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import mirror
from tests.wy_reference import brute_force, brute_force_deltaproduct, chunked_wy


def rand_case(B=1, H=2, T=12, Dk=6, Dv=5, seed=0, r=None, unit=True, s0=True):
    rng = np.random.default_rng(seed)
    sub = () if r is None else (r,)
    q = rng.standard_normal((B, H, T, Dk))
    k = rng.standard_normal((B, H, T, *sub, Dk))
    if unit:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, H, T, *sub, Dv))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, H, T, *sub))))
    g = -np.log1p(np.exp(-rng.standard_normal((B, H, T)))) / 4.0
    S0 = rng.standard_normal((B, H, Dk, Dv)) if s0 else None
    return q, k, v, beta, g, S0


def rel(a, b):
    return np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300)


# ---------------------------------------------------------------- GDN pins

def test_c_oracle_matches_numpy_mirror():
    q, k, v, beta, g, S0 = rand_case(B=2, H=2, T=20, seed=1)
    o, sf = oracle.gdn_fwd(q, k, v, beta, g, S0, scale=0.7)
    om, sm = mirror.gdn_fwd(q, k, v, beta, g, S0, scale=0.7)
    assert rel(o, om) < 1e-13 and rel(sf, sm) < 1e-13


def test_beta_zero_is_pure_decay():
    """beta = 0: S_t = e^{sum_{i<=t} g_i} S0 and o_t = S_t^T q_t (closed form)."""
    q, k, v, beta, g, S0 = rand_case(T=15, seed=2)
    beta[:] = 0.0
    o, sf = oracle.gdn_fwd(q, k, v, beta, g, S0)
    G = np.cumsum(g, axis=-1)
    expect = np.exp(G)[..., None] * np.einsum("bhij,bhti->bhtj", S0, q)
    assert rel(o, expect) < 1e-13
    assert rel(sf, np.exp(G[..., -1])[..., None, None] * S0) < 1e-13


def orthonormal_keys(T, Dk, seed):
    rng = np.random.default_rng(seed)
    Qm, _ = np.linalg.qr(rng.standard_normal((Dk, Dk)))
    return Qm[:T]


def test_exact_overwrite_with_orthonormal_keys():
    """g = 0, beta = 1 and orthonormal keys: S_t = sum_{i<=t} k_i v_i^T, so
    o_t = sum_{i<=t} (q_t.k_i) v_i, and querying k_i returns v_i."""
    T, Dk, Dv = 7, 9, 4
    K = orthonormal_keys(T, Dk, 3)
    rng = np.random.default_rng(4)
    V = rng.standard_normal((T, Dv))
    Q = rng.standard_normal((T, Dk))
    one = lambda x: x[None, None]
    o, sf = oracle.gdn_fwd(one(Q), one(K), one(V), np.ones((1, 1, T)), np.zeros((1, 1, T)))
    expect = np.stack([sum((Q[t] @ K[i]) * V[i] for i in range(t + 1)) for t in range(T)])
    assert np.max(np.abs(o[0, 0] - expect)) < 1e-12
    # reading back with q_t = k_t returns v_t exactly
    o2, _ = oracle.gdn_fwd(one(K), one(K), one(V), np.ones((1, 1, T)), np.zeros((1, 1, T)))
    assert np.max(np.abs(o2[0, 0] - V)) < 1e-12
    assert np.max(np.abs(sf[0, 0] - K.T @ V)) < 1e-12


def test_repeated_key_returns_latest_value():
    Dk, Dv = 5, 3
    K = orthonormal_keys(2, Dk, 5)
    keys = np.stack([K[0], K[1], K[0]])
    vals = np.array([[1.0, 2.0, 3.0], [4.0, 5.0, 6.0], [-7.0, 8.0, 0.5]])
    queries = np.stack([K[0], K[1], K[0]])
    one = lambda x: x[None, None]
    o, _ = oracle.gdn_fwd(one(queries), one(keys), one(vals), np.ones((1, 1, 3)), np.zeros((1, 1, 3)))
    assert np.allclose(o[0, 0, 2], vals[2], atol=1e-13)  # latest write for k_0
    assert np.allclose(o[0, 0, 1], vals[1], atol=1e-13)


def test_brute_force_products_small_T():
    for T in (1, 2, 5, 16):
        q, k, v, beta, g, S0 = rand_case(T=T, seed=10 + T, unit=False)
        o, sf = oracle.gdn_fwd(q, k, v, beta, g, S0, scale=1.3)
        ob, sb = brute_force(q, k, v, beta, g, S0, scale=1.3)
        assert rel(o, ob) < 1e-12 and rel(sf, sb) < 1e-12, T


@pytest.mark.parametrize("C", [1, 2, 16, 64, 100])
def test_chunk_size_independence_via_wy(C):
    """The chunkwise WY form (decay-masked KK^T, (I+A)^-1, w, u, state scan,
    output) is exact algebra: it must equal the token loop for any chunk size,
    including a ragged last chunk (T = 100 is not a multiple of 16 or 64)."""
    q, k, v, beta, g, S0 = rand_case(B=1, H=2, T=100, Dk=8, Dv=6, seed=20)
    o, sf = oracle.gdn_fwd(q, k, v, beta, g, S0, scale=0.5)
    ow, sw = chunked_wy(q, k, v, beta, g, S0, C=C, scale=0.5)
    assert rel(o, ow) < 1e-12 and rel(sf, sw) < 1e-12


def test_split_and_resume_is_identical():
    q, k, v, beta, g, S0 = rand_case(T=40, seed=30)
    o, sf = oracle.gdn_fwd(q, k, v, beta, g, S0)
    t0 = 17
    sl = lambda x, a, b: x[:, :, a:b]
    o1, s1 = oracle.gdn_fwd(*(sl(x, 0, t0) for x in (q, k, v, beta, g)), S0)
    o2, s2 = oracle.gdn_fwd(*(sl(x, t0, 40) for x in (q, k, v, beta, g)), s1)
    assert np.array_equal(np.concatenate([o1, o2], axis=2), o)
    assert np.array_equal(s2, sf)


def test_householder_step_preserves_frobenius_norm():
    """beta = 2, unit keys, g = 0, v = 0: each step is the reflection
    I - 2kk^T, which is orthogonal, so ||S_t||_F = ||S_0||_F."""
    q, k, v, beta, g, S0 = rand_case(T=30, seed=40)
    beta[:] = 2.0
    g[:] = 0.0
    v[:] = 0.0
    _, sf = oracle.gdn_fwd(q, k, v, beta, g, S0)
    assert np.allclose(np.linalg.norm(sf, axis=(-2, -1)), np.linalg.norm(S0, axis=(-2, -1)), rtol=1e-13)


def test_exact_rational_example():
    """A 3-token example in exact rational arithmetic: decay 1/2 (g = -ln 2),
    integer keys and values, beta = 1/2 and 1/4."""
    Dk, Dv = 2, 3
    K = [[1, 0], [1, 1], [0, 2]]
    V = [[1, 2, 3], [0, -1, 1], [2, 2, -2]]
    Qv = [[1, 1], [2, -1], [0, 1]]
    B_ = [Fraction(1, 2), Fraction(1, 4), Fraction(1, 2)]
    S = [[Fraction(0)] * Dv for _ in range(Dk)]
    outs = []
    for t in range(3):
        S = [[Fraction(1, 2) * x for x in row] for row in S]
        p = [sum(S[i][j] * K[t][i] for i in range(Dk)) for j in range(Dv)]
        S = [[S[i][j] + B_[t] * K[t][i] * (V[t][j] - p[j]) for j in range(Dv)] for i in range(Dk)]
        outs.append([sum(S[i][j] * Qv[t][i] for i in range(Dk)) for j in range(Dv)])
    expect = np.array([[float(x) for x in row] for row in outs])
    a = lambda x: np.asarray(x, np.float64)[None, None]
    o, _ = oracle.gdn_fwd(a(Qv), a(K), a(V), a([float(b) for b in B_]), np.full((1, 1, 3), -np.log(2.0)))
    assert np.max(np.abs(o[0, 0] - expect)) < 1e-14


def test_l2norm_flag_equals_prenormalised_inputs():
    q, k, v, beta, g, S0 = rand_case(T=10, seed=50, unit=False)
    o1, s1 = oracle.gdn_fwd(q, k, v, beta, g, S0, l2norm=True)
    qn = q / np.linalg.norm(q, axis=-1, keepdims=True)
    kn = k / np.linalg.norm(k, axis=-1, keepdims=True)
    o2, s2 = oracle.gdn_fwd(qn, kn, v, beta, g, S0)
    assert rel(o1, o2) < 1e-14 and rel(s1, s2) < 1e-14


# Planted mistakes: each wrong variant of the recurrence must fail the brute
# force pin, so the pin is sensitive to the slips it is meant to catch.
def _variant_loop(q, k, v, beta, g, S0, mode):
    B, H, T, Dk = q.shape
    Dv = v.shape[-1]
    o = np.zeros((B, H, T, Dv))
    for b in range(B):
        for h in range(H):
            S = S0[b, h].copy()
            for t in range(T):
                kt, bt = k[b, h, t], beta[b, h, t]
                before = S.T @ q[b, h, t]
                if mode == "decay_after":
                    S = S - bt * np.outer(kt, kt @ S) + bt * np.outer(kt, v[b, h, t])
                    S = np.exp(g[b, h, t]) * S
                else:
                    S = np.exp(g[b, h, t]) * S
                    sign = -1.0 if mode == "sign" else 1.0
                    S = S - sign * bt * np.outer(kt, kt @ S) + bt * np.outer(kt, v[b, h, t])
                o[b, h, t] = before if mode == "exclusive" else S.T @ q[b, h, t]
    return o


@pytest.mark.parametrize("mode", ["decay_after", "sign", "exclusive"])
def test_pins_catch_planted_mistakes(mode):
    q, k, v, beta, g, S0 = rand_case(T=8, seed=60, unit=False)
    ob, _ = brute_force(q, k, v, beta, g, S0)
    assert rel(_variant_loop(q, k, v, beta, g, S0, "none"), ob) < 1e-12
    assert rel(_variant_loop(q, k, v, beta, g, S0, mode), ob) > 1e-3


# ------------------------------------------------------- DeltaProduct pins

def test_deltaproduct_r1_equals_gdn_bitwise():
    q, k, v, beta, g, S0 = rand_case(T=25, seed=70)
    o1, s1 = oracle.gdn_fwd(q, k, v, beta, g, S0, scale=0.9)
    o2, s2 = oracle.deltaproduct_fwd(q, k[:, :, :, None], v[:, :, :, None], beta[..., None], g, S0,
                                     scale=0.9)
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2)


def test_deltaproduct_matches_mirror_and_brute_force():
    q, k, v, beta, g, S0 = rand_case(T=9, seed=80, r=3)
    o, sf = oracle.deltaproduct_fwd(q, k, v, beta, g, S0, scale=1.1)
    om, sm = mirror.deltaproduct_fwd(q, k, v, beta, g, S0, scale=1.1)
    ob, sb = brute_force_deltaproduct(q, k, v, beta, g, S0, scale=1.1)
    assert rel(o, om) < 1e-13 and rel(sf, sm) < 1e-13
    assert rel(o, ob) < 1e-12 and rel(sf, sb) < 1e-12


def test_deltaproduct_is_gdn_over_expanded_rows():
    """Rows (t, j) in order form a GDN sequence of length r*T with the decay on
    row j = 0 only; the DeltaProduct output of token t is the GDN output of
    row (t, r-1) read with q_t."""
    r = 2
    q, k, v, beta, g, S0 = rand_case(T=11, seed=90, r=r)
    B, H, T, _, Dk = k.shape
    o, sf = oracle.deltaproduct_fwd(q, k, v, beta, g, S0)
    gr = np.zeros((B, H, T, r))
    gr[..., 0] = g
    qr = np.repeat(q[:, :, :, None, :], r, axis=3)
    og, sg = oracle.gdn_fwd(qr.reshape(B, H, T * r, Dk), k.reshape(B, H, T * r, Dk),
                            v.reshape(B, H, T * r, -1), beta.reshape(B, H, T * r),
                            gr.reshape(B, H, T * r), S0)
    assert rel(o, og.reshape(B, H, T, r, -1)[:, :, :, r - 1]) < 1e-13
    assert rel(sf, sg) < 1e-13


def test_deltaproduct_zero_beta_substeps_reduce_to_gdn():
    q, k, v, beta, g, S0 = rand_case(T=13, seed=100, r=3)
    beta[..., 1:] = 0.0
    o, sf = oracle.deltaproduct_fwd(q, k, v, beta, g, S0)
    og, sg = oracle.gdn_fwd(q, k[:, :, :, 0], v[:, :, :, 0], beta[..., 0], g, S0)
    assert rel(o, og) < 1e-14 and rel(sf, sg) < 1e-14
