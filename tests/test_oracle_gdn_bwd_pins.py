"""Pins for the fp64 backward of the GDN / DeltaProduct recurrence and of the
block-masked DeltaProduct (gated_deltaproduct test.py: the backward kernels
`gated_chunk_delta_rule_bwd_kernel_dhu`, `gated_chunk_delta_rule_bwd_kernel_dqkw`
and `gated_bwd_prepare_wy_repr_kernel` compute these gradients chunk-wise).

Every gradient is checked against central finite differences of the forward
oracle, which the backward shares no code with, for every input (q, k, v,
beta, g, the initial state), with and without the unit-norm flag, across a
checkpoint boundary of the backward's state rebuild (T = 70 > 64).  Two more
pins tie the backward functions to each other and to the frame scan's: an
all-ones mask makes the masked variant GDN, and frames of one token make the
frame scan GDN with decay = exp(g)."""
import numpy as np
import pytest

import oracle


def case(T=70, r=1, Dk=6, Dv=5, seed=0, masked=False):
    rng = np.random.default_rng(seed)
    B, H = 1, 2
    q = rng.standard_normal((B, H, T, Dk))
    ksh = (B, H, T, Dk) if (masked or r == 0) else (B, H, T, r, Dk)
    vsh = (B, H, T, Dv) if masked else (B, H, T, r, Dv)
    bsh = (B, H, T) if masked else (B, H, T, r)
    k = rng.standard_normal(ksh) / np.sqrt(Dk)
    v = rng.standard_normal(vsh)
    beta = rng.random(bsh)
    g = -0.3 * rng.random((B, H, T))
    s0 = rng.standard_normal((B, H, Dk, Dv))
    go = rng.standard_normal((B, H, T, Dv))
    gs = rng.standard_normal((B, H, Dk, Dv))
    return q, k, v, beta, g, s0, go, gs


def fd_check(fwd, grads, args, go, gs, picks=6, h=1e-6, tol=3e-6, seed=5):
    def loss(a):
        o, sf = fwd(*a)
        return float(np.sum(o * go) + np.sum(sf * gs))

    rng = np.random.default_rng(seed)
    for which in range(len(args)):
        for _ in range(picks):
            idx = tuple(int(rng.integers(0, n)) for n in args[which].shape)
            a = [x.copy() for x in args]
            a[which][idx] += h
            lp = loss(a)
            a[which][idx] -= 2 * h
            lm = loss(a)
            fd = (lp - lm) / (2 * h)
            got = grads[which][idx]
            assert abs(fd - got) <= tol * max(1.0, abs(fd)), (which, idx, fd, got)


@pytest.mark.parametrize("l2norm", [False, True])
def test_gdn_backward_matches_finite_differences(l2norm):
    q, k, v, beta, g, s0, go, gs = case(seed=1 + int(l2norm))
    k, v, beta = k[:, :, :, 0], v[:, :, :, 0], beta[:, :, :, 0]
    scale = 0.7
    grads = oracle.gdn_bwd(q, k, v, beta, g, go, s0, gs, scale=scale, l2norm=l2norm)
    fwd = lambda q_, k_, v_, b_, g_, s_: oracle.gdn_fwd(q_, k_, v_, b_, g_, s_, scale=scale, l2norm=l2norm)
    fd_check(fwd, grads, [q, k, v, beta, g, s0], go, gs)


@pytest.mark.parametrize("r,l2norm", [(2, False), (3, True)])
def test_deltaproduct_backward_matches_finite_differences(r, l2norm):
    q, k, v, beta, g, s0, go, gs = case(T=67, r=r, seed=10 + r)
    grads = oracle.deltaproduct_bwd(q, k, v, beta, g, go, s0, gs, scale=1.3, l2norm=l2norm)
    fwd = lambda *a: oracle.deltaproduct_fwd(*a, scale=1.3, l2norm=l2norm)
    fd_check(fwd, grads, [q, k, v, beta, g, s0], go, gs)


@pytest.mark.parametrize("r,l2norm", [(2, False), (3, True)])
def test_masked_backward_matches_finite_differences(r, l2norm):
    q, k, v, beta, g, s0, go, gs = case(T=66, seed=20 + r, masked=True)
    rng = np.random.default_rng(40 + r)
    mask = rng.standard_normal((r, r))  # not symmetric: catches a transposed mask
    grads = oracle.masked_deltaproduct_bwd(q, k, v, beta, g, mask, go, s0, gs, scale=0.9, l2norm=l2norm)
    fwd = lambda q_, k_, v_, b_, g_, s_: oracle.masked_deltaproduct_fwd(q_, k_, v_, b_, g_, mask, s_, scale=0.9,
                                                                        l2norm=l2norm)
    fd_check(fwd, grads, [q, k, v, beta, g, s0], go, gs)


def test_no_final_state_gradient_and_no_initial_state():
    """None for the final-state gradient is zero, and None for the initial
    state is the zero state: the gradients equal the ones with explicit zeros."""
    q, k, v, beta, g, s0, go, gs = case(T=20, seed=7)
    k, v, beta = k[:, :, :, 0], v[:, :, :, 0], beta[:, :, :, 0]
    a = oracle.gdn_bwd(q, k, v, beta, g, go, None, None)
    b = oracle.gdn_bwd(q, k, v, beta, g, go, np.zeros_like(s0), np.zeros_like(gs))
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


def test_zero_beta_is_decayed_linear_attention():
    """beta = 0 leaves S_t = e^{gamma_t} S_0 (gamma_t = sum of g up to t), so
    o_t = scale e^{gamma_t} S_0^T q_t; the gradients then have closed forms:
    dS_0 = scale sum_t e^{gamma_t} q_t do_t^T,  dq_t = scale e^{gamma_t} S_0 do_t,
    dv = 0,  dg_m = sum_{t >= m} scale e^{gamma_t} q_t^T S_0 do_t."""
    q, k, v, beta, g, s0, go, gs = case(T=9, seed=8)
    k, v = k[:, :, :, 0], v[:, :, :, 0]
    beta = np.zeros(beta.shape[:3])
    scale = 1.7
    dq, dk, dv, db, dg, ds0 = oracle.gdn_bwd(q, k, v, beta, g, go, s0, None, scale=scale)
    gam = np.cumsum(g, axis=-1)
    e = np.exp(gam)
    np.testing.assert_allclose(ds0, scale * np.einsum("bht,bhti,bhtj->bhij", e, q, go), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dq, scale * e[..., None] * np.einsum("bhij,bhtj->bhti", s0, go), rtol=1e-12,
                               atol=1e-12)
    assert np.all(dv == 0.0) and np.all(dk == 0.0)
    per_t = scale * e * np.einsum("bhti,bhij,bhtj->bht", q, s0, go)
    np.testing.assert_allclose(dg, np.cumsum(per_t[..., ::-1], axis=-1)[..., ::-1], rtol=1e-11, atol=1e-12)


def test_all_ones_mask_is_gdn():
    """An all-ones mask makes the block-masked recurrence the GDN recurrence,
    so the two backward functions (written separately) agree."""
    q, k, v, beta, g, s0, go, gs = case(T=30, seed=9, masked=True)
    for r in (2, 3):
        a = oracle.masked_deltaproduct_bwd(q, k, v, beta, g, np.ones((r, r)), go, s0, gs, l2norm=True)
        b = oracle.gdn_bwd(q, k, v, beta, g, go, s0, gs, l2norm=True)
        for x, y in zip(a, b):
            np.testing.assert_allclose(x, y, rtol=1e-10, atol=1e-11)


def test_frames_of_one_token_are_gdn():
    """The frame scan with frames of one token is GDN with decay = exp(g); its
    backward (a separate function) gives the same q, k, v, beta and initial
    state gradients, and ddecay = dg / decay."""
    q, k, v, beta, g, s0, go, gs = case(T=12, seed=11)
    k, v, beta = k[:, :, :, 0], v[:, :, :, 0], beta[:, :, :, 0]
    a = oracle.gdn_bwd(q, k, v, beta, g, go, s0, gs, scale=0.5)
    b = oracle.cam_scan_bwd(q, k, v, beta, np.exp(g), go, s0, gs, scale=0.5)
    for i in (0, 1, 2, 3, 5):
        np.testing.assert_allclose(a[i], b[i], rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(a[4], b[4] * np.exp(g), rtol=1e-10, atol=1e-11)
