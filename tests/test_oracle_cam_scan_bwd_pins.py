"""Pins for the fp64 backward of the frame-level camera scan (fused_cam_gdn.py,
``_cam_scan_bwd_kernel``, forward direction): central finite differences of
the forward oracle, which the backward shares no code with, for every input
(q, k, v, beta, the per-frame decay and the initial state), with and without
the unit-norm flag, and the gradient of the final state."""
import numpy as np
import pytest

import oracle


def case(F=3, S=4, Dk=6, Dv=5, seed=0):
    rng = np.random.default_rng(seed)
    B, H = 1, 2
    q = rng.standard_normal((B, H, F * S, Dk))
    k = rng.standard_normal((B, H, F * S, Dk)) / np.sqrt(Dk)
    v = rng.standard_normal((B, H, F * S, Dv))
    beta = rng.random((B, H, F * S)) / S
    decay = 0.6 + 0.4 * rng.random((B, H, F))
    s0 = rng.standard_normal((B, H, Dk, Dv))
    go = rng.standard_normal((B, H, F * S, Dv))
    gs = rng.standard_normal((B, H, Dk, Dv))
    return q, k, v, beta, decay, s0, go, gs


def loss(args, go, gs, l2norm, scale):
    o, sf = oracle.cam_scan_fwd(*args, scale=scale, l2norm=l2norm)
    return float(np.sum(o * go) + np.sum(sf * gs))


@pytest.mark.parametrize("l2norm", [False, True])
def test_backward_matches_finite_differences(l2norm):
    q, k, v, beta, decay, s0, go, gs = case(seed=1 + int(l2norm))
    scale = 0.8
    grads = oracle.cam_scan_bwd(q, k, v, beta, decay, go, s0, gs, scale=scale, l2norm=l2norm)
    args = [q, k, v, beta, decay, s0]
    rng = np.random.default_rng(5)
    h = 1e-6
    for which in range(6):
        for _ in range(8):
            idx = tuple(int(rng.integers(0, n)) for n in args[which].shape)
            a = [x.copy() for x in args]
            a[which][idx] += h
            lp = loss(a, go, gs, l2norm, scale)
            a[which][idx] -= 2 * h
            lm = loss(a, go, gs, l2norm, scale)
            fd = (lp - lm) / (2 * h)
            assert abs(fd - grads[which][idx]) <= 2e-6 * max(1.0, abs(fd)), (which, idx, fd, grads[which][idx])


def test_frames_of_one_token_match_a_token_level_adjoint():
    """S = 1 makes the frame scan the GDN recurrence with g = log(decay); its
    backward is then checked against finite differences of the GDN oracle."""
    q, k, v, beta, decay, s0, go, gs = case(F=5, S=1, seed=3)
    grads = oracle.cam_scan_bwd(q, k, v, beta, decay, go, s0, None)
    h = 1e-6
    for t in range(5):
        kp, km = k.copy(), k.copy()
        kp[0, 1, t, 2] += h
        km[0, 1, t, 2] -= h
        lp = float(np.sum(oracle.gdn_fwd(q, kp, v, beta, np.log(decay), s0)[0] * go))
        lm = float(np.sum(oracle.gdn_fwd(q, km, v, beta, np.log(decay), s0)[0] * go))
        assert abs((lp - lm) / (2 * h) - grads[1][0, 1, t, 2]) < 1e-6
