"""Pins for the fp64 backward of the camera prep (fused_cam_gdn.py,
``_cam_prep_bwd_kernel``, continued through the full-C RMSNorm): central
finite differences of the forward oracle, which the backward shares no code
with, and the adjoint identity of the linear v path."""
import numpy as np
import pytest

import oracle
from gated_delta_rule_47_gb300.inputs import se3_inverse, se3_poses
import torch


def case(B=1, N=3, H=2, D=16, seed=0, tables=False):
    rng = np.random.default_rng(seed)
    q, k, v = (rng.standard_normal((B, N, H, D)) for _ in range(3))
    P = se3_poses(B * N, torch.Generator().manual_seed(seed))
    pq = P.transpose(-1, -2).reshape(B, N, 4, 4).numpy()
    pkv = se3_inverse(P).reshape(B, N, 4, 4).numpy()
    wq, wk = rng.random(H * D) + 0.5, rng.random(H * D) + 0.5
    g = [rng.standard_normal((B, H, N, D)) for _ in range(3)] + [rng.standard_normal((B, H, N)) for _ in range(2)]
    cos = sin = None
    if tables:
        from oracle import mirror
        cos, sin = mirror.rope_tables(N, D // 2, 100.0)
    return q, k, v, pq, pkv, wq, wk, g, cos, sin


def loss(q, k, v, pq, pkv, wq, wk, g, cos, sin):
    outs = oracle.cam_prep_fwd(q, k, v, pq, pkv, wq, wk, cos, sin, rope_base=100.0, k_scale=0.5, eps=1e-3)
    return sum(float(np.sum(a * b)) for a, b in zip(outs, g))


@pytest.mark.parametrize("tables", [False, True])
def test_backward_matches_finite_differences(tables):
    q, k, v, pq, pkv, wq, wk, g, cos, sin = case(tables=tables)
    dq, dk, dv = oracle.cam_prep_bwd(q, k, v, pq, pkv, g[0], g[1], g[2], g[3], g[4], wq, wk, cos, sin,
                                     rope_base=100.0, k_scale=0.5, eps=1e-3)
    h = 1e-6
    rng = np.random.default_rng(1)
    for which, grad in ((0, dq), (1, dk), (2, dv)):
        for _ in range(12):
            idx = tuple(int(rng.integers(0, n)) for n in q.shape)
            args = [q.copy(), k.copy(), v.copy()]
            args[which][idx] += h
            lp = loss(*args, pq, pkv, wq, wk, g, cos, sin)
            args[which][idx] -= 2 * h
            lm = loss(*args, pq, pkv, wq, wk, g, cos, sin)
            fd = (lp - lm) / (2 * h)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1.0, abs(fd)), (which, idx, fd, grad[idx])


def test_v_path_adjoint_identity():
    """v_out = J v_raw is linear, so <dv_out, J v> = <J^T dv_out, v> exactly."""
    q, k, v, pq, pkv, wq, wk, g, cos, sin = case(N=4, H=3, seed=2)
    _, _, vo, _, _ = oracle.cam_prep_fwd(q, k, v, pq, pkv, wq, wk, rope_base=100.0)
    _, _, dv = oracle.cam_prep_bwd(q, k, v, pq, pkv, g[0], g[1], g[2], None, None, wq, wk, rope_base=100.0)
    assert abs(np.sum(g[2] * vo) - np.sum(dv * v)) < 1e-10
