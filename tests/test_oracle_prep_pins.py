"""Pins for the fp64 camera-prep oracle (fused_cam_gdn.py,
``_torch_cam_prep_reference`` / ``_cam_prep_kernel``): closed forms and
invariants of full-C RMSNorm, ReLU/K-scale, the per-token 4x4 projection and
the interleaved-pair rotary embedding."""
import numpy as np
import torch

import oracle
from oracle import mirror
from gated_delta_rule_47_gb300.inputs import se3_inverse, se3_poses


def raw(B=1, N=6, H=3, D=16, seed=0, positive=False):
    rng = np.random.default_rng(seed)
    x = [rng.standard_normal((B, N, H, D)) for _ in range(3)]
    if positive:
        x = [np.abs(a) + 0.01 for a in x]
    return x


def eye_proj(B, N):
    return np.broadcast_to(np.eye(4), (B, N, 4, 4)).copy()


def flat_tables(N, D):
    return np.ones((N, D // 2)), np.zeros((N, D // 2))


def test_c_matches_numpy_mirror():
    B, N, H, D = 2, 9, 3, 16
    q, k, v = raw(B, N, H, D, seed=1)
    gen = torch.Generator().manual_seed(0)
    P = se3_poses(B * N, gen)
    pq = P.transpose(-1, -2).reshape(B, N, 4, 4).numpy()
    pkv = se3_inverse(P).reshape(B, N, 4, 4).numpy()
    rng = np.random.default_rng(2)
    wq, wk = rng.random(H * D) + 0.5, rng.random(H * D) + 0.5
    a = oracle.cam_prep_fwd(q, k, v, pq, pkv, wq, wk, k_scale=0.5, eps=1e-6)
    b = mirror.cam_prep_fwd(q, k, v, pq, pkv, wq, wk, k_scale=0.5, eps=1e-6)
    for x, y in zip(a, b):
        assert np.max(np.abs(x - y)) < 1e-12


def test_identity_projection_and_zero_angle_give_plain_rmsnorm():
    """P = I and cos = 1, sin = 0: with positive inputs ReLU is the identity,
    so the mean square of q over C = H*D is ms/(ms+eps), that of k is
    k_scale^2 ms/(ms+eps), and v passes through untouched (no norm, ReLU or
    K-scale on v)."""
    B, N, H, D = 1, 5, 4, 16
    q, k, v = raw(B, N, H, D, seed=3, positive=True)
    eps, ks = 1e-2, 0.5
    c, s = flat_tables(N, D)
    qo, ko, vo, pre, post = oracle.cam_prep_fwd(q, k, v, eye_proj(B, N), eye_proj(B, N),
                                                rope_cos=c, rope_sin=s, k_scale=ks, eps=eps)
    C = H * D
    msq = (q ** 2).sum((-1, -2)) / C
    msk = (k ** 2).sum((-1, -2)) / C
    assert np.allclose((qo ** 2).sum((1, 3)) / C, msq / (msq + eps), rtol=1e-13)
    assert np.allclose((ko ** 2).sum((1, 3)) / C, ks ** 2 * msk / (msk + eps), rtol=1e-13)
    assert np.array_equal(vo, v.transpose(0, 2, 1, 3))
    assert np.allclose(pre, post, rtol=1e-14)


def test_relu_zeroes_negative_channels():
    B, N, H, D = 1, 3, 2, 8
    q, k, v = raw(B, N, H, D, seed=4)
    c, s = flat_tables(N, D)
    qo, ko, *_ = oracle.cam_prep_fwd(q, k, v, eye_proj(B, N), eye_proj(B, N), rope_cos=c, rope_sin=s)
    assert np.all(qo[(q < 0).transpose(0, 2, 1, 3)] == 0.0)
    assert np.all(ko[(k < 0).transpose(0, 2, 1, 3)] == 0.0)


def test_rope_preserves_pair_norms():
    B, N, H, D = 1, 40, 2, 16
    q, k, v = raw(B, N, H, D, seed=5)
    c, s = flat_tables(N, D)
    base = oracle.cam_prep_fwd(q, k, v, eye_proj(B, N), eye_proj(B, N), rope_cos=c, rope_sin=s)
    rot = oracle.cam_prep_fwd(q, k, v, eye_proj(B, N), eye_proj(B, N))  # angles from rope_base
    for x0, x1 in zip(base[:3], rot[:3]):
        p0 = (x0[..., D // 2:].reshape(B, H, N, -1, 2) ** 2).sum(-1)
        p1 = (x1[..., D // 2:].reshape(B, H, N, -1, 2) ** 2).sum(-1)
        assert np.allclose(p0, p1, rtol=1e-12)
        assert np.array_equal(x0[..., :D // 2], x1[..., :D // 2])
    assert not np.allclose(base[0][:, :, 1:, D // 2:], rot[0][:, :, 1:, D // 2:])


def test_rope_half_scores_depend_only_on_relative_position():
    """Place the same raw rows at positions (i, j) and (i+s, j+s): the RoPE-half
    score q'_i . k'_j is unchanged."""
    B, N, H, D = 1, 64, 2, 16
    rng = np.random.default_rng(6)
    rowq, rowk = rng.standard_normal((H, D)), rng.standard_normal((H, D))
    q = rng.standard_normal((B, N, H, D))
    k = rng.standard_normal((B, N, H, D))
    v = np.zeros((B, N, H, D))
    i, j, shift = 3, 10, 37
    for p in (i, i + shift):
        q[0, p] = rowq
    for p in (j, j + shift):
        k[0, p] = rowk
    qo, ko, *_ = oracle.cam_prep_fwd(q, k, v, eye_proj(B, N), eye_proj(B, N), rope_base=100.0)
    h = slice(D // 2, D)
    s1 = (qo[0, :, i, h] * ko[0, :, j, h]).sum(-1)
    s2 = (qo[0, :, i + shift, h] * ko[0, :, j + shift, h]).sum(-1)
    assert np.allclose(s1, s2, rtol=1e-10)
    s3 = (qo[0, :, i + 1, h] * ko[0, :, j, h]).sum(-1)
    assert not np.allclose(s1, s3)


def test_projection_half_scores_are_invariant_to_a_common_pose():
    """q uses P^T and k uses P^-1, so the projection-half score of tokens i, j
    is q^T P_i P_j^-1 k: replacing every P_n by P_n G leaves it unchanged.
    The inverses here come from numpy's general inverse."""
    B, N, H, D = 1, 7, 2, 16
    q, k, v = raw(B, N, H, D, seed=7)
    gen = torch.Generator().manual_seed(1)
    P = se3_poses(N, gen).numpy()
    G = se3_poses(1, gen).numpy()[0]

    def run(Ps):
        pq = np.transpose(Ps, (0, 2, 1))[None]
        pkv = np.linalg.inv(Ps)[None]
        return oracle.cam_prep_fwd(q, k, v, pq, pkv, rope_base=10000.0)

    a = run(P)
    b = run(P @ G)
    h = slice(0, D // 2)
    sa = np.einsum("bhid,bhjd->bhij", a[0][..., h], a[1][..., h])
    sb = np.einsum("bhid,bhjd->bhij", b[0][..., h], b[1][..., h])
    assert np.allclose(sa, sb, rtol=1e-9, atol=1e-9)
    # a transposed application (P^T in place of P) breaks the invariance
    bad_a = oracle.cam_prep_fwd(q, k, v, P[None], np.transpose(np.linalg.inv(P), (0, 2, 1))[None])
    bad_b = oracle.cam_prep_fwd(q, k, v, (P @ G)[None], np.transpose(np.linalg.inv(P @ G), (0, 2, 1))[None])
    ta = np.einsum("bhid,bhjd->bhij", bad_a[0][..., h], bad_a[1][..., h])
    tb = np.einsum("bhid,bhjd->bhij", bad_b[0][..., h], bad_b[1][..., h])
    assert not np.allclose(ta, tb, rtol=1e-6)


def test_rigid_rotation_preserves_k_norm():
    """A pure rotation (t = 0) is orthogonal on each group of four, and RoPE is
    orthogonal on each pair, so ||k_post|| = ||k_pre||."""
    B, N, H, D = 1, 8, 3, 16
    q, k, v = raw(B, N, H, D, seed=8)
    gen = torch.Generator().manual_seed(2)
    P = se3_poses(N, gen)
    P[:, :3, 3] = 0.0
    pkv = se3_inverse(P).numpy()[None]
    *_, pre, post = oracle.cam_prep_fwd(q, k, v, P.numpy().transpose(0, 2, 1)[None], pkv)
    assert np.allclose(pre, post, rtol=1e-12)
    P2 = se3_poses(N, gen)
    *_, pre2, post2 = oracle.cam_prep_fwd(q, k, v, P2.numpy().transpose(0, 2, 1)[None],
                                          se3_inverse(P2).numpy()[None])
    assert not np.allclose(pre2, post2)


def test_closed_form_se3_inverse():
    gen = torch.Generator().manual_seed(3)
    P = se3_poses(50, gen)
    assert np.allclose(se3_inverse(P).numpy(), np.linalg.inv(P.numpy()), atol=1e-12)
    R = P[:, :3, :3].numpy()
    assert np.allclose(R @ R.transpose(0, 2, 1), np.eye(3), atol=1e-12)
    assert np.allclose(np.linalg.det(R), 1.0)


def test_k_norm_outputs_are_sums_of_squares():
    B, N, H, D = 2, 5, 2, 16
    q, k, v = raw(B, N, H, D, seed=9)
    gen = torch.Generator().manual_seed(4)
    P = se3_poses(B * N, gen)
    qo, ko, vo, pre, post = oracle.cam_prep_fwd(
        q, k, v, P.transpose(-1, -2).reshape(B, N, 4, 4).numpy(),
        se3_inverse(P).reshape(B, N, 4, 4).numpy(), k_scale=0.5)
    assert np.allclose(post, (ko ** 2).sum(-1), rtol=1e-13)
    ik = 1.0 / np.sqrt((k ** 2).sum((-1, -2)) / (H * D) + 1e-6)
    kn = np.maximum(k * ik[..., None, None], 0.0) * 0.5
    assert np.allclose(pre, (kn ** 2).sum(-1).transpose(0, 2, 1), rtol=1e-13)
    infl = oracle.inflation_sq(pre, post)
    assert np.all(infl > 0)


def _rope_probe(D=16, N=8):
    """v_raw with a known pair (a, b) = (0.6, -0.8) in every rotary pair and
    ones elsewhere; P = I so the projection half passes through.  v skips the
    norm, ReLU and K-scale, so v_out's rotary half is the rotation alone."""
    B, H = 1, 1
    v = np.ones((B, N, H, D))
    v[..., D // 2::2] = 0.6
    v[..., D // 2 + 1::2] = -0.8
    q = np.ones((B, N, H, D))
    k = np.ones((B, N, H, D))
    return q, k, v, eye_proj(B, N)


def _hand_rotated_pair(n, i):
    """fused_cam_gdn.py, ``_prepare_ucpe_rope_tables``: pair i of position n
    turns by th = n * 10000^(-2i/(D/2)); with D = 16, D/2 = 8, that is
    n * 10^-i (10000^(-2i/8) = 10^(-i)), so th(1, 0) = 1 rad and th(7, 3) =
    0.007 rad.  y[2i] = x[2i] cos th - x[2i+1] sin th,
    y[2i+1] = x[2i] sin th + x[2i+1] cos th."""
    th = n * [1.0, 0.1, 0.01, 0.001][i]
    a, b = 0.6, -0.8
    return a * np.cos(th) - b * np.sin(th), a * np.sin(th) + b * np.cos(th)


def test_rope_direction_and_frequencies_against_hand_computed_angles():
    """Pins the rotation's sign and its frequency schedule at positions 1 and
    7, pairs 0 and 3, with the angles the oracle forms itself and with the
    interleaved tables the workloads pass.  A flipped sine, or i in place of
    2i in the exponent (th(7,3) = 7 * 10000^(-3/8) = 0.22 rad), fails."""
    from gated_delta_rule_47_gb300.inputs import rope_tables
    D, N = 16, 8
    q, k, v, P = _rope_probe(D, N)
    tabs = [(None, None), tuple(t.double().numpy() for t in rope_tables(N, D // 2))]
    for c, s in tabs:
        for fn in (oracle.cam_prep_fwd, mirror.cam_prep_fwd):
            _, _, vo, _, _ = fn(q, k, v, P, P, rope_cos=c, rope_sin=s, rope_base=10000.0)
            for n in (1, 7):
                for i in (0, 3):
                    y0, y1 = _hand_rotated_pair(n, i)
                    got = vo[0, 0, n, D // 2 + 2 * i: D // 2 + 2 * i + 2]
                    tol = 1e-12 if c is None else 1e-6  # the tables are fp32
                    assert abs(got[0] - y0) < tol and abs(got[1] - y1) < tol, (n, i, got, (y0, y1))
            # position 0 turns nothing
            assert np.allclose(vo[0, 0, 0, D // 2:], v[0, 0, 0, D // 2:], atol=1e-12)


def test_rope_pin_catches_planted_mistakes():
    """The pin above is sensitive: a sine of the wrong sign, or a frequency
    schedule in i instead of 2i, moves the hand-checked pairs far outside its
    tolerance."""
    n, i = 7, 3
    a, b = 0.6, -0.8
    y0, _ = _hand_rotated_pair(n, i)
    th_bad = n * 10000.0 ** (-i / 8.0)
    assert abs((a * np.cos(th_bad) - b * np.sin(th_bad)) - y0) > 1e-2
    th = n * 1e-3
    assert abs((a * np.cos(th) + b * np.sin(th)) - y0) > 1e-2
