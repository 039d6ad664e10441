"""Pins for the fp64 frame-level camera scan (fused_cam_gdn.py,
``_cam_scan_kernel``, ``_torch_cam_scan_single_chunk``,
``_torch_cam_scan_reference`` and ``_flip_and_shift``), each against something
other than the oracle itself: the pinned token-level GDN oracle, closed forms,
the dense-matrix form of the page's single-chunk torch scan, the flip-and-shift
construction of the reverse mode, and planted mistakes."""
import numpy as np
import pytest

import oracle
from oracle import mirror


def frames_inputs(B=1, H=2, F=4, S=5, Dk=8, Dv=6, seed=0, unit=True):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((B, H, F * S, Dk))
    k = rng.standard_normal((B, H, F * S, Dk))
    if unit:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, H, F * S, Dv))
    beta = rng.random((B, H, F * S)) / S
    decay = np.exp(-rng.random((B, H, F)) / 4)
    s0 = rng.standard_normal((B, H, Dk, Dv))
    return q, k, v, beta, decay, s0


def dense_single_chunk(q, k, v, beta, decay, s0=None):
    """The page's ``_torch_cam_scan_single_chunk`` as explicit matrices, in its
    own (transposed, Dv x Dk) state convention: W_f = d_f (I - sum_s b_s k_s
    k_s^T), U_f = sum_s b_s v_s k_s^T, state <- state W_f + U_f, and each
    frame's outputs are state q_s.  Returns o and the final state in the
    library's Dk x Dv convention."""
    B, H, N, Dk = q.shape
    Dv = v.shape[-1]
    F = decay.shape[-1]
    S = N // F
    o = np.zeros((B, H, N, Dv))
    fin = np.zeros((B, H, Dk, Dv))
    for b in range(B):
        for h in range(H):
            st = np.zeros((Dv, Dk)) if s0 is None else s0[b, h].T.copy()
            for f in range(F):
                sl = slice(f * S, (f + 1) * S)
                K, V, bt = k[b, h, sl], v[b, h, sl], beta[b, h, sl]
                W = decay[b, h, f] * (np.eye(Dk) - (K * bt[:, None]).T @ K)
                U = (V * bt[:, None]).T @ K
                st = st @ W + U
                o[b, h, sl] = (st @ q[b, h, sl].T).T
            fin[b, h] = st.T
    return o, fin


def flip_and_shift(x, axis, pad):
    """Flip along the frame axis and shift right by one, filling with pad
    (fused_cam_gdn.py, ``_flip_and_shift``)."""
    xf = np.flip(x, axis=axis)
    xs = np.take(xf, range(x.shape[axis] - 1), axis=axis)
    shape = list(x.shape)
    shape[axis] = 1
    return np.concatenate([np.full(shape, pad), xs], axis=axis)


def test_c_matches_numpy_mirror_both_directions():
    q, k, v, beta, decay, s0 = frames_inputs(B=2, H=2, F=5, S=3, Dk=8, Dv=8, seed=1)
    a = oracle.cam_scan_fwd(q, k, v, beta, decay, s0, scale=0.7)
    b = mirror.cam_scan_fwd(q, k, v, beta, decay, s0, scale=0.7)
    assert np.max(np.abs(a[0] - b[0])) < 1e-12 and np.max(np.abs(a[1] - b[1])) < 1e-12
    a = oracle.cam_scan_fwd(q, k, v, beta, decay, reverse=True)
    b = mirror.cam_scan_fwd(q, k, v, beta, decay, reverse=True)
    assert np.max(np.abs(a[0] - b[0])) < 1e-12


def test_matches_dense_single_chunk_form():
    q, k, v, beta, decay, s0 = frames_inputs(F=6, S=7, Dk=8, Dv=5, seed=2)
    o, sf = oracle.cam_scan_fwd(q, k, v, beta, decay, s0)
    do, dsf = dense_single_chunk(q, k, v, beta, decay, s0)
    assert np.max(np.abs(o - do)) < 1e-12 and np.max(np.abs(sf - dsf)) < 1e-12


def test_frames_of_one_token_are_the_token_level_gdn():
    """S = 1: one decay and one correction per token, which is the GDN
    recurrence with g = log(decay)."""
    q, k, v, beta, decay, s0 = frames_inputs(F=12, S=1, Dk=8, Dv=6, seed=3)
    o, sf = oracle.cam_scan_fwd(q, k, v, beta, decay, s0, scale=1.3)
    go, gsf = oracle.gdn_fwd(q, k, v, beta, np.log(decay), s0, scale=1.3)
    assert np.max(np.abs(o - go)) < 1e-12 and np.max(np.abs(sf - gsf)) < 1e-12


def test_first_frame_from_zero_state_is_bidirectional_attention():
    """From the zero state nothing is predicted, so after frame 0 the state is
    K^T diag(beta) V and every token of the frame, the earlier ones too, reads
    o_s = sum_{s'} (q_s . k_s') beta_s' v_s'."""
    q, k, v, beta, decay, _ = frames_inputs(F=3, S=6, Dk=8, Dv=4, seed=4)
    o, _ = oracle.cam_scan_fwd(q, k, v, beta, decay)
    sl = slice(0, 6)
    want = np.einsum("bhsd,bhtd,bht,bhtv->bhsv", q[:, :, sl], k[:, :, sl], beta[:, :, sl], v[:, :, sl])
    assert np.max(np.abs(o[:, :, sl] - want)) < 1e-12


def test_beta_zero_is_pure_decay():
    q, k, v, beta, decay, s0 = frames_inputs(F=5, S=4, seed=5)
    o, sf = oracle.cam_scan_fwd(q, k, v, np.zeros_like(beta), decay, s0)
    cum = np.cumprod(decay, axis=-1)  # [B,H,F]
    want = np.repeat(cum, 4, axis=-1)[..., None] * np.einsum("bhkv,bhtk->bhtv", s0, q)
    assert np.max(np.abs(o - want)) < 1e-12
    assert np.max(np.abs(sf - cum[..., -1][..., None, None] * s0)) < 1e-12


def test_orthonormal_keys_make_the_joint_update_sequential():
    """Within a frame of mutually orthogonal unit keys the S corrections
    commute, so the joint update equals S token-level corrections with the
    frame's decay on the first token; with correlated keys it does not (which
    a token-by-token implementation would miss)."""
    rng = np.random.default_rng(6)
    Dk, Dv, S, F = 8, 5, 4, 3
    qm, _ = np.linalg.qr(rng.standard_normal((Dk, Dk)))
    k = np.stack([qm[(f * S) % 8:(f * S) % 8 + S] for f in range(F)]).reshape(1, 1, F * S, Dk)
    q = rng.standard_normal((1, 1, F * S, Dk))
    v = rng.standard_normal((1, 1, F * S, Dv))
    beta = rng.random((1, 1, F * S))
    decay = np.exp(-rng.random((1, 1, F)))
    s0 = rng.standard_normal((1, 1, Dk, Dv))
    g = np.zeros((1, 1, F * S))
    g[..., ::S] = np.log(decay)
    _, sf = oracle.cam_scan_fwd(q, k, v, beta, decay, s0)
    _, gsf = oracle.gdn_fwd(q, k, v, beta, g, s0)
    assert np.max(np.abs(sf - gsf)) < 1e-12
    k2 = k + 0.3 * rng.standard_normal(k.shape)
    _, sf2 = oracle.cam_scan_fwd(q, k2, v, beta, decay, s0)
    _, gsf2 = oracle.gdn_fwd(q, k2, v, beta, g, s0)
    assert np.max(np.abs(sf2 - gsf2)) > 1e-3


def test_reverse_is_flip_and_shift_of_the_forward():
    """fused_cam_gdn.py, ``_torch_cam_scan_reference``: the reverse mode is the
    forward scan over frames taken last to first, with k, v, beta shifted by
    one frame (zero-filled) and the decay shifted with a factor-1 fill, and
    the output flipped back."""
    B, H, F, S, Dk, Dv = 1, 2, 5, 3, 8, 6
    q, k, v, beta, decay, _ = frames_inputs(B, H, F, S, Dk, Dv, seed=7)
    fr = lambda x: x.reshape(B, H, F, S, *x.shape[3:])
    un = lambda x: x.reshape(B, H, F * S, *x.shape[4:])
    qb = un(np.flip(fr(q), axis=2))
    kb = un(flip_and_shift(fr(k), 2, 0.0))
    vb = un(flip_and_shift(fr(v), 2, 0.0))
    bb = un(flip_and_shift(fr(beta), 2, 0.0))
    db = flip_and_shift(decay, 2, 1.0)
    ob, _ = oracle.cam_scan_fwd(qb, kb, vb, bb, db)
    want = un(np.flip(fr(ob), axis=2))
    got, _ = oracle.cam_scan_fwd(q, k, v, beta, decay, reverse=True)
    assert np.max(np.abs(got - want)) < 1e-12
    assert np.max(np.abs(got[:, :, -S:])) == 0.0  # the last frame sees nothing after it


def test_split_and_resume():
    """Frames [0, f0) then [f0, F) from the first part's final state give the
    whole run bit for bit (fused_cam_gdn.py, ``cam_scan_func`` state passing:
    the resumed scan applies frame f0's decay to the loaded state)."""
    q, k, v, beta, decay, s0 = frames_inputs(F=6, S=4, seed=8)
    o, sf = oracle.cam_scan_fwd(q, k, v, beta, decay, s0)
    f0, S = 2, 4
    a = oracle.cam_scan_fwd(q[:, :, :f0 * S], k[:, :, :f0 * S], v[:, :, :f0 * S], beta[:, :, :f0 * S],
                            decay[..., :f0], s0)
    b = oracle.cam_scan_fwd(q[:, :, f0 * S:], k[:, :, f0 * S:], v[:, :, f0 * S:], beta[:, :, f0 * S:],
                            decay[..., f0:], a[1])
    assert np.array_equal(np.concatenate([a[0], b[0]], axis=2), o)
    assert np.array_equal(b[1], sf)


def test_l2norm_flag_equals_normalised_inputs():
    q, k, v, beta, decay, s0 = frames_inputs(F=3, S=4, seed=9, unit=False)
    a = oracle.cam_scan_fwd(q, k, v, beta, decay, s0, l2norm=True)
    qn = q / np.linalg.norm(q, axis=-1, keepdims=True)
    kn = k / np.linalg.norm(k, axis=-1, keepdims=True)
    b = oracle.cam_scan_fwd(qn, kn, v, beta, decay, s0)
    assert np.max(np.abs(a[0] - b[0])) < 1e-12


def test_reverse_mode_takes_no_state():
    q, k, v, beta, decay, s0 = frames_inputs(F=2, S=2, seed=10)
    with pytest.raises(ValueError):
        oracle.cam_scan_fwd(q, k, v, beta, decay, s0, reverse=True)


def test_pins_catch_planted_mistakes():
    """Three plausible slips, planted in a copy of the frame loop, each fail
    the dense single-chunk pin: reading the outputs before the update,
    decaying after it, and updating token by token instead of jointly."""
    q, k, v, beta, decay, s0 = frames_inputs(F=4, S=5, seed=11)
    do, _ = dense_single_chunk(q, k, v, beta, decay, s0)

    def run(kind):
        B, H, N, Dk = q.shape
        F = decay.shape[-1]
        S = N // F
        o = np.zeros((B, H, N, v.shape[-1]))
        for b in range(B):
            for h in range(H):
                St = s0[b, h].copy()
                for f in range(F):
                    sl = slice(f * S, (f + 1) * S)
                    K, V, bt = k[b, h, sl], v[b, h, sl], beta[b, h, sl]
                    if kind == "read_before":
                        o[b, h, sl] = q[b, h, sl] @ (decay[b, h, f] * St)
                    if kind != "decay_after":
                        St = decay[b, h, f] * St
                    if kind == "sequential":
                        for s in range(S):
                            St = St + bt[s] * np.outer(K[s], V[s] - K[s] @ St)
                    else:
                        St = St + K.T @ (bt[:, None] * (V - K @ St))
                    if kind == "decay_after":
                        St = decay[b, h, f] * St
                    if kind != "read_before":
                        o[b, h, sl] = q[b, h, sl] @ St
        return o

    for kind in ("read_before", "decay_after", "sequential"):
        assert np.max(np.abs(run(kind) - do)) > 1e-3, kind
