"""fp64 CPU oracle for the GDN / DeltaProduct forward and backward and the camera branch.

TEST INFRASTRUCTURE ONLY.  The product package never imports this module;
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` do.  It shares no code with the CUDA path.

Two independent restatements of the same definitions live here:

* ``gdn_fwd`` / ``deltaproduct_fwd`` / ``cam_scan_fwd`` / ``cam_prep_fwd`` call the plain C
  implementation in ``gdn_oracle.c`` (compiled on first use with gcc and
  OpenMP, parallel over heads or tokens).
* ``mirror`` holds a pure numpy restatement, token by token, used on small
  cases to cross-check the C code.

The definitions (gated_deltaproduct test.py, state-scan and output kernels;
fused_cam_gdn.py, ``_cam_scan_kernel`` and ``_torch_cam_prep_reference``):

    S_t = exp(g_t) (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
    o_t = scale * S_t^T q_t

DeltaProduct applies the decay once per token and then r such corrections.
The ``*_bwd`` functions are the adjoints of those token loops, written out in
reverse token order (pinned by finite differences of the forward functions).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

from . import mirror  # noqa: F401  (re-exported)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)


def build(force: bool = False) -> str:
    """Compile ``gdn_oracle.c`` into ``_build/liboracle.so`` (gcc, -O2, OpenMP)."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i, d = ctypes.c_int, ctypes.c_double
            lib.oracle_gdn_fwd.argtypes = [_dp] * 8 + [i] * 5 + [d, i]
            lib.oracle_gdn_fwd.restype = i
            lib.oracle_deltaproduct_fwd.argtypes = [_dp] * 8 + [i] * 6 + [d, i]
            lib.oracle_deltaproduct_fwd.restype = i
            lib.oracle_masked_deltaproduct_fwd.argtypes = [_dp] * 9 + [i] * 6 + [d, i]
            lib.oracle_masked_deltaproduct_fwd.restype = i
            lib.oracle_cam_scan_fwd.argtypes = [_dp] * 8 + [i] * 6 + [d, i, i]
            lib.oracle_cam_scan_fwd.restype = i
            lib.oracle_cam_prep_fwd.argtypes = [_dp] * 9 + [d] + [_dp] * 5 + [i] * 4 + [d, d]
            lib.oracle_cam_prep_fwd.restype = i
            lib.oracle_cam_prep_bwd.argtypes = [_dp] * 8 + [d] + [_dp] * 8 + [i] * 4 + [d, d]
            lib.oracle_cam_prep_bwd.restype = i
            lib.oracle_cam_scan_bwd.argtypes = [_dp] * 14 + [i] * 6 + [d, i]
            lib.oracle_cam_scan_bwd.restype = i
            lib.oracle_deltaproduct_bwd.argtypes = [_dp] * 14 + [i] * 6 + [d, i]
            lib.oracle_deltaproduct_bwd.restype = i
            lib.oracle_masked_deltaproduct_bwd.argtypes = [_dp] * 15 + [i] * 6 + [d, i]
            lib.oracle_masked_deltaproduct_bwd.restype = i
            lib.oracle_max_threads.restype = i
            lib.oracle_set_threads.argtypes = [i]
            _lib = lib
    return _lib


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def _f64(x):
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().cpu().double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_dp)


def gdn_fwd(q, k, v, beta, g, initial_state=None, scale=1.0, l2norm=False,
            return_final_state=True):
    """Token-by-token fp64 GDN forward.

    q, k: [B,H,T,Dk]; v: [B,H,T,Dv]; beta, g: [B,H,T]; initial_state: [B,H,Dk,Dv].
    Returns (o [B,H,T,Dv], final_state [B,H,Dk,Dv] or None).
    """
    q, k, v, beta, g = map(_f64, (q, k, v, beta, g))
    s0 = _f64(initial_state)
    B, H, T, Dk = q.shape
    Dv = v.shape[-1]
    assert k.shape == (B, H, T, Dk) and v.shape == (B, H, T, Dv)
    assert beta.shape == (B, H, T) and g.shape == (B, H, T)
    if s0 is not None:
        assert s0.shape == (B, H, Dk, Dv)
    o = np.empty((B, H, T, Dv), np.float64)
    sf = np.empty((B, H, Dk, Dv), np.float64) if return_final_state else None
    rc = _load().oracle_gdn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(s0),
                                _ptr(o), _ptr(sf), B, H, T, Dk, Dv, float(scale), int(bool(l2norm)))
    if rc != 0:
        raise MemoryError("oracle_gdn_fwd failed")
    return o, sf


def deltaproduct_fwd(q, k, v, beta, g, initial_state=None, scale=1.0, l2norm=False,
                     return_final_state=True):
    """fp64 DeltaProduct forward: decay once per token, then r corrections.

    q: [B,H,T,Dk]; k: [B,H,T,r,Dk]; v: [B,H,T,r,Dv]; beta: [B,H,T,r]; g: [B,H,T].
    """
    q, k, v, beta, g = map(_f64, (q, k, v, beta, g))
    s0 = _f64(initial_state)
    B, H, T, r, Dk = k.shape
    Dv = v.shape[-1]
    assert q.shape == (B, H, T, Dk) and v.shape == (B, H, T, r, Dv)
    assert beta.shape == (B, H, T, r) and g.shape == (B, H, T)
    o = np.empty((B, H, T, Dv), np.float64)
    sf = np.empty((B, H, Dk, Dv), np.float64) if return_final_state else None
    rc = _load().oracle_deltaproduct_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g),
                                         _ptr(s0), _ptr(o), _ptr(sf), B, H, T, r, Dk, Dv,
                                         float(scale), int(bool(l2norm)))
    if rc != 0:
        raise MemoryError("oracle_deltaproduct_fwd failed")
    return o, sf


def masked_deltaproduct_fwd(q, k, v, beta, g, mask, initial_state=None, scale=1.0, l2norm=False,
                            return_final_state=True):
    """fp64 block-masked DeltaProduct (gated_deltaproduct test.py, the mask_ij
    variant): the key dim is cut into r = mask.shape[0] slices; per token one
    decay, then every sub-row i predicts with k_t masked slice-wise by
    mask[i][:] and corrects the slice-i rows of the state; one value and beta
    per token; o_t = scale S_t^T q_t.

    q, k: [B,H,T,Dk]; v: [B,H,T,Dv]; beta, g: [B,H,T]; mask: [r,r].
    """
    q, k, v, beta, g, mask = map(_f64, (q, k, v, beta, g, mask))
    s0 = _f64(initial_state)
    B, H, T, Dk = q.shape
    Dv = v.shape[-1]
    r = mask.shape[0]
    assert mask.shape == (r, r) and Dk % r == 0
    assert k.shape == (B, H, T, Dk) and v.shape == (B, H, T, Dv)
    assert beta.shape == (B, H, T) and g.shape == (B, H, T)
    o = np.empty((B, H, T, Dv), np.float64)
    sf = np.empty((B, H, Dk, Dv), np.float64) if return_final_state else None
    rc = _load().oracle_masked_deltaproduct_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(mask),
                                                _ptr(s0), _ptr(o), _ptr(sf), B, H, T, r, Dk, Dv, float(scale),
                                                int(bool(l2norm)))
    if rc != 0:
        raise MemoryError("oracle_masked_deltaproduct_fwd failed")
    return o, sf


def cam_scan_fwd(q, k, v, beta, decay, initial_state=None, scale=1.0, reverse=False, l2norm=False,
                 return_final_state=True):
    """fp64 frame-level camera scan (fused_cam_gdn.py, ``_cam_scan_kernel``).

    q, k: [B,H,N,Dk]; v: [B,H,N,Dv]; beta: [B,H,N]; decay: [B,H,F] factors,
    N = F * S.  Per frame: S <- d_f S, then S += K^T diag(beta)(V - K S) with
    every token predicting from the same decayed state, and o = scale S^T q
    after the frame's update.  reverse=True is the anti-causal mode (frames
    last to first, each reading only the frames after it); it takes no state.
    Returns (o [B,H,N,Dv], final_state [B,H,Dk,Dv] or None).
    """
    q, k, v, beta, decay = map(_f64, (q, k, v, beta, decay))
    s0 = _f64(initial_state)
    B, H, N, Dk = q.shape
    Dv = v.shape[-1]
    F = decay.shape[-1]
    assert decay.shape == (B, H, F) and F > 0 and N % F == 0
    assert k.shape == (B, H, N, Dk) and v.shape == (B, H, N, Dv) and beta.shape == (B, H, N)
    if reverse and (s0 is not None or return_final_state):
        if s0 is not None:
            raise ValueError("the reverse mode takes no initial state")
        return_final_state = False
    o = np.empty((B, H, N, Dv), np.float64)
    sf = np.empty((B, H, Dk, Dv), np.float64) if return_final_state else None
    rc = _load().oracle_cam_scan_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(decay), _ptr(s0),
                                     _ptr(o), _ptr(sf), B, H, F, N // F, Dk, Dv, float(scale),
                                     int(bool(reverse)), int(bool(l2norm)))
    if rc != 0:
        raise MemoryError("oracle_cam_scan_fwd failed")
    return o, sf


def cam_scan_bwd(q, k, v, beta, decay, do, initial_state=None, dfinal_state=None, scale=1.0, l2norm=False):
    """fp64 backward of ``cam_scan_fwd`` (forward direction): gradients
    (dq, dk, dv, dbeta, ddecay, dinitial_state) given do [B,H,N,Dv] and the
    gradient of the final state (None = zero)."""
    q, k, v, beta, decay, do = map(_f64, (q, k, v, beta, decay, do))
    s0, dsf = _f64(initial_state), _f64(dfinal_state)
    B, H, N, Dk = q.shape
    Dv = v.shape[-1]
    F = decay.shape[-1]
    outs = [np.empty((B, H, N, Dk)), np.empty((B, H, N, Dk)), np.empty((B, H, N, Dv)), np.empty((B, H, N)),
            np.empty((B, H, F)), np.empty((B, H, Dk, Dv))]
    rc = _load().oracle_cam_scan_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(decay), _ptr(s0), _ptr(do),
                                     _ptr(dsf), *[_ptr(x) for x in outs], B, H, F, N // F, Dk, Dv, float(scale),
                                     int(bool(l2norm)))
    if rc != 0:
        raise MemoryError("oracle_cam_scan_bwd failed")
    return tuple(outs)


def deltaproduct_bwd(q, k, v, beta, g, do, initial_state=None, dfinal_state=None, scale=1.0, l2norm=False):
    """fp64 backward of ``deltaproduct_fwd``: gradients (dq, dk, dv, dbeta, dg,
    dinitial_state) given do [B,H,T,Dv] and the gradient of the final state
    (None = zero).  k, v, beta carry the sub-step axis: [B,H,T,r,*]."""
    q, k, v, beta, g, do = map(_f64, (q, k, v, beta, g, do))
    s0, dsf = _f64(initial_state), _f64(dfinal_state)
    B, H, T, Dk = q.shape
    r, Dv = k.shape[3], v.shape[-1]
    outs = [np.empty((B, H, T, Dk)), np.empty((B, H, T, r, Dk)), np.empty((B, H, T, r, Dv)),
            np.empty((B, H, T, r)), np.empty((B, H, T)), np.empty((B, H, Dk, Dv))]
    rc = _load().oracle_deltaproduct_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(s0), _ptr(do),
                                         _ptr(dsf), *[_ptr(x) for x in outs], B, H, T, r, Dk, Dv, float(scale),
                                         int(bool(l2norm)))
    if rc != 0:
        raise MemoryError("oracle_deltaproduct_bwd failed")
    return tuple(outs)


def gdn_bwd(q, k, v, beta, g, do, initial_state=None, dfinal_state=None, scale=1.0, l2norm=False):
    """fp64 backward of ``gdn_fwd``: (dq, dk, dv, dbeta, dg, dinitial_state)."""
    dq, dk, dv, db, dg, ds0 = deltaproduct_bwd(q, _f64(k)[:, :, :, None], _f64(v)[:, :, :, None],
                                               _f64(beta)[:, :, :, None], g, do, initial_state,
                                               dfinal_state, scale, l2norm)
    return dq, dk[:, :, :, 0], dv[:, :, :, 0], db[:, :, :, 0], dg, ds0


def masked_deltaproduct_bwd(q, k, v, beta, g, mask, do, initial_state=None, dfinal_state=None, scale=1.0,
                            l2norm=False):
    """fp64 backward of ``masked_deltaproduct_fwd``: (dq, dk, dv, dbeta, dg,
    dinitial_state) given do and the gradient of the final state (None = 0)."""
    q, k, v, beta, g, mask, do = map(_f64, (q, k, v, beta, g, mask, do))
    s0, dsf = _f64(initial_state), _f64(dfinal_state)
    B, H, T, Dk = q.shape
    Dv = v.shape[-1]
    r = mask.shape[0]
    outs = [np.empty((B, H, T, Dk)), np.empty((B, H, T, Dk)), np.empty((B, H, T, Dv)), np.empty((B, H, T)),
            np.empty((B, H, T)), np.empty((B, H, Dk, Dv))]
    rc = _load().oracle_masked_deltaproduct_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(mask),
                                                _ptr(s0), _ptr(do), _ptr(dsf), *[_ptr(x) for x in outs], B, H, T,
                                                r, Dk, Dv, float(scale), int(bool(l2norm)))
    if rc != 0:
        raise MemoryError("oracle_masked_deltaproduct_bwd failed")
    return tuple(outs)


def cam_prep_fwd(q_raw, k_raw, v_raw, proj_q, proj_kv, q_norm_w=None, k_norm_w=None,
                 rope_cos=None, rope_sin=None, rope_base=10000.0, k_scale=0.5, eps=1e-6):
    """fp64 camera-branch prep.  Raw inputs [B,N,H,D]; outputs q,k,v [B,H,N,D]
    and k_pre_sq, k_post_sq [B,H,N]."""
    q_raw, k_raw, v_raw, proj_q, proj_kv = map(_f64, (q_raw, k_raw, v_raw, proj_q, proj_kv))
    q_norm_w, k_norm_w, rope_cos, rope_sin = map(_f64, (q_norm_w, k_norm_w, rope_cos, rope_sin))
    B, N, H, D = q_raw.shape
    assert (rope_cos is None) == (rope_sin is None)
    outs = [np.empty((B, H, N, D), np.float64) for _ in range(3)]
    pre = np.empty((B, H, N), np.float64)
    post = np.empty((B, H, N), np.float64)
    rc = _load().oracle_cam_prep_fwd(_ptr(q_raw), _ptr(k_raw), _ptr(v_raw), _ptr(q_norm_w),
                                     _ptr(k_norm_w), _ptr(proj_q), _ptr(proj_kv),
                                     _ptr(rope_cos), _ptr(rope_sin), float(rope_base),
                                     _ptr(outs[0]), _ptr(outs[1]), _ptr(outs[2]), _ptr(pre),
                                     _ptr(post), B, N, H, D, float(k_scale), float(eps))
    if rc == -2:
        raise ValueError("cam prep needs D even and D/2 divisible by 4")
    if rc != 0:
        raise MemoryError("oracle_cam_prep_fwd failed")
    return outs[0], outs[1], outs[2], pre, post


def cam_prep_bwd(q_raw, k_raw, v_raw, proj_q, proj_kv, dq_out, dk_out, dv_out, dk_pre_sq=None,
                 dk_post_sq=None, q_norm_w=None, k_norm_w=None, rope_cos=None, rope_sin=None, rope_base=10000.0,
                 k_scale=0.5, eps=1e-6):
    """fp64 backward of ``cam_prep_fwd``: the gradients of the raw q, k, v
    [B,N,H,D] given those of q_out, k_out, v_out [B,H,N,D] and of k_pre_sq,
    k_post_sq [B,H,N] (None = zero)."""
    q_raw, k_raw, proj_q, proj_kv, dq_out, dk_out, dv_out = map(
        _f64, (q_raw, k_raw, proj_q, proj_kv, dq_out, dk_out, dv_out))
    dpre, dpost, q_norm_w, k_norm_w, rope_cos, rope_sin = map(
        _f64, (dk_pre_sq, dk_post_sq, q_norm_w, k_norm_w, rope_cos, rope_sin))
    B, N, H, D = q_raw.shape
    assert D <= 512
    outs = [np.empty((B, N, H, D), np.float64) for _ in range(3)]
    rc = _load().oracle_cam_prep_bwd(_ptr(q_raw), _ptr(k_raw), _ptr(q_norm_w), _ptr(k_norm_w), _ptr(proj_q),
                                     _ptr(proj_kv), _ptr(rope_cos), _ptr(rope_sin), float(rope_base), _ptr(dq_out),
                                     _ptr(dk_out), _ptr(dv_out), _ptr(dpre), _ptr(dpost), _ptr(outs[0]),
                                     _ptr(outs[1]), _ptr(outs[2]), B, N, H, D, float(k_scale), float(eps))
    if rc != 0:
        raise MemoryError("oracle_cam_prep_bwd failed")
    return tuple(outs)


def inflation_sq(k_pre_sq, k_post_sq):
    """||k_post||^2 / ||k_pre||^2 with both floored at 1e-12 (fused_cam_gdn.py,
    ``cam_prep_func`` return value)."""
    return np.maximum(k_post_sq, 1e-12) / np.maximum(k_pre_sq, 1e-12)
