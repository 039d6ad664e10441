"""Thin ctypes binding of libgdn.so (argument marshalling only).

Every function here checks that its tensors are CUDA, contiguous and of the
expected dtype and shape, allocates the outputs with torch, and calls the C
entry point of the same name with raw device pointers and the current CUDA
stream.  All computation happens in the library's kernels; there is no
fallback: if ``libgdn.so`` is missing or fails to load, ``load()`` raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libgdn.so")

GDN_F32, GDN_BF16 = 0, 1
GDN_QK_L2NORM = 1
GDN_PATH_SIMT = 2
GDN_CAM_REVERSE = 4
STATUS = {0: "GDN_OK", 1: "GDN_ERR_INVALID_ARG", 2: "GDN_ERR_UNSUPPORTED", 3: "GDN_ERR_MISALIGNED",
          4: "GDN_ERR_WORKSPACE", 5: "GDN_ERR_CUDA", 6: "GDN_ERR_TIMEOUT"}

EXPORTS = ("gdn_status_string", "gdn_version", "gdn_chunk_fwd_workspace_bytes", "gdn_chunk_fwd",
           "deltaproduct_chunk_fwd", "cam_prep_fwd", "gdn_get_device_error", "gdn_set_wait_limit", "gdn_launch_count",
           "gdn_set_cluster_shape", "gdn_chunk_fwd_noalloc", "cam_scan_fwd_workspace_bytes", "cam_scan_fwd",
           "masked_deltaproduct_chunk_fwd", "masked_deltaproduct_chunk_fwd_workspace_bytes",
           "cam_prep_scan_fwd_workspace_bytes", "cam_prep_scan_fwd",
           "cam_prep_bwd", "cam_scan_bwd_workspace_bytes", "cam_scan_bwd", "gdn_chunk_bwd_workspace_bytes",
           "gdn_chunk_bwd", "deltaproduct_chunk_bwd", "masked_deltaproduct_chunk_bwd_workspace_bytes",
           "masked_deltaproduct_chunk_bwd")

_lock = threading.Lock()
_lib = None


class GdnError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} failed: {STATUS.get(status, status)}")


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libgdn.so (built by ``gated_delta_rule_47_gb300.build``) and declare
    the signatures of its entry points."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"libgdn.so not found at {p}; build it with "
                               "`python -m gated_delta_rule_47_gb300.build`")
        lib = ctypes.CDLL(p)
        vp, i, u, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint, ctypes.c_float, ctypes.c_size_t
        lib.gdn_status_string.argtypes = [i]
        lib.gdn_status_string.restype = ctypes.c_char_p
        lib.gdn_version.restype = i
        lib.gdn_chunk_fwd_workspace_bytes.argtypes = [i] * 8
        lib.gdn_chunk_fwd_workspace_bytes.restype = sz
        lib.gdn_chunk_fwd.argtypes = [vp] * 8 + [i] * 6 + [f, u, i, vp, sz, vp]
        lib.gdn_chunk_fwd.restype = i
        lib.gdn_chunk_fwd_noalloc.argtypes = [vp] * 8 + [i] * 6 + [f, u, i, vp]
        lib.gdn_chunk_fwd_noalloc.restype = i
        lib.deltaproduct_chunk_fwd.argtypes = [vp] * 8 + [i] * 7 + [f, u, i, vp, sz, vp]
        lib.deltaproduct_chunk_fwd.restype = i
        lib.masked_deltaproduct_chunk_fwd.argtypes = [vp] * 9 + [i] * 7 + [f, u, i, vp, sz, vp]
        lib.masked_deltaproduct_chunk_fwd_workspace_bytes.argtypes = [i] * 7
        lib.masked_deltaproduct_chunk_fwd_workspace_bytes.restype = sz
        lib.masked_deltaproduct_chunk_fwd.restype = i
        lib.cam_prep_scan_fwd_workspace_bytes.argtypes = [i] * 6
        lib.cam_prep_scan_fwd_workspace_bytes.restype = sz
        lib.cam_prep_scan_fwd.argtypes = [vp] * 7 + [f] + [vp] * 5 + [i] * 5 + [f, f, f, u, i, vp, sz, vp]
        lib.cam_prep_scan_fwd.restype = i
        lib.cam_scan_bwd_workspace_bytes.argtypes = [i] * 7
        lib.cam_scan_bwd_workspace_bytes.restype = sz
        lib.cam_scan_bwd.argtypes = [vp] * 14 + [i] * 6 + [f, u, i, vp, sz, vp]
        lib.cam_scan_bwd.restype = i
        lib.gdn_chunk_bwd_workspace_bytes.argtypes = [i] * 7
        lib.gdn_chunk_bwd_workspace_bytes.restype = sz
        lib.gdn_chunk_bwd.argtypes = [vp] * 14 + [i] * 5 + [f, u, i, vp, sz, vp]
        lib.gdn_chunk_bwd.restype = i
        lib.deltaproduct_chunk_bwd.argtypes = [vp] * 14 + [i] * 6 + [f, u, i, vp, sz, vp]
        lib.deltaproduct_chunk_bwd.restype = i
        lib.masked_deltaproduct_chunk_bwd_workspace_bytes.argtypes = [i] * 7
        lib.masked_deltaproduct_chunk_bwd_workspace_bytes.restype = sz
        lib.masked_deltaproduct_chunk_bwd.argtypes = [vp] * 15 + [i] * 6 + [f, u, i, vp, sz, vp]
        lib.masked_deltaproduct_chunk_bwd.restype = i
        lib.cam_prep_bwd.argtypes = [vp] * 8 + [f] + [vp] * 8 + [i] * 4 + [f, f, i, vp]
        lib.cam_prep_bwd.restype = i
        lib.cam_scan_fwd_workspace_bytes.argtypes = [i] * 7
        lib.cam_scan_fwd_workspace_bytes.restype = sz
        lib.cam_scan_fwd.argtypes = [vp] * 8 + [i] * 6 + [f, u, i, vp, sz, vp]
        lib.cam_scan_fwd.restype = i
        lib.cam_prep_fwd.argtypes = [vp] * 9 + [f] + [vp] * 5 + [i] * 4 + [f, f, i, vp]
        lib.cam_prep_fwd.restype = i
        lib.gdn_get_device_error.argtypes = [vp]
        lib.gdn_get_device_error.restype = i
        lib.gdn_set_wait_limit.argtypes = [ctypes.c_ulonglong]
        lib.gdn_set_wait_limit.restype = i
        lib.gdn_set_cluster_shape.argtypes = [i, i]
        lib.gdn_set_cluster_shape.restype = i
        lib.gdn_launch_count.restype = ctypes.c_ulonglong
        if path is None:
            _lib = lib
        return lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dtype_code(t):
    if t.dtype == torch.bfloat16:
        return GDN_BF16
    if t.dtype == torch.float32:
        return GDN_F32
    raise TypeError(f"unsupported dtype {t.dtype}: use torch.bfloat16 or torch.float32")


def _check(t, name, shape, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def _raise(fn, st):
    if st != 0:
        raise GdnError(fn, st)


def workspace_bytes(B, H, T, Dk, Dv, chunk=64, r=1, dtype=torch.bfloat16):
    code = GDN_BF16 if dtype == torch.bfloat16 else GDN_F32
    n = load().gdn_chunk_fwd_workspace_bytes(B, H, T, r, Dk, Dv, chunk, code)
    if n == ctypes.c_size_t(-1).value:
        raise ValueError("sizes rejected by gdn_chunk_fwd_workspace_bytes")
    return int(n)


def _scan(fn_name, q, k, v, beta, g, r, initial_state, output_final_state, chunk, scale, l2norm,
          o, workspace, stream, simt=False):
    B, H, T, Dk = q.shape
    Dv = v.shape[-1]
    dt = q.dtype
    code = _dtype_code(q)
    sub = () if r is None else (r,)
    _check(q, "q", (B, H, T, Dk), dt)
    _check(k, "k", (B, H, T, *sub, Dk), dt)
    _check(v, "v", (B, H, T, *sub, Dv), dt)
    _check(beta, "beta", (B, H, T, *sub), dt)
    _check(g, "g", (B, H, T), torch.float32)
    if initial_state is not None:
        _check(initial_state, "initial_state", (B, H, Dk, Dv), torch.float32)
    if o is None:
        o = torch.empty(B, H, T, Dv, dtype=dt, device=q.device)
    _check(o, "o", (B, H, T, Dv), dt)
    sf = torch.empty(B, H, Dk, Dv, dtype=torch.float32, device=q.device) if output_final_state else None
    need = workspace_bytes(B, H, T, Dk, Dv, chunk, 1 if r is None else r, dt)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    lib = load()
    flags = (GDN_QK_L2NORM if l2norm else 0) | (GDN_PATH_SIMT if simt else 0)
    common = [_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(initial_state), _ptr(o), _ptr(sf)]
    if r is None:
        st = lib.gdn_chunk_fwd(*common, B, H, T, Dk, Dv, chunk, float(scale), flags, code,
                               _ptr(workspace), ws_bytes, _stream(stream))
    else:
        st = lib.deltaproduct_chunk_fwd(*common, B, H, T, r, Dk, Dv, chunk, float(scale), flags, code,
                                        _ptr(workspace), ws_bytes, _stream(stream))
    _raise(fn_name, st)
    return o, sf


def gdn_chunk_fwd(q, k, v, beta, g, initial_state=None, output_final_state=False, chunk=64,
                  scale=1.0, l2norm=False, o=None, workspace=None, stream=None, simt=False):
    """Chunkwise GDN forward.  q,k [B,H,T,Dk]; v [B,H,T,Dv]; beta [B,H,T] (all
    bf16 or all fp32); g [B,H,T] fp32.  Returns (o, final_state or None).
    simt=True takes the CUDA-core path even where the tensor-core one applies."""
    return _scan("gdn_chunk_fwd", q, k, v, beta, g, None, initial_state, output_final_state, chunk,
                 scale, l2norm, o, workspace, stream, simt)


def gdn_chunk_fwd_noalloc(q, k, v, beta, g, initial_state=None, output_final_state=False, chunk=64,
                          scale=1.0, l2norm=False, o=None, stream=None):
    """gdn_chunk_fwd through the allocation-free entry point: the library uses
    its own fixed scratch array instead of a workspace (B*H <= 64 heads where
    the tensor-core path needs one).  Calls must not overlap on the GPU."""
    B, H, T, Dk = q.shape
    Dv = v.shape[-1]
    dt = q.dtype
    code = _dtype_code(q)
    _check(q, "q", (B, H, T, Dk), dt)
    _check(k, "k", (B, H, T, Dk), dt)
    _check(v, "v", (B, H, T, Dv), dt)
    _check(beta, "beta", (B, H, T), dt)
    _check(g, "g", (B, H, T), torch.float32)
    if initial_state is not None:
        _check(initial_state, "initial_state", (B, H, Dk, Dv), torch.float32)
    if o is None:
        o = torch.empty(B, H, T, Dv, dtype=dt, device=q.device)
    _check(o, "o", (B, H, T, Dv), dt)
    sf = torch.empty(B, H, Dk, Dv, dtype=torch.float32, device=q.device) if output_final_state else None
    flags = GDN_QK_L2NORM if l2norm else 0
    st = load().gdn_chunk_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(initial_state),
                                      _ptr(o), _ptr(sf), B, H, T, Dk, Dv, chunk, float(scale), flags, code,
                                      _stream(stream))
    _raise("gdn_chunk_fwd_noalloc", st)
    return o, sf


def deltaproduct_chunk_fwd(q, k, v, beta, g, initial_state=None, output_final_state=False, chunk=64,
                           scale=1.0, l2norm=False, o=None, workspace=None, stream=None, simt=False):
    """DeltaProduct forward.  q [B,H,T,Dk]; k [B,H,T,r,Dk]; v [B,H,T,r,Dv];
    beta [B,H,T,r]; g [B,H,T] fp32.  chunk counts expanded rows."""
    r = k.shape[3]
    return _scan("deltaproduct_chunk_fwd", q, k, v, beta, g, r, initial_state, output_final_state,
                 chunk, scale, l2norm, o, workspace, stream, simt)


def masked_deltaproduct_workspace_bytes(B, H, T, r, Dk, Dv, dtype=torch.bfloat16):
    code = GDN_BF16 if dtype == torch.bfloat16 else GDN_F32
    return int(load().masked_deltaproduct_chunk_fwd_workspace_bytes(B, H, T, r, Dk, Dv, code))


def masked_deltaproduct_chunk_fwd(q, k, v, beta, g, mask, initial_state=None, output_final_state=False,
                                  chunk=64, scale=1.0, l2norm=False, o=None, workspace=None, stream=None,
                                  simt=False):
    """Block-masked DeltaProduct forward.  q, k [B,H,T,Dk]; v [B,H,T,Dv]; beta
    [B,H,T] (all bf16 or all fp32); g [B,H,T] fp32; mask [r,r] fp32 (CUDA).
    chunk counts sub-rows (tokens x r).  simt keeps the state chain on the
    CUDA cores where the tensor-core chain would run."""
    B, H, T, Dk = q.shape
    Dv = v.shape[-1]
    r = mask.shape[0]
    dt = q.dtype
    code = _dtype_code(q)
    _check(q, "q", (B, H, T, Dk), dt)
    _check(k, "k", (B, H, T, Dk), dt)
    _check(v, "v", (B, H, T, Dv), dt)
    _check(beta, "beta", (B, H, T), dt)
    _check(g, "g", (B, H, T), torch.float32)
    _check(mask, "mask", (r, r), torch.float32)
    if initial_state is not None:
        _check(initial_state, "initial_state", (B, H, Dk, Dv), torch.float32)
    if o is None:
        o = torch.empty(B, H, T, Dv, dtype=dt, device=q.device)
    _check(o, "o", (B, H, T, Dv), dt)
    sf = torch.empty(B, H, Dk, Dv, dtype=torch.float32, device=q.device) if output_final_state else None
    lib = load()
    if workspace is None:
        need = lib.masked_deltaproduct_chunk_fwd_workspace_bytes(B, H, T, r, Dk, Dv, code)
        workspace = torch.empty(max(int(need), 16), dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    flags = (GDN_QK_L2NORM if l2norm else 0) | (GDN_PATH_SIMT if simt else 0)
    st = lib.masked_deltaproduct_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(mask),
                                           _ptr(initial_state), _ptr(o), _ptr(sf), B, H, T, r, Dk, Dv, chunk,
                                           float(scale), flags,
                                           code, _ptr(workspace),
                                           ws_bytes, _stream(stream))
    _raise("masked_deltaproduct_chunk_fwd", st)
    return o, sf


def cam_scan_workspace_bytes(B, H, F, S, Dk, Dv, dtype=torch.bfloat16):
    code = GDN_BF16 if dtype == torch.bfloat16 else GDN_F32
    n = load().cam_scan_fwd_workspace_bytes(B, H, F, S, Dk, Dv, code)
    if n == ctypes.c_size_t(-1).value:
        raise ValueError("sizes rejected by cam_scan_fwd_workspace_bytes")
    return int(n)


def cam_scan_fwd(q, k, v, beta, decay, initial_state=None, output_final_state=False, scale=1.0,
                 reverse=False, l2norm=False, o=None, workspace=None, stream=None, simt=False):
    """Frame-level camera scan.  q, k [B,H,N,Dk]; v [B,H,N,Dv]; beta [B,H,N]
    (all bf16 or all fp32); decay [B,H,F] fp32 factors, N = F * S.  Returns
    (o, final_state or None); reverse=True is the anti-causal mode."""
    B, H, N, Dk = q.shape
    Dv = v.shape[-1]
    F = decay.shape[-1]
    if F <= 0 or N % F != 0:
        raise ValueError(f"{N} tokens do not split into {F} frames")
    S = N // F
    dt = q.dtype
    code = _dtype_code(q)
    _check(q, "q", (B, H, N, Dk), dt)
    _check(k, "k", (B, H, N, Dk), dt)
    _check(v, "v", (B, H, N, Dv), dt)
    _check(beta, "beta", (B, H, N), dt)
    _check(decay, "decay", (B, H, F), torch.float32)
    if initial_state is not None:
        _check(initial_state, "initial_state", (B, H, Dk, Dv), torch.float32)
    if o is None:
        o = torch.empty(B, H, N, Dv, dtype=dt, device=q.device)
    _check(o, "o", (B, H, N, Dv), dt)
    sf = torch.empty(B, H, Dk, Dv, dtype=torch.float32, device=q.device) if output_final_state else None
    need = cam_scan_workspace_bytes(B, H, F, S, Dk, Dv, dt)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    flags = (GDN_QK_L2NORM if l2norm else 0) | (GDN_PATH_SIMT if simt else 0) | (GDN_CAM_REVERSE if reverse else 0)
    st = load().cam_scan_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(decay), _ptr(initial_state), _ptr(o),
                             _ptr(sf), B, H, F, S, Dk, Dv, float(scale), flags, code, _ptr(workspace), ws_bytes,
                             _stream(stream))
    _raise("cam_scan_fwd", st)
    return o, sf


def cam_prep_scan_workspace_bytes(B, N, H, D, F, dtype=torch.bfloat16):
    code = GDN_BF16 if dtype == torch.bfloat16 else GDN_F32
    n = load().cam_prep_scan_fwd_workspace_bytes(B, N, H, D, F, code)
    if n == ctypes.c_size_t(-1).value:
        raise ValueError("sizes rejected by cam_prep_scan_fwd_workspace_bytes")
    return int(n)


def cam_prep_scan_fwd(q_raw, k_raw, v_raw, proj_q, proj_kv, beta, decay, q_norm_w=None, k_norm_w=None,
                      rope_base=10000.0, initial_state=None, output_final_state=False, k_scale=0.5, eps=1e-6,
                      scale=1.0, reverse=False, l2norm=True, o=None, workspace=None, stream=None):
    """Camera prep fused into the frame scan: raw q, k, v [B,N,H,D] bf16 ->
    o [B,H,N,D] = cam_scan_fwd(cam_prep_fwd(...)).  beta [B,H,N] bf16, decay
    [B,H,F] fp32 factors; rotation angles n * rope_base^(-2i/(D/2))."""
    B, N, H, D = q_raw.shape
    F = decay.shape[-1]
    if F <= 0 or N % F != 0:
        raise ValueError(f"{N} tokens do not split into {F} frames")
    dt = q_raw.dtype
    code = _dtype_code(q_raw)
    for name, t in (("q_raw", q_raw), ("k_raw", k_raw), ("v_raw", v_raw)):
        _check(t, name, (B, N, H, D), dt)
    _check(proj_q, "proj_q", (B, N, 4, 4), torch.float32)
    _check(proj_kv, "proj_kv", (B, N, 4, 4), torch.float32)
    _check(beta, "beta", (B, H, N), dt)
    _check(decay, "decay", (B, H, F), torch.float32)
    for name, t in (("q_norm_w", q_norm_w), ("k_norm_w", k_norm_w)):
        if t is not None:
            _check(t, name, (H * D,), torch.float32)
    if initial_state is not None:
        _check(initial_state, "initial_state", (B, H, D, D), torch.float32)
    if o is None:
        o = torch.empty(B, H, N, D, dtype=dt, device=q_raw.device)
    _check(o, "o", (B, H, N, D), dt)
    sf = torch.empty(B, H, D, D, dtype=torch.float32, device=q_raw.device) if output_final_state else None
    if workspace is None:
        workspace = torch.empty(cam_prep_scan_workspace_bytes(B, N, H, D, F, dt), dtype=torch.uint8,
                                device=q_raw.device)
    ws_bytes = workspace.numel() * workspace.element_size()
    flags = (GDN_QK_L2NORM if l2norm else 0) | (GDN_CAM_REVERSE if reverse else 0)
    st = load().cam_prep_scan_fwd(_ptr(q_raw), _ptr(k_raw), _ptr(v_raw), _ptr(q_norm_w), _ptr(k_norm_w),
                                  _ptr(proj_q), _ptr(proj_kv), float(rope_base), _ptr(beta), _ptr(decay),
                                  _ptr(initial_state), _ptr(o), _ptr(sf), B, N, H, D, F, float(k_scale), float(eps),
                                  float(scale), flags, code, _ptr(workspace), ws_bytes, _stream(stream))
    _raise("cam_prep_scan_fwd", st)
    return o, sf


def cam_prep_fwd(q_raw, k_raw, v_raw, proj_q, proj_kv, q_norm_w=None, k_norm_w=None, rope_cos=None,
                 rope_sin=None, rope_base=10000.0, k_scale=0.5, eps=1e-6, with_norms=True, outs=None,
                 stream=None):
    """Fused camera prep.  Raw q,k,v [B,N,H,D] -> q,k,v [B,H,N,D] plus
    ||k||^2 before / after the projection and rotation, [B,H,N] fp32."""
    B, N, H, D = q_raw.shape
    dt = q_raw.dtype
    code = _dtype_code(q_raw)
    for name, t in (("q_raw", q_raw), ("k_raw", k_raw), ("v_raw", v_raw)):
        _check(t, name, (B, N, H, D), dt)
    _check(proj_q, "proj_q", (B, N, 4, 4), torch.float32)
    _check(proj_kv, "proj_kv", (B, N, 4, 4), torch.float32)
    for name, t in (("q_norm_w", q_norm_w), ("k_norm_w", k_norm_w)):
        if t is not None:
            _check(t, name, (H * D,), torch.float32)
    for name, t in (("rope_cos", rope_cos), ("rope_sin", rope_sin)):
        if t is not None:
            _check(t, name, (N, D // 2), torch.float32)
    dev = q_raw.device
    if outs is None:
        outs = tuple(torch.empty(B, H, N, D, dtype=dt, device=dev) for _ in range(3))
    pre = torch.empty(B, H, N, dtype=torch.float32, device=dev) if with_norms else None
    post = torch.empty(B, H, N, dtype=torch.float32, device=dev) if with_norms else None
    st = load().cam_prep_fwd(_ptr(q_raw), _ptr(k_raw), _ptr(v_raw), _ptr(q_norm_w), _ptr(k_norm_w),
                             _ptr(proj_q), _ptr(proj_kv), _ptr(rope_cos), _ptr(rope_sin),
                             float(rope_base), _ptr(outs[0]), _ptr(outs[1]), _ptr(outs[2]), _ptr(pre),
                             _ptr(post), B, N, H, D, float(k_scale), float(eps), code, _stream(stream))
    _raise("cam_prep_fwd", st)
    return outs[0], outs[1], outs[2], pre, post


def cam_scan_bwd(q, k, v, beta, decay, do, initial_state=None, dfinal_state=None, scale=1.0, l2norm=False,
                 need_dinitial=False, workspace=None, stream=None, simt=False):
    """Backward of cam_scan_fwd (forward direction).  Returns (dq, dk, dv,
    dbeta, ddecay, dinitial_state or None); dq, dk, dv in the inputs' dtype,
    the rest fp32.  simt=True keeps the token gradients on the CUDA cores."""
    B, H, N, Dk = q.shape
    Dv = v.shape[-1]
    F = decay.shape[-1]
    if F <= 0 or N % F != 0:
        raise ValueError(f"{N} tokens do not split into {F} frames")
    S = N // F
    dt = q.dtype
    code = _dtype_code(q)
    _check(q, "q", (B, H, N, Dk), dt)
    _check(k, "k", (B, H, N, Dk), dt)
    _check(v, "v", (B, H, N, Dv), dt)
    _check(beta, "beta", (B, H, N), dt)
    _check(decay, "decay", (B, H, F), torch.float32)
    _check(do, "do", (B, H, N, Dv), dt)
    for name, t in (("initial_state", initial_state), ("dfinal_state", dfinal_state)):
        if t is not None:
            _check(t, name, (B, H, Dk, Dv), torch.float32)
    dev = q.device
    dq, dk = torch.empty_like(q), torch.empty_like(k)
    dv = torch.empty_like(v)
    dbeta = torch.empty(B, H, N, dtype=torch.float32, device=dev)
    ddecay = torch.empty(B, H, F, dtype=torch.float32, device=dev)
    ds0 = torch.empty(B, H, Dk, Dv, dtype=torch.float32, device=dev) if need_dinitial else None
    lib = load()
    need = lib.cam_scan_bwd_workspace_bytes(B, H, F, S, Dk, Dv, code)
    if workspace is None:
        workspace = torch.empty(int(need), dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size()
    st = lib.cam_scan_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(decay), _ptr(initial_state), _ptr(do),
                          _ptr(dfinal_state), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dbeta), _ptr(ddecay), _ptr(ds0),
                          B, H, F, S, Dk, Dv, float(scale),
                          (GDN_QK_L2NORM if l2norm else 0) | (GDN_PATH_SIMT if simt else 0), code,
                          _ptr(workspace), ws_bytes, _stream(stream))
    _raise("cam_scan_bwd", st)
    return dq, dk, dv, dbeta, ddecay, ds0


def gdn_chunk_bwd_workspace_bytes(B, H, T, Dk, Dv, dtype=torch.bfloat16, r=1):
    code = GDN_BF16 if dtype == torch.bfloat16 else GDN_F32
    return int(load().gdn_chunk_bwd_workspace_bytes(B, H, T, r, Dk, Dv, code))


def deltaproduct_chunk_bwd(q, k, v, beta, g, do, initial_state=None, dfinal_state=None, scale=1.0, l2norm=False,
                           need_dinitial=False, workspace=None, stream=None, simt=False):
    """Backward of deltaproduct_chunk_fwd: k [B,H,T,r,Dk], v [B,H,T,r,Dv],
    beta [B,H,T,r].  Returns (dq, dk, dv, dbeta, dg, dinitial_state or None);
    dq, dk, dv in the inputs' dtype, the rest fp32."""
    B, H, T, Dk = q.shape
    r, Dv = k.shape[3], v.shape[-1]
    dt = q.dtype
    code = _dtype_code(q)
    _check(q, "q", (B, H, T, Dk), dt)
    _check(k, "k", (B, H, T, r, Dk), dt)
    _check(v, "v", (B, H, T, r, Dv), dt)
    _check(beta, "beta", (B, H, T, r), dt)
    _check(g, "g", (B, H, T), torch.float32)
    _check(do, "do", (B, H, T, Dv), dt)
    for name, t in (("initial_state", initial_state), ("dfinal_state", dfinal_state)):
        if t is not None:
            _check(t, name, (B, H, Dk, Dv), torch.float32)
    dev = q.device
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dbeta = torch.empty(B, H, T, r, dtype=torch.float32, device=dev)
    dg = torch.empty(B, H, T, dtype=torch.float32, device=dev)
    ds0 = torch.empty(B, H, Dk, Dv, dtype=torch.float32, device=dev) if need_dinitial else None
    lib = load()
    if workspace is None:
        need = lib.gdn_chunk_bwd_workspace_bytes(B, H, T, r, Dk, Dv, code)
        workspace = torch.empty(max(int(need), 16), dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size()
    flags = (GDN_QK_L2NORM if l2norm else 0) | (GDN_PATH_SIMT if simt else 0)
    st = lib.deltaproduct_chunk_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(initial_state), _ptr(do),
                                    _ptr(dfinal_state), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dbeta), _ptr(dg),
                                    _ptr(ds0), B, H, T, r, Dk, Dv, float(scale), flags,
                                    code,
                                    _ptr(workspace), ws_bytes, _stream(stream))
    _raise("deltaproduct_chunk_bwd", st)
    return dq, dk, dv, dbeta, dg, ds0


def masked_deltaproduct_chunk_bwd(q, k, v, beta, g, mask, do, initial_state=None, dfinal_state=None, scale=1.0,
                                  l2norm=False, need_dinitial=False, workspace=None, stream=None, simt=False):
    """Backward of masked_deltaproduct_chunk_fwd.  Returns (dq, dk, dv, dbeta,
    dg, dinitial_state or None); dq, dk, dv in the inputs' dtype, the rest fp32."""
    B, H, T, Dk = q.shape
    Dv = v.shape[-1]
    r = mask.shape[0]
    dt = q.dtype
    code = _dtype_code(q)
    _check(q, "q", (B, H, T, Dk), dt)
    _check(k, "k", (B, H, T, Dk), dt)
    _check(v, "v", (B, H, T, Dv), dt)
    _check(beta, "beta", (B, H, T), dt)
    _check(g, "g", (B, H, T), torch.float32)
    _check(mask, "mask", (r, r), torch.float32)
    _check(do, "do", (B, H, T, Dv), dt)
    for name, t in (("initial_state", initial_state), ("dfinal_state", dfinal_state)):
        if t is not None:
            _check(t, name, (B, H, Dk, Dv), torch.float32)
    dev = q.device
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dbeta = torch.empty(B, H, T, dtype=torch.float32, device=dev)
    dg = torch.empty(B, H, T, dtype=torch.float32, device=dev)
    ds0 = torch.empty(B, H, Dk, Dv, dtype=torch.float32, device=dev) if need_dinitial else None
    lib = load()
    if workspace is None:
        need = lib.masked_deltaproduct_chunk_bwd_workspace_bytes(B, H, T, r, Dk, Dv, code)
        workspace = torch.empty(max(int(need), 16), dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size()
    flags = (GDN_QK_L2NORM if l2norm else 0) | (GDN_PATH_SIMT if simt else 0)
    st = lib.masked_deltaproduct_chunk_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(mask),
                                           _ptr(initial_state), _ptr(do), _ptr(dfinal_state), _ptr(dq), _ptr(dk),
                                           _ptr(dv), _ptr(dbeta), _ptr(dg), _ptr(ds0), B, H, T, r, Dk, Dv,
                                           float(scale), flags,
                                           code, _ptr(workspace),
                                           ws_bytes, _stream(stream))
    _raise("masked_deltaproduct_chunk_bwd", st)
    return dq, dk, dv, dbeta, dg, ds0


def gdn_chunk_bwd(q, k, v, beta, g, do, initial_state=None, dfinal_state=None, scale=1.0, l2norm=False,
                  need_dinitial=False, workspace=None, stream=None, simt=False):
    """Backward of gdn_chunk_fwd.  Returns (dq, dk, dv, dbeta, dg,
    dinitial_state or None); dq, dk, dv in the inputs' dtype, the rest fp32."""
    B, H, T, Dk = q.shape
    Dv = v.shape[-1]
    dt = q.dtype
    code = _dtype_code(q)
    _check(q, "q", (B, H, T, Dk), dt)
    _check(k, "k", (B, H, T, Dk), dt)
    _check(v, "v", (B, H, T, Dv), dt)
    _check(beta, "beta", (B, H, T), dt)
    _check(g, "g", (B, H, T), torch.float32)
    _check(do, "do", (B, H, T, Dv), dt)
    for name, t in (("initial_state", initial_state), ("dfinal_state", dfinal_state)):
        if t is not None:
            _check(t, name, (B, H, Dk, Dv), torch.float32)
    dev = q.device
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    dbeta = torch.empty(B, H, T, dtype=torch.float32, device=dev)
    dg = torch.empty(B, H, T, dtype=torch.float32, device=dev)
    ds0 = torch.empty(B, H, Dk, Dv, dtype=torch.float32, device=dev) if need_dinitial else None
    lib = load()
    if workspace is None:
        need = lib.gdn_chunk_bwd_workspace_bytes(B, H, T, 1, Dk, Dv, code)
        workspace = torch.empty(max(int(need), 16), dtype=torch.uint8, device=dev)
    ws_bytes = workspace.numel() * workspace.element_size()
    flags = (GDN_QK_L2NORM if l2norm else 0) | (GDN_PATH_SIMT if simt else 0)
    st = lib.gdn_chunk_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g), _ptr(initial_state), _ptr(do),
                           _ptr(dfinal_state), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dbeta), _ptr(dg), _ptr(ds0), B, H, T,
                           Dk, Dv, float(scale), flags,
                           code, _ptr(workspace), ws_bytes, _stream(stream))
    _raise("gdn_chunk_bwd", st)
    return dq, dk, dv, dbeta, dg, ds0


def cam_prep_bwd(q_raw, k_raw, proj_q, proj_kv, dq_out, dk_out, dv_out, dk_pre_sq=None, dk_post_sq=None,
                 q_norm_w=None, k_norm_w=None, rope_cos=None, rope_sin=None, rope_base=10000.0, k_scale=0.5,
                 eps=1e-6, stream=None):
    """Backward of cam_prep_fwd: gradients of the raw q, k, v [B,N,H,D] from
    those of q_out, k_out, v_out [B,H,N,D] (and of k_pre_sq, k_post_sq)."""
    B, N, H, D = q_raw.shape
    dt = q_raw.dtype
    code = _dtype_code(q_raw)
    _check(k_raw, "k_raw", (B, N, H, D), dt)
    _check(proj_q, "proj_q", (B, N, 4, 4), torch.float32)
    _check(proj_kv, "proj_kv", (B, N, 4, 4), torch.float32)
    for name, t in (("dq_out", dq_out), ("dk_out", dk_out), ("dv_out", dv_out)):
        _check(t, name, (B, H, N, D), dt)
    for name, t in (("dk_pre_sq", dk_pre_sq), ("dk_post_sq", dk_post_sq)):
        if t is not None:
            _check(t, name, (B, H, N), torch.float32)
    outs = tuple(torch.empty(B, N, H, D, dtype=dt, device=q_raw.device) for _ in range(3))
    st = load().cam_prep_bwd(_ptr(q_raw), _ptr(k_raw), _ptr(q_norm_w), _ptr(k_norm_w), _ptr(proj_q), _ptr(proj_kv),
                             _ptr(rope_cos), _ptr(rope_sin), float(rope_base), _ptr(dq_out), _ptr(dk_out),
                             _ptr(dv_out), _ptr(dk_pre_sq), _ptr(dk_post_sq), _ptr(outs[0]), _ptr(outs[1]),
                             _ptr(outs[2]), B, N, H, D, float(k_scale), float(eps), code, _stream(stream))
    _raise("cam_prep_bwd", st)
    return outs


def device_error(stream=None) -> int:
    """Synchronise ``stream`` and read/clear the library's device error word."""
    return int(load().gdn_get_device_error(_stream(stream)))


def set_wait_limit(us: int) -> None:
    """Wall-clock limit in microseconds of each bounded device wait (0 = default)."""
    _raise("gdn_set_wait_limit", load().gdn_set_wait_limit(int(us)))


def set_cluster_shape(heads_per_cluster: int = 0, wy_ctas_per_cluster: int = 0) -> None:
    """Cluster shape of the tcgen05 path (0, 0: automatic)."""
    _raise("gdn_set_cluster_shape", load().gdn_set_cluster_shape(int(heads_per_cluster), int(wy_ctas_per_cluster)))


def launch_count() -> int:
    """Kernels the library has launched in this process so far."""
    return int(load().gdn_launch_count())


def status_string(code: int) -> str:
    return load().gdn_status_string(int(code)).decode()
