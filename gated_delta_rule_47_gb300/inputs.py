"""Seeded synthetic inputs shared by the CUDA path and the fp64 checker.

This module holds no arithmetic of the method itself: it only draws random
tensors with the value distributions of the workloads (unit-norm q/k, normal
v, sigmoid beta, log-sigmoid decay, random SE(3) camera poses, rotary tables)
and rounds them to the compute dtype.  Everything is drawn on the CPU with a
``torch.Generator`` so that both consumers receive identical bytes.

Draw order for the scan inputs: q, k, v, beta-logit, g-logit, then the
optional initial state.  q and k are normalised in fp32 before the cast.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

_DTYPES = {"f32": torch.float32, "bf16": torch.bfloat16}


def torch_dtype(name: str) -> torch.dtype:
    return _DTYPES[name]


def _unit_rows(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)


def gdn_inputs(B, H, T, Dk, Dv, seed, dtype="bf16", g_mu=0.0, g_div=16.0, r=None,
               initial_state=False, normalise_qk=True):
    """Inputs of one scan workload as CPU tensors.

    GDN (r is None): q, k [B,H,T,Dk]; v [B,H,T,Dv]; beta [B,H,T]; g [B,H,T] fp32.
    DeltaProduct (r given): k [B,H,T,r,Dk]; v [B,H,T,r,Dv]; beta [B,H,T,r]; each
    sub-step gets its own unit key, value and beta.
    q, k ~ N(0,1) normalised per row; v ~ N(0,1); beta = sigmoid(N(0,1));
    g = logsigmoid(N(g_mu,1)) / g_div; initial_state ~ N(0,1) fp32 if asked for.
    q, k, v, beta are rounded to ``dtype``; g and the state stay fp32.
    """
    gen = torch.Generator().manual_seed(int(seed))
    sub = () if r is None else (int(r),)
    q = torch.randn(B, H, T, Dk, generator=gen)
    k = torch.randn(B, H, T, *sub, Dk, generator=gen)
    v = torch.randn(B, H, T, *sub, Dv, generator=gen)
    beta_logit = torch.randn(B, H, T, *sub, generator=gen)
    g_logit = torch.randn(B, H, T, generator=gen) + g_mu
    s0 = torch.randn(B, H, Dk, Dv, generator=gen) if initial_state else None
    if normalise_qk:
        q, k = _unit_rows(q), _unit_rows(k)
    td = _DTYPES[dtype]
    out = {
        "q": q.to(td).contiguous(),
        "k": k.to(td).contiguous(),
        "v": v.to(td).contiguous(),
        "beta": torch.sigmoid(beta_logit).to(td).contiguous(),
        "g": (torch.nn.functional.logsigmoid(g_logit) / g_div).float().contiguous(),
    }
    if s0 is not None:
        out["initial_state"] = s0.float().contiguous()
    return out


def mixed_decay(B, H, T, seed, r=1, chunk_rows=64, strong=2.0):
    """Per-token log-decay g [B,H,T] fp32 whose 64-row chunks cycle through
    three regimes, so that one head holds all of them: strong forgetting
    (about -strong*r per token: a chunk's cumulative decay spans well over
    80 nats), the workloads' weak decay logsigmoid(N(0,1))/16, and a chunk
    whose cumulative decay spans about 70 nats.  r is the number of rows per
    token (DeltaProduct sub-steps), so that chunks are counted in rows."""
    gen = torch.Generator().manual_seed(int(seed))
    z = torch.randn(B, H, T, generator=gen)
    regime = ((torch.arange(T) * r) // chunk_rows) % 3
    tok_per_chunk = chunk_rows / r
    strong_g = -strong * r * (1.0 + 0.25 * z.abs())
    weak_g = torch.nn.functional.logsigmoid(z) / 16.0
    border_g = torch.full_like(z, -70.0 / tok_per_chunk)
    g = torch.where(regime == 0, strong_g, torch.where(regime == 1, weak_g, border_g))
    return g.float().contiguous()


def orthonormal_keys(B, H, T, D, seed):
    """[B,H,T,D] fp32 keys whose T <= D rows per head are orthonormal (rows of
    a random orthogonal matrix from the QR factorisation of a Gaussian)."""
    assert T <= D
    gen = torch.Generator().manual_seed(int(seed))
    a = torch.randn(B * H, D, D, generator=gen, dtype=torch.float64)
    qm, _ = torch.linalg.qr(a)
    return qm[:, :T, :].reshape(B, H, T, D).float().contiguous()


def slice_mask(r, seed):
    """An r x r mask for the block-masked DeltaProduct: a random correlation
    matrix (X X^T scaled to a unit diagonal, X ~ N(0,1)^{r x r}), fp32.  Being
    positive semi-definite with a unit diagonal, it keeps the transition
    I - beta (k k^T) o M contractive for unit keys and beta <= 1."""
    gen = torch.Generator().manual_seed(int(seed))
    x = torch.randn(r, r, generator=gen, dtype=torch.float64)
    m = x @ x.T
    d = torch.sqrt(torch.diagonal(m))
    return (m / d[:, None] / d[None, :]).float().contiguous()


def frame_gates(B, H, F, S, seed, dtype="bf16"):
    """Gates of the frame-level camera scan: beta [B,H,F*S] = sigmoid(N(0,1)) / S
    in ``dtype`` (each frame's S corrections enter at once, so their sum is
    scaled by the frame size, which keeps I - K^T diag(beta) K contractive for
    unit keys), and one decay factor per frame, decay [B,H,F] =
    exp(logsigmoid(N(0,1)) / 16) in fp32."""
    gen = torch.Generator().manual_seed(int(seed))
    beta_logit = torch.randn(B, H, F * S, generator=gen)
    g_logit = torch.randn(B, H, F, generator=gen)
    return (torch.sigmoid(beta_logit) / S).to(_DTYPES[dtype]).contiguous(), \
        torch.exp(torch.nn.functional.logsigmoid(g_logit) / 16.0).float().contiguous()


def cam_scan_inputs(B, H, F, S, Dk, Dv, seed, dtype="bf16", initial_state=False, normalise_qk=True):
    """Inputs of one frame-scan workload as CPU tensors: q, k [B,H,F*S,Dk]
    (N(0,1), unit rows unless normalise_qk is False), v [B,H,F*S,Dv] ~ N(0,1),
    the frame gates of ``frame_gates`` and, if asked, an initial state ~ N(0,1)
    [B,H,Dk,Dv] fp32.  Draw order: q, k, v, initial state, then the gates."""
    gen = torch.Generator().manual_seed(int(seed))
    N = F * S
    q = torch.randn(B, H, N, Dk, generator=gen)
    k = torch.randn(B, H, N, Dk, generator=gen)
    v = torch.randn(B, H, N, Dv, generator=gen)
    s0 = torch.randn(B, H, Dk, Dv, generator=gen) if initial_state else None
    if normalise_qk:
        q, k = _unit_rows(q), _unit_rows(k)
    td = _DTYPES[dtype]
    beta, decay = frame_gates(B, H, F, S, seed + 7919, dtype)
    out = {"q": q.to(td).contiguous(), "k": k.to(td).contiguous(), "v": v.to(td).contiguous(),
           "beta": beta, "decay": decay}
    if s0 is not None:
        out["initial_state"] = s0.float().contiguous()
    return out


def quaternion_rotations(n: int, gen: torch.Generator) -> torch.Tensor:
    """n rotation matrices from uniformly random unit quaternions (normalised
    4-D Gaussians), fp64, shape [n,3,3]."""
    qt = torch.randn(n, 4, generator=gen, dtype=torch.float64)
    qt = qt / qt.norm(dim=-1, keepdim=True)
    w, x, y, z = qt.unbind(-1)
    R = torch.stack([
        1 - 2 * (y * y + z * z), 2 * (x * y - z * w), 2 * (x * z + y * w),
        2 * (x * y + z * w), 1 - 2 * (x * x + z * z), 2 * (y * z - x * w),
        2 * (x * z - y * w), 2 * (y * z + x * w), 1 - 2 * (x * x + y * y),
    ], dim=-1).reshape(n, 3, 3)
    return R


def se3_poses(n: int, gen: torch.Generator) -> torch.Tensor:
    """n random poses P = [[R, t], [0, 1]] with t ~ N(0,1)^3, fp64 [n,4,4]."""
    R = quaternion_rotations(n, gen)
    t = torch.randn(n, 3, generator=gen, dtype=torch.float64)
    P = torch.zeros(n, 4, 4, dtype=torch.float64)
    P[:, :3, :3] = R
    P[:, :3, 3] = t
    P[:, 3, 3] = 1.0
    return P


def se3_inverse(P: torch.Tensor) -> torch.Tensor:
    """Closed-form inverse [[R^T, -R^T t], [0, 1]] of a batch of SE(3) poses
    (fused_cam_gdn.py, ``_invert_SE3``)."""
    Rt = P[..., :3, :3].transpose(-1, -2)
    out = torch.zeros_like(P)
    out[..., :3, :3] = Rt
    out[..., :3, 3] = -(Rt @ P[..., :3, 3:4]).squeeze(-1)
    out[..., 3, 3] = 1.0
    return out


def rope_tables(N: int, D_half: int, base: float = 10000.0):
    """Rotary tables in the interleaved encoding y[d] = x[d] cos[d] + x[d^1] sin[d]
    (fused_cam_gdn.py, ``_prepare_ucpe_rope_tables``): cos[n,2i] = cos[n,2i+1] =
    cos(th), sin[n,2i] = -sin(th), sin[n,2i+1] = sin(th), th = n base^(-2i/D_half),
    with n the flattened token index.  Angles in fp64, tables rounded to fp32."""
    i = torch.arange(D_half // 2, dtype=torch.float64)
    th = torch.arange(N, dtype=torch.float64)[:, None] * torch.pow(
        torch.tensor(base, dtype=torch.float64), -2.0 * i / D_half)[None, :]
    cos = torch.repeat_interleave(torch.cos(th), 2, dim=-1)
    sin = torch.stack([-torch.sin(th), torch.sin(th)], dim=-1).reshape(N, D_half)
    return cos.float().contiguous(), sin.float().contiguous()


def cam_inputs(B, N, H, D, seed, dtype="bf16", tables=True, g_mu=0.0, g_div=16.0):
    """Camera-branch workload: raw q, k, v [B,N,H,D] ~ N(0,1) in ``dtype``; unit
    norm weights [H*D] fp32; one random SE(3) pose P per (b,n) with
    proj_q = P^T and proj_kv = P^-1 ([B,N,4,4] fp32); rotary tables [N,D/2]
    fp32 (or None); and the scan's beta [B,H,N] (dtype) and g [B,H,N] fp32."""
    gen = torch.Generator().manual_seed(int(seed))
    td = _DTYPES[dtype]
    q = torch.randn(B, N, H, D, generator=gen).to(td).contiguous()
    k = torch.randn(B, N, H, D, generator=gen).to(td).contiguous()
    v = torch.randn(B, N, H, D, generator=gen).to(td).contiguous()
    P = se3_poses(B * N, gen)
    proj_q = P.transpose(-1, -2).reshape(B, N, 4, 4).float().contiguous()
    proj_kv = se3_inverse(P).reshape(B, N, 4, 4).float().contiguous()
    beta_logit = torch.randn(B, H, N, generator=gen)
    g_logit = torch.randn(B, H, N, generator=gen) + g_mu
    out = {
        "q_raw": q, "k_raw": k, "v_raw": v,
        "q_norm_w": torch.ones(H * D), "k_norm_w": torch.ones(H * D),
        "proj_q": proj_q, "proj_kv": proj_kv,
        "beta": torch.sigmoid(beta_logit).to(td).contiguous(),
        "g": (torch.nn.functional.logsigmoid(g_logit) / g_div).float().contiguous(),
    }
    if tables:
        out["rope_cos"], out["rope_sin"] = rope_tables(N, D // 2)
    else:
        out["rope_cos"] = out["rope_sin"] = None
    return out


@dataclass(frozen=True)
class Workload:
    """One named workload: sizes, dtype, distribution knobs and seed."""
    name: str
    kind: str  # "gdn" | "deltaproduct" | "cam" | "masked_dp"
    B: int
    H: int
    T: int
    D: int
    chunk: int
    dtype: str
    seed: int
    r: int = 1
    g_mu: float = 0.0
    extra: dict = field(default_factory=dict)

    @property
    def tokens(self) -> int:
        return self.B * self.T

    def make(self, **overrides):
        kw = dict(B=self.B, H=self.H, T=self.T, seed=self.seed, dtype=self.dtype, g_mu=self.g_mu)
        kw.update(overrides)
        if self.kind == "cam":
            N = kw.pop("T")
            kw.pop("g_mu")
            return cam_inputs(kw["B"], N, kw["H"], self.D, kw["seed"], dtype=kw["dtype"])
        if self.kind == "masked_dp":
            out = gdn_inputs(kw["B"], kw["H"], kw["T"], self.D, self.D, kw["seed"], dtype=kw["dtype"],
                             g_mu=kw["g_mu"])
            out["mask"] = slice_mask(self.r, kw["seed"] + 1)
            return out
        r = None if self.kind == "gdn" else self.r
        return gdn_inputs(kw["B"], kw["H"], kw["T"], self.D, self.D, kw["seed"], dtype=kw["dtype"],
                          g_mu=kw["g_mu"], r=r)


# The five workloads of the method's benchmark description.
WORKLOADS = {
    "gdn_tiny_f32": Workload("gdn_tiny_f32", "gdn", 1, 2, 256, 64, 64, "f32", 0),
    "gdn_b4h16t4096d128_bf16": Workload("gdn_b4h16t4096d128_bf16", "gdn", 4, 16, 4096, 128, 64, "bf16", 1),
    "gdn_long_b1h32t32768d128_bf16": Workload("gdn_long_b1h32t32768d128_bf16", "gdn", 1, 32, 32768, 128, 64,
                                              "bf16", 2, g_mu=2.0),
    "deltaproduct_r2_b4h16t4096d128_bf16": Workload("deltaproduct_r2_b4h16t4096d128_bf16", "deltaproduct",
                                                    4, 16, 4096, 128, 64, "bf16", 3, r=2),
    "cam_b2n32760h16d128_bf16": Workload("cam_b2n32760h16d128_bf16", "cam", 2, 16, 21 * 30 * 52, 128, 64,
                                         "bf16", 4),
    # the block-masked DeltaProduct variant at the DeltaProduct workload's sizes:
    # one key, value and beta per token (GDN's distributions), r = 2 slices
    # coupled by a random correlation mask; chunk counts sub-rows
    "masked_dp_r2_b4h16t4096d128_bf16": Workload("masked_dp_r2_b4h16t4096d128_bf16", "masked_dp", 4, 16, 4096,
                                                 128, 64, "bf16", 5, r=2),
}


def to_f64(x):
    """CPU fp64 numpy copy of a tensor (None passes through)."""
    if x is None:
        return None
    return np.ascontiguousarray(x.detach().cpu().double().numpy())


def split_heads_np(x, idx):
    """Select a list of flattened (b,h) heads from a [B,H,...] array as [1,len,...]."""
    B, H = x.shape[:2]
    flat = x.reshape(B * H, *x.shape[2:])
    return flat[list(idx)][None]


__all__ = ["gdn_inputs", "cam_inputs", "mixed_decay", "orthonormal_keys", "frame_gates", "cam_scan_inputs",
           "slice_mask", "rope_tables", "se3_poses", "se3_inverse",
           "quaternion_rotations", "WORKLOADS", "Workload", "to_f64", "split_heads_np",
           "torch_dtype"]
