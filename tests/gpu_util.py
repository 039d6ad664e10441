"""Helpers shared by the GPU parity tests: build-and-load of the library,
device copies of seeded inputs, the parity metric, and head sampling."""
from __future__ import annotations

import numpy as np
import torch

from gated_delta_rule_47_gb300 import binding, build
from gated_delta_rule_47_gb300.inputs import to_f64

# max|o - o_ref| / max|o_ref| bounds of the method's accuracy targets.
TOL_F32 = 1e-4
TOL_BF16 = 1e-2

_built = False


def ensure_lib():
    global _built
    if not _built:
        build.build()
        binding.load()
        _built = True


def to_dev(d, device="cuda"):
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def rel_err(x, ref):
    x = to_f64(x) if isinstance(x, torch.Tensor) else np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    assert x.shape == ref.shape, (x.shape, ref.shape)
    assert np.all(np.isfinite(x)), "non-finite values in the CUDA output"
    return float(np.max(np.abs(x - ref)) / max(np.max(np.abs(ref)), 1e-30))


def heads(x, idx):
    """Rows of the flattened (b,h) axis, as a [1, len(idx), ...] tensor/array."""
    B, H = x.shape[:2]
    flat = x.reshape(B * H, *x.shape[2:])
    return flat[list(idx)].unsqueeze(0) if isinstance(x, torch.Tensor) else flat[list(idx)][None]


def sample_heads(B, H, n, seed=0):
    rng = np.random.default_rng(seed)
    idx = sorted(set([0, B * H - 1] + list(rng.choice(B * H, size=min(n, B * H), replace=False))))
    return idx[: max(n, 2)]
