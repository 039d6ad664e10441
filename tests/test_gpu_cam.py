"""GPU parity of the fused camera prep, and of the camera workload end to end
(prep, then the scan with unit-normalised q/k), against the fp64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_47_gb300 import binding
from gated_delta_rule_47_gb300.inputs import WORKLOADS, cam_inputs, to_f64
from tests.gpu_util import TOL_BF16, TOL_F32, ensure_lib, heads, rel_err, sample_heads, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def run_prep(inp, **kw):
    d = to_dev(inp)
    out = binding.cam_prep_fwd(d["q_raw"], d["k_raw"], d["v_raw"], d["proj_q"], d["proj_kv"],
                               d["q_norm_w"], d["k_norm_w"], d["rope_cos"], d["rope_sin"], **kw)
    torch.cuda.synchronize()
    return out


def ref_prep(inp, **kw):
    return oracle.cam_prep_fwd(inp["q_raw"], inp["k_raw"], inp["v_raw"], inp["proj_q"], inp["proj_kv"],
                               inp["q_norm_w"], inp["k_norm_w"], inp["rope_cos"], inp["rope_sin"], **kw)


@pytest.mark.parametrize("dtype,tol", [("f32", TOL_F32), ("bf16", TOL_BF16)])
@pytest.mark.parametrize("tables", [True, False])
@pytest.mark.parametrize("B,N,H,D", [(1, 37, 16, 128), (2, 13, 4, 64), (1, 9, 3, 32), (1, 300, 2, 128)])
def test_prep_small(dtype, tol, tables, B, N, H, D):
    inp = cam_inputs(B, N, H, D, seed=N + H, dtype=dtype, tables=tables)
    g = torch.Generator().manual_seed(5)
    inp["q_norm_w"] = torch.rand(H * D, generator=g) + 0.5
    inp["k_norm_w"] = torch.rand(H * D, generator=g) + 0.5
    got = run_prep(inp, k_scale=0.5, eps=1e-6)
    ref = ref_prep(inp, k_scale=0.5, eps=1e-6)
    for x, y in zip(got, ref):
        assert rel_err(x, y) <= tol


def test_prep_fp32_angles_formed_in_kernel_at_long_positions():
    """fp32 prep without tables over the camera workload's length (positions
    0 .. 32759): the kernel forms th = n * 10000^(-2i/(D/2)) and reduces it
    modulo 2 pi in double before the fp32 sine and cosine, so even the
    largest positions stay within the fp32 bound."""
    inp = cam_inputs(1, 21 * 30 * 52, 2, 128, seed=17, dtype="f32", tables=False)
    got = run_prep(inp, k_scale=0.5, eps=1e-6)
    ref = ref_prep(inp, k_scale=0.5, eps=1e-6)
    for x, y in zip(got, ref):
        assert rel_err(x, y) <= TOL_F32
    # the rotary half of the last thousand positions on its own
    late = (slice(None), slice(None), slice(-1000, None), slice(64, None))
    for x, y in zip(got[:3], ref[:3]):
        assert rel_err(x[late].contiguous(), y[late]) <= TOL_F32


def test_prep_without_norm_outputs():
    inp = cam_inputs(1, 20, 16, 128, seed=3)
    q, k, v, pre, post = run_prep(inp, with_norms=False)
    assert pre is None and post is None
    ref = ref_prep(inp)
    assert rel_err(k, ref[1]) <= TOL_BF16


def test_camera_workload_full_size():
    """Full camera workload in the bench's launch configuration: the prep
    outputs are compared element by element; the scan on them is compared on
    sampled heads against the oracle run on the oracle's own prep output."""
    w = WORKLOADS["cam_b2n32760h16d128_bf16"]
    inp = w.make()
    q, k, v, pre, post = run_prep(inp, k_scale=0.5, eps=1e-6)
    ref = ref_prep(inp, k_scale=0.5, eps=1e-6)
    for x, y in zip((q, k, v, pre, post), ref):
        assert rel_err(x, y) <= TOL_BF16
    dev_beta, dev_g = inp["beta"].cuda(), inp["g"].cuda()
    o, _ = binding.gdn_chunk_fwd(q, k, v, dev_beta, dev_g, chunk=w.chunk, l2norm=True)
    torch.cuda.synchronize()
    assert torch.isfinite(o).all()
    idx = sample_heads(w.B, w.H, 2, seed=w.seed)
    ro, _ = oracle.gdn_fwd(heads(ref[0], idx), heads(ref[1], idx), heads(ref[2], idx),
                           heads(to_f64(inp["beta"]), idx), heads(to_f64(inp["g"]), idx), l2norm=True)
    assert rel_err(heads(o, idx).cpu(), ro) <= TOL_BF16
