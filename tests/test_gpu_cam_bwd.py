"""GPU parity of the camera-prep backward (fused_cam_gdn.py,
``_cam_prep_bwd_kernel``, continued through the full-C RMSNorm) against the
fp64 oracle backward (itself pinned by finite differences), through the C
ABI.  Metric: max|g - g_ref| / max|g_ref| <= 1e-4 (fp32), 1e-2 (bf16).  bf16
with rotary tables and C <= 2048 takes the streamed kernel (stages of three
positions, so N = 37, 13, 9 and 300 end on full and partial stages, and B = 2
crosses a batch row); C = 4096 and the other cases take the per-token kernel."""
import pytest
import torch

import oracle
from gated_delta_rule_47_gb300 import binding
from gated_delta_rule_47_gb300.inputs import WORKLOADS, cam_inputs
from tests.gpu_util import TOL_BF16, TOL_F32, ensure_lib, rel_err, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def grads(B, N, H, D, seed, dtype):
    g = torch.Generator().manual_seed(seed)
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    up = [torch.randn(B, H, N, D, generator=g).to(td).contiguous() for _ in range(3)]
    sq = [torch.randn(B, H, N, generator=g).contiguous() for _ in range(2)]
    return up, sq


@pytest.mark.parametrize("dtype,tol", [("f32", TOL_F32), ("bf16", TOL_BF16)])
@pytest.mark.parametrize("tables", [True, False])
@pytest.mark.parametrize("B,N,H,D", [(1, 37, 16, 128), (2, 13, 4, 64), (1, 9, 3, 32), (1, 300, 2, 128), (1, 7, 32, 128)])
def test_prep_backward(dtype, tol, tables, B, N, H, D):
    inp = cam_inputs(B, N, H, D, seed=N + H + 1, dtype=dtype, tables=tables)
    g = torch.Generator().manual_seed(11)
    inp["q_norm_w"] = torch.rand(H * D, generator=g) + 0.5
    inp["k_norm_w"] = torch.rand(H * D, generator=g) + 0.5
    up, sq = grads(B, N, H, D, seed=3, dtype=dtype)
    d = to_dev(inp)
    got = binding.cam_prep_bwd(d["q_raw"], d["k_raw"], d["proj_q"], d["proj_kv"], up[0].cuda(), up[1].cuda(),
                               up[2].cuda(), sq[0].cuda(), sq[1].cuda(), d["q_norm_w"], d["k_norm_w"], d["rope_cos"],
                               d["rope_sin"])
    torch.cuda.synchronize()
    ref = oracle.cam_prep_bwd(inp["q_raw"], inp["k_raw"], inp["v_raw"], inp["proj_q"], inp["proj_kv"], up[0], up[1],
                              up[2], sq[0], sq[1], inp["q_norm_w"], inp["k_norm_w"], inp["rope_cos"],
                              inp["rope_sin"])
    for x, y in zip(got, ref):
        assert rel_err(x, y) <= tol


def test_prep_backward_camera_workload_size():
    """The camera workload's size (B2, N 32760, H16, D128, bf16, rotary
    tables): every output element against the oracle."""
    w = WORKLOADS["cam_b2n32760h16d128_bf16"]
    inp = w.make()
    up, sq = grads(w.B, w.T, w.H, w.D, seed=4, dtype="bf16")
    d = to_dev(inp)
    got = binding.cam_prep_bwd(d["q_raw"], d["k_raw"], d["proj_q"], d["proj_kv"], up[0].cuda(), up[1].cuda(),
                               up[2].cuda(), None, None, d["q_norm_w"], d["k_norm_w"], d["rope_cos"], d["rope_sin"])
    torch.cuda.synchronize()
    ref = oracle.cam_prep_bwd(inp["q_raw"], inp["k_raw"], inp["v_raw"], inp["proj_q"], inp["proj_kv"], up[0], up[1],
                              up[2], None, None, inp["q_norm_w"], inp["k_norm_w"], inp["rope_cos"], inp["rope_sin"])
    for x, y in zip(got, ref):
        assert rel_err(x, y) <= TOL_BF16


@pytest.mark.parametrize("B,N,H,D", [(1, 1, 16, 128), (2, 4, 8, 128), (1, 5, 4, 64)])
@pytest.mark.parametrize("pre,post,weights", [(True, False, False), (False, True, True), (False, False, False)])
def test_prep_backward_optional_inputs(B, N, H, D, pre, post, weights):
    """bf16 with rotary tables (the streamed kernel): a single token, a full stage
    and a partial one, with the norm weights and each ||k||^2 gradient left out or
    given on its own, and D = 64 beside the D = 128 specialisation."""
    inp = cam_inputs(B, N, H, D, seed=N + 7 * H, dtype="bf16", tables=True)
    g = torch.Generator().manual_seed(13)
    qw = torch.rand(H * D, generator=g) + 0.5 if weights else None
    kw = torch.rand(H * D, generator=g) + 0.5 if weights else None
    up, sq = grads(B, N, H, D, seed=5, dtype="bf16")
    dpre, dpost = (sq[0] if pre else None), (sq[1] if post else None)
    d = to_dev(inp)
    got = binding.cam_prep_bwd(d["q_raw"], d["k_raw"], d["proj_q"], d["proj_kv"], up[0].cuda(), up[1].cuda(),
                               up[2].cuda(), dpre.cuda() if pre else None, dpost.cuda() if post else None,
                               qw.cuda() if weights else None, kw.cuda() if weights else None, d["rope_cos"],
                               d["rope_sin"])
    torch.cuda.synchronize()
    ref = oracle.cam_prep_bwd(inp["q_raw"], inp["k_raw"], inp["v_raw"], inp["proj_q"], inp["proj_kv"], up[0], up[1],
                              up[2], dpre, dpost, qw, kw, inp["rope_cos"], inp["rope_sin"])
    for x, y in zip(got, ref):
        assert rel_err(x, y) <= TOL_BF16
