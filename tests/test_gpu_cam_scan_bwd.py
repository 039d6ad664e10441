"""GPU parity of the frame-scan backward (fused_cam_gdn.py,
``_cam_scan_bwd_kernel``, forward direction) against the fp64 oracle
backward, itself pinned by finite differences, through the C ABI.  Metric:
max|g - g_ref| / max|g_ref| per gradient, at most 1e-4 for fp32 tensors and
1e-2 for bf16 tensors."""
import pytest
import torch

import oracle
from gated_delta_rule_47_gb300 import binding
from gated_delta_rule_47_gb300.inputs import cam_scan_inputs
from tests.gpu_util import TOL_BF16, TOL_F32, ensure_lib, rel_err, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


@pytest.mark.parametrize("l2norm", [False, True])
@pytest.mark.parametrize("dtype,tol", [("f32", TOL_F32), ("bf16", TOL_BF16)])
@pytest.mark.parametrize("F,S,Dk,Dv", [(4, 37, 128, 128), (3, 16, 64, 64), (5, 7, 64, 128), (2, 70, 128, 64),
                                        (3, 300, 128, 128), (2, 129, 128, 128)])
def test_frame_scan_backward(F, S, Dk, Dv, dtype, tol, l2norm):
    inp = cam_scan_inputs(1, 2, F, S, Dk, Dv, seed=F * S + Dk, dtype=dtype, initial_state=True,
                          normalise_qk=not l2norm)
    g = torch.Generator().manual_seed(7)
    td = inp["q"].dtype
    do = torch.randn(1, 2, F * S, Dv, generator=g).to(td)
    dsf = torch.randn(1, 2, Dk, Dv, generator=g)
    d = to_dev(inp)
    got = binding.cam_scan_bwd(d["q"], d["k"], d["v"], d["beta"], d["decay"], do.cuda(), d["initial_state"],
                               dsf.cuda(), scale=0.9, l2norm=l2norm, need_dinitial=True)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    ref = oracle.cam_scan_bwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["decay"], do, inp["initial_state"], dsf,
                              scale=0.9, l2norm=l2norm)
    for name, x, y in zip(("dq", "dk", "dv", "dbeta", "ddecay", "ds0"), got, ref):
        assert rel_err(x, y) <= tol, name


@pytest.mark.parametrize("l2norm", [False, True])
def test_tensor_core_and_cuda_core_token_gradients_agree(l2norm):
    """The tensor-core token kernel (bf16, D 128, 128-token tiles, bf16 hi/lo
    operands) and the CUDA-core one (fp32, 64-token tiles) on the same inputs,
    across ragged tiles: both within the bf16 bound of each other."""
    inp = cam_scan_inputs(1, 3, 3, 200, 128, 128, seed=12, dtype="bf16", initial_state=True,
                          normalise_qk=not l2norm)
    g = torch.Generator().manual_seed(9)
    do = torch.randn(1, 3, 600, 128, generator=g).to(torch.bfloat16).cuda()
    dsf = torch.randn(1, 3, 128, 128, generator=g).cuda()
    d = to_dev(inp)
    args = (d["q"], d["k"], d["v"], d["beta"], d["decay"], do, d["initial_state"], dsf)
    a = binding.cam_scan_bwd(*args, l2norm=l2norm, need_dinitial=True)
    b = binding.cam_scan_bwd(*args, l2norm=l2norm, need_dinitial=True, simt=True)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    for name, x, y in zip(("dq", "dk", "dv", "dbeta", "ddecay", "ds0"), a, b):
        assert rel_err(x, y.double().cpu().numpy()) <= TOL_BF16, name


def test_camera_workload_shape_sampled_heads():
    """The camera workload's shape (B2 H16, 21 frames of 1560 tokens, D128,
    bf16, unit-norm q and k): every head's gradients on the GPU, two heads
    against the oracle."""
    from tests.gpu_util import heads
    B, H, F, S = 2, 16, 21, 1560
    inp = cam_scan_inputs(B, H, F, S, 128, 128, seed=8, dtype="bf16", normalise_qk=False)
    do = torch.randn(B, H, F * S, 128, generator=torch.Generator().manual_seed(2)).to(torch.bfloat16)
    d = to_dev(inp)
    got = binding.cam_scan_bwd(d["q"], d["k"], d["v"], d["beta"], d["decay"], do.cuda(), l2norm=True)
    torch.cuda.synchronize()
    idx = [3, 30]
    sub = {k: heads(v, idx) for k, v in inp.items()}
    ref = oracle.cam_scan_bwd(sub["q"], sub["k"], sub["v"], sub["beta"], sub["decay"], heads(do, idx), l2norm=True)
    for name, x, y in zip(("dq", "dk", "dv", "dbeta", "ddecay"), got[:5], ref[:5]):
        assert rel_err(heads(x, idx).cpu(), y) <= TOL_BF16, name


@pytest.mark.parametrize("F,S", [(1, 50), (1, 128), (2, 1)])
def test_single_frame_and_single_token_frames(F, S):
    """The tensor-core frame products and chains at their edges (bf16, D 128):
    one frame (the chains take a single step each way, so the reverse chain's
    one-frame-ahead load of P never runs) and frames of one token."""
    inp = cam_scan_inputs(1, 2, F, S, 128, 128, seed=40 + F * S, dtype="bf16", initial_state=True)
    g = torch.Generator().manual_seed(11)
    do = torch.randn(1, 2, F * S, 128, generator=g).to(torch.bfloat16)
    dsf = torch.randn(1, 2, 128, 128, generator=g)
    d = to_dev(inp)
    got = binding.cam_scan_bwd(d["q"], d["k"], d["v"], d["beta"], d["decay"], do.cuda(), d["initial_state"],
                               dsf.cuda(), need_dinitial=True)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    ref = oracle.cam_scan_bwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["decay"], do, inp["initial_state"], dsf)
    for name, x, y in zip(("dq", "dk", "dv", "dbeta", "ddecay", "ds0"), got, ref):
        assert rel_err(x, y) <= TOL_BF16, name
