"""GPU parity of the camera prep fused into the frame scan (fused_cam_gdn.py,
``cam_prep_func`` then ``_cam_scan_kernel``) against the fp64 oracle's prep
followed by its frame scan, through the C ABI, and against the two unfused
library calls.  Metric: max|o - o_ref| / max|o_ref| <= 1e-2 (bf16 tensors,
fp32 state)."""
import pytest
import torch

import oracle
from gated_delta_rule_47_gb300 import binding
from gated_delta_rule_47_gb300.inputs import cam_inputs, frame_gates, to_f64
from tests.gpu_util import TOL_BF16, ensure_lib, heads, rel_err, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def make(B, N, H, F, seed, weights=True):
    inp = cam_inputs(B, N, H, 128, seed=seed, tables=False)
    if weights:
        g = torch.Generator().manual_seed(seed + 1)
        inp["q_norm_w"] = torch.rand(H * 128, generator=g) + 0.5
        inp["k_norm_w"] = torch.rand(H * 128, generator=g) + 0.5
    inp["beta"], inp["decay"] = frame_gates(B, H, F, N // F, seed=seed + 2)
    return inp


def run_fused(inp, reverse=False, l2norm=True, s0=None, final=False):
    d = to_dev(inp)
    o, sf = binding.cam_prep_scan_fwd(d["q_raw"], d["k_raw"], d["v_raw"], d["proj_q"], d["proj_kv"], d["beta"],
                                      d["decay"], d["q_norm_w"], d["k_norm_w"], rope_base=10000.0,
                                      initial_state=None if s0 is None else s0.cuda(), output_final_state=final,
                                      reverse=reverse, l2norm=l2norm)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    return o, sf


def run_oracle(inp, reverse=False, l2norm=True, s0=None, idx=None):
    q, k, v, _, _ = oracle.cam_prep_fwd(inp["q_raw"], inp["k_raw"], inp["v_raw"], inp["proj_q"], inp["proj_kv"],
                                        inp["q_norm_w"], inp["k_norm_w"], rope_base=10000.0, k_scale=0.5, eps=1e-6)
    beta, decay = to_f64(inp["beta"]), to_f64(inp["decay"])
    if idx is not None:
        q, k, v, beta, decay = (heads(x, idx) for x in (q, k, v, beta, decay))
        s0 = None if s0 is None else heads(to_f64(s0), idx)
    return oracle.cam_scan_fwd(q, k, v, beta, decay, s0, reverse=reverse, l2norm=l2norm,
                               return_final_state=not reverse)


@pytest.mark.parametrize("reverse", [False, True], ids=["fwd", "rev"])
@pytest.mark.parametrize("B,N,H,F", [(1, 3 * 70, 3, 3), (2, 4 * 130, 2, 4), (1, 5 * 7, 16, 5)])
def test_fused_against_oracle(B, N, H, F, reverse):
    """Frames of 70, 130 and 7 tokens: 64- and 128-token tiles with ragged
    tails inside each frame; up to 16 heads in the raw rows."""
    inp = make(B, N, H, F, seed=N + H)
    o, _ = run_fused(inp, reverse=reverse)
    ro, _ = run_oracle(inp, reverse=reverse)
    assert rel_err(o, ro) <= TOL_BF16


def test_fused_state_passing_and_no_unit_norm():
    inp = make(1, 2 * 96, 2, 2, seed=5)
    s0 = torch.randn(1, 2, 128, 128, generator=torch.Generator().manual_seed(9)) * 0.1
    o, sf = run_fused(inp, l2norm=False, s0=s0, final=True)
    ro, rs = run_oracle(inp, l2norm=False, s0=s0)
    assert rel_err(o, ro) <= TOL_BF16
    assert rel_err(sf, rs) <= TOL_BF16


def test_fused_matches_prep_then_scan():
    """The fused call and the two separate library calls agree within the bf16
    tolerance (the separate path rounds the prepped q, k, v to bf16 in HBM)."""
    inp = make(2, 3 * 200, 4, 3, seed=21)
    o, _ = run_fused(inp)
    d = to_dev(inp)
    q, k, v, _, _ = binding.cam_prep_fwd(d["q_raw"], d["k_raw"], d["v_raw"], d["proj_q"], d["proj_kv"],
                                         d["q_norm_w"], d["k_norm_w"], rope_base=10000.0)
    o2, _ = binding.cam_scan_fwd(q, k, v, d["beta"], d["decay"], l2norm=True)
    torch.cuda.synchronize()
    assert rel_err(o, to_f64(o2)) <= TOL_BF16


def test_camera_workload_full_size_sampled_heads():
    """The camera workload: B2, 21 frames of 30 x 52 tokens, H16, D128, in the
    launch configuration the bench times; sampled heads against the oracle's
    prep and frame scan."""
    B, F, S, H = 2, 21, 30 * 52, 16
    inp = make(B, F * S, H, F, seed=4, weights=False)
    o, _ = run_fused(inp)
    assert torch.isfinite(o).all()
    idx = [0, 21]
    ro, _ = run_oracle(inp, idx=idx)
    assert rel_err(heads(o, idx).cpu(), ro) <= TOL_BF16
