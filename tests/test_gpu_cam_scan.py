"""GPU parity of the frame-level camera scan (fused_cam_gdn.py,
``_cam_scan_kernel``; reverse mode ``_torch_cam_scan_reference``) against the
fp64 oracle, through the C ABI: forward and reverse, tensor-core and CUDA-core
paths, ragged frames, the unit-norm flag, state passing, and the camera
workload's full size on sampled heads.  Metric: max|o - o_ref| / max|o_ref|,
at most 1e-4 for fp32 tensors and 1e-2 for bf16 tensors with the fp32 state."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_47_gb300 import binding
from gated_delta_rule_47_gb300.inputs import cam_scan_inputs, to_f64
from tests.gpu_util import TOL_BF16, TOL_F32, ensure_lib, heads, rel_err, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def run(inp, reverse=False, l2norm=False, scale=1.0, simt=False, final=None):
    d = to_dev(inp)
    final = (not reverse) if final is None else final
    o, sf = binding.cam_scan_fwd(d["q"], d["k"], d["v"], d["beta"], d["decay"],
                                 None if reverse else d.get("initial_state"), output_final_state=final,
                                 scale=scale, reverse=reverse, l2norm=l2norm, simt=simt)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    return o, sf


def ref(inp, reverse=False, l2norm=False, scale=1.0):
    return oracle.cam_scan_fwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["decay"],
                               None if reverse else inp.get("initial_state"), scale=scale, reverse=reverse,
                               l2norm=l2norm, return_final_state=not reverse)


@pytest.mark.parametrize("reverse", [False, True], ids=["fwd", "rev"])
@pytest.mark.parametrize("F,S", [(4, 130), (3, 64), (5, 7), (6, 1), (1, 300)])
def test_tensor_core_path(F, S, reverse):
    """bf16, Dk = Dv = 128: frames of 130 tokens (two 64-token tiles and a
    2-token tail, 128-token output tiles and a 2-token tail), exact tiles,
    frames shorter than a tile, one-token frames, and a single frame."""
    inp = cam_scan_inputs(2, 2, F, S, 128, 128, seed=10 * F + S, dtype="bf16", initial_state=True)
    o, sf = run(inp, reverse=reverse, scale=0.8)
    ro, rs = ref(inp, reverse=reverse, scale=0.8)
    assert rel_err(o, ro) <= TOL_BF16
    if not reverse:
        assert rel_err(sf, rs) <= TOL_BF16
    else:
        assert torch.count_nonzero(o[:, :, -S:]) == 0  # the last frame reads the zero state


@pytest.mark.parametrize("reverse", [False, True], ids=["fwd", "rev"])
@pytest.mark.parametrize("dtype,tol", [("f32", TOL_F32), ("bf16", TOL_BF16)])
@pytest.mark.parametrize("Dk,Dv", [(64, 64), (128, 128), (64, 128), (128, 64)])
def test_cuda_core_path(Dk, Dv, dtype, tol, reverse):
    inp = cam_scan_inputs(1, 2, 4, 37, Dk, Dv, seed=Dk + Dv, dtype=dtype, initial_state=True)
    o, sf = run(inp, reverse=reverse, simt=True)
    ro, rs = ref(inp, reverse=reverse)
    assert rel_err(o, ro) <= tol
    if not reverse:
        assert rel_err(sf, rs) <= tol


@pytest.mark.parametrize("path", ["tc", "simt"])
def test_unit_norm_flag(path):
    inp = cam_scan_inputs(1, 3, 3, 150, 128, 128, seed=31, dtype="bf16", initial_state=True, normalise_qk=False)
    o, sf = run(inp, l2norm=True, simt=path == "simt")
    ro, rs = ref(inp, l2norm=True)
    assert rel_err(o, ro) <= TOL_BF16
    assert rel_err(sf, rs) <= TOL_BF16


def test_split_and_resume():
    inp = cam_scan_inputs(1, 2, 6, 100, 128, 128, seed=41, dtype="bf16", initial_state=True)
    o, sf = run(inp)
    f0, S = 2, 100
    a = {k: (v[:, :, :f0 * S].contiguous() if k in ("q", "k", "v", "beta") else v) for k, v in inp.items()}
    a["decay"] = inp["decay"][..., :f0].contiguous()
    o1, s1 = run(a)
    b = {k: v[:, :, f0 * S:].contiguous() for k, v in inp.items() if k in ("q", "k", "v", "beta")}
    b["decay"] = inp["decay"][..., f0:].contiguous()
    b["initial_state"] = s1.cpu()
    o2, s2 = run(b)
    assert rel_err(torch.cat([o1, o2], dim=2), to_f64(o)) <= 1e-2
    assert rel_err(s2, to_f64(sf)) <= 1e-2


def test_tensor_core_and_cuda_core_paths_agree():
    inp = cam_scan_inputs(2, 2, 3, 200, 128, 128, seed=51, dtype="bf16", initial_state=True)
    o1, s1 = run(inp)
    o2, s2 = run(inp, simt=True)
    assert rel_err(o1, to_f64(o2)) <= TOL_BF16
    assert rel_err(s1, to_f64(s2)) <= TOL_BF16


def test_camera_workload_shape_sampled_heads():
    """The camera workload's shape: B2 H16, 21 frames of 30 x 52 = 1560 tokens,
    D128, bf16, in the launch configuration the bench times; checked on
    sampled heads against the oracle, both directions."""
    B, H, F, S = 2, 16, 21, 1560
    inp = cam_scan_inputs(B, H, F, S, 128, 128, seed=4, dtype="bf16")
    idx = [0, 17, 31]
    sub = {k: heads(v, idx) for k, v in inp.items()}
    for reverse in (False, True):
        o, _ = run(inp, reverse=reverse, final=False)
        assert torch.isfinite(o).all()
        ro, _ = ref(sub, reverse=reverse)
        assert rel_err(heads(o, idx).cpu(), ro) <= TOL_BF16


def test_no_frames_pass_the_state_through():
    """F = 0 through the C entry point: nothing is launched, and the final
    state receives the initial state."""
    import ctypes
    s0 = torch.randn(1, 2, 64, 64, device="cuda")
    sf = torch.full_like(s0, 7.0)
    lib = binding.load()
    st = lib.cam_scan_fwd(None, None, None, None, None, ctypes.c_void_p(s0.data_ptr()), None,
                          ctypes.c_void_p(sf.data_ptr()), 1, 2, 0, 5, 64, 64, 1.0, 0, binding.GDN_F32, None, 0,
                          ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert st == 0
    assert torch.equal(sf, s0)
