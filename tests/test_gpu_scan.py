"""GPU parity of the chunkwise GDN / DeltaProduct forward against the fp64
oracle, through the C ABI.  Metric: max|o - o_ref| / max|o_ref|, at most 1e-4
for fp32 tensors and 1e-2 for bf16 tensors with the fp32 state."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_47_gb300 import binding
from gated_delta_rule_47_gb300.inputs import WORKLOADS, gdn_inputs, to_f64
from tests.gpu_util import TOL_BF16, TOL_F32, ensure_lib, heads, rel_err, sample_heads, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def run_gdn(inp, chunk=64, l2norm=False, scale=1.0, final=True):
    d = to_dev(inp)
    o, sf = binding.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d.get("initial_state"),
                                  output_final_state=final, chunk=chunk, scale=scale, l2norm=l2norm)
    torch.cuda.synchronize()
    return o, sf


def ref_gdn(inp, l2norm=False, scale=1.0):
    return oracle.gdn_fwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"], inp.get("initial_state"),
                          scale=scale, l2norm=l2norm)


def test_tiny_fp32_workload():
    w = WORKLOADS["gdn_tiny_f32"]
    inp = w.make()
    o, sf = run_gdn(inp, chunk=w.chunk)
    ro, rs = ref_gdn(inp)
    assert rel_err(o, ro) <= TOL_F32
    assert rel_err(sf, rs) <= TOL_F32


@pytest.mark.parametrize("dtype,tol", [("f32", TOL_F32), ("bf16", TOL_BF16)])
@pytest.mark.parametrize("chunk", [16, 32, 64])
@pytest.mark.parametrize("Dk,Dv", [(64, 64), (128, 128), (64, 128), (128, 64)])
def test_ragged_tail_and_chunk_sizes(dtype, tol, chunk, Dk, Dv):
    inp = gdn_inputs(2, 2, 203, Dk, Dv, seed=chunk + Dk + Dv, dtype=dtype, initial_state=True)
    o, sf = run_gdn(inp, chunk=chunk, scale=0.75)
    ro, rs = ref_gdn(inp, scale=0.75)
    assert rel_err(o, ro) <= tol
    assert rel_err(sf, rs) <= tol


@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 130])
def test_short_sequences(T):
    inp = gdn_inputs(1, 3, T, 128, 128, seed=T, dtype="bf16", initial_state=True)
    o, sf = run_gdn(inp)
    ro, rs = ref_gdn(inp)
    assert rel_err(o, ro) <= TOL_BF16
    assert rel_err(sf, rs) <= TOL_BF16


def test_empty_sequence_passes_state_through():
    inp = gdn_inputs(1, 2, 0, 64, 64, seed=1, dtype="f32", initial_state=True)
    o, sf = run_gdn(inp)
    assert o.shape == (1, 2, 0, 64)
    assert torch.equal(sf.cpu(), inp["initial_state"])
    inp.pop("initial_state")
    _, sf0 = run_gdn(inp)
    assert torch.count_nonzero(sf0) == 0


def test_split_and_resume_on_gpu():
    inp = gdn_inputs(1, 2, 300, 128, 128, seed=7, dtype="f32", initial_state=True)
    o, sf = run_gdn(inp)
    t0 = 128
    a = {k: (v[:, :, :t0].contiguous() if k in ("q", "k", "v", "beta", "g") else v) for k, v in inp.items()}
    o1, s1 = run_gdn(a)
    b = {k: v[:, :, t0:].contiguous() for k, v in inp.items() if k in ("q", "k", "v", "beta", "g")}
    b["initial_state"] = s1.cpu()
    o2, s2 = run_gdn(b)
    assert rel_err(torch.cat([o1, o2], dim=2), to_f64(o)) <= 1e-5
    assert rel_err(s2, to_f64(sf)) <= 1e-5


def test_l2norm_flag():
    inp = gdn_inputs(1, 2, 150, 128, 128, seed=9, dtype="bf16", normalise_qk=False)
    o, _ = run_gdn(inp, l2norm=True)
    ro, _ = ref_gdn(inp, l2norm=True)
    assert rel_err(o, ro) <= TOL_BF16


@pytest.mark.parametrize("dtype,tol", [("f32", TOL_F32), ("bf16", TOL_BF16)])
@pytest.mark.parametrize("r,chunk", [(2, 64), (3, 64), (3, 16), (4, 32)])
def test_deltaproduct_small(dtype, tol, r, chunk):
    inp = gdn_inputs(2, 2, 77, 128, 128, seed=r, dtype=dtype, r=r, initial_state=True)
    d = to_dev(inp)
    o, sf = binding.deltaproduct_chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["initial_state"],
                                           output_final_state=True, chunk=chunk)
    ro, rs = oracle.deltaproduct_fwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"],
                                     inp["initial_state"])
    assert rel_err(o, ro) <= tol
    assert rel_err(sf, rs) <= tol


def test_deltaproduct_r1_is_gdn():
    inp = gdn_inputs(1, 2, 100, 128, 128, seed=11, dtype="bf16")
    d = to_dev(inp)
    o1, _ = binding.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"])
    o2, _ = binding.deltaproduct_chunk_fwd(d["q"], d["k"][:, :, :, None].contiguous(),
                                           d["v"][:, :, :, None].contiguous(),
                                           d["beta"][..., None].contiguous(), d["g"])
    assert torch.equal(o1, o2)


# --- full-size workloads in the launch configuration the bench times, checked on
# --- sampled heads that the oracle recomputes from the same inputs.

@pytest.mark.parametrize("name", ["gdn_b4h16t4096d128_bf16", "gdn_long_b1h32t32768d128_bf16"])
def test_full_size_gdn_sampled_heads(name):
    w = WORKLOADS[name]
    inp = w.make()
    o, _ = run_gdn(inp, chunk=w.chunk, final=False)
    idx = sample_heads(w.B, w.H, 3 if w.T <= 4096 else 2, seed=w.seed)
    sub = {k: heads(v, idx) for k, v in inp.items()}
    ro, _ = ref_gdn(sub)
    assert rel_err(heads(o, idx).cpu(), ro) <= TOL_BF16
    assert torch.isfinite(o).all()


def test_full_size_deltaproduct_sampled_heads():
    w = WORKLOADS["deltaproduct_r2_b4h16t4096d128_bf16"]
    inp = w.make()
    d = to_dev(inp)
    o, _ = binding.deltaproduct_chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], chunk=w.chunk)
    torch.cuda.synchronize()
    idx = sample_heads(w.B, w.H, 3, seed=w.seed)
    sub = {k: heads(v, idx) for k, v in inp.items()}
    ro, _ = oracle.deltaproduct_fwd(sub["q"], sub["k"], sub["v"], sub["beta"], sub["g"])
    assert rel_err(heads(o, idx).cpu(), ro) <= TOL_BF16
    assert torch.isfinite(o).all()


# --- the tensor-core path (bf16, Dk = Dv = 128, chunk 64, r in {1,2,4}) against
# --- the oracle and against the CUDA-core path on the same inputs.

@pytest.mark.parametrize("T", [64, 300, 1000])
def test_tensor_core_and_cuda_core_paths_agree(T):
    inp = gdn_inputs(2, 3, T, 128, 128, seed=T + 5, dtype="bf16", initial_state=True)
    d = to_dev(inp)
    args = (d["q"], d["k"], d["v"], d["beta"], d["g"], d["initial_state"])
    o_tc, s_tc = binding.gdn_chunk_fwd(*args, output_final_state=True)
    o_sm, s_sm = binding.gdn_chunk_fwd(*args, output_final_state=True, simt=True)
    torch.cuda.synchronize()
    ro, rs = ref_gdn(inp)
    assert rel_err(o_tc, ro) <= TOL_BF16 and rel_err(s_tc, rs) <= TOL_BF16
    assert rel_err(o_sm, ro) <= TOL_BF16 and rel_err(s_sm, rs) <= TOL_BF16
    assert binding.device_error() == 0


@pytest.mark.parametrize("r", [2, 4])
def test_tensor_core_deltaproduct(r):
    inp = gdn_inputs(1, 2, 150, 128, 128, seed=40 + r, dtype="bf16", r=r, initial_state=True)
    d = to_dev(inp)
    o, sf = binding.deltaproduct_chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["initial_state"],
                                           output_final_state=True, chunk=64)
    ro, rs = oracle.deltaproduct_fwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"],
                                     inp["initial_state"])
    assert rel_err(o, ro) <= TOL_BF16
    assert rel_err(sf, rs) <= TOL_BF16


@pytest.mark.parametrize("hc,nwy", [(1, 1), (1, 2), (1, 3), (2, 1), (2, 3), (3, 2), (4, 1), (4, 5)])
def test_tensor_core_cluster_shapes(hc, nwy):
    """Every cluster shape gives the oracle's results: hc scan CTAs share the
    WY pipelines of nwy CTAs, which take the cluster's (head, chunk) items in
    turn. Six heads leave the last cluster of hc = 4 half empty, and T = 300
    gives five chunks per head with a ragged last one."""
    inp = gdn_inputs(2, 3, 300, 128, 128, seed=90 + 10 * hc + nwy, dtype="bf16", initial_state=True)
    d = to_dev(inp)
    try:
        binding.set_cluster_shape(hc, nwy)
        o, sf = binding.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["initial_state"],
                                      output_final_state=True)
        torch.cuda.synchronize()
    finally:
        binding.set_cluster_shape(0, 0)
    assert binding.device_error() == 0
    ro, rs = ref_gdn(inp)
    assert rel_err(o, ro) <= TOL_BF16
    assert rel_err(sf, rs) <= TOL_BF16


@pytest.mark.parametrize("B,H,T", [(1, 1, 200), (1, 1, 64), (3, 1, 130)])
def test_tensor_core_few_heads_automatic_shape(B, H, T):
    """One to three heads (ring mode, with many more WY pipelines than heads,
    most of them without items); results are unaffected."""
    inp = gdn_inputs(B, H, T, 128, 128, seed=B * 7 + T, dtype="bf16", initial_state=True)
    o, sf = run_gdn(inp)
    assert binding.device_error() == 0
    ro, rs = ref_gdn(inp)
    assert rel_err(o, ro) <= TOL_BF16
    assert rel_err(sf, rs) <= TOL_BF16


@pytest.mark.parametrize("hc,nwy", [(1, 2), (4, 5)])
def test_tensor_core_deltaproduct_cluster_shapes(hc, nwy):
    inp = gdn_inputs(1, 5, 150, 128, 128, seed=60 + hc, dtype="bf16", r=2, initial_state=True)
    d = to_dev(inp)
    try:
        binding.set_cluster_shape(hc, nwy)
        o, sf = binding.deltaproduct_chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["initial_state"],
                                               output_final_state=True, chunk=64)
        torch.cuda.synchronize()
    finally:
        binding.set_cluster_shape(0, 0)
    assert binding.device_error() == 0
    ro, rs = oracle.deltaproduct_fwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"], inp["initial_state"])
    assert rel_err(o, ro) <= TOL_BF16
    assert rel_err(sf, rs) <= TOL_BF16


def test_tensor_core_l2norm_and_scale():
    inp = gdn_inputs(1, 2, 200, 128, 128, seed=77, dtype="bf16", normalise_qk=False, initial_state=True)
    o, sf = run_gdn(inp, l2norm=True, scale=0.5)
    ro, rs = ref_gdn(inp, l2norm=True, scale=0.5)
    assert rel_err(o, ro) <= TOL_BF16
    assert rel_err(sf, rs) <= TOL_BF16


@pytest.mark.parametrize("shape", [(0, 0), (1, 1)])
def test_bounded_wait_gives_up_and_context_survives(shape):
    """A 1-microsecond wait limit makes the kernel's first wait run out (ring
    mode, and a forced cluster shape): the call reports GDN_ERR_TIMEOUT through
    the device error word, and with the default limit restored the next call
    is correct."""
    inp = gdn_inputs(1, 2, 1024, 128, 128, seed=3, dtype="bf16")
    d = to_dev(inp)
    assert binding.device_error() == 0
    try:
        binding.set_cluster_shape(*shape)
        binding.set_wait_limit(1)
        binding.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"])
        assert binding.device_error() == 6
    finally:
        binding.set_wait_limit(0)
        binding.set_cluster_shape(0, 0)
    assert binding.device_error() == 0
    o, _ = binding.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"])
    torch.cuda.synchronize()
    ro, _ = ref_gdn(inp)
    assert rel_err(o, ro) <= TOL_BF16


# --- ring mode: one cooperative grid, WY results through per-head rings of 8
# --- slots in the workspace (the default for up to min(80, SMs / 2) heads).

def test_ring_and_cluster_modes_agree():
    """T = 700 gives 11 chunks per head, so every ring wraps and its slots are
    refilled only after the scan has taken them out."""
    inp = gdn_inputs(2, 5, 700, 128, 128, seed=123, dtype="bf16", initial_state=True)
    d = to_dev(inp)
    args = (d["q"], d["k"], d["v"], d["beta"], d["g"], d["initial_state"])
    assert binding.workspace_bytes(2, 5, 700, 128, 128) > 0
    o_ring, s_ring = binding.gdn_chunk_fwd(*args, output_final_state=True)
    try:
        binding.set_cluster_shape(2, 2)
        o_cl, s_cl = binding.gdn_chunk_fwd(*args, output_final_state=True)
        torch.cuda.synchronize()
    finally:
        binding.set_cluster_shape(0, 0)
    assert binding.device_error() == 0
    ro, rs = ref_gdn(inp)
    for o, sf in ((o_ring, s_ring), (o_cl, s_cl)):
        assert rel_err(o, ro) <= TOL_BF16
        assert rel_err(sf, rs) <= TOL_BF16


def test_ring_workspace_with_stale_contents():
    """The ring's tags carry the launch that wrote them: a workspace full of
    random bytes, then one already used by a call on other inputs, both give
    the right results."""
    B, H, T = 1, 4, 600
    ws = torch.randint(0, 256, (binding.workspace_bytes(B, H, T, 128, 128),), dtype=torch.uint8, device="cuda")
    for seed in (7, 8):
        inp = gdn_inputs(B, H, T, 128, 128, seed=seed, dtype="bf16")
        d = to_dev(inp)
        o, _ = binding.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], workspace=ws)
        torch.cuda.synchronize()
        assert binding.device_error() == 0
        ro, _ = ref_gdn(inp)
        assert rel_err(o, ro) <= TOL_BF16


def test_misaligned_workspace_runs_without_the_ring():
    B, H, T = 1, 2, 300
    n = binding.workspace_bytes(B, H, T, 128, 128)
    buf = torch.empty(n + 16, dtype=torch.uint8, device="cuda")
    inp = gdn_inputs(B, H, T, 128, 128, seed=9, dtype="bf16")
    d = to_dev(inp)
    o, _ = binding.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], workspace=buf[8:8 + n])
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    ro, _ = ref_gdn(inp)
    assert rel_err(o, ro) <= TOL_BF16


def test_ring_mode_head_limit():
    """The most heads ring mode takes on this device, and one more (which goes
    to the cluster mode and needs no workspace)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    most = min(80, sms // 2)
    for BH in (most, most + 1):
        inp = gdn_inputs(1, BH, 100, 128, 128, seed=BH, dtype="bf16", initial_state=True)
        assert (binding.workspace_bytes(1, BH, 100, 128, 128) > 0) == (BH == most)
        o, sf = run_gdn(inp)
        assert binding.device_error() == 0
        ro, rs = ref_gdn(inp)
        assert rel_err(o, ro) <= TOL_BF16
        assert rel_err(sf, rs) <= TOL_BF16


def test_graph_replays_reuse_one_workspace():
    """A call captured in a CUDA graph replays with the ring epoch it was
    captured with.  Every launch that completes zeroes its ring's tags, so
    replays back to back on the same workspace match the eager call bit for
    bit, and so does an eager call on that workspace afterwards."""
    B, H, T = 2, 8, 700
    inp = gdn_inputs(B, H, T, 128, 128, seed=321, dtype="bf16", initial_state=True)
    d = to_dev(inp)
    ws = torch.empty(binding.workspace_bytes(B, H, T, 128, 128), dtype=torch.uint8, device="cuda")
    args = (d["q"], d["k"], d["v"], d["beta"], d["g"], d["initial_state"])
    o_eager, s_eager = binding.gdn_chunk_fwd(*args, output_final_state=True, workspace=ws)
    torch.cuda.synchronize()
    o = torch.empty_like(o_eager)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, capture_error_mode="thread_local"):
        binding.gdn_chunk_fwd(*args, o=o, workspace=ws)
    for _ in range(3):
        o.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert binding.device_error() == 0
        assert torch.equal(o, o_eager)
    o2, s2 = binding.gdn_chunk_fwd(*args, output_final_state=True, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(o2, o_eager) and torch.equal(s2, s_eager)
    ro, _ = ref_gdn(inp)
    assert rel_err(o_eager, ro) <= TOL_BF16


def test_full_size_fp32_sampled_heads():
    """The fp32 path at the headline's size (B4 H16 T4096 D128, 64 chunks per
    head, CUDA cores): sampled heads against the oracle at the fp32 bound."""
    inp = gdn_inputs(4, 16, 4096, 128, 128, seed=31, dtype="f32", initial_state=True)
    d = to_dev(inp)
    o, sf = binding.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["initial_state"],
                                  output_final_state=True)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    idx = sample_heads(4, 16, 2, seed=31)
    sub = {k: heads(v, idx) for k, v in inp.items()}
    ro, rs = oracle.gdn_fwd(sub["q"], sub["k"], sub["v"], sub["beta"], sub["g"], sub["initial_state"])
    assert rel_err(heads(o, idx).cpu(), ro) <= TOL_F32
    assert rel_err(heads(sf, idx).cpu(), rs) <= TOL_F32
