"""GPU parity of the block-masked DeltaProduct (gated_deltaproduct test.py,
the mask_ij variant) against the fp64 oracle, through the C ABI.  Metric:
max|o - o_ref| / max|o_ref|, at most 1e-4 for fp32 tensors and 1e-2 for bf16
tensors with the fp32 state."""
import pytest
import torch

import oracle
from gated_delta_rule_47_gb300 import binding
from gated_delta_rule_47_gb300.inputs import WORKLOADS, gdn_inputs, slice_mask
from tests.gpu_util import TOL_BF16, TOL_F32, ensure_lib, heads, rel_err, sample_heads, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def run(inp, chunk=64, l2norm=False, scale=1.0):
    d = to_dev(inp)
    o, sf = binding.masked_deltaproduct_chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["mask"],
                                                  d.get("initial_state"), output_final_state=True, chunk=chunk,
                                                  scale=scale, l2norm=l2norm)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    return o, sf


def ref(inp, l2norm=False, scale=1.0):
    return oracle.masked_deltaproduct_fwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"], inp["mask"],
                                          inp.get("initial_state"), scale=scale, l2norm=l2norm)


@pytest.mark.parametrize("dtype,tol", [("f32", TOL_F32), ("bf16", TOL_BF16)])
@pytest.mark.parametrize("r,chunk", [(2, 64), (2, 16), (4, 32), (8, 64), (1, 32)])
@pytest.mark.parametrize("D", [64, 128])
def test_against_oracle(dtype, tol, r, chunk, D):
    """77 tokens: several chunks and a ragged tail for every chunk size."""
    inp = gdn_inputs(2, 2, 77, D, D, seed=r * 10 + chunk + D, dtype=dtype, initial_state=True)
    inp["mask"] = slice_mask(r, seed=r)
    o, sf = run(inp, chunk=chunk, scale=0.7)
    ro, rs = ref(inp, scale=0.7)
    assert rel_err(o, ro) <= tol
    assert rel_err(sf, rs) <= tol


def test_general_mask_and_unit_norm_flag():
    """A mask that is not a correlation matrix (any real entries), with the
    unit-norm flag on unnormalised keys."""
    inp = gdn_inputs(1, 3, 90, 128, 128, seed=7, dtype="f32", initial_state=True, normalise_qk=False)
    g = torch.Generator().manual_seed(3)
    inp["mask"] = (torch.randn(4, 4, generator=g) * 0.5).contiguous()
    o, sf = run(inp, chunk=32, l2norm=True)
    ro, rs = ref(inp, l2norm=True)
    assert rel_err(o, ro) <= TOL_F32
    assert rel_err(sf, rs) <= TOL_F32


def test_all_ones_mask_is_gdn():
    inp = gdn_inputs(1, 2, 130, 128, 128, seed=8, dtype="f32", initial_state=True)
    inp["mask"] = torch.ones(2, 2)
    o, sf = run(inp)
    ro, rs = oracle.gdn_fwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"], inp["initial_state"])
    assert rel_err(o, ro) <= TOL_F32
    assert rel_err(sf, rs) <= TOL_F32


def test_full_size_workload_sampled_heads():
    w = WORKLOADS["masked_dp_r2_b4h16t4096d128_bf16"]
    inp = w.make()
    d = to_dev(inp)
    o, _ = binding.masked_deltaproduct_chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["mask"],
                                                 chunk=w.chunk)
    torch.cuda.synchronize()
    assert torch.isfinite(o).all()
    idx = sample_heads(w.B, w.H, 2, seed=w.seed)
    sub = {k: (heads(v, idx) if k != "mask" else v) for k, v in inp.items()}
    ro, _ = oracle.masked_deltaproduct_fwd(sub["q"], sub["k"], sub["v"], sub["beta"], sub["g"], sub["mask"])
    assert rel_err(heads(o, idx).cpu(), ro) <= TOL_BF16


@pytest.mark.parametrize("r", [2, 4])
def test_tensor_core_chain_matches_the_cuda_core_chain(r):
    """bf16 at D = 128 runs the state chain on tcgen05 (bf16 hi / lo split
    products, fp32 state in tensor memory); the fp32 CUDA-core chain gives the
    same output to within one bf16 rounding and the same final state to ~2e-4."""
    inp = gdn_inputs(1, 3, 150, 128, 128, seed=70 + r, dtype="bf16", initial_state=True, normalise_qk=False)
    g = torch.Generator().manual_seed(r)
    inp["mask"] = (torch.randn(r, r, generator=g) * 0.5).contiguous()
    d = to_dev(inp)
    outs = []
    for simt in (False, True):
        outs.append(binding.masked_deltaproduct_chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["mask"],
                                                          d["initial_state"], output_final_state=True, l2norm=True,
                                                          simt=simt))
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    (o1, s1), (o2, s2) = outs
    assert rel_err(o1, o2.double().cpu().numpy()) <= 5e-3
    assert rel_err(s1, s2.double().cpu().numpy()) <= 2e-4


@pytest.mark.parametrize("T", [1, 32, 33])
def test_tensor_core_chain_single_chunk(T):
    """The block-masked forward's tensor-core chain (bf16, D 128, r = 2: 32
    tokens per chunk) over one chunk and one chunk plus a token."""
    inp = gdn_inputs(1, 2, T, 128, 128, seed=90 + T, dtype="bf16", initial_state=True)
    inp["mask"] = slice_mask(2, seed=2)
    o, sf = run(inp)
    ro, rs = ref(inp)
    assert rel_err(o, ro) <= TOL_BF16
    assert rel_err(sf, rs) <= TOL_BF16


@pytest.mark.parametrize("r", [2, 4, 8])
def test_tensor_core_kernels_general_mask_unit_norm(r):
    """bf16 at D = 128 runs the chunk-local kernels on tcgen05 as well (exact
    bf16 key / query products, split products for W, U and the output): a
    general real mask, unnormalised keys with the unit-norm flag, a ragged
    tail, against the oracle."""
    inp = gdn_inputs(1, 2, 200, 128, 128, seed=110 + r, dtype="bf16", initial_state=True, normalise_qk=False)
    g = torch.Generator().manual_seed(20 + r)
    inp["mask"] = (torch.randn(r, r, generator=g) * 0.5).contiguous()
    o, sf = run(inp, l2norm=True, scale=0.6)
    ro, rs = ref(inp, l2norm=True, scale=0.6)
    assert rel_err(o, ro) <= TOL_BF16
    assert rel_err(sf, rs) <= TOL_BF16


@pytest.mark.parametrize("r", [2, 4])
def test_tensor_core_kernels_strong_decay(r):
    """Log-decays near -2 per token (over 60 nats per chunk): the decay
    factors of A, P, W and Kd are formed per element, so nothing overflows."""
    inp = gdn_inputs(1, 2, 140, 128, 128, seed=130 + r, dtype="bf16", g_mu=-2.0, g_div=1.0, initial_state=True)
    inp["mask"] = slice_mask(r, seed=r)
    o, sf = run(inp)
    ro, rs = ref(inp)
    assert torch.isfinite(o).all() and torch.isfinite(sf).all()
    assert rel_err(o, ro) <= TOL_BF16
    assert rel_err(sf, rs) <= TOL_BF16


def test_tensor_core_path_is_deterministic():
    """Two CTAs of the WY kernel share each SM and every kernel of the path
    stages through shared memory: two runs over 2048 chunks give the same
    bits (a race between a CTA's phases would show up as differences in a few
    chunks)."""
    inp = gdn_inputs(1, 16, 4096, 128, 128, seed=150, dtype="bf16", initial_state=True)
    inp["mask"] = slice_mask(2, seed=2)
    o1, s1 = run(inp)
    o2, s2 = run(inp)
    assert torch.equal(o1, o2) and torch.equal(s1, s2)


@pytest.mark.parametrize("r,T", [(1, 1), (4, 17), (8, 8), (8, 9)])
def test_tensor_core_kernels_small_and_ragged(r, T):
    """The tensor-core forward kernels (bf16, D 128) on a single token, a
    ragged first chunk and one chunk exactly, at r = 1, 4 and 8."""
    inp = gdn_inputs(1, 2, T, 128, 128, seed=300 + 10 * r + T, dtype="bf16", initial_state=True)
    inp["mask"] = slice_mask(r, seed=r)
    o, sf = run(inp, scale=0.8)
    ro, rs = ref(inp, scale=0.8)
    assert rel_err(o, ro) <= TOL_BF16
    assert rel_err(sf, rs) <= TOL_BF16
