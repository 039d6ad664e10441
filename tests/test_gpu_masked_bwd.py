"""GPU parity of the block-masked DeltaProduct backward (gated_deltaproduct
test.py: `gated_chunk_delta_rule_bwd_kernel_dhu`,
`gated_chunk_delta_rule_bwd_kernel_dqkw`, `gated_bwd_prepare_wy_repr_kernel`,
for the mask_ij variant) against the fp64 oracle backward, itself pinned by
finite differences of the forward oracle, through the C ABI.  Metric:
max|g - g_ref| / max|g_ref| per gradient, at most 1e-4 with fp32 tensors and
1e-2 with bf16 tensors."""
import pytest
import torch

import oracle
from gated_delta_rule_47_gb300 import binding
from gated_delta_rule_47_gb300.inputs import WORKLOADS, gdn_inputs, slice_mask
from tests.gpu_util import TOL_BF16, TOL_F32, ensure_lib, heads, rel_err, to_dev

pytestmark = pytest.mark.gpu

NAMES = ("dq", "dk", "dv", "dbeta", "dg", "ds0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def case(T, D, r, dtype, l2norm, seed, general_mask=False):
    inp = gdn_inputs(1, 2, T, D, D, seed=seed, dtype=dtype, initial_state=True, normalise_qk=not l2norm)
    if general_mask:
        g = torch.Generator().manual_seed(seed)
        inp["mask"] = (torch.randn(r, r, generator=g) * 0.5).contiguous()
    else:
        inp["mask"] = slice_mask(r, seed=r)
    gen = torch.Generator().manual_seed(seed + 1)
    do = torch.randn(1, 2, T, D, generator=gen).to(inp["q"].dtype)
    dsf = torch.randn(1, 2, D, D, generator=gen)
    return inp, do, dsf


@pytest.mark.parametrize("dtype,tol", [("f32", TOL_F32), ("bf16", TOL_BF16)])
@pytest.mark.parametrize("r,T,D", [(2, 77, 128), (4, 50, 64), (8, 30, 128), (1, 70, 64)])
def test_masked_backward(r, T, D, dtype, tol):
    inp, do, dsf = case(T, D, r, dtype, False, seed=r * 7 + T)
    d = to_dev(inp)
    got = binding.masked_deltaproduct_chunk_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["mask"], do.cuda(),
                                                d["initial_state"], dsf.cuda(), scale=0.8, need_dinitial=True)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    ref = oracle.masked_deltaproduct_bwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"], inp["mask"], do,
                                         inp["initial_state"], dsf, scale=0.8)
    for name, x, y in zip(NAMES, got, ref):
        assert rel_err(x, y) <= tol, name


def test_general_mask_and_unit_norm():
    """A mask that is not a correlation matrix, with unnormalised keys under the unit-norm flag."""
    inp, do, dsf = case(90, 128, 4, "f32", True, seed=5, general_mask=True)
    d = to_dev(inp)
    got = binding.masked_deltaproduct_chunk_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["mask"], do.cuda(),
                                                d["initial_state"], dsf.cuda(), l2norm=True, need_dinitial=True)
    torch.cuda.synchronize()
    ref = oracle.masked_deltaproduct_bwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"], inp["mask"], do,
                                         inp["initial_state"], dsf, l2norm=True)
    for name, x, y in zip(NAMES, got, ref):
        assert rel_err(x, y) <= TOL_F32, name


def test_all_ones_mask_matches_the_gdn_backward():
    """An all-ones mask is GDN: the masked backward and the chunk GDN backward agree."""
    inp, do, dsf = case(100, 128, 2, "f32", False, seed=9)
    inp["mask"] = torch.ones(2, 2)
    d = to_dev(inp)
    a = binding.masked_deltaproduct_chunk_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["mask"], do.cuda(),
                                              d["initial_state"], dsf.cuda(), need_dinitial=True)
    b = binding.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], do.cuda(), d["initial_state"], dsf.cuda(),
                              need_dinitial=True)
    torch.cuda.synchronize()
    for name, x, y in zip(NAMES, a, b):
        assert rel_err(x, y.double().cpu().numpy()) <= TOL_F32, name


def test_full_size_sampled_heads():
    """The block-masked workload (B4 H16 T4096 D128 bf16, r = 2): every head on
    the GPU, two heads against the oracle."""
    w = WORKLOADS["masked_dp_r2_b4h16t4096d128_bf16"]
    inp = w.make()
    do = torch.randn(w.B, w.H, w.T, w.D, generator=torch.Generator().manual_seed(4)).to(torch.bfloat16)
    d = to_dev(inp)
    got = binding.masked_deltaproduct_chunk_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["mask"], do.cuda())
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    idx = [1, 50]
    sub = {k: (heads(v, idx) if k != "mask" else v) for k, v in inp.items()}
    ref = oracle.masked_deltaproduct_bwd(sub["q"], sub["k"], sub["v"], sub["beta"], sub["g"], sub["mask"],
                                         heads(do, idx))
    for name, x, y in zip(NAMES[:5], got[:5], ref[:5]):
        assert rel_err(heads(x, idx).cpu(), y) <= TOL_BF16, name


@pytest.mark.parametrize("r,T", [(2, 100), (4, 40)])
def test_tensor_core_chain_matches_the_cuda_core_chain(r, T):
    """bf16 at D = 128 runs the chains on tcgen05 (bf16 hi / lo split
    products); the fp32 CUDA-core chains agree to within one rounding of the
    bf16 gradients and ~2e-4 on the fp32 ones."""
    inp, do, dsf = case(T, 128, r, "bf16", True, seed=60 + r, general_mask=True)
    d = to_dev(inp)

    def run(simt):
        return binding.masked_deltaproduct_chunk_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["mask"], do.cuda(),
                                                     d["initial_state"], dsf.cuda(), l2norm=True, need_dinitial=True,
                                                     simt=simt)

    tc, simt = run(False), run(True)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    for name, x, y in zip(NAMES, tc, simt):
        tol = 5e-3 if x.dtype == torch.bfloat16 else 2e-4
        assert rel_err(x, y.double().cpu().numpy()) <= tol, name


@pytest.mark.parametrize("r", [2, 4, 8])
def test_tensor_core_wy_general_mask_unit_norm(r):
    """bf16 at D = 128 forms the WY factors, T, K K^T, P and the state-gradient
    term B on tcgen05: a general real mask, unnormalised keys under the
    unit-norm flag and a ragged tail, against the oracle."""
    inp, do, dsf = case(150, 128, r, "bf16", True, seed=40 + r, general_mask=True)
    d = to_dev(inp)
    got = binding.masked_deltaproduct_chunk_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["mask"], do.cuda(),
                                                d["initial_state"], dsf.cuda(), scale=0.7, l2norm=True,
                                                need_dinitial=True)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    ref = oracle.masked_deltaproduct_bwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"], inp["mask"], do,
                                         inp["initial_state"], dsf, scale=0.7, l2norm=True)
    for name, x, y in zip(NAMES, got, ref):
        assert rel_err(x, y) <= TOL_BF16, name


def test_tensor_core_path_is_deterministic():
    """Two runs of the bf16 backward over 512 chunks give the same bits."""
    inp, do, dsf = case(2048, 128, 2, "bf16", False, seed=61)
    inp = {k: (v.repeat(1, 4, *([1] * (v.dim() - 2))) if k != "mask" else v) for k, v in inp.items()}
    d = to_dev(inp)
    do = do.repeat(1, 4, 1, 1).cuda()
    dsf = dsf.repeat(1, 4, 1, 1).cuda()
    outs = []
    for _ in range(2):
        outs.append(binding.masked_deltaproduct_chunk_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["mask"], do,
                                                          d["initial_state"], dsf, need_dinitial=True))
    torch.cuda.synchronize()
    for x, y in zip(*outs):
        assert torch.equal(x, y)


def test_tensor_core_path_strong_decay():
    """Log-decays near -2 per token on the block-masked backward (bf16, D 128,
    r = 2): every decay factor of the tensor-core kernels is formed per element."""
    inp, do, dsf = case(120, 128, 2, "bf16", False, seed=71)
    inp["g"] = (torch.nn.functional.logsigmoid(torch.randn(1, 2, 120, generator=torch.Generator().manual_seed(72))
                                               - 2.0)).float()
    d = to_dev(inp)
    got = binding.masked_deltaproduct_chunk_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["mask"], do.cuda(),
                                                d["initial_state"], dsf.cuda(), need_dinitial=True)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    ref = oracle.masked_deltaproduct_bwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"], inp["mask"], do,
                                         inp["initial_state"], dsf)
    for name, x, y in zip(NAMES, got, ref):
        assert torch.isfinite(x).all(), name
        assert rel_err(x, y) <= TOL_BF16, name


@pytest.mark.parametrize("r,T", [(1, 70), (2, 1), (2, 33), (8, 9)])
def test_tensor_core_path_small_and_ragged(r, T):
    """The tensor-core backward (bf16, D 128) at r = 1 (one sub-row per token),
    with a single token, one chunk plus a token, and r = 8 (eight tokens per
    chunk, so the query rows round up to 16 inside the products)."""
    inp, do, dsf = case(T, 128, r, "bf16", False, seed=200 + 10 * r + T)
    d = to_dev(inp)
    got = binding.masked_deltaproduct_chunk_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["mask"], do.cuda(),
                                                d["initial_state"], dsf.cuda(), scale=0.9, need_dinitial=True)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    ref = oracle.masked_deltaproduct_bwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"], inp["mask"], do,
                                         inp["initial_state"], dsf, scale=0.9)
    for name, x, y in zip(NAMES, got, ref):
        assert rel_err(x, y) <= TOL_BF16, name
