"""GPU parity of the chunkwise GDN / DeltaProduct backward (gated_deltaproduct
test.py: `gated_chunk_delta_rule_bwd_kernel_dhu`,
`gated_chunk_delta_rule_bwd_kernel_dqkw`, `gated_bwd_prepare_wy_repr_kernel`)
against the fp64 oracle backward, itself pinned by finite differences of the
forward oracle, through the C ABI.  Metric: max|g - g_ref| / max|g_ref| per
gradient, at most 1e-4 with fp32 tensors and 1e-2 with bf16 tensors."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_47_gb300 import binding
from gated_delta_rule_47_gb300.inputs import gdn_inputs
from tests.gpu_util import TOL_BF16, TOL_F32, ensure_lib, heads, rel_err, to_dev

pytestmark = pytest.mark.gpu

NAMES = ("dq", "dk", "dv", "dbeta", "dg", "ds0")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def grads_case(B, H, T, Dk, Dv, dtype, l2norm, r=None, seed=0, state=True):
    inp = gdn_inputs(B, H, T, Dk, Dv, seed=seed, dtype=dtype, r=r, initial_state=state, normalise_qk=not l2norm)
    gen = torch.Generator().manual_seed(seed + 1)
    do = torch.randn(B, H, T, Dv, generator=gen).to(inp["q"].dtype)
    dsf = torch.randn(B, H, Dk, Dv, generator=gen) if state else None
    return inp, do, dsf


@pytest.mark.parametrize("l2norm", [False, True])
@pytest.mark.parametrize("dtype,tol", [("f32", TOL_F32), ("bf16", TOL_BF16)])
@pytest.mark.parametrize("T,Dk,Dv", [(150, 128, 128), (64, 64, 64), (1, 128, 64), (97, 64, 128), (200, 128, 64)])
def test_gdn_backward(T, Dk, Dv, dtype, tol, l2norm):
    inp, do, dsf = grads_case(1, 2, T, Dk, Dv, dtype, l2norm, seed=T + Dk + Dv)
    d = to_dev(inp)
    got = binding.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], do.cuda(), d["initial_state"], dsf.cuda(),
                                scale=0.8, l2norm=l2norm, need_dinitial=True)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    ref = oracle.gdn_bwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"], do, inp["initial_state"], dsf,
                         scale=0.8, l2norm=l2norm)
    for name, x, y in zip(NAMES, got, ref):
        assert rel_err(x, y) <= tol, name


@pytest.mark.parametrize("dtype,tol", [("f32", TOL_F32), ("bf16", TOL_BF16)])
@pytest.mark.parametrize("r,T", [(2, 90), (3, 50), (4, 33), (8, 17)])
def test_deltaproduct_backward(r, T, dtype, tol):
    inp, do, dsf = grads_case(1, 2, T, 128, 128, dtype, False, r=r, seed=10 * r + T)
    d = to_dev(inp)
    got = binding.deltaproduct_chunk_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], do.cuda(), d["initial_state"],
                                         dsf.cuda(), need_dinitial=True)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    ref = oracle.deltaproduct_bwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"], do, inp["initial_state"], dsf)
    for name, x, y in zip(NAMES, got, ref):
        assert rel_err(x, y) <= tol, name


def test_deltaproduct_r1_is_gdn():
    """r = 1 of the DeltaProduct entry point computes exactly the GDN backward."""
    inp, do, dsf = grads_case(1, 2, 77, 128, 128, "bf16", True, seed=5)
    d = to_dev(inp)
    a = binding.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], do.cuda(), d["initial_state"], dsf.cuda(),
                              l2norm=True, need_dinitial=True)
    b = binding.deltaproduct_chunk_bwd(d["q"], d["k"][:, :, :, None].contiguous(), d["v"][:, :, :, None].contiguous(),
                                       d["beta"][:, :, :, None].contiguous(), d["g"], do.cuda(), d["initial_state"],
                                       dsf.cuda(), l2norm=True, need_dinitial=True)
    for x, y in zip(a, b):
        assert torch.equal(x.reshape(y.shape), y)


def test_no_state_and_no_final_gradient():
    """No initial state (zero) and no final-state gradient (zero)."""
    inp, do, _ = grads_case(2, 1, 130, 128, 128, "bf16", False, seed=3, state=False)
    d = to_dev(inp)
    got = binding.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], do.cuda(), need_dinitial=True)
    torch.cuda.synchronize()
    ref = oracle.gdn_bwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"], do)
    for name, x, y in zip(NAMES, got, ref):
        assert rel_err(x, y) <= TOL_BF16, name


def test_empty_sequence_passes_the_final_gradient_through():
    """T = 0: the initial state's gradient is the final state's (zeros without one)."""
    B, H, Dk, Dv = 1, 3, 64, 128
    e = lambda *s: torch.empty(*s, dtype=torch.bfloat16, device="cuda")
    q, k, v, beta = e(B, H, 0, Dk), e(B, H, 0, Dk), e(B, H, 0, Dv), e(B, H, 0)
    g = torch.empty(B, H, 0, device="cuda")
    do = e(B, H, 0, Dv)
    dsf = torch.randn(B, H, Dk, Dv, device="cuda")
    got = binding.gdn_chunk_bwd(q, k, v, beta, g, do, None, dsf, need_dinitial=True)
    torch.cuda.synchronize()
    assert torch.equal(got[5], dsf)
    got = binding.gdn_chunk_bwd(q, k, v, beta, g, do, None, None, need_dinitial=True)
    torch.cuda.synchronize()
    assert torch.count_nonzero(got[5]) == 0


def test_zero_keys_under_the_unit_norm():
    """Zero key and query rows stay zero under the unit-norm map; their
    gradients follow the map's floor (x / 1e-12) as in the oracle."""
    inp, do, dsf = grads_case(1, 1, 70, 64, 64, "f32", True, seed=4)
    inp["k"][0, 0, 5] = 0.0
    inp["q"][0, 0, 9] = 0.0
    d = to_dev(inp)
    got = binding.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], do.cuda(), d["initial_state"], dsf.cuda(),
                                l2norm=True, need_dinitial=True)
    torch.cuda.synchronize()
    ref = oracle.gdn_bwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"], do, inp["initial_state"], dsf,
                         l2norm=True)
    for name, x, y in zip(NAMES, got, ref):
        if name in ("dq", "dk"):  # the floored rows are ~1e12 larger: compare them on their own
            row = 9 if name == "dq" else 5
            xr, yr = x[0, 0, row].double().cpu().numpy(), y[0, 0, row]
            assert np.max(np.abs(xr - yr)) <= 1e-3 * max(np.max(np.abs(yr)), 1.0), name
            x = x.clone()
            x[0, 0, row] = 0
            y = y.copy()
            y[0, 0, row] = 0
        assert rel_err(x, y) <= TOL_F32, name


def test_full_size_sampled_heads():
    """B4 H16 T4096 D128 bf16 (the headline forward's shape): every head's
    gradients on the GPU, three heads against the oracle."""
    B, H, T = 4, 16, 4096
    inp, do, dsf = grads_case(B, H, T, 128, 128, "bf16", False, seed=21, state=False)
    d = to_dev(inp)
    got = binding.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], do.cuda())
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    idx = [0, 37, 63]
    sub = {k: heads(v, idx) for k, v in inp.items()}
    ref = oracle.gdn_bwd(sub["q"], sub["k"], sub["v"], sub["beta"], sub["g"], heads(do, idx))
    for name, x, y in zip(NAMES[:5], got[:5], ref[:5]):
        assert rel_err(heads(x, idx).cpu(), y) <= TOL_BF16, name


@pytest.mark.parametrize("cut", [37, 64, 100])
def test_split_and_resume(cut):
    """The backward over T tokens equals two calls chained through the state
    arguments: the tail's backward given the forward state at the cut (and the
    final-state gradient), then the head's backward given the tail's
    initial-state gradient as its final-state gradient; the cut need not fall
    on a chunk boundary."""
    T = 150
    inp, do, dsf = grads_case(1, 2, T, 128, 128, "f32", True, seed=31)
    d = to_dev(inp)
    dsf = dsf.cuda()
    full = binding.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], do.cuda(), d["initial_state"], dsf,
                                 l2norm=True, need_dinitial=True)
    head = {k: (v[:, :, :cut].contiguous() if k != "initial_state" else v) for k, v in d.items()}
    tail = {k: (v[:, :, cut:].contiguous() if k != "initial_state" else v) for k, v in d.items()}
    _, s_cut = binding.gdn_chunk_fwd(head["q"], head["k"], head["v"], head["beta"], head["g"],
                                     initial_state=d["initial_state"], output_final_state=True, l2norm=True)
    gt = binding.gdn_chunk_bwd(tail["q"], tail["k"], tail["v"], tail["beta"], tail["g"],
                               do[:, :, cut:].contiguous().cuda(), s_cut, dsf, l2norm=True, need_dinitial=True)
    gh = binding.gdn_chunk_bwd(head["q"], head["k"], head["v"], head["beta"], head["g"],
                               do[:, :, :cut].contiguous().cuda(), d["initial_state"], gt[5], l2norm=True,
                               need_dinitial=True)
    torch.cuda.synchronize()
    for i, name in enumerate(NAMES[:5]):
        joined = torch.cat([gh[i], gt[i]], dim=2)
        assert rel_err(joined, full[i].double().cpu().numpy()) <= TOL_F32, name
    assert rel_err(gh[5], full[5].double().cpu().numpy()) <= TOL_F32


@pytest.mark.parametrize("r,T", [(1, 300), (2, 130), (4, 70)])
def test_tensor_core_chain_matches_the_cuda_core_chain(r, T):
    """bf16 tensors at Dk = Dv = 128 run both state chains on tcgen05 (bf16
    hi / lo split products, fp32 state in tensor memory); the fp32 CUDA-core
    chains give the same gradients to within the split products' ~2^-16
    relative error, over several chunks with a ragged tail, an initial state
    and a final-state gradient.  The bf16 gradients may differ by one rounding
    of the output (2^-8 of an element); the fp32 ones only by the chains'
    arithmetic."""
    inp, do, dsf = grads_case(1, 3, T, 128, 128, "bf16", True, r=(r if r > 1 else None), seed=40 + r)
    d = to_dev(inp)

    def run(simt):
        if r == 1:
            return binding.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], do.cuda(), d["initial_state"],
                                         dsf.cuda(), l2norm=True, need_dinitial=True, simt=simt)
        return binding.deltaproduct_chunk_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], do.cuda(),
                                              d["initial_state"], dsf.cuda(), l2norm=True, need_dinitial=True,
                                              simt=simt)

    tc, simt = run(False), run(True)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    for name, x, y in zip(NAMES, tc, simt):
        tol = 5e-3 if x.dtype == torch.bfloat16 else 2e-4
        assert rel_err(x, y.double().cpu().numpy()) <= tol, name


def test_chain_bounded_wait_gives_up_and_context_survives():
    """A 1-microsecond wait limit makes the tensor-core chains' waits run out:
    the call reports GDN_ERR_TIMEOUT through the device error word, and with
    the default limit restored the next call is correct."""
    inp, do, dsf = grads_case(1, 2, 1024, 128, 128, "bf16", False, seed=50)
    d = to_dev(inp)
    assert binding.device_error() == 0
    try:
        binding.set_wait_limit(1)
        binding.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], do.cuda(), d["initial_state"], dsf.cuda(),
                              need_dinitial=True)
        torch.cuda.synchronize()
        assert binding.device_error() == 6
    finally:
        binding.set_wait_limit(0)
    assert binding.device_error() == 0
    got = binding.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], do.cuda(), d["initial_state"],
                                dsf.cuda(), need_dinitial=True)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    ref = oracle.gdn_bwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"], do, inp["initial_state"], dsf)
    for name, x, y in zip(NAMES, got, ref):
        assert rel_err(x, y) <= TOL_BF16, name


@pytest.mark.parametrize("T", [1, 40, 64, 65])
def test_tensor_core_chain_single_chunk_and_ragged(T):
    """The tensor-core chains (bf16, D 128) over one chunk (T <= 64: each chain
    takes one step, the final state comes from the initial one) and over one
    full chunk plus one token, against the oracle."""
    inp, do, dsf = grads_case(1, 2, T, 128, 128, "bf16", False, seed=70 + T)
    d = to_dev(inp)
    got = binding.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], do.cuda(), d["initial_state"],
                                dsf.cuda(), need_dinitial=True)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    ref = oracle.gdn_bwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"], do, inp["initial_state"], dsf)
    for name, x, y in zip(NAMES, got, ref):
        assert rel_err(x, y) <= TOL_BF16, name


def test_full_size_fp32_sampled_heads():
    """The fp32 backward (CUDA-core chains) over 64 chunks per head: every head
    on the GPU, two heads against the oracle at the fp32 bound."""
    B, H, T = 2, 8, 4096
    inp, do, dsf = grads_case(B, H, T, 128, 128, "f32", False, seed=33)
    d = to_dev(inp)
    got = binding.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], do.cuda(), d["initial_state"],
                                dsf.cuda(), need_dinitial=True)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    idx = [0, 13]
    sub = {k: heads(v, idx) for k, v in inp.items()}
    ref = oracle.gdn_bwd(sub["q"], sub["k"], sub["v"], sub["beta"], sub["g"], heads(do, idx),
                         sub["initial_state"], heads(dsf, idx))
    for name, x, y in zip(NAMES, got, ref):
        assert rel_err(heads(x, idx).cpu(), y) <= TOL_F32, name


@pytest.mark.parametrize("r,T", [(2, 150), (4, 90), (8, 40)])
def test_tensor_core_wy_deltaproduct_unit_norm(r, T):
    """bf16 DeltaProduct at D = 128 forms the WY factors, T, K K^T, P and B on
    tcgen05: unnormalised sub-step keys under the unit-norm flag, against the
    oracle."""
    inp, do, dsf = grads_case(1, 2, T, 128, 128, "bf16", True, r=r, seed=70 + r)
    d = to_dev(inp)
    got = binding.deltaproduct_chunk_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], do.cuda(), d["initial_state"],
                                         dsf.cuda(), scale=0.6, l2norm=True, need_dinitial=True)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    ref = oracle.deltaproduct_bwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"], do, inp["initial_state"], dsf,
                                  scale=0.6, l2norm=True)
    for name, x, y in zip(NAMES, got, ref):
        assert rel_err(x, y) <= TOL_BF16, name


def test_tensor_core_path_is_deterministic():
    """Two runs of the bf16 GDN backward over 512 chunks give the same bits."""
    inp, do, dsf = grads_case(1, 16, 2048, 128, 128, "bf16", False, seed=81)
    d = to_dev(inp)
    do, dsf = do.cuda(), dsf.cuda()
    outs = [binding.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], do, d["initial_state"], dsf,
                                  need_dinitial=True) for _ in range(2)]
    torch.cuda.synchronize()
    for x, y in zip(*outs):
        assert torch.equal(x, y)


def test_tensor_core_path_strong_decay():
    """Log-decays near -2 per token (over 100 nats per 64-row chunk): the
    backward's tensor-core kernels form every decay factor per element, so the
    gradients still match the oracle."""
    inp = gdn_inputs(1, 2, 150, 128, 128, seed=91, dtype="bf16", g_mu=-2.0, g_div=1.0, initial_state=True)
    gen = torch.Generator().manual_seed(92)
    do = torch.randn(1, 2, 150, 128, generator=gen).to(torch.bfloat16)
    dsf = torch.randn(1, 2, 128, 128, generator=gen)
    d = to_dev(inp)
    got = binding.gdn_chunk_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], do.cuda(), d["initial_state"],
                                dsf.cuda(), need_dinitial=True)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    ref = oracle.gdn_bwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"], do, inp["initial_state"], dsf)
    for name, x, y in zip(NAMES, got, ref):
        assert torch.isfinite(x).all(), name
        assert rel_err(x, y) <= TOL_BF16, name
