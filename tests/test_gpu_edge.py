"""GPU parity in the regimes the workloads' weak gates never reach, and the
method's own degenerate cases, through the C ABI.

* Strong forgetting: chunks whose cumulative decay spans more than 80 nats
  make the tensor-core path form every decay factor e^{g_t - g_s} directly
  instead of as a product of row and column factors; chunks of that kind,
  weak ones and ones just under the limit alternate within each head, for
  GDN and DeltaProduct r = 2, 4, in the ring mode and in a forced cluster
  shape, against the fp64 oracle.
* beta = 0 with an initial state is pure decay: S_T = e^{sum g} S_0 and
  o_t = scale e^{G_t} S_0^T q_t in closed form.
* g = 0, beta = 1 and orthonormal keys overwrite exactly: the state maps k_i
  to v_i, so o_t = sum_{i<=t} (q_t . k_i) v_i, and querying a stored key
  returns its value.
* beta = 2 with unit keys, g = 0 and v = 0 is a product of reflections: the
  state's Frobenius norm is preserved.
Tolerances are max|o - o_ref| / max|o_ref| <= 1e-4 for fp32 tensors and
<= 1e-2 for bf16 tensors with the fp32 state."""
import numpy as np
import pytest
import torch

import oracle
from gated_delta_rule_47_gb300 import binding
from gated_delta_rule_47_gb300.inputs import gdn_inputs, mixed_decay, orthonormal_keys, to_f64
from tests.gpu_util import TOL_BF16, TOL_F32, ensure_lib, rel_err, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def call(inp, r=None, simt=False, l2norm=False, scale=1.0, shape=(0, 0), chunk=64):
    """One forward through the binding (GDN when r is None) with an optional
    forced cluster shape; returns (o, final_state) on the device."""
    d = to_dev(inp)
    try:
        binding.set_cluster_shape(*shape)
        if r is None:
            o, sf = binding.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d.get("initial_state"),
                                          output_final_state=True, chunk=chunk, scale=scale, l2norm=l2norm,
                                          simt=simt)
        else:
            o, sf = binding.deltaproduct_chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"],
                                                   d.get("initial_state"), output_final_state=True,
                                                   chunk=chunk, scale=scale, l2norm=l2norm, simt=simt)
        torch.cuda.synchronize()
    finally:
        binding.set_cluster_shape(0, 0)
    assert binding.device_error() == 0
    return o, sf


def oracle_of(inp, r=None, l2norm=False, scale=1.0):
    if r is None:
        return oracle.gdn_fwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"], inp.get("initial_state"),
                              scale=scale, l2norm=l2norm)
    return oracle.deltaproduct_fwd(inp["q"], inp["k"], inp["v"], inp["beta"], inp["g"], inp.get("initial_state"),
                                   scale=scale, l2norm=l2norm)


# ------------------------------------------------------------ strong forgetting

@pytest.mark.parametrize("shape", [(0, 0), (2, 2)], ids=["ring", "cluster2x2"])
@pytest.mark.parametrize("r", [1, 2, 4])
def test_strong_decay_chunks_tensor_core(r, shape):
    """300 rows per head: four full 64-row chunks and a 44-row tail, cycling
    strong (> 80 nats per chunk), weak and just-under-the-limit decay."""
    T = 300 // r
    inp = gdn_inputs(2, 3, T, 128, 128, seed=200 + r, dtype="bf16", r=None if r == 1 else r,
                     initial_state=True)
    inp["g"] = mixed_decay(2, 3, T, seed=300 + r, r=r)
    g = inp["g"].double()
    span = [float((g[..., c * 64 // r:(c + 1) * 64 // r].sum(-1)).abs().min()) for c in range(3)]
    assert span[0] > 80 and span[2] < 80  # the chunks reach both branches
    rr = None if r == 1 else r
    o, sf = call(inp, r=rr, shape=shape)
    ro, rs = oracle_of(inp, r=rr)
    assert rel_err(o, ro) <= TOL_BF16
    assert rel_err(sf, rs) <= TOL_BF16


@pytest.mark.parametrize("dtype,tol", [("f32", TOL_F32), ("bf16", TOL_BF16)])
def test_strong_decay_cuda_core_path(dtype, tol):
    inp = gdn_inputs(1, 2, 203, 64, 128, seed=211, dtype=dtype, initial_state=True)
    inp["g"] = mixed_decay(1, 2, 203, seed=212)
    o, sf = call(inp, simt=True)
    ro, rs = oracle_of(inp)
    assert rel_err(o, ro) <= tol
    assert rel_err(sf, rs) <= tol


# ------------------------------------------------------------ beta = 0: pure decay

def pure_decay_closed_form(inp, scale):
    g = to_f64(inp["g"])
    G = np.cumsum(g, axis=-1)  # [B,H,T]
    S0 = to_f64(inp["initial_state"])
    q = to_f64(inp["q"])
    o = scale * np.exp(G)[..., None] * np.einsum("bhkv,bhtk->bhtv", S0, q)
    return o, np.exp(G[..., -1])[..., None, None] * S0


@pytest.mark.parametrize("path,dtype,tol,shape", [
    ("tc", "bf16", TOL_BF16, (0, 0)), ("tc", "bf16", TOL_BF16, (1, 2)),
    ("simt", "f32", TOL_F32, (0, 0)), ("simt", "bf16", TOL_BF16, (0, 0))])
def test_beta_zero_is_pure_decay(path, dtype, tol, shape):
    T = 150
    inp = gdn_inputs(1, 3, T, 128, 128, seed=220, dtype=dtype, initial_state=True)
    inp["beta"] = torch.zeros_like(inp["beta"])
    inp["g"] = (inp["g"] * 4).contiguous()  # reaches e^{-10} or so by the end
    o, sf = call(inp, simt=path == "simt", scale=0.5, shape=shape)
    co, cs = pure_decay_closed_form(inp, 0.5)
    assert rel_err(o, co) <= tol
    assert rel_err(sf, cs) <= tol


def test_beta_zero_deltaproduct_tensor_core():
    inp = gdn_inputs(1, 2, 70, 128, 128, seed=221, dtype="bf16", r=2, initial_state=True)
    inp["beta"] = torch.zeros_like(inp["beta"])
    o, sf = call(inp, r=2)
    co, cs = pure_decay_closed_form(inp, 1.0)
    assert rel_err(o, co) <= TOL_BF16
    assert rel_err(sf, cs) <= TOL_BF16


# ------------------------------------------------------------ g = 0, beta = 1: overwrite

def overwrite_inputs(D, T, dtype, seed):
    inp = gdn_inputs(1, 2, T, D, D, seed=seed, dtype="f32")
    k = orthonormal_keys(1, 2, T, D, seed=seed + 1)
    q = inp["q"].clone()
    q[:, :, 1::2] = k[:, :, : (T // 2)]  # odd tokens query an earlier key: t = 2j+1 asks for k_j
    td = torch.bfloat16 if dtype == "bf16" else torch.float32
    return {"q": q.to(td).contiguous(), "k": k.to(td).contiguous(), "v": inp["v"].to(td).contiguous(),
            "beta": torch.ones(1, 2, T, dtype=td), "g": torch.zeros(1, 2, T)}


def overwrite_closed_form(inp):
    q, k, v = to_f64(inp["q"]), to_f64(inp["k"]), to_f64(inp["v"])
    scores = np.einsum("bhtd,bhsd->bhts", q, k)
    scores = np.tril(scores)  # inclusive causal
    return np.einsum("bhts,bhsv->bhtv", scores, v)


@pytest.mark.parametrize("path,D", [("simt", 64), ("simt", 128)])
def test_overwrite_with_orthonormal_keys_fp32(path, D):
    T = min(D, 100)
    inp = overwrite_inputs(D, T, "f32", seed=230 + D)
    o, _ = call(inp, simt=True)
    assert rel_err(o, overwrite_closed_form(inp)) <= TOL_F32
    # querying k_j returns v_j
    got = to_f64(o)[:, :, 1::2]
    want = to_f64(inp["v"])[:, :, : T // 2]
    assert np.max(np.abs(got - want)) <= 1e-4 * np.max(np.abs(want))


@pytest.mark.parametrize("shape", [(0, 0), (2, 1)], ids=["ring", "cluster2x1"])
def test_overwrite_with_orthonormal_keys_tensor_core(shape):
    inp = overwrite_inputs(128, 100, "bf16", seed=240)
    o, sf = call(inp, shape=shape)
    ro, rs = oracle_of(inp)
    assert rel_err(o, ro) <= TOL_BF16
    assert rel_err(sf, rs) <= TOL_BF16
    # the bf16-rounded keys are orthonormal to about 2^-8, so the closed form
    # holds to that order too
    assert rel_err(o, overwrite_closed_form(inp)) <= 3e-2


# ------------------------------------------------------------ beta = 2: reflections

@pytest.mark.parametrize("path,dtype,tol", [("tc", "bf16", TOL_BF16), ("simt", "f32", TOL_F32)])
def test_reflections_preserve_state_norm(path, dtype, tol):
    T = 200
    inp = gdn_inputs(1, 2, T, 128, 128, seed=250, dtype=dtype, initial_state=True, normalise_qk=False)
    inp["beta"] = torch.full_like(inp["beta"], 2.0)
    inp["v"] = torch.zeros_like(inp["v"])
    inp["g"] = torch.zeros_like(inp["g"])
    o, sf = call(inp, simt=path == "simt", l2norm=True)
    ro, rs = oracle_of(inp, l2norm=True)
    assert rel_err(o, ro) <= tol
    assert rel_err(sf, rs) <= tol
    n0 = np.linalg.norm(to_f64(inp["initial_state"]).reshape(2, -1), axis=-1)
    nT = np.linalg.norm(to_f64(sf).reshape(2, -1), axis=-1)
    assert np.max(np.abs(nT / n0 - 1.0)) <= tol
