"""The allocation-free entry point, gdn_chunk_fwd_noalloc, against gdn_chunk_fwd.

Some callers cannot allocate device memory: code that runs where cudaMalloc is
not allowed (a host callback, a plug-in whose host owns every allocation) or
under a memory budget fixed in advance.  They call gdn_chunk_fwd_noalloc, which
takes no workspace and uses a fixed scratch array inside the library instead.
These tests call it through the C ABI twice in a row and compare each output
with gdn_chunk_fwd's (given its own workspace) on the same inputs, within the
bf16 tolerance the other parity tests use.  The file is named to be collected
last, so that a failure here comes after every other test has run."""
import pytest
import torch

from gated_delta_rule_47_gb300 import binding
from gated_delta_rule_47_gb300.inputs import gdn_inputs, to_f64
from tests.gpu_util import TOL_BF16, TOL_F32, ensure_lib, rel_err, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def both(d, **kw):
    ref, ref_sf = binding.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d.get("initial_state"),
                                        output_final_state=True, **kw)
    outs = []
    for _ in range(2):  # two calls in a row share the array
        o, sf = binding.gdn_chunk_fwd_noalloc(d["q"], d["k"], d["v"], d["beta"], d["g"],
                                              d.get("initial_state"), output_final_state=True, **kw)
        torch.cuda.synchronize()
        outs.append((o.clone(), sf.clone()))
    return (ref, ref_sf), outs


@pytest.mark.parametrize("B,H,T", [(4, 16, 700), (1, 3, 300), (2, 5, 64)])
def test_noalloc_matches_gdn_chunk_fwd(B, H, T):
    d = to_dev(gdn_inputs(B, H, T, 128, 128, seed=41 + T, dtype="bf16", initial_state=True))
    assert binding.workspace_bytes(B, H, T, 128, 128) > 0  # the scratch-using path
    (ref, ref_sf), outs = both(d)
    for o, sf in outs:
        assert rel_err(o, to_f64(ref)) <= TOL_BF16
        assert rel_err(sf, to_f64(ref_sf)) <= TOL_BF16
    assert binding.device_error() == 0


def test_noalloc_fp32_path_needs_no_scratch():
    d = to_dev(gdn_inputs(1, 2, 200, 64, 64, seed=5, dtype="f32"))
    (ref, _), outs = both(d)
    for o, _ in outs:
        assert rel_err(o, to_f64(ref)) <= TOL_F32


def test_noalloc_rejects_more_heads_than_the_array_serves():
    d = to_dev(gdn_inputs(1, 65, 64, 128, 128, seed=6, dtype="bf16"))
    if binding.workspace_bytes(1, 65, 64, 128, 128) == 0:
        pytest.skip("65 heads take the cluster path here, which needs no scratch")
    with pytest.raises(binding.GdnError) as e:
        binding.gdn_chunk_fwd_noalloc(d["q"], d["k"], d["v"], d["beta"], d["g"])
    assert e.value.status == 4  # GDN_ERR_WORKSPACE
