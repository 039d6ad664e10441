"""The allocation-free entry point, gdn_chunk_fwd_noalloc, against gdn_chunk_fwd.

Some callers cannot allocate device memory: code that runs where cudaMalloc is
not allowed (a host callback, a plug-in whose host owns every allocation) or
under a memory budget fixed in advance.  They call gdn_chunk_fwd_noalloc, which
takes no workspace and uses a fixed scratch array inside the library instead.
These tests call it through the C ABI twice in a row and check that each output
is bit for bit gdn_chunk_fwd's (given its own workspace) on the same inputs:
both run the same kernel on the same inputs, and a stale or partly overwritten
ring slot in the shared array would show as a difference.  The file is named to
be collected last, so that a failure here comes after every other test has
run."""
import pytest
import torch

import oracle
from gated_delta_rule_47_gb300 import binding
from gated_delta_rule_47_gb300.inputs import gdn_inputs
from tests.gpu_util import TOL_BF16, ensure_lib, heads, rel_err, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def ref_call(d):
    return binding.gdn_chunk_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d.get("initial_state"),
                                 output_final_state=True)


def noalloc_call(d):
    return binding.gdn_chunk_fwd_noalloc(d["q"], d["k"], d["v"], d["beta"], d["g"], d.get("initial_state"),
                                         output_final_state=True)


@pytest.mark.parametrize("B,H,T", [(4, 16, 700), (1, 3, 300), (2, 5, 64)])
def test_noalloc_matches_gdn_chunk_fwd(B, H, T):
    d = to_dev(gdn_inputs(B, H, T, 128, 128, seed=41 + T, dtype="bf16", initial_state=True))
    assert binding.workspace_bytes(B, H, T, 128, 128) > 0  # the scratch-using path
    ref, ref_sf = ref_call(d)
    for _ in range(2):  # two calls in a row share the array
        o, sf = noalloc_call(d)
        torch.cuda.synchronize()
        assert torch.equal(o, ref)
        assert torch.equal(sf, ref_sf)
    assert binding.device_error() == 0


def test_noalloc_head_counts_change_between_unsynchronised_calls():
    """64, then 5, then 48 heads, enqueued back to back on one stream with no
    synchronisation: each call's tags sit where the previous call kept ring
    payload, and every result is still gdn_chunk_fwd's."""
    cases = [(4, 16, 400), (1, 5, 300), (3, 16, 200)]
    ins = [to_dev(gdn_inputs(B, H, T, 128, 128, seed=500 + B * H, dtype="bf16", initial_state=True))
           for B, H, T in cases]
    refs = [ref_call(d) for d in ins]
    torch.cuda.synchronize()
    outs = [noalloc_call(d) for d in ins]
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    for (o, sf), (ro, rs) in zip(outs, refs):
        assert torch.equal(o, ro)
        assert torch.equal(sf, rs)


def test_noalloc_fp32_path_needs_no_scratch():
    d = to_dev(gdn_inputs(1, 2, 200, 64, 64, seed=5, dtype="f32"))
    ref, ref_sf = ref_call(d)
    for _ in range(2):
        o, sf = noalloc_call(d)
        torch.cuda.synchronize()
        assert torch.equal(o, ref)
        assert torch.equal(sf, ref_sf)


def test_noalloc_more_heads_than_the_array_serves_run_without_scratch():
    """65 heads: the array's ring holds 64, so the tensor-core path runs in its
    cluster mode, which needs no scratch; checked against the oracle on
    sampled heads, and two calls agree bit for bit."""
    B, H, T = 1, 65, 130
    inp = gdn_inputs(B, H, T, 128, 128, seed=6, dtype="bf16", initial_state=True)
    d = to_dev(inp)
    o1, s1 = noalloc_call(d)
    torch.cuda.synchronize()
    o2, s2 = noalloc_call(d)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    assert torch.equal(o1, o2) and torch.equal(s1, s2)
    idx = [0, 31, 64]
    sub = {k: heads(v, idx) for k, v in inp.items()}
    ro, rs = oracle.gdn_fwd(sub["q"], sub["k"], sub["v"], sub["beta"], sub["g"], sub["initial_state"])
    assert rel_err(heads(o1, idx).cpu(), ro) <= TOL_BF16
    assert rel_err(heads(s1, idx).cpu(), rs) <= TOL_BF16
