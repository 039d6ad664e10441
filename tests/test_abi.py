"""The C-ABI library loads and exports every entry point gdn.h declares, and
its host-side argument checks reject bad calls before anything is launched.
No call here reaches a kernel, so these run without a GPU."""
import ctypes
import os
import re

import pytest

from gated_delta_rule_47_gb300 import binding, build

HEADER = os.path.join(build.INCLUDE, "gdn.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?(?:unsigned\s+long\s+long|\w+)\s*\*?\s*(\w+)\s*\(",
                                 text, flags=re.M)))


def test_header_declares_the_documented_entry_points():
    names = declared_functions()
    for n in ("gdn_chunk_fwd", "deltaproduct_chunk_fwd", "cam_prep_fwd", "gdn_status_string",
              "gdn_chunk_fwd_workspace_bytes", "gdn_get_device_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(binding.EXPORTS) <= set(declared_functions())


def test_status_strings(lib):
    for code, name in binding.STATUS.items():
        assert binding.status_string(code) == name
    assert binding.status_string(99) == "GDN_ERR_UNKNOWN"
    assert lib.gdn_version() >= 100


def test_workspace_query(lib):
    f = lib.gdn_chunk_fwd_workspace_bytes
    bad = ctypes.c_size_t(-1).value
    assert f(1, 2, 256, 1, 64, 64, 64, binding.GDN_F32) != bad
    assert f(1, 2, 256, 1, 96, 64, 64, binding.GDN_F32) == bad   # Dk unsupported
    assert f(1, 2, 256, 1, 64, 64, 48, binding.GDN_F32) == bad   # chunk unsupported
    assert f(1, 2, 256, 3, 64, 64, 64, binding.GDN_F32) != bad   # 21 tokens per chunk
    assert f(1, 2, 256, 9, 64, 64, 64, binding.GDN_F32) == bad   # r > 8
    assert f(-1, 2, 256, 1, 64, 64, 64, binding.GDN_F32) == bad


FAKE = 0x10000  # never dereferenced: every call below fails its host checks first


def scan_call(lib, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, beta=FAKE, g=FAKE, s0=None, o=FAKE, sf=None, B=1, H=1, T=8,
             Dk=64, Dv=64, chunk=64, scale=1.0, flags=0, dtype=binding.GDN_F32, ws=None, wsb=0)
    a.update(kw)
    return lib.gdn_chunk_fwd(a["q"], a["k"], a["v"], a["beta"], a["g"], a["s0"], a["o"], a["sf"],
                             a["B"], a["H"], a["T"], a["Dk"], a["Dv"], a["chunk"], a["scale"],
                             a["flags"], a["dtype"], a["ws"], a["wsb"], None)


def test_scan_argument_checks(lib):
    assert scan_call(lib, q=None) == 1
    assert scan_call(lib, dtype=7) == 1
    assert scan_call(lib, flags=4) == 1
    assert scan_call(lib, B=-1) == 1
    assert scan_call(lib, Dk=96) == 2
    assert scan_call(lib, chunk=128) == 2
    assert scan_call(lib, v=FAKE + 8) == 3
    assert scan_call(lib, s0=FAKE + 4) == 3


def test_deltaproduct_argument_checks(lib):
    f = lib.deltaproduct_chunk_fwd
    args = lambda r, chunk: [FAKE] * 5 + [None, FAKE, None, 1, 1, 8, r, 64, 64, chunk, 1.0, 0,
                                          binding.GDN_BF16, None, 0, None]
    assert f(*args(0, 64)) == 1      # r < 1
    assert f(*args(16, 64)) == 2     # r > 8


def test_cam_prep_argument_checks(lib):
    f = lib.cam_prep_fwd

    def call(D=128, H=16, cos=None, sin=None, base=10000.0, q=FAKE, dtype=binding.GDN_BF16):
        return f(q, FAKE, FAKE, None, None, FAKE, FAKE, cos, sin, base, FAKE, FAKE, FAKE, None, None,
                 1, 4, H, D, 0.5, 1e-6, dtype, None)

    assert call(D=12) == 1               # D/2 not divisible by 4
    assert call(D=24) == 2               # not a multiple of 16
    assert call(H=64, D=128) == 2        # H*D > 4096
    assert call(cos=FAKE) == 1           # one table without the other
    assert call(base=0.0) == 1
    assert call(q=None) == 1
    assert call(q=FAKE + 2) == 3
    assert call(dtype=5) == 1


def test_cluster_shape_checks(lib):
    """The cluster-shape override accepts 1..4 heads and at least one WY CTA
    per cluster (at most 16 CTAs), and 0, 0 restores the automatic choice."""
    for hc, nwy in ((0, 1), (5, 1), (1, 0), (4, 13), (-1, 2)):
        assert lib.gdn_set_cluster_shape(hc, nwy) == 1, (hc, nwy)
    for hc, nwy in ((1, 1), (4, 5), (2, 14)):
        assert lib.gdn_set_cluster_shape(hc, nwy) == 0
    assert lib.gdn_set_cluster_shape(0, 0) == 0


def test_cam_scan_argument_checks(lib):
    f = lib.cam_scan_fwd
    u = 0x10000

    def call(q=u, s0=None, sf=None, B=1, H=2, F=3, S=5, Dk=64, Dv=64, flags=0, dtype=binding.GDN_F32):
        return f(q, u, u, u, u, s0, u, sf, B, H, F, S, Dk, Dv, 1.0, flags, dtype, None, 0, None)

    assert call(s0=u, flags=binding.GDN_CAM_REVERSE) == 2      # no state in the reverse mode
    assert call(sf=u, flags=binding.GDN_CAM_REVERSE) == 2
    assert call(S=0) == 1                                      # a frame holds at least one token
    assert call(F=-1) == 1
    assert call(flags=8) == 1
    assert call(Dk=96) == 2
    assert call(dtype=7) == 1
    assert call(q=None) == 1
    assert call(q=u + 8) == 3
    q = lib.cam_scan_fwd_workspace_bytes
    bad = ctypes.c_size_t(-1).value
    assert q(1, 2, 3, 5, 64, 64, binding.GDN_F32) == 0         # the CUDA-core path needs none
    assert q(1, 2, 3, 0, 64, 64, binding.GDN_F32) == bad
    assert q(1, 2, 3, 5, 96, 64, binding.GDN_F32) == bad


def test_masked_deltaproduct_argument_checks(lib):
    f = lib.masked_deltaproduct_chunk_fwd
    u = 0x10000

    def call(r=2, Dk=64, chunk=64, flags=0, mask=u, q=u, dtype=binding.GDN_F32, ws=u, ws_bytes=1 << 40):
        return f(q, u, u, u, u, mask, None, u, None, 1, 2, 8, r, Dk, 64, chunk, 1.0, flags, dtype, ws, ws_bytes,
                 None)

    assert call(ws=None) == 4      # workspace missing
    assert call(ws_bytes=16) == 4  # or short
    assert call(r=3) == 2          # r must divide Dk
    assert call(r=16, Dk=128) == 2  # r <= 8
    assert call(chunk=48) == 2
    assert call(chunk=0) == 1
    assert call(flags=4) == 1      # GDN_QK_L2NORM and GDN_PATH_SIMT only
    assert call(mask=None) == 1
    assert call(q=u + 4) == 3
    assert call(dtype=3) == 1
    q = lib.masked_deltaproduct_chunk_fwd_workspace_bytes
    per = 2 * 64 * 64 + 2 * 64 * 64 + 64 * 64 + 64 * 64 + 64  # W, Kd, U, Vn, S, P, gamma at D = 64
    assert q(1, 2, 40, 2, 64, 64, binding.GDN_F32) == 4 * 2 * 2 * per  # 40 tokens: two chunks of 32
    assert q(1, 2, 0, 2, 64, 64, binding.GDN_F32) == 0
    assert q(1, 2, 40, 3, 64, 64, binding.GDN_F32) == ctypes.c_size_t(-1).value


def test_cam_prep_scan_argument_checks(lib):
    f = lib.cam_prep_scan_fwd
    u = 0x10000

    def call(D=128, F=3, N=30, H=2, dtype=binding.GDN_BF16, base=10000.0, flags=0, s0=None, ws=u, wsb=1 << 30):
        return f(u, u, u, None, None, u, u, base, u, u, s0, u, None, 1, N, H, D, F, 0.5, 1e-6, 1.0, flags, dtype,
                 ws, wsb, None)

    assert call(D=64) == 2
    assert call(H=33) == 2                              # H * D <= 4096
    assert call(dtype=binding.GDN_F32) == 2
    assert call(base=0.0) == 1
    assert call(flags=binding.GDN_CAM_REVERSE, s0=u) == 2
    assert call(N=31) == 1                              # N is not a whole number of frames
    assert call(flags=2) == 1                           # no CUDA-core switch here
    assert call(ws=None) == 4
    q = lib.cam_prep_scan_fwd_workspace_bytes
    assert q(1, 30, 2, 128, 3, binding.GDN_BF16) == 2 * 3 * 131072 + 30 * 8
    assert q(1, 30, 2, 64, 3, binding.GDN_BF16) == ctypes.c_size_t(-1).value


def test_cam_prep_bwd_argument_checks(lib):
    f = lib.cam_prep_bwd
    u = 0x10000

    def call(D=128, H=4, dtype=binding.GDN_BF16, cos=None, sin=None, base=10000.0, q=u):
        return f(q, u, None, None, u, u, cos, sin, base, u, u, u, None, None, u, u, u, 1, 8, H, D, 0.5, 1e-6, dtype,
                 None)

    assert call(D=36) == 1                 # D/2 not a multiple of 4
    assert call(H=64) == 2                 # H * D > 4096
    assert call(cos=u) == 1                # one table without the other
    assert call(base=0.0) == 1
    assert call(dtype=4) == 1
    assert call(q=None) == 1
    assert call(q=u + 4) == 3


def test_cam_scan_bwd_argument_checks(lib):
    f = lib.cam_scan_bwd
    u = 0x10000

    def call(flags=0, Dk=64, S=5, dtype=binding.GDN_F32, q=u, ws=u):
        return f(q, u, u, u, u, None, u, None, u, u, u, u, u, None, 1, 2, 3, S, Dk, 64, 1.0, flags, dtype, ws,
                 1 << 40, None)

    assert call(flags=binding.GDN_CAM_REVERSE) == 2
    assert call(flags=8) == 1
    assert call(Dk=96) == 2
    assert call(S=0) == 1
    assert call(dtype=5) == 1
    assert call(q=None) == 1
    assert call(q=u + 4) == 3
    assert call(ws=None) == 4
    # G, H, P and dX per frame, the states entering each frame and the last, one share per tile
    assert lib.cam_scan_bwd_workspace_bytes(1, 2, 3, 5, 64, 64, binding.GDN_F32) == 4 * (
        2 * 3 * 4 * 64 * 64 + 2 * 4 * 64 * 64 + 64)
    # bf16 at D = 128 adds the bf16 hi / lo images of the states (F + 1) and gradients (F), 64 KB each
    assert lib.cam_scan_bwd_workspace_bytes(1, 2, 3, 5, 128, 128, binding.GDN_BF16) == 4 * (
        2 * 3 * 4 * 128 * 128 + 2 * 4 * 128 * 128 + 64) + 2 * 7 * 65536


def test_chunk_bwd_argument_checks(lib):
    f = lib.deltaproduct_chunk_bwd
    u = 0x10000
    bad = ctypes.c_size_t(-1).value

    def call(r=1, flags=0, Dk=64, T=70, dtype=binding.GDN_F32, q=u, ws=u, ws_bytes=1 << 40):
        return f(q, u, u, u, u, None, u, None, u, u, u, u, u, None, 1, 2, T, r, Dk, 64, 1.0, flags, dtype, ws,
                 ws_bytes, None)

    assert call(r=0) == 1
    assert call(r=9) == 1
    assert call(flags=binding.GDN_CAM_REVERSE) == 1
    assert call(Dk=96) == 2
    assert call(T=-1) == 1
    assert call(dtype=5) == 1
    assert call(q=None) == 1
    assert call(q=u + 4) == 3
    assert call(ws=None) == 4
    assert call(ws_bytes=16) == 4
    assert lib.gdn_chunk_bwd(u, u, u, u, u, None, u, None, None, u, u, u, u, None, 1, 2, 5, 64, 64, 1.0, 0,
                             binding.GDN_F32, u, 1 << 40, None) == 1  # dq missing
    wsb = lib.gdn_chunk_bwd_workspace_bytes
    per = 3 * 64 * 64 + 2 * 64 * 64 + 2 * 64 * 64 + 3 * 64 * 64 + 64  # floats per head and chunk at D = 64
    assert wsb(1, 2, 70, 1, 64, 64, binding.GDN_F32) == 4 * 2 * 2 * per  # 70 tokens: 2 chunks of 64
    assert wsb(1, 2, 70, 3, 64, 64, binding.GDN_F32) == 4 * 2 * 4 * per  # 21 tokens per chunk
    assert wsb(1, 2, 0, 1, 64, 64, binding.GDN_F32) == 0
    assert wsb(1, 2, 70, 9, 64, 64, binding.GDN_F32) == bad
    assert wsb(1, 2, 70, 1, 96, 64, binding.GDN_F32) == bad


def test_masked_bwd_argument_checks(lib):
    f = lib.masked_deltaproduct_chunk_bwd
    u = 0x10000

    def call(r=2, flags=0, Dk=64, dtype=binding.GDN_F32, mask=u, ws=u, ws_bytes=1 << 40):
        return f(u, u, u, u, u, mask, None, u, None, u, u, u, u, u, None, 1, 2, 40, r, Dk, 64, 1.0, flags, dtype, ws,
                 ws_bytes, None)

    assert call(r=3) == 2          # r must divide 64 and Dk
    assert call(r=16) == 2
    assert call(flags=4) == 1      # GDN_QK_L2NORM and GDN_PATH_SIMT only
    assert call(Dk=96) == 2
    assert call(dtype=4) == 1
    assert call(mask=None) == 1
    assert call(ws=None) == 4
    assert call(ws_bytes=16) == 4
    q = lib.masked_deltaproduct_chunk_bwd_workspace_bytes
    per = 3 * 64 * 64 + 2 * 64 * 64 + 2 * 64 * 64 + 3 * 64 * 64 + 64
    assert q(1, 2, 40, 2, 64, 64, binding.GDN_F32) == 4 * 2 * 2 * per  # 40 tokens: two chunks of 32
    assert q(1, 2, 40, 3, 64, 64, binding.GDN_F32) == ctypes.c_size_t(-1).value
