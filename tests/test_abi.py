"""C-ABI checks that need no GPU: the library loads, exports every function
declared in include/qfp4.h, and rejects bad arguments on the host before
launching anything."""
import os
import re

import pytest

from block_scaled_fp4_tcgen05_gb300 import qfp4

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qfp4.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qfp4_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(qfp4.LIB_PATH):
        import __graft_entry__
        __graft_entry__.build()
    return qfp4.load()


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(qfp4.SIGNATURES), "binding signatures out of sync with the header"


def test_version_and_strings(lib):
    assert qfp4.version() >= 100
    for code in (0, -1, -2, -3, -4, -5, -6, -7, 12345):
        assert isinstance(qfp4.status_string(code), str) and qfp4.status_string(code)


def test_sizes(lib):
    assert qfp4.block_size(0) == 32 and qfp4.block_size(1) == 16 and qfp4.block_size(9) == 0
    assert qfp4.sf_mma_bytes(128, 4) == 512
    assert qfp4.sf_mma_bytes(129, 5) == 2 * 2 * 512
    assert qfp4.sf_mma_bytes(0, 8) == 0
    assert qfp4.sf_mma_grouped_bytes(8192, 8, 256) == (64 + 8) * 64 * 512


FAKE = 1 << 40          # a 16-byte aligned address that is never dereferenced


def test_quantize_rejects_bad_arguments(lib):
    L = lib.qfp4_quantize
    ok_args = dict(fmt=1, X=FAKE, M=16, K=256, gs=FAKE, Q=FAKE, SF=FAKE, layout=0, stream=None)

    def call(**kw):
        a = dict(ok_args, **kw)
        return L(a["fmt"], a["X"], a["M"], a["K"], a["gs"], a["Q"], a["SF"], a["layout"], a["stream"])

    assert call(fmt=3) == -1
    assert call(layout=5) == -1
    assert call(M=-1) == -1
    assert call(K=200) == -2
    assert call(X=None) == -1
    assert call(gs=None) == -1                  # NVFP4 needs a global scale
    assert call(X=FAKE + 8) == -3
    assert call(Q=FAKE + 4) == -3
    assert call(SF=FAKE + 2) == -3
    assert call(M=0) == 0                       # empty: nothing to do, nothing launched
    # (M + 128) * (K / 16) must stay below 2^32 - 4096 (32-bit block indices)
    assert call(M=(1 << 32) // 16 - 128 - 256, K=256) == -2
    assert call(M=(1 << 32) // 16 - 128 - 257, K=256, X=None) == -1   # just inside: reaches the pointer checks


def test_gemm_rejects_bad_arguments(lib):
    L = lib.qfp4_gemm_nt
    base = [1, 256, 256, 256, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 0, None]

    def call(i=None, v=None):
        a = list(base)
        if i is not None:
            a[i] = v
        return L(*a)

    assert call(0, 3) == -1
    assert call(1, -1) == -1
    assert call(1, 0) == 0                      # empty D: nothing to do, nothing launched
    assert call(2, 0) == 0
    assert call(2, 100) == -2                   # N % 128
    assert call(3, 192) == -2                   # K % 128
    assert call(4, None) == -1
    assert call(4, FAKE + 8) == -3
    assert call(10, FAKE + 2) == -3


def test_grouped_and_interleave_reject_bad_arguments(lib):
    assert lib.qfp4_gemm_nt_grouped(1, 0, FAKE, 10, 10, 256, 256, FAKE, FAKE, FAKE, FAKE,
                                    None, None, FAKE, None, 0, None) == -1
    assert lib.qfp4_gemm_nt_grouped(1, 300, FAKE, 10, 10, 256, 256, FAKE, FAKE, FAKE, FAKE,
                                    None, None, FAKE, None, 0, None) == -2
    assert lib.qfp4_quantize_grouped(1, FAKE, 10, 256, 2, FAKE, None, FAKE, FAKE, None) == -1
    assert lib.qfp4_quantize_grouped(1, FAKE, 10, 256, 257, FAKE, FAKE, FAKE, FAKE, None) == -2
    assert lib.qfp4_gemm_nt_grouped(1, 257, FAKE, 10, 10, 256, 256, FAKE, FAKE, FAKE, FAKE,
                                    None, None, FAKE, None, 0, None) == -2
    assert lib.qfp4_gemm_nt_grouped(1, 2, FAKE, 10, -1, 256, 256, FAKE, FAKE, FAKE, FAKE,
                                    None, None, FAKE, None, 0, None) == -1     # max_group_rows < 0
    assert lib.qfp4_global_scale_grouped(FAKE, 10, 16, 257, FAKE, FAKE, None) == -2
    assert lib.qfp4_sf_interleave(FAKE, 10, 10, FAKE, 7, None) == -1
    assert lib.qfp4_sf_interleave(FAKE, 10, 10, FAKE + 1, 1, None) == -3
    assert lib.qfp4_sf_interleave(FAKE, 0, 10, FAKE, 1, None) == 0
    assert lib.qfp4_global_scale(FAKE, 10, 12, FAKE, None) == -2
    assert lib.qfp4_global_scale(FAKE + 2, 10, 16, FAKE, None) == -3
    assert lib.qfp4_global_scale(None, 10, 16, FAKE, None) == -1          # X NULL but not empty
    assert lib.qfp4_global_scale(FAKE, 10, 16, None, None) == -1          # no gs_out


def test_absmax_gs_rejects_bad_arguments(lib):
    a = lib.qfp4_absmax_gs
    assert a(0, FAKE, FAKE, 256, FAKE, None) == -1             # groups
    assert a(257, FAKE, FAKE, 256, FAKE, None) == -2           # at most 256 groups
    assert a(2, None, FAKE, 256, FAKE, None) == -1             # offsets required
    assert a(2, FAKE, None, 256, FAKE, None) == -1
    assert a(2, FAKE, FAKE, 256, None, None) == -1
    assert a(2, FAKE, FAKE, 12, FAKE, None) == -2              # K % 8
    assert a(2, FAKE, FAKE + 8, 256, FAKE, None) == -3
    assert a(2, FAKE + 2, FAKE, 256, FAKE, None) == -3
    assert a(2, FAKE, FAKE, 256, FAKE + 2, None) == -3


def test_residual_rmsnorm_quantize_rejects_bad_arguments(lib):
    L = lib.qfp4_residual_rmsnorm_quantize
    ok = dict(fmt=1, X=FAKE, R=FAKE, gm=FAKE, M=16, K=256, eps=1e-6, Y=FAKE, gs=FAKE, Q=FAKE, SF=FAKE, lay=1)

    def call(**kw):
        a = dict(ok, **kw)
        return L(a["fmt"], a["X"], a["R"], a["gm"], a["M"], a["K"], a["eps"], a["Y"], a["gs"], a["Q"], a["SF"],
                 a["lay"], None)

    assert call(fmt=2) == -1
    assert call(lay=3) == -1
    assert call(M=-1) == -1
    assert call(eps=-1.0) == -1 and call(eps=float("nan")) == -1 and call(eps=float("inf")) == -1
    assert call(K=200) == -2                    # K % 128
    assert call(K=65536 + 128) == -2            # longer rows than one CTA holds
    assert call(M=0) == 0 and call(K=0) == 0     # empty: nothing launched
    assert call(X=None) == -1 and call(gm=None) == -1 and call(Q=None) == -1 and call(SF=None) == -1
    assert call(gs=None) == -1                  # NVFP4 writes the row scales
    assert call(X=FAKE + 8) == -3 and call(R=FAKE + 8) == -3 and call(Y=FAKE + 8) == -3
    assert call(gm=FAKE + 8) == -3 and call(Q=FAKE + 4) == -3 and call(SF=FAKE + 2) == -3
    assert call(gs=FAKE + 2) == -3


def test_sparse_entry_points_reject_bad_arguments(lib):
    c = lib.qfp4_sparse24_compress
    assert c(FAKE, 16, 256, FAKE, FAKE, 7, None) == -1          # layout
    assert c(FAKE, -1, 256, FAKE, FAKE, 0, None) == -1
    assert c(FAKE, 16, 96, FAKE, FAKE, 0, None) == -2           # K % 64
    assert c(FAKE, 16, 256, FAKE, FAKE, 1, None) == -2          # tiled metadata wants K % 512
    assert c(None, 16, 256, FAKE, FAKE, 0, None) == -1
    assert c(FAKE + 8, 16, 256, FAKE, FAKE, 0, None) == -3
    assert c(FAKE, 16, 256, FAKE, FAKE + 2, 0, None) == -3
    assert c(FAKE, 0, 256, FAKE, FAKE, 0, None) == 0
    assert qfp4.sparse24_meta_bytes(130, 512, 1) == 256 * 32 and qfp4.sparse24_meta_bytes(130, 512, 0) == 130 * 32
    g = lib.qfp4_gemm_nt_sparse24
    base = [2, 256, 256, 512, FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, None, FAKE, None]

    def call(i=None, v=None):
        a = list(base)
        if i is not None:
            a[i] = v
        return g(*a)

    assert call(0, 5) == -1
    assert call(0, 1) == -2                                      # the sparse MMA's scales are per 32
    assert call(1, -1) == -1
    assert call(2, 384) == -2                                    # N % 256
    assert call(3, 256) == -2                                    # K % 512
    assert call(1, 0) == 0                                       # empty D
    assert call(4, None) == -1
    assert call(6, FAKE + 8) == -3
    assert call(11, FAKE + 2) == -3


def test_boundary_names_of_the_scope_table(lib):
    """The entry points the scope of this library names, with the argument
    counts given there: the three core calls, the per-expert global scale
    (row count on the device), the grouped quantiser and the grouped GEMM
    with its workspace pair, the workspace size query and the status calls."""
    want = {"qfp4_quantize": 9, "qfp4_sf_interleave": 6, "qfp4_gemm_nt": 14,
            "qfp4_gemm_workspace_bytes": 4, "qfp4_sf_mma_bytes": 2, "qfp4_absmax_gs": 6,
            "qfp4_quantize_grouped": 10, "qfp4_gemm_nt_grouped": 17, "qfp4_poll_device_status": 1,
            "qfp4_status_string": 1}
    for name, nargs in want.items():
        assert hasattr(lib, name), name
        assert len(qfp4.SIGNATURES[name][1]) == nargs, name
    # the grouped GEMM carries (workspace, ws_bytes) right before the stream
    args = qfp4.SIGNATURES["qfp4_gemm_nt_grouped"][1]
    assert args[-3] is qfp4._vp and args[-2] is qfp4._sz


def test_two_level_entry_points_reject_bad_arguments(lib):
    # per-row global scales
    assert lib.qfp4_global_scale_rows(FAKE, -1, 16, FAKE, None) == -1
    assert lib.qfp4_global_scale_rows(FAKE, 10, 12, FAKE, None) == -2          # cols % 8
    assert lib.qfp4_global_scale_rows(FAKE, 10, 16, None, None) == -1
    assert lib.qfp4_global_scale_rows(FAKE + 2, 10, 16, FAKE, None) == -3
    assert lib.qfp4_global_scale_rows(FAKE, 10, 16, FAKE + 2, None) == -3
    assert lib.qfp4_global_scale_rows(None, 0, 16, None, None) == 0            # no rows: nothing launched
    # quantisation with per-row global scales
    q = lib.qfp4_quantize_rows
    assert q(3, FAKE, 16, 256, FAKE, FAKE, FAKE, 0, None) == -1               # format
    assert q(1, FAKE, 16, 256, FAKE, FAKE, FAKE, 5, None) == -1               # layout
    assert q(1, FAKE, 16, 200, FAKE, FAKE, FAKE, 0, None) == -2               # K % 128
    assert q(1, FAKE, 16, 256, None, FAKE, FAKE, 0, None) == -1               # NVFP4 needs gs_rows
    assert q(1, FAKE, 16, 256, FAKE + 2, FAKE, FAKE, 0, None) == -3
    assert q(1, FAKE + 8, 16, 256, FAKE, FAKE, FAKE, 0, None) == -3
    assert q(1, FAKE, 0, 256, FAKE, FAKE, FAKE, 0, None) == 0                 # empty
    # GEMM with the row/column rescale
    g = lib.qfp4_gemm_nt_scaled
    base = [1, 256, 256, 256, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 0, None]

    def call(i=None, v=None):
        a = list(base)
        if i is not None:
            a[i] = v
        return g(*a)

    assert call(0, 3) == -1
    assert call(1, -1) == -1
    assert call(1, 0) == 0                                                       # empty D
    assert call(2, 100) == -2                                                    # N % 128
    assert call(10, FAKE + 2) == -3                                              # row_scale alignment
    assert call(11, FAKE + 2) == -3                                              # col_scale alignment


def test_grouped_two_level_entry_points_reject_bad_arguments(lib):
    q = lib.qfp4_quantize_grouped_rows
    assert q(2, FAKE, 10, 256, 2, FAKE, FAKE, FAKE, FAKE, None) == -1          # format
    assert q(1, FAKE, 10, 256, 0, FAKE, FAKE, FAKE, FAKE, None) == -1          # groups
    assert q(1, FAKE, 10, 200, 2, FAKE, FAKE, FAKE, FAKE, None) == -2          # K % 128
    assert q(1, FAKE, 10, 256, 2, FAKE, None, FAKE, FAKE, None) == -1          # NVFP4 needs gs_rows
    assert q(1, FAKE, 10, 256, 2, FAKE, FAKE + 2, FAKE, FAKE, None) == -3
    g = lib.qfp4_gemm_nt_grouped_scaled
    assert g(1, 0, FAKE, 10, 10, 256, 256, FAKE, FAKE, FAKE, FAKE, None, None, None, None, FAKE, None, 0,
             None) == -1
    assert g(1, 2, FAKE, 10, 10, 256, 256, FAKE, FAKE, FAKE, FAKE, None, None, FAKE + 2, None, FAKE, None, 0,
             None) == -3
    assert g(1, 2, FAKE, 10, 10, 256, 256, FAKE, FAKE, FAKE, FAKE, None, None, None, FAKE + 2, FAKE, None, 0,
             None) == -3


def test_swiglu_entry_points_reject_bad_arguments(lib):
    L = lib.qfp4_gemm_swiglu_quantize
    ok_args = dict(fmt=1, M=300, I=256, K=512, A=FAKE, Asf=FAKE, W=FAKE, Wsf=FAKE, ga=None, gw=None,
                   go=FAKE, Q=FAKE, SF=FAKE, stream=None)

    def call(**kw):
        a = dict(ok_args, **kw)
        return L(a["fmt"], a["M"], a["I"], a["K"], a["A"], a["Asf"], a["W"], a["Wsf"], a["ga"], a["gw"],
                 a["go"], a["Q"], a["SF"], a["stream"])

    assert call(fmt=2) == -1
    assert call(M=-1) == -1
    assert call(I=100) == -2                    # I % 128
    assert call(K=200) == -2
    assert call(M=0) == 0 and call(I=0) == 0     # empty H: nothing launched
    assert call(go=None) == -1                  # NVFP4 needs the output's global scale
    assert call(Q=None) == -1
    assert call(Q=FAKE + 8) == -3
    assert call(SF=FAKE + 2) == -3
    assert call(A=None) == -1
    assert call(W=FAKE + 4) == -3
    G = lib.qfp4_gemm_swiglu_quantize_grouped
    assert G(1, 2, None, 300, 256, 512, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, FAKE, FAKE, None) == -1
    assert G(1, 0, FAKE, 300, 256, 512, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, FAKE, FAKE, None) == -1
    assert G(1, 257, FAKE, 300, 256, 512, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, FAKE, FAKE, None) == -2
    assert G(1, 2, FAKE + 2, 300, 256, 512, FAKE, FAKE, FAKE, FAKE, None, None, FAKE, FAKE, FAKE, None) == -3
    assert G(0, 2, FAKE, 0, 256, 512, FAKE, FAKE, FAKE, FAKE, None, None, None, FAKE, FAKE, None) == 0


def test_test_build_probes_only_in_the_test_build(lib):
    """The encoder probes and the fault injection live in the test build only;
    the probes check their arguments on the host before any launch."""
    for name in ("qfp4_test_inject_skip_release", "qfp4_test_scale_codes", "qfp4_test_element_codes"):
        assert not hasattr(lib, name), name
    if not os.path.exists(qfp4.FAULTINJ_PATH):
        import __graft_entry__
        __graft_entry__.build()
    t = qfp4.load_fault_injection()
    dummy = 16
    assert t.qfp4_test_scale_codes(7, 0, 8, 1.0, dummy, None) == -1      # format
    assert t.qfp4_test_scale_codes(qfp4.NVFP4, 0, 8, 1.0, None, None) == -1
    assert t.qfp4_test_scale_codes(qfp4.NVFP4, 0xFFFFFFF0, 32, 1.0, dummy, None) == -1   # past 2^32
    assert t.qfp4_test_element_codes(qfp4.NVFP4, 0, 8, 0.0, dummy, None) == -1          # s = 0
    assert t.qfp4_test_element_codes(qfp4.MXFP4, 0, 8, 255.0, dummy, None) == -1        # code 255
    assert t.qfp4_test_scale_codes(qfp4.NVFP4, 0, 0, 1.0, dummy, None) == 0                         # nothing to do
