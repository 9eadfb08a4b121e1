"""Thin Python binding of libqfp4.so (see include/qfp4.h).

Argument marshalling only: every function takes torch tensors (or raw
integers for pointers), passes their device addresses and sizes to the C ABI
and raises ``Qfp4Error`` on a non-zero status.  All computation happens in
the CUDA kernels of the library.  There is no fallback: if the library is
missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

MXFP4 = 0
NVFP4 = 1
NVFP4_B32 = 2
SF_ROWMAJOR = 0
SF_MMA = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqfp4.so")
_lock = threading.Lock()
_lib = None

# (restype, argtypes) per exported symbol, mirroring include/qfp4.h
_i32, _i64, _sz, _vp, _cp = ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_char_p
SIGNATURES = {
    "qfp4_version": (_i32, []),
    "qfp4_status_string": (_cp, [_i32]),
    "qfp4_device_check": (_i32, []),
    "qfp4_poll_device_status": (_i32, [_vp]),
    "qfp4_block_size": (_i32, [_i32]),
    "qfp4_sf_mma_bytes": (_sz, [_i64, _i64]),
    "qfp4_sf_mma_grouped_bytes": (_sz, [_i64, _i64, _i64]),
    "qfp4_global_scale": (_i32, [_vp, _i64, _i64, _vp, _vp]),
    "qfp4_global_scale_grouped": (_i32, [_vp, _i64, _i64, _i64, _vp, _vp, _vp]),
    "qfp4_quantize": (_i32, [_i32, _vp, _i64, _i64, _vp, _vp, _vp, _i32, _vp]),
    "qfp4_global_scale_rows": (_i32, [_vp, _i64, _i64, _vp, _vp]),
    "qfp4_quantize_rows": (_i32, [_i32, _vp, _i64, _i64, _vp, _vp, _vp, _i32, _vp]),
    "qfp4_gemm_nt_scaled": (_i32, [_i32, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                   _sz, _vp]),
    "qfp4_quantize_grouped_rows": (_i32, [_i32, _vp, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp]),
    "qfp4_gemm_nt_grouped_scaled": (_i32, [_i32, _i64, _vp, _i64, _i64, _i64, _i64, _vp, _vp, _vp, _vp,
                                           _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "qfp4_absmax_gs": (_i32, [_i64, _vp, _vp, _i64, _vp, _vp]),
    "qfp4_sparse24_meta_bytes": (_sz, [_i64, _i64, _i32]),
    "qfp4_sparse24_compress": (_i32, [_vp, _i64, _i64, _vp, _vp, _i32, _vp]),
    "qfp4_gemm_nt_sparse24": (_i32, [_i32, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                     _vp]),
    "qfp4_gemm_swiglu_quantize": (_i32, [_i32, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                         _vp]),
    "qfp4_gemm_swiglu_quantize_grouped": (_i32, [_i32, _i64, _vp, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp,
                                                 _vp, _vp, _vp, _vp, _vp]),
    "qfp4_quantize_grouped": (_i32, [_i32, _vp, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp]),
    "qfp4_residual_rmsnorm_quantize": (_i32, [_i32, _vp, _vp, _vp, _i64, _i64, ctypes.c_float, _vp, _vp, _vp,
                                              _vp, _i32, _vp]),
    "qfp4_sf_interleave": (_i32, [_vp, _i64, _i64, _vp, _i32, _vp]),
    "qfp4_gemm_workspace_bytes": (_sz, [_i32, _i64, _i64, _i64]),
    "qfp4_gemm_nt": (_i32, [_i32, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "qfp4_gemm_nt_noalloc": (_i32, [_i32, _i64, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "qfp4_gemm_nt_grouped": (_i32, [_i32, _i64, _vp, _i64, _i64, _i64, _i64, _vp, _vp, _vp, _vp,
                                    _vp, _vp, _vp, _vp, _sz, _vp]),
}


class Qfp4Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status_string(status)} ({status})")


def load() -> ctypes.CDLL:
    """Open libqfp4.so (built by build.py / __graft_entry__.build())."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libqfp4.so not built ({LIB_PATH}); run __graft_entry__.build()")
            lib = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
        return _lib


FAULTINJ_PATH = os.path.join(_HERE, "libqfp4_faultinj.so")
_faultinj = None


def load_fault_injection() -> ctypes.CDLL:
    """Open the test build (libqfp4_faultinj.so, built by
    build.build(variant="faultinj")): the same entry points with a 5 ms wait
    limit, plus qfp4_test_inject_skip_release(int) and the encoder probes
    qfp4_test_scale_codes / qfp4_test_element_codes.  For tests only; the
    product path always uses load()."""
    global _faultinj
    with _lock:
        if _faultinj is None:
            if not os.path.exists(FAULTINJ_PATH):
                raise RuntimeError(f"fault-injection build missing ({FAULTINJ_PATH})")
            lib = ctypes.CDLL(FAULTINJ_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            lib.qfp4_test_inject_skip_release.restype = _i32
            lib.qfp4_test_inject_skip_release.argtypes = [_i32]
            for name in ("qfp4_test_scale_codes", "qfp4_test_element_codes"):
                fn = getattr(lib, name)
                fn.restype = _i32
                fn.argtypes = [_i32, ctypes.c_uint32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p]
            _faultinj = lib
        return _faultinj


def status_string(status: int) -> str:
    return load().qfp4_status_string(int(status)).decode()


def _p(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, rc: int) -> None:
    if rc != 0:
        raise Qfp4Error(fn, rc)


def version() -> int:
    return load().qfp4_version()


def device_check() -> int:
    return load().qfp4_device_check()


def poll_device_status(stream=None) -> int:
    return load().qfp4_poll_device_status(_stream(stream))


def block_size(fmt: int) -> int:
    return load().qfp4_block_size(fmt)


def sf_mma_bytes(rows: int, cols: int) -> int:
    return int(load().qfp4_sf_mma_bytes(rows, cols))


def sf_mma_grouped_bytes(total_rows: int, groups: int, cols: int) -> int:
    return int(load().qfp4_sf_mma_grouped_bytes(total_rows, groups, cols))


def gemm_workspace_bytes(fmt: int, M: int, N: int, K: int) -> int:
    return int(load().qfp4_gemm_workspace_bytes(fmt, M, N, K))


def global_scale(X, gs_out, stream=None) -> None:
    rows, cols = X.shape
    _check("qfp4_global_scale",
           load().qfp4_global_scale(_p(X), rows, cols, _p(gs_out), _stream(stream)))


def global_scale_grouped(X, row_offsets, gs_out, stream=None) -> None:
    rows, cols = X.shape
    groups = row_offsets.numel() - 1
    _check("qfp4_global_scale_grouped",
           load().qfp4_global_scale_grouped(_p(X), rows, cols, groups, _p(row_offsets), _p(gs_out),
                                            _stream(stream)))


def absmax_gs(row_offsets, X, gs_out, stream=None) -> None:
    """Per-group global scales with the row count read on the device from
    row_offsets[groups]; X is [>= that many rows, K]."""
    K = X.shape[1]
    groups = row_offsets.numel() - 1
    _check("qfp4_absmax_gs",
           load().qfp4_absmax_gs(groups, _p(row_offsets), _p(X), K, _p(gs_out), _stream(stream)))


def quantize(fmt, X, gs, Q, SF, sf_layout=SF_ROWMAJOR, stream=None) -> None:
    M, K = X.shape
    _check("qfp4_quantize",
           load().qfp4_quantize(fmt, _p(X), M, K, _p(gs), _p(Q), _p(SF), sf_layout, _stream(stream)))


def global_scale_rows(X, gs_out, stream=None) -> None:
    """Per-row NVFP4 global scales: gs_out[r] = amax(row r) / (6*448)."""
    rows, cols = X.shape
    _check("qfp4_global_scale_rows",
           load().qfp4_global_scale_rows(_p(X), rows, cols, _p(gs_out), _stream(stream)))


def quantize_rows(fmt, X, gs_rows, Q, SF, sf_layout=SF_ROWMAJOR, stream=None) -> None:
    """Quantise with one global scale per row (two-level NVFP4)."""
    M, K = X.shape
    _check("qfp4_quantize_rows",
           load().qfp4_quantize_rows(fmt, _p(X), M, K, _p(gs_rows), _p(Q), _p(SF), sf_layout, _stream(stream)))


def quantize_grouped(fmt, X, row_offsets, gs, Q, SF_mma, stream=None) -> None:
    rows, K = X.shape
    groups = row_offsets.numel() - 1
    _check("qfp4_quantize_grouped",
           load().qfp4_quantize_grouped(fmt, _p(X), rows, K, groups, _p(row_offsets), _p(gs), _p(Q),
                                        _p(SF_mma), _stream(stream)))


def quantize_grouped_rows(fmt, X, row_offsets, gs_rows, Q, SF_mma, stream=None) -> None:
    """Grouped quantiser with one global scale per row (per-group MMA scale layout)."""
    rows, K = X.shape
    groups = row_offsets.numel() - 1
    _check("qfp4_quantize_grouped_rows",
           load().qfp4_quantize_grouped_rows(fmt, _p(X), rows, K, groups, _p(row_offsets), _p(gs_rows), _p(Q),
                                             _p(SF_mma), _stream(stream)))


def residual_rmsnorm_quantize(fmt, X, R, gamma, eps, Y, gs_rows, Q, SF, sf_layout=SF_MMA, stream=None) -> None:
    """y = bf16(X + R) into Y (R and Y may be None), z = RMSNorm(y) * gamma,
    per-row global scales of z into gs_rows (NVFP4) and z quantised into Q, SF."""
    M, K = X.shape
    _check("qfp4_residual_rmsnorm_quantize",
           load().qfp4_residual_rmsnorm_quantize(fmt, _p(X), _p(R), _p(gamma), M, K, float(eps), _p(Y), _p(gs_rows),
                                                 _p(Q), _p(SF), sf_layout, _stream(stream)))


def sf_interleave(SF_in, rows, cols, SF_out, layout=SF_MMA, stream=None) -> None:
    _check("qfp4_sf_interleave",
           load().qfp4_sf_interleave(_p(SF_in), rows, cols, _p(SF_out), layout, _stream(stream)))


def gemm_nt_scaled(fmt, M, N, K, A, A_sf, B, B_sf, gs_a, gs_b, row_scale, col_scale, D, workspace=None,
                   ws_bytes=0, stream=None) -> None:
    """The GEMM with the two-level epilogue: row m of D times row_scale[m],
    column n times col_scale[n] (either may be None)."""
    _check("qfp4_gemm_nt_scaled",
           load().qfp4_gemm_nt_scaled(fmt, M, N, K, _p(A), _p(A_sf), _p(B), _p(B_sf), _p(gs_a), _p(gs_b),
                                      _p(row_scale), _p(col_scale), _p(D), _p(workspace), ws_bytes,
                                      _stream(stream)))


def gemm_nt(fmt, M, N, K, A, A_sf, B, B_sf, gs_a, gs_b, D, workspace=None, ws_bytes=0,
            stream=None) -> None:
    _check("qfp4_gemm_nt",
           load().qfp4_gemm_nt(fmt, M, N, K, _p(A), _p(A_sf), _p(B), _p(B_sf), _p(gs_a), _p(gs_b),
                               _p(D), _p(workspace), ws_bytes, _stream(stream)))


def gemm_nt_grouped(fmt, row_offsets, total_rows, max_group_rows, N, K, A, A_sf, B, B_sf,
                    gs_a, gs_b, D, workspace=None, ws_bytes=0, stream=None) -> None:
    groups = row_offsets.numel() - 1
    _check("qfp4_gemm_nt_grouped",
           load().qfp4_gemm_nt_grouped(fmt, groups, _p(row_offsets), total_rows, max_group_rows, N, K,
                                       _p(A), _p(A_sf), _p(B), _p(B_sf), _p(gs_a), _p(gs_b), _p(D),
                                       _p(workspace), ws_bytes, _stream(stream)))


def gemm_nt_grouped_scaled(fmt, row_offsets, total_rows, max_group_rows, N, K, A, A_sf, B, B_sf,
                           gs_a, gs_b, row_scale, col_scale, D, workspace=None, ws_bytes=0,
                           stream=None) -> None:
    """Grouped GEMM with the two-level epilogue: row m times row_scale[m],
    column n of group e times col_scale[e*N + n] (either may be None)."""
    groups = row_offsets.numel() - 1
    _check("qfp4_gemm_nt_grouped_scaled",
           load().qfp4_gemm_nt_grouped_scaled(fmt, groups, _p(row_offsets), total_rows, max_group_rows, N, K,
                                              _p(A), _p(A_sf), _p(B), _p(B_sf), _p(gs_a), _p(gs_b),
                                              _p(row_scale), _p(col_scale), _p(D), _p(workspace), ws_bytes,
                                              _stream(stream)))


def sparse24_meta_bytes(rows: int, K: int, layout: int = SF_MMA) -> int:
    return int(load().qfp4_sparse24_meta_bytes(rows, K, layout))


def sparse24_compress(W, W_comp, W_meta, layout=SF_MMA, stream=None) -> None:
    """2:4 pair-sparse packed W [rows, K/2] -> kept bytes [rows, K/4] and metadata."""
    rows, K = W.shape[0], W.shape[1] * 2
    _check("qfp4_sparse24_compress",
           load().qfp4_sparse24_compress(_p(W), rows, K, _p(W_comp), _p(W_meta), layout, _stream(stream)))


def gemm_nt_sparse24(fmt, M, N, K, X, X_sf, W_comp, W_meta, W_sf, gs_x, gs_w, D, row_scale=None, col_scale=None,
                     stream=None) -> None:
    _check("qfp4_gemm_nt_sparse24",
           load().qfp4_gemm_nt_sparse24(fmt, M, N, K, _p(X), _p(X_sf), _p(W_comp), _p(W_meta), _p(W_sf), _p(gs_x),
                                        _p(gs_w), _p(row_scale), _p(col_scale), _p(D), _stream(stream)))


def gemm_swiglu_quantize(fmt, M, I, K, A, A_sf, W, W_sf, gs_a, gs_w, gs_out, Q_out, SF_out,
                         stream=None) -> None:
    """Up-projection with SwiGLU, requantised: W holds the gate and up rows
    interleaved in groups of the block size; writes H = silu(gate) * up
    quantised into Q_out [M, I/2] and SF_out (MMA layout for [M, I/g])."""
    _check("qfp4_gemm_swiglu_quantize",
           load().qfp4_gemm_swiglu_quantize(fmt, M, I, K, _p(A), _p(A_sf), _p(W), _p(W_sf), _p(gs_a), _p(gs_w),
                                            _p(gs_out), _p(Q_out), _p(SF_out), _stream(stream)))


def gemm_swiglu_quantize_grouped(fmt, row_offsets, total_rows, I, K, A, A_sf, W, W_sf, gs_a, gs_w, gs_out,
                                 Q_out, SF_out, stream=None) -> None:
    """Per-expert version; SF_out in the per-group MMA layout."""
    groups = row_offsets.numel() - 1
    _check("qfp4_gemm_swiglu_quantize_grouped",
           load().qfp4_gemm_swiglu_quantize_grouped(fmt, groups, _p(row_offsets), total_rows, I, K, _p(A),
                                                    _p(A_sf), _p(W), _p(W_sf), _p(gs_a), _p(gs_w), _p(gs_out),
                                                    _p(Q_out), _p(SF_out), _stream(stream)))
