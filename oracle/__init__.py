"""CPU oracle for block-scaled FP4 -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does.

This module is argument marshalling around ``oracle.c`` (plain C, built with
gcc, no code shared with the CUDA library).  The arithmetic lives in the C
file; see its header for the definitions and the pages they follow.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

MXFP4 = 0
NVFP4 = 1
NVFP4_B32 = 2       # NVFP4 with one UE4M3 scale per 32 elements (the 2:4-sparse path)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def _paths():
    """Source and library to use.  QFP4_ORACLE_SOURCE names a modified copy
    of oracle.c (the pin suite's planted-mistake check builds one per
    mistake); its library is built beside it, never over the real one."""
    src = os.environ.get("QFP4_ORACLE_SOURCE")
    if src:
        src = os.path.abspath(src)
        return src, os.path.join(os.path.dirname(src), "liboracle.so")
    return _SRC, _LIB_PATH


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library (gcc, OpenMP, strict IEEE fp32)."""
    src, lib_path = _paths()
    os.makedirs(os.path.dirname(lib_path), exist_ok=True)
    stale = (not os.path.exists(lib_path)
             or os.path.getmtime(lib_path) < os.path.getmtime(src))
    if force or stale:
        tmp = lib_path + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-shared", "-fPIC", "-o", tmp, src, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, lib_path)
    return lib_path


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        c_i64, c_int, c_f, c_d, c_p = (ctypes.c_int64, ctypes.c_int, ctypes.c_float,
                                       ctypes.c_double, ctypes.c_void_p)
        sigs = {
            "oracle_e2m1_value": (c_d, [c_int]),
            "oracle_ue8m0_value": (c_d, [c_int]),
            "oracle_ue4m3_value": (c_d, [c_int]),
            "oracle_scale_value": (c_d, [c_int, c_int]),
            "oracle_block_size": (c_int, [c_int]),
            "oracle_e2m1_round": (c_int, [c_f]),
            "oracle_ue4m3_round": (c_int, [c_f]),
            "oracle_ue8m0_round": (c_int, [c_f]),
            "oracle_scale_round": (c_int, [c_int, c_f]),
            "oracle_global_scale": (c_f, [c_p, c_i64]),
            "oracle_global_scale_bf16": (c_f, [c_p, c_i64]),
            "oracle_quantize_f32": (c_int, [c_int, c_p, c_i64, c_i64, c_f, c_p, c_p]),
            "oracle_quantize_bf16": (c_int, [c_int, c_p, c_i64, c_i64, c_f, c_p, c_p]),
            "oracle_dequantize": (c_int, [c_int, c_p, c_p, c_i64, c_i64, c_f, c_p]),
            "oracle_sf_mma_bytes": (c_i64, [c_i64, c_i64]),
            "oracle_sf_to_mma": (c_int, [c_p, c_i64, c_i64, c_p]),
            "oracle_sf_from_mma": (c_int, [c_p, c_i64, c_i64, c_p]),
            "oracle_gemm_nt": (c_int, [c_int, c_i64, c_i64, c_i64, c_p, c_p, c_p, c_p,
                                       c_f, c_f, c_p, c_p]),
            "oracle_gemm_nt_entries": (c_int, [c_int, c_i64, c_p, c_p, c_p, c_p, c_f, c_f,
                                               c_i64, c_p, c_p, c_p, c_p]),
            "oracle_global_scale_rows_bf16": (c_int, [c_p, c_i64, c_i64, c_p]),
            "oracle_quantize_bf16_rows": (c_int, [c_int, c_p, c_i64, c_i64, c_p, c_p, c_p]),
            "oracle_gemm_nt_scaled": (c_int, [c_int, c_i64, c_i64, c_i64, c_p, c_p, c_p, c_p,
                                              c_f, c_f, c_p, c_p, c_p, c_p]),
            "oracle_gemm_nt_scaled_entries": (c_int, [c_int, c_i64, c_p, c_p, c_p, c_p, c_f, c_f, c_p, c_p,
                                                      c_i64, c_p, c_p, c_p, c_p]),
            "oracle_swiglu_f64": (c_int, [c_p, c_p, c_i64, c_p]),
            "oracle_residual_rmsnorm": (c_int, [c_p, c_p, c_p, c_i64, c_i64, c_d, c_p, c_p, c_p]),
            "oracle_sparse24_decompress": (c_int, [c_p, c_p, c_i64, c_i64, c_p]),
            "oracle_sparse24_compress": (c_int, [c_p, c_i64, c_i64, c_p, c_p]),
            "oracle_e2m1_round_n": (c_int, [c_p, c_i64, c_p]),
            "oracle_scale_round_n": (c_int, [c_int, c_p, c_i64, c_p]),
            "oracle_num_threads": (c_int, []),
            "oracle_set_num_threads": (None, [c_int]),
            "oracle_scale_codes_bits": (c_int, [c_int, ctypes.c_uint32, c_i64, ctypes.c_float, c_p]),
            "oracle_element_codes_bits": (c_int, [ctypes.c_uint32, c_i64, ctypes.c_float, c_p]),
        }
        for name, (res, args) in sigs.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def block_size(fmt: int) -> int:
    return _load().oracle_block_size(fmt)


# ---- scalar format functions -------------------------------------------------

def e2m1_value(code: int) -> float:
    return _load().oracle_e2m1_value(int(code))


def ue8m0_value(byte: int) -> float:
    return _load().oracle_ue8m0_value(int(byte))


def ue4m3_value(byte: int) -> float:
    return _load().oracle_ue4m3_value(int(byte))


def scale_value(fmt: int, byte: int) -> float:
    return _load().oracle_scale_value(int(fmt), int(byte))


def e2m1_round(q: float) -> int:
    return _load().oracle_e2m1_round(float(np.float32(q)))


def ue4m3_round(t: float) -> int:
    return _load().oracle_ue4m3_round(float(np.float32(t)))


def ue8m0_round(t: float) -> int:
    return _load().oracle_ue8m0_round(float(np.float32(t)))


def e2m1_round_array(q: np.ndarray) -> np.ndarray:
    """Vector form of e2m1_round, one C call per element (fp32 input)."""
    lib = _load()
    q = np.ascontiguousarray(q, dtype=np.float32).ravel()
    return np.fromiter((lib.oracle_e2m1_round(float(v)) for v in q), dtype=np.uint8, count=q.size)


# ---- tensors -----------------------------------------------------------------

def global_scale(x: np.ndarray) -> np.float32:
    """gs = amax / (6*448) in fp32.  ``x`` is fp32, or bf16 bits as uint16."""
    lib = _load()
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        return np.float32(lib.oracle_global_scale_bf16(_ptr(x), x.size))
    x = x.astype(np.float32, copy=False)
    return np.float32(lib.oracle_global_scale(_ptr(x), x.size))


def global_scale_rows(x: np.ndarray) -> np.ndarray:
    """Per-row gs[m] = amax of row m / (6*448) (fp32 [M]); ``x`` is bf16 bits as uint16."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.uint16)
    M, K = x.shape
    gs = np.zeros(M, dtype=np.float32)
    if lib.oracle_global_scale_rows_bf16(_ptr(x), M, K, _ptr(gs)) != 0:
        raise ValueError("bad shape")
    return gs


def quantize(fmt: int, x: np.ndarray, gs=1.0):
    """x [M, K] fp32, or bf16 bits as uint16 -> (Q uint8 [M, K/2], SF uint8 [M, K/g]).
    ``gs`` is one global scale, or (bf16 input) an array of one per row."""
    lib = _load()
    x = np.ascontiguousarray(x)
    M, K = x.shape
    g = block_size(fmt)
    Q = np.zeros((M, K // 2), dtype=np.uint8)
    SF = np.zeros((M, K // g), dtype=np.uint8)
    if np.ndim(gs) == 1:
        if x.dtype != np.uint16:
            raise ValueError("per-row global scales take bf16 input")
        gsr = np.ascontiguousarray(gs, dtype=np.float32)
        assert gsr.size == M
        if lib.oracle_quantize_bf16_rows(fmt, _ptr(x), M, K, _ptr(gsr), _ptr(Q), _ptr(SF)) != 0:
            raise ValueError("oracle quantize rejected its input (shape or non-finite value)")
        return Q, SF
    if x.dtype == np.uint16:
        rc = lib.oracle_quantize_bf16(fmt, _ptr(x), M, K, float(np.float32(gs)), _ptr(Q), _ptr(SF))
    else:
        x = np.ascontiguousarray(x, dtype=np.float32)
        rc = lib.oracle_quantize_f32(fmt, _ptr(x), M, K, float(np.float32(gs)), _ptr(Q), _ptr(SF))
    if rc != 0:
        raise ValueError("oracle quantize rejected its input (shape or non-finite value)")
    return Q, SF


def dequantize(fmt: int, Q: np.ndarray, SF: np.ndarray, gs: float = 1.0) -> np.ndarray:
    lib = _load()
    Q = np.ascontiguousarray(Q, dtype=np.uint8)
    SF = np.ascontiguousarray(SF, dtype=np.uint8)
    M = Q.shape[0]
    K = Q.shape[1] * 2
    _check_sf(fmt, SF, M, K)
    X = np.zeros((M, K), dtype=np.float64)
    if lib.oracle_dequantize(fmt, _ptr(Q), _ptr(SF), M, K, float(np.float32(gs)), _ptr(X)) != 0:
        raise ValueError("bad shape")
    return X


def sf_mma_bytes(rows: int, cols: int) -> int:
    return int(_load().oracle_sf_mma_bytes(rows, cols))


def sf_to_mma(SF: np.ndarray) -> np.ndarray:
    lib = _load()
    SF = np.ascontiguousarray(SF, dtype=np.uint8)
    rows, cols = SF.shape
    out = np.zeros(sf_mma_bytes(rows, cols), dtype=np.uint8)
    lib.oracle_sf_to_mma(_ptr(SF), rows, cols, _ptr(out))
    return out


def sf_from_mma(buf: np.ndarray, rows: int, cols: int) -> np.ndarray:
    lib = _load()
    buf = np.ascontiguousarray(buf, dtype=np.uint8)
    assert buf.size >= sf_mma_bytes(rows, cols)
    out = np.zeros((rows, cols), dtype=np.uint8)
    lib.oracle_sf_from_mma(_ptr(buf), rows, cols, _ptr(out))
    return out


def _opt_f32(v, n):
    if v is None:
        return None, None
    a = np.ascontiguousarray(v, dtype=np.float32)
    assert a.size == n
    return a, _ptr(a)


def _check_sf(fmt: int, sf: np.ndarray, rows: int, K: int):
    """Scale factors must be row-major [rows, K/g] for the format's block g."""
    g = block_size(fmt)
    if K % g != 0 or sf.size != rows * (K // g):
        raise ValueError(f"scale factors: {sf.size} bytes for [{rows}, {K}/{g}]")


def gemm_nt(fmt: int, A: np.ndarray, A_sf: np.ndarray, B: np.ndarray, B_sf: np.ndarray,
            gs_a: float = 1.0, gs_b: float = 1.0, row_scale=None, col_scale=None):
    """Full reference GEMM. Returns (D fp64 [M,N], T fp64 [M,N]); SF row-major.
    ``row_scale`` [M] and ``col_scale`` [N] (fp32, optional) rescale row m and
    column n of D (the two-level epilogue)."""
    lib = _load()
    A, A_sf, B, B_sf = (np.ascontiguousarray(v, dtype=np.uint8) for v in (A, A_sf, B, B_sf))
    M, N, K = A.shape[0], B.shape[0], A.shape[1] * 2
    _check_sf(fmt, A_sf, M, K)
    _check_sf(fmt, B_sf, N, K)
    D = np.zeros((M, N), dtype=np.float64)
    T = np.zeros((M, N), dtype=np.float64)
    if row_scale is not None or col_scale is not None:
        rs, rsp = _opt_f32(row_scale, M)
        cs, csp = _opt_f32(col_scale, N)
        rc = lib.oracle_gemm_nt_scaled(fmt, M, N, K, _ptr(A), _ptr(A_sf), _ptr(B), _ptr(B_sf),
                                       float(np.float32(gs_a)), float(np.float32(gs_b)), rsp, csp,
                                       _ptr(D), _ptr(T))
        if rc != 0:
            raise ValueError("bad shape")
        return D, T
    rc = lib.oracle_gemm_nt(fmt, M, N, K, _ptr(A), _ptr(A_sf), _ptr(B), _ptr(B_sf),
                            float(np.float32(gs_a)), float(np.float32(gs_b)), _ptr(D), _ptr(T))
    if rc != 0:
        raise ValueError("bad shape")
    return D, T


def gemm_nt_entries(fmt: int, A, A_sf, B, B_sf, gs_a, gs_b, mi, ni, row_scale=None, col_scale=None):
    """Reference values at sampled (m, n) positions. Returns (D, T) fp64 [count]."""
    lib = _load()
    A, A_sf, B, B_sf = (np.ascontiguousarray(v, dtype=np.uint8) for v in (A, A_sf, B, B_sf))
    K = A.shape[1] * 2
    _check_sf(fmt, A_sf, A.shape[0], K)
    _check_sf(fmt, B_sf, B.shape[0], K)
    mi = np.ascontiguousarray(mi, dtype=np.int64)
    ni = np.ascontiguousarray(ni, dtype=np.int64)
    if mi.size != ni.size or (mi.size and (mi.min() < 0 or mi.max() >= A.shape[0]
                                           or ni.min() < 0 or ni.max() >= B.shape[0])):
        raise ValueError("sampled positions out of range")
    D = np.zeros(mi.size, dtype=np.float64)
    T = np.zeros(mi.size, dtype=np.float64)
    if row_scale is not None or col_scale is not None:
        rs, rsp = _opt_f32(row_scale, A.shape[0])
        cs, csp = _opt_f32(col_scale, B.shape[0])
        rc = lib.oracle_gemm_nt_scaled_entries(fmt, K, _ptr(A), _ptr(A_sf), _ptr(B), _ptr(B_sf),
                                               float(np.float32(gs_a)), float(np.float32(gs_b)), rsp, csp,
                                               mi.size, _ptr(mi), _ptr(ni), _ptr(D), _ptr(T))
        if rc != 0:
            raise ValueError("bad shape")
        return D, T
    rc = lib.oracle_gemm_nt_entries(fmt, K, _ptr(A), _ptr(A_sf), _ptr(B), _ptr(B_sf),
                                    float(np.float32(gs_a)), float(np.float32(gs_b)),
                                    mi.size, _ptr(mi), _ptr(ni), _ptr(D), _ptr(T))
    if rc != 0:
        raise ValueError("bad shape")
    return D, T


# ---- SwiGLU of the MoE up-projection, and its requantisation ------------------

def swiglu(G: np.ndarray, U: np.ndarray) -> np.ndarray:
    """H = silu(G) * U = G * U / (1 + exp(-G)), elementwise in fp64."""
    lib = _load()
    G = np.ascontiguousarray(G, dtype=np.float64)
    U = np.ascontiguousarray(U, dtype=np.float64)
    if G.shape != U.shape:
        raise ValueError("gate and up outputs differ in shape")
    H = np.zeros(G.shape, dtype=np.float64)
    if lib.oracle_swiglu_f64(_ptr(G), _ptr(U), G.size, _ptr(H)) != 0:
        raise ValueError("bad size")
    return H


def swiglu_up(fmt: int, A, A_sf, Wg, Wg_sf, Wu, Wu_sf, gs_a: float = 1.0, gs_w: float = 1.0):
    """Exact output of an up-projection with SwiGLU: tokens A [M, K/2], gate
    and up weight rows Wg, Wu [I, K/2], all with row-major scale factors.
        G = gemm_nt(A, Wg),  U = gemm_nt(A, Wu)   (exact sums, times gs_a gs_w)
        H = silu(G) * U
    Returns (H, G, U, TG, TU), fp64 [M, I]; TG and TU are the scaled sums of
    |a_k w_k| in which the GEMM's accumulation error is bounded."""
    G, TG = gemm_nt(fmt, A, A_sf, Wg, Wg_sf, gs_a, gs_w)
    U, TU = gemm_nt(fmt, A, A_sf, Wu, Wu_sf, gs_a, gs_w)
    return swiglu(G, U), G, U, TG, TU


def swiglu_requantize(fmt: int, H: np.ndarray, gs2: float = 1.0):
    """The requantised SwiGLU output: H rounded to fp32, then the quantiser's
    rule with the next layer's activation global scale gs2 (NVFP4; MXFP4 has
    none).  Returns (Q [M, I/2], SF row-major [M, I/g])."""
    return quantize(fmt, np.asarray(H, dtype=np.float64).astype(np.float32), gs2)


def _e2m1_round_n(q: np.ndarray) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.float32)
    out = np.zeros(q.shape, dtype=np.uint8)
    _load().oracle_e2m1_round_n(_ptr(q), q.size, _ptr(out))
    return out


def _scale_round_n(fmt: int, t: np.ndarray) -> np.ndarray:
    t = np.ascontiguousarray(t, dtype=np.float32)
    out = np.zeros(t.shape, dtype=np.uint8)
    _load().oracle_scale_round_n(fmt, _ptr(t), t.size, _ptr(out))
    return out


def _f32_down(x: np.ndarray) -> np.ndarray:
    """Largest fp32 value <= x (elementwise, x fp64)."""
    y = x.astype(np.float32)
    return np.where(y.astype(np.float64) > x, np.nextafter(y, np.float32(-np.inf)), y)


def _f32_up(x: np.ndarray) -> np.ndarray:
    """Smallest fp32 value >= x."""
    y = x.astype(np.float32)
    return np.where(y.astype(np.float64) < x, np.nextafter(y, np.float32(np.inf)), y)


def requant_valid(fmt: int, Q: np.ndarray, SF: np.ndarray, H: np.ndarray, delta: np.ndarray,
                  gs2=1.0, gs2_hi=None) -> np.ndarray:
    """Which blocks of a quantised matrix are what the quantiser's rule gives
    for SOME fp32 matrix within delta of H (elementwise), and some global
    scale in [gs2, gs2_hi]?

    Where the value being quantised comes out of an fp32 computation, only H
    (exact) and a bound delta on the distance are known; any fp32 value in
    [H - delta, H + delta] is then a correct input.  Where the global scale is
    itself computed that way (an amax over the row), it is known only to lie
    in an interval; gs2_hi = None means it is exactly gs2.  The rule is
    monotone in every step, so a block passes when
      - its scale byte lies between the codes the rule gives for the smallest
        block amax over the largest scale and the largest amax over the
        smallest scale, and
      - with the scales s that byte gives over the interval, each element's
        code lies between the codes of the smallest and the largest quotient
        of its range by s (codes ordered along the real line, -0 just below
        +0); if s is 0 every code must be 0.
    Q [M, I/2] packed, SF row-major [M, I/g], H and delta fp64 [M, I]; gs2
    and gs2_hi scalars or per-row arrays [M], > 0 (NVFP4; ignored for
    MXFP4).  Returns a bool mask [M, I/g]."""
    g = block_size(fmt)
    H = np.asarray(H, dtype=np.float64)
    delta = np.asarray(delta, dtype=np.float64)
    M, I = H.shape
    if I % g or Q.shape != (M, I // 2) or SF.shape != (M, I // g) or delta.shape != H.shape:
        raise ValueError("shapes")
    if np.any(delta < 0) or not np.all(np.isfinite(H)):
        raise ValueError("delta must be >= 0 and H finite")

    def per_row(v):
        a = np.asarray(v, dtype=np.float32)
        return np.broadcast_to(a.reshape(-1, 1) if a.ndim else a, (M, 1)).astype(np.float32)

    if fmt == MXFP4:
        gs_lo = gs_hi = per_row(1.0)
    else:
        gs_lo = per_row(gs2)
        gs_hi = gs_lo if gs2_hi is None else per_row(gs2_hi)
    if not (np.all(gs_lo > 0) and np.all(gs_hi >= gs_lo)):
        raise ValueError("the global scales must be positive and gs2 <= gs2_hi")
    lo, hi = _f32_down(H - delta), _f32_up(H + delta)
    a_small = np.where((lo <= 0) & (hi >= 0), np.float32(0), np.minimum(np.abs(lo), np.abs(hi)))
    a_large = np.maximum(np.abs(lo), np.abs(hi))
    amax_lo = a_small.reshape(M, I // g, g).max(axis=-1)
    amax_hi = a_large.reshape(M, I // g, g).max(axis=-1)
    six = np.float32(6.0)
    code_lo = _scale_round_n(fmt, (amax_lo / six) / gs_hi)
    code_hi = _scale_round_n(fmt, (amax_hi / six) / gs_lo)
    sf_ok = (SF >= code_lo) & (SF <= code_hi)
    table = np.array([scale_value(fmt, b) for b in range(256)], dtype=np.float64)
    with np.errstate(invalid="ignore", divide="ignore", over="ignore"):
        dec = table[SF].astype(np.float32)
        s_lo = np.repeat(dec * gs_lo, g, axis=1)
        s_hi = np.repeat(dec * gs_hi, g, axis=1)
        zero = s_hi == 0
        finite = np.isfinite(s_lo) & np.isfinite(s_hi)
        one = np.float32(1)
        sl = np.where(zero | ~finite, one, s_lo)
        sh = np.where(zero | ~finite, one, s_hi)
        corners = np.stack([lo / sl, lo / sh, hi / sl, hi / sh])
        c_lo = _e2m1_round_n(corners.min(axis=0))
        c_hi = _e2m1_round_n(corners.max(axis=0))
    key = np.array([4.0 * e2m1_value(c) for c in range(16)])
    key[8] = -1.0                                    # -0 sits just below +0
    nib = np.stack([Q & 15, Q >> 4], axis=-1).reshape(M, I)
    el_ok = np.where(zero, nib == 0, (key[c_lo] <= key[nib]) & (key[nib] <= key[c_hi]))
    el_ok &= finite
    return sf_ok & el_ok.reshape(M, I // g, g).all(axis=-1)


# ---- residual add and RMSNorm in front of the quantiser ------------------------

def residual_rmsnorm(x: np.ndarray, r, gamma: np.ndarray, eps: float = 1e-6):
    """y = bf16(x + r) (the new residual stream; r may be None), and
    z = y / sqrt(mean(y^2) + eps) * gamma in fp64.  x, r: bf16 bits [M, K];
    gamma: bf16 bits [K].  Returns (y bf16 bits [M, K], z fp64 [M, K],
    1/rms fp64 [M])."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.uint16)
    M, K = x.shape
    gamma = np.ascontiguousarray(gamma, dtype=np.uint16)
    if gamma.shape != (K,):
        raise ValueError("gamma must be [K]")
    rp = None
    if r is not None:
        r = np.ascontiguousarray(r, dtype=np.uint16)
        if r.shape != x.shape:
            raise ValueError("residual shape")
        rp = _ptr(r)
    y = np.zeros((M, K), dtype=np.uint16)
    z = np.zeros((M, K), dtype=np.float64)
    inv = np.zeros(M, dtype=np.float64)
    if lib.oracle_residual_rmsnorm(_ptr(x), rp, _ptr(gamma), M, K, float(eps), _ptr(y), _ptr(z), _ptr(inv)) != 0:
        raise ValueError("bad arguments")
    return y, z, inv


def rows_global_scale_exact(z: np.ndarray) -> np.ndarray:
    """The two-level rule's per-row global scale of an exact fp64 matrix:
    amax over the row / (6 * 448), in fp64 (a kernel computes it in fp32
    from its own z)."""
    return np.abs(np.asarray(z, dtype=np.float64)).max(axis=1) / 2688.0


# ---- 2:4 pair-granular sparse operand ------------------------------------------

def sparse24_decompress(Wc: np.ndarray, meta: np.ndarray, K: int) -> np.ndarray:
    """Compressed rows Wc [rows, K/4] and metadata [rows, K/16] -> the dense
    packed operand [rows, K/2] (two kept pairs of every four, see oracle.c)."""
    Wc = np.ascontiguousarray(Wc, dtype=np.uint8)
    meta = np.ascontiguousarray(meta, dtype=np.uint8)
    rows = Wc.shape[0]
    if Wc.shape != (rows, K // 4) or meta.shape != (rows, K // 16):
        raise ValueError("shapes")
    W = np.zeros((rows, K // 2), dtype=np.uint8)
    if _load().oracle_sparse24_decompress(_ptr(Wc), _ptr(meta), rows, K, _ptr(W)) != 0:
        raise ValueError("bad metadata (needs i0 < i1 in every group) or K % 16 != 0")
    return W


def sparse24_compress(W: np.ndarray):
    """Dense packed operand [rows, K/2] with at most two non-zero pairs in
    every group of four -> (Wc [rows, K/4], meta [rows, K/16])."""
    W = np.ascontiguousarray(W, dtype=np.uint8)
    rows, K = W.shape[0], W.shape[1] * 2
    Wc = np.zeros((rows, K // 4), dtype=np.uint8)
    meta = np.zeros((rows, K // 16), dtype=np.uint8)
    if _load().oracle_sparse24_compress(_ptr(W), rows, K, _ptr(Wc), _ptr(meta)) != 0:
        raise ValueError("a group holds more than two non-zero pairs, or K % 16 != 0")
    return Wc, meta


def gemm_nt_sparse24(fmt: int, A, A_sf, Wc, meta, W_sf, gs_a: float = 1.0, gs_w: float = 1.0):
    """D = A @ W^T with W given 2:4 pair-sparse: the dense GEMM of the
    decompressed operand (its scale factors are those of the dense K)."""
    K = np.asarray(A).shape[1] * 2
    return gemm_nt(fmt, A, A_sf, sparse24_decompress(Wc, meta, K), W_sf, gs_a, gs_w)


def scale_codes_bits(fmt: int, first: int, n: int, gs=1.0) -> np.ndarray:
    """Scale bytes the quantiser's rule gives for amax = the floats whose
    bit patterns are first .. first + n - 1 (no NaN or Inf among them)."""
    out = np.empty(n, dtype=np.uint8)
    if _load().oracle_scale_codes_bits(fmt, first, n, float(np.float32(gs)), _ptr(out)) != 0:
        raise ValueError("bad range")
    return out


def element_codes_bits(first: int, n: int, s) -> np.ndarray:
    """E2M1 codes of x / s for x = the floats whose bit patterns are first ..
    first + n - 1 (no NaN or Inf among them), block scale s > 0."""
    out = np.empty(n, dtype=np.uint8)
    if _load().oracle_element_codes_bits(first, n, float(np.float32(s)), _ptr(out)) != 0:
        raise ValueError("bad range or scale")
    return out


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Thread count of the oracle's OpenMP loops (for timing it on n cores)."""
    _load().oracle_set_num_threads(int(n))
