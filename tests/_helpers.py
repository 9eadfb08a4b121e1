"""Shared helpers of the test suite: device buffers, the GEMM acceptance rule
and small pipelines that drive the CUDA path through the C ABI."""
from __future__ import annotations

import numpy as np
import torch

from block_scaled_fp4_tcgen05_gb300 import qfp4

MX, NV = qfp4.MXFP4, qfp4.NVFP4

# Acceptance rule for the GEMM (per element):
#   |D_gpu - D_ref| <= 2^-8 |D_ref| + 1e-6 * T,   T = |gs_a gs_b| sum_k |a_k b_k|
REL_TOL = 2.0 ** -8
ABS_TOL_T = 1e-6


def to_dev_bf16(bits: np.ndarray) -> torch.Tensor:
    """uint16 bf16 bit patterns (host) -> bfloat16 CUDA tensor."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16).copy())
    return t.view(torch.bfloat16).cuda()


def to_dev_u8(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8).copy()).cuda()


def to_host(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy()


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def dev_scalar(x: float) -> torch.Tensor:
    return torch.tensor([np.float32(x)], dtype=torch.float32, device="cuda")


def tolerance_ratio(d_gpu: np.ndarray, d_ref: np.ndarray, t_ref: np.ndarray) -> float:
    """max over elements of err / bound (<= 1 passes); exact zero bound needs zero error."""
    err = np.abs(d_gpu - d_ref)
    bound = REL_TOL * np.abs(d_ref) + ABS_TOL_T * t_ref
    if np.any((bound == 0) & (err != 0)):
        return float("inf")
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(bound > 0, err / bound, 0.0)
    return float(r.max()) if r.size else 0.0


def assert_gemm_close(d_gpu, d_ref, t_ref, what=""):
    ratio = tolerance_ratio(d_gpu, d_ref, t_ref)
    if not ratio <= 1.0:
        err = np.abs(d_gpu - d_ref)
        bound = REL_TOL * np.abs(d_ref) + ABS_TOL_T * t_ref
        bad = np.argwhere(err > bound)
        sample = bad[:8].tolist()
        raise AssertionError(f"{what}: {len(bad)} elements out of tolerance (max ratio {ratio:.3g}); "
                             f"first {sample}: gpu {[d_gpu[tuple(i)] for i in sample]} "
                             f"ref {[d_ref[tuple(i)] for i in sample]}")
    return ratio


def run_gemm(fmt, A, A_sf_rm, B, B_sf_rm, gs_a=None, gs_b=None):
    """Host packed operands + row-major SF -> GPU GEMM (SF interleaved on the
    device) -> D as float64 host array."""
    M, N, K = A.shape[0], B.shape[0], A.shape[1] * 2
    g = qfp4.block_size(fmt)
    dA, dB = to_dev_u8(A), to_dev_u8(B)
    sfa = torch.zeros(qfp4.sf_mma_bytes(M, K // g), dtype=torch.uint8, device="cuda")
    sfb = torch.zeros(qfp4.sf_mma_bytes(N, K // g), dtype=torch.uint8, device="cuda")
    qfp4.sf_interleave(to_dev_u8(A_sf_rm), M, K // g, sfa, qfp4.SF_MMA)
    qfp4.sf_interleave(to_dev_u8(B_sf_rm), N, K // g, sfb, qfp4.SF_MMA)
    ga = dev_scalar(gs_a) if gs_a is not None else None
    gb = dev_scalar(gs_b) if gs_b is not None else None
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    ws_bytes = qfp4.gemm_workspace_bytes(fmt, M, N, K)
    ws = torch.zeros(max(ws_bytes, 1), dtype=torch.uint8, device="cuda") if ws_bytes else None
    qfp4.gemm_nt(fmt, M, N, K, dA, sfa, dB, sfb, ga, gb, D, ws, ws_bytes)
    torch.cuda.synchronize()
    assert qfp4.poll_device_status() == 0
    return bf16_to_f64(D)


def swiglu_delta(G, U, TG, TU, K):
    """Bound on |H_kernel - H| for the fused SwiGLU epilogue, from the exact
    G, U (fp64) and their sums of |a_k w_k| (TG, TU):
      - the fp32 accumulation of G and U: at most one rounding per 64-K MMA
        step of partial sums bounded by T, taken four times over for the
        tensor core's internal sums, plus the rounding of acc * gs;
      - silu's derivative lies in [-0.1, 1.1], so an error e_G in G moves
        silu(G) * U by at most 1.1 e_G (|U| + e_U), and e_U moves it by
        |silu(G)| e_U;
      - the epilogue's own arithmetic: e^-|g| (Cody-Waite reduction onto the
        hardware exp2, below 2^-22.7 relative), a reciprocal estimate with one
        correction and two products, measured below 2^-21.9 of H on GB300;
        2^-19 |H| is allowed for it."""
    from oracle import swiglu
    steps = max(1, K // 64)
    e_g = 4.0 * steps * 2.0 ** -24 * TG + 2.0 ** -22 * np.abs(G)
    e_u = 4.0 * steps * 2.0 ** -24 * TU + 2.0 ** -22 * np.abs(U)
    silu = np.abs(swiglu(G, np.ones_like(G)))
    H = swiglu(G, U)
    return 1.1 * (np.abs(U) + e_u) * e_g + silu * e_u + 2.0 ** -19 * np.abs(H)
