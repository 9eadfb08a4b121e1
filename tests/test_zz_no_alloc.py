"""The allocation-free GEMM entry point, qfp4_gemm_nt_noalloc, for callers
that may not allocate device memory themselves (a fixed device-memory budget
planned ahead, or a host framework whose allocator must own every
allocation).  It keeps the decode split-K scratch in a static device array
inside the library instead of a caller workspace.  Each case calls it twice
in a row through the C ABI and checks both results against qfp4_gemm_nt
with a workspace, within the GEMM tolerance of the other tests
(|D - D_ref| <= 2^-8 |D_ref| + 1e-6 sum_k |a_k b_k|); a shape whose scratch
exceeds the array must be refused with QFP4_ERR_WORKSPACE.

This file is named to be collected last: if it fails, a run that stops at
the first failure has run every other test already.  It also runs alone in a
fresh process."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_tcgen05_gb300 import qfp4, synth
from tests._helpers import MX, NV, assert_gemm_close, bf16_to_f64, dev_scalar, to_dev_u8

pytestmark = pytest.mark.gpu

QFP4_ERR_WORKSPACE = -7
SCRATCH_BYTES = (8 << 20) + 4096        # the array's size, as the header states it


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    qfp4.load()
    assert qfp4.device_check() == 0


def operands(fmt, M, N, K, seed):
    gen = synth.rng(seed)
    g = qfp4.block_size(fmt)
    A = gen.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    B = gen.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    lo, hi = (118, 136) if fmt == MX else (1, 0x7F)
    Asf = gen.integers(lo, hi, size=(M, K // g), dtype=np.uint8)
    Bsf = gen.integers(lo, hi, size=(N, K // g), dtype=np.uint8)
    dev = []
    for q, sf, rows in ((A, Asf, M), (B, Bsf, N)):
        m = torch.zeros(qfp4.sf_mma_bytes(rows, K // g), dtype=torch.uint8, device="cuda")
        qfp4.sf_interleave(to_dev_u8(sf), rows, K // g, m, qfp4.SF_MMA)
        dev += [to_dev_u8(q), m]
    return (A, Asf, B, Bsf), dev


def call_noalloc(fmt, M, N, K, dev, ga, gb, D):
    lib = qfp4.load()
    return lib.qfp4_gemm_nt_noalloc(fmt, M, N, K, dev[0].data_ptr(), dev[1].data_ptr(), dev[2].data_ptr(),
                                    dev[3].data_ptr(), ga.data_ptr() if ga is not None else None,
                                    gb.data_ptr() if gb is not None else None, D.data_ptr(),
                                    torch.cuda.current_stream().cuda_stream)


# decode shapes that split K (S = 4 and S = 8 on a GB300), a decode shape
# that does not, and a prefill shape (CTA pairs, no scratch at all)
@pytest.mark.parametrize("fmt,M,N,K", [(NV, 128, 4096, 14336), (MX, 64, 2048, 8192), (NV, 128, 14336, 4096),
                                       (NV, 300, 512, 1024)])
def test_noalloc_matches_gemm_nt(fmt, M, N, K):
    (A, Asf, B, Bsf), dev = operands(fmt, M, N, K, 6100 + M + N + K)
    gs_a, gs_b = (0.25, 1.5) if fmt == NV else (1.0, 1.0)
    ga, gb = (dev_scalar(gs_a), dev_scalar(gs_b)) if fmt == NV else (None, None)
    ws_bytes = qfp4.gemm_workspace_bytes(fmt, M, N, K)
    assert ws_bytes <= SCRATCH_BYTES
    ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")
    D_ref = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    qfp4.gemm_nt(fmt, M, N, K, dev[0], dev[1], dev[2], dev[3], ga, gb, D_ref, ws, ws_bytes)
    torch.cuda.synchronize()
    assert qfp4.poll_device_status() == 0
    d_ref = bf16_to_f64(D_ref)
    _, t = oracle.gemm_nt(fmt, A, Asf, B, Bsf, gs_a, gs_b)
    outs = []
    for _ in range(2):
        D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert call_noalloc(fmt, M, N, K, dev, ga, gb, D) == 0
        torch.cuda.synchronize()
        assert qfp4.poll_device_status() == 0
        d = bf16_to_f64(D)
        assert_gemm_close(d, d_ref, t, f"no-alloc vs qfp4_gemm_nt {M}x{N}x{K}")
        outs.append(d)
    # same kernels, same summation order: the two calls agree bit for bit
    assert np.array_equal(outs[0], outs[1])


def test_noalloc_refuses_scratch_beyond_the_array():
    """A decode shape whose split-K partials need more than the array holds
    is refused before anything is launched (D keeps its contents)."""
    fmt, M, K = NV, 128, 8192
    for N in (4864, 4608, 4352):
        if qfp4.gemm_workspace_bytes(fmt, M, N, K) > SCRATCH_BYTES:
            break
    else:
        pytest.skip("no decode shape on this GPU needs more scratch than the array holds")
    z = torch.zeros(16, dtype=torch.uint8, device="cuda")
    D = torch.full((M, N), 3.0, dtype=torch.bfloat16, device="cuda")
    assert call_noalloc(fmt, M, N, K, [z, z, z, z], None, None, D) == QFP4_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((D.float() == 3.0).all())
