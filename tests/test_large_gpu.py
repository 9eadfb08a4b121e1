"""Parity past 2^31 elements: X is 131200 x 16384 BF16 (4.3 GB), so every byte
offset into X, the packed codes and the scale factors needs 64 bits.

The rows of X repeat a block of 4099 rows (an odd prime, so an offset that
wrapped at any power of two would land on a row holding other data).  The
oracle quantises that block once; the expected codes and scale bytes are its
rows repeated.  The GEMM's output rows repeat too, bit for bit (identical A
rows against the same B), and sampled outputs from every part of D, including
the first rows whose elements lie past 2^31, are checked against the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_tcgen05_gb300 import qfp4, synth
from tests._helpers import MX, NV, assert_gemm_close, to_dev_bf16, to_dev_u8, to_host

pytestmark = pytest.mark.gpu

P = 4099                             # rows in the repeated block
M, N, K = 131200, 256, 16384
FIRST_PAST_2_31 = (1 << 31) // K     # row 131072: its elements start at 2^31


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    qfp4.load()
    assert qfp4.device_check() == 0


def tile_rows(block: torch.Tensor, rows: int) -> torch.Tensor:
    """[rows, ...] device tensor whose row r is block[r % len(block)]."""
    out = torch.empty((rows,) + tuple(block.shape[1:]), dtype=block.dtype, device=block.device)
    p = block.shape[0]
    for r0 in range(0, rows, p):
        n = min(p, rows - r0)
        out[r0:r0 + n].copy_(block[:n])
    return out


@pytest.mark.parametrize("fmt", [MX, NV])
def test_past_2_31_elements(fmt):
    assert M * K > 2**31 and 2 * M * K > 2**32 and M > FIRST_PAST_2_31
    g = qfp4.block_size(fmt)

    # activations: device global scale and both SF layouts, against the oracle
    xa = synth.activations_bf16(9100 + fmt, P, K)
    X = tile_rows(to_dev_bf16(xa), M)
    gs = torch.ones(1, dtype=torch.float32, device="cuda")
    if fmt == NV:
        qfp4.global_scale(X, gs)
    Q = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
    SF = torch.empty((M, K // g), dtype=torch.uint8, device="cuda")
    Qm = torch.empty_like(Q)
    SFm = torch.empty((qfp4.sf_mma_bytes(M, K // g),), dtype=torch.uint8, device="cuda")
    qfp4.quantize(fmt, X, gs, Q, SF, qfp4.SF_ROWMAJOR)
    qfp4.quantize(fmt, X, gs, Qm, SFm, qfp4.SF_MMA)
    torch.cuda.synchronize()
    assert qfp4.poll_device_status() == 0
    del X

    # every row of the block occurs in X, so X's amax is the block's
    gs_ref = oracle.global_scale(xa) if fmt == NV else np.float32(1.0)
    assert np.float32(gs.item()) == gs_ref, "global scale"
    q_ref, sf_ref = oracle.quantize(fmt, xa, gs_ref)
    q_exp = tile_rows(to_dev_u8(q_ref), M)
    assert torch.equal(Q, q_exp), "packed codes"
    assert torch.equal(Qm, q_exp), "packed codes (MMA-layout run)"
    del q_exp, Q
    sf_full = np.ascontiguousarray(np.tile(sf_ref, (-(-M // P), 1))[:M])
    assert torch.equal(SF, to_dev_u8(sf_full)), "row-major scale bytes"
    assert np.array_equal(to_host(SFm), oracle.sf_to_mma(sf_full)), "MMA-layout scale bytes"
    del SF, sf_full

    # weights: quantised on the device, checked, then the GEMM
    xw = synth.weights_bf16(9200 + fmt, N, K)
    Xw = to_dev_bf16(xw)
    gw = torch.ones(1, dtype=torch.float32, device="cuda")
    if fmt == NV:
        qfp4.global_scale(Xw, gw)
    Bq = torch.empty((N, K // 2), dtype=torch.uint8, device="cuda")
    Bsf = torch.empty((qfp4.sf_mma_bytes(N, K // g),), dtype=torch.uint8, device="cuda")
    qfp4.quantize(fmt, Xw, gw, Bq, Bsf, qfp4.SF_MMA)
    torch.cuda.synchronize()
    gw_ref = oracle.global_scale(xw) if fmt == NV else np.float32(1.0)
    assert np.float32(gw.item()) == gw_ref
    qw_ref, sfw_ref = oracle.quantize(fmt, xw, gw_ref)
    assert np.array_equal(to_host(Bq), qw_ref)
    assert np.array_equal(to_host(Bsf), oracle.sf_to_mma(sfw_ref))

    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    qfp4.gemm_nt(fmt, M, N, K, Qm, SFm, Bq, Bsf, gs if fmt == NV else None, gw if fmt == NV else None, D)
    torch.cuda.synchronize()
    assert qfp4.poll_device_status() == 0

    # identical A rows against the same B give identical D rows
    for r0 in range(P, M, P):
        n = min(P, M - r0)
        assert torch.equal(D[r0:r0 + n], D[:n]), f"D rows {r0}..{r0 + n - 1} differ from rows 0..{n - 1}"

    gen = synth.rng(9300 + fmt)
    rows = np.array([0, P - 1, FIRST_PAST_2_31 - 1, FIRST_PAST_2_31, M - 1])
    mi = np.concatenate([gen.integers(0, M, 20000), np.repeat(rows, N)])
    ni = np.concatenate([gen.integers(0, N, 20000), np.tile(np.arange(N), len(rows))])
    d_ref, t_ref = oracle.gemm_nt_entries(fmt, q_ref, sf_ref, qw_ref, sfw_ref, gs_ref, gw_ref, mi % P, ni)
    d = D[torch.from_numpy(mi).cuda(), torch.from_numpy(ni).cuda()].float().cpu().numpy().astype(np.float64)
    assert_gemm_close(d, d_ref, t_ref, "sampled past 2^31")
