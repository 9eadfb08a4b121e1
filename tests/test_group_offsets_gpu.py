"""Grouped calls with unusable device row offsets: every grouped kernel checks
the offsets before it touches its outputs (start at 0, never decrease, end at
the row count the host passed, no group above max_group_rows for the GEMMs).
A failing check must leave the outputs as they were and make the status poll
return QFP4_ERR_INVALID_ARG; the next poll is clean again."""
import numpy as np
import pytest
import torch

from block_scaled_fp4_tcgen05_gb300 import qfp4, synth
from tests._helpers import NV, MX, to_dev_bf16

pytestmark = pytest.mark.gpu

INVALID = -1
ROWS, K = 300, 512


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    qfp4.load()
    assert qfp4.device_check() == 0
    torch.cuda.synchronize()
    qfp4.poll_device_status()        # start from a clean status word


def bad_offsets():
    return {
        "end_past_rows": [0, 100, 200, ROWS + 1],
        "end_short": [0, 100, 200, ROWS - 1],
        "start_not_zero": [1, 100, 200, ROWS],
        "decreasing": [0, 200, 100, ROWS],
    }


def dev_offs(o):
    return torch.tensor(o, dtype=torch.int32, device="cuda")


def expect_invalid_then_clean():
    torch.cuda.synchronize()
    assert qfp4.poll_device_status() == INVALID
    assert qfp4.poll_device_status() == 0


def filled(shape, dtype, value):
    t = torch.empty(shape, dtype=dtype, device="cuda")
    t.view(torch.uint8).fill_(value)
    return t


@pytest.mark.parametrize("case", sorted(bad_offsets()))
@pytest.mark.parametrize("fmt", [MX, NV])
def test_grouped_quantiser_and_scales(case, fmt):
    offs = dev_offs(bad_offsets()[case])
    groups = offs.numel() - 1
    g = qfp4.block_size(fmt)
    X = to_dev_bf16(synth.activations_bf16(synth.SEED_BASE + 900, ROWS, K))
    gs = torch.ones(groups, dtype=torch.float32, device="cuda")
    Q = filled((ROWS, K // 2), torch.uint8, 0xAB)
    SF = filled((qfp4.sf_mma_grouped_bytes(ROWS, groups, K // g),), torch.uint8, 0xCD)
    qfp4.quantize_grouped(fmt, X, offs, gs, Q, SF)
    expect_invalid_then_clean()
    assert torch.all(Q == 0xAB), "codes written despite bad offsets"
    assert torch.all(SF == 0), "scale buffer must hold the zeros the call clears it to"
    if fmt == NV:
        gs_rows = torch.ones(ROWS, dtype=torch.float32, device="cuda")
        qfp4.quantize_grouped_rows(NV, X, offs, gs_rows, Q, SF)
        expect_invalid_then_clean()
        assert torch.all(Q == 0xAB)
        gs_out = torch.full((groups,), 7.0, dtype=torch.float32, device="cuda")
        qfp4.global_scale_grouped(X, offs, gs_out)
        expect_invalid_then_clean()
        assert torch.all(gs_out == 0.0), "skipped groups read as amax 0"
        if case in ("start_not_zero", "decreasing"):
            # the row count comes from offs[groups]; only the other checks apply
            gs_out.fill_(7.0)
            qfp4.absmax_gs(offs, X, gs_out)
            expect_invalid_then_clean()
            assert torch.all(gs_out == 0.0)


def grouped_operands(fmt, groups, N):
    g = qfp4.block_size(fmt)
    A = torch.zeros((ROWS, K // 2), dtype=torch.uint8, device="cuda")
    Asf = torch.zeros((qfp4.sf_mma_grouped_bytes(ROWS, groups, K // g),), dtype=torch.uint8, device="cuda")
    B = torch.zeros((groups * N, K // 2), dtype=torch.uint8, device="cuda")
    Bsf = torch.zeros((groups * qfp4.sf_mma_bytes(N, K // g),), dtype=torch.uint8, device="cuda")
    return A, Asf, B, Bsf


@pytest.mark.parametrize("case", sorted(bad_offsets()) + ["group_above_max"])
@pytest.mark.parametrize("N", [256, 384])        # CTA-pair and single-CTA grouped kernels
def test_grouped_gemm(case, N):
    o = [0, 100, 200, ROWS] if case == "group_above_max" else bad_offsets()[case]
    max_rows = 99 if case == "group_above_max" else 200
    offs = dev_offs(o)
    groups = offs.numel() - 1
    A, Asf, B, Bsf = grouped_operands(NV, groups, N)
    D = filled((ROWS, N), torch.bfloat16, 0x5A)
    gs = torch.ones(groups, dtype=torch.float32, device="cuda")
    qfp4.gemm_nt_grouped(NV, offs, ROWS, max_rows, N, K, A, Asf, B, Bsf, gs, gs, D)
    expect_invalid_then_clean()
    assert torch.all(D.view(torch.uint8) == 0x5A), "D written despite bad offsets"
    rs = torch.ones(ROWS, dtype=torch.float32, device="cuda")
    cs = torch.ones(groups * N, dtype=torch.float32, device="cuda")
    qfp4.gemm_nt_grouped_scaled(NV, offs, ROWS, max_rows, N, K, A, Asf, B, Bsf, gs, gs, rs, cs, D)
    expect_invalid_then_clean()
    assert torch.all(D.view(torch.uint8) == 0x5A)


@pytest.mark.parametrize("case", sorted(bad_offsets()))
def test_grouped_swiglu(case):
    offs = dev_offs(bad_offsets()[case])
    groups = offs.numel() - 1
    I = 128
    A, Asf, W, Wsf = grouped_operands(NV, groups, 2 * I)
    Qh = filled((ROWS, I // 2), torch.uint8, 0x3C)
    SFh = torch.empty((qfp4.sf_mma_grouped_bytes(ROWS, groups, I // 16),), dtype=torch.uint8, device="cuda")
    gs = torch.ones(groups, dtype=torch.float32, device="cuda")
    qfp4.gemm_swiglu_quantize_grouped(NV, offs, ROWS, I, K, A, Asf, W, Wsf, gs, gs, gs, Qh, SFh)
    expect_invalid_then_clean()
    assert torch.all(Qh == 0x3C)


def test_valid_offsets_still_pass():
    """The check accepts what it should: empty groups, a group exactly at
    max_group_rows, offsets ending at the row count."""
    offs = dev_offs([0, 0, 150, 150, ROWS])
    groups = 4
    N = 256
    A, Asf, B, Bsf = grouped_operands(NV, groups, N)
    D = filled((ROWS, N), torch.bfloat16, 0x5A)
    gs = torch.ones(groups, dtype=torch.float32, device="cuda")
    qfp4.gemm_nt_grouped(NV, offs, ROWS, 150, N, K, A, Asf, B, Bsf, gs, gs, D)
    torch.cuda.synchronize()
    assert qfp4.poll_device_status() == 0
    assert torch.all(D.float() == 0.0)             # zero operands: D = 0 everywhere
