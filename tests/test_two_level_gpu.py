"""GPU parity of the two-level path against the CPU oracle: per-row global
scales (bit-exact), quantisation with one global scale per row (bit-exact)
and the GEMM with a per-row and per-column rescale in its epilogue (within
|D - D_ref| <= 2^-8 |D_ref| + 1e-6 T, T including the scales)."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_tcgen05_gb300 import qfp4, synth
from tests._helpers import MX, NV, assert_gemm_close, bf16_to_f64, dev_scalar, to_dev_bf16, to_dev_u8, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    qfp4.load()
    assert qfp4.device_check() == 0


def dev_f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


# ----------------------------------------------------------------- per-row global scales

@pytest.mark.parametrize("rows,cols", [(1, 8), (37, 384), (300, 1024), (4096, 4096)])
def test_global_scale_rows_bitexact(rows, cols):
    x = synth.activations_bf16(3000 + rows + cols, rows, cols)
    if rows > 3:
        x[2] = 0                                   # an all-zero row: gs 0
    gs = torch.full((rows,), -1.0, dtype=torch.float32, device="cuda")
    qfp4.global_scale_rows(to_dev_bf16(x), gs)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(gs), oracle.global_scale_rows(x))


# ----------------------------------------------------------------- per-row quantisation

@pytest.mark.parametrize("M,K", [(1, 128), (37, 384), (300, 1024), (4096, 4096)])
def test_quantize_rows_bitexact(M, K):
    x = synth.activations_bf16(4000 + M + K, M, K)
    if M > 3:
        x[1] = 0
    gs = oracle.global_scale_rows(x)
    q_ref, sf_ref = oracle.quantize(NV, x, gs)
    X = to_dev_bf16(x)
    for layout in (qfp4.SF_ROWMAJOR, qfp4.SF_MMA):
        Q = torch.full((M, K // 2), 0xAB, dtype=torch.uint8, device="cuda")
        nsf = M * (K // 16) if layout == qfp4.SF_ROWMAJOR else qfp4.sf_mma_bytes(M, K // 16)
        SF = torch.full((nsf,), 0xCD, dtype=torch.uint8, device="cuda")
        qfp4.quantize_rows(NV, X, dev_f32(gs), Q, SF, layout)
        torch.cuda.synchronize()
        assert qfp4.poll_device_status() == 0
        assert np.array_equal(to_host(Q), q_ref)
        want = sf_ref.reshape(-1) if layout == qfp4.SF_ROWMAJOR else oracle.sf_to_mma(sf_ref)
        assert np.array_equal(to_host(SF), want)


def test_quantize_rows_mxfp4_is_plain_quantize():
    x = synth.activations_bf16(4100, 130, 512)
    q_ref, sf_ref = oracle.quantize(MX, x, 1.0)
    Q = torch.empty((130, 256), dtype=torch.uint8, device="cuda")
    SF = torch.empty((130, 16), dtype=torch.uint8, device="cuda")
    qfp4.quantize_rows(MX, to_dev_bf16(x), None, Q, SF, qfp4.SF_ROWMAJOR)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(Q), q_ref) and np.array_equal(to_host(SF), sf_ref)


# ----------------------------------------------------------------- row / column rescaled GEMM

def operands(fmt, M, N, K, seed):
    gen = synth.rng(seed)
    g = qfp4.block_size(fmt)
    A = gen.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    B = gen.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    lo, hi = (118, 136) if fmt == MX else (1, 0x7F)
    Asf = gen.integers(lo, hi, size=(M, K // g), dtype=np.uint8)
    Bsf = gen.integers(lo, hi, size=(N, K // g), dtype=np.uint8)
    rs = (np.exp(gen.normal(0, 1.5, M)) * np.where(gen.random(M) < 0.1, -1, 1)).astype(np.float32)
    cs = np.exp(gen.normal(0, 1.5, N)).astype(np.float32)
    return A, Asf, B, Bsf, rs, cs


def run_scaled(fmt, A, Asf, B, Bsf, gs_a, gs_b, rs, cs, plain=False):
    M, N, K = A.shape[0], B.shape[0], A.shape[1] * 2
    g = qfp4.block_size(fmt)
    sfa = torch.zeros(qfp4.sf_mma_bytes(M, K // g), dtype=torch.uint8, device="cuda")
    sfb = torch.zeros(qfp4.sf_mma_bytes(N, K // g), dtype=torch.uint8, device="cuda")
    qfp4.sf_interleave(to_dev_u8(Asf), M, K // g, sfa, qfp4.SF_MMA)
    qfp4.sf_interleave(to_dev_u8(Bsf), N, K // g, sfb, qfp4.SF_MMA)
    ga = dev_scalar(gs_a) if gs_a is not None else None
    gb = dev_scalar(gs_b) if gs_b is not None else None
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    if plain:
        qfp4.gemm_nt(fmt, M, N, K, to_dev_u8(A), sfa, to_dev_u8(B), sfb, ga, gb, D)
    else:
        qfp4.gemm_nt_scaled(fmt, M, N, K, to_dev_u8(A), sfa, to_dev_u8(B), sfb, ga, gb,
                            dev_f32(rs) if rs is not None else None, dev_f32(cs) if cs is not None else None, D)
    torch.cuda.synchronize()
    assert qfp4.poll_device_status() == 0
    return D


# shapes chosen to reach every kernel: M <= 128 (A and B swapped on CTA pairs),
# N % 256 == 0 (CTA pairs; MXFP4 with K % 512 == 0 on two-K-block stages),
# and N % 256 != 0 (single-CTA tiles)
SHAPES = [(64, 1024, 512), (128, 384, 768), (300, 512, 1024), (513, 768, 768), (300, 640, 512),
          (260, 384, 1024)]


@pytest.mark.parametrize("fmt", [MX, NV])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemm_scaled_vs_oracle(fmt, M, N, K):
    A, Asf, B, Bsf, rs, cs = operands(fmt, M, N, K, 5000 + M + N + K + fmt)
    gs_a, gs_b = (None, None) if fmt == MX else (0.75, 3.0e-3)
    for r, c in ((rs, cs), (rs, None), (None, cs)):
        D = run_scaled(fmt, A, Asf, B, Bsf, gs_a, gs_b, r, c)
        d_ref, t_ref = oracle.gemm_nt(fmt, A, Asf, B, Bsf, gs_a or 1.0, gs_b or 1.0, r, c)
        assert_gemm_close(bf16_to_f64(D), d_ref, t_ref,
                          f"{M}x{N}x{K} rows {'on' if r is not None else 'off'} cols {'on' if c is not None else 'off'}")


@pytest.mark.parametrize("fmt", [MX, NV])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemm_scaled_without_scales_is_plain(fmt, M, N, K):
    A, Asf, B, Bsf, _, _ = operands(fmt, M, N, K, 6000 + M + N + K + fmt)
    gs_a, gs_b = (None, None) if fmt == MX else (0.75, 3.0e-3)
    d1 = run_scaled(fmt, A, Asf, B, Bsf, gs_a, gs_b, None, None)
    d2 = run_scaled(fmt, A, Asf, B, Bsf, gs_a, gs_b, None, None, plain=True)
    assert torch.equal(d1.view(torch.int16), d2.view(torch.int16))


def test_two_level_nvfp4_pipeline_4096():
    """The accuracy path end to end on the device at 4096^3: per-row global
    scales and per-row quantisation of the activations and of the weights
    (bit-exact), then the GEMM with those scales as row and column rescales,
    checked on sampled outputs and whole rows."""
    M = N = K = 4096
    xa = synth.activations_bf16(7001, M, K)
    xw = synth.weights_bf16(7002, N, K)
    out = []
    for x in (xa, xw):
        rows = x.shape[0]
        X = to_dev_bf16(x)
        gs = torch.empty(rows, dtype=torch.float32, device="cuda")
        qfp4.global_scale_rows(X, gs)
        Q = torch.empty((rows, K // 2), dtype=torch.uint8, device="cuda")
        SF = torch.empty(qfp4.sf_mma_bytes(rows, K // 16), dtype=torch.uint8, device="cuda")
        qfp4.quantize_rows(NV, X, gs, Q, SF, qfp4.SF_MMA)
        torch.cuda.synchronize()
        gs_ref = oracle.global_scale_rows(x)
        assert np.array_equal(to_host(gs), gs_ref)
        q_ref, sf_ref = oracle.quantize(NV, x, gs_ref)
        assert np.array_equal(to_host(Q), q_ref)
        assert np.array_equal(to_host(SF), oracle.sf_to_mma(sf_ref))
        out.append((Q, SF, gs, q_ref, sf_ref, gs_ref))
    (Qa, SFa, gsa, qa, sfa, gsa_ref), (Qb, SFb, gsb, qb, sfb, gsb_ref) = out
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    qfp4.gemm_nt_scaled(NV, M, N, K, Qa, SFa, Qb, SFb, None, None, gsa, gsb, D)
    torch.cuda.synchronize()
    assert qfp4.poll_device_status() == 0
    gen = synth.rng(7003)
    rows = (0, 77, M - 1)
    mi = np.concatenate([gen.integers(0, M, 20000), np.repeat(np.array(rows), N)])
    ni = np.concatenate([gen.integers(0, N, 20000), np.tile(np.arange(N), len(rows))])
    d_ref, t_ref = oracle.gemm_nt_entries(NV, qa, sfa, qb, sfb, 1.0, 1.0, mi, ni, gsa_ref, gsb_ref)
    assert_gemm_close(bf16_to_f64(D)[mi, ni], d_ref, t_ref, "two-level 4096^3 sampled")


# ----------------------------------------------------------------- grouped (MoE) two-level

@pytest.mark.parametrize("N", [256, 384])
def test_grouped_two_level_nvfp4(N):
    """Per-row global scales of the concatenated activations and of each
    expert's weight rows, grouped per-row quantisation (bit-exact, per-group
    scale layout), then the grouped GEMM with row and column rescales against
    the oracle per expert.  N = 256 runs CTA pairs, N = 384 single CTAs."""
    counts = np.array([300, 17, 0, 140, 256])
    E, K, g = len(counts), 512, 16
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    rows = int(offs[-1])
    xa = synth.activations_bf16(8000 + N, rows, K)
    xw = synth.weights_bf16(8001 + N, E * N, K)
    d_offs = torch.from_numpy(offs).cuda()
    w_offs = torch.arange(0, (E + 1) * N, N, dtype=torch.int32, device="cuda")
    out = []
    for x, o, nrow in ((xa, d_offs, rows), (xw, w_offs, E * N)):
        X = to_dev_bf16(x)
        gs = torch.empty(nrow, dtype=torch.float32, device="cuda")
        qfp4.global_scale_rows(X, gs)
        Q = torch.empty((nrow, K // 2), dtype=torch.uint8, device="cuda")
        SF = torch.full((qfp4.sf_mma_grouped_bytes(nrow, E, K // g),), 0xEE, dtype=torch.uint8, device="cuda")
        qfp4.quantize_grouped_rows(NV, X, o, gs, Q, SF)
        torch.cuda.synchronize()
        out.append((Q, SF, gs, to_host(Q), to_host(SF), to_host(gs)))
    (Qa, SFa, gsa, qa_h, sfa_h, gsa_h), (Qb, SFb, gsb, qb_h, sfb_h, gsb_h) = out
    assert np.array_equal(gsa_h, oracle.global_scale_rows(xa))
    assert np.array_equal(gsb_h, oracle.global_scale_rows(xw))
    # quantised bytes and the per-group scale layout
    kc = K // g // 4
    for x, q_h, sf_h, gs_h, seg in ((xa, qa_h, sfa_h, gsa_h, offs), (xw, qb_h, sfb_h, gsb_h, np.arange(0, (E + 1) * N, N))):
        tile = 0
        for e in range(E):
            lo, hi = int(seg[e]), int(seg[e + 1])
            if hi == lo:
                continue
            q_ref, sf_ref = oracle.quantize(NV, x[lo:hi], gs_h[lo:hi])
            assert np.array_equal(q_h[lo:hi], q_ref), e
            ref_mma = oracle.sf_to_mma(sf_ref)
            assert np.array_equal(sf_h[tile * kc * 512:tile * kc * 512 + ref_mma.size], ref_mma), e
            tile += -(-(hi - lo) // 128)
    D = torch.empty((rows, N), dtype=torch.bfloat16, device="cuda")
    qfp4.gemm_nt_grouped_scaled(NV, d_offs, rows, int(counts.max()), N, K, Qa, SFa, Qb, SFb, None, None, gsa, gsb, D)
    D0 = torch.empty((rows, N), dtype=torch.bfloat16, device="cuda")
    D1 = torch.empty((rows, N), dtype=torch.bfloat16, device="cuda")
    qfp4.gemm_nt_grouped_scaled(NV, d_offs, rows, int(counts.max()), N, K, Qa, SFa, Qb, SFb, None, None,
                                None, None, D0)
    qfp4.gemm_nt_grouped(NV, d_offs, rows, int(counts.max()), N, K, Qa, SFa, Qb, SFb, None, None, D1)
    torch.cuda.synchronize()
    assert qfp4.poll_device_status() == 0
    assert torch.equal(D0.view(torch.int16), D1.view(torch.int16))      # no scales: the plain grouped GEMM
    Dh = bf16_to_f64(D)
    for e in range(E):
        lo, hi = int(offs[e]), int(offs[e + 1])
        if hi == lo:
            continue
        sfa_e = oracle.sf_from_mma(np.ascontiguousarray(sfa_h[sum(-(-int(c) // 128) for c in counts[:e]) * kc * 512:]),
                                   hi - lo, K // g)
        sfb_e = oracle.sf_from_mma(np.ascontiguousarray(sfb_h[e * (N // 128) * kc * 512:]), N, K // g)
        d_ref, t_ref = oracle.gemm_nt(NV, qa_h[lo:hi], sfa_e, qb_h[e * N:(e + 1) * N], sfb_e, 1.0, 1.0,
                                      gsa_h[lo:hi], gsb_h[e * N:(e + 1) * N])
        assert_gemm_close(Dh[lo:hi], d_ref, t_ref, f"expert {e}")
