"""GPU parity of the tensor-core GEMM against the CPU oracle, within
|D - D_ref| <= 2^-8 |D_ref| + 1e-6 sum_k |a_k b_k| per element."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_tcgen05_gb300 import qfp4, synth
from tests._helpers import (MX, NV, assert_gemm_close, bf16_to_f64, dev_scalar, run_gemm,
                            to_dev_bf16, to_dev_u8, to_host)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    qfp4.load()
    assert qfp4.device_check() == 0


def pack(codes):
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


def one_sf(fmt):
    return 127 if fmt == MX else 0x38          # 1.0


# ----------------------------------------------------------------- probes

@pytest.mark.parametrize("fmt", [MX, NV])
@pytest.mark.parametrize("M", [128, 256, 384])
def test_all_ones_closed_form(fmt, M):
    N, K = 256, 512
    g = qfp4.block_size(fmt)
    A, B = pack(np.full((M, K), 2)), pack(np.full((N, K), 2))
    sa, sb = (126, 129) if fmt == MX else (0x30, 0x40)
    Asf = np.full((M, K // g), sa, np.uint8)
    Bsf = np.full((N, K // g), sb, np.uint8)
    d = run_gemm(fmt, A, Asf, B, Bsf, 1.0, 1.0)
    want = K * oracle.scale_value(fmt, sa) * oracle.scale_value(fmt, sb)
    assert np.all(d == want), np.unique(d)[:10]


@pytest.mark.parametrize("fmt", [MX, NV])
@pytest.mark.parametrize("M", [128, 256])
def test_one_hot_elements(fmt, M):
    """Single non-zero FP4 element per A row at a distinct k: pins the nibble
    order and the K position inside the 128-byte swizzled rows (single-CTA
    tiles at M = 128, CTA-pair tiles at M = 256)."""
    N, K = 256, 512
    g = qfp4.block_size(fmt)
    codes = np.zeros((M, K), np.uint8)
    ks = (np.arange(M) * 37) % K
    codes[np.arange(M), ks] = 7                          # 6.0
    A = pack(codes)
    bc = np.zeros((N, K), np.uint8)
    bc[:, :] = (np.arange(K)[None, :] % 7) + 1           # distinct per k
    bc[:, :] += ((np.arange(N)[:, None] % 2) * 8).astype(np.uint8)   # sign alternates per n
    B = pack(bc)
    Asf = np.full((M, K // g), one_sf(fmt), np.uint8)
    Bsf = np.full((N, K // g), one_sf(fmt), np.uint8)
    d = run_gemm(fmt, A, Asf, B, Bsf, 1.0, 1.0)
    d_ref, t_ref = oracle.gemm_nt(fmt, A, Asf, B, Bsf, 1.0, 1.0)
    assert_gemm_close(d, d_ref, t_ref, "one-hot elements")


@pytest.mark.parametrize("fmt", [MX, NV])
@pytest.mark.parametrize("M", [128, 256])
def test_one_hot_scales(fmt, M):
    """All elements 1.0; A's scale bytes distinct per (row, block) and B's per
    (column, block): pins the scale-factor layout in tensor memory."""
    N, K = 256, 1024
    g = qfp4.block_size(fmt)
    kg = K // g
    A, B = pack(np.full((M, K), 2)), pack(np.full((N, K), 2))
    gen = synth.rng(3)
    if fmt == MX:
        Asf = gen.integers(112, 142, size=(M, kg), dtype=np.uint8)
        Bsf = gen.integers(112, 142, size=(N, kg), dtype=np.uint8)
    else:
        Asf = gen.integers(1, 0x7F, size=(M, kg), dtype=np.uint8)
        Bsf = gen.integers(1, 0x7F, size=(N, kg), dtype=np.uint8)
    d = run_gemm(fmt, A, Asf, B, Bsf, 1.0, 1.0)
    d_ref, t_ref = oracle.gemm_nt(fmt, A, Asf, B, Bsf, 1.0, 1.0)
    assert_gemm_close(d, d_ref, t_ref, "one-hot scales")


# ----------------------------------------------------------------- small cases

def test_small_mxfp4_128x256x256():
    """The small MXFP4 workload: fp32 N(0,1) operands quantised by the oracle."""
    case = synth.SMALL_MX
    gen = synth.rng(case.seed)
    a = synth.normal_f32(gen, (case.M, case.K))
    b = synth.normal_f32(gen, (case.N, case.K))
    A, Asf = oracle.quantize(MX, a)
    B, Bsf = oracle.quantize(MX, b)
    d = run_gemm(MX, A, Asf, B, Bsf)
    d_ref, t_ref = oracle.gemm_nt(MX, A, Asf, B, Bsf)
    assert_gemm_close(d, d_ref, t_ref, case.name)


def random_operands(fmt, M, N, K, seed):
    gen = synth.rng(seed)
    g = qfp4.block_size(fmt)
    A = gen.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    B = gen.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    lo, hi = (118, 136) if fmt == MX else (1, 0x7F)
    Asf = gen.integers(lo, hi, size=(M, K // g), dtype=np.uint8)
    Bsf = gen.integers(lo, hi, size=(N, K // g), dtype=np.uint8)
    return A, Asf, B, Bsf


@pytest.mark.parametrize("fmt", [MX, NV])
@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (100, 256, 384), (128, 384, 256),
                                   (300, 640, 1024), (513, 256, 2048), (256, 1280, 640),
                                   (300, 512, 1024), (640, 1536, 768), (1100, 2048, 384)])
def test_random_shapes(fmt, M, N, K):
    A, Asf, B, Bsf = random_operands(fmt, M, N, K, M * 7 + N + K + fmt)
    gs_a, gs_b = (None, None) if fmt == MX else (0.37, 2.5e-3)
    d = run_gemm(fmt, A, Asf, B, Bsf, gs_a, gs_b)
    d_ref, t_ref = oracle.gemm_nt(fmt, A, Asf, B, Bsf, gs_a or 1.0, gs_b or 1.0)
    assert_gemm_close(d, d_ref, t_ref, f"{M}x{N}x{K}")


def test_global_scale_doubles_exactly():
    A, Asf, B, Bsf = random_operands(NV, 256, 512, 512, 5)
    d1 = run_gemm(NV, A, Asf, B, Bsf, 0.75, 1.5)
    d2 = run_gemm(NV, A, Asf, B, Bsf, 1.5, 1.5)
    assert np.array_equal(d2, 2.0 * d1)


# ----------------------------------------------------------------- full pipeline

def device_quantize(fmt, xbits):
    """gs (NVFP4) -> quantize (row-major SF) -> interleave, all on the device;
    returns device buffers and the host copies for the oracle."""
    M, K = xbits.shape
    g = qfp4.block_size(fmt)
    X = to_dev_bf16(xbits)
    gs = torch.ones(1, dtype=torch.float32, device="cuda")
    if fmt == NV:
        qfp4.global_scale(X, gs)
    Q = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
    SF = torch.empty((M, K // g), dtype=torch.uint8, device="cuda")
    SFm = torch.empty((qfp4.sf_mma_bytes(M, K // g),), dtype=torch.uint8, device="cuda")
    qfp4.quantize(fmt, X, gs, Q, SF, qfp4.SF_ROWMAJOR)
    qfp4.sf_interleave(SF, M, K // g, SFm, qfp4.SF_MMA)
    torch.cuda.synchronize()
    return Q, SFm, gs, to_host(Q), to_host(SF), np.float32(gs.item())


def sampled_check(fmt, qa, qb, D, n_samples, seed, full_rows=(0,)):
    M, N = D.shape
    gen = synth.rng(seed)
    mi = np.concatenate([gen.integers(0, M, n_samples), np.repeat(np.array(full_rows) % M, N)])
    ni = np.concatenate([gen.integers(0, N, n_samples), np.tile(np.arange(N), len(full_rows))])
    d_ref, t_ref = oracle.gemm_nt_entries(fmt, qa[3], qa[4], qb[3], qb[4], qa[5], qb[5], mi, ni)
    d = bf16_to_f64(D)[mi, ni]
    return assert_gemm_close(d, d_ref, t_ref, "sampled")


@pytest.mark.parametrize("case", [synth.PREFILL_NV, synth.DECODE_UP, synth.DECODE_ATTN],
                         ids=lambda c: c.name)
def test_pipeline_full_size(case):
    """Activations and weights quantised on the device (bit-exact against the
    oracle), then the GEMM at full size, checked on sampled outputs."""
    xa = synth.activations_bf16(case.seed, case.M, case.K)
    xw = synth.weights_bf16(case.seed + 1000, case.N, case.K)
    qa = device_quantize(case.fmt, xa)
    qb = device_quantize(case.fmt, xw)
    for q, x in ((qa, xa), (qb, xw)):
        gs_ref = oracle.global_scale(x) if case.fmt == NV else np.float32(1.0)
        assert q[5] == gs_ref
        q_ref, sf_ref = oracle.quantize(case.fmt, x, gs_ref)
        assert np.array_equal(q[3], q_ref) and np.array_equal(q[4], sf_ref)
    D = torch.empty((case.M, case.N), dtype=torch.bfloat16, device="cuda")
    ws_bytes = qfp4.gemm_workspace_bytes(case.fmt, case.M, case.N, case.K)
    ws = torch.zeros(max(ws_bytes, 1), dtype=torch.uint8, device="cuda")
    qfp4.gemm_nt(case.fmt, case.M, case.N, case.K, qa[0], qa[1], qb[0], qb[1], qa[2], qb[2], D,
                 ws, ws_bytes)
    torch.cuda.synchronize()
    assert qfp4.poll_device_status() == 0
    sampled_check(case.fmt, qa, qb, D, 20000, case.seed, full_rows=(0, case.M - 1, 77))


@pytest.mark.parametrize("case", synth.COMPUTE_SWEEP, ids=lambda c: c.name)
def test_compute_sweep_full_size(case):
    xa = synth.activations_bf16(case.seed, case.M, case.K)
    xw = synth.weights_bf16(case.seed + 1000, case.N, case.K)
    qa = device_quantize(case.fmt, xa)
    qb = device_quantize(case.fmt, xw)
    D = torch.empty((case.M, case.N), dtype=torch.bfloat16, device="cuda")
    qfp4.gemm_nt(case.fmt, case.M, case.N, case.K, qa[0], qa[1], qb[0], qb[1], qa[2], qb[2], D)
    torch.cuda.synchronize()
    assert qfp4.poll_device_status() == 0
    sampled_check(case.fmt, qa, qb, D, 8000, case.seed, full_rows=(case.M // 2,))


def test_grouped_moe_up_projection():
    """Per-expert NVFP4 up-projection in one launch: device per-expert global
    scales and grouped quantisation, then the grouped GEMM."""
    case = synth.MOE_UP
    counts = synth.moe_counts(case.seed, case.tokens, case.experts, case.topk)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    rows = int(offs[-1])
    E, N, K = case.experts, case.N, case.K
    g = qfp4.block_size(NV)
    xa = synth.activations_bf16(case.seed, rows, K)
    xw = synth.weights_bf16(case.seed + 1000, E * N, K)
    d_offs = torch.from_numpy(offs).cuda()
    X = to_dev_bf16(xa)
    gs_a = torch.empty(E, dtype=torch.float32, device="cuda")
    qfp4.global_scale_grouped(X, d_offs, gs_a)
    Qa = torch.empty((rows, K // 2), dtype=torch.uint8, device="cuda")
    SFa = torch.empty((qfp4.sf_mma_grouped_bytes(rows, E, K // g),), dtype=torch.uint8, device="cuda")
    qfp4.quantize_grouped(NV, X, d_offs, gs_a, Qa, SFa)
    # weights: per-expert global scale, quantised per expert, SF interleaved over [E*N, K/g]
    W = to_dev_bf16(xw)
    w_offs = torch.arange(0, (E + 1) * N, N, dtype=torch.int32, device="cuda")
    gs_b = torch.empty(E, dtype=torch.float32, device="cuda")
    qfp4.global_scale_grouped(W, w_offs, gs_b)
    Qb = torch.empty((E * N, K // 2), dtype=torch.uint8, device="cuda")
    SFb = torch.empty((qfp4.sf_mma_grouped_bytes(E * N, E, K // g),), dtype=torch.uint8, device="cuda")
    qfp4.quantize_grouped(NV, W, w_offs, gs_b, Qb, SFb)
    D = torch.empty((rows, N), dtype=torch.bfloat16, device="cuda")
    qfp4.gemm_nt_grouped(NV, d_offs, rows, int(counts.max()), N, K, Qa, SFa, Qb, SFb, gs_a, gs_b, D)
    torch.cuda.synchronize()
    assert qfp4.poll_device_status() == 0
    Qa_h, Qb_h, gsa_h, gsb_h = to_host(Qa), to_host(Qb), to_host(gs_a), to_host(gs_b)
    Dh = bf16_to_f64(D)
    gen = synth.rng(case.seed + 7)
    worst = 0.0
    for e in range(E):
        if counts[e] == 0:
            continue
        xa_e = xa[offs[e]:offs[e + 1]]
        xw_e = xw[e * N:(e + 1) * N]
        assert gsa_h[e] == oracle.global_scale(xa_e) and gsb_h[e] == oracle.global_scale(xw_e)
        qa_ref, sfa_ref = oracle.quantize(NV, xa_e, gsa_h[e])
        qb_ref, sfb_ref = oracle.quantize(NV, xw_e, gsb_h[e])
        assert np.array_equal(Qa_h[offs[e]:offs[e + 1]], qa_ref)
        assert np.array_equal(Qb_h[e * N:(e + 1) * N], qb_ref)
        n_s = 3000
        mi = gen.integers(0, counts[e], n_s)
        ni = gen.integers(0, N, n_s)
        d_ref, t_ref = oracle.gemm_nt_entries(NV, qa_ref, sfa_ref, qb_ref, sfb_ref, gsa_h[e], gsb_h[e], mi, ni)
        worst = max(worst, assert_gemm_close(Dh[offs[e] + mi, ni], d_ref, t_ref, f"expert {e}"))
    assert worst <= 1.0


# ----------------------------------------------------------------- decode (M <= 128)

def expected_splits(M, N, K):
    """The split count the decode kernel picks: the largest of 8, 4, 2 with
    ceil(N/256) * S CTA pairs on the GPU at once, S <= ceil(K/256), and at
    least 16 of the ceil(K/256) K-blocks taken off each pair."""
    pairs = torch.cuda.get_device_properties(0).multi_processor_count // 2
    tiles, kblocks = -(-N // 256), -(-K // 256)
    if M > 128 or K < 256:
        return 1
    for s in (8, 4, 2):
        if tiles * s <= pairs and s <= kblocks and kblocks - -(-kblocks // s) >= 16:
            return s
    return 1


def decode_workspace(fmt, M, N, K):
    """Zero-filled workspace for the decode split-K (None when it needs none)."""
    ws_bytes = qfp4.gemm_workspace_bytes(fmt, M, N, K)
    splits = expected_splits(M, N, K)
    if splits == 1:
        assert ws_bytes == 0
        return None, 0
    tiles, mpad = -(-N // 256), -(-M // 32) * 32
    counters = -(-(tiles * 2 * 2 * 4) // 256) * 256        # (count, generation) per pair tile and CTA
    assert ws_bytes == counters + tiles * splits * 2 * 128 * mpad * 4
    return torch.zeros(ws_bytes, dtype=torch.uint8, device="cuda"), ws_bytes


@pytest.mark.parametrize("fmt", [MX, NV])
@pytest.mark.parametrize("M,N,K", [(1, 128, 256), (37, 384, 1024), (128, 1024, 4096), (100, 2048, 2304),
                                   (128, 4096, 128), (64, 256, 8192), (128, 4096, 512), (77, 1024, 5120),
                                   (64, 256, 4736), (33, 640, 5248), (128, 4096, 14336), (5, 384, 16384),
                                   (128, 2048, 8192)])
def test_decode_shapes(fmt, M, N, K):
    """M <= 128 runs the decode kernel (A and B swapped on CTA pairs; ragged
    token counts, a weight tile of only 128 rows, and a trailing half K-block
    among the shapes), with K split over 2, 4 or 8 CTA pairs per weight tile
    when that saves enough K-blocks and a workspace is given: S = 8 at
    77 x 1024 x 5120 (ranges of 2 and 3 K-blocks), 64 x 256 x 4736 (the half
    K-block in the last range), 33 x 640 x 5248 (an empty second weight tile
    in the last pair), 5 x 384 x 16384, 64 x 256 x 8192 and 128 x 2048 x 8192;
    S = 4 at 128 x 4096 x 14336; one range for the rest.
    Both paths must match the oracle, and each must be bit-identical across
    repeated calls (the split partials are summed in a fixed order)."""
    A, Asf, B, Bsf = random_operands(fmt, M, N, K, M + N + K + 3 * fmt)
    gs_a, gs_b = (None, None) if fmt == MX else (0.125, 3.0)
    g = qfp4.block_size(fmt)
    ws, ws_bytes = decode_workspace(fmt, M, N, K)
    dA, dB = to_dev_u8(A), to_dev_u8(B)
    sfa = torch.zeros(qfp4.sf_mma_bytes(M, K // g), dtype=torch.uint8, device="cuda")
    sfb = torch.zeros(qfp4.sf_mma_bytes(N, K // g), dtype=torch.uint8, device="cuda")
    qfp4.sf_interleave(to_dev_u8(Asf), M, K // g, sfa, qfp4.SF_MMA)
    qfp4.sf_interleave(to_dev_u8(Bsf), N, K // g, sfb, qfp4.SF_MMA)
    ga = dev_scalar(gs_a) if gs_a else None
    gb = dev_scalar(gs_b) if gs_b else None
    d_ref, t_ref = oracle.gemm_nt(fmt, A, Asf, B, Bsf, gs_a or 1.0, gs_b or 1.0)
    paths = [(None, 0)] + ([(ws, ws_bytes)] if ws is not None else [])
    for w, wb in paths:
        outs = []
        for _ in range(3):
            D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
            qfp4.gemm_nt(fmt, M, N, K, dA, sfa, dB, sfb, ga, gb, D, w, wb)
            torch.cuda.synchronize()
            outs.append(bf16_to_f64(D))
        assert qfp4.poll_device_status() == 0
        what = f"decode {M}x{N}x{K} {'split-K' if w is not None else 'one range'}"
        assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2]), what
        assert_gemm_close(outs[0], d_ref, t_ref, what)
    if ws is not None:
        # every call leaves the arrival counts at zero for the next one; the
        # generation word beside each count advanced once per call (3 calls)
        # for the 128-row weight tiles that exist (N % 256 == 128 leaves the
        # last pair's second tile empty)
        words = ws[:-(-N // 256) * 2 * 2 * 4].view(torch.int32).cpu().numpy()
        assert not words[0::2].any()
        tiles_exist = np.arange(words.size // 2) < N // 128
        assert np.array_equal(words[1::2], np.where(tiles_exist, 3, 0))


@pytest.mark.parametrize("fmt", [MX, NV])
def test_decode_split_k_two_level(fmt):
    """The split-K reduction applies the two-level epilogue (row scale per
    token, column scale per weight row) like the single-range drain."""
    M, N, K = 96, 2048, 8192
    A, Asf, B, Bsf = random_operands(fmt, M, N, K, 4242 + fmt)
    g = qfp4.block_size(fmt)
    ws, ws_bytes = decode_workspace(fmt, M, N, K)
    assert ws is not None
    gen = synth.rng(77 + fmt)
    rs = (2.0 ** gen.integers(-3, 4, M)).astype(np.float32) * np.float32(1.25)
    cs = (2.0 ** gen.integers(-3, 4, N)).astype(np.float32) * np.float32(0.75)
    sfa = torch.zeros(qfp4.sf_mma_bytes(M, K // g), dtype=torch.uint8, device="cuda")
    sfb = torch.zeros(qfp4.sf_mma_bytes(N, K // g), dtype=torch.uint8, device="cuda")
    qfp4.sf_interleave(to_dev_u8(Asf), M, K // g, sfa, qfp4.SF_MMA)
    qfp4.sf_interleave(to_dev_u8(Bsf), N, K // g, sfb, qfp4.SF_MMA)
    ga, gb = (dev_scalar(0.5), dev_scalar(1.5)) if fmt == NV else (None, None)
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    qfp4.gemm_nt_scaled(fmt, M, N, K, to_dev_u8(A), sfa, to_dev_u8(B), sfb, ga, gb,
                        torch.from_numpy(rs).cuda(), torch.from_numpy(cs).cuda(), D, ws, ws_bytes)
    torch.cuda.synchronize()
    assert qfp4.poll_device_status() == 0
    d_ref, t_ref = oracle.gemm_nt(fmt, A, Asf, B, Bsf, 0.5 if fmt == NV else 1.0, 1.5 if fmt == NV else 1.0,
                                  row_scale=rs, col_scale=cs)
    assert_gemm_close(bf16_to_f64(D), d_ref, t_ref, "split-K two-level")


# ----------------------------------------------------------------- grouped vs dense

@pytest.mark.parametrize("N", [14336, 14464])
def test_grouped_equals_dense_per_group(N):
    """The grouped launch computes every group with the same kernel and the
    same K order as a dense launch over that group's rows, so the outputs must
    be bit-identical, and identical across repeated launches.  Scale factors
    vary along K, so a K-block combined with another K-block's scales shows.
    N = 14336 runs the CTA-pair kernel, N = 14464 the single-CTA one."""
    counts = np.array([2193, 1698, 128, 1553, 1387, 16, 142, 1075])
    E, K, g = len(counts), 4096, 16
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    rows = int(offs[-1])
    gen = torch.Generator(device="cuda").manual_seed(1234 + N)
    A = torch.randint(0, 256, (rows, K // 2), dtype=torch.uint8, device="cuda", generator=gen)
    B = torch.randint(0, 256, (E * N, K // 2), dtype=torch.uint8, device="cuda", generator=gen)
    SFa = torch.randint(40, 60, (qfp4.sf_mma_grouped_bytes(rows, E, K // g),), dtype=torch.uint8,
                        device="cuda", generator=gen)
    SFb = torch.randint(40, 60, (qfp4.sf_mma_grouped_bytes(E * N, E, K // g),), dtype=torch.uint8,
                        device="cuda", generator=gen)
    gs_a = torch.rand(E, device="cuda", generator=gen) + 0.5
    gs_b = torch.rand(E, device="cuda", generator=gen) + 0.5
    d_offs = torch.from_numpy(offs).cuda()
    outs = []
    for _ in range(2):
        D = torch.zeros((rows, N), dtype=torch.bfloat16, device="cuda")
        qfp4.gemm_nt_grouped(NV, d_offs, rows, int(counts.max()), N, K, A, SFa, B, SFb, gs_a, gs_b, D)
        torch.cuda.synchronize()
        outs.append(D)
    assert qfp4.poll_device_status() == 0
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16))
    kc = K // g // 4
    tile = 0
    for e in range(E):
        m = int(counts[e])
        sfa_e = SFa[tile * kc * 512:(tile + (m + 127) // 128) * kc * 512]
        sfb_e = SFb[e * (N // 128) * kc * 512:(e + 1) * (N // 128) * kc * 512]
        tile += (m + 127) // 128
        De = torch.empty((m, N), dtype=torch.bfloat16, device="cuda")
        qfp4.gemm_nt(NV, m, N, K, A[offs[e]:offs[e + 1]], sfa_e, B[e * N:(e + 1) * N], sfb_e,
                     gs_a[e:e + 1], gs_b[e:e + 1], De)
        torch.cuda.synchronize()
        same = torch.equal(De.view(torch.int16), outs[0][offs[e]:offs[e + 1]].view(torch.int16))
        assert same, f"group {e} ({m} rows) differs from the dense launch"


# ----------------------------------------------------------------- degenerate shapes

def test_degenerate_shapes():
    """M == 0 or N == 0: nothing to compute; K == 0: an empty sum, D == 0."""
    D = torch.full((4, 256), 7.0, dtype=torch.bfloat16, device="cuda")
    z = torch.zeros(16, dtype=torch.uint8, device="cuda")
    qfp4.gemm_nt(NV, 0, 256, 256, z, z, z, z, None, None, D)
    qfp4.gemm_nt(NV, 4, 0, 256, z, z, z, z, None, None, D)
    torch.cuda.synchronize()
    assert bool((D.float() == 7.0).all())
    qfp4.gemm_nt(NV, 4, 256, 0, z, z, z, z, None, None, D)
    torch.cuda.synchronize()
    assert qfp4.poll_device_status() == 0
    assert bool((D.float() == 0.0).all()) and not bool(torch.signbit(D.float()).any())
