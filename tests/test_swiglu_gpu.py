"""GPU parity of the up-projection with SwiGLU and requantisation
(qfp4_gemm_swiglu_quantize[_grouped]) against the oracle.

The kernel's gate and up sums come out of fp32 accumulators and pass through
an exponential before they are rounded to codes, so the check is the
oracle's requant_valid: every block must be what the quantiser's rule gives
for some fp32 input within the propagated error bound of the exact
H = silu(G) * U (tests/_helpers.swiglu_delta).  As a sanity bound on top,
at least 99% of the blocks must equal the rule applied to the exact H."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_tcgen05_gb300 import qfp4, synth
from tests._helpers import MX, NV, dev_scalar, swiglu_delta, to_dev_bf16, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    qfp4.load()
    assert qfp4.device_check() == 0


def interleave_perm(I, g):
    """Row order of W: groups of g gate rows, then the g up rows of the same
    outputs (gate rows are 0..I-1 and up rows I..2I-1 of [gate; up])."""
    b = np.arange(I // g)[:, None] * g + np.arange(g)[None, :]
    return np.concatenate([b, I + b], axis=1).reshape(-1)


def quantize_dev(fmt, xbits, gs=None):
    """Device global scale (NVFP4, unless given) and quantisation with
    row-major scale bytes; returns (Q, SF_rowmajor, gs) on the device."""
    M, K = xbits.shape
    g = qfp4.block_size(fmt)
    X = to_dev_bf16(xbits)
    if gs is None:
        gs = torch.ones(1, dtype=torch.float32, device="cuda")
        if fmt == NV:
            qfp4.global_scale(X, gs)
    Q = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
    SF = torch.empty((M, K // g), dtype=torch.uint8, device="cuda")
    qfp4.quantize(fmt, X, gs, Q, SF, qfp4.SF_ROWMAJOR)
    return Q, SF, gs


def to_mma(SF_rm):
    rows, cols = SF_rm.shape
    out = torch.empty((qfp4.sf_mma_bytes(rows, cols),), dtype=torch.uint8, device="cuda")
    qfp4.sf_interleave(SF_rm, rows, cols, out, qfp4.SF_MMA)
    return out


def weights(fmt, I, K, seed):
    """Gate and up weights quantised together (one global scale) on the
    device and interleaved; returns the device W, W_sf (MMA layout), gs_w and
    the oracle's gate and up operands."""
    g = qfp4.block_size(fmt)
    wcat = np.concatenate([synth.weights_bf16(seed, I, K), synth.weights_bf16(seed + 1, I, K)])
    Qc, SFc, gw = quantize_dev(fmt, wcat)
    gw_ref = oracle.global_scale(wcat) if fmt == NV else np.float32(1.0)
    qc_ref, sfc_ref = oracle.quantize(fmt, wcat, gw_ref)
    torch.cuda.synchronize()
    assert np.float32(gw.item()) == gw_ref
    assert np.array_equal(to_host(Qc), qc_ref) and np.array_equal(to_host(SFc), sfc_ref)
    perm = torch.from_numpy(interleave_perm(I, g)).cuda()
    W = Qc[perm].contiguous()
    W_sf = to_mma(SFc[perm].contiguous())
    ref = (qc_ref[:I], sfc_ref[:I], qc_ref[I:], sfc_ref[I:], gw_ref)
    return W, W_sf, gw, ref


def check_blocks(fmt, qh, sfh, H, delta, gs_out, what):
    ok = oracle.requant_valid(fmt, qh, sfh, H, delta, gs_out)
    if not ok.all():
        bad = np.argwhere(~ok)[:6].tolist()
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} blocks invalid, first {bad}")
    g = qfp4.block_size(fmt)
    q_ref, sf_ref = oracle.swiglu_requantize(fmt, H, gs_out)
    M, I = H.shape
    same_codes = (qh == q_ref).reshape(M, I // g, g // 2).all(axis=-1)
    exact = float(((sfh == sf_ref) & same_codes).mean())
    assert exact >= 0.99, f"{what}: only {exact:.4f} of the blocks equal the rule on the exact H"
    return exact


@pytest.mark.parametrize("fmt", [MX, NV])
@pytest.mark.parametrize("M,I,K", [(300, 256, 512), (77, 128, 256), (1, 384, 1024), (513, 256, 768)])
def test_swiglu_quantize_vs_oracle(fmt, M, I, K):
    g = qfp4.block_size(fmt)
    xa = synth.activations_bf16(8100 + M + K, M, K)
    Qa, SFa, ga = quantize_dev(fmt, xa)
    SFa_m = to_mma(SFa)
    W, W_sf, gw, (qg, sfg, qu, sfu, gw_ref) = weights(fmt, I, K, 8200 + I + fmt)
    ga_ref = oracle.global_scale(xa) if fmt == NV else np.float32(1.0)
    qa_ref, sfa_ref = oracle.quantize(fmt, xa, ga_ref)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(Qa), qa_ref) and np.array_equal(to_host(SFa), sfa_ref)
    H, G, U, TG, TU = oracle.swiglu_up(fmt, qa_ref, sfa_ref, qg, sfg, qu, sfu, ga_ref, gw_ref)
    gs_out = np.float32(max(np.abs(H).max(), 1e-30) / 2688.0) if fmt == NV else np.float32(1.0)

    Qh = torch.full((M, I // 2), 0x5A, dtype=torch.uint8, device="cuda")
    SFh = torch.full((qfp4.sf_mma_bytes(M, I // g),), 0xA5, dtype=torch.uint8, device="cuda")
    go = dev_scalar(gs_out) if fmt == NV else None
    qfp4.gemm_swiglu_quantize(fmt, M, I, K, Qa, SFa_m, W, W_sf, ga if fmt == NV else None,
                              gw if fmt == NV else None, go, Qh, SFh)
    torch.cuda.synchronize()
    assert qfp4.poll_device_status() == 0
    sfh_m = to_host(SFh)
    sfh = oracle.sf_from_mma(sfh_m, M, I // g)
    assert np.array_equal(sfh_m, oracle.sf_to_mma(sfh)), "scale layout or its zero padding"
    check_blocks(fmt, to_host(Qh), sfh, H, swiglu_delta(G, U, TG, TU, K), gs_out, f"M={M} I={I} K={K}")


def test_swiglu_quantize_full_size_sampled_rows():
    """Llama-3-8B ffn-up shape (4096 tokens, I = 14336, K = 4096), NVFP4,
    checked on 64 whole rows: the tile edges (0, 255/256, 4095) and a seeded
    sample spread over every 256-row pair tile."""
    fmt, M, I, K = NV, 4096, 14336, 4096
    g = 16
    xa = synth.activations_bf16(8300, M, K)
    Qa, SFa, ga = quantize_dev(fmt, xa)
    SFa_m = to_mma(SFa)
    W, W_sf, gw, (qg, sfg, qu, sfu, gw_ref) = weights(fmt, I, K, 8400)
    ga_ref = oracle.global_scale(xa)
    edges = [0, 1, 127, 128, 255, 256, 2047, 4095]
    pick = synth.rng(8301).choice(np.setdiff1d(np.arange(M), edges), 64 - len(edges), replace=False)
    rows = np.sort(np.concatenate([edges, pick]))
    qa_ref, sfa_ref = oracle.quantize(fmt, xa[rows], ga_ref)
    torch.cuda.synchronize()
    assert np.float32(ga.item()) == ga_ref
    assert np.array_equal(to_host(Qa)[rows], qa_ref) and np.array_equal(to_host(SFa)[rows], sfa_ref)
    H, G, U, TG, TU = oracle.swiglu_up(fmt, qa_ref, sfa_ref, qg, sfg, qu, sfu, ga_ref, gw_ref)
    gs_out = np.float32(np.abs(H).max() / 2688.0)

    Qh = torch.empty((M, I // 2), dtype=torch.uint8, device="cuda")
    SFh = torch.full((qfp4.sf_mma_bytes(M, I // g),), 0xA5, dtype=torch.uint8, device="cuda")
    qfp4.gemm_swiglu_quantize(fmt, M, I, K, Qa, SFa_m, W, W_sf, ga, gw, dev_scalar(gs_out), Qh, SFh)
    torch.cuda.synchronize()
    assert qfp4.poll_device_status() == 0
    sfh = oracle.sf_from_mma(to_host(SFh), M, I // g)[rows]
    check_blocks(fmt, to_host(Qh)[rows], sfh, H, swiglu_delta(G, U, TG, TU, K), gs_out, "4096x14336x4096")


@pytest.mark.parametrize("fmt", [MX, NV])
def test_swiglu_quantize_grouped(fmt):
    """Three experts with 150, 0 and 300 rows: per-expert weights and global
    scales, H written in the per-group scale layout."""
    g = qfp4.block_size(fmt)
    I, K = 256, 512
    counts = np.array([150, 0, 300])
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    E, T = len(counts), int(offs[-1])
    xa = synth.activations_bf16(8500 + fmt, T, K)
    X = to_dev_bf16(xa)
    d_offs = torch.from_numpy(offs).cuda()
    ga = torch.ones(E, dtype=torch.float32, device="cuda")
    if fmt == NV:
        qfp4.global_scale_grouped(X, d_offs, ga)
    Qa = torch.empty((T, K // 2), dtype=torch.uint8, device="cuda")
    SFa = torch.empty((qfp4.sf_mma_grouped_bytes(T, E, K // g),), dtype=torch.uint8, device="cuda")
    qfp4.quantize_grouped(fmt, X, d_offs, ga if fmt == NV else None, Qa, SFa)
    Ws, Wsfs, gws, refs = [], [], [], []
    for e in range(E):
        W, W_sf, gw, ref = weights(fmt, I, K, 8600 + 10 * e + fmt)
        Ws.append(W), Wsfs.append(W_sf), gws.append(gw), refs.append(ref)
    W = torch.cat(Ws)
    W_sf = torch.cat(Wsfs)
    gw = torch.cat(gws)
    torch.cuda.synchronize()
    ga_h = to_host(ga)
    Hs, gs_out = [], np.ones(E, dtype=np.float32)
    for e in range(E):
        lo, hi = int(offs[e]), int(offs[e + 1])
        if hi == lo:
            Hs.append(None)
            continue
        ga_ref = oracle.global_scale(xa[lo:hi]) if fmt == NV else np.float32(1.0)
        assert ga_h[e] == ga_ref
        qa_ref, sfa_ref = oracle.quantize(fmt, xa[lo:hi], ga_ref)
        assert np.array_equal(to_host(Qa)[lo:hi], qa_ref)
        qg, sfg, qu, sfu, gw_ref = refs[e]
        Hs.append(oracle.swiglu_up(fmt, qa_ref, sfa_ref, qg, sfg, qu, sfu, ga_ref, gw_ref))
        if fmt == NV:
            gs_out[e] = np.float32(np.abs(Hs[e][0]).max() / 2688.0)
    Qh = torch.full((T, I // 2), 0x5A, dtype=torch.uint8, device="cuda")
    SFh = torch.full((qfp4.sf_mma_grouped_bytes(T, E, I // g),), 0xA5, dtype=torch.uint8, device="cuda")
    go = torch.from_numpy(gs_out).cuda() if fmt == NV else None
    qfp4.gemm_swiglu_quantize_grouped(fmt, d_offs, T, I, K, Qa, SFa, W, W_sf, ga if fmt == NV else None,
                                      gw if fmt == NV else None, go, Qh, SFh)
    torch.cuda.synchronize()
    assert qfp4.poll_device_status() == 0
    qh, sfh_m = to_host(Qh), to_host(SFh)
    kc = (I // g) // 4
    tile = 0
    for e in range(E):
        lo, hi = int(offs[e]), int(offs[e + 1])
        if hi == lo:
            continue
        H, G, U, TG, TU = Hs[e]
        sfh = oracle.sf_from_mma(np.ascontiguousarray(sfh_m[tile * kc * 512:]), hi - lo, I // g)
        check_blocks(fmt, qh[lo:hi], sfh, H, swiglu_delta(G, U, TG, TU, K), gs_out[e], f"expert {e}")
        tile += -(-(hi - lo) // 128)


def test_swiglu_quantize_empty_sum():
    """K = 0: H = 0, so every scale byte and every code is 0."""
    M, I = 50, 128
    Qh = torch.full((M, I // 2), 0x5A, dtype=torch.uint8, device="cuda")
    SFh = torch.full((qfp4.sf_mma_bytes(M, I // 16),), 0xA5, dtype=torch.uint8, device="cuda")
    qfp4.gemm_swiglu_quantize(NV, M, I, 0, None, None, None, None, None, None, dev_scalar(1.0), Qh, SFh)
    torch.cuda.synchronize()
    assert int(Qh.max()) == 0 and int(SFh.max()) == 0


def test_swiglu_quantize_zero_output_scale():
    """gs_out = 0 with a non-zero H: every block target is (amax/6)/0 = +inf,
    which saturates the UE4M3 scale byte to 0x7E (448), and the element scale
    s = 448 * 0 = 0 makes every code +0 (the zero-scale reading); the oracle
    gives the same bytes."""
    fmt, M, I, K = NV, 77, 128, 256
    g = 16
    xa = synth.activations_bf16(8700, M, K)
    Qa, SFa, ga = quantize_dev(fmt, xa)
    W, W_sf, gw, (qg, sfg, qu, sfu, gw_ref) = weights(fmt, I, K, 8800)
    ga_ref = oracle.global_scale(xa)
    qa_ref, sfa_ref = oracle.quantize(fmt, xa, ga_ref)
    H = oracle.swiglu_up(fmt, qa_ref, sfa_ref, qg, sfg, qu, sfu, ga_ref, gw_ref)[0]
    q_ref, sf_ref = oracle.swiglu_requantize(fmt, H, np.float32(0.0))
    nonzero = np.abs(H).reshape(M, I // g, g).max(axis=-1) > 0
    assert nonzero.all(), "the case wants every block of H non-zero"
    assert np.all(sf_ref == 0x7E) and not q_ref.any()
    Qh = torch.full((M, I // 2), 0x5A, dtype=torch.uint8, device="cuda")
    SFh = torch.full((qfp4.sf_mma_bytes(M, I // g),), 0xA5, dtype=torch.uint8, device="cuda")
    qfp4.gemm_swiglu_quantize(fmt, M, I, K, Qa, to_mma(SFa), W, W_sf, ga, gw, dev_scalar(0.0), Qh, SFh)
    torch.cuda.synchronize()
    assert qfp4.poll_device_status() == 0
    assert not to_host(Qh).any(), "codes must all be +0 under a zero element scale"
    assert np.array_equal(oracle.sf_from_mma(to_host(SFh), M, I // g), sf_ref)
