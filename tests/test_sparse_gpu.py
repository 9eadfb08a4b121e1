"""GPU parity of the 2:4 pair-sparse FP4 path against the oracle: the
compressor (bit-exact kept bytes and metadata, both layouts), the NVFP4
quantiser with 32-element blocks the sparse path uses (bit-exact), and the
sparse GEMM (|D - D_ref| <= 2^-8 |D_ref| + 1e-6 sum_k |x_k w_k|)."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_tcgen05_gb300 import qfp4, synth
from tests._helpers import assert_gemm_close, bf16_to_f64, dev_scalar, to_dev_bf16, to_dev_u8, to_host

pytestmark = pytest.mark.gpu

NV32 = qfp4.NVFP4_B32
INVALID = -1


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    qfp4.load()
    assert qfp4.device_check() == 0


def meta_rowmajor_to_tiled(meta, rows, K):
    """Row-major metadata [rows, K/16] -> the tiled layout
    [ceil(rows/128)][K/512][128][32], padding rows holding pairs 0 and 1."""
    rp = -(-rows // 128) * 128
    m = np.full((rp, K // 16), 0x44, np.uint8)
    m[:rows] = meta
    return np.ascontiguousarray(m.reshape(rp // 128, 128, K // 512, 32).transpose(0, 2, 1, 3)).reshape(-1)


def quantize_dev(x, fmt=NV32, layout=qfp4.SF_ROWMAJOR):
    rows, K = x.shape
    X = to_dev_bf16(x)
    gs = torch.empty(1, dtype=torch.float32, device="cuda")
    qfp4.global_scale(X, gs)
    Q = torch.empty((rows, K // 2), dtype=torch.uint8, device="cuda")
    nsf = qfp4.sf_mma_bytes(rows, K // 32) if layout == qfp4.SF_MMA else rows * (K // 32)
    SF = torch.empty((nsf,), dtype=torch.uint8, device="cuda")
    qfp4.quantize(fmt, X, gs, Q, SF, layout)
    return Q, SF, gs


def prune_mask(rows, K, seed):
    """A random choice of 2 of every 4 pair bytes along K (all six patterns)."""
    gen = synth.rng(seed)
    pats = np.array([(a, b) for a in range(4) for b in range(a + 1, 4)])
    sel = pats[gen.integers(0, 6, (rows, K // 8))]
    mask = np.zeros((rows, K // 8, 4), bool)
    np.put_along_axis(mask, sel, True, axis=2)
    return mask.reshape(rows, K // 2)


def sparse_operands(M, N, K, seed):
    """Activations and pruned weights quantised on the device (bit-exact
    against the oracle), the weights compressed on the device (bit-exact),
    and the oracle's own operands for the reference."""
    xa = synth.activations_bf16(seed, M, K)
    xw = synth.weights_bf16(seed + 1, N, K)
    Qx, SFx, gx = quantize_dev(xa, layout=qfp4.SF_MMA)
    Qw, SFw, gw = quantize_dev(xw)
    gx_ref, gw_ref = oracle.global_scale(xa), oracle.global_scale(xw)
    qx_ref, sfx_ref = oracle.quantize(NV32, xa, gx_ref)
    qw_ref, sfw_ref = oracle.quantize(NV32, xw, gw_ref)
    torch.cuda.synchronize()
    assert np.float32(gx.item()) == gx_ref and np.float32(gw.item()) == gw_ref
    assert np.array_equal(to_host(Qx), qx_ref)
    assert np.array_equal(oracle.sf_from_mma(to_host(SFx), M, K // 32), sfx_ref)
    assert np.array_equal(to_host(Qw), qw_ref) and np.array_equal(to_host(SFw).reshape(N, K // 32), sfw_ref)
    mask = prune_mask(N, K, seed + 2)
    w_pruned = np.where(mask, qw_ref, 0).astype(np.uint8)
    Wc_ref, meta_ref = oracle.sparse24_compress(w_pruned)
    Wp = to_dev_u8(w_pruned)
    Wc = torch.empty((N, K // 4), dtype=torch.uint8, device="cuda")
    meta = torch.empty((qfp4.sparse24_meta_bytes(N, K, qfp4.SF_MMA),), dtype=torch.uint8, device="cuda")
    qfp4.sparse24_compress(Wp, Wc, meta, qfp4.SF_MMA)
    torch.cuda.synchronize()
    assert qfp4.poll_device_status() == 0
    assert np.array_equal(to_host(Wc), Wc_ref), "compressed weights"
    assert np.array_equal(to_host(meta), meta_rowmajor_to_tiled(meta_ref, N, K)), "tiled metadata"
    SFw_m = torch.empty((qfp4.sf_mma_bytes(N, K // 32),), dtype=torch.uint8, device="cuda")
    qfp4.sf_interleave(SFw, N, K // 32, SFw_m, qfp4.SF_MMA)
    dev = (Qx, SFx, Wc, meta, SFw_m, gx, gw)
    ref = (qx_ref, sfx_ref, Wc_ref, meta_ref, sfw_ref, gx_ref, gw_ref)
    return dev, ref


@pytest.mark.parametrize("M,N,K", [(256, 256, 512), (300, 512, 1024), (77, 256, 2048), (128, 768, 1536),
                                   (1000, 1024, 512), (513, 256, 4096)])
def test_sparse_gemm_vs_oracle(M, N, K):
    """One tile and one stage; ragged token counts (a pair's second token
    tile partly or wholly past M); several weight tiles; long K."""
    (Qx, SFx, Wc, meta, SFw, gx, gw), (qx, sfx, wc, mt, sfw, gxr, gwr) = sparse_operands(M, N, K, 9700 + M + N)
    outs = []
    for _ in range(2):
        D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        qfp4.gemm_nt_sparse24(NV32, M, N, K, Qx, SFx, Wc, meta, SFw, gx, gw, D)
        torch.cuda.synchronize()
        outs.append(bf16_to_f64(D))
    assert qfp4.poll_device_status() == 0
    assert np.array_equal(outs[0], outs[1]), "repeated launches differ"
    d_ref, t_ref = oracle.gemm_nt_sparse24(NV32, qx, sfx, wc, mt, sfw, gxr, gwr)
    assert_gemm_close(outs[0], d_ref, t_ref, f"sparse {M}x{N}x{K}")


def test_sparse_gemm_two_level():
    """Per-row (token) and per-column (weight row) fp32 rescale in the
    epilogue, as the deployed two-level sparse kernel does."""
    M, N, K = 300, 512, 1024
    (Qx, SFx, Wc, meta, SFw, gx, gw), (qx, sfx, wc, mt, sfw, gxr, gwr) = sparse_operands(M, N, K, 9800)
    gen = synth.rng(9801)
    rs = (np.exp(gen.normal(0, 1.0, M)) * np.where(gen.random(M) < 0.1, -1, 1)).astype(np.float32)
    cs = np.exp(gen.normal(0, 1.0, N)).astype(np.float32)
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    qfp4.gemm_nt_sparse24(NV32, M, N, K, Qx, SFx, Wc, meta, SFw, gx, gw, D,
                          torch.from_numpy(rs).cuda(), torch.from_numpy(cs).cuda())
    torch.cuda.synchronize()
    assert qfp4.poll_device_status() == 0
    W = oracle.sparse24_decompress(wc, mt, K)
    d_ref, t_ref = oracle.gemm_nt(NV32, qx, sfx, W, sfw, gxr, gwr, row_scale=rs, col_scale=cs)
    assert_gemm_close(bf16_to_f64(D), d_ref, t_ref, "sparse two-level")


def test_sparse_gemm_one_hot_positions():
    """Kept elements 1.0 at unit scales, one A element per row: D[m, n] is
    x[m, k] summed over exactly the dense positions k row n keeps, for every
    metadata pattern, with -0 pairs (codes 8) among the kept ones."""
    M, N, K = 256, 256, 512
    gen = synth.rng(9900)
    mask = prune_mask(N, K, 9901)
    wb = np.where(mask, np.uint8(0x22), np.uint8(0)).astype(np.uint8)     # kept pairs: 1.0, 1.0
    neg0 = mask & (gen.random(mask.shape) < 0.1)
    wb = np.where(neg0, np.uint8(0x88), wb)                                # some kept pairs -0, -0
    xa = np.zeros((M, K), np.uint8)
    xa[np.arange(M), (np.arange(M) * 37) % K] = 4                          # 2.0 at one k per row
    qx = (xa[:, 0::2] | (xa[:, 1::2] << 4)).astype(np.uint8)
    sfx = np.full((M, K // 32), 0x38, np.uint8)
    sfw = np.full((N, K // 32), 0x38, np.uint8)
    Wc_ref, meta_ref = oracle.sparse24_compress(wb)
    Wc = torch.empty((N, K // 4), dtype=torch.uint8, device="cuda")
    meta = torch.empty((qfp4.sparse24_meta_bytes(N, K, qfp4.SF_MMA),), dtype=torch.uint8, device="cuda")
    qfp4.sparse24_compress(to_dev_u8(wb), Wc, meta, qfp4.SF_MMA)
    SFx = torch.zeros((qfp4.sf_mma_bytes(M, K // 32),), dtype=torch.uint8, device="cuda")
    SFw = torch.zeros((qfp4.sf_mma_bytes(N, K // 32),), dtype=torch.uint8, device="cuda")
    qfp4.sf_interleave(to_dev_u8(sfx), M, K // 32, SFx, qfp4.SF_MMA)
    qfp4.sf_interleave(to_dev_u8(sfw), N, K // 32, SFw, qfp4.SF_MMA)
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    qfp4.gemm_nt_sparse24(NV32, M, N, K, to_dev_u8(qx), SFx, Wc, meta, SFw, None, None, D)
    torch.cuda.synchronize()
    assert qfp4.poll_device_status() == 0
    assert np.array_equal(to_host(Wc), Wc_ref)
    d = bf16_to_f64(D)
    k_of = (np.arange(M) * 37) % K
    dense_w = oracle.dequantize(NV32, wb, sfw)                          # [N, K], the kept 1.0 / -0 values
    want = 2.0 * dense_w[:, k_of].T                                     # [M, N]
    assert np.array_equal(d, want)


def test_compress_rowmajor_and_rejects_non_sparse():
    rows, K = 130, 256
    mask = prune_mask(rows, K, 9950)
    w = np.where(mask, synth.rng(9951).integers(0, 256, (rows, K // 2), dtype=np.uint8), 0).astype(np.uint8)
    Wc_ref, meta_ref = oracle.sparse24_compress(w)
    Wc = torch.empty((rows, K // 4), dtype=torch.uint8, device="cuda")
    meta = torch.empty((qfp4.sparse24_meta_bytes(rows, K, qfp4.SF_ROWMAJOR),), dtype=torch.uint8, device="cuda")
    qfp4.sparse24_compress(to_dev_u8(w), Wc, meta, qfp4.SF_ROWMAJOR)
    torch.cuda.synchronize()
    assert qfp4.poll_device_status() == 0
    assert np.array_equal(to_host(Wc), Wc_ref) and np.array_equal(to_host(meta).reshape(rows, K // 16), meta_ref)
    bad = w.copy()
    bad[7, 8:12] = 0x11                        # four non-zero pairs in one group
    qfp4.sparse24_compress(to_dev_u8(bad), Wc, meta, qfp4.SF_ROWMAJOR)
    torch.cuda.synchronize()
    assert qfp4.poll_device_status() == INVALID
    assert qfp4.poll_device_status() == 0


def test_sparse_gemm_full_size_square():
    """Square 8192 (the headline sparse shape), sampled outputs against the
    oracle on the decompressed weights."""
    M = N = K = 8192
    xa = synth.activations_bf16(9960, M, K)
    xw = synth.weights_bf16(9961, N, K)
    Qx, SFx, gx = quantize_dev(xa, layout=qfp4.SF_MMA)
    Qw, SFw, gw = quantize_dev(xw)
    mask = torch.from_numpy(prune_mask(N, K, 9962)).cuda()
    Wp = torch.where(mask, Qw, torch.zeros_like(Qw))
    Wc = torch.empty((N, K // 4), dtype=torch.uint8, device="cuda")
    meta = torch.empty((qfp4.sparse24_meta_bytes(N, K, qfp4.SF_MMA),), dtype=torch.uint8, device="cuda")
    qfp4.sparse24_compress(Wp, Wc, meta, qfp4.SF_MMA)
    SFw_m = torch.empty((qfp4.sf_mma_bytes(N, K // 32),), dtype=torch.uint8, device="cuda")
    qfp4.sf_interleave(SFw, N, K // 32, SFw_m, qfp4.SF_MMA)
    D = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    qfp4.gemm_nt_sparse24(NV32, M, N, K, Qx, SFx, Wc, meta, SFw_m, gx, gw, D)
    torch.cuda.synchronize()
    assert qfp4.poll_device_status() == 0
    rows = np.array([0, 255, 256, 4097, 8191])
    gen = synth.rng(9963)
    mi = np.concatenate([np.repeat(rows, 64), gen.integers(0, M, 3000)])
    ni = np.concatenate([np.tile(gen.integers(0, N, 64), len(rows)), gen.integers(0, N, 3000)])
    gx_ref = oracle.global_scale(xa)
    gw_ref = oracle.global_scale(xw)
    qx_ref, sfx_ref = oracle.quantize(NV32, xa[np.unique(mi)], gx_ref)
    remap = {m: i for i, m in enumerate(np.unique(mi))}
    nsel = np.unique(ni)
    qw_ref, sfw_ref = oracle.quantize(NV32, xw[nsel], gw_ref)
    wp = np.where(to_host(mask)[nsel], qw_ref, 0).astype(np.uint8)
    nmap = {n: i for i, n in enumerate(nsel)}
    d_ref, t_ref = oracle.gemm_nt_entries(NV32, qx_ref, sfx_ref, wp, sfw_ref, gx_ref, gw_ref,
                                          np.array([remap[m] for m in mi]), np.array([nmap[n] for n in ni]))
    d = bf16_to_f64(D)[mi, ni]
    assert_gemm_close(d, d_ref, t_ref, "sparse 8192^3 sampled")
