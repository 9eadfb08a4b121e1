"""GPU parity of the HBM-bound kernels against the CPU oracle, bit-exact:
global scale, quantiser (row-major and MMA scale layouts, grouped) and the
scale-factor interleave."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_tcgen05_gb300 import qfp4, synth
from tests._helpers import MX, NV, dev_scalar, to_dev_bf16, to_dev_u8, to_host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    qfp4.load()
    assert qfp4.device_check() == 0


def quantize_dev(fmt, xbits, gs, layout=qfp4.SF_ROWMAJOR):
    M, K = xbits.shape
    g = qfp4.block_size(fmt)
    X = to_dev_bf16(xbits)
    Q = torch.full((M, K // 2), 0xAB, dtype=torch.uint8, device="cuda")
    if layout == qfp4.SF_ROWMAJOR:
        SF = torch.full((M, K // g), 0xCD, dtype=torch.uint8, device="cuda")
    else:
        SF = torch.full((qfp4.sf_mma_bytes(M, K // g),), 0xCD, dtype=torch.uint8, device="cuda")
    qfp4.quantize(fmt, X, dev_scalar(gs) if gs is not None else None, Q, SF, layout)
    torch.cuda.synchronize()
    return to_host(Q), to_host(SF)


def check_quantize(fmt, xbits, gs):
    q_ref, sf_ref = oracle.quantize(fmt, xbits, gs if gs is not None else 1.0)
    Q, SF = quantize_dev(fmt, xbits, gs, qfp4.SF_ROWMAJOR)
    bad = np.argwhere(Q != q_ref)
    assert bad.size == 0, f"{len(bad)} packed bytes differ, first {bad[:5].tolist()}"
    assert np.array_equal(SF, sf_ref)
    Q2, SFm = quantize_dev(fmt, xbits, gs, qfp4.SF_MMA)
    assert np.array_equal(Q2, q_ref)
    assert np.array_equal(SFm, oracle.sf_to_mma(sf_ref))


@pytest.mark.parametrize("fmt", [MX, NV])
@pytest.mark.parametrize("M,K", [(1, 128), (37, 384), (130, 1024), (256, 4096)])
def test_quantize_activations_bitexact(fmt, M, K):
    x = synth.activations_bf16(1000 + M + K, M, K)
    gs = oracle.global_scale(x) if fmt == NV else None
    check_quantize(fmt, x, gs)


@pytest.mark.parametrize("fmt", [MX, NV])
def test_quantize_weights_bitexact(fmt):
    x = synth.weights_bf16(77, 512, 2048)
    check_quantize(fmt, x, oracle.global_scale(x) if fmt == NV else None)


@pytest.mark.parametrize("fmt", [MX, NV])
def test_quantize_special_values(fmt):
    """Zero blocks, bf16 subnormals, huge values, signed zeros, mixed scales."""
    gen = synth.rng(5)
    rows = []
    rows.append(np.zeros(256, np.float32))
    rows.append(np.full(256, -0.0, np.float32))
    rows.append((gen.standard_normal(256) * 1e-39).astype(np.float32))      # subnormal bf16
    rows.append((gen.standard_normal(256) * 1e37).astype(np.float32))
    r = gen.standard_normal(256).astype(np.float32)
    r[::7] = 0.0
    r[1::7] = -0.0
    rows.append(r)
    rows.append(np.geomspace(1e-30, 1e30, 256).astype(np.float32) * np.where(np.arange(256) % 2, -1, 1))
    x = synth.f32_to_bf16_bits(np.stack(rows))
    # gs = 0 is what an all-zero tensor gets: (amax / 6) / gs is then NaN or
    # +inf, and NaN must take scale code 0 like the oracle's rounding does
    for gs in ([None] if fmt == MX else [np.float32(1.0), np.float32(3.1e-3), np.float32(1e-30),
                                          np.float32(7e25), oracle.global_scale(x), np.float32(0.0)]):
        check_quantize(fmt, x, gs)


def test_quantize_on_grid_roundtrip_exact_ties():
    """Inputs exactly on midpoints of the E2M1 grid times a power-of-two scale:
    every element is an exact tie and must go to the even code."""
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    for fmt, gs in ((MX, None), (NV, np.float32(0.125))):
        g = qfp4.block_size(fmt)
        blocks = []
        for sc in (2.0 ** -3, 1.0, 2.0 ** 5):
            for sign in (1.0, -1.0):
                b = np.zeros(g, np.float32)
                b[0] = 6.0 * sc * (1.0 if gs is None else gs)
                b[1:8] = sign * mids * sc * (1.0 if gs is None else gs)
                blocks.append(b)
        x = synth.f32_to_bf16_bits(np.concatenate(blocks).reshape(1, -1))
        pad = (-x.shape[1]) % 128
        x = np.pad(x, ((0, 0), (0, pad)))
        check_quantize(fmt, x, gs)


def test_quantize_nvfp4_near_ties():
    """NVFP4 with global scales tuned so x / s lands within a few fp32 ulps of
    an E2M1 midpoint: the quotient must be the correctly rounded one."""
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    x0 = np.float32(1.0)
    count = 0
    for m in mids:
        for code in (0x30, 0x3B, 0x46, 0x52):
            dec = np.float32(oracle.ue4m3_value(code))
            gs0 = np.float32(x0 / (np.float32(m) * dec))
            for k in range(-3, 4):
                gs = gs0
                for _ in range(abs(k)):
                    gs = np.nextafter(gs, np.float32(np.inf if k > 0 else 0), dtype=np.float32)
                amax_el = np.float32(6.0) * dec * gs
                row = np.zeros(128, np.float32)
                row[0] = amax_el
                row[1] = x0
                row[2] = -x0
                row[3] = np.float32(x0 * 1.5)
                xb = synth.f32_to_bf16_bits(row.reshape(1, -1))
                check_quantize(NV, xb, gs)
                count += 1
    assert count == 7 * 4 * 7


@pytest.mark.parametrize("fmt", [MX, NV])
def test_quantize_full_size_16384x4096(fmt):
    """The decode-batch quantizer workload at full size, bit-exact."""
    x = synth.activations_bf16(synth.QUANT_SEED, synth.QUANT_ROWS, synth.QUANT_COLS)
    gs = oracle.global_scale(x) if fmt == NV else None
    q_ref, sf_ref = oracle.quantize(fmt, x, gs if gs is not None else 1.0)
    Q, SFm = quantize_dev(fmt, x, gs, qfp4.SF_MMA)
    assert np.array_equal(Q, q_ref)
    assert np.array_equal(SFm, oracle.sf_to_mma(sf_ref))


@pytest.mark.parametrize("rows,cols", [(1, 8), (16, 16), (200, 64), (4096, 256), (16384, 256)])
def test_global_scale_bitexact(rows, cols):
    x = synth.activations_bf16(rows * 7 + cols, rows, cols)
    gs = torch.empty(1, dtype=torch.float32, device="cuda")
    qfp4.global_scale(to_dev_bf16(x), gs)
    torch.cuda.synchronize()
    assert np.float32(gs.item()) == oracle.global_scale(x)


def test_global_scale_many_launches():
    """The one-tensor global scale reduces through a pool of device slots that
    every launch hands back at zero: more launches than the pool has slots,
    back to back on one stream, on tensors whose maxima differ (and an empty
    and an all-zero one among them), each bit-exact."""
    shapes = [(1, 8), (3, 16), (130, 64), (0, 8), (257, 40)]
    xs = []
    for i, (r, c) in enumerate(shapes):
        x = synth.activations_bf16(4000 + i, r, c) if r else np.zeros((0, c), np.uint16)
        xs.append((to_dev_bf16(x) if r else torch.zeros((1, c), dtype=torch.bfloat16, device="cuda"), r, c,
                   oracle.global_scale(x) if r else np.float32(0.0)))
    zero = torch.zeros((5, 24), dtype=torch.bfloat16, device="cuda")
    n = 1100 + 7
    out = torch.full((n,), -1.0, dtype=torch.float32, device="cuda")
    want = []
    for k in range(n):
        if k % 11 == 5:
            qfp4.global_scale(zero, out[k:k + 1])
            want.append(np.float32(0.0))
        else:
            X, r, c, w = xs[k % len(xs)]
            qfp4.global_scale(X[:r] if r else X[:0], out[k:k + 1])
            want.append(w)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(out), np.array(want, dtype=np.float32))


def test_global_scale_grouped_many_launches():
    """The per-group global scales reduce through a pool of 64 device slots:
    more launches than that, alternating the two entry points (row count on
    the host, row count read on the device) and group layouts with empty
    groups, each bit-exact against the oracle per group."""
    layouts = [np.array([5, 0, 130, 1], dtype=np.int64), np.array([0, 0, 64], dtype=np.int64),
               np.array([300, 17, 0, 0, 2, 9, 1, 44], dtype=np.int64)]
    cases = []
    for i, counts in enumerate(layouts):
        offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
        x = synth.activations_bf16(5000 + i, int(offs[-1]), 96)
        want = np.array([oracle.global_scale(x[offs[e]:offs[e + 1]]) if counts[e] else np.float32(0.0)
                         for e in range(len(counts))], dtype=np.float32)
        cases.append((to_dev_bf16(x), torch.from_numpy(offs).cuda(), want))
    results = []
    for k in range(70):
        X, d_offs, want = cases[k % len(cases)]
        gs = torch.full((len(want),), -1.0, dtype=torch.float32, device="cuda")
        if k % 2:
            qfp4.absmax_gs(d_offs, X, gs)
        else:
            qfp4.global_scale_grouped(X, d_offs, gs)
        results.append((gs, want))
    torch.cuda.synchronize()
    assert qfp4.poll_device_status() == 0
    for k, (gs, want) in enumerate(results):
        assert np.array_equal(to_host(gs), want), k


def test_global_scale_grouped_bitexact():
    counts = synth.moe_counts(5)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    x = synth.activations_bf16(9, int(offs[-1]), 512)
    gs = torch.empty(len(counts), dtype=torch.float32, device="cuda")
    qfp4.global_scale_grouped(to_dev_bf16(x), torch.from_numpy(offs).cuda(), gs)
    torch.cuda.synchronize()
    got = to_host(gs)
    for e in range(len(counts)):
        seg = x[offs[e]:offs[e + 1]]
        want = oracle.global_scale(seg) if seg.size else np.float32(0.0)
        assert got[e] == want, e


@pytest.mark.parametrize("fmt", [MX, NV])
def test_quantize_grouped_bitexact(fmt):
    counts = np.array([5, 0, 130, 128, 1, 300, 0, 77], dtype=np.int64)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    K = 512
    g = qfp4.block_size(fmt)
    x = synth.activations_bf16(11, int(offs[-1]), K)
    gs_host = np.array([oracle.global_scale(x[offs[e]:offs[e + 1]]) if counts[e] else np.float32(1.0)
                        for e in range(len(counts))], dtype=np.float32)
    Q = torch.empty((int(offs[-1]), K // 2), dtype=torch.uint8, device="cuda")
    SF = torch.full((qfp4.sf_mma_grouped_bytes(int(offs[-1]), len(counts), K // g),), 0xEE,
                    dtype=torch.uint8, device="cuda")
    qfp4.quantize_grouped(fmt, to_dev_bf16(x), torch.from_numpy(offs).cuda(),
                          torch.from_numpy(gs_host).cuda() if fmt == NV else None, Q, SF)
    torch.cuda.synchronize()
    Qh, SFh = to_host(Q), to_host(SF)
    tile = 0
    for e in range(len(counts)):
        if counts[e] == 0:
            continue
        q_ref, sf_ref = oracle.quantize(fmt, x[offs[e]:offs[e + 1]], gs_host[e] if fmt == NV else 1.0)
        assert np.array_equal(Qh[offs[e]:offs[e + 1]], q_ref), e
        ref_mma = oracle.sf_to_mma(sf_ref)
        start = tile * (K // g // 4) * 512
        assert np.array_equal(SFh[start:start + ref_mma.size], ref_mma), e
        tile += -(-int(counts[e]) // 128)
    assert SFh[tile * (K // g // 4) * 512:].max(initial=0) == 0


@pytest.mark.parametrize("rows,cols", [(1, 1), (128, 4), (129, 7), (64, 16), (130, 48), (300, 64), (4096, 256),
                                       (8192, 512)])
def test_sf_interleave_bitexact(rows, cols):
    sf = synth.rng(rows + cols).integers(0, 255, size=(rows, cols), dtype=np.uint8)
    out = torch.full((qfp4.sf_mma_bytes(rows, cols),), 0x5A, dtype=torch.uint8, device="cuda")
    qfp4.sf_interleave(to_dev_u8(sf), rows, cols, out, qfp4.SF_MMA)
    back = torch.zeros((rows, cols), dtype=torch.uint8, device="cuda")
    qfp4.sf_interleave(out, rows, cols, back, qfp4.SF_ROWMAJOR)
    torch.cuda.synchronize()
    assert np.array_equal(to_host(out), oracle.sf_to_mma(sf))
    assert np.array_equal(to_host(back), sf)


def test_quantize_all_zero_tensor_nvfp4():
    """An all-zero tensor: global scale 0, every block scale code 0 and every
    element code 0, through the device global scale and the quantiser."""
    x = np.zeros((130, 512), np.uint16)
    X = to_dev_bf16(x)
    gs = torch.full((1,), -1.0, dtype=torch.float32, device="cuda")
    qfp4.global_scale(X, gs)
    torch.cuda.synchronize()
    assert gs.item() == 0.0 == oracle.global_scale(x)
    check_quantize(NV, x, np.float32(0.0))


# ----------------------------------------------------------------- exhaustive element path

def exhaustive_input(fmt, gs):
    """Every (scale code, element) pair the quantiser can meet for this gs:
    for each reachable scale code c, blocks whose first element is the largest
    positive bf16 value that yields c, filled with every bf16 value (both
    signs, and +-0) of magnitude at most that value."""
    g = qfp4.block_size(fmt)
    per_row = 128 // g if fmt == NV else 256 // g          # rows of 128 (NV) or 256 (MX) elements
    pos = np.arange(1, 0x7F80, dtype=np.uint16)             # positive finite bf16
    nb = len(pos)
    probe = np.zeros(((nb + per_row - 1) // per_row * per_row, g), np.uint16)
    probe[:nb, 0] = pos
    _, sf = oracle.quantize(fmt, probe.reshape(-1, per_row * g), gs)
    codes = sf.reshape(-1)[:nb]
    blocks = []
    for c in np.unique(codes):
        amax = pos[codes == c].max()
        mags = pos[pos <= amax]
        vals = np.concatenate([mags, mags | 0x8000, np.array([0, 0x8000], np.uint16)])
        fill = g - 1
        nblk = (len(vals) + fill - 1) // fill
        b = np.zeros((nblk, g), np.uint16)
        b[:, 0] = amax
        flat = np.zeros(nblk * fill, np.uint16)
        flat[:len(vals)] = vals
        b[:, 1:] = flat.reshape(nblk, fill)
        blocks.append(b)
    allb = np.concatenate(blocks)
    pad = (-len(allb)) % per_row
    allb = np.concatenate([allb, np.zeros((pad, g), np.uint16)])
    return allb.reshape(-1, per_row * g), len(np.unique(codes))


@pytest.mark.parametrize("fmt,gs", [(NV, np.float32(1.0)), (NV, np.float32(0.01371)),
                                    (NV, np.float32(7.3e-6)), (MX, None)])
def test_quantize_exhaustive_element_path(fmt, gs):
    """Bit-exact against the oracle over every bf16 element value with every
    reachable scale code (a few million elements per case): pins the scale
    encoding, the quotient x / s and its E2M1 rounding at every input the
    kernel can see for this global scale."""
    x, ncodes = exhaustive_input(fmt, gs if gs is not None else np.float32(1.0))
    assert ncodes >= (100 if fmt == NV else 200)
    check_quantize(fmt, x, gs)


def every_amax_input(seed):
    """One NVFP4 block per positive finite bf16 magnitude v (bit patterns
    0x0000..0x7F7F): v at a random position, the other 15 elements random
    fractions of v (rounded to bf16, so never above v), every sign random;
    rows of 256 blocks, zero-padded."""
    gen = synth.rng(seed)
    vals = np.arange(0, 0x7F80, dtype=np.uint32)
    amax = (vals << 16).view(np.float32)
    n = len(vals)
    others = synth.f32_to_bf16_bits(amax[:, None] * gen.random((n, 15)).astype(np.float32))
    blk = np.concatenate([vals.astype(np.uint16)[:, None], others], axis=1)
    blk = np.take_along_axis(blk, gen.permuted(np.tile(np.arange(16), (n, 1)), axis=1), axis=1)
    blk = np.where(gen.random((n, 16)) < 0.5, blk | np.uint16(0x8000), blk).astype(np.uint16)
    pad = (-n) % 256
    blk = np.concatenate([blk, np.zeros((pad, 16), np.uint16)])
    return blk.reshape(-1, 256 * 16)


_RANDOM_GS = [np.float32(2.0 ** e) for e in synth.rng(12).uniform(-100.0, 100.0, 4)]


@pytest.mark.parametrize("gs", [np.float32(1.0), np.float32(0.01371), np.float32(7.3e-6), np.float32(3.1e-3),
                                np.float32(1e-30), np.float32(7e25), np.float32(2.0 ** -100),
                                np.float32(2.0 ** 100), np.float32(2.0 ** -101), np.float32(1.5 * 2.0 ** 100)]
                         + _RANDOM_GS)
def test_quantize_nvfp4_every_block_amax(gs):
    """Bit-exact against the oracle with every positive finite bf16 magnitude
    as the maximum of some block: pins the scale code of every amax a
    per-tensor NVFP4 quantisation can see, for global scales inside and just
    outside [2^-100, 2^100] (where the kernel reads codes from a table built
    at launch) and for random ones across that range."""
    check_quantize(NV, every_amax_input(31), gs)


def quantize_grouped_check(x, counts, gs_host):
    """Grouped NVFP4 quantisation of x (bf16 bits) against the oracle, group
    by group: codes and per-group MMA-layout scale tiles, bit-exact."""
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    K = x.shape[1]
    Q = torch.empty((int(offs[-1]), K // 2), dtype=torch.uint8, device="cuda")
    SF = torch.full((qfp4.sf_mma_grouped_bytes(int(offs[-1]), len(counts), K // 16),), 0xEE,
                    dtype=torch.uint8, device="cuda")
    qfp4.quantize_grouped(NV, to_dev_bf16(x), torch.from_numpy(offs).cuda(), torch.from_numpy(gs_host).cuda(), Q, SF)
    torch.cuda.synchronize()
    Qh, SFh = to_host(Q), to_host(SF)
    tile = 0
    for e in range(len(counts)):
        if counts[e] == 0:
            continue
        q_ref, sf_ref = oracle.quantize(NV, x[offs[e]:offs[e + 1]], gs_host[e])
        assert np.array_equal(Qh[offs[e]:offs[e + 1]], q_ref), e
        ref_mma = oracle.sf_to_mma(sf_ref)
        start = tile * (K // 64) * 512
        assert np.array_equal(SFh[start:start + ref_mma.size], ref_mma), e
        tile += -(-int(counts[e]) // 128)


def test_quantize_grouped_nvfp4_every_block_amax():
    """Every positive finite bf16 magnitude as a block maximum in each of four
    groups with their own global scales: two inside the scale-code tables'
    range, one below it (per-block arithmetic for that group only) and one
    far above; bit-exact against the oracle."""
    x = every_amax_input(31)                     # 128 rows, every magnitude once
    # four groups of 128 rows, each with every magnitude once (rolls by whole blocks)
    x = np.concatenate([x, np.roll(x, 16, axis=1), np.roll(x, 160, axis=1), x[::-1]])
    gs_host = np.array([1.0, 0.0137, 2.0 ** -101, 7e25], dtype=np.float32)
    quantize_grouped_check(x, np.array([128, 128, 128, 128]), gs_host)


def test_quantize_grouped_nvfp4_more_groups_than_tables():
    """Twelve groups (more than the kernel keeps scale-code tables for), with
    ragged and empty groups: each group's gs and RN(1/gs) come from shared
    memory and the per-block arithmetic; bit-exact against the oracle."""
    counts = np.array([33, 0, 140, 1, 256, 7, 0, 129, 64, 3, 300, 17], dtype=np.int64)
    x = synth.activations_bf16(23, int(counts.sum()), 1024)
    offs = np.concatenate([[0], np.cumsum(counts)])
    gs_host = np.array([oracle.global_scale(x[offs[e]:offs[e + 1]]) if counts[e] else np.float32(1.0)
                        for e in range(len(counts))], dtype=np.float32)
    gs_host[4] = np.float32(2.0 ** -110)
    quantize_grouped_check(x, counts, gs_host)
