"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each test ties one oracle function to a closed form, a library conversion
(torch's float8 types), a brute-force search, an invariant of the method, or
a value printed on the pages / worked by hand from the format definitions
(fixtures under tests/golden/).  No GPU is used.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_tcgen05_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
MX, NV, NV32 = oracle.MXFP4, oracle.NVFP4, oracle.NVFP4_B32


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _e2m1_golden():
    vals = {}
    for code, val, negzero in _golden_rows("e2m1_values.txt"):
        vals[int(code)] = (float(val), int(negzero))
    return vals


E2M1 = _e2m1_golden()
GRID = np.array([E2M1[c][0] for c in range(8)], dtype=np.float64)


# --------------------------------------------------------------------------
# decoding
# --------------------------------------------------------------------------

def test_e2m1_decode_matches_format_table():
    for code in range(16):
        v = oracle.e2m1_value(code)
        want, negzero = E2M1[code]
        assert v == want
        assert math.copysign(1.0, v) < 0 if negzero else True


def test_e2m1_products_bruteforce():
    """All 256 code x code products equal the table products, exactly."""
    seen = set()
    for a in range(16):
        for b in range(16):
            p = oracle.e2m1_value(a) * oracle.e2m1_value(b)
            assert Fraction(p) == Fraction(E2M1[a][0]) * Fraction(E2M1[b][0])
            seen.add(abs(p))
    assert max(seen) == 36.0
    assert len(seen) == len({abs(x * y) for x in GRID for y in GRID})


def test_ue4m3_decode_vs_torch_float8():
    codes = torch.arange(0, 0x7F, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).tolist()
    for c, r in zip(codes.tolist(), ref):
        assert oracle.ue4m3_value(c) == r
    assert oracle.ue4m3_value(0x7E) == 448.0
    assert oracle.ue4m3_value(0x08) == 2.0 ** -6
    assert oracle.ue4m3_value(0x01) == 2.0 ** -9
    assert math.isnan(oracle.ue4m3_value(0x7F))
    assert math.isnan(oracle.ue4m3_value(0x80))


def test_ue8m0_decode_vs_closed_form_and_torch():
    codes = torch.arange(0, 255, dtype=torch.uint8)
    ref = codes.view(torch.float8_e8m0fnu).to(torch.float64).tolist()
    for c, r in zip(codes.tolist(), ref):
        v = oracle.ue8m0_value(c)
        assert v == math.ldexp(1.0, c - 127)
        assert v == r
    assert math.isnan(oracle.ue8m0_value(255))


# --------------------------------------------------------------------------
# rounding
# --------------------------------------------------------------------------

def _nearest_even_grid(q):
    """Brute force: nearest magnitude on the grid, tie -> even code, sign kept."""
    q = np.asarray(q, dtype=np.float32)
    # beyond 7 every input is nearest to 6; clamping keeps the fp64 distances exact
    a = np.minimum(np.abs(q.astype(np.float64)), 7.0)
    d = np.abs(a[:, None] - GRID[None, :])
    idx = np.argmin(d, axis=1)                    # first (lower) index on ties
    nxt = np.minimum(idx + 1, 7)
    tie = (d[np.arange(a.size), nxt] == d[np.arange(a.size), idx]) & (nxt != idx)
    idx = np.where(tie & (idx % 2 == 1), nxt, idx)
    return (idx | np.where(np.signbit(q), 8, 0)).astype(np.uint8)


def test_e2m1_round_hand_cases():
    for inp, code in _golden_rows("e2m1_rounding_cases.txt"):
        assert oracle.e2m1_round(np.float32(float(inp))) == int(code), inp


def test_e2m1_round_bruteforce_random():
    gen = synth.rng(7)
    q = np.concatenate([
        gen.uniform(-7.5, 7.5, 200_000).astype(np.float32),
        (gen.standard_normal(50_000) * 3).astype(np.float32),
    ])
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], dtype=np.float32)
    near = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(9))])
    q = np.concatenate([q, near, -near, np.float32([0.0, -0.0, 6.0, -6.0, 1e30, -1e30])])
    got = oracle.e2m1_round_array(q)
    want = _nearest_even_grid(q)
    assert np.array_equal(got, want)


def test_scale_round_hand_cases():
    for fmt, t, code in _golden_rows("scale_rounding_cases.txt"):
        fn = oracle.ue8m0_round if fmt == "ue8m0" else oracle.ue4m3_round
        assert fn(np.float32(float(t))) == int(code), (fmt, t)


def test_ue4m3_round_vs_torch_float8():
    """Below the 448/480 tie torch's float8_e4m3fn conversion is RNE with
    subnormals, exactly the rounding the scale rule asks for."""
    gen = synth.rng(11)
    t = np.concatenate([
        np.exp(gen.uniform(np.log(1e-5), np.log(463.0), 20_000)).astype(np.float32),
        gen.uniform(0, 0.02, 5_000).astype(np.float32),
    ])
    vals = np.array([oracle.ue4m3_value(c) for c in range(0x7F)], dtype=np.float64)
    mids = ((vals[:-1] + vals[1:]) / 2).astype(np.float32)   # exact in fp32
    t = np.concatenate([t, mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9))])
    t = t[t < 464.0]
    ref = torch.from_numpy(t).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.ue4m3_round(v) for v in t], dtype=np.uint8)
    assert np.array_equal(got, ref)


def test_ue8m0_round_vs_torch_away_from_ties():
    """torch's float8_e8m0fnu conversion rounds to nearest (ties upward); away
    from the exact 1.5*2^e ties it must agree with round-to-nearest-even."""
    gen = synth.rng(13)
    t = np.exp(gen.uniform(np.log(1e-30), np.log(1e30), 20_000)).astype(np.float32)
    m, _ = np.frexp(t)
    t = t[m != 0.75]
    ref = torch.from_numpy(t).to(torch.float8_e8m0fnu).view(torch.uint8).numpy()
    got = np.array([oracle.ue8m0_round(v) for v in t], dtype=np.uint8)
    assert np.array_equal(got, ref)
    # exact ties: the even code
    for e in range(-20, 21):
        t = np.float32(1.5 * 2.0 ** e)
        lo = e + 127
        assert oracle.ue8m0_round(t) == (lo if lo % 2 == 0 else lo + 1)


# --------------------------------------------------------------------------
# quantiser
# --------------------------------------------------------------------------

def _grid_blocks(fmt, rows, blocks, seed, gs):
    """Inputs already on the grid code * scale * gs, with a +-6 in every block
    so that the block's own scale is recovered exactly."""
    g = oracle.block_size(fmt)
    gen = synth.rng(seed)
    codes = gen.integers(0, 16, size=(rows, blocks, g))
    pos6 = gen.integers(0, g, size=(rows, blocks))
    sign6 = gen.integers(0, 2, size=(rows, blocks)) * 8
    np.put_along_axis(codes, pos6[..., None], (7 + sign6)[..., None], axis=2)
    if fmt == MX:
        sfb = gen.integers(110, 145, size=(rows, blocks))
    else:
        sfb = gen.integers(1, 0x7F, size=(rows, blocks))
    x = np.zeros((rows, blocks, g), dtype=np.float64)
    for r in range(rows):
        for b in range(blocks):
            s = (oracle.ue8m0_value(sfb[r, b]) if fmt == MX else oracle.ue4m3_value(sfb[r, b])) * gs
            x[r, b] = [math.copysign(E2M1[c][0], -1.0 if c >= 8 else 1.0) * s for c in codes[r, b]]
    return x.reshape(rows, blocks * g).astype(np.float32), codes.reshape(rows, blocks * g), sfb


@pytest.mark.parametrize("fmt,gs", [(MX, 1.0), (NV, 1.0), (NV, 2.0 ** -3), (NV, 2.0 ** 5), (NV32, 2.0 ** -3)])
def test_quantize_roundtrip_exact_on_grid(fmt, gs):
    x, codes, sfb = _grid_blocks(fmt, 6, 8, 21 + fmt, gs)
    assert np.array_equal(x.astype(np.float64) / 1.0, x)     # representable
    Q, SF = oracle.quantize(fmt, x, gs)
    assert np.array_equal(SF, sfb.astype(np.uint8))
    lo, hi = Q & 15, Q >> 4
    got = np.stack([lo, hi], axis=-1).reshape(codes.shape)
    assert np.array_equal(got, codes.astype(np.uint8))
    back = oracle.dequantize(fmt, Q, SF, gs)
    assert np.array_equal(back, x.astype(np.float64))


def test_quantize_zero_block_and_saturation():
    x = np.zeros((1, 32), dtype=np.float32)
    Q, SF = oracle.quantize(NV, x, 0.5)
    assert SF.tolist() == [[0, 0]] and Q.max() == 0
    Q, SF = oracle.quantize(MX, x, 1.0)
    assert SF.tolist() == [[0]] and Q.max() == 0
    # an all-zero tensor has global scale 0; t = (0/6)/0 is NaN and takes
    # scale code 0 like t = 0, and a non-zero block with gs = 0 has t = +inf,
    # which saturates to 0x7E while s = 448 * 0 = 0 still zeroes its elements
    assert oracle.global_scale(np.zeros((2, 16), np.uint16)) == 0.0
    Q, SF = oracle.quantize(NV, x, 0.0)
    assert SF.tolist() == [[0, 0]] and Q.max() == 0
    y = np.zeros((1, 32), dtype=np.float32)
    y[0, 20] = 1.0
    Q, SF = oracle.quantize(NV, y, 0.0)
    assert SF.tolist() == [[0, 0x7E]] and Q.max() == 0
    # NVFP4 scale saturation: t = amax/6/gs of 448, 464, 470, 1e6 -> 0x7E
    for t in (448.0, 464.0, 470.0, 1e6):
        x = np.zeros((1, 16), dtype=np.float32)
        x[0, 3] = np.float32(t * 6)
        Q, SF = oracle.quantize(NV, x, 1.0)
        assert SF[0, 0] == 0x7E
        # q = 6t/448 > 6 for t > 448: saturates to code 7, nibble of element 3
        assert (Q[0, 1] >> 4) == 7


def test_quantize_hand_worked_mx_block():
    """One MXFP4 block worked by hand: amax = 9 -> t = 1.5 -> tie between
    2^0 and 2^1 -> even code 128 (scale 2); q = x / 2."""
    x = np.zeros((1, 32), dtype=np.float32)
    x[0, :6] = [9.0, -4.5, 1.0, 0.5, -2.5, 3.0]
    Q, SF = oracle.quantize(MX, x, 1.0)
    assert SF[0, 0] == 128
    nib = [Q[0, i // 2] >> (4 * (i % 2)) & 15 for i in range(6)]
    # q = 4.5 -> 4 (code 6); -2.25 -> -2 (12); 0.5 -> 0.5 (1); 0.25 -> tie -> 0;
    # -1.25 -> tie -> -1 (10); 1.5 -> 1.5 (3)
    assert nib == [6, 12, 1, 0, 10, 3]


def test_quantize_element_error_property():
    """Every element lands on the nearest grid point of x/s (or saturates),
    with s recomputed from the emitted scale byte."""
    for fmt in (MX, NV):
        xb = synth.activations_bf16(3 + fmt, 16, 256)
        x = synth.bf16_bits_to_f32(xb)
        gs = oracle.global_scale(xb) if fmt == NV else np.float32(1.0)
        Q, SF = oracle.quantize(fmt, xb, gs)
        g = oracle.block_size(fmt)
        codes = np.stack([Q & 15, Q >> 4], axis=-1).reshape(x.shape)
        for r in range(x.shape[0]):
            for k in range(x.shape[1]):
                s = np.float32(np.float32(oracle.scale_value(fmt, SF[r, k // g])) * np.float32(gs))
                q = np.float32(x[r, k]) / s
                v = abs(E2M1[int(codes[r, k])][0])
                if abs(q) >= 6.0:
                    assert v == 6.0
                else:
                    assert abs(abs(q) - v) <= np.min(np.abs(abs(q) - GRID)) + 0.0


def test_mxfp4_has_no_global_scale():
    """MXFP4 carries only its UE8M0 block scales (DeepGEMM PR, "Summary");
    a global scale handed to it is ignored by the quantiser, the dequantiser
    and the GEMM alike."""
    xb = synth.activations_bf16(17, 8, 256)
    Q1, SF1 = oracle.quantize(MX, xb, 1.0)
    Q2, SF2 = oracle.quantize(MX, xb, 0.37)
    assert np.array_equal(Q1, Q2) and np.array_equal(SF1, SF2)
    assert np.array_equal(oracle.dequantize(MX, Q1, SF1, 0.37), oracle.dequantize(MX, Q1, SF1, 1.0))
    Qw, SFw = oracle.quantize(MX, synth.weights_bf16(18, 4, 256))
    d1, t1 = oracle.gemm_nt(MX, Q1, SF1, Qw, SFw, 1.0, 1.0)
    d2, t2 = oracle.gemm_nt(MX, Q1, SF1, Qw, SFw, 0.37, 3.0)
    assert np.array_equal(d1, d2) and np.array_equal(t1, t2)
    mi, ni = np.array([0, 7, 3]), np.array([1, 0, 3])
    e1, _ = oracle.gemm_nt_entries(MX, Q1, SF1, Qw, SFw, 1.0, 1.0, mi, ni)
    e2, _ = oracle.gemm_nt_entries(MX, Q1, SF1, Qw, SFw, 0.37, 3.0, mi, ni)
    assert np.array_equal(e1, e2) and np.array_equal(e1, d1[mi, ni])


def test_global_scale_puts_largest_block_at_448():
    xb = synth.activations_bf16(5, 64, 512)
    gs = oracle.global_scale(xb)
    x = synth.bf16_bits_to_f32(xb)
    assert gs == np.float32(np.float32(np.abs(x).max()) / np.float32(2688.0))
    Q, SF = oracle.quantize(NV, xb, gs)
    assert SF.max() == 0x7E


def test_byte_accounting_matches_qgemm_page():
    (row,) = _golden_rows("byte_accounting.txt")
    printed = float(row[1])
    x = np.ones((4, 1024), dtype=np.float32)
    Q, SF = oracle.quantize(MX, x)
    bits_mx = 8.0 * (Q.nbytes + SF.nbytes) / x.size
    assert bits_mx == 4.25
    assert round(8.0 / bits_mx, 2) == printed
    Q, SF = oracle.quantize(NV, x)
    assert 8.0 * (Q.nbytes + SF.nbytes) / x.size == 4.5


# --------------------------------------------------------------------------
# GEMM
# --------------------------------------------------------------------------

def _pack(codes):
    codes = np.asarray(codes, dtype=np.uint8)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


@pytest.mark.parametrize("fmt", [MX, NV, NV32])
def test_gemm_all_ones_closed_form(fmt):
    g = oracle.block_size(fmt)
    M, N, K = 3, 5, 256
    A = _pack(np.full((M, K), 2))          # code 2 = 1.0
    B = _pack(np.full((N, K), 2))
    sa, sb = (125, 131) if fmt == MX else (0x30, 0x45)
    Asf = np.full((M, K // g), sa, dtype=np.uint8)
    Bsf = np.full((N, K // g), sb, dtype=np.uint8)
    gs_a, gs_b = (1.0, 1.0) if fmt == MX else (0.375, 2.5)
    D, T = oracle.gemm_nt(fmt, A, Asf, B, Bsf, gs_a, gs_b)
    dec = oracle.ue8m0_value if fmt == MX else oracle.ue4m3_value
    want = K * dec(sa) * dec(sb) * gs_a * gs_b
    assert np.all(D == want) and np.all(T == abs(want))


@pytest.mark.parametrize("fmt", [MX, NV, NV32])
def test_gemm_one_hot_pins_nibble_order(fmt):
    """A single non-zero element at (m0, k0): the k index <-> nibble mapping
    (even k low nibble) and the block index k0 // g are both exercised."""
    g = oracle.block_size(fmt)
    M, N, K = 4, 3, 128
    for k0 in (0, 1, 17, 46, 127):
        codes = np.zeros((M, K), dtype=np.uint8)
        codes[2, k0] = 7                               # 6.0
        A = _pack(codes)
        Asf = np.full((M, K // g), 127 if fmt == MX else 56, dtype=np.uint8)   # 1.0
        Asf[2, k0 // g] = 129 if fmt == MX else 64                             # 4.0 / 2.0
        bc = np.zeros((N, K), dtype=np.uint8)
        bc[:, k0] = [2, 11, 5]                          # 1, -1.5, 3
        B = _pack(bc)
        Bsf = np.full((N, K // g), 128 if fmt == MX else 64, dtype=np.uint8)  # 2.0
        D, _ = oracle.gemm_nt(fmt, A, Asf, B, Bsf, 1.0, 1.0)
        sa = 4.0 if fmt == MX else 2.0
        want = np.zeros((M, N))
        want[2] = np.array([1.0, -1.5, 3.0]) * 6.0 * sa * 2.0
        assert np.array_equal(D, want), k0


def _random_operands(fmt, M, N, K, seed):
    gen = synth.rng(seed)
    g = oracle.block_size(fmt)
    A = gen.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    B = gen.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    lo, hi = (118, 136) if fmt == MX else (1, 0x7F)
    Asf = gen.integers(lo, hi, size=(M, K // g), dtype=np.uint8)
    Bsf = gen.integers(lo, hi, size=(N, K // g), dtype=np.uint8)
    return A, Asf, B, Bsf


@pytest.mark.parametrize("fmt", [MX, NV, NV32])
def test_gemm_vs_numpy_matmul_of_independent_decode(fmt):
    """Decode with the golden table and torch's float8 decoders, multiply with
    numpy's matmul (fp64): must match the oracle to fp64 rounding."""
    M, N, K = 24, 40, 512
    A, Asf, B, Bsf = _random_operands(fmt, M, N, K, 31 + fmt)
    gs_a, gs_b = (1.0, 1.0) if fmt == MX else (np.float32(0.0123), np.float32(3.7))
    g = oracle.block_size(fmt)
    table = np.array([math.copysign(E2M1[c][0], -1.0 if c >= 8 else 1.0) for c in range(16)])
    sfdt = torch.float8_e8m0fnu if fmt == MX else torch.float8_e4m3fn

    def deq(Q, SF):
        codes = np.stack([Q & 15, Q >> 4], axis=-1).reshape(Q.shape[0], -1)
        sf = torch.from_numpy(SF.copy()).view(sfdt).to(torch.float64).numpy()
        return table[codes] * np.repeat(sf, g, axis=1)

    ref = (deq(A, Asf) @ deq(B, Bsf).T) * (float(gs_a) * float(gs_b))
    D, T = oracle.gemm_nt(fmt, A, Asf, B, Bsf, gs_a, gs_b)
    assert np.allclose(D, ref, rtol=1e-12, atol=1e-12 * np.abs(T).max())
    Tref = np.abs(deq(A, Asf)) @ np.abs(deq(B, Bsf)).T * abs(float(gs_a) * float(gs_b))
    assert np.allclose(T, Tref, rtol=1e-12)


@pytest.mark.parametrize("fmt", [MX, NV, NV32])
def test_gemm_tiny_exact_bruteforce(fmt):
    """2x3 outputs, K = 64, exact rational arithmetic in pure Python."""
    M, N, K = 2, 3, 64
    A, Asf, B, Bsf = _random_operands(fmt, M, N, K, 41 + fmt)
    g = oracle.block_size(fmt)
    gs_a, gs_b = (1.0, 1.0) if fmt == MX else (0.25, 8.0)

    def val(Q, SF, r, k):
        byte = int(Q[r, k // 2])
        code = (byte >> 4) if k % 2 else (byte & 15)
        mag = Fraction(E2M1[code][0]) if code < 8 else -Fraction(E2M1[code - 8][0])
        b = int(SF[r, k // g])
        if fmt == MX:
            s = Fraction(2) ** (b - 127)
        else:
            e, m = b >> 3, b & 7
            s = Fraction(m, 512) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
        return mag * s

    D, _ = oracle.gemm_nt(fmt, A, Asf, B, Bsf, gs_a, gs_b)
    for m in range(M):
        for n in range(N):
            exact = sum(val(A, Asf, m, k) * val(B, Bsf, n, k) for k in range(K))
            exact *= Fraction(gs_a) * Fraction(gs_b)
            assert Fraction(D[m, n]) == exact


def test_gemm_global_scale_identity():
    A, Asf, B, Bsf = _random_operands(NV, 8, 16, 256, 51)
    D1, T1 = oracle.gemm_nt(NV, A, Asf, B, Bsf, 1.0, 1.0)
    D2, T2 = oracle.gemm_nt(NV, A, Asf, B, Bsf, 2.0 ** 3, 2.0 ** -2)
    assert np.array_equal(D2, 2.0 * D1) and np.array_equal(T2, 2.0 * T1)


@pytest.mark.parametrize("fmt", [MX, NV])
def test_gemm_row_col_rescale_identity(fmt):
    """Two-level epilogue: D(rs, cs)[m,n] = rs[m] cs[n] D(1,1)[m,n], exact in
    fp64 for power-of-two scales (and T alike); NULL scales are ones; sampled
    entries agree with the full product."""
    A, Asf, B, Bsf = _random_operands(fmt, 12, 20, 256, 53 + fmt)
    gen = np.random.default_rng(9)
    rs = (2.0 ** gen.integers(-6, 7, 12)).astype(np.float32)
    cs = (2.0 ** gen.integers(-6, 7, 20)).astype(np.float32)
    D1, T1 = oracle.gemm_nt(fmt, A, Asf, B, Bsf, 0.5, 0.25)
    D2, T2 = oracle.gemm_nt(fmt, A, Asf, B, Bsf, 0.5, 0.25, rs, cs)
    outer = rs.astype(np.float64)[:, None] * cs.astype(np.float64)[None, :]
    assert np.array_equal(D2, outer * D1) and np.array_equal(T2, outer * T1)
    Dr, _ = oracle.gemm_nt(fmt, A, Asf, B, Bsf, 0.5, 0.25, rs, None)
    Dc, _ = oracle.gemm_nt(fmt, A, Asf, B, Bsf, 0.5, 0.25, None, cs)
    assert np.array_equal(Dr, rs.astype(np.float64)[:, None] * D1)
    assert np.array_equal(Dc, cs.astype(np.float64)[None, :] * D1)
    mi, ni = gen.integers(0, 12, 50), gen.integers(0, 20, 50)
    De, Te = oracle.gemm_nt_entries(fmt, A, Asf, B, Bsf, 0.5, 0.25, mi, ni, rs, cs)
    assert np.array_equal(De, D2[mi, ni]) and np.array_equal(Te, T2[mi, ni])


def test_per_row_global_scale_and_quantise_reduce_to_per_tensor():
    """Per-row global scales are the per-tensor rule on each row alone, and
    quantising with them equals quantising each row alone with its scale."""
    x = synth.activations_bf16(81, 7, 256)
    x[3] = 0                                     # an all-zero row: gs 0
    gs = oracle.global_scale_rows(x)
    for m in range(7):
        assert gs[m] == oracle.global_scale(x[m:m + 1])
    assert gs[3] == 0.0
    Q, SF = oracle.quantize(NV, x, gs)
    for m in range(7):
        q1, s1 = oracle.quantize(NV, x[m:m + 1], gs[m])
        assert np.array_equal(Q[m:m + 1], q1) and np.array_equal(SF[m:m + 1], s1)


def test_gemm_ue8m0_increment_doubles_one_block():
    """Scale byte + 1 on one block of one A row adds exactly that block's
    contribution once more (it doubles)."""
    A, Asf, B, Bsf = _random_operands(MX, 4, 6, 256, 61)
    D0, _ = oracle.gemm_nt(MX, A, Asf, B, Bsf)
    Asf1 = Asf.copy()
    Asf1[1, 3] += 1
    D1, _ = oracle.gemm_nt(MX, A, Asf1, B, Bsf)
    only = np.zeros_like(A)
    only[1, 3 * 16:4 * 16] = A[1, 3 * 16:4 * 16]        # block 3 = bytes 48..63
    Dblk, _ = oracle.gemm_nt(MX, only, Asf, B, Bsf)
    assert np.array_equal(D1 - D0, Dblk)
    assert np.array_equal(np.delete(D1, 1, axis=0), np.delete(D0, 1, axis=0))


@pytest.mark.parametrize("fmt,g", [(NV, 16), (NV32, 32)])
def test_ue4m3_scale_step_doubles_exactly_one_block(fmt, g):
    """One UE4M3 scale byte of one A row raised by one exponent step (0x38,
    1.0, to 0x40, 2.0) adds exactly the contribution of that row's g elements
    of the block once more: 16 for NVFP4, 32 for the per-32 format of the
    sparse path."""
    M, N, K = 3, 5, 256
    A, _, B, _ = _random_operands(fmt, M, N, K, 62 + fmt)
    assert oracle.block_size(fmt) == g
    Asf = np.full((M, K // g), 0x38, np.uint8)
    Bsf = np.full((N, K // g), 0x38, np.uint8)
    D0, _ = oracle.gemm_nt(fmt, A, Asf, B, Bsf, 0.5, 4.0)
    Asf1 = Asf.copy()
    Asf1[2, 3] = 0x40
    D1, _ = oracle.gemm_nt(fmt, A, Asf1, B, Bsf, 0.5, 4.0)
    only = np.zeros_like(A)
    only[2, 3 * g // 2:4 * g // 2] = A[2, 3 * g // 2:4 * g // 2]       # elements 3g .. 4g-1
    Dblk, _ = oracle.gemm_nt(fmt, only, Asf, B, Bsf, 0.5, 4.0)
    assert np.array_equal(D1 - D0, Dblk) and np.any(Dblk != 0)
    assert np.array_equal(np.delete(D1, 2, axis=0), np.delete(D0, 2, axis=0))


def test_gemm_entries_equal_full():
    A, Asf, B, Bsf = _random_operands(NV, 32, 48, 256, 71)
    D, T = oracle.gemm_nt(NV, A, Asf, B, Bsf, 0.5, 0.125)

    mi = np.array([0, 5, 31, 17])
    ni = np.array([47, 0, 3, 22])
    d, t = oracle.gemm_nt_entries(NV, A, Asf, B, Bsf, 0.5, 0.125, mi, ni)
    assert np.array_equal(d, D[mi, ni]) and np.array_equal(t, T[mi, ni])


# --------------------------------------------------------------------------
# scale-factor interleave
# --------------------------------------------------------------------------

@pytest.mark.parametrize("rows,cols", [(128, 4), (256, 16), (300, 7), (1, 1), (129, 5)])
def test_sf_interleave_vs_numpy_reshape(rows, cols):
    """The 5D layout [rows/128][cols/4][32][4][4] built with numpy reshapes."""
    gen = synth.rng(rows * 100 + cols)
    sf = gen.integers(1, 255, size=(rows, cols), dtype=np.uint8)
    R, C = -(-rows // 128) * 128, -(-cols // 4) * 4
    pad = np.zeros((R, C), dtype=np.uint8)
    pad[:rows, :cols] = sf
    # row r = rt*128 + j*32 + i, col c = ct*4 + kk  ->  [rt][ct][i][j][kk]
    want = pad.reshape(R // 128, 4, 32, C // 4, 4).transpose(0, 3, 2, 1, 4).reshape(-1)
    got = oracle.sf_to_mma(sf)
    assert got.size == oracle.sf_mma_bytes(rows, cols) == want.size
    assert np.array_equal(got, want)
    assert np.array_equal(oracle.sf_from_mma(got, rows, cols), sf)


# --------------------------------------------------------------------------
# SwiGLU of the up-projection, and the validity check of its requantisation
# --------------------------------------------------------------------------

def test_swiglu_closed_forms():
    """silu(x) = x * sigmoid(x): its limits, one value worked from e, the
    identity silu(x) - silu(-x) = x, and exact linearity in the up operand."""
    U = np.array([3.0, -2.5, 0.75, 1e3])
    assert np.all(oracle.swiglu(np.zeros(4), U) == 0.0)                    # silu(0) = 0
    G = np.array([40.0, 100.0, 1e4, 3.5e38])
    assert np.array_equal(oracle.swiglu(G, U), G * U)                    # sigmoid -> 1
    assert np.all(oracle.swiglu(np.array([-746.0, -1e4, -3e38, -800.0]), U) == 0.0)   # -> 0
    e = math.e
    assert oracle.swiglu(np.array([1.0]), np.array([2.0]))[0] == pytest.approx(2 * e / (e + 1), rel=1e-15)
    assert oracle.swiglu(np.array([-1.0]), np.array([1.0]))[0] == pytest.approx(-1 / (e + 1), rel=1e-15)
    x = synth.rng(401).normal(0, 4, 1000)
    odd = oracle.swiglu(x, np.ones_like(x)) - oracle.swiglu(-x, np.ones_like(x))
    assert np.allclose(odd, x, rtol=1e-15, atol=1e-300)
    u = synth.rng(402).normal(0, 1, 1000)
    assert np.array_equal(oracle.swiglu(x, 2.0 * u), 2.0 * oracle.swiglu(x, u))


def test_swiglu_up_gate_and_up_roles():
    """G comes from the gate rows and U from the up rows: doubling the up
    weights (one UE8M0 step on every scale byte) doubles H exactly, doubling
    the gate weights does not; zero gate weights give H = 0."""
    A, Asf, Wg, Wgsf = _random_operands(MX, 6, 8, 256, 403)
    _, _, Wu, Wusf = _random_operands(MX, 6, 8, 256, 404)
    H, G, U, TG, TU = oracle.swiglu_up(MX, A, Asf, Wg, Wgsf, Wu, Wusf)
    assert np.array_equal(G, oracle.gemm_nt(MX, A, Asf, Wg, Wgsf)[0])
    assert np.array_equal(U, oracle.gemm_nt(MX, A, Asf, Wu, Wusf)[0])
    H2u = oracle.swiglu_up(MX, A, Asf, Wg, Wgsf, Wu, Wusf + 1)[0]
    assert np.array_equal(H2u, 2.0 * H)
    H2g = oracle.swiglu_up(MX, A, Asf, Wg, Wgsf + 1, Wu, Wusf)[0]
    assert not np.allclose(H2g, 2.0 * H)
    H0 = oracle.swiglu_up(MX, A, Asf, np.zeros_like(Wg), Wgsf, Wu, Wusf)[0]
    assert np.all(H0 == 0.0)
    # NVFP4: the global scales multiply G and U before the nonlinearity
    A, Asf, Wg, Wgsf = _random_operands(NV, 4, 16, 256, 405)
    _, _, Wu, Wusf = _random_operands(NV, 4, 16, 256, 406)
    Hs, Gs, Us, _, _ = oracle.swiglu_up(NV, A, Asf, Wg, Wgsf, Wu, Wusf, 0.5, 0.25)
    H1, G1, U1, _, _ = oracle.swiglu_up(NV, A, Asf, Wg, Wgsf, Wu, Wusf)
    assert np.array_equal(Gs, G1 * 0.125) and np.array_equal(Us, U1 * 0.125)
    assert np.array_equal(Hs, oracle.swiglu(G1 * 0.125, U1 * 0.125))


def _requant_case(fmt, M, I, seed):
    gen = synth.rng(seed)
    H = gen.normal(0, 1, (M, I)) * np.exp(gen.normal(0, 1, (M, 1)))
    gs2 = np.float32(np.abs(H).max() / 2688.0) if fmt == NV else np.float32(1.0)
    return H, gs2


@pytest.mark.parametrize("fmt", [MX, NV])
def test_requant_valid_is_exact_at_zero_width(fmt):
    """With delta = 0 and H already fp32, exactly the rule's own output
    passes: any other scale byte or any other element code fails."""
    H, gs2 = _requant_case(fmt, 8, 256, 407 + fmt)
    H = H.astype(np.float32).astype(np.float64)
    Q, SF = oracle.swiglu_requantize(fmt, H, gs2)
    z = np.zeros_like(H)
    assert oracle.requant_valid(fmt, Q, SF, H, z, gs2).all()
    g = oracle.block_size(fmt)
    gen = synth.rng(409)
    for _ in range(40):
        r, j = int(gen.integers(0, 8)), int(gen.integers(0, 256 // g))
        SF2 = SF.copy()
        SF2[r, j] = (int(SF[r, j]) + (1 if gen.integers(0, 2) else -1)) % 256
        ok = oracle.requant_valid(fmt, Q, SF2, H, z, gs2)
        assert not ok[r, j] and ok.sum() == ok.size - 1
        k = int(gen.integers(0, 256))
        Q2 = Q.copy()
        Q2[r, k // 2] ^= np.uint8((1 + int(gen.integers(0, 15))) << (4 * (k % 2)))
        ok = oracle.requant_valid(fmt, Q2, SF, H, z, gs2)
        assert not ok[r, k // g] and ok.sum() == ok.size - 1


@pytest.mark.parametrize("fmt", [MX, NV])
def test_requant_valid_accepts_every_input_in_the_box(fmt):
    """Whatever fp32 matrix inside [H - delta, H + delta] the rule is given,
    its output passes (random points, and both corners of the box)."""
    H, gs2 = _requant_case(fmt, 16, 512, 410 + fmt)
    delta = 2e-3 * np.abs(H) + 1e-4 * np.abs(H).max()
    gen = synth.rng(412 + fmt)
    points = [H - delta, H + delta] + [H + delta * gen.uniform(-1, 1, H.shape) for _ in range(12)]
    for h in points:
        h32 = np.clip(h.astype(np.float32), oracle._f32_down(H - delta), oracle._f32_up(H + delta))
        Q, SF = oracle.quantize(fmt, h32, gs2)
        assert oracle.requant_valid(fmt, Q, SF, H, delta, gs2).all()


def test_requant_valid_tie_and_zero_scale():
    """A value on an E2M1 tie takes either neighbour once delta > 0, but not
    a code two steps away; an all-zero NVFP4 block takes scale 0 and +0 codes
    only."""
    H = np.zeros((1, 16))
    H[0, 0] = 6.0                 # amax 6 with gs 1: scale 1.0, so x / s = x
    H[0, 1] = 0.25                # tie between codes 0 (0) and 1 (0.5)
    Q, SF = oracle.swiglu_requantize(NV, H, 1.0)
    assert SF[0, 0] == 0x38 and (Q[0, 0] >> 4) == 0
    delta = np.full_like(H, 1e-6)
    assert oracle.requant_valid(NV, Q, SF, H, delta, 1.0).all()
    Q1 = Q.copy()
    Q1[0, 0] = (Q[0, 0] & 15) | (1 << 4)                                   # 0.5
    assert oracle.requant_valid(NV, Q1, SF, H, delta, 1.0).all()
    assert not oracle.requant_valid(NV, Q1, SF, H, np.zeros_like(H), 1.0).any()
    Q2 = Q.copy()
    Q2[0, 0] = (Q[0, 0] & 15) | (2 << 4)                                   # 1.0
    assert not oracle.requant_valid(NV, Q2, SF, H, delta, 1.0).any()
    Z = np.zeros((1, 16))
    Qz, SFz = oracle.swiglu_requantize(NV, Z, 1.0)
    assert SFz[0, 0] == 0 and Qz.max() == 0
    assert oracle.requant_valid(NV, Qz, SFz, Z, np.zeros_like(Z), 1.0).all()
    Qn = Qz.copy()
    Qn[0, 3] = 8                                                          # -0
    assert not oracle.requant_valid(NV, Qn, SFz, Z, np.zeros_like(Z), 1.0).any()


# --------------------------------------------------------------------------
# residual add and RMSNorm in front of the quantiser
# --------------------------------------------------------------------------

def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(torch.bfloat16)


def _bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


def test_residual_add_rounds_like_torch_bf16():
    """y = bf16(x + r): torch's float -> bfloat16 conversion (nearest even)
    of the fp32 sum, on random values and on sums placed exactly halfway
    between two bf16 values."""
    gen = synth.rng(501)
    x = synth.f32_to_bf16_bits(gen.normal(0, 1, (64, 128)).astype(np.float32))
    r = synth.f32_to_bf16_bits(gen.normal(0, 3, (64, 128)).astype(np.float32))
    # ties: x = 1 + 2^-7 (bf16), r = 2^-8 -> x + r sits between two bf16 values
    x[0, :4] = synth.f32_to_bf16_bits(np.array([1 + 2 ** -7, 1.0, 1 + 2 ** -6, 3.0], np.float32))
    r[0, :4] = synth.f32_to_bf16_bits(np.array([2 ** -8, 2 ** -8, 2 ** -8, 2 ** -7 * 3 / 2], np.float32))
    y, _, _ = oracle.residual_rmsnorm(x, r, np.full(128, 0x3F80, np.uint16))
    want = _bits((_bf16(x).float() + _bf16(r).float()).to(torch.bfloat16))
    assert np.array_equal(y, want)
    y0, _, _ = oracle.residual_rmsnorm(x, None, np.full(128, 0x3F80, np.uint16))
    assert np.array_equal(y0, x)


def test_rmsnorm_closed_forms():
    """Rows worked by hand: [3, 4] has mean square 12.5, so z = [3, 4] * sqrt(2)
    / 5; a constant row c = 0.5 with eps = 0.25 gives sqrt(0.5); with eps = 0
    every row has mean square 1 after the norm; gamma scales z linearly and
    doubling the input leaves z unchanged."""
    one = np.full(2, 0x3F80, np.uint16)
    x = synth.f32_to_bf16_bits(np.array([[3.0, 4.0]], np.float32))
    _, z, inv = oracle.residual_rmsnorm(x, None, one, 0.0)
    assert z[0] == pytest.approx(np.array([3.0, 4.0]) * math.sqrt(2) / 5, rel=1e-15)
    c = synth.f32_to_bf16_bits(np.full((1, 16), 0.5, np.float32))
    _, z, _ = oracle.residual_rmsnorm(c, None, np.full(16, 0x3F80, np.uint16), 0.25)
    assert np.allclose(z, math.sqrt(0.5), rtol=1e-15, atol=0)
    xb = synth.activations_bf16(502, 8, 256)
    ones = np.full(256, 0x3F80, np.uint16)
    _, z, _ = oracle.residual_rmsnorm(xb, None, ones, 0.0)
    assert np.allclose((z ** 2).mean(axis=1), 1.0, rtol=1e-13)
    x2 = synth.f32_to_bf16_bits(2.0 * synth.bf16_bits_to_f32(xb))
    _, z2, _ = oracle.residual_rmsnorm(x2, None, ones, 0.0)
    assert np.array_equal(z2, z)
    twos = np.full(256, 0x4000, np.uint16)
    _, zg, _ = oracle.residual_rmsnorm(xb, None, twos, 0.0)
    assert np.array_equal(zg, 2.0 * z)
    # the residual enters before the norm: x + r with r = x is x doubled
    _, zr, _ = oracle.residual_rmsnorm(xb, xb, ones, 0.0)
    assert np.array_equal(zr, z)
    _, zr1, _ = oracle.residual_rmsnorm(xb, xb, ones, 1.0)
    _, z1, _ = oracle.residual_rmsnorm(xb, None, ones, 1.0)
    assert not np.allclose(zr1, z1)             # eps does not scale with the input


def test_rows_global_scale_exact_matches_the_bf16_rule():
    xb = synth.activations_bf16(503, 16, 512)
    got = oracle.rows_global_scale_exact(synth.bf16_bits_to_f32(xb).astype(np.float64))
    want = oracle.global_scale_rows(xb)
    assert np.all(np.abs(got - want) <= np.spacing(want.astype(np.float32)))


@pytest.mark.parametrize("fmt", [MX, NV])
def test_requant_valid_per_row_scales_and_intervals(fmt):
    """Per-row global scales check each row with its own scale; with an
    interval [lo, hi] the rule's output for any scale inside it passes, and
    an output made with a scale outside a point interval can fail."""
    H, _ = _requant_case(fmt, 12, 256, 504 + fmt)
    gen = synth.rng(506 + fmt)
    gs = np.float32(np.abs(H).max(axis=1) / 2688.0)
    z = np.zeros_like(H)
    H32 = H.astype(np.float32).astype(np.float64)
    Q = np.zeros((12, 128), np.uint8)
    SF = np.zeros((12, 256 // oracle.block_size(fmt)), np.uint8)
    for m in range(12):
        Q[m:m + 1], SF[m:m + 1] = oracle.quantize(fmt, H32[m:m + 1].astype(np.float32), gs[m])
    assert oracle.requant_valid(fmt, Q, SF, H32, z, gs).all()
    for m in (0, 5, 11):
        ok_m = oracle.requant_valid(fmt, Q[m:m + 1], SF[m:m + 1], H32[m:m + 1], z[m:m + 1], gs[m])
        assert ok_m.all()
    if fmt == MX:
        return
    lo = (gs * np.float32(0.97)).astype(np.float32)
    hi = (gs * np.float32(1.05)).astype(np.float32)
    for _ in range(6):
        gsx = np.where(gen.uniform(size=12) < 0.5, lo, hi) if _ < 2 else \
            (lo + (hi - lo) * gen.uniform(size=12).astype(np.float32)).astype(np.float32)
        Qx = np.zeros_like(Q)
        SFx = np.zeros_like(SF)
        for m in range(12):
            Qx[m:m + 1], SFx[m:m + 1] = oracle.quantize(NV, H32[m:m + 1].astype(np.float32), gsx[m])
        assert oracle.requant_valid(NV, Qx, SFx, H32, z, lo, hi).all()
    Qh = np.zeros_like(Q)
    SFh = np.zeros_like(SF)
    for m in range(12):
        Qh[m:m + 1], SFh[m:m + 1] = oracle.quantize(NV, H32[m:m + 1].astype(np.float32), hi[m])
    assert not oracle.requant_valid(NV, Qh, SFh, H32, z, gs).all()


# --------------------------------------------------------------------------
# 2:4 pair-granular sparse operand
# --------------------------------------------------------------------------

def test_sparse24_hand_worked_groups():
    """Two groups worked by hand: [00 21 00 43] keeps pairs 1 and 3 (nibble
    1 | 3 << 2 = 0xD); [10 00 00 00] keeps pair 0 and the lowest zero pair 1
    (nibble 4); the even group sits in the low nibble of the metadata byte."""
    W = np.array([[0x00, 0x21, 0x00, 0x43, 0x10, 0x00, 0x00, 0x00]], np.uint8)
    Wc, meta = oracle.sparse24_compress(W)
    assert Wc.tolist() == [[0x21, 0x43, 0x10, 0x00]]
    assert meta.tolist() == [[0xD | (0x4 << 4)]]
    assert np.array_equal(oracle.sparse24_decompress(Wc, meta, 16), W)
    # -0 codes count as zero pairs: 0x88 and 0x08 do not take a slot
    W2 = np.array([[0x88, 0x31, 0x08, 0x75, 0, 0, 0, 0]], np.uint8)
    Wc2, meta2 = oracle.sparse24_compress(W2)
    assert Wc2[0, :2].tolist() == [0x31, 0x75] and (meta2[0, 0] & 15) == (1 | 3 << 2)
    with pytest.raises(ValueError):
        oracle.sparse24_compress(np.array([[0x11, 0x22, 0x33, 0, 0, 0, 0, 0]], np.uint8))
    with pytest.raises(ValueError):                          # i0 >= i1 is not a valid group
        oracle.sparse24_decompress(np.zeros((1, 4), np.uint8), np.array([[0x3 | (0x1 << 2)]], np.uint8), 16)


def _random_sparse24(rows, K, seed):
    """Random 2:4 operand: in every group of four bytes, two random pair
    positions hold bytes whose elements are both non-zero."""
    gen = synth.rng(seed)
    W = np.zeros((rows, K // 2), np.uint8)
    nz = lambda size: gen.integers(1, 8, size) | (gen.integers(0, 2, size) << 3)   # non-zero E2M1 codes
    for r in range(rows):
        for j in range(K // 8):
            i = gen.choice(4, 2, replace=False)
            W[r, 4 * j + i] = (nz(2) | (nz(2) << 4)).astype(np.uint8)
    return W


def test_sparse24_round_trips():
    W = _random_sparse24(16, 256, 511)
    Wc, meta = oracle.sparse24_compress(W)
    assert np.array_equal(oracle.sparse24_decompress(Wc, meta, 256), W)
    gen = synth.rng(512)
    pairs = np.array([(a, b) for a in range(4) for b in range(a + 1, 4)])
    sel = pairs[gen.integers(0, 6, (16, 32))]
    nibs = (sel[..., 0] | (sel[..., 1] << 2)).astype(np.uint8)
    meta2 = (nibs[:, 0::2] | (nibs[:, 1::2] << 4)).astype(np.uint8)
    Wc2 = _random_sparse24(16, 128, 513)[:, :64]                            # bytes with non-zero elements
    Wc2 = np.where(Wc2 == 0, np.uint8(0x11), Wc2)
    W2 = oracle.sparse24_decompress(Wc2, meta2, 256)
    Wc3, meta3 = oracle.sparse24_compress(W2)
    assert np.array_equal(Wc3, Wc2) and np.array_equal(meta3, meta2)


@pytest.mark.parametrize("fmt", [MX, NV, NV32])
def test_sparse24_gemm_keeps_exactly_the_selected_positions(fmt):
    """All kept elements 1.0 (code 2) with unit scales: D[m, n] is the sum of
    a[m, k] over the positions k that row n keeps, found here from the
    metadata by hand-written indexing."""
    g = oracle.block_size(fmt)
    M, N, K = 5, 6, 128
    W = _random_sparse24(N, K, 514 + fmt)
    W = np.where(W != 0, np.uint8(0x22), W)                   # both elements 1.0
    Wc, meta = oracle.sparse24_compress(W)
    one = 127 if fmt == MX else 0x38
    Wsf = np.full((N, K // g), one, np.uint8)
    A, Asf, _, _ = _random_operands(fmt, M, 1, K, 515 + fmt)
    D, _ = oracle.gemm_nt_sparse24(fmt, A, Asf, Wc, meta, Wsf)
    a = oracle.dequantize(fmt, A, Asf)
    want = np.zeros((M, N))
    for n in range(N):
        for j in range(K // 8):
            nib = (meta[n, j // 2] >> (4 * (j % 2))) & 15
            for p in (nib & 3, nib >> 2):
                want[:, n] += a[:, 8 * j + 2 * p] + a[:, 8 * j + 2 * p + 1]
    assert np.allclose(D, want, rtol=1e-15, atol=0)


def test_requant_valid_box_across_zero():
    """When every element's range spans zero, an all-zero input lies in the
    box, so the all-zero output (scale byte 0, +0 codes) must pass."""
    for fmt in (MX, NV):
        H = np.full((1, 32), 1e-3) * synth.rng(520 + fmt).choice([-1.0, 1.0], (1, 32))
        delta = np.full_like(H, 2e-3)
        g = oracle.block_size(fmt)
        Q0 = np.zeros((1, 16), np.uint8)
        SF0 = np.zeros((1, 32 // g), np.uint8)
        assert oracle.requant_valid(fmt, Q0, SF0, H, delta, 1.0).all()
        Qr, SFr = oracle.quantize(fmt, H.astype(np.float32), 1.0)
        assert oracle.requant_valid(fmt, Qr, SFr, H, delta, 1.0).all()


def test_requant_valid_underflowing_scale():
    """A non-zero NVFP4 block far below the global scale takes scale byte 0,
    which decodes to 0, so the rule writes +0 for every element, negative
    ones included: that output passes, and -0 codes for the negative
    elements do not."""
    H = np.array([[3e-12, -2e-12, 1e-12, -4e-12] * 4])
    Q, SF = oracle.swiglu_requantize(NV, H, 1.0)
    assert SF.tolist() == [[0]] and Q.max() == 0
    z = np.zeros_like(H)
    assert oracle.requant_valid(NV, Q, SF, H, z, 1.0).all()
    neg = np.stack([Q & 15, Q >> 4], axis=-1).reshape(1, 16)
    neg[H < 0] = 8
    Qn = (neg[:, 0::2] | (neg[:, 1::2] << 4)).astype(np.uint8)
    assert not oracle.requant_valid(NV, Qn, SF, H, z, 1.0).any()


def test_bit_range_codes_follow_the_quantiser_steps():
    """The bit-range forms behind the exhaustive GPU check of the encoders:
    element codes equal E2M1 rounding of numpy's IEEE fp32 quotient x / s,
    and scale codes equal the scale byte the whole quantiser gives a block
    whose largest magnitude is that value."""
    starts = (0x00000000, 0x3E7FFF00, 0x3F7FFF80, 0x40A00000 - 64, 0x7F7FFF00,
              0x80000000, 0xBF400000 - 100, 0xC0C00000 - 200)
    n = 256
    for first in starts:
        bits = np.arange(first, first + n, dtype=np.uint64).astype(np.uint32)
        x = bits.view(np.float32)
        for s in (np.float32(1.0), np.float32(3.0), np.float32(0.37), np.float32(2.0 ** -100)):
            with np.errstate(over="ignore"):
                q = x / s
            assert np.array_equal(oracle.element_codes_bits(first, n, s), oracle.e2m1_round_array(q)), (hex(first), s)
        if first >= 0x80000000:
            continue
        for fmt, gs in ((NV, np.float32(1.0)), (NV, np.float32(0.0137)), (NV, np.float32(1e-30)), (MX, np.float32(1.0))):
            g = oracle.block_size(fmt)
            blocks = np.zeros((n, g), np.float32)
            blocks[:, 3] = x
            _, sf = oracle.quantize(fmt, blocks, gs)
            assert np.array_equal(oracle.scale_codes_bits(fmt, first, n, gs), sf[:, 0]), (hex(first), fmt, gs)
