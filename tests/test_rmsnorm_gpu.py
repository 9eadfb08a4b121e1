"""GPU parity of the residual-add + RMSNorm quantiser
(qfp4_residual_rmsnorm_quantize) against the oracle.

y = bf16(x + r) must be bit-exact.  z comes out of an fp32 sum of squares, a
square root and two products, so it is known only to within a relative
error the header states, eps_z = ((L + 2)/2 + 4) * 2^-24 with L = EPT + 10 the
longest chain of additions in the kernel's sum (first-order error analysis
of a sum of positive terms, one division by K, one addition of eps, a square
root, a reciprocal and two products, each correctly rounded).  So:
  - the row's global scale (NVFP4) must lie in amax(z)(1 +- eps_z) / 2688,
    widened by the rounding of that division;
  - every block must be what the quantiser's rule gives for some fp32 input
    within eps_z |z| of the exact z, with the kernel's own row scale
    (oracle.requant_valid);
  - and, as a sanity bound, at least 99% of the blocks must equal the rule
    applied to the exact z rounded to fp32 with that row scale."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_tcgen05_gb300 import qfp4, synth
from tests._helpers import MX, NV, to_dev_bf16, to_host

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    qfp4.load()
    assert qfp4.device_check() == 0


def ept_for(fmt, K):
    e = qfp4.block_size(fmt)
    while K // e > 1024:
        e *= 2
    return e


def eps_z(fmt, K):
    L = ept_for(fmt, K) + 10
    return ((L + 2) / 2 + 4) * U * 1.01


def run(fmt, M, K, with_r, layout, seed, eps=1e-6):
    g = qfp4.block_size(fmt)
    x = synth.activations_bf16(seed, M, K)
    r = synth.activations_bf16(seed + 1, M, K) if with_r else None
    gamma = synth.norm_weight_bf16(seed + 2, K)
    X = to_dev_bf16(x)
    R = to_dev_bf16(r) if with_r else None
    Gm = to_dev_bf16(gamma)
    Y = torch.full((M, K), 7.0, dtype=torch.bfloat16, device="cuda") if with_r else None
    gs = torch.full((M,), -1.0, dtype=torch.float32, device="cuda")
    Q = torch.full((M, K // 2), 0x5A, dtype=torch.uint8, device="cuda")
    sf_bytes = qfp4.sf_mma_bytes(M, K // g) if layout == qfp4.SF_MMA else M * (K // g)
    SF = torch.full((sf_bytes,), 0xA5, dtype=torch.uint8, device="cuda")
    qfp4.residual_rmsnorm_quantize(fmt, X, R, Gm, eps, Y, gs if fmt == NV else None, Q, SF, layout)
    torch.cuda.synchronize()
    assert qfp4.poll_device_status() == 0
    return x, r, gamma, Y, gs, Q, SF


def gs_interval(z, e):
    """The interval the kernel's row global scale must lie in, from the exact
    z alone: amax(z)(1 +- eps_z) / 2688, widened outward by the rounding of
    the division (fp32 bounds)."""
    amax = np.abs(z).max(axis=1)
    lo = (amax * (1 - e) / 2688.0 * (1 - 2 * U)).astype(np.float32)
    hi = (amax * (1 + e) / 2688.0 * (1 + 2 * U)).astype(np.float32)
    return amax, lo, hi


def check_rows(fmt, K, q_h, sf, gs_k, z, what):
    """Kernel codes, scale bytes and (NVFP4) row scales of rows with exact
    output z, checked against what the oracle alone fixes."""
    M = z.shape[0]
    g = qfp4.block_size(fmt)
    e = eps_z(fmt, K)
    amax, lo, hi = gs_interval(z, e)
    live = amax > 0
    # a row whose z is all zero: global scale 0, every scale byte 0, every code +0
    assert not q_h[~live].any() and not sf[~live].any(), f"{what}: zero rows"
    if fmt == NV:
        assert np.all(gs_k[~live] == 0), f"{what}: zero rows' global scale"
        assert np.all((gs_k[live] >= lo[live]) & (gs_k[live] <= hi[live])), f"{what}: row scale outside its bound"
    ok = oracle.requant_valid(fmt, q_h[live], sf[live], z[live], e * np.abs(z[live]),
                              lo[live] if fmt == NV else 1.0, hi[live] if fmt == NV else None)
    if not ok.all():
        bad = np.argwhere(~ok)[:6].tolist()
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} blocks invalid, first {bad}")
    # sanity bound: the rule on the exact z (fp32) with the exact row scale
    z32 = z.astype(np.float32)
    gs_ref = (amax / 2688.0).astype(np.float32)
    same = 0
    for m in np.flatnonzero(live):
        q_ref, sf_ref = oracle.quantize(fmt, z32[m:m + 1], gs_ref[m] if fmt == NV else 1.0)
        codes_ok = (q_h[m] == q_ref[0]).reshape(K // g, g // 2).all(axis=-1)
        same += int(((sf[m] == sf_ref[0]) & codes_ok).sum())
    frac = same / max(1, int(live.sum()) * (K // g))
    assert frac >= 0.99, f"{what}: only {frac:.4f} of the blocks equal the rule on the exact z"
    return frac


def check(fmt, M, K, x, r, gamma, Y, gs, Q, SF, layout, eps=1e-6, what=""):
    g = qfp4.block_size(fmt)
    y_ref, z, _ = oracle.residual_rmsnorm(x, r, gamma, eps)
    if Y is not None:
        assert np.array_equal(to_host(Y.view(torch.int16)).view(np.uint16), y_ref), f"{what}: y not bit-exact"
    sf_h = to_host(SF)
    if layout == qfp4.SF_MMA:
        sf = oracle.sf_from_mma(sf_h, M, K // g)
        assert np.array_equal(sf_h, oracle.sf_to_mma(sf)), f"{what}: scale layout or its zero padding"
    else:
        sf = sf_h.reshape(M, K // g)
    return check_rows(fmt, K, to_host(Q), sf, to_host(gs).astype(np.float32) if fmt == NV else None, z, what)


@pytest.mark.parametrize("fmt", [MX, NV])
@pytest.mark.parametrize("M,K,with_r,layout", [(1, 128, True, qfp4.SF_MMA), (77, 4096, True, qfp4.SF_MMA),
                                               (129, 1024, True, qfp4.SF_ROWMAJOR), (64, 4096, False, qfp4.SF_MMA),
                                               (300, 14336, True, qfp4.SF_MMA), (40, 2560, True, qfp4.SF_ROWMAJOR),
                                               (33, 40960, True, qfp4.SF_MMA)])
def test_residual_rmsnorm_quantize_vs_oracle(fmt, M, K, with_r, layout):
    """Ragged row counts (MMA-layout padding), K from one 128-element tile to
    40960 (two to four scale blocks per thread), with and without the
    residual input."""
    x, r, gamma, Y, gs, Q, SF = run(fmt, M, K, with_r, layout, 9100 + M + K + fmt)
    check(fmt, M, K, x, r, gamma, Y, gs, Q, SF, layout, what=f"{M}x{K}")


def test_residual_rmsnorm_full_size_sampled_rows():
    """X[16384, 4096] with a residual (the quantiser's full-size workload),
    NVFP4 into the MMA layout, checked on 64 sampled whole rows."""
    fmt, M, K = NV, 16384, 4096
    x, r, gamma, Y, gs, Q, SF = run(fmt, M, K, True, qfp4.SF_MMA, 9500)
    rows = np.unique(np.concatenate([[0, 127, 128, M - 1], synth.rng(9501).choice(M, 60, replace=False)]))
    sf_all = oracle.sf_from_mma(to_host(SF), M, K // 16)
    y_ref, z, _ = oracle.residual_rmsnorm(x[rows], r[rows], gamma)
    assert np.array_equal(to_host(Y.view(torch.int16)).view(np.uint16)[rows], y_ref)
    check_rows(fmt, K, to_host(Q)[rows], sf_all[rows], to_host(gs)[rows], z, "16384x4096")


def test_residual_rmsnorm_special_rows():
    """An all-zero row (z = 0: global scale 0, every scale byte 0, every code
    +0), a row that is zero after the residual cancels it, and a large eps."""
    fmt, M, K = NV, 4, 512
    x = synth.activations_bf16(9600, M, K)
    r = x.copy()
    r[1] ^= 0x8000                               # row 1: x + (-x) = 0
    x[2] = 0
    r[2] = 0                                     # row 2: both zero
    gamma = synth.norm_weight_bf16(9601, K)
    for eps in (1e-6, 10.0):
        X, R, Gm = to_dev_bf16(x), to_dev_bf16(r), to_dev_bf16(gamma)
        Y = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
        gs = torch.empty(M, dtype=torch.float32, device="cuda")
        Q = torch.empty((M, K // 2), dtype=torch.uint8, device="cuda")
        SF = torch.empty((M * (K // 16),), dtype=torch.uint8, device="cuda")
        qfp4.residual_rmsnorm_quantize(fmt, X, R, Gm, eps, Y, gs, Q, SF, qfp4.SF_ROWMAJOR)
        torch.cuda.synchronize()
        assert qfp4.poll_device_status() == 0
        gs_h, q_h, sf_h = to_host(gs), to_host(Q), to_host(SF).reshape(M, K // 16)
        for m in (1, 2):
            assert gs_h[m] == 0.0 and not q_h[m].any() and not sf_h[m].any()
        check(fmt, M, K, x, r, gamma, Y, gs, Q, SF, qfp4.SF_ROWMAJOR, eps=eps, what=f"eps={eps}")
