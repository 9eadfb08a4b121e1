"""Every finite fp32 value through the device encoders of the fp32 quantisers
(the residual-add + RMSNorm quantiser and the SwiGLU epilogue use
block_scale and encode8_f32), against the oracle: as a block maximum (the
scale byte, under several global scales) and as an element (the E2M1 code,
under several block scales, both quotient paths).  The test build's probes
run the device functions over ranges of bit patterns; the oracle applies the
quantiser's steps to the same patterns.  Bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from block_scaled_fp4_tcgen05_gb300 import qfp4
from tests._helpers import MX, NV

pytestmark = pytest.mark.gpu

CHUNK = 1 << 27
POSITIVE = (0x00000000, 0x7F800000)          # +0 .. the largest finite value
NEGATIVE = (0x80000000, 0xFF800000)          # -0 .. the most negative finite value


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    return qfp4.load_fault_injection()


@pytest.fixture(scope="module")
def buf(lib):
    return torch.empty(CHUNK, dtype=torch.uint8, device="cuda")


def sweep(probe, fmt, param, ranges, reference, buf):
    checked = 0
    for lo, hi in ranges:
        for first in range(lo, hi, CHUNK):
            n = min(CHUNK, hi - first)
            assert probe(fmt, first, n, float(param), buf.data_ptr(), None) == 0
            torch.cuda.synchronize()
            got = buf[:n].cpu().numpy()
            want = reference(first, n)
            if not np.array_equal(got, want):
                bad = np.flatnonzero(got != want)[:5]
                raise AssertionError(
                    f"{len(np.flatnonzero(got != want))} codes differ in [{first:#010x}, +{n}); first: "
                    + ", ".join(f"bits {first + int(i):#010x} device {got[i]} oracle {want[i]}" for i in bad))
            checked += n
    return checked


@pytest.mark.parametrize("fmt,gs", [(NV, np.float32(1.0)), (NV, np.float32(0.0137)), (NV, np.float32(1e-30)),
                                    (MX, np.float32(1.0))])
def test_scale_byte_of_every_fp32_block_maximum(lib, buf, fmt, gs):
    """The scale byte for every finite amax >= 0: NVFP4 with a unit global
    scale, a typical one (amax / 2688 of an activation tensor) and one small
    enough that t = (amax / 6) / gs leaves the fast-division range; MXFP4."""
    n = sweep(lib.qfp4_test_scale_codes, fmt, gs, [POSITIVE],
              lambda first, n: oracle.scale_codes_bits(fmt, first, n, gs), buf)
    assert n == 0x7F800000


@pytest.mark.parametrize("fmt,param", [(NV, np.float32(1.0)), (NV, np.float32(1.6576)),
                                       (NV, np.float32(2.0 ** -70)), (NV, np.float32(2.0 ** 70)),
                                       (MX, 127), (MX, 147), (MX, 0), (MX, 254)])
def test_e2m1_code_of_every_fp32_element(lib, buf, fmt, param):
    """The E2M1 code of every finite x, both signs.  NVFP4 block scales: 1, an
    arbitrary value (the corrected quotient does the work), and scales outside
    [2^-64, 2^64] (IEEE division throughout); within a scale, groups whose
    maximum exceeds s * 2^60 take the IEEE division as in the kernels.  MXFP4
    scale codes: unity, 2^20, and both ends of the UE8M0 range."""
    s = np.float32(param) if fmt == NV else np.float32(2.0 ** (int(param) - 127))
    n = sweep(lib.qfp4_test_element_codes, fmt, param, [POSITIVE, NEGATIVE],
              lambda first, n: oracle.element_codes_bits(first, n, s), buf)
    assert n == 2 * 0x7F800000
