"""A device-side bounded wait made to run out on purpose, in the allowed
form: a barrier arrival that never comes (no trap, no bad address).

Every wait in the library's kernels is bounded; one that runs out records
QFP4_ERR_TIMEOUT in the device status word, the kernel leaves through its
abort path (in-flight copies given time to land, tensor memory freed) and the
context stays usable.  The fault-injection test build (libqfp4_faultinj.so:
the same sources with QFP4_FAULT_INJECTION, a 5 ms wait limit and the hook
qfp4_test_inject_skip_release) lets the leader epilogue of the first CTA
pair skip its release of the accumulator after its first tile, so that the
MMA issuer's next wait, and then every other role's of that pair, run out.
No copy engine transfer completes on that barrier.

The test expects QFP4_ERR_TIMEOUT from qfp4_poll_device_status within well
under a second, then runs the same GEMM with the hook disarmed and checks it
bit for bit against the released library."""
import time

import numpy as np
import pytest
import torch

from block_scaled_fp4_tcgen05_gb300 import qfp4, synth
from tests._helpers import NV, dev_scalar, to_dev_u8

pytestmark = pytest.mark.gpu

QFP4_ERR_TIMEOUT = -5


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    qfp4.load()
    assert qfp4.device_check() == 0


def _fault_lib():
    from block_scaled_fp4_tcgen05_gb300 import build
    build.build(variant="faultinj")          # no-op when already built
    return qfp4.load_fault_injection()


def _operands(M, N, K, seed):
    gen = synth.rng(seed)
    A = gen.integers(0, 256, size=(M, K // 2), dtype=np.uint8)
    B = gen.integers(0, 256, size=(N, K // 2), dtype=np.uint8)
    dev = []
    for q, rows in ((A, M), (B, N)):
        sf = gen.integers(1, 0x7F, size=(rows, K // 16), dtype=np.uint8)
        m = torch.zeros(qfp4.sf_mma_bytes(rows, K // 16), dtype=torch.uint8, device="cuda")
        qfp4.sf_interleave(to_dev_u8(sf), rows, K // 16, m, qfp4.SF_MMA)
        dev += [to_dev_u8(q), m]
    return dev


def _call(lib, M, N, K, dev, ga, gb, D):
    return lib.qfp4_gemm_nt(NV, M, N, K, dev[0].data_ptr(), dev[1].data_ptr(), dev[2].data_ptr(),
                            dev[3].data_ptr(), ga.data_ptr(), gb.data_ptr(), D.data_ptr(), None, 0,
                            torch.cuda.current_stream().cuda_stream)


def test_bounded_wait_runs_out_and_the_context_stays_usable():
    lib = _fault_lib()
    # 256 pair tiles on at most 76 pairs: the first pair has a second tile,
    # whose MMAs wait for the release that is skipped
    M, N, K = 4096, 4096, 256
    dev = _operands(M, N, K, 7700)
    ga, gb = dev_scalar(0.5), dev_scalar(2.0)
    D_ref = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    qfp4.gemm_nt(NV, M, N, K, dev[0], dev[1], dev[2], dev[3], ga, gb, D_ref)
    torch.cuda.synchronize()
    assert qfp4.poll_device_status() == 0
    assert lib.qfp4_poll_device_status(None) == 0            # nothing pending in the test library

    assert lib.qfp4_test_inject_skip_release(1) == 0
    D = torch.full((M, N), 3.0, dtype=torch.bfloat16, device="cuda")
    t0 = time.perf_counter()
    assert _call(lib, M, N, K, dev, ga, gb, D) == 0           # the launch itself is fine
    torch.cuda.synchronize()                                  # the kernel ends (no hang)
    elapsed = time.perf_counter() - t0
    assert lib.qfp4_poll_device_status(None) == QFP4_ERR_TIMEOUT
    assert elapsed < 1.0, f"the 5 ms waits took {elapsed:.3f} s to run out"
    assert lib.qfp4_poll_device_status(None) == 0             # the status word was cleared

    # disarmed: the same call is correct again in the same context
    assert lib.qfp4_test_inject_skip_release(0) == 0
    D2 = torch.full((M, N), 3.0, dtype=torch.bfloat16, device="cuda")
    assert _call(lib, M, N, K, dev, ga, gb, D2) == 0
    torch.cuda.synchronize()
    assert lib.qfp4_poll_device_status(None) == 0
    assert torch.equal(D2.view(torch.int16), D_ref.view(torch.int16))
