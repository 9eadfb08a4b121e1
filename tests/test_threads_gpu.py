"""Two host threads calling the library at once, each on its own CUDA stream.

The host side of the library keeps process-wide state: the per-kernel shared
memory attribute set once per device, the cache of encoded tensor maps, the
cached cluster occupancy of the decode kernel.  All of it sits behind
mutexes.  Here one thread runs prefill-sized GEMMs (CTA pairs) and the
quantiser while the other runs split-K decode GEMMs with their own
workspace; every result must equal, bit for bit, the one the same call gave
before in a single thread (the kernels are deterministic), and no device
status may be raised."""
import threading

import numpy as np
import pytest
import torch

from block_scaled_fp4_tcgen05_gb300 import qfp4, synth
from tests._helpers import NV, dev_scalar, to_dev_u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    qfp4.load()
    assert qfp4.device_check() == 0


def _operands(M, N, K, seed):
    gen = synth.rng(seed)
    dev = []
    for rows in (M, N):
        q = gen.integers(0, 256, size=(rows, K // 2), dtype=np.uint8)
        sf = gen.integers(1, 0x7F, size=(rows, K // 16), dtype=np.uint8)
        m = torch.zeros(qfp4.sf_mma_bytes(rows, K // 16), dtype=torch.uint8, device="cuda")
        qfp4.sf_interleave(to_dev_u8(sf), rows, K // 16, m, qfp4.SF_MMA)
        dev += [to_dev_u8(q), m]
    return dev


def test_two_threads_two_streams():
    ga, gb = dev_scalar(0.5), dev_scalar(1.5)
    # thread 1: prefill GEMM on CTA pairs, then quantise its inputs' source
    Mp, Np, Kp = 1024, 2048, 1024
    pre = _operands(Mp, Np, Kp, 8100)
    x = synth.activations_bf16(8101, 512, 2048)
    X = torch.from_numpy(x.view(np.int16).copy()).view(torch.bfloat16).cuda()
    gsx = torch.empty(1, dtype=torch.float32, device="cuda")
    # thread 2: decode GEMM that splits K (workspace of its own)
    Md, Nd, Kd = 128, 4096, 8192
    dec = _operands(Md, Nd, Kd, 8102)
    ws_bytes = qfp4.gemm_workspace_bytes(NV, Md, Nd, Kd)
    ws = torch.zeros(max(ws_bytes, 16), dtype=torch.uint8, device="cuda")

    def prefill(D, stream=None):
        qfp4.gemm_nt(NV, Mp, Np, Kp, pre[0], pre[1], pre[2], pre[3], ga, gb, D, stream=stream)

    def quant(Q, SF, stream=None):
        qfp4.global_scale(X, gsx, stream=stream)
        qfp4.quantize(NV, X, gsx, Q, SF, qfp4.SF_MMA, stream=stream)

    def decode(D, stream=None):
        qfp4.gemm_nt(NV, Md, Nd, Kd, dec[0], dec[1], dec[2], dec[3], ga, gb, D, ws, ws_bytes, stream=stream)

    # single-threaded references
    Dp_ref = torch.empty((Mp, Np), dtype=torch.bfloat16, device="cuda")
    Dd_ref = torch.empty((Md, Nd), dtype=torch.bfloat16, device="cuda")
    Q_ref = torch.empty((512, 1024), dtype=torch.uint8, device="cuda")
    SF_ref = torch.empty(qfp4.sf_mma_bytes(512, 2048 // 16), dtype=torch.uint8, device="cuda")
    prefill(Dp_ref)
    decode(Dd_ref)
    quant(Q_ref, SF_ref)
    torch.cuda.synchronize()
    assert qfp4.poll_device_status() == 0

    iters = 30
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    Dp = [torch.empty_like(Dp_ref) for _ in range(iters)]
    Dd = [torch.empty_like(Dd_ref) for _ in range(iters)]
    Qs = [torch.empty_like(Q_ref) for _ in range(iters)]
    SFs = [torch.empty_like(SF_ref) for _ in range(iters)]
    errors = []
    start = threading.Barrier(2)

    def worker1():
        try:
            start.wait()
            with torch.cuda.stream(s1):
                for i in range(iters):
                    prefill(Dp[i], stream=s1)
                    quant(Qs[i], SFs[i], stream=s1)
        except Exception as e:          # reported on the main thread
            errors.append(e)

    def worker2():
        try:
            start.wait()
            with torch.cuda.stream(s2):
                for i in range(iters):
                    decode(Dd[i], stream=s2)
        except Exception as e:
            errors.append(e)

    t1, t2 = threading.Thread(target=worker1), threading.Thread(target=worker2)
    t1.start(); t2.start()
    t1.join(); t2.join()
    torch.cuda.synchronize()
    assert not errors, errors
    assert qfp4.poll_device_status() == 0
    for i in range(iters):
        assert torch.equal(Dp[i].view(torch.int16), Dp_ref.view(torch.int16)), f"prefill call {i}"
        assert torch.equal(Dd[i].view(torch.int16), Dd_ref.view(torch.int16)), f"decode call {i}"
        assert torch.equal(Qs[i], Q_ref) and torch.equal(SFs[i], SF_ref), f"quantise call {i}"
