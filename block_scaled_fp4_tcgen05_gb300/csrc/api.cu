// api.cu -- library-wide entry points of libqfp4: version, status text,
// device check and the device status poll.
#include <cstdint>
#include <cuda_runtime.h>
#include <mutex>
#include <set>
#include <utility>

#include "qfp4_common.cuh"
#include "qfp4_gemm_internal.cuh"

namespace qfp4 {

int ensure_thread_context()
{
    // The runtime makes the primary context current on a host thread only
    // when that thread makes certain runtime calls; a driver-API call (the
    // tensor-map encode) from a thread that has made none fails with
    // CUDA_ERROR_INVALID_CONTEXT.  cudaSetDevice binds the current device's
    // primary context to the calling thread; done once per thread and device.
    thread_local int bound = -1;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return QFP4_ERR_CUDA;
    if (dev != bound) {
        if (cudaSetDevice(dev) != cudaSuccess) return QFP4_ERR_CUDA;
        bound = dev;
    }
    return QFP4_OK;
}

int ensure_smem_attr(const void *kern, int bytes)
{
    static std::mutex mu;
    static std::set<std::pair<const void *, int>> done;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return QFP4_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (done.count({kern, dev})) return QFP4_OK;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return QFP4_ERR_CUDA;
    done.insert({kern, dev});
    return QFP4_OK;
}

}  // namespace qfp4

extern "C" int qfp4_version(void) { return 100; }   // 0.1.0

extern "C" const char *qfp4_status_string(int status)
{
    switch (status) {
    case QFP4_OK: return "ok";
    case QFP4_ERR_INVALID_ARG: return "invalid argument";
    case QFP4_ERR_UNSUPPORTED: return "unsupported shape or option";
    case QFP4_ERR_MISALIGNED: return "pointer not aligned as required";
    case QFP4_ERR_CUDA: return "CUDA call failed";
    case QFP4_ERR_TIMEOUT: return "device-side bounded wait ran out";
    case QFP4_ERR_ARCH: return "current device is not an sm_103 GPU";
    case QFP4_ERR_WORKSPACE: return "workspace missing or too small";
    default: return "unknown status";
    }
}

extern "C" int qfp4_device_check(void)
{
    int dev = 0, major = 0, minor = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return QFP4_ERR_CUDA;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return QFP4_ERR_CUDA;
    return (major == 10 && minor == 3) ? QFP4_OK : QFP4_ERR_ARCH;
}

extern "C" int qfp4_poll_device_status(void *stream)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t q = 0, g = 0, gp = 0, gd = 0, gs = 0;
    int rc = qfp4::read_clear_status_quant(s, &q);
    if (rc == QFP4_OK) rc = qfp4::read_clear_status_gemm(s, &g);
    if (rc == QFP4_OK) rc = qfp4::read_clear_status_gemm_pair(s, &gp);
    if (rc == QFP4_OK) rc = qfp4::read_clear_status_gemm_decode(s, &gd);
    if (rc == QFP4_OK) rc = qfp4::read_clear_status_gemm_sparse(s, &gs);
    if (rc != QFP4_OK) return rc;
    const uint32_t all = q | g | gp | gd | gs;
    if (all & qfp4::kStatusTimeout) return QFP4_ERR_TIMEOUT;
    if (all & (qfp4::kStatusBadGroup | qfp4::kStatusBadSparsity)) return QFP4_ERR_INVALID_ARG;
    return QFP4_OK;
}
