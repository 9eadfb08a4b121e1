// qfp4_common.cuh -- shared host/device helpers of libqfp4 (not part of the ABI).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/qfp4.h"

namespace qfp4 {

// Device status word: one per translation unit that launches kernels.  A
// kernel that gives up on a bounded wait ORs in a bit; qfp4_poll_device_status
// reads and clears every unit's word.
enum : uint32_t { kStatusTimeout = 1u, kStatusBadGroup = 2u, kStatusBadSparsity = 4u };

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

inline int block_elems(int fmt)
{
    return fmt == QFP4_NVFP4 ? 16 : (fmt == QFP4_MXFP4 || fmt == QFP4_NVFP4_B32) ? 32 : 0;
}

inline int launch_status(cudaError_t e)
{
    return e == cudaSuccess ? QFP4_OK : QFP4_ERR_CUDA;
}

// Raises `kern`'s dynamic shared-memory limit to `bytes` on the current
// device, once per (kernel, device); later calls only look the pair up.
// Safe to call from several host threads (a mutex guards the record).
int ensure_smem_attr(const void *kern, int bytes);

// Makes the current device's primary context current on the calling host
// thread (needed before driver-API calls from a thread that has made no
// runtime call yet).  Once per (thread, device).
int ensure_thread_context();

// Grouped launches read per-group row offsets from device memory.  They are
// usable only if they start at 0, never decrease, end at the row count the
// host sized the launch for and, when max_rows > 0, give no group more than
// max_rows rows.  A kernel that finds them otherwise records kStatusBadGroup
// and writes nothing.
__device__ __forceinline__ bool group_offsets_valid(const int32_t *offs, int groups, int64_t total_rows,
                                                    int64_t max_rows)
{
    if (offs[0] != 0 || offs[groups] != total_rows) return false;
    for (int e = 0; e < groups; ++e) {
        const int64_t rows = static_cast<int64_t>(offs[e + 1]) - offs[e];
        if (rows < 0 || (max_rows > 0 && rows > max_rows)) return false;
    }
    return true;
}

inline int sm_count()
{
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

// Programmatic dependent launch.  Every kernel of this library is launched
// with programmatic stream serialisation: it may start (set up barriers,
// tensor memory and descriptors) while the previous kernel on the stream is
// still finishing, and it calls pdl_wait() before its first access to global
// memory; that returns once the previous kernel has completed and its writes
// are visible.  A preceding kernel that was launched without this attribute
// (any other library's) is simply waited for in full.
__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Allows the next kernel on the stream to begin launching now (it still
// waits for this kernel to complete before it touches memory).
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Per-unit status readers (defined in each .cu that owns a status word).
int read_clear_status_quant(cudaStream_t s, uint32_t *out);
int read_clear_status_gemm(cudaStream_t s, uint32_t *out);
int read_clear_status_gemm_sparse(cudaStream_t s, uint32_t *out);

}  // namespace qfp4
