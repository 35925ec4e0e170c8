// Host-side helpers shared by the pkv entry points: argument checks, the
// per-device attribute cache and the driver entry point for tensor maps.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <utility>

#include "../../include/pkv.h"

namespace pkv {

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bool is_pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }

inline int ilog2(int64_t x)
{
    int r = 0;
    while ((int64_t(1) << (r + 1)) <= x) ++r;
    return r;
}

struct DeviceInfo {
    int device = -1;
    int sm_count = 0;
    int max_smem_optin = 0;
};

// Attributes of the current device (cached per device id).  Returns false if
// no device is current / visible.
bool current_device_info(DeviceInfo *info);

// cuTensorMapEncodeTiled obtained through the runtime's driver entry point
// (no link-time dependency on libcuda).  nullptr if unavailable.
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);
EncodeTiledFn encode_tiled_fn();

// Launch with programmatic stream serialization (see griddep_wait in
// pkv_device.cuh): the kernel may start before its predecessor in the stream
// finishes and waits on the device for it before touching memory.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Remember why a call is about to return PKV_ECUDA (per host thread), for
// pkv_last_cuda_error().
void record_cuda_error(const char *where, const char *what);

inline pkv_status cuda_fail(const char *where, cudaError_t e)
{
    record_cuda_error(where, cudaGetErrorString(e));
    return PKV_ECUDA;
}

// Status of the launch just made (clears the runtime's sticky launch error).
inline pkv_status launch_status(const char *where)
{
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? PKV_OK : cuda_fail(where, e);
}

}  // namespace pkv
