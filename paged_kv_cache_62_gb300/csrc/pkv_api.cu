// Library-wide entry points (version, status strings) and host helpers.
#include <cstdio>
#include <mutex>

#include "pkv_host.h"

namespace pkv {

static thread_local char g_last_cuda_error[256] = "";

void record_cuda_error(const char *where, const char *what)
{
    std::snprintf(g_last_cuda_error, sizeof g_last_cuda_error, "%s: %s", where, what);
}

bool current_device_info(DeviceInfo *info)
{
    static std::mutex mu;
    static DeviceInfo cache[64];
    int dev = -1;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        record_cuda_error("cudaGetDevice", e != cudaSuccess ? cudaGetErrorString(e) : "device index out of range");
        return false;
    }
    std::lock_guard<std::mutex> lock(mu);
    DeviceInfo &c = cache[dev];
    if (c.device != dev) {
        int sms = 0, smem = 0;
        cudaError_t a = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (a == cudaSuccess) a = cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (a != cudaSuccess) {
            cudaGetLastError();
            record_cuda_error("cudaDeviceGetAttribute", cudaGetErrorString(a));
            return false;
        }
        c.sm_count = sms;
        c.max_smem_optin = smem;
        c.device = dev;
    }
    *info = c;
    return true;
}

EncodeTiledFn encode_tiled_fn()
{
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        cudaGetLastError();
    });
    return fn;
}

}  // namespace pkv

extern "C" int pkv_abi_version(void) { return 2; }

extern "C" const char *pkv_last_cuda_error(void) { return pkv::g_last_cuda_error; }

extern "C" const char *pkv_status_string(int status)
{
    switch (status) {
    case PKV_OK: return "ok";
    case PKV_EINVAL: return "invalid argument (pointer, size, shape or alignment)";
    case PKV_EUNSUPPORTED: return "unsupported configuration";
    case PKV_ECUDA: return "CUDA call or kernel launch failed";
    case PKV_EWORKSPACE: return "workspace missing or too small";
    case PKV_EBOUNDS: return "size beyond a limit of the library";
    case PKV_EFULL: return "not enough free blocks";
    default: return "unknown pkv status";
    }
}
