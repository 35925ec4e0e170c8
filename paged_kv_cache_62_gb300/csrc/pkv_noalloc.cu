// Allocation-free decode entry point (include/pkv.h, pkv_paged_decode_noalloc).
//
// Some callers cannot hand the library a workspace: an engine that gave
// (nearly) all free device memory to its KV block pool at start-up, or a host
// framework whose plugin interface passes only inputs and outputs and forbids
// device allocations while it runs.  For them the decode scratch is a fixed
// array owned by this library.  It sits in a translation unit of its own, with
// no kernel, so that the CUDA runtime loads it (and its device memory is
// taken) only when a caller first asks for its address -- the first
// pkv_paged_decode_noalloc call on a device -- never for callers of the other
// entry points.  From then on every device that loaded it holds it until the
// process exits.
#include <mutex>

#include "pkv_host.h"

namespace pkv {

constexpr size_t kStaticScratchBytes = size_t(PKV_NOALLOC_SCRATCH_BYTES);
static __device__ __align__(256) uint8_t g_decode_scratch[kStaticScratchBytes];

// Device address of g_decode_scratch on the current device.  The name of the
// array in host code is only a host-side stand-in, so the address is asked of
// the runtime once per device (with that device current; the lookup also
// loads the array's module on that device) and cached.
static void *static_scratch_address(pkv_status *status)
{
    static std::mutex mu;
    static void *addr[64] = {};
    int dev = -1;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        record_cuda_error("cudaGetDevice", e != cudaSuccess ? cudaGetErrorString(e) : "device index out of range");
        *status = PKV_ECUDA;
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        const cudaError_t se = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (se != cudaSuccess || !p) {
            cudaGetLastError();
            record_cuda_error("cudaGetSymbolAddress", se != cudaSuccess ? cudaGetErrorString(se) : "null address");
            *status = PKV_ECUDA;
            return nullptr;
        }
        addr[dev] = p;
    }
    return addr[dev];
}

}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_paged_decode_noalloc(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                                               const int32_t *block_tables, int32_t max_blocks_per_seq,
                                               const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                                               int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                               int32_t num_blocks, int32_t max_context_len, float scale,
                                               uint16_t *out, int32_t num_workers, int32_t *err_word,
                                               pkv_stream_t stream)
{
    // Size check first, on the host only: reject what does not fit the fixed scratch.
    const size_t need = pkv_paged_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim);
    if (need > kStaticScratchBytes) return PKV_EWORKSPACE;
    if (need == 0)  // invalid sizes: the regular checks answer
        return pkv_paged_decode(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                                num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, max_context_len, scale,
                                out, nullptr, 0, num_workers, err_word, stream);
    // The address lookup also serves as the set-up of a device: a call with num_seqs == 0 does it
    // (and loads the array) without launching anything.
    pkv_status st = PKV_OK;
    void *scratch = static_scratch_address(&st);
    if (!scratch) return st;
    return pkv_paged_decode(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                            num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, max_context_len, scale, out,
                            scratch, kStaticScratchBytes, num_workers, err_word, stream);
}
