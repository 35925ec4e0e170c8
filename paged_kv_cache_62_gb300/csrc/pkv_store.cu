// Decode-step slot computation and the store_kvcache scatter.
//
// pkv_decode_slot_mapping: slot of the token each sequence appends --
//   block_tables[b][pos / bs] * bs + pos % bs with pos = context_lens[b] - 1
//   (nano-vLLM lab manual §5.2.3 / B.2.3; nano-vllm KV-cache post §3.1, §4.4).
// pkv_kv_store: row slot_mapping[t] of k_cache / v_cache becomes a copy of
//   k[t] / v[t]; slot -1 skips the row (MinivLLM review, "注意力内核的三个分支").
//
// pkv_decode_store: both in one launch for a decode step (one new token per
//   sequence, at position context_lens[b] - 1).
// pkv_kv_store_fp8: the same scatter into E4M3 caches, each element stored as
//   the E4M3 code of x / scale[kv head] (an IEEE binary32 division, then the
//   conversion's round to nearest even, saturating at +-448).
// pkv_copy_blocks: copy-on-write block copies, block dst of both caches
//   becomes a bit copy of block src (nano-vllm KV-cache post §2.2; mini-vLLM
//   README §1, copy-on-write of a half-full shared block).
//
// The first two are tiny, latency-bound launches.  The store moves whole cache rows
// (num_kv_heads * head_dim bf16, 2 KiB for Qwen3-0.6B) with 16-byte vector
// loads/stores: one CTA per token, consecutive threads on consecutive 16-byte
// chunks of the row, so every warp access is a fully coalesced 512-byte run.
#include <algorithm>

#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {

__global__ void decode_slot_mapping_kernel(const int32_t *__restrict__ block_tables, int32_t max_blocks,
                                           const int32_t *__restrict__ context_lens, int32_t num_seqs,
                                           int32_t block_size, int32_t log2_bs, int32_t num_blocks,
                                           int32_t *__restrict__ slot_mapping, int32_t num_tokens,
                                           int32_t *err)
{
    griddep_launch_dependents();
    griddep_wait();
    const int32_t t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= num_tokens) return;
    int32_t slot = -1;
    if (t < num_seqs) {
        const int32_t len = __ldg(context_lens + t);
        if (len > 0) {
            const int32_t pos = len - 1;
            const int32_t logical = pos >> log2_bs;
            if (logical >= max_blocks) {
                flag_error(err, PKV_ERR_CONTEXT_RANGE);
            } else {
                const int32_t phys = __ldg(block_tables + static_cast<int64_t>(t) * max_blocks + logical);
                if (phys < 0 || phys >= num_blocks)
                    flag_error(err, PKV_ERR_BLOCK_RANGE);
                else
                    slot = phys * block_size + (pos & (block_size - 1));
            }
        } else if (len < 0) {
            flag_error(err, PKV_ERR_CONTEXT_RANGE);
        }
    }
    slot_mapping[t] = slot;
}

__global__ void kv_store_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                                const int32_t *__restrict__ slot_mapping, uint4 *__restrict__ k_cache,
                                uint4 *__restrict__ v_cache, int64_t num_slots, int32_t row_vecs, int32_t *err)
{
    griddep_launch_dependents();
    griddep_wait();
    const int32_t t = blockIdx.x;
    const int64_t s = __ldg(slot_mapping + t);
    if (s == -1) return;
    if (s < 0 || s >= num_slots) {
        if (threadIdx.x == 0) flag_error(err, PKV_ERR_SLOT_RANGE);
        return;
    }
    const uint4 *ks = k + static_cast<int64_t>(t) * row_vecs;
    const uint4 *vs = v + static_cast<int64_t>(t) * row_vecs;
    uint4 *kd = k_cache + s * row_vecs;
    uint4 *vd = v_cache + s * row_vecs;
    for (int32_t i = threadIdx.x; i < row_vecs; i += blockDim.x) {
        const uint4 a = __ldg(ks + i);
        const uint4 b = __ldg(vs + i);
        kd[i] = a;
        vd[i] = b;
    }
}

// A decode step's store in one launch: CTA b computes the slot of position
// L_b - 1 (every thread loads the same length and table entry, so no
// barrier is needed) and copies row b of k and v there.
__global__ void decode_store_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                                    const int32_t *__restrict__ block_tables, int32_t max_blocks,
                                    const int32_t *__restrict__ context_lens, int32_t block_size, int32_t log2_bs,
                                    int32_t num_blocks, uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                                    int32_t row_vecs, int32_t *__restrict__ slot_mapping, int32_t *err)
{
    griddep_launch_dependents();
    griddep_wait();
    const int32_t b = blockIdx.x;
    const int32_t len = __ldg(context_lens + b);
    int64_t slot = -1;
    if (len > 0) {
        const int32_t pos = len - 1;
        const int32_t logical = pos >> log2_bs;
        if (logical >= max_blocks) {
            if (threadIdx.x == 0) flag_error(err, PKV_ERR_CONTEXT_RANGE);
        } else {
            const int32_t phys = __ldg(block_tables + int64_t(b) * max_blocks + logical);
            if (phys < 0 || phys >= num_blocks) {
                if (threadIdx.x == 0) flag_error(err, PKV_ERR_BLOCK_RANGE);
            } else {
                slot = int64_t(phys) * block_size + (pos & (block_size - 1));
            }
        }
    } else if (len < 0 && threadIdx.x == 0) {
        flag_error(err, PKV_ERR_CONTEXT_RANGE);
    }
    if (slot_mapping && threadIdx.x == 0) slot_mapping[b] = int32_t(slot);
    if (slot < 0) return;
    const uint4 *ks = k + int64_t(b) * row_vecs;
    const uint4 *vs = v + int64_t(b) * row_vecs;
    uint4 *kd = k_cache + slot * row_vecs;
    uint4 *vd = v_cache + slot * row_vecs;
    for (int32_t i = threadIdx.x; i < row_vecs; i += blockDim.x) {
        const uint4 a = __ldg(ks + i);
        const uint4 c = __ldg(vs + i);
        kd[i] = a;
        vd[i] = c;
    }
}

// One CTA per token; thread i quantises the 8-element group i of the row
// (group i belongs to kv head i / (D / 8)).
__global__ void kv_store_fp8_kernel(const uint4 *__restrict__ k, const uint4 *__restrict__ v,
                                    const int32_t *__restrict__ slot_mapping, uint2 *__restrict__ k_cache,
                                    uint2 *__restrict__ v_cache, int64_t num_slots, int32_t row_groups,
                                    int32_t head_groups, const float *__restrict__ k_scale,
                                    const float *__restrict__ v_scale, int32_t *err)
{
    griddep_launch_dependents();
    griddep_wait();
    const int32_t t = blockIdx.x;
    const int64_t s = __ldg(slot_mapping + t);
    if (s == -1) return;
    if (s < 0 || s >= num_slots) {
        if (threadIdx.x == 0) flag_error(err, PKV_ERR_SLOT_RANGE);
        return;
    }
    for (int32_t i = threadIdx.x; i < row_groups; i += blockDim.x) {
        const int32_t h = i / head_groups;
        const int64_t src = int64_t(t) * row_groups + i, dst = s * row_groups + i;
        k_cache[dst] = quantise8_e4m3(__ldg(k + src), __ldg(k_scale + h));
        v_cache[dst] = quantise8_e4m3(__ldg(v + src), __ldg(v_scale + h));
    }
}

// Copy-on-write block copies.  The work is cut into 32 KiB chunks of one
// block of one cache; a persistent grid walks the chunks, every thread keeping
// eight 16-byte loads in flight (the copy is bound by HBM read + write).  Loads
// go through L2 only; stores are plain (marking them streaming measured 8 %
// slower on GB300).  Measured on 120 pairs of 512 KiB blocks: the same time as
// torch's own device copy of the same bytes.
constexpr int kCopyThreads = 256;
constexpr int kCopyVecs = 8;                                 // 16-byte vectors in flight per thread
constexpr int64_t kChunkVecs = kCopyThreads * kCopyVecs;     // vectors per chunk (32 KiB)

__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(uint4 *__restrict__ k_cache,
                                                                   uint4 *__restrict__ v_cache,
                                                                   const int32_t *__restrict__ pairs,
                                                                   int32_t num_pairs, int32_t num_blocks,
                                                                   int64_t block_vecs, int64_t chunks_per_block,
                                                                   int32_t *err)
{
    griddep_launch_dependents();
    griddep_wait();
    const int64_t total = int64_t(num_pairs) * 2 * chunks_per_block;
    for (int64_t c = blockIdx.x; c < total; c += gridDim.x) {
        const int64_t pc = c / chunks_per_block;  // (pair, cache)
        const int64_t part = c - pc * chunks_per_block;
        const int32_t i = int32_t(pc >> 1);
        const int32_t src = __ldg(pairs + 2 * i), dst = __ldg(pairs + 2 * i + 1);
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
            if (threadIdx.x == 0 && (pc & 1) == 0 && part == 0) flag_error(err, PKV_ERR_BLOCK_RANGE);
            continue;
        }
        if (src == dst) continue;
        uint4 *base = (pc & 1) ? v_cache : k_cache;
        const uint4 *from = base + int64_t(src) * block_vecs;
        uint4 *to = base + int64_t(dst) * block_vecs;
        const int64_t v0 = part * kChunkVecs + threadIdx.x;
        uint4 x[kCopyVecs];
#pragma unroll
        for (int j = 0; j < kCopyVecs; ++j) {
            const int64_t v = v0 + int64_t(j) * kCopyThreads;
            if (v < block_vecs) x[j] = __ldcg(from + v);
        }
#pragma unroll
        for (int j = 0; j < kCopyVecs; ++j) {
            const int64_t v = v0 + int64_t(j) * kCopyThreads;
            if (v < block_vecs) to[v] = x[j];
        }
    }
}

}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_decode_slot_mapping(const int32_t *block_tables, int32_t max_blocks_per_seq,
                                              const int32_t *context_lens, int32_t num_seqs, int32_t block_size,
                                              int32_t num_blocks, int32_t *slot_mapping, int32_t num_tokens,
                                              int32_t *err_word, pkv_stream_t stream)
{
    if (num_seqs < 0 || num_tokens < num_seqs || max_blocks_per_seq <= 0 || num_blocks <= 0) return PKV_EINVAL;
    if (!is_pow2(block_size)) return PKV_EINVAL;
    if (static_cast<int64_t>(num_blocks) * block_size > INT32_MAX) return PKV_EBOUNDS;
    if (num_tokens == 0) return PKV_OK;
    if (!slot_mapping || (num_seqs > 0 && (!block_tables || !context_lens))) return PKV_EINVAL;
    const int threads = 128;
    const int blocks = (num_tokens + threads - 1) / threads;
    const cudaError_t e =
        launch_pdl(decode_slot_mapping_kernel, dim3(blocks), dim3(threads), 0, reinterpret_cast<cudaStream_t>(stream),
                   block_tables, max_blocks_per_seq, context_lens, num_seqs, block_size, ilog2(block_size),
                   num_blocks, slot_mapping, num_tokens, err_word);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return cuda_fail("decode_slot_mapping_kernel launch", e);
    }
    return launch_status("decode_slot_mapping_kernel launch");
}

extern "C" pkv_status pkv_kv_store(const uint16_t *k, const uint16_t *v, const int32_t *slot_mapping,
                                   int32_t num_tokens, uint16_t *k_cache, uint16_t *v_cache, int32_t num_blocks,
                                   int32_t block_size, int32_t num_kv_heads, int32_t head_dim, int32_t *err_word,
                                   pkv_stream_t stream)
{
    if (num_tokens < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
        return PKV_EINVAL;
    const int64_t row_bytes = static_cast<int64_t>(num_kv_heads) * head_dim * 2;
    if (row_bytes % 16 != 0 || row_bytes / 16 > INT32_MAX) return PKV_EINVAL;
    if (num_tokens == 0) return PKV_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PKV_EINVAL;
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache)) return PKV_EINVAL;
    const int32_t row_vecs = static_cast<int32_t>(row_bytes / 16);
    const int threads = row_vecs >= 256 ? 256 : ((row_vecs + 31) / 32) * 32;
    const cudaError_t e =
        launch_pdl(kv_store_kernel, dim3(num_tokens), dim3(threads), 0, reinterpret_cast<cudaStream_t>(stream),
                   reinterpret_cast<const uint4 *>(k), reinterpret_cast<const uint4 *>(v), slot_mapping,
                   reinterpret_cast<uint4 *>(k_cache), reinterpret_cast<uint4 *>(v_cache),
                   static_cast<int64_t>(num_blocks) * block_size, row_vecs, err_word);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return cuda_fail("kv_store_kernel launch", e);
    }
    return launch_status("kv_store_kernel launch");
}

// A wait on an mbarrier that nothing completes: the bounded wait gives up at
// its time limit, the kernel flags PKV_ERR_WAIT_TIMEOUT and returns (the
// timeout path of every wait in the library, exercised without a fault).
__global__ void diag_wait_timeout_kernel(int32_t *err)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncwarp();
    if (!mbar_wait_bounded(&bar, 0u) && threadIdx.x == 0) flag_error(err, PKV_ERR_WAIT_TIMEOUT);
}

extern "C" pkv_status pkv_diag_wait_timeout(int32_t *err_word, pkv_stream_t stream)
{
    if (!err_word) return PKV_EINVAL;
    diag_wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(err_word);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail("diag_wait_timeout_kernel launch", e);
    return launch_status("diag_wait_timeout_kernel launch");
}

extern "C" pkv_status pkv_copy_blocks(uint16_t *k_cache, uint16_t *v_cache, const int32_t *pairs,
                                      int32_t num_pairs, int32_t num_blocks, int32_t block_size,
                                      int32_t num_kv_heads, int32_t head_dim, int32_t *err_word,
                                      pkv_stream_t stream)
{
    if (num_pairs < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
        return PKV_EINVAL;
    const int64_t block_bytes = int64_t(block_size) * num_kv_heads * head_dim * 2;
    if (block_bytes % 16 != 0) return PKV_EINVAL;
    if (num_pairs == 0) return PKV_OK;
    if (!k_cache || !v_cache || !pairs) return PKV_EINVAL;
    if (!aligned16(k_cache) || !aligned16(v_cache)) return PKV_EINVAL;
    DeviceInfo dev;
    if (!current_device_info(&dev)) return PKV_ECUDA;
    const int64_t block_vecs = block_bytes / 16;
    const int64_t chunks_per_block = (block_vecs + kChunkVecs - 1) / kChunkVecs;
    const int64_t total = int64_t(num_pairs) * 2 * chunks_per_block;
    // persistent grid: up to 8 CTAs of 256 threads per SM, never more CTAs than chunks
    const int64_t grid = std::min<int64_t>(total, int64_t(dev.sm_count) * 8);
    const cudaError_t e = launch_pdl(copy_blocks_kernel, dim3(unsigned(grid)), dim3(kCopyThreads), 0,
                                     reinterpret_cast<cudaStream_t>(stream), reinterpret_cast<uint4 *>(k_cache),
                                     reinterpret_cast<uint4 *>(v_cache), pairs, num_pairs, num_blocks, block_vecs,
                                     chunks_per_block, err_word);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return cuda_fail("copy_blocks_kernel launch", e);
    }
    return launch_status("copy_blocks_kernel launch");
}

extern "C" pkv_status pkv_kv_store_fp8(const uint16_t *k, const uint16_t *v, const int32_t *slot_mapping,
                                       int32_t num_tokens, uint8_t *k_cache, uint8_t *v_cache, int32_t num_blocks,
                                       int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                                       const float *k_scale, const float *v_scale, int32_t *err_word,
                                       pkv_stream_t stream)
{
    if (num_tokens < 0 || num_blocks <= 0 || block_size <= 0 || num_kv_heads <= 0 || head_dim <= 0)
        return PKV_EINVAL;
    if (head_dim % 8 != 0 || int64_t(num_kv_heads) * head_dim / 8 > INT32_MAX) return PKV_EINVAL;
    if (num_tokens == 0) return PKV_OK;
    if (!k || !v || !slot_mapping || !k_cache || !v_cache || !k_scale || !v_scale) return PKV_EINVAL;
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache)) return PKV_EINVAL;
    const int32_t row_groups = num_kv_heads * (head_dim / 8);
    const int threads = row_groups >= 256 ? 256 : ((row_groups + 31) / 32) * 32;
    const cudaError_t e =
        launch_pdl(kv_store_fp8_kernel, dim3(num_tokens), dim3(threads), 0, reinterpret_cast<cudaStream_t>(stream),
                   reinterpret_cast<const uint4 *>(k), reinterpret_cast<const uint4 *>(v), slot_mapping,
                   reinterpret_cast<uint2 *>(k_cache), reinterpret_cast<uint2 *>(v_cache),
                   static_cast<int64_t>(num_blocks) * block_size, row_groups, head_dim / 8, k_scale, v_scale, err_word);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return cuda_fail("kv_store_fp8_kernel launch", e);
    }
    return launch_status("kv_store_fp8_kernel launch");
}

extern "C" pkv_status pkv_decode_store(const uint16_t *k, const uint16_t *v, const int32_t *block_tables,
                                       int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs,
                                       uint16_t *k_cache, uint16_t *v_cache, int32_t num_blocks, int32_t block_size,
                                       int32_t num_kv_heads, int32_t head_dim, int32_t *slot_mapping,
                                       int32_t *err_word, pkv_stream_t stream)
{
    if (num_seqs < 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 || num_kv_heads <= 0 || head_dim <= 0)
        return PKV_EINVAL;
    if (!is_pow2(block_size)) return PKV_EINVAL;
    if (static_cast<int64_t>(num_blocks) * block_size > INT32_MAX) return PKV_EBOUNDS;
    const int64_t row_bytes = static_cast<int64_t>(num_kv_heads) * head_dim * 2;
    if (row_bytes % 16 != 0 || row_bytes / 16 > INT32_MAX) return PKV_EINVAL;
    if (num_seqs == 0) return PKV_OK;
    if (!k || !v || !block_tables || !context_lens || !k_cache || !v_cache) return PKV_EINVAL;
    if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache)) return PKV_EINVAL;
    const int32_t row_vecs = static_cast<int32_t>(row_bytes / 16);
    const int threads = row_vecs >= 256 ? 256 : ((row_vecs + 31) / 32) * 32;
    const cudaError_t e =
        launch_pdl(decode_store_kernel, dim3(num_seqs), dim3(threads), 0, reinterpret_cast<cudaStream_t>(stream),
                   reinterpret_cast<const uint4 *>(k), reinterpret_cast<const uint4 *>(v), block_tables,
                   max_blocks_per_seq, context_lens, block_size, ilog2(block_size), num_blocks,
                   reinterpret_cast<uint4 *>(k_cache), reinterpret_cast<uint4 *>(v_cache), row_vecs, slot_mapping,
                   err_word);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return cuda_fail("decode_store_kernel launch", e);
    }
    return launch_status("decode_store_kernel launch");
}
