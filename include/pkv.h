/*
 * pkv.h -- C ABI of libpkv.so, the GB300 (sm_103a) paged KV cache hot path.
 *
 * The library implements the two device operations that a paged-KV decode
 * step needs, plus the slot computation that feeds the first one:
 *
 *   pkv_decode_slot_mapping  slot_mapping of the token each sequence appends
 *   pkv_kv_store             store_kvcache: scatter new K/V rows into the cache
 *   pkv_paged_decode         q_len = 1 GQA PagedAttention over the block tables
 *
 * Conventions shared by every entry point
 *   - All array pointers are DEVICE pointers owned by the caller.  The library
 *     allocates no device memory, keeps no state that affects results (only
 *     host-side memos such as encoded tensor maps) and never synchronises the
 *     stream.  Work is enqueued asynchronously on `stream` (NULL = the legacy
 *     default stream); the return code covers only host-side argument checks
 *     and the launch itself.
 *   - bf16 arrays hold IEEE bfloat16 values (uint16 bit patterns); index arrays
 *     are int32.  Every multi-dimensional array is dense, row-major
 *     (C-contiguous) with the shape given below, and must start on a 16-byte
 *     boundary.
 *   - Problems that only the device can see (a slot or block id outside the
 *     cache, a context length outside its table) never trap: the kernel skips
 *     the offending access and ORs a PKV_ERR_* bit into *err_word (a device
 *     int32, may be NULL).  Read it after synchronising; clear it yourself.
 *     Output values are unspecified for a call that set a bit.
 *   - Out-of-place only: outputs may not alias inputs.
 *   - Entry points may be called from several host threads on different
 *     streams; calls are independent.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t (struct CUstream_st *). */
typedef struct CUstream_st *pkv_stream_t;

typedef enum {
    PKV_OK = 0,
    PKV_EINVAL = -1,       /* bad pointer, size, shape or alignment            */
    PKV_EUNSUPPORTED = -2, /* valid request outside the compiled variants      */
    PKV_ECUDA = -3,        /* a CUDA runtime/driver call or launch failed      */
    PKV_EWORKSPACE = -4,   /* workspace missing or smaller than required       */
    PKV_EBOUNDS = -5,      /* a size beyond a limit of the library: PKV_MAX_SEQS,
                              PKV_MAX_WORKERS, num_blocks * block_size < 2^31,
                              or a block table row too short for a sequence     */
    PKV_EFULL = -6         /* block allocator: not enough free blocks          */
} pkv_status;

/* Bits ORed into *err_word by the kernels. */
#define PKV_ERR_SLOT_RANGE 0x1    /* slot_mapping entry not -1 and outside [0, num_blocks*block_size) */
#define PKV_ERR_BLOCK_RANGE 0x2   /* block table entry that must be read lies outside [0, num_blocks) */
#define PKV_ERR_CONTEXT_RANGE 0x4 /* context_len < 0 or above min(max_context_len, max_blocks*block_size) */
#define PKV_ERR_WAIT_TIMEOUT 0x8  /* a bounded wait on an asynchronous copy gave up                    */
#define PKV_ERR_WORKSPACE 0x10    /* decode workspace control block not in a state this library left   */

/* Version of this ABI (bumped on any incompatible change). */
PKV_API int pkv_abi_version(void);

/* Static text for a pkv_status value (never NULL). */
PKV_API const char *pkv_status_string(int status);

/* Why the most recent call on this host thread returned PKV_ECUDA: the CUDA
 * call that failed and its error text ("" if none yet).  The text stays
 * valid until the next failing call on the same thread. */
PKV_API const char *pkv_last_cuda_error(void);

/*
 * pkv_decode_slot_mapping -- the cache slot of the token each sequence
 * appends in this decode step.
 *
 * Defined by the nano-vLLM lab manual (§5.2.3 and appendix B.2.3) and the
 * nano-vllm KV-cache post (§3.1, §3.5, §4.4): the physical row of logical
 * position pos is block_tables[b][pos / block_size] * block_size +
 * pos % block_size; in a decode step the appended token sits at
 * pos = context_lens[b] - 1 because context_lens already count it
 * (lab manual §5.2.1; post §4.4: context_lens [431, 434] give slots
 * [430, 689] with block_size 256).
 *
 *   block_tables  [num_seqs, max_blocks_per_seq] int32, unused entries -1
 *   context_lens  [num_seqs] int32
 *   slot_mapping  [num_tokens] int32 output; num_tokens >= num_seqs.
 *                 Row t < num_seqs gets the slot of sequence t (or -1 when
 *                 context_lens[t] == 0); rows t >= num_seqs are padding and
 *                 get -1 (lab manual appendix B.4: padding rows must not
 *                 write the cache).
 *   num_blocks    physical blocks in the cache (for the range check)
 * A context length that does not fit its table row, or a table entry outside
 * [0, num_blocks), yields -1 for that row and sets the matching err bit.
 */
PKV_API pkv_status pkv_decode_slot_mapping(const int32_t *block_tables, int32_t max_blocks_per_seq,
                                   const int32_t *context_lens, int32_t num_seqs,
                                   int32_t block_size, int32_t num_blocks,
                                   int32_t *slot_mapping, int32_t num_tokens,
                                   int32_t *err_word, pkv_stream_t stream);

/*
 * pkv_kv_store -- store_kvcache: write each new token's K and V rows into
 * the paged cache through slot_mapping.
 *
 * Defined by the MinivLLM review (section "注意力内核的三个分支": the store
 * kernel writes k[t], v[t] into the cache row slot_mapping[t] of a cache laid
 * out [num_blocks, block_size, num_kv_heads, head_dim], and returns at once
 * for slot -1) and the nano-vllm KV-cache post (§3.1: the per-layer k_cache /
 * v_cache views of the single preallocated pool).
 *
 *   k, v          [num_tokens, num_kv_heads, head_dim] bf16
 *   slot_mapping  [num_tokens] int32; -1 = padding row, nothing written
 *   k_cache,
 *   v_cache       [num_blocks, block_size, num_kv_heads, head_dim] bf16
 * The result is a bit copy.  Two rows with the same slot (other than -1) in
 * one call are not allowed; which one lands is unspecified.
 * A slot outside [-1, num_blocks*block_size) is skipped and sets
 * PKV_ERR_SLOT_RANGE.  head_dim * num_kv_heads * 2 bytes must be a multiple
 * of 16.  num_tokens == 0 is a no-op.
 */
PKV_API pkv_status pkv_kv_store(const uint16_t *k, const uint16_t *v, const int32_t *slot_mapping,
                        int32_t num_tokens, uint16_t *k_cache, uint16_t *v_cache,
                        int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                        int32_t head_dim, int32_t *err_word, pkv_stream_t stream);

/*
 * pkv_decode_store -- a decode step's store in one launch: the slot of each
 * sequence's new token (pkv_decode_slot_mapping) and the store of its K and V
 * rows there (pkv_kv_store), fused.
 *
 * Row b of k and v (one new token per sequence) goes to the slot of position
 * context_lens[b] - 1: block_tables[b][pos / block_size] * block_size +
 * pos % block_size (nano-vLLM lab manual §5.2.3, nano-vllm KV-cache post §4.4;
 * store as in the MinivLLM review, "注意力内核的三个分支").  A sequence with
 * context_lens[b] == 0 is a padding row: nothing is written.
 *
 *   k, v          [num_seqs, num_kv_heads, head_dim] bf16
 *   block_tables  [num_seqs, max_blocks_per_seq] int32; context_lens [num_seqs]
 *   k_cache,
 *   v_cache       [num_blocks, block_size, num_kv_heads, head_dim] bf16
 *   slot_mapping  may be NULL; else [num_seqs] int32 receives the slots (-1
 *                 for padding rows and rejected ones)
 * Errors as the two calls it fuses (PKV_ERR_CONTEXT_RANGE, PKV_ERR_BLOCK_RANGE;
 * the row is then skipped).  block_size a power of two; head_dim *
 * num_kv_heads * 2 bytes a multiple of 16.
 */
PKV_API pkv_status pkv_decode_store(const uint16_t *k, const uint16_t *v, const int32_t *block_tables,
                                    int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs,
                                    uint16_t *k_cache, uint16_t *v_cache, int32_t num_blocks,
                                    int32_t block_size, int32_t num_kv_heads, int32_t head_dim,
                                    int32_t *slot_mapping, int32_t *err_word, pkv_stream_t stream);

/*
 * Bytes of device workspace that pkv_paged_decode needs for these sizes
 * (split-K partial states, one arrival counter per (sequence, kv head), and a
 * small load-balance record).  Depends only on the arguments; 0 means the
 * sizes are invalid.  Context lengths and the block size do not enter: the
 * kernel runs one persistent CTA per SM (at most 512 slices of the work
 * list), and a slice leaves at most two partial states per kv head, so the
 * partial states are bounded by the slice count and the batch, whatever the
 * lengths.  The workspace must be zero-filled (cudaMemset) once
 * before its first use; from then on the library keeps it consistent, for
 * any sizes of later calls.  Calls with up to 16384 arrival counters
 * (num_seqs * num_kv_heads) keep them in a region no other data ever uses;
 * larger calls clear theirs with a cudaMemsetAsync on the stream before the
 * launch.  Its control block carries a call epoch that the
 * last CTA of every call advances on the device, so nothing per call is
 * baked into the launch and a captured CUDA graph may replay a call any
 * number of times; the per-(sequence, kv head) arrival counters return to
 * zero when a call completes; per-SM speed estimates size each SM's share of
 * the next call (speed only, never results).  A control block that is not in
 * a state the library left (not zero-filled before first use, overwritten)
 * sets PKV_ERR_WORKSPACE.  Calls that may run at the same time need separate
 * workspaces; reusing one workspace for consecutive calls on a stream lets
 * the estimates settle.
 */
PKV_API size_t pkv_paged_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                       int32_t num_kv_heads, int32_t head_dim);

/* Upper limits of pkv_paged_decode (beyond them: PKV_EBOUNDS). */
#define PKV_MAX_SEQS 16384
#define PKV_MAX_WORKERS 4096

/*
 * pkv_paged_decode -- decode-phase PagedAttention (one query token per
 * sequence, grouped-query attention).
 *
 * Defined by the mini-vLLM README (§5 "Triton PagedAttention Decode Kernel":
 * the kernel walks each sequence's physical blocks through its block table,
 * kv_head = q_head / (num_q_heads / num_kv_heads), bf16 storage with fp32
 * accumulation, online softmax with running max m, sum l and weighted sum
 * acc) and the MinivLLM review (section "注意力内核的三个分支": the block
 * table is looked up per token, block_tables[b, t / block_size], slot
 * t % block_size).  For sequence b, query head h and L = context_lens[b]:
 *     out[b, h] = sum_{j<L} softmax_j(scale * q[b, h] . K_j) * V_j
 * where K_j, V_j are row j % block_size of physical block
 * block_tables[b][j / block_size], kv head h / (num_q_heads / num_kv_heads).
 * L == 0 gives out[b, h] = 0.  scale is the final multiplier (pass
 * 1/sqrt(head_dim) for standard attention).
 *
 *   q             [num_seqs, num_q_heads, head_dim] bf16
 *   k_cache,
 *   v_cache       [num_blocks, block_size, num_kv_heads, head_dim] bf16
 *   block_tables  [num_seqs, max_blocks_per_seq] int32 (-1 padded; only the
 *                 first ceil(L / block_size) entries of a row are read)
 *   context_lens  [num_seqs] int32
 *   max_context_len  host-side upper bound of context_lens (no device->host
 *                 read is made); lengths above it are a device error
 *   out           [num_seqs, num_q_heads, head_dim] bf16, rounded to nearest
 *   workspace     device buffer of at least
 *                 pkv_paged_decode_workspace_size(...) bytes, 16-byte aligned
 *   num_workers   0 (the default): one CTA per SM; each SM takes a
 *                 contiguous share of the work sized by the speed it showed
 *                 in earlier calls on this workspace -- or, when the call
 *                 has fewer units (bounded with max_context_len) than the
 *                 GPU has SMs, one CTA per unit.  Otherwise a fixed, even
 *                 split over about num_workers consumer warps (CTAs of 8
 *                 warps), 1..PKV_MAX_WORKERS.  A tuning control, and the
 *                 way to reproducible results: with a fixed split the
 *                 partial states and their merge order depend only on the
 *                 inputs, so two calls on the same inputs give bit-identical
 *                 outputs.  The default split moves with the measured SM
 *                 speeds, and with it the rounding of the split-K merge
 *                 (outputs may differ in their last bits from call to call).
 * Supported: head_dim in {64, 128}; num_q_heads / num_kv_heads in 1..16
 * (bf16 caches; 1..8 for E4M3 caches);
 * block_size a power of two in [8, 1024]; num_seqs <= PKV_MAX_SEQS;
 * num_blocks * block_size < 2^31.
 * The work list is (sequence, kv-head group, 16 to 256-token unit); each
 * CTA takes a contiguous range of it, so one sequence may be spread over
 * several CTAs; their partial softmax states are merged in the same kernel
 * by the CTA that completes the sequence's count (split-K /
 * flash-decoding).  Each kernel is launched with programmatic stream
 * serialization and waits on the device for the previous kernel in the stream
 * before it reads any input.
 */
PKV_API pkv_status pkv_paged_decode(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                            const int32_t *block_tables, int32_t max_blocks_per_seq,
                            const int32_t *context_lens, int32_t num_seqs,
                            int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                            int32_t block_size, int32_t num_blocks, int32_t max_context_len,
                            float scale, uint16_t *out, void *workspace, size_t workspace_bytes,
                            int32_t num_workers, int32_t *err_word, pkv_stream_t stream);

/*
 * pkv_paged_decode_store -- a decode step's store and attention in one
 * launch: pkv_decode_store followed by pkv_paged_decode, with the same
 * results (cache bit for bit, outputs within the decode tolerance).
 *
 * Row b of k_new and v_new ([num_seqs, num_kv_heads, head_dim] bf16, 16-byte
 * aligned) is the K and V of sequence b's token at position
 * context_lens[b] - 1 (already counted in context_lens): it is written to
 * that position's cache row (block_tables[b][pos / block_size] * block_size +
 * pos % block_size), and the attention uses it.  slot_mapping may be NULL;
 * else [num_seqs] int32 receives the rows written (-1 for padding rows,
 * rejected lengths and rejected block ids).  The block holding a sequence's
 * new token must not be shared with another sequence of the call (copy-on-
 * write gives every sequence its own last block).  Other arguments, limits
 * and errors as pkv_paged_decode; PKV_ERR_BLOCK_RANGE also covers the new
 * token's block (nothing stored then).
 */
PKV_API pkv_status pkv_paged_decode_store(const uint16_t *q, const uint16_t *k_new, const uint16_t *v_new,
                                          uint16_t *k_cache, uint16_t *v_cache, const int32_t *block_tables,
                                          int32_t max_blocks_per_seq, const int32_t *context_lens,
                                          int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                          int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                          int32_t max_context_len, float scale, uint16_t *out,
                                          int32_t *slot_mapping, void *workspace, size_t workspace_bytes,
                                          int32_t num_workers, int32_t *err_word, pkv_stream_t stream);

/*
 * pkv_paged_decode_noalloc -- pkv_paged_decode for callers that cannot
 * allocate device memory.  (The pages have no counterpart of this call; it
 * exists for callers of this library.)
 *
 * Who needs it: an engine that handed (nearly) all free device memory to its
 * KV block pool at start-up and has nothing left for a workspace, or a host
 * framework whose plugin interface passes only inputs and outputs and forbids
 * device allocations while it runs.  This call takes the same arguments as
 * pkv_paged_decode minus the workspace and computes the same result; its
 * scratch is a fixed array of PKV_NOALLOC_SCRATCH_BYTES inside the library,
 * which every device that loads the library holds until the process exits.
 * It allocates nothing (no cudaMalloc, cudaFree or allocating library call).
 *
 *   - Sizes whose workspace (pkv_paged_decode_workspace_size) exceeds
 *     PKV_NOALLOC_SCRATCH_BYTES are rejected with PKV_EWORKSPACE before any
 *     device work; everything else is validated as in pkv_paged_decode.
 *   - The array is loaded on a device, and its device memory taken, by the
 *     first call of this entry point on that device, which also looks up its
 *     device address (once, with that device current).  A call with
 *     num_seqs == 0 does just that and launches nothing: make it, on each
 *     device, before the caller hands the device's free memory to its KV
 *     pool, and before any stream capture.  Callers of the other entry points
 *     never load the array.
 *   - Every call on a device shares the one array, and the array keeps
 *     whatever the last call left in it.  Nothing in it needs to start at
 *     zero: its call epoch and balance record stay valid from call to call,
 *     and the arrival counters sit in a region no other data uses (or, for
 *     calls with more than 16384 of them, are cleared on the stream before
 *     the launch).  Calls that overlap on the GPU -- on different streams,
 *     or from different threads -- race on it: serialise them.
 */
#define PKV_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)

PKV_API pkv_status pkv_paged_decode_noalloc(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                                    const int32_t *block_tables, int32_t max_blocks_per_seq,
                                    const int32_t *context_lens, int32_t num_seqs,
                                    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                    int32_t block_size, int32_t num_blocks, int32_t max_context_len,
                                    float scale, uint16_t *out, int32_t num_workers,
                                    int32_t *err_word, pkv_stream_t stream);

/*
 * pkv_paged_attention -- paged attention for several new tokens per sequence:
 * a chunk of a prefill over a cached prefix, or a batch that mixes prefill
 * chunks with decode steps (one new token).
 *
 * The nano-vllm KV-cache post (§3.5) builds the slots of such a chunk and the
 * mini-vLLM README names the prefill over a cached prefix as the next step.
 * Sequence b holds L = context_lens[b] tokens in the cache (the chunk's K/V
 * already stored there, pkv_kv_store), the last n = cu_seqlens_q[b+1] -
 * cu_seqlens_q[b] of them new; query row r = cu_seqlens_q[b] + i (i < n) sits
 * at position L - n + i and attends causally the keys j <= L - n + i:
 *     out[r, h] = sum_{j<=p} softmax_j(scale * q[r, h] . K_j) V_j,  p = L - n + i,
 * K_j, V_j read through sequence b's block table row as in pkv_paged_decode.
 *
 *   q, out        [num_rows, num_q_heads, head_dim] bf16, num_rows =
 *                 cu_seqlens_q[num_seqs] (the host-known row count)
 *   cu_seqlens_q  [num_seqs + 1] int32, device, non-decreasing from 0
 *   context_lens  [num_seqs] int32, device: cached tokens per sequence,
 *                 new ones included
 *   workspace     pkv_paged_attention_workspace_size(num_rows, ...) bytes,
 *                 zero-filled before first use (as pkv_paged_decode's)
 *   new_per_seq   0: the offsets cu_seqlens_q say how many new tokens each
 *                 sequence has.  n > 0: every sequence has exactly n
 *                 (rows b * n .. b * n + n - 1, num_rows = num_seqs * n;
 *                 cu_seqlens_q may be NULL) -- a speculative-decoding verify
 *                 step, say.
 * Consecutive queries of a sequence share passes over its keys: with
 * G = num_q_heads / num_kv_heads and q = max(1, 16 / G), chunks of Q
 * queries (the last one of a sequence possibly shorter) each read the keys
 * the chunk's last query sees once for all its Q * G (query, head) pairs,
 * every query keeping its own causal bound; Q = q when the call has at most
 * 2q new tokens per sequence on average, else Q = 8q (64 at G = 2).  A
 * sequence of n new tokens over L cached ones so streams about (n / Q) * L
 * key rows, not n * L.  With new_per_seq = n <= q, each sequence is one such
 * pass without the expansion kernel.
 * Rows inconsistent with the offsets (n > L, rows outside every sequence's
 * range) give zeros and PKV_ERR_CONTEXT_RANGE.  num_rows <= PKV_MAX_SEQS;
 * other limits, num_workers and errors as pkv_paged_decode.
 */
PKV_API size_t pkv_paged_attention_workspace_size(int32_t num_rows, int32_t num_q_heads,
                                                  int32_t num_kv_heads, int32_t head_dim);
PKV_API pkv_status pkv_paged_attention(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                                       const int32_t *block_tables, int32_t max_blocks_per_seq,
                                       const int32_t *cu_seqlens_q, const int32_t *context_lens,
                                       int32_t num_seqs, int32_t num_rows, int32_t num_q_heads,
                                       int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                       int32_t num_blocks, int32_t max_context_len, float scale,
                                       uint16_t *out, int32_t new_per_seq, void *workspace,
                                       size_t workspace_bytes, int32_t num_workers, int32_t *err_word,
                                       pkv_stream_t stream);

/*
 * E4M3 (fp8) KV cache.  The mini-vLLM README lists "no FP8 KV" among its gaps
 * to production vLLM (§ "与 production vLLM 的关键差距") and gives no format;
 * this library stores the OCP 8-bit floating point E4M3 encoding
 * ("float8_e4m3fn": sign, 4 exponent bits with bias 7, 3 mantissa bits,
 * largest finite 448, no infinities, 0x7F / 0xFF NaN) with one scale per kv
 * head for K and one for V, both caller-chosen device float32 arrays
 * [num_kv_heads] (for example a calibrated max |x| / 448): an element x is
 * stored as the code of x / scale and read back as value(code) * scale.
 * Caches hold one byte per element: [num_blocks, block_size, num_kv_heads,
 * head_dim] uint8, half the bytes of the bf16 layout.
 *
 * pkv_kv_store_fp8 -- pkv_kv_store into E4M3 caches: row slot_mapping[t]
 * becomes the codes of k[t] / k_scale (per kv head) -- one IEEE binary32
 * division of the bf16 value, then round to nearest even, saturating at
 * +-448 (NaN stays NaN).  Slot -1 and range errors as pkv_kv_store;
 * head_dim must be a multiple of 8.
 */
PKV_API pkv_status pkv_kv_store_fp8(const uint16_t *k, const uint16_t *v, const int32_t *slot_mapping,
                                    int32_t num_tokens, uint8_t *k_cache, uint8_t *v_cache,
                                    int32_t num_blocks, int32_t block_size, int32_t num_kv_heads,
                                    int32_t head_dim, const float *k_scale, const float *v_scale,
                                    int32_t *err_word, pkv_stream_t stream);

/*
 * pkv_paged_decode_fp8 -- pkv_paged_decode over E4M3 caches: K_j and V_j are
 * the codes' values times k_scale / v_scale of their kv head; everything else
 * (shapes, workspace, num_workers, errors, supported sizes) as
 * pkv_paged_decode.  The K scale is folded into the query prescale and the V
 * scale into the final division (both exact up to fp32 rounding), so the
 * inner loop reads one byte per element.
 */
PKV_API pkv_status pkv_paged_decode_fp8(const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                                        const float *k_scale, const float *v_scale,
                                        const int32_t *block_tables, int32_t max_blocks_per_seq,
                                        const int32_t *context_lens, int32_t num_seqs,
                                        int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                        int32_t block_size, int32_t num_blocks, int32_t max_context_len,
                                        float scale, uint16_t *out, void *workspace, size_t workspace_bytes,
                                        int32_t num_workers, int32_t *err_word, pkv_stream_t stream);

/*
 * pkv_paged_decode_store_fp8 -- pkv_paged_decode_store over E4M3 caches:
 * row b of k_new / v_new (bf16, [num_seqs, num_kv_heads, head_dim], 16-byte
 * aligned) is quantised exactly as pkv_kv_store_fp8 does (the E4M3 code of
 * x / scale[kv head]), stored at position context_lens[b] - 1 and attended
 * over with the other codes (as pkv_paged_decode_fp8).  Same result as
 * pkv_decode_slot_mapping + pkv_kv_store_fp8 + pkv_paged_decode_fp8;
 * arguments, slot_mapping and errors as pkv_paged_decode_store.
 */
PKV_API pkv_status pkv_paged_decode_store_fp8(const uint16_t *q, const uint16_t *k_new, const uint16_t *v_new,
                                              uint8_t *k_cache, uint8_t *v_cache, const float *k_scale,
                                              const float *v_scale, const int32_t *block_tables,
                                              int32_t max_blocks_per_seq, const int32_t *context_lens,
                                              int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                              int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                              int32_t max_context_len, float scale, uint16_t *out,
                                              int32_t *slot_mapping, void *workspace, size_t workspace_bytes,
                                              int32_t num_workers, int32_t *err_word, pkv_stream_t stream);

/*
 * pkv_copy_blocks -- batched copy-on-write block copies.
 *
 * Defined by the nano-vllm KV-cache post (§2.2: sequences that share a
 * physical block keep sharing it until one of them writes a different token
 * there; that write first copies the block to a new one) and the mini-vLLM
 * README (§1: copy-on-write of a half-full shared block).  For every pair i,
 * physical block dst = pairs[2i + 1] of k_cache and of v_cache becomes a bit
 * copy of block src = pairs[2i] (block_size rows x num_kv_heads x head_dim
 * bf16 values each); src == dst leaves the block as it is.
 *
 *   k_cache,
 *   v_cache   [num_blocks, block_size, num_kv_heads, head_dim] bf16, device
 *   pairs     [num_pairs][2] int32 (src, dst), device
 * The dst blocks of one call must be distinct and must not be the src of
 * another pair of the same call (the copies run concurrently); a pair with an
 * id outside [0, num_blocks) is skipped and sets PKV_ERR_BLOCK_RANGE.
 * block_size * num_kv_heads * head_dim * 2 must be a multiple of 16 bytes.
 * Memory-bound: it reads and writes 2 * block bytes per pair.
 */
PKV_API pkv_status pkv_copy_blocks(uint16_t *k_cache, uint16_t *v_cache, const int32_t *pairs,
                                   int32_t num_pairs, int32_t num_blocks, int32_t block_size,
                                   int32_t num_kv_heads, int32_t head_dim, int32_t *err_word,
                                   pkv_stream_t stream);

/*
 * Host-side block allocator: which physical blocks hold each sequence's
 * tokens, with reference counts for shared blocks (the nano-vllm KV-cache
 * post, §3.3 "BlockManager 的设计").  The free list is a FIFO of block ids,
 * initially 0, 1, ..., num_blocks - 1: allocation takes from the front,
 * release appends to the back (§3.3.1).  A block's reference count is the
 * number of sequences whose table holds it.  Which blocks may be shared
 * (prefix hashing in the post, §3.4) is the caller's decision: sharing is
 * explicit.  Not thread-safe: one allocator per host thread, or a lock.
 * Sequence ids are any int32 >= 0 not in use.  On any error the allocator is
 * left as it was.
 */
typedef struct pkv_block_allocator pkv_block_allocator;

/* A pool of num_blocks blocks of block_size tokens.  NULL on bad sizes. */
PKV_API pkv_block_allocator *pkv_allocator_create(int32_t num_blocks, int32_t block_size);
PKV_API void pkv_allocator_destroy(pkv_block_allocator *a);

/* A new sequence of num_tokens tokens (its prefill): its first shared_blocks
 * blocks are the first shared_blocks blocks of sequence parent_id (each one's
 * count + 1, the post's REUSE path, §3.3.3), the rest are fresh blocks from
 * the front of the free list.  Shared blocks must be whole blocks the parent
 * holds and must not include the block of the sequence's last token
 * (shared_blocks * block_size < num_tokens).  PKV_EFULL if the free list is
 * too short; PKV_EINVAL for an id in use, an unknown parent or a bad count. */
PKV_API pkv_status pkv_allocator_add(pkv_block_allocator *a, int32_t seq_id, int32_t num_tokens,
                                     int32_t parent_id, int32_t shared_blocks);

/* child_id becomes a copy of parent_id: the same tokens and table, every
 * block's count + 1 (parallel sampling, beam search: §2.2 of the post). */
PKV_API pkv_status pkv_allocator_fork(pkv_block_allocator *a, int32_t parent_id, int32_t child_id);

/* One decode step of seq_id: its new token goes to position p = its token
 * count.  If p % block_size == 0 the token opens a fresh block (the post's
 * may_append, §3.3.4).  Otherwise, if its last block is shared (count > 1),
 * copy-on-write: a fresh block replaces it in this sequence's table, the old
 * block's count drops by one, and (*cow_src, *cow_dst) name the copy that
 * pkv_copy_blocks must make before the token is stored; else both are -1.
 * cow_src / cow_dst may be NULL.  PKV_EFULL if a block is needed and none
 * is free. */
PKV_API pkv_status pkv_allocator_append(pkv_block_allocator *a, int32_t seq_id, int32_t *cow_src,
                                        int32_t *cow_dst);

/* The sequence ends (or is preempted): its table is walked backwards and
 * every block's count drops by one; a block at zero goes to the back of the
 * free list (§3.3.5). */
PKV_API pkv_status pkv_allocator_free(pkv_block_allocator *a, int32_t seq_id);

/* Free blocks; a block's count (-1 for a bad id); a sequence's tokens (-1 if unknown). */
PKV_API int32_t pkv_allocator_num_free(const pkv_block_allocator *a);
PKV_API int32_t pkv_allocator_ref_count(const pkv_block_allocator *a, int32_t block_id);
PKV_API int32_t pkv_allocator_num_tokens(const pkv_block_allocator *a, int32_t seq_id);

/* Decode inputs for a batch, in host memory: row i of block_tables
 * [n][max_blocks] is the table of seq_ids[i], -1 padded; context_lens[i]
 * (may be NULL) its token count.  PKV_EINVAL if a sequence is unknown,
 * PKV_EBOUNDS if one holds more than max_blocks blocks (nothing is written
 * then). */
PKV_API pkv_status pkv_allocator_tables(const pkv_block_allocator *a, const int32_t *seq_ids, int32_t n,
                                        int32_t *block_tables, int32_t max_blocks, int32_t *context_lens);

/* ------------------------------------------------------------------------
 * Diagnostics.  Not part of the paged-KV operations; they exercise the
 * library's failure paths without a GPU fault.
 * ------------------------------------------------------------------------ */

/*
 * pkv_diag_wait_timeout -- one warp waits on a barrier that nothing completes.
 * Every wait on an asynchronous copy in the library is bounded (about 2 s);
 * this one runs out, sets PKV_ERR_WAIT_TIMEOUT in *err_word (device) and
 * returns, leaving the context usable.  It takes the wait's time limit to
 * complete.  err_word NULL: PKV_EINVAL.
 */
PKV_API pkv_status pkv_diag_wait_timeout(int32_t *err_word, pkv_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
