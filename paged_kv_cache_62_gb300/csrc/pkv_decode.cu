// Decode-phase PagedAttention entry points (include/pkv.h): argument checks,
// the launch of the bf16-cache kernels (the kernel itself is in
// pkv_decode_kernel.cuh) and the workspace size.
#include "pkv_decode_kernel.cuh"

using namespace pkv;

extern "C" size_t pkv_paged_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                                  int32_t head_dim)
{
    if (num_seqs < 0 || num_seqs > PKV_MAX_SEQS || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        num_q_heads % num_kv_heads != 0)
        return 0;
    return ws_layout(num_seqs, num_q_heads / num_kv_heads, num_kv_heads, head_dim).total;
}

// Shared by the bf16 and the E4M3 entry points (k_scale / v_scale: the
// latter's per-kv-head scales, device arrays).  qn > 1: entry b holds up to qn
// queries that share its K/V stream as qn * G virtual heads of a kv head --
// with row_cnt null, every entry is a sequence with qn new tokens (q / out rows
// b * qn + i; context_lens the sequences' whole lengths); otherwise entry b
// holds row_cnt[b] queries at rows b + i (row_seq[b]: its sequence,
// context_lens[b]: the length its last query sees).
static pkv_status decode_call(bool fp8, bool qs, int32_t qn, const uint16_t *q, const void *k_cache, const void *v_cache,
                              const float *k_scale, const float *v_scale, const int32_t *row_seq,
                              const int32_t *row_cnt, const int32_t *block_tables,
                              int32_t max_blocks_per_seq, const int32_t *context_lens, int32_t num_seqs,
                              int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                              int32_t num_blocks, int32_t max_context_len, float scale, uint16_t *out,
                              void *workspace, size_t workspace_bytes, int32_t num_workers, int32_t *err_word,
                              pkv_stream_t stream, const uint16_t *k_new = nullptr, const uint16_t *v_new = nullptr,
                              int32_t *slot_out = nullptr)
{
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 ||
        head_dim <= 0 || block_size <= 0 || num_blocks <= 0 || max_blocks_per_seq <= 0 || max_context_len < 0 ||
        num_workers < 0 || !std::isfinite(scale))
        return PKV_EINVAL;
    if (num_seqs > PKV_MAX_SEQS || num_workers > PKV_MAX_WORKERS) return PKV_EBOUNDS;
    if (head_dim != 64 && head_dim != 128) return PKV_EUNSUPPORTED;
    if (qn < 1) return PKV_EINVAL;
    const int gq = num_q_heads / num_kv_heads;  // query heads per kv head
    const int G = gq * qn;                      // virtual heads per kv head sharing one K/V stream
    if (G > (fp8 ? 8 : 16)) return PKV_EUNSUPPORTED;  // virtual heads per warp: the MMA tile's rows
    if (!is_pow2(block_size) || block_size < 8 || block_size > 1024) return PKV_EUNSUPPORTED;
    if (int64_t(num_blocks) * block_size > INT32_MAX) return PKV_EBOUNDS;
    if (num_seqs == 0) return PKV_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out) return PKV_EINVAL;
    if (fp8 && (!k_scale || !v_scale)) return PKV_EINVAL;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out)) return PKV_EINVAL;
    const int64_t len_limit = std::min<int64_t>(max_context_len, int64_t(max_blocks_per_seq) * block_size);
    // unit counts (and positions in the unit list) are kept in 32 bits
    const int64_t max_units = int64_t(num_kv_heads) * num_seqs * ((len_limit + 7) / 8);
    if (max_units > INT32_MAX) return PKV_EBOUNDS;
    if (qs && (fp8 || !row_cnt)) return PKV_EINVAL;  // query-split entries are chunks of bf16 calls
    if ((k_new || v_new) && (qs || qn != 1 || row_seq || !k_new || !v_new || !aligned16(k_new) ||
                             !aligned16(v_new)))
        return PKV_EINVAL;  // the fused store goes with a decode
    const WsLayout ws = ws_layout(num_seqs, G, num_kv_heads, head_dim, qs);
    if (!workspace || workspace_bytes < ws.total || !aligned16(workspace)) return PKV_EWORKSPACE;

    DeviceInfo dev;
    if (!current_device_info(&dev)) return PKV_ECUDA;

    LaunchArgs a{};  // every field starts at zero; those a call uses are set below
    DecodeParams &p = a.p;
    uint8_t *wsb = static_cast<uint8_t *>(workspace);
    p.q = q;
    p.block_tables = block_tables;
    p.context_lens = context_lens;
    p.out = out;
    p.ws_count = reinterpret_cast<unsigned long long *>(wsb + ws.count_off);
    p.ws_bal = reinterpret_cast<BalanceState *>(wsb + ws.bal_off);
    p.ws_ml = reinterpret_cast<float *>(wsb + ws.ml_off);
    p.ws_acc = reinterpret_cast<float *>(wsb + ws.acc_off);
    p.err = err_word;
    p.B = num_seqs;
    p.Hq = num_q_heads;
    p.Hkv = num_kv_heads;
    p.bs = block_size;
    p.log2_bs = ilog2(block_size);
    p.NB = num_blocks;
    p.max_blocks = max_blocks_per_seq;
    p.len_limit = int32_t(len_limit);
    // query-split entries of 128 rows run on the tensor-memory CTAs where they can
    const bool tc5 = qs && !fp8 && tc5_eligible(head_dim, G, gq, block_size, num_seqs, dev.max_smem_optin);
    p.hg = qs ? 1 : head_group(num_kv_heads, G);
    p.nhg = num_kv_heads / p.hg;
    p.sub = qs ? team_warps(G) : warp_slices(G, p.hg);
    p.toks = warp_tokens(G, fp8, qs, tc5) * (qs ? 1 : p.sub);
    p.boxtok = std::min(p.toks, block_size);
    p.nbox = p.toks / p.boxtok;
    p.lg_nbox = ilog2(p.nbox);
    p.cons = tc5 ? kTc5Consumers : p.hg * p.sub;
    p.nst = 2;
    p.num_workers = 0;
    p.per_segment = 0;
    p.scale_log2 = float(double(scale) * 1.4426950408889634);
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.row_seq = row_seq;
    p.qn = qn;
    p.gq = gq;
    p.row_cnt = row_cnt;
    p.k_new = k_new;
    p.v_new = v_new;
    p.k_cache_w = static_cast<uint8_t *>(const_cast<void *>(k_cache));
    p.v_cache_w = static_cast<uint8_t *>(const_cast<void *>(v_cache));
    p.slot_out = k_new ? slot_out : nullptr;
    p.qstride = row_cnt ? 1 : qn;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.device = dev.device;
    a.sm_count = dev.sm_count;
    a.max_smem = dev.max_smem_optin;
    a.requested_workers = num_workers;
    // A call with fewer units than SMs (bounded from the host-known lengths) runs one CTA per unit
    // with the fixed split: the CTAs without work would only add set-up and contention
    // (tiny and Qwen2.5-shaped batches: 9.2 -> 7.9 and 17.9 -> 14.1 us per graph-replayed call).
    // Regular CTAs with at most kSegmentUnits units per (entry, head group) run one CTA per segment
    // instead: a few units in one CTA's pipeline cost less than the split-K pieces and merge of a
    // split (per back-to-back call: tiny workload 8.3 -> 7.0 us, Qwen2.5-shaped 14.2 -> 9.0 us).
    if (num_workers == 0) {
        const int64_t per_seg = (len_limit + p.toks - 1) / p.toks;
        const int64_t units_max = int64_t(num_seqs) * p.nhg * per_seg;
        if (units_max < dev.sm_count) {
            if (!qs && per_seg <= kSegmentUnits && int64_t(num_seqs) * p.nhg <= kMaxSlots) {
                p.per_segment = 1;
                a.requested_workers = num_seqs * p.nhg * p.cons;
            } else {
                a.requested_workers = int32_t(std::max<int64_t>(1, units_max)) * p.cons;
            }
        }
    }
    a.stream = reinterpret_cast<cudaStream_t>(stream);

    LaunchFn fn = fp8    ? pick_decode_fp8(head_dim, G)
                  : tc5  ? pick_decode_tc5(head_dim)
                  : qs   ? pick_decode_qs(head_dim, G)
                  : G > 8 ? pick_decode_wide(head_dim, G)
                         : (head_dim == 64 ? pick_group<64, false, false>(G) : pick_group<128, false, false>(G));
    if (!fn) return PKV_EUNSUPPORTED;
    if (ws.count_clear) {  // counters outside the fixed region start at zero (see WsLayout)
        const cudaError_t ce = cudaMemsetAsync(p.ws_count, 0, ws.count_bytes, a.stream);
        if (ce != cudaSuccess) {
            cudaGetLastError();
            return cuda_fail("cudaMemsetAsync (arrival counters)", ce);
        }
    }
    return fn(a);
}

extern "C" pkv_status pkv_paged_decode(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                                       const int32_t *block_tables, int32_t max_blocks_per_seq,
                                       const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                                       int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                       int32_t num_blocks, int32_t max_context_len, float scale, uint16_t *out,
                                       void *workspace, size_t workspace_bytes, int32_t num_workers,
                                       int32_t *err_word, pkv_stream_t stream)
{
    return decode_call(false, false, 1, q, k_cache, v_cache, nullptr, nullptr, nullptr, nullptr, block_tables,
                       max_blocks_per_seq, context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                       num_blocks, max_context_len, scale, out, workspace, workspace_bytes, num_workers, err_word,
                       stream);
}

extern "C" pkv_status pkv_paged_decode_store(const uint16_t *q, const uint16_t *k_new, const uint16_t *v_new,
                                             uint16_t *k_cache, uint16_t *v_cache, const int32_t *block_tables,
                                             int32_t max_blocks_per_seq, const int32_t *context_lens,
                                             int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                             int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                             int32_t max_context_len, float scale, uint16_t *out,
                                             int32_t *slot_mapping, void *workspace, size_t workspace_bytes,
                                             int32_t num_workers, int32_t *err_word, pkv_stream_t stream)
{
    if (num_seqs > 0 && (!k_new || !v_new)) return PKV_EINVAL;
    return decode_call(false, false, 1, q, k_cache, v_cache, nullptr, nullptr, nullptr, nullptr, block_tables,
                       max_blocks_per_seq, context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                       num_blocks, max_context_len, scale, out, workspace, workspace_bytes, num_workers, err_word,
                       stream, k_new, v_new, slot_mapping);
}

extern "C" pkv_status pkv_paged_decode_store_fp8(const uint16_t *q, const uint16_t *k_new, const uint16_t *v_new,
                                                 uint8_t *k_cache, uint8_t *v_cache, const float *k_scale,
                                                 const float *v_scale, const int32_t *block_tables,
                                                 int32_t max_blocks_per_seq, const int32_t *context_lens,
                                                 int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                                 int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                                 int32_t max_context_len, float scale, uint16_t *out,
                                                 int32_t *slot_mapping, void *workspace, size_t workspace_bytes,
                                                 int32_t num_workers, int32_t *err_word, pkv_stream_t stream)
{
    if (num_seqs > 0 && (!k_new || !v_new)) return PKV_EINVAL;
    return decode_call(true, false, 1, q, k_cache, v_cache, k_scale, v_scale, nullptr, nullptr, block_tables,
                       max_blocks_per_seq, context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                       num_blocks, max_context_len, scale, out, workspace, workspace_bytes, num_workers, err_word,
                       stream, k_new, v_new, slot_mapping);
}

extern "C" pkv_status pkv_paged_decode_fp8(const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                                           const float *k_scale, const float *v_scale, const int32_t *block_tables,
                                           int32_t max_blocks_per_seq, const int32_t *context_lens,
                                           int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                           int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                           int32_t max_context_len, float scale, uint16_t *out, void *workspace,
                                           size_t workspace_bytes, int32_t num_workers, int32_t *err_word,
                                           pkv_stream_t stream)
{
    return decode_call(true, false, 1, q, k_cache, v_cache, k_scale, v_scale, nullptr, nullptr, block_tables,
                       max_blocks_per_seq, context_lens,
                       num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, max_context_len, scale,
                       out, workspace, workspace_bytes, num_workers, err_word, stream);
}

// ------------------------------------------------------------------ several query rows per sequence
namespace pkv {

// Query row r = cu_seqlens_q[b] + i of sequence b (n = cu_seqlens_q[b+1] -
// cu_seqlens_q[b] new tokens, L = context_lens[b] in the cache) sits at
// position L - n + i: it sees the L - n + i + 1 keys before it.  The rows of
// a sequence are cut into chunks of up to `chunk` consecutive queries that share
// one K/V stream; a chunk is entry r of the decode kernel, r the row of its
// first query: row_seq[r] = b, row_cnt[r] = its query count, row_len[r] = the
// keys its last query sees.  Rows that start no chunk get row_cnt = 0 and
// row_len = 0 (no work, no output).  One thread per row finds its sequence by
// binary search over cu_seqlens_q, so every row gets a sequence in
// [0, num_seqs) even when the offsets are inconsistent; such rows (not inside
// their sequence's range, n > L, offsets not starting at 0) are entries of
// their own or their chunk's with length 0 (zero output) and set
// PKV_ERR_CONTEXT_RANGE.  With cu_seqlens_q null, every sequence has
// new_per_seq rows (row r belongs to sequence r / new_per_seq).
__global__ void expand_rows_kernel(const int32_t *__restrict__ cu_seqlens_q, int32_t new_per_seq,
                                   const int32_t *__restrict__ context_lens, int32_t num_seqs, int32_t num_rows,
                                   int32_t chunk, int32_t *__restrict__ row_seq, int32_t *__restrict__ row_len,
                                   int32_t *__restrict__ row_cnt, int32_t *err)
{
    griddep_launch_dependents();
    griddep_wait();
    const int32_t r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= num_rows) return;
    int32_t lo = 0, r0 = 0, r1 = 0;
    if (cu_seqlens_q) {
        int32_t hi = num_seqs;  // the last b with cu_seqlens_q[b] <= r
        while (hi - lo > 1) {
            const int32_t mid = (lo + hi) >> 1;
            if (__ldg(cu_seqlens_q + mid) <= r)
                lo = mid;
            else
                hi = mid;
        }
        r0 = __ldg(cu_seqlens_q + lo);
        r1 = __ldg(cu_seqlens_q + lo + 1);
    } else {
        lo = min(r / new_per_seq, num_seqs - 1);
        r0 = lo * new_per_seq;
        r1 = r0 + new_per_seq;
    }
    const int32_t L = __ldg(context_lens + lo);
    const int32_t n = r1 - r0, i = r - r0;
    const bool inside = r0 <= r && r < r1;
    const bool ok = (!cu_seqlens_q || __ldg(cu_seqlens_q) == 0) && inside && n <= L && r1 <= num_rows;
    if (!ok) flag_error(err, PKV_ERR_CONTEXT_RANGE);
    int32_t cnt = 1, len = 0;  // a row outside its sequence's range: an entry of its own, zero output
    if (inside) {
        cnt = i % chunk == 0 ? min(min(chunk, n - i), num_rows - r) : 0;  // never past the last row
        len = ok && cnt > 0 ? L - n + i + cnt : 0;
    }
    row_seq[r] = lo;
    row_len[r] = len;
    row_cnt[r] = cnt;
}

inline size_t rows_bytes(int32_t num_rows) { return align256(size_t(num_rows) * 4); }

// Queries per warp: as many as keep its qg * G virtual heads within the rows
// of the MMA tile it uses: 8 for a regular CTA (same-n entries), 16 for a
// query-split one.  A query-split entry holds the queries of all team_warps
// warps of its CTA.
inline int32_t chunk_queries(int32_t num_q_heads, int32_t num_kv_heads, int32_t rows = 8)
{
    return std::max(1, rows / (num_q_heads / num_kv_heads));
}

inline int32_t qs_queries(int32_t num_q_heads, int32_t num_kv_heads)
{
    return chunk_queries(num_q_heads, num_kv_heads, 16);
}

inline int32_t entry_queries(int32_t num_q_heads, int32_t num_kv_heads)
{
    const int32_t qg = qs_queries(num_q_heads, num_kv_heads);
    return qg * team_warps(qg * (num_q_heads / num_kv_heads));
}

}  // namespace pkv

extern "C" size_t pkv_paged_attention_workspace_size(int32_t num_rows, int32_t num_q_heads, int32_t num_kv_heads,
                                                     int32_t head_dim)
{
    const size_t base = pkv_paged_decode_workspace_size(num_rows, num_q_heads, num_kv_heads, head_dim);
    if (base == 0) return 0;
    // decode workspace: same-n calls (entries of n <= qg queries, n * G virtual heads), or one
    // chunk entry per row (qg * G virtual heads a warp, on a regular or a query-split CTA); then the
    // three row arrays
    const int32_t gq = num_q_heads / num_kv_heads, qg = qs_queries(num_q_heads, num_kv_heads);
    size_t dec = std::max(base, ws_layout(num_rows, gq * qg, num_kv_heads, head_dim, true).total);
    for (int32_t qn = 2; qn <= qg; ++qn)
        dec = std::max(dec, ws_layout(num_rows, gq * qn, num_kv_heads, head_dim).total);
    return align256(dec) + 3 * rows_bytes(num_rows);
}

extern "C" pkv_status pkv_paged_attention(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                                          const int32_t *block_tables, int32_t max_blocks_per_seq,
                                          const int32_t *cu_seqlens_q, const int32_t *context_lens, int32_t num_seqs,
                                          int32_t num_rows, int32_t num_q_heads, int32_t num_kv_heads,
                                          int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                          int32_t max_context_len, float scale, uint16_t *out, int32_t new_per_seq,
                                          void *workspace, size_t workspace_bytes, int32_t num_workers,
                                          int32_t *err_word, pkv_stream_t stream)
{
    if (num_seqs < 0 || num_rows < 0 || new_per_seq < 0) return PKV_EINVAL;
    if (num_rows == 0) return PKV_OK;
    if (num_seqs == 0 || !context_lens || (new_per_seq == 0 && !cu_seqlens_q)) return PKV_EINVAL;
    if (new_per_seq > 0 && int64_t(num_seqs) * new_per_seq != num_rows) return PKV_EINVAL;
    if (num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads != 0) return PKV_EINVAL;
    const size_t need = pkv_paged_attention_workspace_size(num_rows, num_q_heads, num_kv_heads, head_dim);
    if (need == 0) return num_rows > PKV_MAX_SEQS ? PKV_EBOUNDS : PKV_EINVAL;
    if (!workspace || workspace_bytes < need || !aligned16(workspace)) return PKV_EWORKSPACE;
    // Up to qg queries of a sequence fit one regular CTA warp's MMA tile (qg * G <= 16 virtual heads):
    // the CTA's warps split the K/V tokens, as in decode.  Longer runs of new tokens go to query-split
    // CTAs, whose warps split an entry of up to 8 * qg queries and share every K/V tile.
    const int32_t qg = qs_queries(num_q_heads, num_kv_heads);
    if (new_per_seq > 1 && new_per_seq <= qg)
        // every sequence's n new tokens share its K/V stream: read once, n * G virtual heads
        return decode_call(false, false, new_per_seq, q, k_cache, v_cache, nullptr, nullptr, nullptr, nullptr,
                           block_tables, max_blocks_per_seq, context_lens, num_seqs, num_q_heads, num_kv_heads,
                           head_dim, block_size, num_blocks, max_context_len, scale, out, workspace,
                           workspace_bytes, num_workers, err_word, stream);
    // chunks of a sequence's queries, one entry per row; few new tokens per sequence on average (at
    // most two regular chunks): chunks of qg on regular CTAs, else chunks of 8 * qg on query-split ones.
    // The row arrays sit after the decode workspace.
    const bool qs = int64_t(num_rows) > 2 * int64_t(qg) * num_seqs;
    const int32_t chunk = qs ? entry_queries(num_q_heads, num_kv_heads) : qg;
    uint8_t *wsb = static_cast<uint8_t *>(workspace);
    const size_t dec_bytes = need - 3 * rows_bytes(num_rows);
    int32_t *row_seq = reinterpret_cast<int32_t *>(wsb + dec_bytes);
    int32_t *row_len = reinterpret_cast<int32_t *>(wsb + dec_bytes + rows_bytes(num_rows));
    int32_t *row_cnt = reinterpret_cast<int32_t *>(wsb + dec_bytes + 2 * rows_bytes(num_rows));
    const cudaError_t e = launch_pdl(expand_rows_kernel, dim3((num_rows + 255) / 256), dim3(256), 0,
                                     reinterpret_cast<cudaStream_t>(stream), new_per_seq > 0 ? nullptr : cu_seqlens_q,
                                     new_per_seq, context_lens, num_seqs, num_rows, chunk, row_seq, row_len,
                                     row_cnt, err_word);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return cuda_fail("expand_rows_kernel launch", e);
    }
    const pkv_status st = launch_status("expand_rows_kernel launch");
    if (st != PKV_OK) return st;
    return decode_call(false, qs, qg, q, k_cache, v_cache, nullptr, nullptr, row_seq, row_cnt, block_tables,
                       max_blocks_per_seq, row_len, num_rows, num_q_heads, num_kv_heads, head_dim, block_size,
                       num_blocks, max_context_len, scale, out, workspace, dec_bytes, num_workers, err_word, stream);
}
