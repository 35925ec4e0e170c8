/*
 * Oracle for the paged KV cache hot path -- TEST INFRASTRUCTURE ONLY.
 *
 * This file is a plain, slow, obviously correct CPU restatement of what the
 * paged KV cache computes, in fp64.  It exists to check the CUDA library
 * against.  Only the test suite, the package smoke check and the CPU-baseline
 * leg of the benchmark may load it; the library itself never does, and it
 * shares no code, header or table with the CUDA sources.
 *
 * Sources (all restated, nothing copied):
 *  [P1] nano-vLLM inference lab manual ("5. 动手改造：从跑通到可测量的推理服务"),
 *       §5.2.1 (context_lens include the position about to be written),
 *       §5.2.3 and appendix B.2.3 (slot = block_table[pos // B] * B + pos % B),
 *       appendix B.1.2 (softmax attention worked example),
 *       appendix B.4 (padding rows carry slot -1 and context_len 0 and must
 *       not write the real cache).
 *  [P2] "mini-vLLM v0.4 -- From-Scratch LLM Inference Serving Runtime",
 *       §5 "Triton PagedAttention Decode Kernel" (q_len = 1 decode, GQA map
 *       kv_head = q_head // (Hq / Hkv), fp16/bf16 storage, fp32 accumulation,
 *       online softmax state m / l / acc).
 *  [P3] "MinivLLM：六步搭出一个 Qwen3 推理引擎", section "注意力内核的三个分支"
 *       (store_kvcache: cache layout [num_blocks, block_size, Hkv, D],
 *       slot -1 skips the row; decode kernel looks up block_tables[b, t // bs]
 *       for every token t, slot t % bs).
 *  [P4] "大模型推理引擎学习入门-2：带你理解 nano-vllm 的 KV Cache 以及 Paged
 *       Attention", §3.1 (slot = block_table[i] * block_size + offset, per-layer
 *       k_cache/v_cache views), §3.5 (slot_mapping), §4.4 (decode example:
 *       context_lens [431, 434] -> slot_mapping [430, 689]), §2.2 (shared
 *       blocks are copied before a divergent write: copy-on-write).
 *
 * Numbers: K/V/q are bf16 bit patterns (uint16), widened exactly to double.
 * Every sum, exp and division is done in double.  The attention uses the
 * plain two-pass softmax (max, then exponentials, then one division); the
 * partial-state functions at the end restate the split-and-merge identity
 * that the online softmax of [P2] §5 relies on.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)
#define ORACLE_EBOUNDS (-5)

/* bf16 -> double: a bf16 value is the top 16 bits of an IEEE binary32. */
static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ---------------------------------------------------------------------------
 * 8-bit floating point E4M3, the "fp8 KV cache" the mini-vLLM README names as
 * missing (§ "与 production vLLM 的关键差距"); the pages give no format, so
 * this is the OCP 8-bit floating point E4M3 encoding that production engines
 * store K/V in ("float8_e4m3fn"): sign bit, 4 exponent bits with bias 7,
 * 3 mantissa bits; exponent field 0 holds subnormals m * 2^-9; no infinities;
 * exponent 15 with mantissa 7 (0x7F / 0xFF) is NaN, so the largest finite
 * magnitude is 1.75 * 2^8 = 448.
 * ------------------------------------------------------------------------- */
static double e4m3_to_double(uint8_t c)
{
    const int e = (c >> 3) & 0xF, m = c & 7;
    const double sign = (c & 0x80) ? -1.0 : 1.0;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) return sign * ldexp((double)m, -9);
    return sign * ldexp(1.0 + m / 8.0, e - 7);
}

/* Nearest finite E4M3 value to y, ties to the code with an even last bit
 * (round to nearest even), magnitudes beyond 448 saturating to 448; NaN gives
 * 0x7F.  Done by brute force over the 127 finite non-negative codes, which
 * is the definition of rounding to the nearest representable value. */
static uint8_t e4m3_from_float(float y)
{
    if (isnan(y)) return 0x7F;
    const uint8_t sign = signbit(y) ? 0x80 : 0;
    const double a = fabs((double)y);
    int best = 0;
    double best_err = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        const double err = fabs(e4m3_to_double((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0)) {
            best = c;
            best_err = err;
        }
    }
    return (uint8_t)(sign | best);
}

int oracle_e4m3_decode(const uint8_t *codes, int64_t n, double *out)
{
    if ((n > 0 && (!codes || !out)) || n < 0) return ORACLE_EINVAL;
    for (int64_t i = 0; i < n; ++i) out[i] = e4m3_to_double(codes[i]);
    return ORACLE_OK;
}

int oracle_e4m3_encode(const float *x, int64_t n, uint8_t *out)
{
    if ((n > 0 && (!x || !out)) || n < 0) return ORACLE_EINVAL;
    for (int64_t i = 0; i < n; ++i) out[i] = e4m3_from_float(x[i]);
    return ORACLE_OK;
}

int oracle_version(void) { return 1; }

/* ---------------------------------------------------------------------------
 * Slot of logical position `pos` of the sequence whose block table is `row`
 * ([P1] §5.2.3 / B.2.3; [P4] §3.1): the logical block is pos // block_size,
 * the offset inside it is pos % block_size, and the physical row number is
 * physical_block * block_size + offset.
 * Returns -1 through *slot_out when the logical block lies beyond the table.
 * ------------------------------------------------------------------------- */
int oracle_slot_of(const int32_t *row, int32_t max_blocks, int32_t block_size,
                   int64_t pos, int64_t *slot_out)
{
    if (!row || !slot_out || block_size <= 0 || pos < 0) return ORACLE_EINVAL;
    int64_t logical_block = pos / block_size;
    int64_t offset = pos % block_size;
    if (logical_block >= max_blocks) { *slot_out = -1; return ORACLE_EBOUNDS; }
    *slot_out = (int64_t)row[logical_block] * block_size + offset;
    return ORACLE_OK;
}

/* ---------------------------------------------------------------------------
 * Decode-step slot_mapping ([P1] §5.2.1, [P4] §4.4, [P1] B.4): one new token
 * per sequence; sequence t's context_len already counts that token, so its
 * position is context_lens[t] - 1.  Rows t >= num_seqs (padding up to
 * num_tokens) and rows with context_len 0 get -1.
 * ------------------------------------------------------------------------- */
int oracle_decode_slot_mapping(const int32_t *block_tables, int32_t max_blocks,
                               const int32_t *context_lens, int32_t num_seqs,
                               int32_t block_size, int32_t num_tokens,
                               int32_t *slot_mapping)
{
    if (!block_tables || !context_lens || !slot_mapping) return ORACLE_EINVAL;
    if (num_seqs < 0 || num_tokens < 0 || max_blocks <= 0 || block_size <= 0)
        return ORACLE_EINVAL;
    int rc = ORACLE_OK;
    for (int32_t t = 0; t < num_tokens; ++t) {
        slot_mapping[t] = -1;
        if (t >= num_seqs) continue;
        int32_t len = context_lens[t];
        if (len <= 0) continue;
        int64_t slot;
        if (oracle_slot_of(block_tables + (int64_t)t * max_blocks, max_blocks,
                           block_size, (int64_t)len - 1, &slot) != ORACLE_OK) {
            rc = ORACLE_EBOUNDS;
            continue;
        }
        slot_mapping[t] = (int32_t)slot;
    }
    return rc;
}

/* ---------------------------------------------------------------------------
 * store_kvcache ([P3] "注意力内核的三个分支", [P4] §3.1): for every token t
 * whose slot s is not -1, row s of the cache (all Hkv heads x D values) becomes
 * a bit copy of k[t] (and likewise v[t]).  Nothing else changes.
 * row_elems = Hkv * D; num_slots = num_blocks * block_size.
 * ------------------------------------------------------------------------- */
int oracle_kv_store(const uint16_t *k, const uint16_t *v, const int32_t *slot_mapping,
                    int32_t num_tokens, uint16_t *k_cache, uint16_t *v_cache,
                    int64_t num_slots, int32_t row_elems)
{
    if (!k || !v || !slot_mapping || !k_cache || !v_cache) return ORACLE_EINVAL;
    if (num_tokens < 0 || num_slots < 0 || row_elems <= 0) return ORACLE_EINVAL;
    int rc = ORACLE_OK;
    for (int32_t t = 0; t < num_tokens; ++t) {
        int64_t s = slot_mapping[t];
        if (s == -1) continue;
        if (s < 0 || s >= num_slots) { rc = ORACLE_EBOUNDS; continue; }
        memcpy(k_cache + s * row_elems, k + (int64_t)t * row_elems, sizeof(uint16_t) * (size_t)row_elems);
        memcpy(v_cache + s * row_elems, v + (int64_t)t * row_elems, sizeof(uint16_t) * (size_t)row_elems);
    }
    return rc;
}

/* ---------------------------------------------------------------------------
 * store_kvcache into an E4M3 cache: as oracle_kv_store, but element (h, d) of
 * row t is stored as the E4M3 code of the binary32 quotient x / scale[h]
 * (one IEEE single-precision division of the bf16 value by the kv head's
 * scale, then the rounding of e4m3_from_float).  The per-kv-head scales k_scale
 * and v_scale are the caller's (a calibrated max |x| / 448, say).
 * ------------------------------------------------------------------------- */
int oracle_kv_store_fp8(const uint16_t *k, const uint16_t *v, const int32_t *slot_mapping,
                        int32_t num_tokens, uint8_t *k_cache, uint8_t *v_cache, int64_t num_slots,
                        int32_t hkv, int32_t d, const float *k_scale, const float *v_scale)
{
    if (!k || !v || !slot_mapping || !k_cache || !v_cache || !k_scale || !v_scale) return ORACLE_EINVAL;
    if (num_tokens < 0 || num_slots < 0 || hkv <= 0 || d <= 0) return ORACLE_EINVAL;
    const int64_t row = (int64_t)hkv * d;
    int rc = ORACLE_OK;
    for (int32_t t = 0; t < num_tokens; ++t) {
        int64_t s = slot_mapping[t];
        if (s == -1) continue;
        if (s < 0 || s >= num_slots) { rc = ORACLE_EBOUNDS; continue; }
        for (int64_t i = 0; i < row; ++i) {
            const int32_t h = (int32_t)(i / d);
            const float xk = (float)bf16_bits_to_double(k[t * row + i]);
            const float xv = (float)bf16_bits_to_double(v[t * row + i]);
            const float qk = xk / k_scale[h];
            const float qv = xv / v_scale[h];
            k_cache[s * row + i] = e4m3_from_float(qk);
            v_cache[s * row + i] = e4m3_from_float(qv);
        }
    }
    return rc;
}

/* ---------------------------------------------------------------------------
 * Copy-on-write block copy ([P4] §2.2: before a sequence writes into a
 * physical block that other sequences share, the block is copied to a new one;
 * [P2] §1: copy-on-write of a half-full shared block).  For each pair i in
 * order, physical block dst = pairs[2i + 1] of both caches becomes a bit copy
 * of block src = pairs[2i] (all block_size x Hkv x D values); src == dst
 * leaves it as it is.  An id outside [0, num_blocks) makes the pair skipped
 * and the call return ORACLE_EBOUNDS.  block_elems = block_size * Hkv * D.
 * ------------------------------------------------------------------------- */
int oracle_copy_blocks(uint16_t *k_cache, uint16_t *v_cache, const int32_t *pairs, int32_t num_pairs,
                       int32_t num_blocks, int64_t block_elems)
{
    if (!k_cache || !v_cache || (num_pairs > 0 && !pairs)) return ORACLE_EINVAL;
    if (num_pairs < 0 || num_blocks <= 0 || block_elems <= 0) return ORACLE_EINVAL;
    int rc = ORACLE_OK;
    for (int32_t i = 0; i < num_pairs; ++i) {
        const int64_t src = pairs[2 * i], dst = pairs[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) { rc = ORACLE_EBOUNDS; continue; }
        if (src == dst) continue;
        memcpy(k_cache + dst * block_elems, k_cache + src * block_elems, sizeof(uint16_t) * (size_t)block_elems);
        memcpy(v_cache + dst * block_elems, v_cache + src * block_elems, sizeof(uint16_t) * (size_t)block_elems);
    }
    return rc;
}

/* ---------------------------------------------------------------------------
 * Paged decode attention ([P2] §5, [P3] "注意力内核的三个分支", [P1] B.1.2).
 * For sequence b with L = context_lens[b] and query head h:
 *   g     = h / (Hq / Hkv)                                  (GQA map)
 *   K_j   = k_cache[block_tables[b][j / bs]][j % bs][g][:]   for j < L
 *   s_j   = scale * sum_d q[b][h][d] * K_j[d]
 *   w_j   = exp(s_j - max_j s_j)
 *   out   = sum_j w_j V_j / sum_j w_j ;  L == 0 gives out = 0.
 * Layouts: q [B, Hq, D]; caches [num_blocks, bs, Hkv, D]; block_tables
 * [B, max_blocks]; out [B, Hq, D] (double).
 * ------------------------------------------------------------------------- */
typedef struct {
    const uint16_t *q, *k_cache, *v_cache;
    const uint8_t *k8, *v8;           /* E4M3 caches instead of bf16 (then k_cache, v_cache unused) */
    const float *k_scale, *v_scale;   /* their per-kv-head scales */
    const int32_t *block_tables, *context_lens;
    const int32_t *row_seq;           /* query row -> sequence whose table it reads (NULL: the row itself) */
    int32_t num_seqs, hq, hkv, d, block_size, num_blocks, max_blocks;
    double scale;
    double *out;
    int32_t nthreads, tid;
    int status;
} decode_job;

/* Element idx of the K (is_v = 0) or V cache, kv head g: a bf16 value, or an
 * E4M3 code times the kv head's scale. */
static double kv_elem(const decode_job *J, int is_v, int64_t idx, int32_t g)
{
    if (J->k8)
        return is_v ? e4m3_to_double(J->v8[idx]) * (double)J->v_scale[g]
                    : e4m3_to_double(J->k8[idx]) * (double)J->k_scale[g];
    return bf16_bits_to_double(is_v ? J->v_cache[idx] : J->k_cache[idx]);
}

/* One (sequence, query head) item.  Returns 0 or ORACLE_EBOUNDS. */
static int decode_one(const decode_job *J, int32_t b, int32_t h, double *scores)
{
    const int32_t d_all = J->d;
    const int32_t group = J->hq / J->hkv;
    const int32_t g = h / group;
    const int32_t len = J->context_lens[b];
    double *o = J->out + ((int64_t)b * J->hq + h) * d_all;
    for (int32_t d = 0; d < d_all; ++d) o[d] = 0.0;
    if (len == 0) return ORACLE_OK;
    if (len < 0 || (int64_t)len > (int64_t)J->max_blocks * J->block_size) return ORACLE_EBOUNDS;

    const uint16_t *qv = J->q + ((int64_t)b * J->hq + h) * d_all;
    const int32_t *row = J->block_tables + (int64_t)(J->row_seq ? J->row_seq[b] : b) * J->max_blocks;

    /* pass 1: scores and their maximum */
    double m = -INFINITY;
    for (int32_t j = 0; j < len; ++j) {
        int32_t phys = row[j / J->block_size];
        if (phys < 0 || phys >= J->num_blocks) return ORACLE_EBOUNDS;
        int64_t base = (((int64_t)phys * J->block_size + j % J->block_size) * J->hkv + g) * d_all;
        double dot = 0.0;
        for (int32_t d = 0; d < d_all; ++d)
            dot += bf16_bits_to_double(qv[d]) * kv_elem(J, 0, base + d, g);
        scores[j] = J->scale * dot;
        if (scores[j] > m) m = scores[j];
    }
    /* pass 2: weights, their sum and the weighted sum of V rows */
    double denom = 0.0;
    for (int32_t j = 0; j < len; ++j) {
        int32_t phys = row[j / J->block_size];
        int64_t base = (((int64_t)phys * J->block_size + j % J->block_size) * J->hkv + g) * d_all;
        double w = exp(scores[j] - m);
        denom += w;
        for (int32_t d = 0; d < d_all; ++d)
            o[d] += w * kv_elem(J, 1, base + d, g);
    }
    for (int32_t d = 0; d < d_all; ++d) o[d] /= denom;
    return ORACLE_OK;
}

static void *decode_worker(void *arg)
{
    decode_job *J = (decode_job *)arg;
    int32_t max_len = J->max_blocks * J->block_size;
    double *scores = (double *)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
    if (!scores) { J->status = ORACLE_EINVAL; return NULL; }
    int64_t items = (int64_t)J->num_seqs * J->hq;
    for (int64_t it = J->tid; it < items; it += J->nthreads) {
        int rc = decode_one(J, (int32_t)(it / J->hq), (int32_t)(it % J->hq), scores);
        if (rc != ORACLE_OK) J->status = rc;
    }
    free(scores);
    return NULL;
}

static int run_decode(decode_job proto, int32_t nthreads);

int oracle_paged_decode(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                        const int32_t *block_tables, int32_t max_blocks,
                        const int32_t *context_lens, int32_t num_seqs, int32_t hq,
                        int32_t hkv, int32_t d, int32_t block_size, int32_t num_blocks,
                        double scale, double *out, int32_t nthreads)
{
    if (!k_cache || !v_cache) return ORACLE_EINVAL;
    decode_job J = {q, k_cache, v_cache, NULL, NULL, NULL, NULL, block_tables, context_lens, NULL,
                    num_seqs, hq, hkv, d, block_size, num_blocks, max_blocks, scale, out, 1, 0, ORACLE_OK};
    return run_decode(J, nthreads);
}

/* ---------------------------------------------------------------------------
 * Paged attention with several new tokens per sequence (chunked prefill over a
 * cached prefix, or a mixed batch of prefills and decodes): sequence b holds
 * L = context_lens[b] tokens in the cache, the last n = cu_seqlens_q[b+1] -
 * cu_seqlens_q[b] of them new; its query row r = cu_seqlens_q[b] + i (i < n)
 * sits at position p = L - n + i and attends the keys j <= p (causal
 * attention over the cached prefix and the new tokens before it: the
 * nano-vllm KV-cache post §3.5 builds the slots of such a chunk, the mini-vLLM
 * README names the prefill with a cached prefix as the next step).  Each row
 * is the decode definition above with context length p + 1 and sequence b's
 * block table.  q, out: [T, Hq, D] with T = cu_seqlens_q[B].  n > L, or a
 * decreasing cu_seqlens_q, is ORACLE_EINVAL.
 * ------------------------------------------------------------------------- */
int oracle_paged_attention(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                           const int32_t *block_tables, int32_t max_blocks, const int32_t *cu_seqlens_q,
                           const int32_t *context_lens, int32_t num_seqs, int32_t hq, int32_t hkv, int32_t d,
                           int32_t block_size, int32_t num_blocks, double scale, double *out, int32_t nthreads)
{
    if (!cu_seqlens_q || !context_lens || num_seqs < 0 || cu_seqlens_q[0] != 0) return ORACLE_EINVAL;
    const int32_t T = cu_seqlens_q[num_seqs];
    int32_t *row_seq = (int32_t *)malloc(sizeof(int32_t) * (size_t)(T > 0 ? T : 1));
    int32_t *row_len = (int32_t *)malloc(sizeof(int32_t) * (size_t)(T > 0 ? T : 1));
    if (!row_seq || !row_len) { free(row_seq); free(row_len); return ORACLE_EINVAL; }
    int rc = ORACLE_OK;
    for (int32_t b = 0; b < num_seqs && rc == ORACLE_OK; ++b) {
        const int32_t n = cu_seqlens_q[b + 1] - cu_seqlens_q[b], L = context_lens[b];
        if (n < 0 || n > L) { rc = ORACLE_EINVAL; break; }
        for (int32_t i = 0; i < n; ++i) {
            row_seq[cu_seqlens_q[b] + i] = b;
            row_len[cu_seqlens_q[b] + i] = L - n + i + 1;
        }
    }
    if (rc == ORACLE_OK) {
        decode_job J = {q, k_cache, v_cache, NULL, NULL, NULL, NULL, block_tables, row_len, row_seq,
                        T, hq, hkv, d, block_size, num_blocks, max_blocks, scale, out, 1, 0, ORACLE_OK};
        rc = run_decode(J, nthreads);
    }
    free(row_seq);
    free(row_len);
    return rc;
}

/* The same attention over E4M3 caches: K_j, V_j are the codes' values times
 * k_scale[g], v_scale[g] (per kv head), everything else as above. */
int oracle_paged_decode_fp8(const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                            const float *k_scale, const float *v_scale,
                            const int32_t *block_tables, int32_t max_blocks,
                            const int32_t *context_lens, int32_t num_seqs, int32_t hq,
                            int32_t hkv, int32_t d, int32_t block_size, int32_t num_blocks,
                            double scale, double *out, int32_t nthreads)
{
    if (!k_cache || !v_cache || !k_scale || !v_scale) return ORACLE_EINVAL;
    decode_job J = {q, NULL, NULL, k_cache, v_cache, k_scale, v_scale, block_tables, context_lens, NULL,
                    num_seqs, hq, hkv, d, block_size, num_blocks, max_blocks, scale, out, 1, 0, ORACLE_OK};
    return run_decode(J, nthreads);
}

static int run_decode(decode_job proto, int32_t nthreads)
{
    const uint16_t *q = proto.q;
    const int32_t *block_tables = proto.block_tables, *context_lens = proto.context_lens;
    const int32_t num_seqs = proto.num_seqs, hq = proto.hq, hkv = proto.hkv, d = proto.d;
    const int32_t block_size = proto.block_size, max_blocks = proto.max_blocks;
    double *out = proto.out;
    if (!q || !block_tables || !context_lens || !out) return ORACLE_EINVAL;
    if (num_seqs < 0 || hq <= 0 || hkv <= 0 || d <= 0 || block_size <= 0 || max_blocks <= 0)
        return ORACLE_EINVAL;
    if (hq % hkv != 0) return ORACLE_EINVAL; /* [P2] §5: the group size must divide */
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;

    decode_job jobs[256];
    pthread_t threads[256];
    for (int32_t t = 0; t < nthreads; ++t) {
        jobs[t] = proto;
        jobs[t].nthreads = nthreads;
        jobs[t].tid = t;
        jobs[t].status = ORACLE_OK;
    }
    if (nthreads == 1) {
        decode_worker(&jobs[0]);
    } else {
        for (int32_t t = 0; t < nthreads; ++t) pthread_create(&threads[t], NULL, decode_worker, &jobs[t]);
        for (int32_t t = 0; t < nthreads; ++t) pthread_join(threads[t], NULL);
    }
    int rc = ORACLE_OK;
    for (int32_t t = 0; t < nthreads; ++t)
        if (jobs[t].status != ORACLE_OK) rc = jobs[t].status;
    return rc;
}

/* ---------------------------------------------------------------------------
 * Split-K partial state and merge (the online-softmax state of [P2] §5,
 * applied to disjoint token ranges).  For the tokens j in [j0, j1) of
 * (b, h):
 *   m   = max s_j,   l = sum exp(s_j - m),   acc = sum exp(s_j - m) V_j.
 * An empty range gives m = -inf, l = 0, acc = 0.
 * Merging n states: M = max m_i; l = sum exp(m_i - M) l_i;
 * out = sum exp(m_i - M) acc_i / l  (states with m_i = -inf contribute 0;
 * if every state is empty, out = 0).
 * ------------------------------------------------------------------------- */
int oracle_partial_state(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                         const int32_t *block_tables, int32_t max_blocks, int32_t b,
                         int32_t h, int32_t hq, int32_t hkv, int32_t d, int32_t block_size,
                         int32_t num_blocks, double scale, int32_t j0, int32_t j1,
                         double *m_out, double *l_out, double *acc_out)
{
    if (!q || !k_cache || !v_cache || !block_tables || !m_out || !l_out || !acc_out) return ORACLE_EINVAL;
    if (hq % hkv != 0 || j0 < 0 || j1 < j0) return ORACLE_EINVAL;
    const int32_t g = h / (hq / hkv);
    const uint16_t *qv = q + ((int64_t)b * hq + h) * d;
    const int32_t *row = block_tables + (int64_t)b * max_blocks;
    for (int32_t e = 0; e < d; ++e) acc_out[e] = 0.0;
    *m_out = -INFINITY;
    *l_out = 0.0;
    if (j1 == j0) return ORACLE_OK;
    if ((int64_t)j1 > (int64_t)max_blocks * block_size) return ORACLE_EBOUNDS;
    double *s = (double *)malloc(sizeof(double) * (size_t)(j1 - j0));
    if (!s) return ORACLE_EINVAL;
    double m = -INFINITY;
    for (int32_t j = j0; j < j1; ++j) {
        int32_t phys = row[j / block_size];
        if (phys < 0 || phys >= num_blocks) { free(s); return ORACLE_EBOUNDS; }
        int64_t base = (((int64_t)phys * block_size + j % block_size) * hkv + g) * d;
        double dot = 0.0;
        for (int32_t e = 0; e < d; ++e)
            dot += bf16_bits_to_double(qv[e]) * bf16_bits_to_double(k_cache[base + e]);
        s[j - j0] = scale * dot;
        if (s[j - j0] > m) m = s[j - j0];
    }
    double l = 0.0;
    for (int32_t j = j0; j < j1; ++j) {
        int32_t phys = row[j / block_size];
        int64_t base = (((int64_t)phys * block_size + j % block_size) * hkv + g) * d;
        double w = exp(s[j - j0] - m);
        l += w;
        for (int32_t e = 0; e < d; ++e) acc_out[e] += w * bf16_bits_to_double(v_cache[base + e]);
    }
    free(s);
    *m_out = m;
    *l_out = l;
    return ORACLE_OK;
}

int oracle_merge_states(const double *m, const double *l, const double *acc, int32_t n,
                        int32_t d, double *out)
{
    if (!m || !l || !acc || !out || n < 0 || d <= 0) return ORACLE_EINVAL;
    double big = -INFINITY;
    for (int32_t i = 0; i < n; ++i)
        if (m[i] > big) big = m[i];
    for (int32_t e = 0; e < d; ++e) out[e] = 0.0;
    if (big == -INFINITY) return ORACLE_OK;
    double denom = 0.0;
    for (int32_t i = 0; i < n; ++i) {
        if (m[i] == -INFINITY) continue;
        double f = exp(m[i] - big);
        denom += f * l[i];
        for (int32_t e = 0; e < d; ++e) out[e] += f * acc[(int64_t)i * d + e];
    }
    for (int32_t e = 0; e < d; ++e) out[e] /= denom;
    return ORACLE_OK;
}
