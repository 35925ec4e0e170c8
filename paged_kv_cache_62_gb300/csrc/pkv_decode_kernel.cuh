// Decode-phase PagedAttention for sm_103a (q_len = 1, grouped-query attention).
//
// What it computes (mini-vLLM README §5 "Triton PagedAttention Decode Kernel";
// MinivLLM review, section "注意力内核的三个分支"): for sequence b, query head
// h and L = context_lens[b],
//     out[b, h] = softmax_j(scale * q[b, h] . K_j) V_j,   j < L,
// with K_j / V_j read from row j % bs of physical block block_tables[b][j / bs]
// at kv head h / G (G = Hq / Hkv), accumulated in fp32 with the online softmax
// state (m, l, acc) of the README.
//
// How (GB300 design):
//  * Kv heads are taken in groups of HG (the largest divisor of Hkv that is
//    at most the CTA's 8 consumer warps).  A unit of work is TOKS = TW * SUB
//    consecutive tokens of one (sequence, head group), TW = 16 tokens per
//    warp (32 for E4M3 caches) and SUB warps per head (see team_warps): the
//    group's cache rows, moved by one 4-D TMA tensor copy per physical-block
//    span and cache into a shared-memory stage as 128-byte-swizzled rows (see
//    Tc).  Each CTA warms L2 with its first units while it sets up (see
//    BalanceState::hint).
//  * One CTA per SM: a producer warp streams units through a ring of 2-16
//    stages (mbarrier transaction counts for "full", consumer arrivals for
//    "empty"); HG * SUB consumer warps take one TW-token slice of one kv head
//    each, so every consumer works on every stage and the CTA's warps finish
//    together.  Block-table entries for 32 boxes at a time are fetched by the
//    producer's lanes one batch ahead; q rows arrive by bulk copy in a
//    separate 2-slot ring.
//  * A consumer serves all G query heads of its kv head from one K/V read,
//    on the warp-level tensor cores: S^T = Q K^T and O^T += V^T P^T as
//    m16n8k16 MMAs with fp32 accumulators, K and V fed by ldmatrix from the
//    swizzled stage, P kept in registers as two bf16 parts (see attend_tile);
//    up to 16 virtual heads (queries x heads) fill the tile's two 8-row
//    halves; the online softmax rescales only when a score passes the running
//    max by a slack, and exponentials are ex2 of log2e-prescaled scores.
//    Query-split CTAs (QS) instead give every warp all tokens of one kv head
//    and its own queries: long runs of new tokens share K/V passes.  Their
//    tensor-memory variant (TC5) runs a 128-row entry against 128-key tiles
//    on the 5th-generation tensor cores: tcgen05.mma issued by one thread,
//    scores, weights and output in tensor memory, 8 softmax warps (see
//    tc5_softmax_warps).
//  * The decode step's store can run in the same launch: the tile holding a
//    sequence's new token takes its K/V row from the step's inputs and writes
//    it to the cache (see DecodeParams::k_new).
//  * The batch's unit list is cut into one slice per SM id, each slice's size
//    following the finishing times the previous call on the workspace saw.
//    A CTA whose slice covers a whole (sequence, head group) writes bf16
//    output directly; otherwise it leaves per-head partial states (m, l, acc)
//    in the workspace and counts its units in on a per-(sequence, kv head)
//    counter; the CTA that completes the count merges the pieces (split-K /
//    flash-decoding without a second kernel).
//
// This header holds the kernel and its launch templates; pkv_decode.cu
// instantiates the bf16-cache kernels for up to 8 virtual heads and defines
// the C entry points, pkv_decode_wide.cu the bf16 ones for 9 to 16,
// pkv_decode_qs.cu the query-split ones, pkv_decode_tc5.cu their tensor-memory
// variant, pkv_decode_fp8.cu the E4M3 ones.
#pragma once
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <mutex>
#include <type_traits>
#include <unordered_map>
#include <vector>

#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {

constexpr int kMaxStages = 16;    // ring depth (as many as fit: 3 of 64 KiB, 12 of 16 KiB)
constexpr int kMaxSlots = 512;    // slices: SM ids (adaptive) or CTAs (fixed split)
constexpr int kSegmentUnits = 8;  // small calls: one CTA per segment when no segment has more units
constexpr uint32_t kTableMagic = 0x62616c31u;
constexpr uint32_t kEpochMagic = 0x65706f63u;
constexpr int32_t kHintMagic = 0x6869;
// Units of a slice's first block warmed into L2 at the start of a call (measured on the Qwen3-0.6B-shaped
// batch, 64 KiB units: 3 -> 94.6 us, 6 -> 93.1, 8 -> 92.6, 12 -> 92.0 per call; none: 96.5; 16, the whole
// 256-token block, about 0.3 us less than 12 graph-replayed).
constexpr int kHintUnits = 16;
// Context lengths a set-up thread loads at once in the unit scan.
constexpr int kScanBatch = 16;

// Consumer warps per CTA and tokens each takes from a stage (a stage holds
// team_warps * warp_tokens token rows of head_dim: 64 KiB for head_dim 128).
// A warp's tile is made of 16-token sub-tiles, each the n extent of two
// m16n8k16 score products and the k extent of one output product: one for
// bf16 caches, two for E4M3 caches (the same bytes a stage; two independent
// sub-tiles give the consumer twice the independent MMA chains, and the
// widening of E4M3 codes makes that path consumer-bound).  A warp's
// registers do not grow with the group size (G query heads are rows of one
// MMA tile), so every group size runs 8 consumers.
__host__ __device__ constexpr int team_warps(int) { return 8; }
// Tensor-memory (tcgen05) query-split CTAs: 8 warps that own the 128 rows of
// the tile, two per row (the softmax and the epilogue: warp w takes rows
// 32 (w % 4) .. + 31 and keys 64 (w / 4) .. + 63 of every tile), one warp that
// issues the tensor-core products, then the producer warp.
constexpr int kTc5SoftmaxWarps = 8;
constexpr int kTc5Consumers = kTc5SoftmaxWarps + 1;
constexpr int kTc5Keys = 128;          // keys per tile (one unit): the N extent of one score product
// TMEM columns (512): two score buffers of 128 columns, each later holding its tile's weights P in its
// first 64 columns (bf16 pairs of keys 2c, 2c + 1 in column c; key half h in columns 32 h .. 32 h + 31);
// the output (D <= 128 columns, from column 256); and two Q tiles of 64 columns from column 384 (row r of
// the tile in lane r, dims 2c, 2c + 1 in column c).
constexpr uint32_t kTc5Cols = 512, kTc5OCol = 256, kTc5QCol = 384;
constexpr uint32_t kTc5SlabBytes = 128u * 128u;  // one 64-dim slab of 128 rows of a K or V slot
// The K tiles stream through a ring of nst slots (a slot is free again once its scores are read); the V
// tiles through a ring of kTc5VSlots (free again once their output product is done).
constexpr int kTc5VSlots = 3;
static_assert(kTc5Keys * 128 == int(kTc5SlabBytes), "a stage's K or V slab holds one tile of 128-byte rows");

// Query-split CTAs (qs; long runs of new tokens, see paged_decode_kernel)
// take 32-token tiles too: one kv head's stage is small, and every warp
// works on every token.  Their tensor-memory variant (tc5) takes kTc5Keys keys
// a tile: the N extent of one score product.
__host__ __device__ constexpr int warp_tokens(int, bool fp8, bool qs = false, bool tc5 = false)
{
    return tc5 ? kTc5Keys : (fp8 || qs ? 32 : 16);
}

// ------------------------------------------------------------------ load balance state
// In the adaptive mode a slice's size follows what the previous call on this
// workspace saw: a slice that finished late gets a little less work, one
// that finished early a little more (SMs of a GB300 stream HBM at somewhat
// different rates).  This only moves work around: any table
// contents, garbage included, give correct results.
struct BalanceState {
    float weight[2][kMaxSlots];           // weight a slice had in the call that wrote the entry (0: no SM)
    float elapsed[2][kMaxSlots];          // its run time in us (<= 0: present, nothing measured)
    uint32_t tag[2][kMaxSlots];           // (call number of the writer) ^ kTableMagic
    unsigned long long claim[kMaxSlots];  // (gen << 32) | 1 once a CTA took the slice this call
    // First copy of each SM id's own slice in the call that wrote the entry: (cache row, kv head
    // coordinate, gen ^ kHintMagic, sequence b) and (logical block of the row in b's table, b's length, 0, 0).
    // The next call warms L2 with the rows from there to the end of that block while it sets up (a
    // slice's first unit moves little from one decode step to the next), if b's table still maps
    // that logical block to the row's block.  Only a hint; any contents are safe.
    int4 hint[kMaxSlots][2];
    // Control block.  Call number e of a workspace runs with gen = e + 1 (never 0, the value
    // of zero-filled tags).  `done` counts the CTAs of the call that have read the block; the
    // one that completes the count leaves epoch = e + 1, stamp = (e + 1) ^ kEpochMagic,
    // done = 0.  A zero-filled workspace reads as call 0.
    uint32_t epoch, stamp, done, pad;
};

struct DecodeParams {
    const uint16_t *q;
    const int32_t *block_tables;
    const int32_t *context_lens;
    uint16_t *out;
    unsigned long long *ws_count;  // [B * Hkv] arrival counters: (gen << 32) | units arrived
    float *ws_ml;                  // [slots][G][2] (m, l) per partial
    float *ws_acc;                 // [slots][G][D] unnormalised accumulators
    BalanceState *ws_bal;
    int32_t *err;
    int32_t B, Hq, Hkv, bs, log2_bs, NB, max_blocks, len_limit;
    int32_t hg, nhg, sub, toks;  // kv heads per group, groups, warp slices per head, tokens per unit
    int32_t boxtok, nbox;        // tokens per TMA box (min(toks, bs)) and boxes per unit
    int32_t nst, cons, lg_nbox;  // ring stages, consumer warps (hg * sub), log2(nbox)
    int32_t num_workers;         // > 0: fixed split over about num_workers / consumers CTAs; 0: adaptive
    int32_t per_segment;         // fixed split with one slice per (entry, head group): no split-K pieces
    int32_t qslots;              // Q row buffers: 2 (the next segment's rows load during this one), or 1
                                 // where that buys the ring another stage
    float scale_log2;            // scale * log2(e)
    const float *k_scale, *v_scale;  // E4M3 caches: per-kv-head scales (unused for bf16 caches)
    const int32_t *row_seq;          // several query rows per sequence: row -> the sequence whose table it
                                     // reads (null: row b reads table row b)
    // Several new tokens per sequence sharing one K/V stream: the kernel's G "heads" of a kv head are
    // qn queries x gq query heads (virtual head hh = query hh / gq, head hh % gq).  Entry b holds
    // cnt <= qn queries (row_cnt[b], or qn where row_cnt is null); its query i is q / out row
    // b * qstride + i and sees the keys before position L - cnt + i + 1 (L: entry b's context length).
    // Decode: qn = 1, gq = G, qstride = 1.
    int32_t qn, gq, qstride;
    const int32_t *row_cnt;
    // Store fused into a decode (qn = 1): row b of k_new / v_new [B, Hkv, D] (bf16) is the K/V of
    // sequence b's token at position L - 1; the kernel writes it (E4M3 caches: its codes under the kv
    // head's scales) to that token's cache row (k_cache_w / v_cache_w, [NB * bs, Hkv, D] elements) and
    // attends with it; slot_out[b] (nullable) receives the row (-1 when nothing was stored).  k_new
    // null: a plain decode.
    const uint16_t *k_new, *v_new;
    uint8_t *k_cache_w, *v_cache_w;
    int32_t *slot_out;
};

// What the producer tells the consumers about the unit in a stage.
struct alignas(16) UnitMeta {
    int32_t b, g, u, n;            // unit u of the n units of (b, group g); b < 0: no more work
    int32_t L, flags, slice, cnt;  // context length of b, kFirst | kLast | kSliceEnd, slice of the unit,
                                   // queries of entry b
    int32_t newrow, pad[3];        // fused store: cache row of token L - 1 if the unit holds it, else -1
};
constexpr int kFirst = 1;     // first unit of (b, g) in this slice
constexpr int kLast = 2;      // last unit of (b, g) in this slice
constexpr int kSliceEnd = 4;  // last unit of the slice

// Shared-memory layout, computed the same way on the host (size) and device (offsets).
struct CtaLayout {
    uint32_t kv_bytes, stage_bytes, q_bytes, comb_bytes;
    uint32_t off_v, off_q, off_comb, off_meta, off_bar, off_bound, off_wts, off_red, off_sh, off_scan, total;
};

__host__ __device__ inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

// Floats per state in the combine buffer: G * (D + 2) rounded up to a
// multiple of 4, so every block (and its float4 rows) is 16-byte aligned.
__host__ __device__ inline int comb_stride(int D, int G) { return int(align_up(uint32_t(G * (D + 2)), 4)); }

// Whether a kernel variant may run with one Q row buffer: regular bf16 CTAs of 8 virtual heads, where
// at head_dim 128 and 8 kv heads a CTA the second buffer (32 KiB) costs the ring its third stage.  The
// other variants keep two, a fixed count that keeps their code as it was (fewer heads fit three stages
// beside two buffers; the 16-row tiles miss a third stage either way).
__host__ __device__ constexpr bool one_q_buffer_ok(int G, bool fp8, bool qs, bool tc5)
{
    return G == 8 && !fp8 && !qs && !tc5;
}

// es: bytes per cached element (2 for bf16, 1 for E4M3); qs: query-split
// CTA (all sub warps of a kv head on the same tokens, each with its own G
// virtual heads); tc5: its tensor-memory variant (Q slots hold the 128-row
// tile as 128-byte-swizzled 64-dim slabs).
__host__ __device__ inline CtaLayout cta_layout(int D, int G, int es, int hg, int sub, int nst, int B,
                                                bool qs = false, bool tc5 = false, int qslots = 2)
{
    CtaLayout l;
    const int toks = warp_tokens(G, es == 1, qs, tc5) * (qs ? 1 : sub);
    l.kv_bytes = uint32_t(toks * hg * D * es);
    // stages start on the 1024-byte swizzle period; tc5: a stage is a K slot, the V slots follow the ring
    l.stage_bytes = align_up((tc5 ? 1 : 2) * l.kv_bytes, 1024);
    l.q_bytes = tc5 ? 0u : align_up(uint32_t(hg * (qs ? sub : 1) * G * D * 2), 128);  // tc5: Q in tensor memory
    // states of the non-leading warps of every head (the leader keeps its own in registers); tc5: the
    // values each row's two key halves exchange ([2 tile parities][2 halves][128 rows] floats)
    l.comb_bytes = tc5 ? 2u * 2u * 128u * 4u
                       : (sub > 1 && !qs ? align_up(uint32_t(hg * (sub - 1) * comb_stride(D, G) * 4), 128) : 0u);
    uint32_t o = uint32_t(nst) * l.stage_bytes;
    l.off_v = o;
    if (tc5) o += uint32_t(kTc5VSlots) * align_up(l.kv_bytes, 1024);
    l.off_q = o;
    o += uint32_t(qslots) * l.q_bytes;
    l.off_comb = o;
    o += l.comb_bytes;
    l.off_meta = o;
    o += uint32_t(nst) * uint32_t(sizeof(UnitMeta));
    l.off_bar = o;
    // full / empty per stage, q full / empty x2, combine full / free; tc5: scores full x2, scores read x2,
    // weights full x2, output product done x2, drain, a row's two halves met (one per lane quarter) x4,
    // all softmax warps met, a Q tile written, full / empty per V slot (the stages' pair then covers the
    // K slots), and per K slot its meta written
    o += uint32_t(2 * nst + 6 + (tc5 ? 15 + 2 * kTc5VSlots + nst : 0)) * 8;
    l.off_bound = align_up(o, 16);
    o = l.off_bound + (kMaxSlots + 1) * 8;
    l.off_wts = o;
    o += kMaxSlots * 4;
    l.off_red = o;
    o += 64 * 4;
    l.off_sh = o;
    o += 32;
    l.off_scan = o;
    o += uint32_t(B + 1) * 4;
    l.total = o;
    return l;
}

// Kv-head grouping: HG = the largest divisor of Hkv that is <= team_warps(G);
// the warps of a CTA split as HG heads x SUB token slices, SUB the largest
// power of two <= team_warps(G) / HG (a power of two, so a unit is a whole
// number of power-of-two TMA boxes).
inline int head_group(int Hkv, int G)
{
    for (int g = team_warps(G); g > 1; --g)
        if (Hkv % g == 0) return g;
    return 1;
}

inline int warp_slices(int G, int hg)
{
    int s = 1;
    while (2 * s * hg <= team_warps(G)) s *= 2;
    return s;
}

// Workspace regions.  The arrival counters of a call must read as zero (or as
// another call's tag) when it starts.  A completed call leaves its counters at
// zero, but a call of other sizes on the same workspace may have used the same
// words for partial states, whose bits can be anything.  So calls with up to
// kFixedCounters counters keep them in a region at a fixed offset that nothing
// else ever uses; a larger call keeps them after that region, and the host
// clears them on the stream before its launch (count_clear).
constexpr size_t kFixedCounters = 16384;

struct WsLayout {
    size_t bal_off, count_off, count_bytes, ml_off, acc_off, total;
    bool count_clear;  // counters outside the fixed region: cleared by the host before the launch
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Piece slots.  Only a segment (an entry's units of one head group) that
// crosses a slice boundary leaves pieces, and a slice holds at most two of
// them: its first segment (the one holding the slice's first unit, when it
// began in an earlier slice or goes on into a later one) and its last
// segment (going on into the next slice).  Two numberings, whichever needs
// fewer slots:
//   by entry (B * nhg < kMaxSlots): (slice + b * nhg + group) * hg + h,
//     injective because slices and segments are both ordered along the
//     unit list;
//   by slice (otherwise): (2 slice + [not the slice's first segment]) * hg + h,
//     2 * kMaxSlots * hg slots whatever the batch.
// Query-split CTAs (qs) keep one piece per warp: slot * team_warps + warp,
// and one arrival counter per (entry, kv head, warp).
__host__ __device__ inline bool slots_by_slice(int32_t B, int32_t nhg) { return int64_t(B) * nhg >= kMaxSlots; }

inline WsLayout ws_layout(int32_t B, int32_t G, int32_t Hkv, int32_t D, bool qs = false)
{
    const int hg = qs ? 1 : head_group(Hkv, G);
    const size_t subq = qs ? size_t(team_warps(G)) : 1;
    const size_t slots = (slots_by_slice(B, Hkv / hg) ? 2 * size_t(kMaxSlots)
                                                       : size_t(kMaxSlots) + size_t(B) * size_t(Hkv / hg)) *
                         size_t(hg) * subq;
    WsLayout w;
    w.bal_off = 0;
    const size_t fixed_off = align256(sizeof(BalanceState)), fixed_end = fixed_off + kFixedCounters * 8;
    const size_t counters = size_t(B) * size_t(Hkv) * subq;
    w.count_clear = counters > kFixedCounters;
    w.count_off = w.count_clear ? fixed_end : fixed_off;
    w.count_bytes = counters * 8;
    w.ml_off = w.count_clear ? align256(fixed_end + w.count_bytes) : fixed_end;
    w.acc_off = w.ml_off + align256(slots * size_t(G) * 2 * 4);
    w.total = w.acc_off + slots * size_t(G) * size_t(D) * 4;
    return w;
}

// ------------------------------------------------------------------ unit list walking
// Units in (b, group, u) order; scan[b] = sum over earlier sequences of their
// units per group, so the list holds nhg * scan[B] units.
struct Walker {
    int32_t b, g, u, n;
};

__device__ __forceinline__ void walker_advance(Walker &w, const int32_t *scan, int32_t nhg, int32_t B)
{
    if (++w.u < w.n) return;
    w.u = 0;
    if (++w.g < nhg) return;
    w.g = 0;
    do {
        ++w.b;
        w.n = (w.b < B) ? scan[w.b + 1] - scan[w.b] : 1;
    } while (w.n == 0);
}

// Position of unit x (0 <= x < nhg * scan[B]).
__device__ __forceinline__ Walker walker_locate(const int32_t *scan, int32_t B, int32_t nhg, long long x)
{
    int lo = 0, hi = B;  // nhg*scan[lo] <= x < nhg*scan[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if ((long long)nhg * scan[mid] <= x)
            lo = mid;
        else
            hi = mid;
    }
    Walker w;
    w.b = lo;
    w.n = scan[lo + 1] - scan[lo];
    const int32_t rem = int32_t(x - (long long)nhg * scan[lo]);  // < nhg * n <= total units < 2^31
    w.g = rem / w.n;
    w.u = rem - w.g * w.n;
    return w;
}

// Barrier of the CTA's nt set-up threads (its consumer warps, threads 0 .. nt - 1): the
// producer warp runs its own part of the set-up meanwhile and meets them at __syncthreads.
__device__ __forceinline__ void setup_sync(int nt)
{
    asm volatile("bar.sync 1, %0;" ::"r"(nt) : "memory");
}

// Units per sequence -> exclusive prefix in scan[0..B].
// `tmp` needs 32 ints of shared memory that is free during the call.
static __device__ void unit_prefix_scan(const DecodeParams &p, int32_t *scan, int32_t *tmp, int nt)
{
    const int tid = threadIdx.x;
    const int lane = tid & 31, wid = tid >> 5, nw = nt >> 5;
    // thread tid counts the units of its run of entries [lo, hi), the lengths loaded kScanBatch at a
    // time (all in flight together: one memory round trip a batch, not one an entry)
    const int per = (p.B + nt - 1) / nt;
    const int lo = min(p.B, tid * per), hi = min(p.B, lo + per);
    int32_t sum = 0;
    for (int i0 = lo; i0 < hi; i0 += kScanBatch) {
        int32_t len[kScanBatch];
#pragma unroll
        for (int k = 0; k < kScanBatch; ++k) len[k] = i0 + k < hi ? __ldg(p.context_lens + i0 + k) : 0;
#pragma unroll
        for (int k = 0; k < kScanBatch; ++k) {
            if (i0 + k >= hi) break;
            int32_t n = 0;
            // several queries of a sequence sharing a stream need at least one key each (the row
            // arrays of a chunked call are built that way; a same-n call can break it)
            if (len[k] < 0 || len[k] > p.len_limit || (!p.row_cnt && p.qn > 1 && len[k] < p.qn)) {
                if (blockIdx.x == 0) flag_error(p.err, PKV_ERR_CONTEXT_RANGE);
            } else {
                n = (len[k] + p.toks - 1) / p.toks;
            }
            scan[i0 + k] = n;
            sum += n;
        }
    }
    int32_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t v = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) tmp[wid] = incl;
    setup_sync(nt);
    if (wid == 0) {
        const int32_t v = lane < nw ? tmp[lane] : 0;
        int32_t inc = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t u = __shfl_up_sync(kFull, inc, o);
            if (lane >= o) inc += u;
        }
        if (lane < nw) tmp[lane] = inc - v;
    }
    setup_sync(nt);
    int32_t run = tmp[wid] + incl - sum;
    for (int i = lo; i < hi; ++i) {
        const int32_t n = scan[i];
        scan[i] = run;
        run += n;
    }
    if (lo < hi && hi == p.B) scan[p.B] = run;
    setup_sync(nt);
}

// ------------------------------------------------------------------ one tile
// Slack (log2 units) a score may exceed the running max before the running
// state is rescaled: weights stay <= 2^kRescaleSlack, which fp32 holds with
// ample room, and most tiles skip the rescale entirely.
constexpr float kRescaleSlack = 8.0f;

// Stage layout.  The producer copies the cached rows (one token, one kv head)
// of a box of boxtok tokens and HG kv heads as NP parts of RB bytes each, one
// 4-D TMA copy per box and cache landing as [kv head][part][token][RB bytes],
// so the boxtok rows of a (kv head, part) are consecutive RB-byte rows of
// shared memory, swizzled by the copy: 16-byte chunk c of row R lands at
// chunk c ^ (R & 7) (128-byte rows) or c ^ ((R >> 1) & 3) (64-byte rows,
// 64-dim E4M3 caches).
// The chunks of eight consecutive tokens then sit in eight different bank
// groups, and one ldmatrix reads them without a conflict.
// HR: 8-row halves of the MMA tile that hold a warp's virtual heads (2 when
// a warp has more than 8).
template <int D, bool FP8, bool QS = false, int HR_ = 1>
struct Tc {
    static constexpr int ES = FP8 ? 1 : 2;              // bytes per cached element
    static constexpr int ROWB = D * ES;                 // bytes per cached row
    static constexpr int RB = ROWB >= 128 ? 128 : 64;   // bytes per shared-memory row
    static constexpr int NP = ROWB / RB;                // parts per cached row
    static constexpr int NCP = ROWB / 32;               // 16-byte chunk pairs per row (one ldmatrix.x4 each)
    static constexpr int KS = D / 16;                   // k-steps of the score product
    static constexpr int MT = D / 16;                   // m-tiles of the output product
    static constexpr int NT = FP8 || QS ? 2 : 1;        // 16-token sub-tiles of a warp's tile
    static constexpr int TW = 16 * NT;                  // tokens of a warp's tile (warp_tokens)
    static constexpr int HR = HR_;                      // 8-row halves of the MMA tile holding virtual heads
};

__host__ __device__ constexpr int row_bytes_smem(int D, int es) { return D * es >= 128 ? 128 : 64; }

template <int RB>
__device__ __forceinline__ uint32_t swizzled_chunk(uint32_t c, uint32_t R)
{
    return RB == 128 ? (c ^ (R & 7u)) : (c ^ ((R >> 1) & 3u));
}

// Byte offsets, from a stage's K (or V) region, of the 16-byte row pieces this
// lane hands to ldmatrix for sub-tile st of the warp's tile (token
// j * TW + 16 st + tl of the unit): tl = 8 * (lane / 16) + lane % 8, chunk
// 2i + (lane / 8) % 2 of the row.  Matrix q of an .x4 load is then
// (tokens 0-7 | 8-15 of the sub-tile) x (chunk 2i | 2i + 1) for q = 0 (0-7, 2i),
// 1 (0-7, 2i+1), 2 (8-15, 2i), 3 (8-15, 2i+1).
// Kept factored (a few registers instead of NT x NCP): chunk pair i lies in
// row part i / (RB / 32) (part stride boxtok RB bytes), and since boxtok is a
// multiple of 8 the swizzle key of its row is that of the token alone, so the
// piece's chunk is ((i % (RB / 32)) << 5) ^ kx.
template <int D, bool FP8, bool QS>
struct LaneOffsets {
    using T = Tc<D, FP8, QS>;
    uint32_t base[T::NT];  // row of the sub-tile's token, part 0, chunk 0
    uint32_t part;         // bytes between a row's parts
    uint32_t kx;           // the lane's chunk bit and the row's swizzle key, as a byte offset
    __device__ __forceinline__ uint32_t at(int st, int i) const
    {
        constexpr int per = T::RB / 32;  // chunk pairs per part
        return base[st] + uint32_t(i / per) * part + ((uint32_t(i % per) << 5) ^ kx);
    }
};

template <int D, bool FP8, bool QS>
__device__ __forceinline__ void lane_offsets(LaneOffsets<D, FP8, QS> &off, int lane, int j, int h, int hg, int boxtok)
{
    using T = Tc<D, FP8, QS>;
    const int tl = ((lane >> 4) << 3) | (lane & 7), e = (lane >> 3) & 1;
    const int lg = __ffs(boxtok) - 1;
    const uint32_t box_bytes = uint32_t(boxtok * hg * T::ROWB);
    off.part = uint32_t(boxtok * T::RB);
#pragma unroll
    for (int st = 0; st < T::NT; ++st) {
        const int t = j * T::TW + 16 * st + tl;
        const int bi = t >> lg, r = t & (boxtok - 1);
        off.base[st] = uint32_t(bi) * box_bytes + uint32_t(h * T::NP * boxtok + r) * T::RB;
        if (st == 0) off.kx = uint32_t(e ^ (T::RB == 128 ? (r & 7) : ((r >> 1) & 3))) << 4;  // the same for every st
    }
}

// Head dim held by output fragment element (m-tile mt, half: 0 for c0/c1,
// 1 for c2/c3) of the thread in row group g = lane / 4.  bf16 caches: the
// transposed V tile puts dim 16 mt + g in rows g and 16 mt + 8 + g in rows
// g + 8; E4M3 caches: dims 16 mt + 2g and 16 mt + 2g + 1 (the byte pairs of
// a 16-bit transpose, split by a byte permute).
template <bool FP8>
__device__ __forceinline__ int dim_of(int mt, int half, int g)
{
    return FP8 ? 16 * mt + 2 * g + half : 16 * mt + 8 * half + g;
}

__device__ __forceinline__ uint32_t f16x2_of(float lo, float hi)
{
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// f16 pair, magnitudes past the f16 range saturating to +-65504 (NaN stays NaN).
__device__ __forceinline__ uint32_t f16x2_sat(float lo, float hi)
{
    uint32_t h;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(hi), "f"(lo));
    return h;
}

// One warp tile (NT sub-tiles of 16 tokens) of one (sequence, kv head) for its
// query heads (virtual heads) on the tensor cores, m16n8k16 with fp32
// accumulators:
//   S^T = Q K^T    rows: virtual heads (the thread's rows are g = lane / 4
//                  and, with HR = 2, g + 8; rows past the warp's heads are
//                  zero), columns: 8 tokens per n-tile, k: head dims;
//   P = 2^(S - m)  the online-softmax weights of the thread's rows;
//   O^T += V^T P^T rows: head dims, columns: 8 virtual heads per half
//                  (HR halves), k: tokens.
// The S^T accumulator fragment of a sub-tile's two n-tiles is, register for
// register, the P^T operand fragment of its output product (rows 0-7 for
// half 0, rows 8-15 for half 1), so P never leaves the registers.  kb / vb:
// shared addresses of the stage's K and V regions.  lim[hr]: tokens (from the
// tile's first) below it count for the thread's row of half hr (the causal
// bound of its query); TAIL: tokens from `valid` on are not the sequence's
// (their rows may hold anything, even NaN), so their V values are zeroed
// before the product.  E4M3 caches run the products in f16 (every E4M3 value
// is exact in f16, and so is every bf16 query element of magnitude
// 2^-14 .. 65504; smaller ones keep f16's subnormal steps of 2^-24, larger
// ones saturate at 65504); the kv head's K scale is in ksc, its V scale is
// applied by the caller.
template <int D, bool FP8, bool QS, int HR_, bool TAIL>
__device__ __forceinline__ void attend_tile(uint32_t kb, uint32_t vb,
                                            const LaneOffsets<D, FP8, QS> &off,
                                            const uint32_t (&qa)[Tc<D, FP8, QS, HR_>::KS][2 * Tc<D, FP8, QS, HR_>::HR],
                                            float ksc, const int (&lim)[Tc<D, FP8, QS, HR_>::HR], int valid,
                                            float (&m)[Tc<D, FP8, QS, HR_>::HR], float (&l)[Tc<D, FP8, QS, HR_>::HR],
                                            float (&o)[Tc<D, FP8, QS, HR_>::MT][Tc<D, FP8, QS, HR_>::HR][4], int lane)
{
    using T = Tc<D, FP8, QS, HR_>;
    constexpr int NT = T::NT, HR = T::HR;
    // accumulation chains per n-tile (bf16: halves the MMA dependency depth; not with 16 rows, whose
    // registers would spill at D = 128)
    constexpr int CH = NT == 1 && HR == 1 ? 2 : 1;
    const int r4 = lane & 3;
    // A operand of k-step ks: rows g (qa[ks][0], [1]) and g + 8 (qa[ks][2], [3], zero when HR = 1)
    auto a1 = [&](int ks) { return HR == 2 ? qa[ks][2 % (2 * HR)] : 0u; };
    auto a3 = [&](int ks) { return HR == 2 ? qa[ks][3 % (2 * HR)] : 0u; };
    float sa[NT][CH][2][4];  // [sub-tile][chain][n-tile][fragment]
#pragma unroll
    for (int st = 0; st < NT; ++st)
#pragma unroll
        for (int c = 0; c < CH; ++c)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) sa[st][c][nt][e] = 0.f;
#pragma unroll
    for (int i = 0; i < T::NCP; ++i) {
#pragma unroll
        for (int st = 0; st < NT; ++st) {
            uint32_t r0, r1, r2, r3;
            ldsm_x4(kb + off.at(st, i), r0, r1, r2, r3);
            if constexpr (!FP8) {
                // chunks 2i, 2i+1 = dims 16i..16i+15 = k-step i; r0/r1 tokens 0-7, r2/r3 tokens 8-15
                mma_bf16_16816(sa[st][i % CH][0], qa[i][0], a1(i), qa[i][1], a3(i), r0, r1);
                mma_bf16_16816(sa[st][i % CH][1], qa[i][0], a1(i), qa[i][1], a3(i), r2, r3);
            } else {
                // chunk 2i (2i+1) = k-step 2i (2i+1); a register holds four codes 4r..4r+3 of a
                // token: dims (4r, 4r+1) are k-slots (2r, 2r+1), dims (4r+2, 4r+3) k-slots (2r+8, 2r+9)
                uint32_t b[4][2];
                e4m3x4_to_f16x2x2(r0, b[0][0], b[0][1]);
                e4m3x4_to_f16x2x2(r1, b[1][0], b[1][1]);
                e4m3x4_to_f16x2x2(r2, b[2][0], b[2][1]);
                e4m3x4_to_f16x2x2(r3, b[3][0], b[3][1]);
                mma_f16_16816(sa[st][0][0], qa[2 * i][0], a1(2 * i), qa[2 * i][1], a3(2 * i), b[0][0], b[0][1]);
                mma_f16_16816(sa[st][0][1], qa[2 * i][0], a1(2 * i), qa[2 * i][1], a3(2 * i), b[2][0], b[2][1]);
                mma_f16_16816(sa[st][CH - 1][0], qa[2 * i + 1][0], a1(2 * i + 1), qa[2 * i + 1][1],
                              a3(2 * i + 1), b[1][0], b[1][1]);
                mma_f16_16816(sa[st][CH - 1][1], qa[2 * i + 1][0], a1(2 * i + 1), qa[2 * i + 1][1],
                              a3(2 * i + 1), b[3][0], b[3][1]);
            }
        }
    }
    // the thread's scores: row g (half 0, fragment elements c0, c1) and row g + 8 (half 1, c2, c3),
    // tokens 16 st + 8 nt + 2 r4 + e
    float x[HR][NT * 4];  // -inf past the row's bound
#pragma unroll
    for (int hr = 0; hr < HR; ++hr)
#pragma unroll
        for (int st = 0; st < NT; ++st)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int k = 4 * st + 2 * nt + e;
                    float sum = sa[st][0][nt][2 * hr + e];
                    if constexpr (CH == 2) sum += sa[st][1][nt][2 * hr + e];
                    x[hr][k] = 16 * st + 8 * nt + 2 * r4 + e < lim[hr] ? sum * ksc : -INFINITY;
                }
    float mx[HR];
    bool grow = false;
#pragma unroll
    for (int hr = 0; hr < HR; ++hr) {
        mx[hr] = x[hr][0];
#pragma unroll
        for (int k = 1; k < NT * 4; ++k) mx[hr] = fmaxf(mx[hr], x[hr][k]);
        mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(kFull, mx[hr], 1));  // the four threads of a row
        mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(kFull, mx[hr], 2));
        grow |= mx[hr] > m[hr] + kRescaleSlack;
    }
    // Online softmax (m, l, acc).  The running max only moves when some score passes it by more
    // than the slack; the first tile with a valid token for the row always moves it (m = -inf).
    if (__any_sync(kFull, grow)) {
#pragma unroll
        for (int hr = 0; hr < HR; ++hr) {
            const float mn = fmaxf(m[hr], mx[hr]);
            const float alpha = mn == -INFINITY ? 1.0f : ex2(m[hr] - mn);  // 0 on the row's first valid tile
            l[hr] *= alpha;
            m[hr] = mn;
            // output columns 2 r4 and 2 r4 + 1 of half hr are the rows of threads 8 r4 and 8 r4 + 4
            const float a0 = __shfl_sync(kFull, alpha, 8 * r4), a1v = __shfl_sync(kFull, alpha, 8 * r4 + 4);
#pragma unroll
            for (int mt = 0; mt < T::MT; ++mt) {
                o[mt][hr][0] *= a0;
                o[mt][hr][1] *= a1v;
                o[mt][hr][2] *= a0;
                o[mt][hr][3] *= a1v;
            }
        }
    }
    // The weights as the output product's operand.  bf16 caches: two parts, hi = bf16(p) and lo =
    // bf16(p - hi); hi + lo carries p to 2^-17 of itself and both products are exact in the fp32
    // accumulators, so the output is the fp32 weights' sum to about fp32 precision.  E4M3 caches: one
    // f16 part (2^-12 of p; the products run in f16 there, and the consumers are the bound, so a
    // second product would cost time).
    uint32_t pb[HR][NT][2], pl[HR][NT][2];
#pragma unroll
    for (int hr = 0; hr < HR; ++hr) {
        // 2^(-inf) = 0 for the masked tokens; a row without any valid token so far (m = -inf) takes 0
        const float mr = m[hr] == -INFINITY ? 0.f : m[hr];
        float pr[NT * 4];
#pragma unroll
        for (int k = 0; k < NT * 4; ++k) pr[k] = ex2(x[hr][k] - mr);
        float ps = 0.f;
#pragma unroll
        for (int k = 0; k < NT * 4; ++k) ps += pr[k];
        l[hr] += ps;
#pragma unroll
        for (int st = 0; st < NT; ++st)
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                const float p0 = pr[4 * st + 2 * c], p1 = pr[4 * st + 2 * c + 1];
                if constexpr (FP8) {
                    pb[hr][st][c] = f16x2_of(p0, p1);
                    pl[hr][st][c] = 0u;
                } else {
                    pb[hr][st][c] = pack_bf16x2(p0, p1);
                    pl[hr][st][c] = pack_bf16x2(p0 - __uint_as_float(pb[hr][st][c] << 16),
                                                p1 - __uint_as_float(pb[hr][st][c] & 0xffff0000u));
                }
            }
    }

#pragma unroll
    for (int st = 0; st < NT; ++st) {
        // transposed V tiles: the low half of a register is token 2 r4 (8 + 2 r4) of the sub-tile, the
        // high half the next one
        uint32_t keep0 = 0xffffffffu, keep1 = 0xffffffffu;
        if constexpr (TAIL) {
            const int v0 = valid - 16 * st;
            keep0 = (2 * r4 < v0 ? 0x0000ffffu : 0u) | (2 * r4 + 1 < v0 ? 0xffff0000u : 0u);
            keep1 = (2 * r4 + 8 < v0 ? 0x0000ffffu : 0u) | (2 * r4 + 9 < v0 ? 0xffff0000u : 0u);
        }
#pragma unroll
        for (int i = 0; i < T::NCP; ++i) {
            uint32_t r0, r1, r2, r3;
            ldsm_x4_t(vb + off.at(st, i), r0, r1, r2, r3);
            if constexpr (TAIL) {
                r0 &= keep0;
                r1 &= keep0;
                r2 &= keep1;
                r3 &= keep1;
            }
            if constexpr (!FP8) {
                // m-tile i: dims 16i + g (r0: tokens 0-7, r2: tokens 8-15) and 16i + 8 + g (r1, r3)
#pragma unroll
                for (int hr = 0; hr < HR; ++hr) {
                    mma_bf16_16816(o[i][hr], r0, r1, r2, r3, pb[hr][st][0], pb[hr][st][1]);
                    mma_bf16_16816(o[i][hr], r0, r1, r2, r3, pl[hr][st][0], pl[hr][st][1]);
                }
            } else {
                // a register holds (token 2r4: dims 2g, 2g+1 | token 2r4+1: dims 2g, 2g+1) of a 16-dim
                // chunk; the byte permute pairs the two tokens per dim: low half dim 2g, high half dim 2g+1
                uint32_t a[4][2];
                e4m3x4_to_f16x2x2(__byte_perm(r0, 0u, 0x3120), a[0][0], a[0][1]);
                e4m3x4_to_f16x2x2(__byte_perm(r1, 0u, 0x3120), a[1][0], a[1][1]);
                e4m3x4_to_f16x2x2(__byte_perm(r2, 0u, 0x3120), a[2][0], a[2][1]);
                e4m3x4_to_f16x2x2(__byte_perm(r3, 0u, 0x3120), a[3][0], a[3][1]);
#pragma unroll
                for (int hr = 0; hr < HR; ++hr) {
                    mma_f16_16816(o[2 * i][hr], a[0][0], a[0][1], a[2][0], a[2][1], pb[hr][st][0], pb[hr][st][1]);
                    mma_f16_16816(o[2 * i + 1][hr], a[1][0], a[1][1], a[3][0], a[3][1], pb[hr][st][0],
                                  pb[hr][st][1]);
                }
            }
        }
    }
}

// ------------------------------------------------------------------ load balance
__device__ __forceinline__ unsigned smid()
{
    unsigned v;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(v));
    return v;
}

__device__ __forceinline__ unsigned nsmid()
{
    unsigned v;
    asm volatile("mov.u32 %0, %%nsmid;" : "=r"(v));
    return v;
}

// Sums of two floats per thread over the nt set-up threads (fixed order:
// identical in every CTA).  `red` holds 2 * 32 floats.
__device__ __forceinline__ float2 block_sum2(float2 v, float *red, int nt)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = nt >> 5;
    v.x = warp_sum(v.x);
    v.y = warp_sum(v.y);
    setup_sync(nt);
    if (lane == 0) {
        red[2 * wid] = v.x;
        red[2 * wid + 1] = v.y;
    }
    setup_sync(nt);
    float2 t = make_float2(0.f, 0.f);
    for (int i = 0; i < nw; ++i) {
        t.x += red[2 * i];
        t.y += red[2 * i + 1];
    }
    return t;
}

// The balance entries this thread reads in build_partition (slices tid + k nt
// for k < kBalE, nt set-up threads), loaded up front so that their memory
// round trip overlaps the context-length loads of unit_prefix_scan.  Both
// table halves are loaded, before this call's number is known;
// build_partition keeps the entry whose tag names the previous call.
constexpr int kBalE = 4;
struct BalanceIn {
    float w[2][kBalE], t[2][kBalE];  // [table half][entry k]
    uint32_t tag[2][kBalE];
};
// the fewest set-up threads a CTA has: 5 consumer warps (a head group of 5)
static_assert(kBalE * 5 * 32 >= kMaxSlots, "the balance entries of the set-up threads must cover every slice");

__device__ __forceinline__ BalanceIn load_balance(const DecodeParams &p, bool adaptive, int nslots, int nt)
{
    BalanceIn in;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int k = 0; k < kBalE; ++k) {
            const int i = threadIdx.x + k * nt;
            in.w[h][k] = 1.0f;
            in.t[h][k] = 0.f;
            in.tag[h][k] = 0u;
            if (adaptive && i < nslots) {
                // plain L2 loads; the half this call writes is told apart by its tag
                in.tag[h][k] = __ldcg(&p.ws_bal->tag[h][i]);
                in.w[h][k] = __ldcg(&p.ws_bal->weight[h][i]);
                in.t[h][k] = __ldcg(&p.ws_bal->elapsed[h][i]);
            }
        }
    return in;
}

// Slice bounds of this call.  Adaptive mode: each slice entry of the table
// half written by the previous call on this workspace (call - 1) keeps its
// weight scaled by clamp(sqrt(mean elapsed / its elapsed), 0.9, 1.12)
// (weight 0: an SM id without a CTA) -- a damped step: a slice's time also
// varies with the data it held, and the full step overcorrects (consecutive
// calls' finishing times then anti-correlate); entries from any other call
// count as unknown (weight 1).  Fixed mode: equal weights.  Every CTA computes the same bounds from the
// same inputs in the same order; leaves the weights in w[].  Run by the nt
// set-up threads.
static __device__ void build_partition(const DecodeParams &p, uint32_t gen, bool adaptive, int nslots, long long T,
                                long long *bound, float *w, float *red, const BalanceIn &in, int nt)
{
    const int tid = threadIdx.x;
    const uint32_t want = (gen - 1u) ^ kTableMagic;
    // pass 1: raw weights (kept in w) and elapsed times (kept in bound[] as float bits)
    float tsum = 0.f, tcnt = 0.f;
    float *el = reinterpret_cast<float *>(bound);
#pragma unroll
    for (int k = 0; k < kBalE; ++k) {
        const int i = tid + k * nt;
        if (i >= nslots) break;
        float x = 1.0f, t = 0.f;
        const bool h1 = in.tag[1][k] == want;  // the half the previous call wrote (selects, no indexing)
        if (adaptive && (h1 || in.tag[0][k] == want)) {
            x = h1 ? in.w[1][k] : in.w[0][k];
            t = h1 ? in.t[1][k] : in.t[0][k];
            if (!(x >= 0.f) || !(x < 1.0e6f)) x = 1.0f;
            if (!(t < 1.0e9f)) t = 0.f;
            if (x > 0.f && t > 0.f) {
                tsum += t;
                tcnt += 1.f;
            }
        }
        w[i] = x;
        el[i] = t;
    }
    const float2 tt = block_sum2(make_float2(tsum, tcnt), red, nt);
    tsum = tt.x;
    tcnt = tt.y;
    const float tmean = tcnt > 0.f ? tsum / tcnt : 0.f;
    // pass 2: scale by the finishing-time ratio, then bound every weight to [1/4, 4] x mean
    float wsum = 0.f, wcnt = 0.f;
    for (int i = tid; i < nslots; i += nt) {
        float x = w[i];
        const float t = el[i];
        if (x > 0.f && t > 0.f && tmean > 0.f) x *= fminf(fmaxf(sqrtf(tmean / t), 0.9f), 1.12f);
        w[i] = x;
        if (x > 0.f) {
            wsum += x;
            wcnt += 1.f;
        }
    }
    const float2 ww = block_sum2(make_float2(wsum, wcnt), red, nt);
    wsum = ww.x;
    wcnt = ww.y;
    const float wmean = wcnt > 0.f ? wsum / wcnt : 1.0f;
    for (int i = tid; i < nslots; i += nt) {
        float x = wcnt > 0.f ? w[i] / wmean : 1.0f;  // mean 1 over present slices; none: equal weights
        if (x > 0.f) x = fminf(fmaxf(x, 0.25f), 4.0f);
        w[i] = x;
    }
    setup_sync(nt);
    // bounds: the weights in fixed point (2^16 per unit weight, at most 2^18 a slice), their exact
    // integer prefix over the slices, then 2^20 tickets for the whole list -> tiles (a shift, no
    // division).  Exact integers keep the bounds nondecreasing however the sums associate (a float
    // prefix split over threads could drop a bound by one unit after a zero-weight slice).  Thread
    // tid takes slices [tid per, (tid + 1) per), per <= kBalE; its sum is scanned over the set-up
    // threads (warp shuffles, then the warp totals in red[]).
    {
        const int lane = tid & 31, wid = tid >> 5, nw = nt >> 5;
        const int per = (nslots + nt - 1) / nt;
        const int lo = min(nslots, tid * per), hi = min(nslots, lo + per);
        int32_t *ired = reinterpret_cast<int32_t *>(red);
        int32_t run = 0;
        for (int i = lo; i < hi; ++i) run += int32_t(w[i] * 65536.0f);
        int32_t incl = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t v = __shfl_up_sync(kFull, incl, o);
            if (lane >= o) incl += v;
        }
        if (lane == 31) ired[wid] = incl;
        setup_sync(nt);
        if (wid == 0) {
            const int32_t v = lane < nw ? ired[lane] : 0;
            int32_t inc = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t u = __shfl_up_sync(kFull, inc, o);
                if (lane >= o) inc += u;
            }
            if (lane < nw) ired[lane] = inc - v;  // warp offsets
            if (lane == 31) ired[32] = inc;       // total
        }
        setup_sync(nt);
        const int32_t total = ired[32];
        // an exact, nondecreasing prefix times one positive factor, rounded down: nondecreasing
        // tickets.  No weights: equal slices (i < 512: 32-bit).
        const float tickets = total > 0 ? 1048576.0f / float(total) : 0.f;
        int32_t acc = ired[wid] + incl - run;
        for (int i = lo; i < hi; ++i) {
            const int pre = total > 0 ? int(fminf(float(acc) * tickets, 1048576.0f)) : (i << 20) / nslots;
            bound[i] = (T * pre) >> 20;
            acc += int32_t(w[i] * 65536.0f);
        }
        if (tid == 0) bound[nslots] = T;
    }
    // bounds are monotone: the integer prefix only grows and pre is clamped to [0, 2^20]
    setup_sync(nt);
}

__device__ __forceinline__ bool try_claim(unsigned long long *word, uint32_t gen)
{
    const unsigned long long cur = *reinterpret_cast<volatile unsigned long long *>(word);
    if (uint32_t(cur >> 32) == gen) return false;
    return atomicCAS(word, cur, (static_cast<unsigned long long>(gen) << 32) | 1ull) == cur;
}

// Warp-collective: claim a non-empty slice that no CTA took yet, among the
// slices this CTA looks after (s = blockIdx.x + k * gridDim.x).  -1 if none.
// With `record`, also writes the balance entries of the looked-after slices
// that are empty this call (nobody else writes them): present if an SM
// claimed it, absent otherwise.
static __device__ int claim_leftover(const DecodeParams &p, uint32_t gen, const long long *bound, int nslots, int wp,
                              bool record)
{
    const int lane = threadIdx.x & 31;
    for (int k0 = 0; blockIdx.x + (long long)k0 * gridDim.x < nslots; k0 += 32) {
        const long long s = blockIdx.x + (long long)(k0 + lane) * gridDim.x;
        bool cand = false;
        if (s < nslots) {
            const unsigned long long cur = *reinterpret_cast<volatile unsigned long long *>(&p.ws_bal->claim[s]);
            const bool claimed = uint32_t(cur >> 32) == gen;
            if (bound[s + 1] > bound[s]) {
                cand = !claimed;
            } else if (record) {
                p.ws_bal->weight[wp][s] = claimed ? 1.0f : 0.0f;
                p.ws_bal->elapsed[wp][s] = claimed ? -1.0f : 0.0f;
                p.ws_bal->tag[wp][s] = gen ^ kTableMagic;
            }
        }
        unsigned m = __ballot_sync(kFull, cand);
        while (m) {
            const int l = __ffs(m) - 1;
            int ok = 0;
            if (lane == l) ok = try_claim(&p.ws_bal->claim[s], gen);
            if (__shfl_sync(kFull, ok, l)) return int(__shfl_sync(kFull, s, l));
            m &= m - 1;
        }
    }
    return -1;
}

// ------------------------------------------------------------------ split-K merge (a6)
// Count the `units` of one piece of (b, kv head) in.  The counter word is
// (gen << 32) | units arrived; a word from another call (another gen: a call
// that gave up half-way, or the zero left by a completed one) counts as
// zero.  Returns 1 for the piece that completes the pair's `total` units
// (and resets the word to 0).  Counting units, not pieces, lets any
// partition of the unit list merge correctly.
__device__ __forceinline__ int arrive_last(unsigned long long *ctr, uint32_t gen, uint32_t units, uint32_t total,
                                           int32_t *err)
{
    // first guess: the counter is at rest (0: the merge of the previous call reset it, or the workspace is
    // new), so the first arrival of a segment takes one round trip; any other value comes back from the
    // failed exchange and the loop goes on from it
    unsigned long long cur = 0ull;
    for (int it = 0; it < (1 << 20); ++it) {
        const uint32_t n = ((uint32_t(cur >> 32) == gen) ? uint32_t(cur) : 0u) + units;
        const unsigned long long next = (static_cast<unsigned long long>(gen) << 32) | n;
        const unsigned long long seen = atomicCAS(ctr, cur, next);
        if (seen == cur) {
            if (n != total) return 0;
            atomicExch(ctr, 0ull);
            return 1;
        }
        cur = seen;
    }
    flag_error(err, PKV_ERR_WAIT_TIMEOUT);  // unreachable in practice: a handful of CTAs contend
    return 0;
}

// Slice that holds unit x (non-empty by construction), 0 <= x < bound[nslots].
__device__ __forceinline__ int slice_of(const long long *bound, int nslots, long long x)
{
    int lo = 0, hi = nslots;  // bound[lo] <= x < bound[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (bound[mid] <= x)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

// Merge the partial states of (b, kv head kvh) left by the non-empty slices
// sf..sl (the segment's first unit is x0) from their piece slots (see
// ws_layout: by slice, f = 1 only in slice sf when the segment is not that
// slice's first, x0 > bound[sf]), and write the outputs of the
// entry's nvh virtual heads that are queries:
//   M = max m_i,  l = sum 2^(m_i - M) l_i,  out = sum 2^(m_i - M) acc_i / l
// (the online-softmax algebra; m in log2 units).  The pieces were written by
// other SMs, so they are read through L2 (ld.global.cg), BATCH pieces at a
// time with independent loads, folded into a running (M, l, acc).
template <int D, int G, bool FP8, bool QS>
__device__ __forceinline__ void merge_pieces(const DecodeParams &p, const long long *bound, int sf, int sl,
                                             long long x0, int g, int h, int jq, int b, int kvh, int nvh, int lane)
{
    constexpr int PER = D / 32;                                // output values per lane
    constexpr int HB = G < 8 ? G : 8;                          // heads merged together (more would spill)
    constexpr int BATCH = HB <= 2 ? 4 : (HB <= 5 ? 2 : 1);     // pieces loaded together
    using Vec = typename std::conditional<PER == 4, float4, float2>::type;
    const float2 *ml = reinterpret_cast<const float2 *>(p.ws_ml);
    for (int h0 = 0; h0 < nvh; h0 += HB) {  // virtual heads past the entry's queries are not written
        float M[HB], lsum[HB], a[HB][PER];
#pragma unroll
        for (int i = 0; i < HB; ++i) {
            M[i] = -INFINITY;
            lsum[i] = 0.f;
#pragma unroll
            for (int e = 0; e < PER; ++e) a[i][e] = 0.f;
        }
        for (int s0 = sf; s0 <= sl; s0 += BATCH) {
            float2 st[BATCH][HB];
            Vec v[BATCH][HB];
            bool use[BATCH];
#pragma unroll
            for (int k = 0; k < BATCH; ++k) {
                const int s = s0 + k;
                use[k] = s <= sl && bound[s + 1] > bound[s];  // empty slices left nothing
                const int sk = use[k] ? s : sf;
                const long long slot = ((slots_by_slice(p.B, p.nhg)
                                             ? 2LL * sk + ((sk == sf && x0 != bound[sf]) ? 1 : 0)
                                             : sk + (long long)b * p.nhg + g) * p.hg + h) * (QS ? p.sub : 1) + jq;
#pragma unroll
                for (int i = 0; i < HB; ++i) {
                    const int hh = min(h0 + i, G - 1);  // a block past G re-reads the last head (not written)
                    st[k][i] = __ldcg(ml + slot * G + hh);
                    v[k][i] = __ldcg(reinterpret_cast<const Vec *>(p.ws_acc + (slot * G + hh) * D + lane * PER));
                }
            }
#pragma unroll
            for (int i = 0; i < HB; ++i) {
                float mb = M[i];
#pragma unroll
                for (int k = 0; k < BATCH; ++k)
                    if (use[k]) mb = fmaxf(mb, st[k][i].x);
                // 0 while nothing has been folded in (M = -inf); a head with no valid token in any piece
                // so far (several queries per stream) keeps its zero state
                const float r = mb == -INFINITY ? 1.0f : ex2(M[i] - mb);
                lsum[i] *= r;
#pragma unroll
                for (int e = 0; e < PER; ++e) a[i][e] *= r;
#pragma unroll
                for (int k = 0; k < BATCH; ++k) {
                    const float f = (use[k] && st[k][i].x != -INFINITY) ? ex2(st[k][i].x - mb) : 0.f;
                    lsum[i] = fmaf(f, st[k][i].y, lsum[i]);
                    const float *x = reinterpret_cast<const float *>(&v[k][i]);
#pragma unroll
                    for (int e = 0; e < PER; ++e) a[i][e] = fmaf(f, x[e], a[i][e]);
                }
                M[i] = mb;
            }
        }
#pragma unroll
        for (int i = 0; i < HB; ++i) {
            const int hh = h0 + i;
            if (hh >= nvh) break;
            const float inv = (FP8 ? __ldg(p.v_scale + kvh) : 1.0f) / lsum[i];
            uint16_t *o = p.out + ((int64_t(b) * p.qstride + jq * p.qn + hh / p.gq) * p.Hq + int64_t(kvh) * p.gq +
                                   hh % p.gq) * D + lane * PER;
            if constexpr (PER == 4)
                *reinterpret_cast<uint2 *>(o) = make_uint2(pack_bf16x2(a[i][0] * inv, a[i][1] * inv),
                                                           pack_bf16x2(a[i][2] * inv, a[i][3] * inv));
            else
                *reinterpret_cast<uint32_t *>(o) = pack_bf16x2(a[i][0] * inv, a[i][1] * inv);
        }
    }
}

// ------------------------------------------------------------------ tensor-memory query-split CTA (tc5)
// A query-split entry of 128 rows -- 128 / gq queries x gq query heads of one kv head, row r = query
// r / gq, head r % gq, in blocks of G = 16 rows that play the part of the query-split CTA's warps (jq) --
// against 128-key tiles of that kv head, on the 5th-generation tensor cores:
//   S = Q K^T      128 x 128 fp32 in tensor memory (two buffers); Q in tensor memory (written there by the
//                  softmax threads from the query rows when a segment starts, two tiles), K
//                  128-byte-swizzled K-major in shared memory (a K slot of the ring);
//   P = 2^(S - m)  by 8 warps, two threads per row (TMEM lane r; each takes 64 of the keys): masks, the
//                  row's running max m (the two halves exchange their tile max) and sum l (fp32 weights),
//                  P written over its own scores in tensor memory (once both halves read theirs: the
//                  exchange of the tile max orders it) rounded to bf16, the product's operand
//                  type (as flash-attention kernels do; a second product for the rounding error, as the
//                  decode path carries, would double the output product's tensor-core time);
//   O += P V       128 x D fp32 in tensor memory, P the A operand from tensor memory, V a V slot's rows
//                  as an MN-major operand from shared memory; O is rescaled in place (read, scaled, written
//                  back) only when a row's max passes m by the slack, which after a segment's first tiles is
//                  rare.
// The MMA warp issues each product as soon as its inputs are ready (see tc5_mma_warp), so the tensor core
// computes the next scores and the current output product while the softmax warps work on a tile.
// Ordering: scores -> sfull[j % 2] (tcgen05.commit); scores read -> sfree[j % 2] (8 warps; it frees the
// unit's K slot and meta); weights written -> pfull[j % 2] (8 warps); output product done -> odone[j % 2]
// and the V slot's vempty (commits); a segment's Q tile written -> qready (8 warps); a unit's meta written
// -> mready[slot] (the producer, before the unit's copy is issued).  A score buffer takes S(k) once the
// output product of unit k - 2, which read its weights there, is done.  A segment's last unit writes the
// next segment's Q tile (into the other Q tile, from the next unit's meta) right after its weights and
// before its epilogue, so the next segment's first scores run while the epilogue waits for the last output
// product and writes O out.  No barrier can run two phases ahead of its waiter: each one's next phase
// needs the waiter's own next step.
struct Tc5Smem {
    const UnitMeta *metas;
    // full / empty: a K slot (and its unit's meta); vfull / vempty: a V slot
    uint64_t *full, *empty, *vfull, *vempty, *qready, *sfull, *sfree, *pfull, *odone, *drain, *pair, *team;
    uint64_t *mready;  // [nst] a K slot's meta written (its copy may still be on the way)
    uint8_t *vbase;                  // V slot 0
    uint32_t stage_addr, v_addr;     // shared addresses of K slot 0 and V slot 0
};

__host__ __device__ inline uint32_t tc5_vslot_bytes(const CtaLayout &lay) { return align_up(lay.kv_bytes, 1024); }

// O += P(u) V(u): the weights of unit u (buffer u % 2) times the V rows of its V slot.
template <int D>
__device__ __forceinline__ void tc5_output_product(const CtaLayout &lay, const Tc5Smem &m, uint32_t tmem,
                                                   uint32_t u, bool first)
{
    constexpr uint32_t IP = idesc_bf16_f32(128, D, true);
    tc_fence_after();
    const uint32_t va = m.v_addr + (u % kTc5VSlots) * tc5_vslot_bytes(lay);
    const uint32_t pa = tmem + (u & 1u) * 128u;  // the weights, over the unit's scores
    // V: keys along K (8-key groups 1024 bytes apart: 16 keys = 2048 bytes), dims along N (64-dim blocks
    // one slab apart)
#pragma unroll
    for (int ks = 0; ks < kTc5Keys / 16; ++ks)
        tc_mma_bf16_ta(tmem + kTc5OCol, pa + uint32_t(8 * ks),
                       smem_desc_sw128(va + uint32_t(ks) * 2048u, kTc5SlabBytes, 1024), IP, !(first && ks == 0));
    tc_commit(&m.odone[u & 1u]);
    tc_commit(&m.vempty[u % kTc5VSlots]);  // the V slot may take the next copy
}

// The MMA warp: lane 0 issues every tensor-core product of the CTA, each as soon as its inputs are
// ready -- S(k) once unit k's K slot has landed (and, on a segment's first unit, its Q tile is written,
// and the output product of unit k - 2 is done), P(k)V once the weights of unit k are written and its V
// slot has landed --
// polling both without blocking on either, so a late copy never holds back an output product whose
// weights are ready.  A K slot (and its unit's meta) is released when the softmax warps have read that
// unit's scores, a V slot when the unit's output product is done.  Before it returns it waits for all
// products to complete (also when it gave up: no progress for the wait limit).
template <int D>
__device__ void tc5_mma_warp(const DecodeParams &p, const CtaLayout &lay, const Tc5Smem &m, uint32_t tmem)
{
    constexpr uint32_t IS = idesc_bf16_f32(128, kTc5Keys, false);
    const int lane = threadIdx.x & 31;
    bool dead = false;
    if (lane == 0) {
        int s = 0;                       // K slot of unit ns
        uint32_t ph = 0;                 // its parity
        uint32_t ns = 0, npv = 0;        // next unit to score, next unit to multiply by V
        uint32_t segs = 0;               // segments begun (Q tiles used)
        bool have_meta = false, ended = false;
        int flags = 0;
        uint32_t nrel = 0;               // units whose K slots were released (their scores read)
        int slot_of[4] = {0, 0, 0, 0};   // K slots of units nrel .. ns - 1 (at most 3)
        bool first_of[2] = {false, false};
        uint64_t t0 = global_ns();
        for (uint32_t it = 0;; ++it) {
            bool progress = false;
            // K slots of units whose scores (and meta) the softmax warps have read
            if (nrel < ns && mbar_test_wait(smem_u32(&m.sfree[nrel & 1u]), (nrel >> 1) & 1u)) {
                mbar_arrive(&m.empty[slot_of[nrel & 3u]]);
                ++nrel;
                progress = true;
            }
            // the next scores: unit ns's K slot (and meta), its Q tile on a segment's first unit, and its
            // score buffer free (the output product of unit ns - 2 done); at most two units ahead of the
            // output products and one ahead of the K slot releases
            if (!ended && ns < npv + 2 && nrel + 1 >= ns) {
                if (!have_meta && mbar_test_wait(smem_u32(&m.full[s]), ph)) {
                    have_meta = true;
                    flags = m.metas[s].flags;
                    if (m.metas[s].b < 0) ended = true;
                }
                if (have_meta && !ended) {
                    const bool qok = !(flags & kFirst) || mbar_test_wait(smem_u32(m.qready), segs & 1u);
                    const bool bok = ns < 2 || mbar_test_wait(smem_u32(&m.odone[ns & 1u]), ((ns >> 1) - 1) & 1u);
                    if (qok && bok) {
                        if (flags & kFirst) ++segs;
                        tc_fence_after();
                        const uint32_t qa = tmem + kTc5QCol + ((segs - 1) & 1u) * 64u;
                        const uint32_t ka = m.stage_addr + uint32_t(s) * lay.stage_bytes;
#pragma unroll
                        for (int ks = 0; ks < D / 16; ++ks) {
                            const uint32_t within = uint32_t(ks & 3) * 32, slab = uint32_t(ks >> 2);
                            tc_mma_bf16_ta(tmem + (ns & 1u) * 128u, qa + uint32_t(8 * ks),
                                           smem_desc_sw128(ka + slab * kTc5SlabBytes + within, 16, 1024), IS, ks > 0);
                        }
                        tc_commit(&m.sfull[ns & 1u]);
                        slot_of[ns & 3u] = s;
                        first_of[ns & 1u] = (flags & kFirst) != 0;
                        ++ns;
                        have_meta = false;
                        if (++s == p.nst) {
                            s = 0;
                            ph ^= 1u;
                        }
                        progress = true;
                    }
                }
            }
            // the next output product, once its weights are written and its V slot has landed
            if (npv < ns && mbar_test_wait(smem_u32(&m.pfull[npv & 1u]), (npv >> 1) & 1u) &&
                mbar_test_wait(smem_u32(&m.vfull[npv % kTc5VSlots]), (npv / kTc5VSlots) & 1u)) {
                tc5_output_product<D>(lay, m, tmem, npv, first_of[npv & 1u]);
                ++npv;
                progress = true;
            }
            if (ended && npv == ns) break;
            if (progress) {
                t0 = global_ns();
            } else if ((it & 255u) == 0 && global_ns() - t0 > kWaitLimitNs) {
                dead = true;
                break;
            }
        }
        if (dead) flag_error(p.err, PKV_ERR_WAIT_TIMEOUT);
        // every product issued has completed before the tensor memory is freed
        tc_commit(m.drain);
    }
    __syncwarp();
    if (!mbar_wait_bounded(m.drain, 0u) && lane == 0) flag_error(p.err, PKV_ERR_WAIT_TIMEOUT);
}

// A tensor-memory CTA's piece of a segment: the 128 rows' (m, l) at ws_ml[tile * 128 + row] and their
// unnormalised outputs at ws_acc[tile * 128 D ..], laid out as [D / 4][128 rows][4] so that a warp's
// 32 rows move 512 contiguous bytes per access; tile numbers the 128-row blocks of the slot space of
// ws_layout (slot = tile * 8 + row / 16).
__device__ __forceinline__ long long tc5_piece_tile(const DecodeParams &p, int slice, bool slice_first, int b, int g)
{
    return slots_by_slice(p.B, p.nhg) ? 2LL * slice + (slice_first ? 0 : 1) : slice + (long long)b * p.nhg + g;
}

// The pieces of one (entry, kv head) segment, merged by the CTA whose piece completed its unit count:
// thread (row, half) folds columns [half D / 2, (half + 1) D / 2) of the row over the pieces left by the
// non-empty slices sf..sl, in slice order (the CTA's own piece, that of slice own, read back from tensor
// memory: the same values it stored), then writes the row's bf16 output if the row is one of the entry's
// queries:
//   M = max m_i,  l = sum 2^(m_i - M) l_i,  out = sum 2^(m_i - M) acc_i / l.
template <int D>
__device__ void tc5_merge(const DecodeParams &p, const long long *bound, int sf, int sl, int own, float own_m,
                          float own_l, uint32_t own_o, long long x0, int g, int b, int row, int half, bool row_ok,
                          int qi)
{
    constexpr int C = D / 2;  // columns of this thread
    const float2 *ml = reinterpret_cast<const float2 *>(p.ws_ml);
    float M = -INFINITY, lsum = 0.f, a[C];
#pragma unroll
    for (int e = 0; e < C; ++e) a[e] = 0.f;
    // the running state takes piece (m, l) with weight f = 2^(m - M'), itself r = 2^(M - M')
    auto rescale = [&](float2 st, float &r, float &f) {
        const float mb = fmaxf(M, st.x);
        r = M == -INFINITY ? 0.f : ex2(M - mb);
        f = ex2(st.x - mb);
        lsum = fmaf(f, st.y, lsum * r);
        M = mb;
    };
    for (int sk = sf; sk <= sl; ++sk) {
        if (bound[sk + 1] <= bound[sk]) continue;  // an empty slice left nothing
        float r, f;
        if (sk == own) {
            // (the load is warp-wide: every lane takes part, also for a row that saw no key here)
            const bool has = own_m != -INFINITY;
            if (has) rescale(make_float2(own_m, own_l), r, f);
            __syncwarp();  // lanes that left an earlier piece early meet again
#pragma unroll
            for (int cc = 0; cc < C / 32; ++cc) {
                uint32_t w[32];
                tmem_ld32(own_o + uint32_t(cc * 32), w);
                if (has) {
#pragma unroll
                    for (int i = 0; i < 32; ++i) a[32 * cc + i] = fmaf(f, __uint_as_float(w[i]), a[32 * cc + i] * r);
                }
            }
        } else {
            const long long tile = tc5_piece_tile(p, sk, !(sk == sf && x0 != bound[sf]), b, g);
            const float2 st = __ldcg(ml + tile * 128 + row);
            const float4 *src = reinterpret_cast<const float4 *>(p.ws_acc + tile * 128 * D) + half * (C / 4) * 128 + row;
            float4 v[C / 4];
#pragma unroll
            for (int k = 0; k < C / 4; ++k) v[k] = __ldcg(src + k * 128);
            if (st.x == -INFINITY) continue;
            rescale(st, r, f);
#pragma unroll
            for (int k = 0; k < C / 4; ++k) {
                a[4 * k] = fmaf(f, v[k].x, a[4 * k] * r);
                a[4 * k + 1] = fmaf(f, v[k].y, a[4 * k + 1] * r);
                a[4 * k + 2] = fmaf(f, v[k].z, a[4 * k + 2] * r);
                a[4 * k + 3] = fmaf(f, v[k].w, a[4 * k + 3] * r);
            }
        }
    }
    if (!row_ok) return;
    const float inv = lsum > 0.f ? 1.0f / lsum : 0.f;
    uint16_t *o = p.out + ((long long)(b + qi) * p.Hq + (long long)g * p.gq + (row % p.gq)) * D + half * C;
#pragma unroll
    for (int k = 0; k < C / 8; ++k)
        *reinterpret_cast<uint4 *>(o + 8 * k) =
            make_uint4(pack_bf16x2(a[8 * k] * inv, a[8 * k + 1] * inv),
                       pack_bf16x2(a[8 * k + 2] * inv, a[8 * k + 3] * inv),
                       pack_bf16x2(a[8 * k + 4] * inv, a[8 * k + 5] * inv),
                       pack_bf16x2(a[8 * k + 6] * inv, a[8 * k + 7] * inv));
}

static_assert(team_warps(16) * 16 == 128, "a tensor-memory piece tile is 8 slots of 16 rows");

// The softmax warps: thread t of the 256 takes row r = 32 (w % 4) + lane (TMEM lane r; w = t / 32) and
// keys 64 h .. 64 h + 63 of every tile, h = w / 4.  The two threads of a row (warps w and w + 4) hold the
// same running max: they exchange their tile max each tile; each keeps the sum of its own keys' weights.
// When a segment starts they write its Q tile (dims 64 h .. 64 h + 63 of row r) into tensor memory.
template <int D, int G>
__device__ void tc5_softmax_warps(const DecodeParams &p, const CtaLayout &lay, const Tc5Smem &m, uint32_t tmem,
                                  float *xch, const long long *bound, const int32_t *scan, int *sh,
                                  const float *wts, int nslots, uint32_t gen, int wp, bool adaptive)
{
    constexpr int KH = kTc5Keys / 2;  // keys of a half
    constexpr int DH = D / 2;         // dims of a half (of Q and of the output)
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int quarter = warp & 3, half = warp >> 2;
    const int row = 32 * quarter + lane;
    const uint32_t tlane = tmem + (uint32_t(32 * quarter) << 16);  // this warp's lane quarter
    const int qi = row / p.gq;                                      // query of the row within its entry
    const int home = sh[0];
    const float c = p.scale_log2;
    int s = 0;
    uint32_t ph = 0, j = 0, segs = 0;
    float mrun = -INFINITY, lrun = 0.f;
    bool row_ok = false;
    int shift = 0, u_first = 0;
    uint32_t meets = 0;  // exchanges with the row's other half so far (the same in both warps)
    uint32_t teams = 0;  // meetings of all softmax warps so far (the same in every one)
    // a wait that may give up: the kernel's error word, and out of the loop
    auto wait = [&](uint64_t *bar, uint32_t parity) {
        if (mbar_wait_bounded(bar, parity)) return true;
        if (lane == 0) flag_error(p.err, PKV_ERR_WAIT_TIMEOUT);
        return false;
    };
    auto meet_all = [&]() {
        __syncwarp();
        if (lane == 0) mbar_arrive(m.team);
        return wait(m.team, teams++ & 1u);
    };
    // give v to the row's other half and take its value (slots alternate by exchange, so a warp one
    // exchange ahead does not overwrite a value its partner has yet to read); false if the wait gave up
    auto exchange = [&](float v, float &other) {
        float *slot = xch + (meets & 1u) * 256u;
        slot[half * 128 + row] = v;
        __syncwarp();
        if (lane == 0) mbar_arrive(&m.pair[quarter]);
        if (!wait(&m.pair[quarter], meets++ & 1u)) return false;
        other = slot[(1 - half) * 128 + row];
        return true;
    };
    // A segment's Q tile into tensor memory (tile segs % 2: the tile before it was last read by the
    // segment before the previous one's scores, all of which were read back): this thread's 64 dims of
    // its row, zeros for rows that are not queries of the entry.
    auto write_q = [&](const UnitMeta &sg) {
        uint32_t w[32];
        if (qi < sg.cnt) {
            const uint4 *src = reinterpret_cast<const uint4 *>(
                p.q + ((long long)(sg.b + qi) * p.Hq + (long long)sg.g * p.gq + (row % p.gq)) * D + half * DH);
#pragma unroll
            for (int k = 0; k < DH / 8; ++k) {
                const uint4 v = __ldg(src + k);
                w[4 * k] = v.x;
                w[4 * k + 1] = v.y;
                w[4 * k + 2] = v.z;
                w[4 * k + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int k = 0; k < DH / 2; ++k) w[k] = 0u;
        }
        const uint32_t qa = tlane + kTc5QCol + (segs & 1u) * 64u + uint32_t(half * DH / 2);
        if constexpr (DH / 2 == 32) {
            tmem_st32(qa, w);
        } else {
            uint32_t w16[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) w16[k] = w[k];
            tmem_st16(qa, w16);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(m.qready);
        ++segs;
    };
    // the next segment's Q tile is already written: the first one before the loop, each later one at the
    // end of the segment before it
    bool q_early = false;
    if (wait(&m.mready[0], 0u)) {
        const UnitMeta f0 = m.metas[0];
        if (f0.b >= 0 && (f0.flags & kFirst)) {
            write_q(f0);
            q_early = true;
        }
    }
    for (;;) {
        if (!wait(&m.full[s], ph)) break;
        const UnitMeta mt = m.metas[s];
        if (mt.b < 0) break;
        const bool first = (mt.flags & kFirst) != 0;
        const int kvh = mt.g;  // hg = 1
        if (first) {
            row_ok = qi < mt.cnt;
            shift = (mt.cnt - 1) - qi;  // the row's query sees this many fewer of the entry's last keys
            mrun = -INFINITY;
            lrun = 0.f;
            u_first = mt.u;
            if (!q_early) write_q(mt);
            q_early = false;
        }
        const int tok0 = mt.u * kTc5Keys;
        const int valid = min(kTc5Keys, mt.L - tok0);
        const int lim = row_ok ? min(valid, mt.L - tok0 - shift) - KH * half : 0;  // keys of this half
        if (valid < kTc5Keys) {
            // V rows past the sequence's end hold anything (NaN included) and 0 * NaN is NaN: zero them,
            // once the V copy has landed
            if (!wait(&m.vfull[j % kTc5VSlots], (j / kTc5VSlots) & 1u)) break;
            uint8_t *vrows = m.vbase + size_t(j % kTc5VSlots) * tc5_vslot_bytes(lay);
            const int per_part = (kTc5Keys - valid) * 8, n = per_part * (D / 64);
            for (int i = t; i < n; i += 32 * kTc5SoftmaxWarps) {
                const int part = i / per_part, r = i - part * per_part;
                *reinterpret_cast<uint4 *>(vrows + part * kTc5SlabBytes + valid * 128 + r * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();  // for the tensor core
        }
        if (!wait(&m.sfull[j & 1u], (j >> 1) & 1u)) break;
        tc_fence_after();
        const uint32_t sbuf = tlane + (j & 1u) * 128u;  // the unit's score buffer (and then its weights)
        // raw scores s of the half's keys (at or past the row's bound: -inf); weights 2^(s c - m)
        float x[KH];
        {
            uint32_t r[KH];
            tmem_ld64(sbuf + uint32_t(KH * half), r);
            if (lim >= KH) {
#pragma unroll
                for (int i = 0; i < KH; ++i) x[i] = __uint_as_float(r[i]);
            } else {
#pragma unroll
                for (int i = 0; i < KH; ++i) x[i] = i < lim ? __uint_as_float(r[i]) : -INFINITY;
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&m.sfree[j & 1u]);  // the unit's K slot (and meta) may be reused
        float mx4[4] = {x[0], x[1], x[2], x[3]};
#pragma unroll
        for (int i = 4; i < KH; ++i) mx4[i & 3] = fmaxf(mx4[i & 3], x[i]);
        float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * c;  // c > 0
        float other;
        if (!exchange(mx, other)) break;
        mx = fmaxf(mx, other);  // the row's tile max: the same in both halves
        float alpha = 1.0f;
        bool resc = false;
        if (mx > mrun + kRescaleSlack) {  // also the row's first tile with a key (mrun = -inf)
            if (!first && mrun != -INFINITY) {
                alpha = ex2(mrun - mx);
                lrun *= alpha;
                resc = true;
            }
            mrun = mx;
        }
        // O's rows scaled in place (alpha = 1 for rows that keep their max), this thread's half of the
        // columns, once P(j - 1) V is in
        if (__any_sync(kFull, resc)) {
            if (!wait(&m.odone[(j - 1) & 1u], ((j - 1) >> 1) & 1u)) break;
            tc_fence_after();
#pragma unroll 1
            for (int cc = half * (D / 64); cc < (half + 1) * (D / 64); ++cc) {
                uint32_t r[32];
                tmem_ld32(tlane + kTc5OCol + cc * 32, r);
#pragma unroll
                for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                tmem_st32(tlane + kTc5OCol + cc * 32, r);
            }
        }
        // weights rounded to bf16 (the output product's operand), over the scores in this half's 32 columns
        // of the unit's buffer (both halves read their scores before the exchange); the row sum adds the fp32
        // weights (2^-inf = 0 for the masked keys; a row without any key so far takes m = 0 and gets zeros)
        {
            const float mneg = mrun == -INFINITY ? 0.f : -mrun;
            float ps[4] = {0.f, 0.f, 0.f, 0.f};
            uint32_t w[32];
#pragma unroll
            for (int k = 0; k < KH / 2; ++k) {
                const float p0 = ex2(fmaf(x[2 * k], c, mneg)), p1 = ex2(fmaf(x[2 * k + 1], c, mneg));
                ps[k & 3] += p0 + p1;
                w[k] = pack_bf16x2(p0, p1);
            }
            lrun += (ps[0] + ps[1]) + (ps[2] + ps[3]);
            tmem_st32(sbuf + 32u * half, w);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&m.pfull[j & 1u]);

        if (mt.flags & kLast) {  // the segment's part in this slice ends: O once its last product is done
            // First the next segment's Q tile, so that its first scores run during this epilogue: the
            // next unit's meta, written before its K copy is issued (the producer issues it without
            // waiting for anything past this unit's weights)
            {
                const int sn = s + 1 == p.nst ? 0 : s + 1;
                if (!wait(&m.mready[sn], s + 1 == p.nst ? ph ^ 1u : ph)) break;
                const UnitMeta nx = m.metas[sn];
                if (nx.b >= 0 && (nx.flags & kFirst)) {
                    write_q(nx);
                    q_early = true;
                }
            }
            if (!wait(&m.odone[j & 1u], (j >> 1) & 1u)) break;
            tc_fence_after();
            float lother;
            if (!exchange(lrun, lother)) break;
            const float L = lrun + lother;  // the row's sum (both halves share the max)
            const int piece = mt.u - u_first + 1;
            // this thread's columns of the row: [half D / 2, (half + 1) D / 2)
            if (piece == mt.n) {  // the whole segment ran here: bf16 output
                const float inv = L > 0.f ? 1.0f / L : 0.f;
                uint16_t *orow = p.out + ((long long)(mt.b + qi) * p.Hq + (long long)kvh * p.gq + (row % p.gq)) * D;
#pragma unroll 1
                for (int cc = half * (D / 64); cc < (half + 1) * (D / 64); ++cc) {
                    uint32_t r[32];
                    tmem_ld32(tlane + kTc5OCol + cc * 32, r);
                    if (row_ok) {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            *reinterpret_cast<uint4 *>(orow + cc * 32 + 8 * k) = make_uint4(
                                pack_bf16x2(__uint_as_float(r[8 * k]) * inv, __uint_as_float(r[8 * k + 1]) * inv),
                                pack_bf16x2(__uint_as_float(r[8 * k + 2]) * inv, __uint_as_float(r[8 * k + 3]) * inv),
                                pack_bf16x2(__uint_as_float(r[8 * k + 4]) * inv, __uint_as_float(r[8 * k + 5]) * inv),
                                pack_bf16x2(__uint_as_float(r[8 * k + 6]) * inv, __uint_as_float(r[8 * k + 7]) * inv));
                    }
                }
            } else {
                // a piece: (m, l, acc) of every row into the slice's piece tile (tc5_piece_tile); the CTA
                // whose piece completes the (entry, kv head) count merges all 128 rows
                const long long x0 = (long long)p.nhg * scan[mt.b] + (long long)mt.g * mt.n;
                const bool firstseg = u_first > 0 || x0 == bound[mt.slice];
                const long long tile = tc5_piece_tile(p, mt.slice, firstseg, mt.b, mt.g);
                float4 *dst = reinterpret_cast<float4 *>(p.ws_acc + tile * 128 * D) + row;
#pragma unroll 1
                for (int cc = half * (D / 64); cc < (half + 1) * (D / 64); ++cc) {
                    uint32_t r[32];
                    tmem_ld32(tlane + kTc5OCol + cc * 32, r);
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        dst[(cc * 8 + k) * 128] =
                            make_float4(__uint_as_float(r[4 * k]), __uint_as_float(r[4 * k + 1]),
                                        __uint_as_float(r[4 * k + 2]), __uint_as_float(r[4 * k + 3]));
                }
                if (half == 0) reinterpret_cast<float2 *>(p.ws_ml)[tile * 128 + row] = make_float2(mrun, L);
                // the whole piece is written before it is counted in: every thread's stores precede the
                // meeting (release / acquire at CTA scope), and the counting thread's fence at device scope
                // carries them (fences are cumulative)
                if (!meet_all()) break;
                if (t == 0) {
                    __threadfence();
                    sh[5] = arrive_last(p.ws_count + ((long long)mt.b * p.Hkv + kvh) * p.sub, gen, uint32_t(piece),
                                        uint32_t(mt.n), p.err);
                }
                if (!meet_all()) break;
                if (sh[5]) {
                    __threadfence();
                    tc5_merge<D>(p, bound, slice_of(bound, nslots, x0), slice_of(bound, nslots, x0 + mt.n - 1),
                                 mt.slice, mrun, L, tlane + kTc5OCol + uint32_t(half * (D / 2)), x0, mt.g, mt.b, row,
                                 half, row_ok, qi);
                }
            }
            tc_fence_before();  // the reads of O come before the next segment's first product overwrites it
        }
        if ((mt.flags & kSliceEnd) && adaptive && t == 0) {
            // balance record for the next call (as the regular consumers leave it)
            const bool own = mt.slice == home;
            const float us = float(global_ns() - *reinterpret_cast<const volatile unsigned long long *>(sh + 2)) * 1e-3f;
            p.ws_bal->weight[wp][mt.slice] = own ? wts[mt.slice] : 0.f;
            p.ws_bal->elapsed[wp][mt.slice] = own ? fmaxf(us, 1e-3f) : 0.f;
            p.ws_bal->tag[wp][mt.slice] = gen ^ kTableMagic;
        }
        ++j;
        if (++s == p.nst) {
            s = 0;
            ph ^= 1u;
        }
    }
    tc_fence_before();
}

// ------------------------------------------------------------------ main kernel
// Block: p.cons consumer warps and one producer warp (warp p.cons).  Consumer
// warp w takes kv head w / sub of the group and, per unit, either the TW-token
// slice w % sub (QS false: a unit is TW * sub tokens) or all TW tokens for
// its own qn queries w % sub of the entry's (QS true, hg = 1: the query-split
// CTA for long runs of new tokens, where the entry's up to sub * qn queries
// share every K/V tile).  TC5 (with QS): the same entries on the tensor-memory
// consumers (see tc5_softmax_warps).
template <int D, int G, bool FP8, bool QS, bool TC5 = false>
__global__ void __launch_bounds__(TC5 ? (kTc5Consumers + 1) * 32 : (team_warps(G) + 1) * 32, 1)
    paged_decode_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                        const DecodeParams p)
{
    static_assert(!TC5 || (QS && !FP8 && G == 16 && (D == 64 || D == 128)), "tensor-memory CTAs: bf16 query-split");
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int ES = FP8 ? 1 : 2;  // bytes per cached element
    const int qslots = one_q_buffer_ok(G, FP8, QS, TC5) ? p.qslots : 2;
    const CtaLayout lay = cta_layout(D, G, ES, p.hg, p.sub, p.nst, p.B, QS, TC5, qslots);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    uint8_t *stage0 = smem;
    uint8_t *qbuf = smem + lay.off_q;
    float *comb = reinterpret_cast<float *>(smem + lay.off_comb);
    UnitMeta *metas = reinterpret_cast<UnitMeta *>(smem + lay.off_meta);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + lay.off_bar);  // [nst] stage loaded (tx count)
    uint64_t *empty = full + p.nst;                                     // [nst] stage released by consumers
    uint64_t *qfull = empty + p.nst;                                    // [2] q rows loaded
    uint64_t *qempty = qfull + 2;                                       // [2] q rows taken by consumers
    uint64_t *cfull = qempty + 2;                                       // states written for a combine
    uint64_t *cfree = cfull + 1;                                        // combine buffer read again
    long long *bound = reinterpret_cast<long long *>(smem + lay.off_bound);
    float *wts = reinterpret_cast<float *>(smem + lay.off_wts);
    float *red = reinterpret_cast<float *>(smem + lay.off_red);
    // [0] own slice, [2..3] its start time, [4] tensor-memory address (TC5), [5] a piece completed its
    // segment (TC5)
    int *sh = reinterpret_cast<int *>(smem + lay.off_sh);
    int32_t *scan = reinterpret_cast<int32_t *>(smem + lay.off_scan);
    uint64_t *tc5_bar = cfree + 1;  // TC5: sfull[2], sfree[2], pfull[2], odone[2], drain, pair[4], team, qready
    uint64_t *vfull = tc5_bar + 15;        // TC5: [kTc5VSlots] a V slot loaded
    uint64_t *vempty = vfull + kTc5VSlots;  // TC5: [kTc5VSlots] a V slot released
    uint64_t *mready = vempty + kTc5VSlots;  // TC5: [nst] a K slot's meta written (before its copy lands)

    if (threadIdx.x == 32 * p.cons) {  // none of this reads what the previous kernel writes
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
        // TC5: a stage and a Q slot are released by one tcgen05.commit of the MMA warp
        const uint32_t releases = TC5 ? 1u : uint32_t(p.cons);
        for (int i = 0; i < p.nst; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], releases);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&qfull[i], 1);
            mbar_init(&qempty[i], releases);
        }
        mbar_init(cfull, uint32_t(p.cons - p.hg));  // the non-leading warps' states
        mbar_init(cfree, uint32_t(p.hg));           // read again by the leaders
        if constexpr (TC5) {
            for (int i = 0; i < 2; ++i) {                   // [i]: of a unit j with j % 2 == i
                mbar_init(&tc5_bar[i], 1);                  // scores computed
                mbar_init(&tc5_bar[2 + i], kTc5SoftmaxWarps);  // scores read
                mbar_init(&tc5_bar[4 + i], kTc5SoftmaxWarps);  // weights written
                mbar_init(&tc5_bar[6 + i], 1);              // output product done
            }
            mbar_init(&tc5_bar[8], 1);                      // every product done (before TMEM is freed)
            for (int i = 0; i < 4; ++i) mbar_init(&tc5_bar[9 + i], 2);  // the two warps of lane quarter i met
            mbar_init(&tc5_bar[13], kTc5SoftmaxWarps);      // all softmax warps met
            mbar_init(&tc5_bar[14], kTc5SoftmaxWarps);      // a segment's Q tile written
            for (int i = 0; i < kTc5VSlots; ++i) {
                mbar_init(&vfull[i], 1);
                mbar_init(&vempty[i], 1);
            }
            for (int i = 0; i < p.nst; ++i) mbar_init(&mready[i], 1);
        }
        fence_barrier_init();
    }
    if constexpr (TC5)
        if (warp == kTc5SoftmaxWarps) tmem_alloc(reinterpret_cast<uint32_t *>(sh + 4), kTc5Cols);
    griddep_launch_dependents();  // lets the next kernel in the stream get scheduled; it waits for this grid
    griddep_wait();               // inputs may come from the previous kernel in the stream

    // Slices: one per SM id, sized by measured finishing times (adaptive), or one per CTA (fixed).
    const bool adaptive = p.num_workers == 0;
    int nslots = int(gridDim.x);
    if (adaptive) nslots = int(min(nsmid(), unsigned(kMaxSlots)));
    const uint32_t epoch = __ldcg(&p.ws_bal->epoch);  // the workspace's control block: this call's number
    const uint32_t gen = epoch + 1u;                   // tags of this call; zero-filled words never match
    const int wp = int(gen & 1u);                      // this call writes one half of the balance table
    const unsigned my_sm = smid();
    // The set-up splits in two parts that run at the same time, each about two memory round trips
    // long.  The consumer warps (threads 0 .. 32 cons - 1, their own barrier) issue the control
    // block, balance entries and context lengths together, then scan and partition.  The producer
    // warp's lane 0 claims this SM id's slice (an exchange: the first CTA of this call to run on the
    // SM id finds another call's tag there) and warms L2 from the hint; both need the call number
    // first, and the hint a block-table entry after it.
    const int nset = 32 * p.cons;
    if (warp == p.cons) {
        if (lane == 0) {
            const uint32_t stamp = __ldcg(&p.ws_bal->stamp);
            const bool hint = p.num_workers == 0 && !p.row_seq && my_sm < unsigned(kMaxSlots);
            int4 h0 = make_int4(-1, -1, -1, -1), h1 = make_int4(-1, -1, -1, -1);
            if (hint) {
                h0 = __ldcg(&p.ws_bal->hint[my_sm][0]);
                h1 = __ldcg(&p.ws_bal->hint[my_sm][1]);
            }
            unsigned long long home_word = static_cast<unsigned long long>(gen) << 32;
            if (adaptive && int(my_sm) < nslots)
                home_word = atomicExch(&p.ws_bal->claim[my_sm], (static_cast<unsigned long long>(gen) << 32) | 1ull);
            // Warm L2 with up to kHintUnits units from the first copy this SM id's slice made in the
            // previous call on the workspace, if the sequence's table still maps that block (then
            // these are rows this call reads).
            if (hint && h0.z == (int32_t(epoch) ^ kHintMagic) && h0.w >= 0 && h0.w < p.B && h1.x >= 0 &&
                h1.x < p.max_blocks && h0.x >= 0 && h0.x < p.NB * p.bs && h0.y >= 0 && h0.y + p.hg <= p.Hkv &&
                __ldg(p.block_tables + (long long)h0.w * p.max_blocks + h1.x) == (h0.x >> p.log2_bs)) {
                const int32_t in_block = h0.x & (p.bs - 1);
                // rows of the block the sequence holds now (one decode step later: one more)
                const int32_t held = min(p.bs, h1.y + 1 - h1.x * p.bs);
                for (int i = 0; i < kHintUnits && in_block + i * p.toks < held && in_block + (i + 1) * p.toks <= p.bs;
                     ++i) {
                    tma_prefetch_4d(&kmap, 0, h0.x + i * p.toks, 0, h0.y);
                    tma_prefetch_4d(&vmap, 0, h0.x + i * p.toks, 0, h0.y);
                }
            }
            const bool ctl_ok = stamp == (epoch ^ kEpochMagic) || (epoch == 0u && stamp == 0u);
            if (!ctl_ok && blockIdx.x == 0) flag_error(p.err, PKV_ERR_WORKSPACE);
            int home = -1;
            if (!adaptive)
                home = int(blockIdx.x);
            else if (uint32_t(home_word >> 32) != gen)
                home = int(my_sm);
            sh[0] = home;
        }
    } else {
        const BalanceIn bal_in = load_balance(p, adaptive, nslots, nset);
        // the query count of this thread's first entry to check for zeros below, loaded with the rest
        const long long b_first = blockIdx.x + (long long)threadIdx.x * gridDim.x;
        const int rows_first = p.row_cnt && b_first < p.B ? __ldg(p.row_cnt + b_first) : p.qn;
        unit_prefix_scan(p, scan, reinterpret_cast<int32_t *>(smem), nset);
        const long long T = (long long)p.nhg * scan[p.B];
        // Entries without units (L == 0, or a rejected length) get zeros in their query rows; CTAs
        // share the job (CTA c takes entries c, c + grid, ...), a set-up thread checks one of them at a
        // time, and a warp zeroes the rows of its threads' entries together.
        for (long long k0 = 0; blockIdx.x + k0 * gridDim.x < p.B; k0 += nset) {
            const long long b = blockIdx.x + (k0 + threadIdx.x) * gridDim.x;
            int rows = 0;
            if (b < p.B && scan[b + 1] == scan[b]) {
                if (p.slot_out) p.slot_out[b] = -1;  // fused store: nothing stored
                rows = k0 == 0 ? rows_first : (p.row_cnt ? __ldg(p.row_cnt + b) : p.qn);
            }
            for (unsigned zm = __ballot_sync(kFull, rows > 0); zm; zm &= zm - 1) {
                const int l = __ffs(zm) - 1;
                const long long bz = __shfl_sync(kFull, b, l);
                const int nz = __shfl_sync(kFull, rows, l) * p.Hq * D / 8;
                uint4 *o = reinterpret_cast<uint4 *>(p.out + bz * p.qstride * p.Hq * D);
                for (int i = lane; i < nz; i += 32) o[i] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        if (p.per_segment) {
            // slice i = segment (entry i / nhg, group i % nhg), whole: the grid has one CTA per segment
            for (int i = threadIdx.x; i <= nslots; i += nset) {
                long long x = T;
                if (i < nslots && i < p.B * p.nhg) {
                    const int b = i / p.nhg, g = i - b * p.nhg;
                    x = (long long)p.nhg * scan[b] + (long long)g * (scan[b + 1] - scan[b]);
                }
                bound[i] = x;
            }
            setup_sync(nset);
        } else {
            build_partition(p, gen, adaptive, nslots, T, bound, wts, red, bal_in, nset);
        }
    }
    if constexpr (TC5) tc_fence_before();
    __syncthreads();
    if constexpr (TC5) tc_fence_after();

    if (warp == p.cons) {
        // ============================== producer warp ==============================
        const uint64_t policy = policy_evict_first();
        const uint32_t box_bytes = uint32_t(p.boxtok * p.hg * D * ES);
        uint32_t kk = 0, segs = 0;  // units issued, q-ring uses
        uint32_t vunits = 0;        // TC5: V tiles issued
        int rs = 0;                 // ring slot of unit kk (kk % nst, kept without a division)
        uint32_t rph = 0;           // parity of that slot's use (kk / nst) & 1
        bool dead = false;
        int slice = sh[0];
        if (slice < 0 && adaptive) slice = claim_leftover(p, gen, bound, nslots, wp, false);
        while (slice >= 0 && !dead) {
            const long long lo = bound[slice], hi = bound[slice + 1];
            if (lane == 0 && slice == sh[0])
                *reinterpret_cast<unsigned long long *>(sh + 2) = global_ns();
            const long long nunits = hi - lo, nboxes = nunits * p.nbox;
            // TC5: the slice's units from its last (entry, kv head) segment on, then from its start: the
            // part of that segment which continues in the next slice (and the part of the first segment
            // which continued from the previous one) finishes early, so the merge of a split segment
            // happens amid the run, not at its end.  Segments stay whole and in order (and a merge folds
            // its pieces in slice order), so the results are unchanged.
            long long rot = 0;
            if constexpr (TC5) {
                if (nunits > 1) {
                    const Walker last = walker_locate(scan, p.B, p.nhg, hi - 1);
                    rot = max(0LL, hi - 1 - last.u - lo);
                }
            }
            auto unit_at = [&](long long k) {  // unit processed k-th
                const long long y = k + rot;
                return lo + (y >= nunits ? y - nunits : y);
            };
            // Block-table prefetch, 32 boxes per batch: lane j of `cur` holds the entry (and the
            // context length) of box kb + j; `nxt` is loaded one batch ahead.  Two register sets,
            // because the scoreboard tracks a register for the whole warp.
            Walker iw = nunits > 0 ? walker_locate(scan, p.B, p.nhg, lo + rot) : Walker{0, 0, 0, 1};
            int32_t cur_e = -1, cur_L = 0, cur_c = 1, nxt_e = -1, nxt_L = 0, nxt_c = 1;
            auto prefetch_batch = [&](long long kb) {  // boxes [kb, kb + 32) -> nxt, one per lane
                const long long x = kb + lane;
                if (x < nboxes) {
                    const Walker mine = walker_locate(scan, p.B, p.nhg, unit_at(x >> p.lg_nbox));
                    const int32_t pos = mine.u * p.toks + int32_t(x & (p.nbox - 1)) * p.boxtok;
                    // The entry is only used for pos < L, where pos / bs < max_blocks (lengths
                    // beyond the table were rejected by the scan); clamping keeps the load in
                    // the row and lets it go out together with the length's.
                    const int32_t blk = min(pos >> p.log2_bs, p.max_blocks - 1);
                    nxt_L = __ldg(p.context_lens + mine.b);
                    nxt_c = p.row_cnt ? __ldg(p.row_cnt + mine.b) : p.qn;
                    const int32_t trow = p.row_seq ? __ldg(p.row_seq + mine.b) : mine.b;
                    nxt_e = __ldg(p.block_tables + (long long)trow * p.max_blocks + blk);
                }
            };
            // TC5: the query rows of segment w into L2 (the softmax warps load them into tensor memory at
            // the end of the segment before): 8 qn queries x gq heads of kv head g, D values each, as
            // 128-byte lines, lane-strided (plain prefetches: they do not queue behind the copies)
            auto prefetch_q = [&](const Walker &w) {
                const int nq = min(team_warps(G) * p.qn, p.B - w.b);
                const int lines = p.gq * D * 2 / 128;
                for (int i = lane; i < nq * lines; i += 32) {
                    const int r = i / lines, c = i - r * lines;
                    prefetch_l2(reinterpret_cast<const uint8_t *>(
                                    p.q + ((long long)(w.b + r) * p.Hq + (long long)w.g * p.gq) * D) +
                                c * 128);
                }
            };
            if (nunits > 0) {
                prefetch_batch(0);
                cur_e = nxt_e;
                cur_L = nxt_L;
                cur_c = nxt_c;
            }
            for (long long k = 0; k < nunits; ++k) {
                const long long kb0 = k * p.nbox;  // nbox is a power of two <= 32: batches start on units
                if ((kb0 & 31) == 0 && k > 0) {
                    cur_e = nxt_e;
                    cur_L = nxt_L;
                    cur_c = nxt_c;
                    if (kb0 + 32 < nboxes) prefetch_batch(kb0 + 32);
                }
                const int s = rs;
                if (kk >= uint32_t(p.nst) && !mbar_wait_bounded(&empty[s], rph ^ 1u)) {
                    dead = true;
                    break;
                }
                const int src = int(kb0 & 31);
                const int32_t len = __shfl_sync(kFull, cur_L, src);
                const int32_t cnt = __shfl_sync(kFull, cur_c, src);
                const int32_t e = __shfl_sync(kFull, cur_e, (src + lane) & 31);  // lane j: box j's entry
                const long long x = unit_at(k);
                const int flags = ((x == lo || iw.u == 0) ? kFirst : 0) |
                                  ((x == hi - 1 || iw.u == iw.n - 1) ? kLast : 0) |
                                  (k == nunits - 1 ? kSliceEnd : 0);
                if (flags & kFirst) {  // q rows of this (b, group) for the consumers
                    const int qs = int(segs & uint32_t(qslots - 1));
                    const uint32_t quse = segs >> (qslots - 1);  // earlier uses of the buffer
                    if (!TC5 && quse > 0 && !mbar_wait_bounded(&qempty[qs], (quse - 1) & 1u)) {
                        dead = true;
                        break;
                    }
                    if constexpr (TC5) {
                        // the consumers load the entry's Q tile themselves (into tensor memory); its rows
                        // were warmed in L2 when the segment before it was issued (here: a slice's first)
                        if (k == 0) prefetch_q(iw);
                    } else if (p.qn == 1 && !QS) {  // the group's G * hg query rows are contiguous
                        const uint32_t qb = uint32_t(p.hg * G * D * 2);
                        if (lane == 0) {
                            mbar_arrive_expect_tx(&qfull[qs], qb);
                            bulk_load(qbuf + qs * lay.q_bytes,
                                      p.q + ((long long)iw.b * p.Hq + (long long)iw.g * p.hg * G) * D, qb,
                                      &qfull[qs]);
                        }
                    } else {
                        // cnt queries: kv head h's virtual heads i * gq .. i * gq + gq - 1 come from row
                        // b * qstride + i; one copy of gq rows per (h, i < cnt), lane t copying pair t
                        // (the slots of virtual heads past cnt * gq are not loaded: the consumers zero them).
                        // Query-split (hg = 1): query i is virtual head (i % qn) * gq.. of warp i / qn,
                        // whose G rows start at (i / qn) * G = (i - i % qn) * gq: the same offset i * gq.
                        if (lane == 0) mbar_arrive_expect_tx(&qfull[qs], uint32_t(p.hg * cnt * p.gq * D * 2));
                        __syncwarp();
                        for (int t = lane; t < p.hg * cnt; t += 32) {
                            const int hh = t / cnt, qi = t - hh * cnt;
                            bulk_load(qbuf + qs * lay.q_bytes + size_t((hh * G + qi * p.gq) * D) * 2,
                                      p.q + (((long long)iw.b * p.qstride + qi) * p.Hq +
                                             (long long)(iw.g * p.hg + hh) * p.gq) * D,
                                      uint32_t(p.gq * D * 2), &qfull[qs]);
                        }
                    }
                    ++segs;
                }
                // box j of the unit: tokens [pos, pos + boxtok) of one physical block
                const int32_t pos = iw.u * p.toks + lane * p.boxtok;
                int32_t row = -1;
                if (lane < p.nbox && pos < len) {
                    if (e >= 0 && e < p.NB)
                        row = e * p.bs + (pos & (p.bs - 1));
                    else
                        flag_error(p.err, PKV_ERR_BLOCK_RANGE);
                }
                const uint32_t nrows = __popc(__ballot_sync(kFull, row >= 0));
                // fused store: the cache row of the sequence's new token (position L - 1), if this unit
                // holds it (-1 where its block id was rejected)
                int32_t newrow = -1;
                const int32_t u0 = iw.u * p.toks;
                if (p.k_new && len - 1 >= u0 && len - 1 < u0 + p.toks) {
                    const int32_t off = len - 1 - u0;
                    const int32_t rb = __shfl_sync(kFull, row, off >> (__ffs(p.boxtok) - 1));
                    newrow = rb >= 0 ? rb + (off & (p.boxtok - 1)) : -1;
                    if (lane == 0 && iw.g == 0 && p.slot_out) p.slot_out[iw.b] = newrow;
                }
                uint8_t *st = stage0 + s * lay.stage_bytes;
                if (lane == 0) {
                    UnitMeta &mt = metas[s];
                    mt.b = iw.b;
                    mt.g = iw.g;
                    mt.u = iw.u;
                    mt.n = iw.n;
                    mt.L = len;
                    mt.flags = flags;
                    mt.slice = slice;
                    mt.cnt = cnt;
                    mt.newrow = newrow;
                    if constexpr (TC5) mbar_arrive(&mready[s]);  // the meta, for a look ahead
                    // TC5: full[s] counts the K half only; the V half has barriers of its own
                    mbar_arrive_expect_tx(&full[s], (TC5 ? 1u : 2u) * nrows * box_bytes);
                }
                __syncwarp();
                if (k == 0 && lane == 0 && adaptive && !p.row_seq && slice == sh[0] && row >= 0 &&
                    my_sm < unsigned(kMaxSlots)) {
                    p.ws_bal->hint[my_sm][0] = make_int4(row, iw.g * p.hg, int32_t(gen) ^ kHintMagic, iw.b);
                    p.ws_bal->hint[my_sm][1] = make_int4((iw.u * p.toks) >> p.log2_bs, len, 0, 0);
                }
                if constexpr (TC5) {
                    // K now (its half of the stage is free once the previous scores of the slot are done);
                    // V once the slot's previous output product is done
                    if (row >= 0) tma_load_4d(st + lane * box_bytes, &kmap, 0, row, 0, iw.g, &full[s], policy);
                    const uint32_t vs = vunits % kTc5VSlots;
                    if (vunits >= kTc5VSlots && !mbar_wait_bounded(&vempty[vs], ((vunits / kTc5VSlots) - 1) & 1u)) {
                        ++kk;  // its K copy is on the way
                        dead = true;
                        break;
                    }
                    if (lane == 0) mbar_arrive_expect_tx(&vfull[vs], nrows * box_bytes);
                    __syncwarp();
                    if (row >= 0)
                        tma_load_4d(smem + lay.off_v + vs * align_up(lay.kv_bytes, 1024) + lane * box_bytes, &vmap, 0,
                                    row, 0, iw.g, &vfull[vs], policy);
                    ++vunits;
                } else if (row >= 0) {  // box j: lane j, one copy per cache
                    tma_load_4d(st + lane * box_bytes, &kmap, 0, row, 0, iw.g * p.hg, &full[s], policy);
                    tma_load_4d(st + lay.kv_bytes + lane * box_bytes, &vmap, 0, row, 0, iw.g * p.hg, &full[s],
                                policy);
                }
                ++kk;
                if (++rs == p.nst) {
                    rs = 0;
                    rph ^= 1u;
                }
                if (k + 1 < nunits) {
                    if (rot > 0 && k + 1 == nunits - rot)
                        iw = walker_locate(scan, p.B, p.nhg, lo);  // from the slice's last unit to its first
                    else
                        walker_advance(iw, scan, p.nhg, p.B);
                    if constexpr (TC5)
                        if (flags & kLast) prefetch_q(iw);  // the next segment's query rows
                }
                if (k == 0 && nboxes > 32) prefetch_batch(32);  // after the first copies are on their way
            }
            slice = (adaptive && !dead) ? claim_leftover(p, gen, bound, nslots, wp, true) : -1;
        }
        if (!dead) {  // end-of-work marker
            if (kk < uint32_t(p.nst) || mbar_wait_bounded(&empty[rs], rph ^ 1u)) {
                if (lane == 0) {
                    metas[rs].b = -1;
                    if constexpr (TC5) mbar_arrive(&mready[rs]);
                    mbar_arrive(&full[rs]);
                }
                ++kk;
            } else {
                dead = true;
            }
        }
        if (dead && lane == 0) flag_error(p.err, PKV_ERR_WAIT_TIMEOUT);
        // let every copy this warp started land before the CTA can retire
        for (uint32_t i = kk > uint32_t(p.nst) ? kk - uint32_t(p.nst) : 0u; i < kk; ++i)
            mbar_wait_bounded(&full[i % uint32_t(p.nst)], (i / uint32_t(p.nst)) & 1u);
        if constexpr (TC5)
            for (uint32_t i = vunits > uint32_t(kTc5VSlots) ? vunits - uint32_t(kTc5VSlots) : 0u; i < vunits; ++i)
                mbar_wait_bounded(&vfull[i % kTc5VSlots], (i / kTc5VSlots) & 1u);
        // Count this CTA in: every thread of it read the control block long ago (the fence orders
        // those reads before the count).  The CTA that completes the count leaves the block ready
        // for the next call.  This is the producer's last act, while the consumers still work
        // through the stages in flight, so the round trip is off the kernel's critical path.
        if (lane == 0) {
            __threadfence();
            if (atomicAdd(&p.ws_bal->done, 1u) == gridDim.x - 1) {
                p.ws_bal->done = 0u;
                p.ws_bal->epoch = epoch + 1u;
                p.ws_bal->stamp = (epoch + 1u) ^ kEpochMagic;
            }
        }
        return;
    }

    // ============================== consumer warps ==============================
    if constexpr (TC5) {
        const uint32_t tmem = uint32_t(sh[4]);
        Tc5Smem tm;
        tm.metas = metas;
        tm.full = full;
        tm.empty = empty;
        tm.vfull = vfull;
        tm.vempty = vempty;
        tm.mready = mready;
        tm.sfull = tc5_bar;
        tm.sfree = tc5_bar + 2;
        tm.pfull = tc5_bar + 4;
        tm.odone = tc5_bar + 6;
        tm.drain = tc5_bar + 8;
        tm.pair = tc5_bar + 9;
        tm.team = tc5_bar + 13;
        tm.qready = tc5_bar + 14;
        tm.vbase = smem + lay.off_v;
        tm.stage_addr = smem_u32(stage0);
        tm.v_addr = smem_u32(smem + lay.off_v);
        if (warp == kTc5SoftmaxWarps)
            tc5_mma_warp<D>(p, lay, tm, tmem);
        else
            tc5_softmax_warps<D, G>(p, lay, tm, tmem, comb, bound, scan, sh, wts, nslots, gen, wp, adaptive);
        named_barrier(2, 32 * kTc5Consumers);  // every tensor-memory access of the CTA is done
        if (warp == kTc5SoftmaxWarps) {
            tc_fence_after();
            tmem_dealloc(tmem, kTc5Cols);
        }
        return;
    } else {
    using TC = Tc<D, FP8, QS, (G > 8 ? 2 : 1)>;
    const int h = warp / p.sub, j = warp - h * p.sub;  // kv head in the group, slice of the unit or queries
    const int jt = QS ? 0 : j;                         // token slice of the unit
    const int jq = QS ? j : 0;                         // block of qn queries of the entry
    const int g8 = lane >> 2, r4 = lane & 3;           // fragment row group and column pair of the thread
    const int home = sh[0];
    LaneOffsets<D, FP8, QS> off;
    lane_offsets<D, FP8, QS>(off, lane, jt, h, p.hg, p.boxtok);
    const uint32_t stage_addr = smem_u32(stage0);
    constexpr int HR = TC::HR;  // halves of the MMA tile's rows that hold virtual heads
    // several queries per stream: the query of row g8 + 8 hr sees shift[hr] fewer of the entry's last
    // tokens (set per entry: the entry's last query sees them all)
    int shift[HR];
    int nvh = G;  // virtual heads of this warp that are queries (the rest are zero rows)
    uint32_t kk = 0, segs = 0, combs = 0;
    int s = 0;           // ring slot of stage kk
    uint32_t sph = 0;    // parity of its use
    uint32_t qa[TC::KS][2 * HR];
    float o[TC::MT][HR][4];
    float m[HR], l[HR];
#pragma unroll
    for (int hr = 0; hr < HR; ++hr) {
        shift[hr] = 0;
        m[hr] = -INFINITY;
        l[hr] = 0.f;
    }
    float ksc = p.scale_log2;
    float vsc = 1.0f;  // E4M3 caches: the kv head's V scale, applied in the final division
    // fused store: this lane's 8 bytes of the new K / V row (4 bf16 elements, or 8 E4M3 codes)
    uint2 kn = make_uint2(0u, 0u), vn = make_uint2(0u, 0u);
    // 16-row tiles hold twice the accumulators: their registers are short, so they load the new row only
    // when its tile comes (one load's latency, once per segment of a decode with more than 8 query heads
    // per kv head), instead of holding it from the segment's start
    constexpr bool kLateNewRow = TC::HR == 2;
    auto load_new_row = [&](const UnitMeta &m_, uint2 &k2, uint2 &v2) {
        const long long row0 = ((long long)m_.b * p.Hkv + m_.g * p.hg + h) * D;
        if constexpr (!FP8) {
            k2 = __ldg(reinterpret_cast<const uint2 *>(p.k_new + row0 + lane * 4));
            v2 = __ldg(reinterpret_cast<const uint2 *>(p.v_new + row0 + lane * 4));
        } else {  // quantised as pkv_kv_store_fp8 does
            const int kvh = m_.g * p.hg + h;
            k2 = quantise8_e4m3(__ldg(reinterpret_cast<const uint4 *>(p.k_new + row0 + lane * 8)),
                                __ldg(p.k_scale + kvh));
            v2 = quantise8_e4m3(__ldg(reinterpret_cast<const uint4 *>(p.v_new + row0 + lane * 8)),
                                __ldg(p.v_scale + kvh));
        }
    };
    int u_first = 0;
    for (;;) {
        if (!mbar_wait_bounded(&full[s], sph)) {
            if (lane == 0) flag_error(p.err, PKV_ERR_WAIT_TIMEOUT);
            break;
        }
        const UnitMeta mt = metas[s];
        if (mt.b < 0) break;
        if (mt.flags & kFirst) {
            const int qs = int(segs & uint32_t(qslots - 1));
            const uint32_t quse = segs >> (qslots - 1);
            ksc = p.scale_log2;  // E4M3 caches: the kv head's K scale joins the score scale
            if constexpr (FP8) {
                ksc *= __ldg(p.k_scale + mt.g * p.hg + h);
                vsc = __ldg(p.v_scale + mt.g * p.hg + h);
            }
            if (!mbar_wait_bounded(&qfull[qs], quse & 1u)) {
                if (lane == 0) flag_error(p.err, PKV_ERR_WAIT_TIMEOUT);
                break;
            }
            if constexpr (!QS && !kLateNewRow) {
                // the segment's new K/V row, used at its last tile (its load's latency hides until then)
                if (p.k_new && lane < TC::ROWB / 8) load_new_row(mt, kn, vn);
            }
            nvh = max(0, min(p.qn, mt.cnt - jq * p.qn)) * p.gq;
            // Q operand fragments of rows g8 (qa[ks][0], [1]) and g8 + 8 (qa[ks][2], [3]; HR = 2), zero
            // past nvh: k-step ks holds dims 16 ks + 2 r4 (+1) and 16 ks + 8 + 2 r4 (+1) (bf16), or
            // 16 ks + 4 r4 (+1) and 16 ks + 4 r4 + 2 (+3) (E4M3 order)
            const uint16_t *qw =
                reinterpret_cast<const uint16_t *>(qbuf + qs * lay.q_bytes) + (h * (QS ? p.sub : 1) + jq) * G * D;
#pragma unroll
            for (int hr = 0; hr < HR; ++hr) {
                const int row = g8 + 8 * hr;
                shift[hr] = (mt.cnt - 1) - (jq * p.qn + row / p.gq);
                const uint16_t *qr = qw + row * D;
#pragma unroll
                for (int ks = 0; ks < TC::KS; ++ks) {
                    qa[ks][2 * hr] = qa[ks][2 * hr + 1] = 0u;
                    if (row < nvh) {
                        if constexpr (!FP8) {
                            qa[ks][2 * hr] = *reinterpret_cast<const uint32_t *>(qr + 16 * ks + 2 * r4);
                            qa[ks][2 * hr + 1] = *reinterpret_cast<const uint32_t *>(qr + 16 * ks + 8 + 2 * r4);
                        } else {
                            const uint2 w = *reinterpret_cast<const uint2 *>(qr + 16 * ks + 4 * r4);
                            qa[ks][2 * hr] = f16x2_sat(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u));
                            qa[ks][2 * hr + 1] =
                                f16x2_sat(__uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
                        }
                    }
                }
#pragma unroll
                for (int mi = 0; mi < TC::MT; ++mi)
#pragma unroll
                    for (int e = 0; e < 4; ++e) o[mi][hr][e] = 0.f;
                m[hr] = -INFINITY;
                l[hr] = 0.f;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&qempty[qs]);
            ++segs;
            u_first = mt.u;
        }
        const int tok0 = mt.u * p.toks + jt * TC::TW;
        const int valid = min(TC::TW, mt.L - tok0);
        if (valid > 0 && nvh > 0) {
            const uint32_t kb = stage_addr + uint32_t(s) * lay.stage_bytes;
            if constexpr (!QS) {
                // fused store: the tile holding the new token takes its K/V row from k_new / v_new (the
                // cache row the copy brought is the previous content) and writes it to the cache; no
                // other CTA reads that row in this kernel (the block of a sequence's last token is its own)
                const int tl = mt.L - 1 - tok0;
                if (p.k_new && mt.newrow >= 0 && tl >= 0 && tl < TC::TW) {
                    if (lane < TC::ROWB / 8) {
                        if constexpr (kLateNewRow) load_new_row(mt, kn, vn);
                        const int t = jt * TC::TW + tl, lg = __ffs(p.boxtok) - 1;
                        const int bi = t >> lg, r = t & (p.boxtok - 1);
                        const int byte = lane * 8, pp = byte / TC::RB, within = byte % TC::RB;
                        const uint32_t R = uint32_t((h * TC::NP + pp) * p.boxtok + r);
                        const uint32_t o = uint32_t(bi * p.boxtok * p.hg * TC::ROWB) + R * TC::RB +
                                           (swizzled_chunk<TC::RB>(uint32_t(within >> 4), R) << 4) + (within & 15);
                        asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(kb + o), "r"(kn.x), "r"(kn.y) : "memory");
                        asm volatile("st.shared.v2.u32 [%0], {%1, %2};" ::"r"(kb + lay.kv_bytes + o), "r"(vn.x),
                                     "r"(vn.y) : "memory");
                        const long long e = ((long long)mt.newrow * p.Hkv + mt.g * p.hg + h) * TC::ROWB + byte;
                        *reinterpret_cast<uint2 *>(p.k_cache_w + e) = kn;
                        *reinterpret_cast<uint2 *>(p.v_cache_w + e) = vn;
                        fence_proxy_async_smem();  // the ring's next copy into this stage comes after
                    }
                    __syncwarp();
                }
            }
            int lim[HR];
#pragma unroll
            for (int hr = 0; hr < HR; ++hr) lim[hr] = min(valid, mt.L - tok0 - shift[hr]);
            if (valid == TC::TW)
                attend_tile<D, FP8, QS, TC::HR, false>(kb, kb + lay.kv_bytes, off, qa, ksc, lim, valid, m, l, o, lane);
            else
                attend_tile<D, FP8, QS, TC::HR, true>(kb, kb + lay.kv_bytes, off, qa, ksc, lim, valid, m, l, o, lane);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        ++kk;
        if (++s == p.nst) {
            s = 0;
            sph ^= 1u;
        }

        if ((mt.flags & kLast) && nvh > 0) {
            // close this warp's part of (b, group) (a query-split warp without queries has none).
            // Row state -> column state: the thread's output columns of half hr are virtual heads
            // 8 hr + 2 r4 + e (e = 0, 1), whose rows belong to threads 8 r4 + 4e (their half-hr row).
            float mc[HR][2], lc[HR][2];
#pragma unroll
            for (int hr = 0; hr < HR; ++hr) {
                float lt = l[hr] + __shfl_xor_sync(kFull, l[hr], 1);
                lt += __shfl_xor_sync(kFull, lt, 2);
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    mc[hr][e] = __shfl_sync(kFull, m[hr], 8 * r4 + 4 * e);
                    lc[hr][e] = __shfl_sync(kFull, lt, 8 * r4 + 4 * e);
                }
            }
            bool leader = true;
            if constexpr (!QS) {
                if (p.sub > 1) {
                    // the token slices of a kv head are combined by the head's first warp (j == 0):
                    // the others leave their states in shared memory ([G][D] sums, then G maxima, G sums)
                    const uint32_t round = combs++;
                    const int cst = comb_stride(D, G);
                    leader = j == 0;
                    if (!leader) {
                        if (round > 0 && !mbar_wait_bounded(cfree, (round - 1) & 1u)) break;
                        float *mine = comb + (h * (p.sub - 1) + j - 1) * cst;
#pragma unroll
                        for (int hr = 0; hr < HR; ++hr)
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const int hh = 8 * hr + 2 * r4 + e;
                                if (hh < G) {
#pragma unroll
                                    for (int mi = 0; mi < TC::MT; ++mi)
#pragma unroll
                                        for (int half = 0; half < 2; ++half)
                                            mine[hh * D + dim_of<FP8>(mi, half, g8)] = o[mi][hr][2 * half + e];
                                    if (g8 == 0) {
                                        mine[G * D + hh] = mc[hr][e];
                                        mine[G * D + G + hh] = lc[hr][e];
                                    }
                                }
                            }
                        __syncwarp();
                        if (lane == 0) mbar_arrive(cfull);
                    } else {
                        if (!mbar_wait_bounded(cfull, round & 1u)) break;
                        const float *others = comb + h * (p.sub - 1) * cst;
#pragma unroll
                        for (int hr = 0; hr < HR; ++hr)
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                const int hh = 8 * hr + 2 * r4 + e;
                                if (hh < G) {
                                    float M = mc[hr][e];
                                    for (int jj = 0; jj < p.sub - 1; ++jj)
                                        M = fmaxf(M, others[jj * cst + G * D + hh]);
                                    // M = -inf only when no slice saw a valid token for this head (several
                                    // queries per stream, a piece past the query's last key): the state stays zero
                                    const bool none = M == -INFINITY;
                                    const float f0 = none ? 0.f : ex2(mc[hr][e] - M);
                                    float ls = f0 * lc[hr][e];
#pragma unroll
                                    for (int mi = 0; mi < TC::MT; ++mi) {
                                        o[mi][hr][e] *= f0;
                                        o[mi][hr][2 + e] *= f0;
                                    }
                                    for (int jj = 0; jj < p.sub - 1; ++jj) {
                                        const float *st2 = others + jj * cst;
                                        // 0: a slice without tokens
                                        const float f = none ? 0.f : ex2(st2[G * D + hh] - M);
                                        ls = fmaf(f, st2[G * D + G + hh], ls);
#pragma unroll
                                        for (int mi = 0; mi < TC::MT; ++mi)
#pragma unroll
                                            for (int half = 0; half < 2; ++half)
                                                o[mi][hr][2 * half + e] =
                                                    fmaf(f, st2[hh * D + dim_of<FP8>(mi, half, g8)],
                                                         o[mi][hr][2 * half + e]);
                                    }
                                    mc[hr][e] = M;
                                    lc[hr][e] = ls;
                                }
                            }
                        __syncwarp();
                        if (lane == 0) mbar_arrive(cfree);
                    }
                }
            }
            if (leader) {
                const int kvh = mt.g * p.hg + h;
                const int piece = mt.u - u_first + 1;
                if (piece == mt.n) {  // this CTA ran the whole (b, group): write the output
#pragma unroll
                    for (int hr = 0; hr < HR; ++hr)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int hh = 8 * hr + 2 * r4 + e;
                            if (hh < nvh) {
                                const float inv = vsc / lc[hr][e];
                                uint16_t *orow = p.out + (((long long)mt.b * p.qstride + jq * p.qn + hh / p.gq) * p.Hq +
                                                          (long long)kvh * p.gq + hh % p.gq) * D;
#pragma unroll
                                for (int mi = 0; mi < TC::MT; ++mi) {
                                    if constexpr (FP8) {
                                        *reinterpret_cast<uint32_t *>(orow + dim_of<FP8>(mi, 0, g8)) =
                                            pack_bf16x2(o[mi][hr][e] * inv, o[mi][hr][2 + e] * inv);
                                    } else {
                                        orow[dim_of<FP8>(mi, 0, g8)] = uint16_t(pack_bf16x2(o[mi][hr][e] * inv, 0.f));
                                        orow[dim_of<FP8>(mi, 1, g8)] =
                                            uint16_t(pack_bf16x2(o[mi][hr][2 + e] * inv, 0.f));
                                    }
                                }
                            }
                        }
                } else {
                    // the segment is its slice's first when it began in an earlier slice or at the
                    // slice's first unit (see ws_layout)
                    const long long x0 = (long long)p.nhg * scan[mt.b] + (long long)mt.g * mt.n;
                    const bool first = u_first > 0 || x0 == bound[mt.slice];
                    const long long slot = ((slots_by_slice(p.B, p.nhg)
                                                 ? 2LL * mt.slice + (first ? 0 : 1)
                                                 : mt.slice + (long long)mt.b * p.nhg + mt.g) * p.hg + h) *
                                               (QS ? p.sub : 1) + jq;
#pragma unroll
                    for (int hr = 0; hr < HR; ++hr)
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int hh = 8 * hr + 2 * r4 + e;
                            if (hh < G) {
                                float *dst = p.ws_acc + (slot * G + hh) * D;
#pragma unroll
                                for (int mi = 0; mi < TC::MT; ++mi) {
                                    if constexpr (FP8) {
                                        *reinterpret_cast<float2 *>(dst + dim_of<FP8>(mi, 0, g8)) =
                                            make_float2(o[mi][hr][e], o[mi][hr][2 + e]);
                                    } else {
                                        dst[dim_of<FP8>(mi, 0, g8)] = o[mi][hr][e];
                                        dst[dim_of<FP8>(mi, 1, g8)] = o[mi][hr][2 + e];
                                    }
                                }
                                if (g8 == 0)
                                    reinterpret_cast<float2 *>(p.ws_ml)[slot * G + hh] = make_float2(mc[hr][e], lc[hr][e]);
                            }
                        }
                    // publish the piece, then count its units in; the CTA that completes the
                    // (b, kv head) merges all pieces
                    __threadfence();
                    __syncwarp();
                    int last = 0;
                    if (lane == 0)
                        last = arrive_last(p.ws_count + ((long long)mt.b * p.Hkv + kvh) * (QS ? p.sub : 1) + jq,
                                           gen, uint32_t(piece), uint32_t(mt.n), p.err);
                    if (__shfl_sync(kFull, last, 0)) {
                        __threadfence();
                        merge_pieces<D, G, FP8, QS>(p, bound, slice_of(bound, nslots, x0),
                                                    slice_of(bound, nslots, x0 + mt.n - 1), x0, mt.g, h, jq, mt.b,
                                                    kvh, nvh, lane);
                    }
                }
            }
            // The segment's state is spent (the next segment starts with kFirst and sets it again);
            // clearing it here tells the compiler so, and it keeps none of it through the merge.
#pragma unroll
            for (int ks = 0; ks < TC::KS; ++ks)
#pragma unroll
                for (int c = 0; c < 2 * HR; ++c) qa[ks][c] = 0u;
#pragma unroll
            for (int mi = 0; mi < TC::MT; ++mi)
#pragma unroll
                for (int hr = 0; hr < HR; ++hr)
#pragma unroll
                    for (int e = 0; e < 4; ++e) o[mi][hr][e] = 0.f;
        }
        if ((mt.flags & kSliceEnd) && adaptive && warp == 0 && lane == 0) {
            // balance record for the next call: this slice's weight and run time, or "absent"
            // when an SM id without a CTA of its own left the slice to this CTA
            const bool own = mt.slice == home;
            const float us =
                float(global_ns() - *reinterpret_cast<volatile unsigned long long *>(sh + 2)) * 1e-3f;
            p.ws_bal->weight[wp][mt.slice] = own ? wts[mt.slice] : 0.f;
            p.ws_bal->elapsed[wp][mt.slice] = own ? fmaxf(us, 1e-3f) : 0.f;
            p.ws_bal->tag[wp][mt.slice] = gen ^ kTableMagic;
        }
    }
    }  // not TC5
}

// ------------------------------------------------------------------ host side
struct LaunchArgs {
    DecodeParams p;
    const void *k_cache, *v_cache;
    int device, sm_count, max_smem;
    int requested_workers;
    cudaStream_t stream;
};

// Tensor map over one cache, each cached row (token, kv head) seen as parts of
// RB bytes (RB / es elements): dims (RB / es, NB * bs rows, parts, Hkv) with
// byte strides (Hkv * D * es, RB, D * es) -- not increasing, which the
// driver takes.  A box is box_rows tokens x all parts x box_heads kv heads and
// lands in shared memory as [kv head][part][token][RB bytes], the copy
// swizzling the RB-byte rows (see the stage layout at Tc).
inline bool encode_cache_map(CUtensorMap *map, const void *base, bool fp8, int D, int Hkv, int64_t rows,
                             int box_heads, int box_rows)
{
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) {
        record_cuda_error("cuTensorMapEncodeTiled", "driver entry point unavailable");
        return false;
    }
    const int es = fp8 ? 1 : 2;  // bytes per element
    const int rb = row_bytes_smem(D, es), parts = D * es / rb;
    const cuuint64_t dims[4] = {cuuint64_t(rb / es), cuuint64_t(rows), cuuint64_t(parts), cuuint64_t(Hkv)};
    const cuuint64_t strides[3] = {cuuint64_t(Hkv) * D * es, cuuint64_t(rb), cuuint64_t(D) * es};
    const cuuint32_t box[4] = {cuuint32_t(rb / es), cuuint32_t(box_rows), cuuint32_t(parts), cuuint32_t(box_heads)};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    const CUresult r = enc(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                           const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           rb == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        char msg[64];
        std::snprintf(msg, sizeof msg, "CUresult %d", int(r));
        record_cuda_error("cuTensorMapEncodeTiled", msg);
        return false;
    }
    return true;
}

// Tensor maps encode only (base address, shape, strides, box), so a map made
// once for a cache tensor stays valid for every later call on it; keep the
// most recent ones (an engine binds one k_cache / v_cache view per layer, as in
// the nano-vllm KV-cache post, §3.2).
inline bool cached_cache_map(CUtensorMap *map, int dev, const void *base, bool fp8, int D, int Hkv, int64_t rows,
                             int box_heads, int box_rows)
{
    struct Entry {
        int dev;
        const void *base;
        bool fp8;
        int D, Hkv;
        int64_t rows;
        int box_heads, box;
        CUtensorMap map;
    };
    constexpr size_t kMaxEntries = 256;
    static std::mutex mu;
    static std::vector<Entry> cache;
    std::lock_guard<std::mutex> lock(mu);
    for (size_t i = 0; i < cache.size(); ++i) {
        const Entry &e = cache[i];
        if (e.dev == dev && e.base == base && e.fp8 == fp8 && e.D == D && e.Hkv == Hkv && e.rows == rows &&
            e.box_heads == box_heads && e.box == box_rows) {
            *map = e.map;
            return true;
        }
    }
    if (!encode_cache_map(map, base, fp8, D, Hkv, rows, box_heads, box_rows)) return false;
    if (cache.size() >= kMaxEntries) cache.erase(cache.begin());
    cache.push_back(Entry{dev, base, fp8, D, Hkv, rows, box_heads, box_rows, *map});
    return true;
}

// cudaFuncSetAttribute once per device and kernel variant (it is a host-side
// driver call; repeating it on every launch costs microseconds).  Keyed on
// <D, G, FP8, QS, TC5>: every variant has the same function-pointer type, so
// the memo must be per instantiation.
template <int D, int G, bool FP8, bool QS, bool TC5, typename Kernel>
inline bool ensure_smem_attribute(Kernel kern, int dev, size_t smem)
{
    static std::mutex mu;
    static size_t configured[64] = {};
    if (dev < 0 || dev >= 64) return false;
    std::lock_guard<std::mutex> lock(mu);
    if (configured[dev] >= smem) return true;
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) {
        cudaGetLastError();
        record_cuda_error("cudaFuncSetAttribute", cudaGetErrorString(e));
        return false;
    }
    configured[dev] = smem;
    return true;
}

template <int D, int G, bool FP8, bool QS, bool TC5 = false>
pkv_status launch_decode(LaunchArgs &a)
{
    DecodeParams &p = a.p;
    // ring depth: as many stages (up to kMaxStages) as the shared memory holds, beside two Q row
    // buffers, or beside one where that fits more stages (a segment's Q rows go into registers at its
    // first tile, so one buffer is free again long before the next segment needs it)
    constexpr int ES = FP8 ? 1 : 2;
    auto depth = [&](int qslots) {
        int n = kMaxStages;
        while (n > 2 && cta_layout(D, G, ES, p.hg, p.sub, n, p.B, QS, TC5, qslots).total > uint32_t(a.max_smem)) --n;
        return n;
    };
    int nst = depth(2);
    p.qslots = 2;
    if (one_q_buffer_ok(G, FP8, QS, TC5) && depth(1) > nst) {
        nst = depth(1);
        p.qslots = 1;
    }
    const CtaLayout lay = cta_layout(D, G, ES, p.hg, p.sub, nst, p.B, QS, TC5, p.qslots);
    if (lay.total > uint32_t(a.max_smem)) return PKV_EUNSUPPORTED;
    p.nst = nst;

    // Adaptive split: one CTA per SM, slices keyed by SM id.  Fixed split:
    // about num_workers / consumers CTAs with equal slices.
    int grid = a.sm_count;
    p.num_workers = 0;
    if (a.requested_workers > 0) {
        grid = (a.requested_workers + p.cons - 1) / p.cons;
        if (grid > kMaxSlots) grid = kMaxSlots;
        p.num_workers = a.requested_workers;
    }
    if (grid > kMaxSlots) grid = kMaxSlots;

    CUtensorMap kmap, vmap;
    const int64_t rows = int64_t(p.NB) * p.bs;
    if (!cached_cache_map(&kmap, a.device, a.k_cache, FP8, D, p.Hkv, rows, p.hg, p.boxtok) ||
        !cached_cache_map(&vmap, a.device, a.v_cache, FP8, D, p.Hkv, rows, p.hg, p.boxtok))
        return PKV_ECUDA;

    auto kern = paged_decode_kernel<D, G, FP8, QS, TC5>;
    if (!ensure_smem_attribute<D, G, FP8, QS, TC5>(kern, a.device, lay.total)) return PKV_ECUDA;
    const cudaError_t e =
        launch_pdl(kern, dim3(grid), dim3((p.cons + 1) * 32), lay.total, a.stream, kmap, vmap, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return cuda_fail("paged_decode_kernel launch", e);
    }
    return launch_status("paged_decode_kernel launch");
}

using LaunchFn = pkv_status (*)(LaunchArgs &);

template <int D, bool FP8, bool QS>
LaunchFn pick_group(int G)
{
    switch (G) {
    case 1: return launch_decode<D, 1, FP8, QS>;
    case 2: return launch_decode<D, 2, FP8, QS>;
    case 3: return launch_decode<D, 3, FP8, QS>;
    case 4: return launch_decode<D, 4, FP8, QS>;
    case 5: return launch_decode<D, 5, FP8, QS>;
    case 6: return launch_decode<D, 6, FP8, QS>;
    case 7: return launch_decode<D, 7, FP8, QS>;
    case 8: return launch_decode<D, 8, FP8, QS>;
    default: return nullptr;
    }
}

// Launchers of the E4M3-cache kernels, the query-split bf16 kernels and the
// regular bf16 kernels for 9 to 16 virtual heads (defined in
// pkv_decode_fp8.cu, pkv_decode_qs.cu and pkv_decode_wide.cu, translation
// units of their own so that the kernel families build in parallel).
LaunchFn pick_decode_fp8(int D, int G);
LaunchFn pick_decode_qs(int D, int G);
LaunchFn pick_decode_wide(int D, int G);  // regular bf16 CTAs, 9 to 16 virtual heads (pkv_decode_wide.cu)
LaunchFn pick_decode_tc5(int D);          // tensor-memory query-split CTAs, 16 virtual heads (pkv_decode_tc5.cu)

// Whether a query-split call can run on the tensor-memory CTAs: bf16 caches, entries of 128 rows
// (16 virtual heads per block: the query heads of a kv head a power of two), 128-key tiles within one
// block (block_size >= 128), and a ring of at least two stages in shared memory.
inline bool tc5_eligible(int D, int G, int gq, int block_size, int B, int max_smem)
{
    if (G != 16 || (D != 64 && D != 128) || block_size < kTc5Keys || (gq & (gq - 1)) != 0) return false;  // one box a tile
    return cta_layout(D, G, 2, 1, team_warps(G), 2, B, true, true).total <= uint32_t(max_smem);
}

}  // namespace pkv
