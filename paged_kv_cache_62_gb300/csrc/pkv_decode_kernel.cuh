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
//    at most the CTA's consumer warps, 8, or 4 for groups of 5+ query heads).
//    A unit of work is TOKS = TW * SUB consecutive tokens of one (sequence,
//    head group), TW = 16 tokens per warp and SUB warps per head (see
//    team_warps): whole contiguous cache rows of the group, moved by
//    one TMA tensor copy per physical-block span into a shared-memory stage.
//  * One CTA per SM: a producer warp streams units through a ring of 2-4
//    stages (mbarrier transaction counts for "full", consumer arrivals for
//    "empty"); HG * SUB consumer warps take one TW-token slice of one kv head
//    each, so every consumer works on every stage and the CTA's warps finish
//    together.  Block-table entries for 32 boxes at a time are fetched by the
//    producer's lanes one batch ahead; q rows arrive by bulk copy in a
//    separate 2-slot ring.
//  * A consumer serves all G query heads of its kv head from one K/V read: a
//    token row is split over D/8 lanes (16 bytes each), partial dot products
//    are finished by a shuffle reduce-scatter, the softmax max is a warp vote
//    plus (rarely) a warp max, exponentials are ex2 of log2e-prescaled scores,
//    and P.V uses the same lane split with packed fp32 FMAs.
//  * The batch's unit list is cut into one slice per SM id, each slice's size
//    following the finishing times the previous call on the workspace saw.
//    A CTA whose slice covers a whole (sequence, head group) writes bf16
//    output directly; otherwise it leaves per-head partial states (m, l, acc)
//    in the workspace and counts its units in on a per-(sequence, kv head)
//    counter; the CTA that completes the count merges the pieces (split-K /
//    flash-decoding without a second kernel).
//
// This header holds the kernel and its launch templates; pkv_decode.cu
// instantiates the bf16-cache kernels and defines the C entry points,
// pkv_decode_fp8.cu instantiates the E4M3-cache kernels.
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

constexpr int kMaxStages = 4;     // ring depth
constexpr int kMaxSlots = 512;    // slices: SM ids (adaptive) or CTAs (fixed split)
constexpr uint32_t kTableMagic = 0x62616c31u;
constexpr uint32_t kEpochMagic = 0x65706f63u;

// Consumer warps per CTA and tokens each takes from a stage (a stage holds
// team_warps * warp_tokens token rows of head_dim, 64 KiB for head_dim 128).
// Measured on the Qwen3-0.6B-shaped batch: 8 warps x 16 tokens with three
// 64 KiB stages beats 16 warps x 8 tokens (17 warps leave 96 registers a
// thread, and the G = 2 loop spills) and 8 warps x 8 tokens with six 32 KiB
// stages (twice the per-stage overhead per token).  Groups of 5 or more query
// heads keep 16G accumulator and query registers a lane: with 8 consumers
// plus the producer, three warps share an SM sub-partition's 16K registers
// (168 a thread) and those groups spill; with 4 consumers at most two do
// (255 a thread).
__host__ __device__ constexpr int team_warps(int G) { return G >= 5 ? 4 : 8; }
__host__ __device__ constexpr int warp_tokens(int) { return 16; }

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
    float scale_log2;            // scale * log2(e)
    const float *k_scale, *v_scale;  // E4M3 caches: per-kv-head scales (unused for bf16 caches)
    const int32_t *row_seq;          // several query rows per sequence: row -> the sequence whose table it
                                     // reads (null: row b reads table row b)
    // Several new tokens per sequence sharing one K/V stream: the kernel's G "heads" of a kv head are
    // qn queries x gq query heads (virtual head hh = query hh / gq, head hh % gq); query i of sequence b
    // is q / out row b * qn + i and sees the keys before position L - qn + i + 1.  Decode: qn = 1, gq = G.
    int32_t qn, gq;
};

// What the producer tells the consumers about the unit in a stage.
struct alignas(16) UnitMeta {
    int32_t b, g, u, n;            // unit u of the n units of (b, group g); b < 0: no more work
    int32_t L, flags, slice, pad;  // context length of b, kFirst | kLast | kSliceEnd, slice of the unit
};
constexpr int kFirst = 1;     // first unit of (b, g) in this slice
constexpr int kLast = 2;      // last unit of (b, g) in this slice
constexpr int kSliceEnd = 4;  // last unit of the slice

template <int D, int G>
struct Shape {
    static constexpr int TW = warp_tokens(G);  // tokens per warp tile
    static constexpr int LPT = D / 8;          // lanes per token row (16 bytes each)
    static constexpr int TPI = 32 / LPT;       // tokens per warp step
    static constexpr int NIT = TW / TPI;       // steps per tile
    static constexpr int DUP = LPT / NIT;      // lanes that end up holding each score
    static_assert(LPT >= NIT && DUP >= 1 && NIT >= 1, "tile does not fit the lane split");
};

// Shared-memory layout, computed the same way on the host (size) and device (offsets).
struct CtaLayout {
    uint32_t kv_bytes, stage_bytes, q_bytes, comb_bytes;
    uint32_t off_q, off_comb, off_meta, off_bar, off_bound, off_wts, off_red, off_sh, off_scan, total;
};

__host__ __device__ inline uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

// Floats per state in the combine buffer: G * (D + 2) rounded up to a
// multiple of 4, so every block (and its float4 rows) is 16-byte aligned.
__host__ __device__ inline int comb_stride(int D, int G) { return int(align_up(uint32_t(G * (D + 2)), 4)); }

// es: bytes per cached element (2 for bf16, 1 for E4M3).
__host__ __device__ inline CtaLayout cta_layout(int D, int G, int es, int hg, int sub, int nst, int B)
{
    CtaLayout l;
    const int toks = warp_tokens(G) * sub;
    l.kv_bytes = uint32_t(toks * hg * D * es);
    l.stage_bytes = align_up(2 * l.kv_bytes, 128);
    l.q_bytes = align_up(uint32_t(hg * G * D * 2), 128);
    // states of the non-leading warps of every head (the leader keeps its own in registers)
    l.comb_bytes = sub > 1 ? align_up(uint32_t(hg * (sub - 1) * comb_stride(D, G) * 4), 128) : 0u;
    uint32_t o = uint32_t(nst) * l.stage_bytes;
    l.off_q = o;
    o += 2 * l.q_bytes;
    l.off_comb = o;
    o += l.comb_bytes;
    l.off_meta = o;
    o += uint32_t(nst) * uint32_t(sizeof(UnitMeta));
    l.off_bar = o;
    o += uint32_t(2 * nst + 6) * 8;  // full / empty per stage, q full / empty x2, combine full / free
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

struct WsLayout {
    size_t bal_off, count_off, ml_off, acc_off, total;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Piece slots: (slice + b * nhg + group) * hg + head-in-group, one per piece.
inline WsLayout ws_layout(int32_t B, int32_t G, int32_t Hkv, int32_t D)
{
    const int hg = head_group(Hkv, G);
    const size_t slots = (size_t(kMaxSlots) + size_t(B) * size_t(Hkv / hg)) * size_t(hg);
    WsLayout w;
    w.bal_off = 0;
    w.count_off = align256(sizeof(BalanceState));
    w.ml_off = w.count_off + align256(size_t(B) * size_t(Hkv) * 8);
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

// Units per sequence -> exclusive prefix in scan[0..B].
// `tmp` needs 32 ints of shared memory that is free during the call.
static __device__ void unit_prefix_scan(const DecodeParams &p, int32_t *scan, int32_t *tmp)
{
    const int tid = threadIdx.x, nt = blockDim.x;
    const int lane = tid & 31, wid = tid >> 5, nw = nt >> 5;
    const int per = (p.B + nt - 1) / nt;
    const int lo = min(p.B, tid * per), hi = min(p.B, lo + per);
    int32_t sum = 0;
    for (int i = lo; i < hi; ++i) {
        const int32_t len = __ldg(p.context_lens + i);
        int32_t n = 0;
        if (len < 0 || len > p.len_limit) {
            if (blockIdx.x == 0) flag_error(p.err, PKV_ERR_CONTEXT_RANGE);
        } else {
            n = (len + p.toks - 1) / p.toks;
        }
        scan[i] = n;
        sum += n;
    }
    int32_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t v = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) tmp[wid] = incl;
    __syncthreads();
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
    __syncthreads();
    int32_t run = tmp[wid] + incl - sum;
    for (int i = lo; i < hi; ++i) {
        const int32_t n = scan[i];
        scan[i] = run;
        run += n;
    }
    if (lo < hi && hi == p.B) scan[p.B] = run;
    __syncthreads();
}

// ------------------------------------------------------------------ one tile
// Slack (log2 units) a score may exceed the running max before the running
// state is rescaled: weights stay <= 2^kRescaleSlack, which fp32 holds with
// ample room, and most tiles skip the warp max and the rescale entirely.
constexpr float kRescaleSlack = 8.0f;

__device__ __forceinline__ void unpack8x2(const uint4 w, float2 f[4])
{
    const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) f[i] = make_float2(__uint_as_float(u[i] << 16), __uint_as_float(u[i] & 0xffff0000u));
}

// Eight E4M3 codes (bytes 0..7 of w, element e in byte e) -> four fp32
// pairs: the hardware conversion to f16 pairs (exact: every E4M3 value is a
// normal f16 or zero), then f16 -> fp32 (exact).
__device__ __forceinline__ void unpack8x2_e4m3(const uint2 w, float2 f[4])
{
    const uint32_t u[2] = {w.x, w.y};
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        uint32_t h0, h1;  // f16 pairs of bytes (1, 0) and (3, 2)
        asm("{.reg .b16 lo, hi;\n\t"
            "mov.b32 {lo, hi}, %2;\n\t"
            "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t"
            "cvt.rn.f16x2.e4m3x2 %1, hi;}"
            : "=r"(h0), "=r"(h1) : "r"(u[i]));
        f[2 * i] = __half22float2(*reinterpret_cast<const __half2 *>(&h0));
        f[2 * i + 1] = __half22float2(*reinterpret_cast<const __half2 *>(&h1));
    }
}

// Eight consecutive cached elements starting at element `e` of `base` as fp32 pairs.
template <bool FP8>
__device__ __forceinline__ void load8(const uint8_t *base, int e, float2 f[4])
{
    if constexpr (FP8)
        unpack8x2_e4m3(*reinterpret_cast<const uint2 *>(base + e), f);
    else
        unpack8x2(*reinterpret_cast<const uint4 *>(base + 2 * e), f);
}

// One TW-token tile of one (sequence, kv head) for the G query heads of the
// group: Ks / Vs point at the tile's first K / V row, consecutive tokens are
// `stride` elements apart (bf16 values, or E4M3 codes whose kv-head scales
// the caller has folded into q2 and the final division).  Element pairs are
// handled with the packed fp32 FMA (two independent round-to-nearest fp32
// FMAs per instruction).
template <int D, int G, bool FP8>
__device__ __forceinline__ void attend_tile(const uint8_t *Ks, const uint8_t *Vs, int stride, int valid,
                                            const float2 (&q2)[G][4], float (&m)[G], float (&l)[G],
                                            float2 (&acc)[G][4], int c, int grp, int rem, int qtail, int gq)
{
    using S = Shape<D, G>;
    constexpr int LPT = S::LPT, TPI = S::TPI, NIT = S::NIT, DUP = S::DUP;

    // scores: lane (grp, c) forms the 8-element partial dot products of tokens i*TPI + grp
    float part[G][NIT];
#pragma unroll
    for (int i = 0; i < NIT; ++i) {
        const int tok = i * TPI + grp;
        float2 k2[4];
        load8<FP8>(Ks, tok * stride + c * 8, k2);
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float2 a = __fmul2_rn(q2[h][0], k2[0]);
#pragma unroll
            for (int j = 1; j < 4; ++j) a = __ffma2_rn(q2[h][j], k2[j], a);
            part[h][i] = a.x + a.y;
        }
    }
    // reduce-scatter over the LPT lanes of a token: afterwards lane c holds the
    // full score of step c / DUP
#pragma unroll
    for (int cnt = NIT, mask = LPT / 2; cnt > 1; cnt >>= 1, mask >>= 1) {
        const bool upper = (c & mask) != 0;
#pragma unroll
        for (int j = 0; j < cnt / 2; ++j) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float send = upper ? part[h][j] : part[h][j + cnt / 2];
                const float keep = upper ? part[h][j + cnt / 2] : part[h][j];
                part[h][j] = keep + __shfl_xor_sync(kFull, send, mask);
            }
        }
    }
#pragma unroll
    for (int mask = DUP / 2; mask > 0; mask >>= 1)
#pragma unroll
        for (int h = 0; h < G; ++h) part[h][0] += __shfl_xor_sync(kFull, part[h][0], mask);

    const int tok_s = (c / DUP) * TPI + grp;
    const bool ok = tok_s < valid;
    float pr[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        // several queries per stream: query h / gq sees qtail - h / gq fewer of the sequence's last
        // tokens (rem: tokens of the sequence from this tile's first on, not clamped to the tile)
        const bool okh = qtail > 0 ? tok_s < min(valid, rem - (qtail - h / gq)) : ok;
        const float s = okh ? part[h][0] : -INFINITY;
        // Online softmax (m, l, acc).  The running max only moves when some
        // score passes it by more than the slack; the first tile with a valid token
        // for the head always moves it (m = -inf before it).
        if (__any_sync(kFull, s > m[h] + kRescaleSlack)) {
            const float mn = fmaxf(m[h], warp_max(s));
            const float alpha = ex2(m[h] - mn);  // 0 on the first tile
            l[h] *= alpha;
            const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[h][j] = __fmul2_rn(acc[h][j], a2);
            m[h] = mn;
        }
        pr[h] = okh ? ex2(s - m[h]) : 0.f;
        l[h] += pr[h];
    }
    // P.V: the weight of token i*TPI + grp sits in lane grp*LPT + i*DUP
#pragma unroll
    for (int i = 0; i < NIT; ++i) {
        const int tok = i * TPI + grp;
        float ph[G];
#pragma unroll
        for (int h = 0; h < G; ++h) ph[h] = __shfl_sync(kFull, pr[h], grp * LPT + i * DUP);
        if (tok < valid) {  // rows past L may hold anything, even NaN: never touch them
            float2 v2[4];
            load8<FP8>(Vs, tok * stride + c * 8, v2);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float2 p2 = make_float2(ph[h], ph[h]);
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[h][j] = __ffma2_rn(p2, v2[j], acc[h][j]);
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

// Sums of two floats per thread over the CTA (fixed order: identical in every
// CTA).  `red` holds 2 * 32 floats.
__device__ __forceinline__ float2 block_sum2(float2 v, float *red)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    v.x = warp_sum(v.x);
    v.y = warp_sum(v.y);
    __syncthreads();
    if (lane == 0) {
        red[2 * wid] = v.x;
        red[2 * wid + 1] = v.y;
    }
    __syncthreads();
    float2 t = make_float2(0.f, 0.f);
    for (int i = 0; i < nw; ++i) {
        t.x += red[2 * i];
        t.y += red[2 * i + 1];
    }
    return t;
}

// The balance entries this thread reads in build_partition (slices tid and
// tid + blockDim.x), loaded up front so that their memory round trip overlaps
// the context-length loads of unit_prefix_scan.  Both table halves are
// loaded, before this call's number is known; build_partition keeps the
// entry whose tag names the previous call.
struct BalanceIn {
    float w[2][2], t[2][2];  // [table half][entry k]
    uint32_t tag[2][2];
};
static_assert(2 * (8 + 1) * 32 >= kMaxSlots, "two balance entries per thread must cover every slice");

__device__ __forceinline__ BalanceIn load_balance(const DecodeParams &p, bool adaptive, int nslots)
{
    BalanceIn in;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int i = threadIdx.x + k * blockDim.x;
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
// same inputs in the same order; leaves the weights in w[].
static __device__ void build_partition(const DecodeParams &p, uint32_t gen, bool adaptive, int nslots, long long T,
                                long long *bound, float *w, float *red, const BalanceIn &in)
{
    const int tid = threadIdx.x, nt = blockDim.x;
    const uint32_t want = (gen - 1u) ^ kTableMagic;
    // pass 1: raw weights (kept in w) and elapsed times (kept in bound[] as float bits)
    float tsum = 0.f, tcnt = 0.f;
    float *el = reinterpret_cast<float *>(bound);
#pragma unroll
    for (int k = 0; k < 2; ++k) {
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
    const float2 tt = block_sum2(make_float2(tsum, tcnt), red);
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
    const float2 ww = block_sum2(make_float2(wsum, wcnt), red);
    wsum = ww.x;
    wcnt = ww.y;
    const float wmean = wcnt > 0.f ? wsum / wcnt : 1.0f;
    for (int i = tid; i < nslots; i += nt) {
        float x = wcnt > 0.f ? w[i] / wmean : 1.0f;  // mean 1 over present slices; none: equal weights
        if (x > 0.f) x = fminf(fmaxf(x, 0.25f), 4.0f);
        w[i] = x;
    }
    __syncthreads();
    // bounds: float prefix of the weights -> 2^20 tickets -> tiles (a shift, no division)
    if (tid < 32) {
        const int per = (nslots + 31) / 32;
        const int lo = min(nslots, tid * per), hi = min(nslots, lo + per);
        float run = 0.f;
        for (int i = lo; i < hi; ++i) run += w[i];
        float incl = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float v = __shfl_up_sync(kFull, incl, o);
            if (tid >= o) incl += v;
        }
        const float total = __shfl_sync(kFull, incl, 31);
        float acc = incl - run;
        for (int i = lo; i < hi; ++i) {
            long long pre = total > 0.f ? (long long)(acc / total * 1048576.0f) : (long long)i * 1048576 / nslots;
            pre = pre < 0 ? 0 : (pre > 1048576 ? 1048576 : pre);
            bound[i] = (T * pre) >> 20;
            acc += w[i];
        }
        __syncwarp();
        if (tid == 0) bound[nslots] = T;
    }
    // bounds are monotone: the float prefix only grows and pre is clamped to [0, 2^20]
    __syncthreads();
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
    unsigned long long cur = *reinterpret_cast<volatile unsigned long long *>(ctr);
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
// sf..sl, piece slots (s + sigma) * hg + h:
//   M = max m_i,  l = sum 2^(m_i - M) l_i,  out = sum 2^(m_i - M) acc_i / l
// (the online-softmax algebra; m in log2 units).  The pieces were written by
// other SMs, so they are read through L2 (ld.global.cg), BATCH pieces at a
// time with independent loads, folded into a running (M, l, acc).
template <int D, int G, bool FP8>
__device__ __forceinline__ void merge_pieces(const DecodeParams &p, const long long *bound, int sf, int sl,
                                             long long sigma, int h, int b, int kvh, int lane)
{
    constexpr int PER = D / 32;                           // output values per lane
    constexpr int BATCH = G <= 2 ? 4 : (G <= 7 ? 2 : 1);  // pieces loaded together (G = 8 would spill)
    using Vec = typename std::conditional<PER == 4, float4, float2>::type;
    const float2 *ml = reinterpret_cast<const float2 *>(p.ws_ml);
    float M[G], lsum[G], a[G][PER];
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
        M[hh] = -INFINITY;
        lsum[hh] = 0.f;
#pragma unroll
        for (int e = 0; e < PER; ++e) a[hh][e] = 0.f;
    }
    for (int s0 = sf; s0 <= sl; s0 += BATCH) {
        float2 st[BATCH][G];
        Vec v[BATCH][G];
        bool use[BATCH];
#pragma unroll
        for (int k = 0; k < BATCH; ++k) {
            const int s = s0 + k;
            use[k] = s <= sl && bound[s + 1] > bound[s];  // empty slices left nothing
            const long long slot = ((use[k] ? s : sf) + sigma) * p.hg + h;
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                st[k][hh] = __ldcg(ml + slot * G + hh);
                v[k][hh] = __ldcg(reinterpret_cast<const Vec *>(p.ws_acc + (slot * G + hh) * D + lane * PER));
            }
        }
#pragma unroll
        for (int hh = 0; hh < G; ++hh) {
            float mb = M[hh];
#pragma unroll
            for (int k = 0; k < BATCH; ++k)
                if (use[k]) mb = fmaxf(mb, st[k][hh].x);
            // 0 while nothing has been folded in (M = -inf); a head with no valid token in any piece
            // so far (several queries per stream) keeps its zero state
            const float r = mb == -INFINITY ? 1.0f : ex2(M[hh] - mb);
            lsum[hh] *= r;
#pragma unroll
            for (int e = 0; e < PER; ++e) a[hh][e] *= r;
#pragma unroll
            for (int k = 0; k < BATCH; ++k) {
                const float f = (use[k] && st[k][hh].x != -INFINITY) ? ex2(st[k][hh].x - mb) : 0.f;
                lsum[hh] = fmaf(f, st[k][hh].y, lsum[hh]);
                const float *x = reinterpret_cast<const float *>(&v[k][hh]);
#pragma unroll
                for (int e = 0; e < PER; ++e) a[hh][e] = fmaf(f, x[e], a[hh][e]);
            }
            M[hh] = mb;
        }
    }
#pragma unroll
    for (int hh = 0; hh < G; ++hh) {
        const float inv = (FP8 ? __ldg(p.v_scale + kvh) : 1.0f) / lsum[hh];
        uint16_t *o = p.out + ((int64_t(b) * p.qn + hh / p.gq) * p.Hq + int64_t(kvh) * p.gq + hh % p.gq) * D +
                      lane * PER;
        if constexpr (PER == 4)
            *reinterpret_cast<uint2 *>(o) = make_uint2(pack_bf16x2(a[hh][0] * inv, a[hh][1] * inv),
                                                       pack_bf16x2(a[hh][2] * inv, a[hh][3] * inv));
        else
            *reinterpret_cast<uint32_t *>(o) = pack_bf16x2(a[hh][0] * inv, a[hh][1] * inv);
    }
}

// ------------------------------------------------------------------ main kernel
// Block: p.cons consumer warps (warp w: kv head w / sub of the group, TW-token
// slice w % sub of every unit) and one producer warp (warp p.cons).
template <int D, int G, bool FP8>
__global__ void __launch_bounds__((team_warps(G) + 1) * 32, 1)
    paged_decode_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                        const DecodeParams p)
{
    using S = Shape<D, G>;
    constexpr int LPT = S::LPT, DUP = S::DUP, TW = S::TW;
    extern __shared__ __align__(1024) uint8_t smem[];
    constexpr int ES = FP8 ? 1 : 2;  // bytes per cached element
    const CtaLayout lay = cta_layout(D, G, ES, p.hg, p.sub, p.nst, p.B);
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
    int *sh = reinterpret_cast<int *>(smem + lay.off_sh);  // [0] own slice, [2..3] its start time
    int32_t *scan = reinterpret_cast<int32_t *>(smem + lay.off_scan);

    if (threadIdx.x == 0) {
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
    }
    griddep_launch_dependents();  // lets the next kernel in the stream get scheduled; it waits for this grid
    griddep_wait();               // inputs may come from the previous kernel in the stream

    // Slices: one per SM id, sized by measured finishing times (adaptive), or one per CTA (fixed).
    const bool adaptive = p.num_workers == 0;
    int nslots = int(gridDim.x);
    if (adaptive) nslots = int(min(nsmid(), unsigned(kMaxSlots)));
    // The set-up's global reads are all issued here, so together they cost about one memory
    // round trip: the workspace's control block (this call's number), the balance entries,
    // the context lengths (in unit_prefix_scan) and, once the call number is in, the claim on
    // this SM id's slice (an exchange: the first CTA of this call to run on the SM id finds
    // another call's tag there), whose answer is needed only after the partition.
    const uint32_t epoch = __ldcg(&p.ws_bal->epoch), stamp = __ldcg(&p.ws_bal->stamp);
    const BalanceIn bal_in = load_balance(p, adaptive, nslots);
    const bool ctl_ok = stamp == (epoch ^ kEpochMagic) || (epoch == 0u && stamp == 0u);
    const uint32_t gen = epoch + 1u;  // tags of this call; zero-filled words never match
    const int wp = int(gen & 1u);     // this call writes one half of the balance table
    const unsigned my_sm = smid();
    unsigned long long home_word = static_cast<unsigned long long>(gen) << 32;
    if (threadIdx.x == 0 && adaptive && int(my_sm) < nslots)
        home_word = atomicExch(&p.ws_bal->claim[my_sm], (static_cast<unsigned long long>(gen) << 32) | 1ull);
    if (!ctl_ok && blockIdx.x == 0 && threadIdx.x == 0) flag_error(p.err, PKV_ERR_WORKSPACE);
    unit_prefix_scan(p, scan, reinterpret_cast<int32_t *>(smem));
    const long long T = (long long)p.nhg * scan[p.B];

    // Sequences without units (L == 0, or a rejected length) get zeros; CTAs share the job.
    for (int b = blockIdx.x; b < p.B; b += gridDim.x)
        if (scan[b + 1] == scan[b])
            for (int i = threadIdx.x; i < p.Hq * D / 8; i += blockDim.x)
                reinterpret_cast<uint4 *>(p.out + int64_t(b) * p.Hq * D)[i] = make_uint4(0u, 0u, 0u, 0u);

    build_partition(p, gen, adaptive, nslots, T, bound, wts, red, bal_in);

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.nst; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], uint32_t(p.cons));
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&qfull[i], 1);
            mbar_init(&qempty[i], uint32_t(p.cons));
        }
        mbar_init(cfull, uint32_t(p.cons - p.hg));  // the non-leading warps' states
        mbar_init(cfree, uint32_t(p.hg));           // read again by the leaders
        fence_barrier_init();
        int home = -1;
        if (!adaptive)
            home = int(blockIdx.x);
        else if (uint32_t(home_word >> 32) != gen)
            home = int(my_sm);
        sh[0] = home;
    }
    __syncthreads();

    if (warp == p.cons) {
        // ============================== producer warp ==============================
        const uint64_t policy = policy_evict_first();
        const uint32_t box_bytes = uint32_t(p.boxtok * p.hg * D * ES);
        uint32_t kk = 0, segs = 0;  // units issued, q-ring uses
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
            // Block-table prefetch, 32 boxes per batch: lane j of `cur` holds the entry (and the
            // context length) of box kb + j; `nxt` is loaded one batch ahead.  Two register sets,
            // because the scoreboard tracks a register for the whole warp.
            Walker iw = nunits > 0 ? walker_locate(scan, p.B, p.nhg, lo) : Walker{0, 0, 0, 1};
            int32_t cur_e = -1, cur_L = 0, nxt_e = -1, nxt_L = 0;
            auto prefetch_batch = [&](long long kb) {  // boxes [kb, kb + 32) -> nxt, one per lane
                const long long x = kb + lane;
                if (x < nboxes) {
                    const Walker mine = walker_locate(scan, p.B, p.nhg, lo + (x >> p.lg_nbox));
                    const int32_t pos = mine.u * p.toks + int32_t(x & (p.nbox - 1)) * p.boxtok;
                    // The entry is only used for pos < L, where pos / bs < max_blocks (lengths
                    // beyond the table were rejected by the scan); clamping keeps the load in
                    // the row and lets it go out together with the length's.
                    const int32_t blk = min(pos >> p.log2_bs, p.max_blocks - 1);
                    nxt_L = __ldg(p.context_lens + mine.b);
                    const int32_t trow = p.row_seq ? __ldg(p.row_seq + mine.b) : mine.b;
                    nxt_e = __ldg(p.block_tables + (long long)trow * p.max_blocks + blk);
                }
            };
            if (nunits > 0) {
                prefetch_batch(0);
                cur_e = nxt_e;
                cur_L = nxt_L;
            }
            for (long long k = 0; k < nunits; ++k) {
                const long long kb0 = k * p.nbox;  // nbox is a power of two <= 16: batches start on units
                if ((kb0 & 31) == 0 && k > 0) {
                    cur_e = nxt_e;
                    cur_L = nxt_L;
                    if (kb0 + 32 < nboxes) prefetch_batch(kb0 + 32);
                }
                const int s = rs;
                if (kk >= uint32_t(p.nst) && !mbar_wait_bounded(&empty[s], rph ^ 1u)) {
                    dead = true;
                    break;
                }
                const int src = int(kb0 & 31);
                const int32_t len = __shfl_sync(kFull, cur_L, src);
                const int32_t e = __shfl_sync(kFull, cur_e, (src + lane) & 31);  // lane j: box j's entry
                const int flags = ((k == 0 || iw.u == 0) ? kFirst : 0) |
                                  ((k == nunits - 1 || iw.u == iw.n - 1) ? kLast : 0) |
                                  (k == nunits - 1 ? kSliceEnd : 0);
                if (flags & kFirst) {  // q rows of this (b, group) for the consumers
                    const int qs = int(segs & 1u);
                    const uint32_t quse = segs >> 1;
                    if (quse > 0 && !mbar_wait_bounded(&qempty[qs], (quse - 1) & 1u)) {
                        dead = true;
                        break;
                    }
                    const uint32_t qb = uint32_t(p.hg * G * D * 2);
                    if (p.qn == 1) {  // the group's G * hg query rows are contiguous
                        if (lane == 0) {
                            mbar_arrive_expect_tx(&qfull[qs], qb);
                            bulk_load(qbuf + qs * lay.q_bytes,
                                      p.q + ((long long)iw.b * p.Hq + (long long)iw.g * p.hg * G) * D, qb,
                                      &qfull[qs]);
                        }
                    } else {
                        // qn queries: kv head h's virtual heads i * gq .. i * gq + gq - 1 come from row
                        // b * qn + i; one copy of gq rows per (h, i), lane t copying pair t
                        if (lane == 0) mbar_arrive_expect_tx(&qfull[qs], qb);
                        __syncwarp();
                        for (int t = lane; t < p.hg * p.qn; t += 32) {
                            const int hh = t / p.qn, qi = t - hh * p.qn;
                            bulk_load(qbuf + qs * lay.q_bytes + size_t((hh * G + qi * p.gq) * D) * 2,
                                      p.q + (((long long)iw.b * p.qn + qi) * p.Hq +
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
                    mbar_arrive_expect_tx(&full[s], 2 * nrows * box_bytes);
                }
                __syncwarp();
                if (row >= 0) {
                    tma_load_3d(st + lane * box_bytes, &kmap, 0, iw.g * p.hg, row, &full[s], policy);
                    tma_load_3d(st + lay.kv_bytes + lane * box_bytes, &vmap, 0, iw.g * p.hg, row, &full[s], policy);
                }
                ++kk;
                if (++rs == p.nst) {
                    rs = 0;
                    rph ^= 1u;
                }
                if (k + 1 < nunits) walker_advance(iw, scan, p.nhg, p.B);
                if (k == 0 && nboxes > 32) prefetch_batch(32);  // after the first copies are on their way
            }
            slice = (adaptive && !dead) ? claim_leftover(p, gen, bound, nslots, wp, true) : -1;
        }
        if (!dead) {  // end-of-work marker
            if (kk < uint32_t(p.nst) || mbar_wait_bounded(&empty[rs], rph ^ 1u)) {
                if (lane == 0) {
                    metas[rs].b = -1;
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
    const int h = warp / p.sub, j = warp - h * p.sub;  // kv head in the group, token slice of the unit
    const int c = lane % LPT, grp = lane / LPT;
    const int stride = p.hg * D;                      // elements between consecutive tokens of a stage
    const int home = sh[0];
    uint32_t kk = 0, segs = 0, combs = 0;
    int s = 0;           // ring slot of stage kk
    uint32_t sph = 0;    // parity of its use
    float2 q2[G][4], acc[G][4];
    float m[G], l[G];
    float vsc = 1.0f;  // E4M3 caches: the kv head's V scale, applied in the final division
    int u_first = 0;
    for (;;) {
        if (!mbar_wait_bounded(&full[s], sph)) {
            if (lane == 0) flag_error(p.err, PKV_ERR_WAIT_TIMEOUT);
            break;
        }
        const UnitMeta mt = metas[s];
        if (mt.b < 0) break;
        const uint8_t *st = stage0 + s * lay.stage_bytes;
        if (mt.flags & kFirst) {
            const int qs = int(segs & 1u);
            float ksc = p.scale_log2;  // E4M3 caches: the kv head's K scale folds into the query prescale
            if constexpr (FP8) {
                ksc *= __ldg(p.k_scale + mt.g * p.hg + h);
                vsc = __ldg(p.v_scale + mt.g * p.hg + h);
            }
            if (!mbar_wait_bounded(&qfull[qs], (segs >> 1) & 1u)) {
                if (lane == 0) flag_error(p.err, PKV_ERR_WAIT_TIMEOUT);
                break;
            }
            const uint16_t *qh = reinterpret_cast<const uint16_t *>(qbuf + qs * lay.q_bytes) + h * G * D;
            const float2 sc = make_float2(ksc, ksc);
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                float2 f[4];
                unpack8x2(*reinterpret_cast<const uint4 *>(qh + hh * D + c * 8), f);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    q2[hh][e] = __fmul2_rn(f[e], sc);
                    acc[hh][e] = make_float2(0.f, 0.f);
                }
                m[hh] = -INFINITY;
                l[hh] = 0.f;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&qempty[qs]);
            ++segs;
            u_first = mt.u;
        }
        const int tok0 = mt.u * p.toks + j * TW;
        const int valid = min(TW, mt.L - tok0);
        if (valid > 0) {
            const int e0 = (j * TW * p.hg + h) * D;  // element offset of this warp's first row in the stage
            attend_tile<D, G, FP8>(st + e0 * ES, st + lay.kv_bytes + e0 * ES, stride, valid, q2, m, l, acc, c,
                                   grp, mt.L - tok0, p.qn - 1, p.gq);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        ++kk;
        if (++s == p.nst) {
            s = 0;
            sph ^= 1u;
        }

        if (mt.flags & kLast) {
            // close this warp's part of (b, group): fold the token groups
#pragma unroll
            for (int mask = LPT; mask < 32; mask <<= 1)
#pragma unroll
                for (int hh = 0; hh < G; ++hh)
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        acc[hh][e].x += __shfl_xor_sync(kFull, acc[hh][e].x, mask);
                        acc[hh][e].y += __shfl_xor_sync(kFull, acc[hh][e].y, mask);
                    }
            float lt[G];
#pragma unroll
            for (int hh = 0; hh < G; ++hh) lt[hh] = warp_sum(l[hh]) * (1.0f / DUP);
            bool leader = true;
            if (p.sub > 1) {
                // the token slices of a kv head are combined by the head's first warp (j == 0):
                // the others leave their states in shared memory
                const uint32_t round = combs++;
                const int cst = comb_stride(D, G);
                leader = j == 0;
                if (!leader) {
                    if (round > 0 && !mbar_wait_bounded(cfree, (round - 1) & 1u)) break;
                    float *mine = comb + (h * (p.sub - 1) + j - 1) * cst;
                    if (grp == 0)
#pragma unroll
                        for (int hh = 0; hh < G; ++hh) {
                            float4 *dst = reinterpret_cast<float4 *>(mine + hh * D + c * 8);
                            dst[0] = make_float4(acc[hh][0].x, acc[hh][0].y, acc[hh][1].x, acc[hh][1].y);
                            dst[1] = make_float4(acc[hh][2].x, acc[hh][2].y, acc[hh][3].x, acc[hh][3].y);
                        }
                    if (lane == 0)
#pragma unroll
                        for (int hh = 0; hh < G; ++hh) {
                            mine[G * D + hh] = m[hh];
                            mine[G * D + G + hh] = lt[hh];
                        }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(cfull);
                } else {
                    if (!mbar_wait_bounded(cfull, round & 1u)) break;
                    const float *others = comb + h * (p.sub - 1) * cst;
#pragma unroll
                    for (int hh = 0; hh < G; ++hh) {
                        float M = m[hh];
                        for (int jj = 0; jj < p.sub - 1; ++jj) M = fmaxf(M, others[jj * cst + G * D + hh]);
                        // M = -inf only when no slice saw a valid token for this head (several queries
                        // per stream, a piece past the query's last key): the state stays zero
                        const bool none = M == -INFINITY;
                        const float f0 = none ? 0.f : ex2(m[hh] - M);
                        float ls = f0 * lt[hh];
                        const float2 f02 = make_float2(f0, f0);
                        float2 a[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) a[e] = __fmul2_rn(acc[hh][e], f02);
                        for (int jj = 0; jj < p.sub - 1; ++jj) {
                            const float *st2 = others + jj * cst;
                            const float f = none ? 0.f : ex2(st2[G * D + hh] - M);  // 0 for a slice with no tokens
                            ls = fmaf(f, st2[G * D + G + hh], ls);
                            const float4 x0 = *reinterpret_cast<const float4 *>(st2 + hh * D + c * 8);
                            const float4 x1 = *reinterpret_cast<const float4 *>(st2 + hh * D + c * 8 + 4);
                            a[0] = make_float2(fmaf(f, x0.x, a[0].x), fmaf(f, x0.y, a[0].y));
                            a[1] = make_float2(fmaf(f, x0.z, a[1].x), fmaf(f, x0.w, a[1].y));
                            a[2] = make_float2(fmaf(f, x1.x, a[2].x), fmaf(f, x1.y, a[2].y));
                            a[3] = make_float2(fmaf(f, x1.z, a[3].x), fmaf(f, x1.w, a[3].y));
                        }
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[hh][e] = a[e];
                        m[hh] = M;
                        lt[hh] = ls;
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(cfree);
                }
            }
            if (leader) {
                const int kvh = mt.g * p.hg + h;
                const int piece = mt.u - u_first + 1;
                if (piece == mt.n) {  // this CTA ran the whole (b, group): write the output
                    if (grp == 0)
#pragma unroll
                        for (int hh = 0; hh < G; ++hh) {
                            const float inv = vsc / lt[hh];
                            uint4 o;
                            o.x = pack_bf16x2(acc[hh][0].x * inv, acc[hh][0].y * inv);
                            o.y = pack_bf16x2(acc[hh][1].x * inv, acc[hh][1].y * inv);
                            o.z = pack_bf16x2(acc[hh][2].x * inv, acc[hh][2].y * inv);
                            o.w = pack_bf16x2(acc[hh][3].x * inv, acc[hh][3].y * inv);
                            *reinterpret_cast<uint4 *>(
                                p.out + (((long long)mt.b * p.qn + hh / p.gq) * p.Hq + (long long)kvh * p.gq + hh % p.gq) * D +
                                c * 8) = o;
                        }
                } else {
                    const long long sigma = (long long)mt.b * p.nhg + mt.g;
                    const long long slot = (mt.slice + sigma) * p.hg + h;
                    if (grp == 0)
#pragma unroll
                        for (int hh = 0; hh < G; ++hh) {
                            float4 *dst = reinterpret_cast<float4 *>(p.ws_acc + ((slot * G + hh) * D + c * 8));
                            dst[0] = make_float4(acc[hh][0].x, acc[hh][0].y, acc[hh][1].x, acc[hh][1].y);
                            dst[1] = make_float4(acc[hh][2].x, acc[hh][2].y, acc[hh][3].x, acc[hh][3].y);
                        }
                    if (lane == 0)
#pragma unroll
                        for (int hh = 0; hh < G; ++hh)
                            reinterpret_cast<float2 *>(p.ws_ml)[slot * G + hh] = make_float2(m[hh], lt[hh]);
                    // publish the piece, then count its units in; the CTA that completes the
                    // (b, kv head) merges all pieces
                    __threadfence();
                    __syncwarp();
                    int last = 0;
                    if (lane == 0)
                        last = arrive_last(p.ws_count + (long long)mt.b * p.Hkv + kvh, gen, uint32_t(piece),
                                           uint32_t(mt.n), p.err);
                    if (__shfl_sync(kFull, last, 0)) {
                        __threadfence();
                        const long long x0 = (long long)p.nhg * scan[mt.b] + (long long)mt.g * mt.n;
                        merge_pieces<D, G, FP8>(p, bound, slice_of(bound, nslots, x0),
                                           slice_of(bound, nslots, x0 + mt.n - 1), sigma, h, mt.b, kvh, lane);
                    }
                }
            }
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
}

// ------------------------------------------------------------------ host side
struct LaunchArgs {
    DecodeParams p;
    const void *k_cache, *v_cache;
    int device, sm_count, max_smem;
    int requested_workers;
    cudaStream_t stream;
};

// Tensor map over one cache: dims (head_dim, kv heads, NB * bs rows); a box is
// box_rows tokens x box_heads kv heads x head_dim (whole contiguous rows of a head group).
inline bool encode_cache_map(CUtensorMap *map, const void *base, bool fp8, int D, int Hkv, int64_t rows,
                             int box_heads, int box_rows)
{
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) {
        record_cuda_error("cuTensorMapEncodeTiled", "driver entry point unavailable");
        return false;
    }
    const cuuint64_t dims[3] = {cuuint64_t(D), cuuint64_t(Hkv), cuuint64_t(rows)};
    const cuuint64_t es = fp8 ? 1 : 2;  // bytes per element
    const cuuint64_t strides[2] = {cuuint64_t(D) * es, cuuint64_t(Hkv) * D * es};
    const cuuint32_t box[3] = {cuuint32_t(D), cuuint32_t(box_heads), cuuint32_t(box_rows)};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUresult r = enc(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                           const_cast<void *>(base), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
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
// <D, G, FP8>: every variant has the same function-pointer type, so the memo
// must be per instantiation.
template <int D, int G, bool FP8, typename Kernel>
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

template <int D, int G, bool FP8>
pkv_status launch_decode(LaunchArgs &a)
{
    DecodeParams &p = a.p;
    // ring depth: as many stages (up to kMaxStages) as the shared memory holds
    int nst = kMaxStages;
    constexpr int ES = FP8 ? 1 : 2;
    while (nst > 2 && cta_layout(D, G, ES, p.hg, p.sub, nst, p.B).total > uint32_t(a.max_smem)) --nst;
    const CtaLayout lay = cta_layout(D, G, ES, p.hg, p.sub, nst, p.B);
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

    auto kern = paged_decode_kernel<D, G, FP8>;
    if (!ensure_smem_attribute<D, G, FP8>(kern, a.device, lay.total)) return PKV_ECUDA;
    const cudaError_t e = launch_pdl(kern, dim3(grid), dim3((p.cons + 1) * 32), lay.total, a.stream, kmap, vmap, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return cuda_fail("paged_decode_kernel launch", e);
    }
    return launch_status("paged_decode_kernel launch");
}

using LaunchFn = pkv_status (*)(LaunchArgs &);

template <int D, bool FP8>
LaunchFn pick_group(int G)
{
    switch (G) {
    case 1: return launch_decode<D, 1, FP8>;
    case 2: return launch_decode<D, 2, FP8>;
    case 3: return launch_decode<D, 3, FP8>;
    case 4: return launch_decode<D, 4, FP8>;
    case 5: return launch_decode<D, 5, FP8>;
    case 6: return launch_decode<D, 6, FP8>;
    case 7: return launch_decode<D, 7, FP8>;
    case 8: return launch_decode<D, 8, FP8>;
    default: return nullptr;
    }
}

// Launchers of the E4M3-cache kernels (defined in pkv_decode_fp8.cu, a
// translation unit of its own so that the two kernel families build in
// parallel).
LaunchFn pick_decode_fp8(int D, int G);

}  // namespace pkv
