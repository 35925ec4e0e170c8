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
//  * The work is the list of 16-token tiles of every (sequence, kv head) pair,
//    in (b, g, tile) order.  Every CTA rebuilds the per-sequence tile prefix
//    sum in shared memory, and worker warp w takes tiles
//    [w*T/P, (w+1)*T/P) -- an even split of the whole batch over all resident
//    warps, so long and short sequences balance without a host round trip.
//  * Each warp is its own pipeline: lane 0 issues TMA tensor copies (one K and
//    one V box of 16 tokens x head_dim for the warp's kv head) into a 3-stage
//    ring of shared-memory tiles, completion tracked by mbarrier transaction
//    counts.  Block-table entries for tile k+32 are fetched while tile k is
//    issued (one register per lane), so table lookups never stall the ring.
//  * One K/V read serves all G query heads of the group.  A token row is
//    split over D/8 lanes (16 bytes each); the per-lane partial dot products
//    of a tile are finished by a shuffle reduce-scatter, the softmax max is a
//    warp max, exponentials are ex2 on log2e-prescaled scores, and P.V uses
//    the same lane split with fp32 accumulators.
//  * A warp whose tile range covers a whole (b, g) writes bf16 output
//    directly; otherwise it leaves its (m, l, acc) in the workspace and counts
//    itself in on a per-(b, g) counter; the warp that brings in the last piece
//    merges them all (split-K / flash-decoding without a second kernel).
#include <algorithm>
#include <atomic>
#include <cstdio>
#include <mutex>
#include <type_traits>
#include <unordered_map>
#include <vector>
#include <cmath>

#include "pkv_device.cuh"
#include "pkv_host.h"

namespace pkv {

constexpr int kTile = 16;      // tokens per tile
constexpr int kMaxWarps = 12;  // warps per CTA (one CTA per SM) for small groups
constexpr int kStages = 2;     // ring depth per warp

// ------------------------------------------------------------------ load balance state
// The tile list is cut into one slice per SM id, each slice into equal
// per-warp ranges.  In the adaptive mode the slices' sizes follow what the
// previous call on this workspace saw: a slice that finished late gets a
// little less work, one that finished early a little more (SMs of a GB300
// stream HBM at noticeably different, but stable, rates).  This only moves
// work around: any table contents, garbage included, give correct results.
constexpr int kMaxSlots = 512;  // slices: SM ids (adaptive) or CTAs (fixed split)
constexpr uint32_t kTableMagic = 0x62616c31u;

struct BalanceState {
    float weight[2][kMaxSlots];           // weight a slice had in the call that wrote the entry (0: no SM)
    float elapsed[2][kMaxSlots];          // its run time in us (<= 0: present, nothing measured)
    uint32_t tag[2][kMaxSlots];           // (call number of the writer) ^ kTableMagic
    unsigned long long claim[kMaxSlots];  // (gen << 32) | 1 once a CTA took the slice this call
};

struct DecodeParams {
    const uint16_t *q;
    const int32_t *block_tables;
    const int32_t *context_lens;
    uint16_t *out;
    unsigned long long *ws_count;  // [B * Hkv] arrival counters: (call generation << 32) | tiles arrived
    float *ws_ml;        // [slots][G][2] (m, l) per partial
    float *ws_acc;       // [slots][G][D] unnormalised accumulators
    BalanceState *ws_bal;  // per-SM speed estimates, claims, call counter
    int32_t *err;
    int32_t B, Hq, Hkv, bs, log2_bs, NB, max_blocks, len_limit;
    int32_t num_workers;  // > 0: fixed split over ceil(num_workers / warps) CTAs; 0: adaptive split by SM
    float scale_log2;     // scale * log2(e)
    uint32_t gen;         // generation of this call (tags counters and claims)
    uint32_t call;        // number of this call on this workspace: call & 1 picks the table half written
};

struct alignas(16) StageMeta {
    int32_t b, g, t, n, L, seg_start, pad0, pad1;
};

template <int D, int G>
struct Shape {
    static constexpr int LPT = D / 8;          // lanes per token row (16 bytes each)
    static constexpr int TPI = 32 / LPT;       // tokens per warp step
    static constexpr int NIT = kTile / TPI;    // steps per tile
    static constexpr int DUP = LPT / NIT;      // lanes that end up holding each score
    static constexpr int KV_BYTES = kTile * D * 2;
    static constexpr int Q_BYTES = G * D * 2;
    static constexpr int STAGE_BYTES = (2 * KV_BYTES + Q_BYTES + 127) / 128 * 128;
    static_assert(LPT >= NIT && DUP >= 1, "tile too large for the lane split");
    // Warps per CTA: as many as the register file allows without spilling
    // (one CTA of WARPS*32 threads per SM, so at most 65536 / (WARPS*32) registers each).
    static constexpr int WARPS = (G <= 3 || (D == 64 && G <= 5)) ? kMaxWarps : 8;
};

struct WsLayout {
    size_t bal_off, count_off, ml_off, acc_off, total;
};

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Piece slots: one per (worker, sequence, kv head) boundary.  Worker ids
// (slice * warps + warp) stay below kWorkerIds in both modes.
constexpr size_t kWorkerIds = size_t(PKV_MAX_WORKERS) + 64;

inline WsLayout ws_layout(int32_t B, int32_t G, int32_t Hkv, int32_t D)
{
    const size_t slots = kWorkerIds + size_t(B) * size_t(Hkv);
    WsLayout w;
    w.bal_off = 0;
    w.count_off = align256(sizeof(BalanceState));
    w.ml_off = w.count_off + align256(size_t(B) * size_t(Hkv) * 8);
    w.acc_off = w.ml_off + align256(slots * size_t(G) * 2 * 4);
    w.total = w.acc_off + slots * size_t(G) * size_t(D) * 4;
    return w;
}

// ------------------------------------------------------------------ work list walking
struct Walker {
    int32_t b, g, t, n;
};

__device__ __forceinline__ void walker_advance(Walker &w, const int32_t *scan, int32_t Hkv, int32_t B)
{
    if (++w.t < w.n) return;
    w.t = 0;
    if (++w.g < Hkv) return;
    w.g = 0;
    do {
        ++w.b;
        w.n = (w.b < B) ? scan[w.b + 1] - scan[w.b] : 1;
    } while (w.n == 0);
}

// Position of global tile x (0 <= x < Hkv * scan[B]).
__device__ __forceinline__ Walker walker_locate(const int32_t *scan, int32_t B, int32_t Hkv, int64_t x)
{
    int lo = 0, hi = B;  // Hkv*scan[lo] <= x < Hkv*scan[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (int64_t(Hkv) * scan[mid] <= x)
            lo = mid;
        else
            hi = mid;
    }
    Walker w;
    w.b = lo;
    w.n = scan[lo + 1] - scan[lo];
    const int64_t rem = x - int64_t(Hkv) * scan[lo];
    w.g = int32_t(rem / w.n);
    w.t = int32_t(rem - int64_t(w.g) * w.n);
    return w;
}

__device__ __forceinline__ void table_lookup(const DecodeParams &p, const Walker &w, int nsub, int32_t &e0,
                                             int32_t &e1, int32_t &len)
{
    const int32_t *row = p.block_tables + int64_t(w.b) * p.max_blocks;
    const int32_t pos0 = w.t * kTile;
    e0 = __ldg(row + (pos0 >> p.log2_bs));
    if (nsub == 2) {
        const int32_t lb1 = (pos0 + kTile / 2) >> p.log2_bs;
        e1 = lb1 < p.max_blocks ? __ldg(row + lb1) : -1;
    }
    len = __ldg(p.context_lens + w.b);
}

// Tiles per sequence -> exclusive prefix in scan[0..B].
// `tmp` needs 32 ints of shared memory that is free during the call.
__device__ void tile_prefix_scan(const DecodeParams &p, int32_t *scan, int32_t *tmp)
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
            n = (len + kTile - 1) / kTile;
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

// One 16-token tile of one (sequence, kv head) for the G query heads of the group.
// Element pairs are handled with the packed fp32 FMA (two independent
// round-to-nearest fp32 FMAs per instruction).
template <int D, int G>
__device__ __forceinline__ void attend_tile(const uint8_t *st, int valid, const float2 (&q2)[G][4], float (&m)[G],
                                            float (&l)[G], float2 (&acc)[G][4], int c, int grp)
{
    using S = Shape<D, G>;
    constexpr int LPT = S::LPT, TPI = S::TPI, NIT = S::NIT, DUP = S::DUP;
    const uint16_t *Ks = reinterpret_cast<const uint16_t *>(st);
    const uint16_t *Vs = reinterpret_cast<const uint16_t *>(st + S::KV_BYTES);

    // scores: lane (grp, c) forms the 8-element partial dot products of tokens i*TPI + grp
    float part[G][NIT];
#pragma unroll
    for (int i = 0; i < NIT; ++i) {
        const int tok = i * TPI + grp;
        float2 k2[4];
        unpack8x2(*reinterpret_cast<const uint4 *>(Ks + tok * D + c * 8), k2);
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
        const float s = ok ? part[h][0] : -INFINITY;
        // Online softmax (m, l, acc).  The running max only moves when some
        // score passes it by more than the slack; the first tile always moves it
        // (m = -inf, and every tile holds at least one valid token).
        if (__any_sync(kFull, s > m[h] + kRescaleSlack)) {
            const float mn = fmaxf(m[h], warp_max(s));
            const float alpha = ex2(m[h] - mn);  // 0 on the first tile
            l[h] *= alpha;
            const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[h][j] = __fmul2_rn(acc[h][j], a2);
            m[h] = mn;
        }
        pr[h] = ok ? ex2(s - m[h]) : 0.f;
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
            unpack8x2(*reinterpret_cast<const uint4 *>(Vs + tok * D + c * 8), v2);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const float2 p2 = make_float2(ph[h], ph[h]);
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[h][j] = __ffma2_rn(p2, v2[j], acc[h][j]);
            }
        }
    }
}

// ------------------------------------------------------------------ partition
// Worker u = slice * nwarps + j owns the tiles
//   [bound[s] + len * j / nwarps, bound[s] + len * (j + 1) / nwarps),  len = bound[s+1] - bound[s].
// Worker ids grow with tile index, so a piece's workspace slot u + (b * Hkv + g)
// is unique (each step along the tile list raises u, or (b, g), or both).
struct Partition {
    const long long *bound;  // [nslots + 1] in shared memory
    int nslots, nwarps;

    __device__ __forceinline__ void range(long long u, long long &b, long long &e) const
    {
        const int s = int(u / nwarps), j = int(u - (long long)s * nwarps);
        const long long lo = bound[s], len = bound[s + 1] - lo;
        b = lo + len * j / nwarps;
        e = lo + len * (j + 1) / nwarps;
    }
    // The (non-empty) worker that owns tile x, 0 <= x < bound[nslots].
    __device__ __forceinline__ long long worker_of(long long x) const
    {
        int lo = 0, hi = nslots;  // bound[lo] <= x < bound[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (bound[mid] <= x)
                lo = mid;
            else
                hi = mid;
        }
        const long long b0 = bound[lo], len = bound[lo + 1] - b0;
        return (long long)lo * nwarps + ((x - b0 + 1) * nwarps - 1) / len;
    }
};

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

// Sum of one float per thread over the CTA (fixed order: identical in every CTA).
__device__ __forceinline__ float block_sum(float v, float *red)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
    v = warp_sum(v);
    __syncthreads();
    if (lane == 0) red[wid] = v;
    __syncthreads();
    float t = 0.f;
    for (int i = 0; i < nw; ++i) t += red[i];
    return t;
}

// Slice bounds of this call.  Adaptive mode: each slice entry of the table
// half written by the previous call on this workspace (call - 1) keeps its
// weight scaled by clamp(mean elapsed / its elapsed, 0.8, 1.25) (weight 0: an
// SM id without a CTA); entries from any other call count as unknown (weight
// 1).  Fixed mode: equal weights.  Every CTA computes the same bounds from the
// same inputs in the same order; leaves the weights in w[].
__device__ void build_partition(const DecodeParams &p, bool adaptive, int nslots, long long T, long long *bound,
                                float *w, float *red)
{
    const int tid = threadIdx.x, nt = blockDim.x;
    const int rp = int(p.call & 1u) ^ 1;
    const uint32_t want = (p.call - 1u) ^ kTableMagic;
    // pass 1: raw weights (kept in w) and elapsed times (kept in bound[] as float bits)
    float tsum = 0.f, tcnt = 0.f;
    float *el = reinterpret_cast<float *>(bound);
    for (int i = tid; i < nslots; i += nt) {
        float x = 1.0f, t = 0.f;
        // plain L2 loads: this half of the table is not written during this call
        if (adaptive && __ldcg(&p.ws_bal->tag[rp][i]) == want) {
            x = __ldcg(&p.ws_bal->weight[rp][i]);
            t = __ldcg(&p.ws_bal->elapsed[rp][i]);
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
    tsum = block_sum(tsum, red);
    tcnt = block_sum(tcnt, red);
    const float tmean = tcnt > 0.f ? tsum / tcnt : 0.f;
    // pass 2: scale by the finishing-time ratio, then bound every weight to [1/4, 4] x mean
    float wsum = 0.f, wcnt = 0.f;
    for (int i = tid; i < nslots; i += nt) {
        float x = w[i];
        const float t = el[i];
        if (x > 0.f && t > 0.f && tmean > 0.f) x *= fminf(fmaxf(tmean / t, 0.8f), 1.25f);
        w[i] = x;
        if (x > 0.f) {
            wsum += x;
            wcnt += 1.f;
        }
    }
    wsum = block_sum(wsum, red);
    wcnt = block_sum(wcnt, red);
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
__device__ int claim_leftover(const DecodeParams &p, const long long *bound, int nslots, int wp, bool record)
{
    const int lane = threadIdx.x & 31;
    for (int k0 = 0; blockIdx.x + (long long)k0 * gridDim.x < nslots; k0 += 32) {
        const long long s = blockIdx.x + (long long)(k0 + lane) * gridDim.x;
        bool cand = false;
        if (s < nslots) {
            const unsigned long long cur = *reinterpret_cast<volatile unsigned long long *>(&p.ws_bal->claim[s]);
            const bool claimed = uint32_t(cur >> 32) == p.gen;
            if (bound[s + 1] > bound[s]) {
                cand = !claimed;
            } else if (record) {
                p.ws_bal->weight[wp][s] = claimed ? 1.0f : 0.0f;
                p.ws_bal->elapsed[wp][s] = claimed ? -1.0f : 0.0f;
                p.ws_bal->tag[wp][s] = p.call ^ kTableMagic;
            }
        }
        unsigned m = __ballot_sync(kFull, cand);
        while (m) {
            const int l = __ffs(m) - 1;
            int ok = 0;
            if (lane == l) ok = try_claim(&p.ws_bal->claim[s], p.gen);
            if (__shfl_sync(kFull, ok, l)) return int(__shfl_sync(kFull, s, l));
            m &= m - 1;
        }
    }
    return -1;
}

// ------------------------------------------------------------------ split-K merge (a6)
// Count the `tiles` of one piece of (b, g) in.  The counter word is (call
// generation << 32) | tiles arrived; a word from another call (other
// generation, or leftover garbage) counts as zero, so the workspace never
// needs clearing.  Returns 1 for the piece that completes the pair's `total`
// tiles (and resets the word to 0).  Counting tiles, not pieces, lets any
// partition of the tile list merge correctly.
__device__ __forceinline__ int arrive_last(unsigned long long *ctr, uint32_t gen, uint32_t tiles, uint32_t total,
                                           int32_t *err)
{
    unsigned long long cur = *reinterpret_cast<volatile unsigned long long *>(ctr);
    for (int it = 0; it < (1 << 20); ++it) {
        const uint32_t n = ((uint32_t(cur >> 32) == gen) ? uint32_t(cur) : 0u) + tiles;
        const unsigned long long next = (static_cast<unsigned long long>(gen) << 32) | n;
        const unsigned long long seen = atomicCAS(ctr, cur, next);
        if (seen == cur) {
            if (n != total) return 0;
            atomicExch(ctr, 0ull);
            return 1;
        }
        cur = seen;
    }
    flag_error(err, PKV_ERR_WAIT_TIMEOUT);  // unreachable in practice: a handful of warps contend
    return 0;
}

// Merge the partial states of (b, g) held by the non-empty workers uf..ul:
//   M = max m_i,  l = sum 2^(m_i - M) l_i,  out = sum 2^(m_i - M) acc_i / l
// (the online-softmax algebra; m in log2 units).  The pieces were written by
// other SMs, so they are read through L2 (ld.global.cg), BATCH pieces at a
// time with independent loads, folded into a running (M, l, acc).
template <int D, int G>
__device__ __forceinline__ void merge_pieces(const DecodeParams &p, const Partition &part, long long bg, long long uf,
                                             long long ul, int b, int g, int lane)
{
    constexpr int PER = D / 32;                               // output values per lane
    constexpr int BATCH = G <= 2 ? 4 : (G <= 4 ? 2 : 1);      // pieces loaded together
    using Vec = typename std::conditional<PER == 4, float4, float2>::type;
    const float2 *ml = reinterpret_cast<const float2 *>(p.ws_ml);
    float M[G], lsum[G], a[G][PER];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        M[h] = -INFINITY;
        lsum[h] = 0.f;
#pragma unroll
        for (int e = 0; e < PER; ++e) a[h][e] = 0.f;
    }
    for (long long u0 = uf; u0 <= ul; u0 += BATCH) {
        float2 st[BATCH][G];
        Vec v[BATCH][G];
        bool use[BATCH];
#pragma unroll
        for (int k = 0; k < BATCH; ++k) {
            long long rb = 0, re = 0;
            if (u0 + k <= ul) part.range(u0 + k, rb, re);
            use[k] = re > rb;                               // empty workers wrote nothing
            const long long slot = (use[k] ? u0 + k : uf) + bg;
#pragma unroll
            for (int h = 0; h < G; ++h) {
                st[k][h] = __ldcg(ml + slot * G + h);
                v[k][h] = __ldcg(reinterpret_cast<const Vec *>(p.ws_acc + (slot * G + h) * D + lane * PER));
            }
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
            float mb = M[h];
#pragma unroll
            for (int k = 0; k < BATCH; ++k)
                if (use[k]) mb = fmaxf(mb, st[k][h].x);
            const float r = ex2(M[h] - mb);  // 0 while nothing has been folded in (M = -inf)
            lsum[h] *= r;
#pragma unroll
            for (int e = 0; e < PER; ++e) a[h][e] *= r;
#pragma unroll
            for (int k = 0; k < BATCH; ++k) {
                const float f = use[k] ? ex2(st[k][h].x - mb) : 0.f;
                lsum[h] = fmaf(f, st[k][h].y, lsum[h]);
                const float *x = reinterpret_cast<const float *>(&v[k][h]);
#pragma unroll
                for (int e = 0; e < PER; ++e) a[h][e] = fmaf(f, x[e], a[h][e]);
            }
            M[h] = mb;
        }
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
        const float inv = 1.0f / lsum[h];
        uint16_t *o = p.out + (int64_t(b) * p.Hq + int64_t(g) * G + h) * D + lane * PER;
        if constexpr (PER == 4)
            *reinterpret_cast<uint2 *>(o) = make_uint2(pack_bf16x2(a[h][0] * inv, a[h][1] * inv),
                                                       pack_bf16x2(a[h][2] * inv, a[h][3] * inv));
        else
            *reinterpret_cast<uint32_t *>(o) = pack_bf16x2(a[h][0] * inv, a[h][1] * inv);
    }
}

// ------------------------------------------------------------------ main kernel
template <int D, int G>
__global__ void __launch_bounds__(Shape<D, G>::WARPS * 32, 1)
    paged_decode_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                        const DecodeParams p)
{
    using S = Shape<D, G>;
    constexpr int LPT = S::LPT, DUP = S::DUP;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int nwarps = blockDim.x >> 5;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = lane % LPT, grp = lane / LPT;

    // shared memory: per-warp stage rings, their metadata and barriers, the
    // slice bounds, the sanitised slice weights, a few scalars, the tile prefix
    uint8_t *stages = smem + size_t(warp) * kStages * S::STAGE_BYTES;
    StageMeta *metas =
        reinterpret_cast<StageMeta *>(smem + size_t(nwarps) * kStages * S::STAGE_BYTES) + warp * kStages;
    uint64_t *bars =
        reinterpret_cast<uint64_t *>(smem + size_t(nwarps) * kStages * (S::STAGE_BYTES + sizeof(StageMeta))) +
        warp * kStages;
    long long *bound = reinterpret_cast<long long *>(smem + size_t(nwarps) * kStages *
                                                                (S::STAGE_BYTES + sizeof(StageMeta) + 8));
    float *wts = reinterpret_cast<float *>(bound + kMaxSlots + 1);
    float *red = wts + kMaxSlots;
    int *slice_sh = reinterpret_cast<int *>(red + 32);  // [0] slice to run next, [1] this CTA's own slice
    int32_t *scan = reinterpret_cast<int32_t *>(slice_sh + 4);

    if (threadIdx.x == 0) {
        prefetch_tensormap(&kmap);
        prefetch_tensormap(&vmap);
    }
    griddep_launch_dependents();  // lets the next kernel in the stream get scheduled; it waits for this grid
    griddep_wait();               // inputs may come from the previous kernel in the stream
    tile_prefix_scan(p, scan, reinterpret_cast<int32_t *>(smem));

    const long long T = (long long)p.Hkv * scan[p.B];
    // Sequences without tiles (L == 0, or a rejected length) get zeros; CTAs share the job.
    for (int b = blockIdx.x; b < p.B; b += gridDim.x)
        if (scan[b + 1] == scan[b])
            for (int i = threadIdx.x; i < p.Hq * D / 8; i += blockDim.x)
                reinterpret_cast<uint4 *>(p.out + int64_t(b) * p.Hq * D)[i] = make_uint4(0u, 0u, 0u, 0u);

    // Slices: one per SM id, sized by measured speed (adaptive), or one per CTA (fixed split).
    const bool adaptive = p.num_workers == 0;
    int nslots = int(gridDim.x);
    if (adaptive) {
        nslots = int(min(nsmid(), unsigned(kMaxSlots)));
        nslots = min(nslots, int(kWorkerIds / nwarps));
    }
    const int wp = int(p.call & 1u);  // this call writes one half of the balance table, reads the other
    build_partition(p, adaptive, nslots, T, bound, wts, red);
    const Partition part{bound, nslots, nwarps};

    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
        fence_barrier_init();
    }
    if (warp == 0) {
        int home = -1;
        if (lane == 0) {
            if (!adaptive)
                home = int(blockIdx.x);
            else if (int(smid()) < nslots && try_claim(&p.ws_bal->claim[smid()], p.gen))
                home = int(smid());
        }
        home = __shfl_sync(kFull, home, 0);
        const int first = (home < 0 && adaptive) ? claim_leftover(p, bound, nslots, wp, false) : home;
        if (lane == 0) {
            slice_sh[0] = first;
            slice_sh[1] = home;
        }
    }
    __syncthreads();

    const uint64_t policy = policy_evict_first();
    const int box = p.bs < kTile ? p.bs : kTile;
    const int nsub = kTile / box;
    uint32_t kk = 0;     // tiles this warp has consumed: selects ring stage and barrier phase
    bool dead = false;   // a wait timed out: do no more work

    // One worker's tile range [begin, end); u is the worker id (sets the piece slots).
    auto run_range = [&](long long begin, long long end, long long u) {
        const int ntiles = int(end - begin);

        // Block-table prefetch in batches of 32 tiles: lane j of `cur` holds the
        // table entries (and context length) of tile kb + j of the current batch;
        // `nxt` is loaded, all lanes at once, one batch ahead.  Two register sets,
        // because the scoreboard tracks a register for the whole warp: a fresh
        // load into the register that the next shuffle reads would stall it.
        Walker fw = walker_locate(scan, p.B, p.Hkv, begin);  // first tile not yet prefetched
        Walker iw = fw;                                       // next tile to issue
        int32_t cur0 = -1, cur1 = -1, curL = 0, nxt0 = -1, nxt1 = -1, nxtL = 0;
        auto prefetch_batch = [&](int kb) {  // tiles [kb, kb + 32) -> nxt; fw moves on to kb + 32
            Walker mine = fw;
    #pragma unroll 1
            for (int j = 0; j < 32 && kb + j < ntiles; ++j) {
                if (lane == j) mine = fw;
                if (kb + j + 1 < ntiles) walker_advance(fw, scan, p.Hkv, p.B);
            }
            if (kb + lane < ntiles) table_lookup(p, mine, nsub, nxt0, nxt1, nxtL);
        };
        prefetch_batch(0);
        cur0 = nxt0;
        cur1 = nxt1;
        curL = nxtL;
        if (ntiles > 32) prefetch_batch(32);

        auto issue = [&](int k, int s) {
            const int src = k & 31;
            if (src == 0 && k > 0) {  // batch boundary: nxt was loaded 32 tiles ago
                cur0 = nxt0;
                cur1 = nxt1;
                curL = nxtL;
                if (k + 32 < ntiles) prefetch_batch(k + 32);
            }
            const int32_t e0 = __shfl_sync(kFull, cur0, src);
            const int32_t e1 = __shfl_sync(kFull, cur1, src);
            const int32_t len = __shfl_sync(kFull, curL, src);
            if (lane == 0) {
                uint8_t *st = stages + s * S::STAGE_BYTES;
                const int seg_start = (k == 0 || iw.t == 0) ? 1 : 0;
                const int32_t pos0 = iw.t * kTile;
                int32_t row0 = -1, row1 = -1;
                if (e0 >= 0 && e0 < p.NB)
                    row0 = e0 * p.bs + (pos0 & (p.bs - 1));
                else
                    flag_error(p.err, PKV_ERR_BLOCK_RANGE);
                if (nsub == 2 && pos0 + box < len) {
                    if (e1 >= 0 && e1 < p.NB)
                        row1 = e1 * p.bs;
                    else
                        flag_error(p.err, PKV_ERR_BLOCK_RANGE);
                }
                const uint32_t sub_bytes = uint32_t(2 * box * D * 2);
                const uint32_t bytes = (row0 >= 0 ? sub_bytes : 0u) + (row1 >= 0 ? sub_bytes : 0u) +
                                       (seg_start ? uint32_t(S::Q_BYTES) : 0u);
                StageMeta &mt = metas[s];
                mt.b = iw.b;
                mt.g = iw.g;
                mt.t = iw.t;
                mt.n = iw.n;
                mt.L = len;
                mt.seg_start = seg_start;
                mbar_arrive_expect_tx(&bars[s], bytes);
                if (row0 >= 0) {
                    tma_load_3d(st, &kmap, 0, iw.g, row0, &bars[s], policy);
                    tma_load_3d(st + S::KV_BYTES, &vmap, 0, iw.g, row0, &bars[s], policy);
                }
                if (row1 >= 0) {
                    tma_load_3d(st + box * D * 2, &kmap, 0, iw.g, row1, &bars[s], policy);
                    tma_load_3d(st + S::KV_BYTES + box * D * 2, &vmap, 0, iw.g, row1, &bars[s], policy);
                }
                if (seg_start)
                    bulk_load(st + 2 * S::KV_BYTES, p.q + (int64_t(iw.b) * p.Hq + int64_t(iw.g) * G) * D,
                              S::Q_BYTES, &bars[s]);
            }
            if (k + 1 < ntiles) walker_advance(iw, scan, p.Hkv, p.B);
        };

        const int prologue = ntiles < kStages ? ntiles : kStages;
        for (int k = 0; k < prologue; ++k) issue(k, int((kk + k) % kStages));

        float2 q2[G][4], acc[G][4];
        float m[G], l[G];
        bool open = false;
        int32_t seg_t0 = 0;
        int k = 0;
        for (; k < ntiles; ++k) {
            const int s = int((kk + k) % kStages);
            if (!mbar_wait_bounded(&bars[s], uint32_t((kk + k) / kStages) & 1u)) {
                if (lane == 0) flag_error(p.err, PKV_ERR_WAIT_TIMEOUT);
                break;
            }
            const StageMeta mt = metas[s];
            const uint8_t *st = stages + s * S::STAGE_BYTES;
            if (!open) {
                open = true;
                seg_t0 = mt.t;
                const uint16_t *qs = reinterpret_cast<const uint16_t *>(st + 2 * S::KV_BYTES);
    #pragma unroll
                for (int h = 0; h < G; ++h) {
                    float2 f[4];
                    unpack8x2(*reinterpret_cast<const uint4 *>(qs + h * D + c * 8), f);
                    const float2 sc = make_float2(p.scale_log2, p.scale_log2);
    #pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        q2[h][j] = __fmul2_rn(f[j], sc);
                        acc[h][j] = make_float2(0.f, 0.f);
                    }
                    m[h] = -INFINITY;
                    l[h] = 0.f;
                }
            }
            const int valid = min(kTile, mt.L - mt.t * kTile);
            attend_tile<D, G>(st, valid, q2, m, l, acc, c, grp);
            __syncwarp();
            if (k + kStages < ntiles) issue(k + kStages, s);

            if (mt.t == mt.n - 1 || k == ntiles - 1) {
                // close the segment: fold the token groups, then write out or leave a partial
    #pragma unroll
                for (int mask = LPT; mask < 32; mask <<= 1)
    #pragma unroll
                    for (int h = 0; h < G; ++h)
    #pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            acc[h][j].x += __shfl_xor_sync(kFull, acc[h][j].x, mask);
                            acc[h][j].y += __shfl_xor_sync(kFull, acc[h][j].y, mask);
                        }
                float lt[G];
    #pragma unroll
                for (int h = 0; h < G; ++h) lt[h] = warp_sum(l[h]) * (1.0f / DUP);
                const int piece_tiles = mt.t - seg_t0 + 1;
                if (piece_tiles == mt.n) {  // this warp ran the whole (b, g): write the output
                    if (grp == 0) {
    #pragma unroll
                        for (int h = 0; h < G; ++h) {
                            const float inv = 1.0f / lt[h];
                            uint4 o;
                            o.x = pack_bf16x2(acc[h][0].x * inv, acc[h][0].y * inv);
                            o.y = pack_bf16x2(acc[h][1].x * inv, acc[h][1].y * inv);
                            o.z = pack_bf16x2(acc[h][2].x * inv, acc[h][2].y * inv);
                            o.w = pack_bf16x2(acc[h][3].x * inv, acc[h][3].y * inv);
                            *reinterpret_cast<uint4 *>(p.out + (int64_t(mt.b) * p.Hq + int64_t(mt.g) * G + h) * D +
                                                       c * 8) = o;
                        }
                    }
                } else {
                    const int64_t slot = u + int64_t(mt.b) * p.Hkv + mt.g;
                    if (grp == 0) {
    #pragma unroll
                        for (int h = 0; h < G; ++h) {
                            float4 *dst = reinterpret_cast<float4 *>(p.ws_acc + ((slot * G + h) * D + c * 8));
                            dst[0] = make_float4(acc[h][0].x, acc[h][0].y, acc[h][1].x, acc[h][1].y);
                            dst[1] = make_float4(acc[h][2].x, acc[h][2].y, acc[h][3].x, acc[h][3].y);
                        }
                    }
                    if (lane == 0)
    #pragma unroll
                        for (int h = 0; h < G; ++h)
                            reinterpret_cast<float2 *>(p.ws_ml)[slot * G + h] = make_float2(m[h], lt[h]);
                    // Publish the piece, then count it in; the warp that brings in the last
                    // piece of this (b, g) merges them all.
                    __threadfence();
                    __syncwarp();
                    const int64_t bg = int64_t(mt.b) * p.Hkv + mt.g;
                    int last = 0;
                    if (lane == 0)
                        last = arrive_last(p.ws_count + bg, p.gen, uint32_t(piece_tiles), uint32_t(mt.n), p.err);
                    if (__shfl_sync(kFull, last, 0)) {
                        __threadfence();
                        const long long x0 = (long long)p.Hkv * scan[mt.b] + (long long)mt.g * mt.n;
                        merge_pieces<D, G>(p, part, bg, part.worker_of(x0), part.worker_of(x0 + mt.n - 1), mt.b,
                                           mt.g, lane);
                    }
                }
                open = false;
            }
        }
        if (k < ntiles) {
            // gave up on a wait: let every copy still in flight land, then stop for good
            for (int j = k; j < ntiles && j < k + kStages; ++j)
                mbar_wait_bounded(&bars[(kk + j) % kStages], uint32_t((kk + j) / kStages) & 1u);
            dead = true;
        }
        kk += uint32_t(ntiles);

    };

    unsigned long long t_home = 0;
    for (;;) {
        const int slice = slice_sh[0];
        if (slice < 0) break;
        const bool home = slice == slice_sh[1];
        if (home && threadIdx.x == 0) t_home = global_ns();
        const long long u = (long long)slice * nwarps + warp;
        long long rb, re;
        part.range(u, rb, re);
        if (re > rb && !dead) run_range(rb, re, u);
        __syncthreads();
        if (warp == 0) {
            int next = -1;
            if (adaptive) {
                if (lane == 0 && bound[slice + 1] > bound[slice]) {
                    // record for the next call: the weight this slice had and how long it took,
                    // or "absent" when an SM id without a CTA of its own left it to this CTA
                    const float us = float(global_ns() - t_home) * 1e-3f;
                    p.ws_bal->weight[wp][slice] = home ? wts[slice] : 0.f;
                    p.ws_bal->elapsed[wp][slice] = home ? fmaxf(us, 1e-3f) : 0.f;
                    p.ws_bal->tag[wp][slice] = p.call ^ kTableMagic;
                }
                next = claim_leftover(p, bound, nslots, wp, true);
            }
            if (lane == 0) slice_sh[0] = next;
        }
        __syncthreads();
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

inline bool encode_cache_map(CUtensorMap *map, const void *base, int D, int Hkv, int64_t rows, int box_rows)
{
    EncodeTiledFn enc = encode_tiled_fn();
    if (!enc) {
        record_cuda_error("cuTensorMapEncodeTiled", "driver entry point unavailable");
        return false;
    }
    const cuuint64_t dims[3] = {cuuint64_t(D), cuuint64_t(Hkv), cuuint64_t(rows)};
    const cuuint64_t strides[2] = {cuuint64_t(D) * 2, cuuint64_t(Hkv) * D * 2};
    const cuuint32_t box[3] = {cuuint32_t(D), 1u, cuuint32_t(box_rows)};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
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
inline bool cached_cache_map(CUtensorMap *map, int dev, const void *base, int D, int Hkv, int64_t rows, int box_rows)
{
    struct Entry {
        int dev;
        const void *base;
        int D, Hkv;
        int64_t rows;
        int box;
        CUtensorMap map;
    };
    constexpr size_t kMaxEntries = 256;
    static std::mutex mu;
    static std::vector<Entry> cache;
    std::lock_guard<std::mutex> lock(mu);
    for (size_t i = 0; i < cache.size(); ++i) {
        const Entry &e = cache[i];
        if (e.dev == dev && e.base == base && e.D == D && e.Hkv == Hkv && e.rows == rows && e.box == box_rows) {
            *map = e.map;
            return true;
        }
    }
    if (!encode_cache_map(map, base, D, Hkv, rows, box_rows)) return false;
    if (cache.size() >= kMaxEntries) cache.erase(cache.begin());
    cache.push_back(Entry{dev, base, D, Hkv, rows, box_rows, *map});
    return true;
}

// cudaFuncSetAttribute once per device and kernel variant (it is a host-side
// driver call; repeating it on every launch costs microseconds).  Keyed on
// <D, G>: every variant has the same function-pointer type, so the memo must
// be per instantiation.
template <int D, int G, typename Kernel>
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

// Number of this call on this workspace (per device).  The kernel keeps its
// load-balance table in the workspace, one half written per call: this number
// picks the half, and the previous call's entries are recognised by its
// number minus one.  A host-side memo only: losing it costs one call of
// balance, never results.
inline uint32_t next_call_number(int dev, const void *workspace)
{
    static std::mutex mu;
    static std::unordered_map<uintptr_t, uint32_t> calls[64];
    if (dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lock(mu);
    auto &m = calls[dev];
    if (m.size() > 65536) m.clear();
    return ++m[reinterpret_cast<uintptr_t>(workspace)];
}

template <int D, int G>
size_t decode_smem_bytes(int nwarps, int B)
{
    using S = Shape<D, G>;
    return size_t(nwarps) * kStages * (S::STAGE_BYTES + sizeof(StageMeta) + 8)  // rings, metadata, barriers
           + size_t(kMaxSlots + 1) * 8 + size_t(kMaxSlots) * 4 + 32 * 4 + 16     // bounds, weights, scalars
           + size_t(B + 1) * 4;                                                  // tile prefix
}

template <int D, int G>
pkv_status launch_decode(LaunchArgs &a)
{
    int nwarps = Shape<D, G>::WARPS;
    while (nwarps > 1 && decode_smem_bytes<D, G>(nwarps, a.p.B) > size_t(a.max_smem)) --nwarps;
    const size_t smem = decode_smem_bytes<D, G>(nwarps, a.p.B);
    if (smem > size_t(a.max_smem)) return PKV_EUNSUPPORTED;

    // Adaptive split: one CTA per SM, slices keyed by SM id.  Fixed split: the
    // requested worker count rounded up to whole CTAs.
    int grid = a.sm_count;
    a.p.num_workers = 0;
    if (a.requested_workers > 0) {
        grid = (a.requested_workers + nwarps - 1) / nwarps;
        if (grid > kMaxSlots) grid = kMaxSlots;
        a.p.num_workers = a.requested_workers;
    }

    const int box = a.p.bs < kTile ? a.p.bs : kTile;
    CUtensorMap kmap, vmap;
    const int64_t rows = int64_t(a.p.NB) * a.p.bs;
    if (!cached_cache_map(&kmap, a.device, a.k_cache, D, a.p.Hkv, rows, box) ||
        !cached_cache_map(&vmap, a.device, a.v_cache, D, a.p.Hkv, rows, box))
        return PKV_ECUDA;

    auto kern = paged_decode_kernel<D, G>;
    if (!ensure_smem_attribute<D, G>(kern, a.device, smem)) return PKV_ECUDA;
    const cudaError_t e = launch_pdl(kern, dim3(grid), dim3(nwarps * 32), smem, a.stream, kmap, vmap, a.p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return cuda_fail("paged_decode_kernel launch", e);
    }
    return launch_status("paged_decode_kernel launch");
}

using LaunchFn = pkv_status (*)(LaunchArgs &);

template <int D>
LaunchFn pick_group(int G)
{
    switch (G) {
    case 1: return launch_decode<D, 1>;
    case 2: return launch_decode<D, 2>;
    case 3: return launch_decode<D, 3>;
    case 4: return launch_decode<D, 4>;
    case 5: return launch_decode<D, 5>;
    case 6: return launch_decode<D, 6>;
    case 7: return launch_decode<D, 7>;
    case 8: return launch_decode<D, 8>;
    default: return nullptr;
    }
}

}  // namespace pkv

using namespace pkv;

extern "C" size_t pkv_paged_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                                  int32_t head_dim)
{
    if (num_seqs < 0 || num_seqs > PKV_MAX_SEQS || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        num_q_heads % num_kv_heads != 0)
        return 0;
    return ws_layout(num_seqs, num_q_heads / num_kv_heads, num_kv_heads, head_dim).total;
}

extern "C" pkv_status pkv_paged_decode(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                                       const int32_t *block_tables, int32_t max_blocks_per_seq,
                                       const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                                       int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                       int32_t num_blocks, int32_t max_context_len, float scale, uint16_t *out,
                                       void *workspace, size_t workspace_bytes, int32_t num_workers,
                                       int32_t *err_word, pkv_stream_t stream)
{
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 ||
        head_dim <= 0 || block_size <= 0 || num_blocks <= 0 || max_blocks_per_seq <= 0 || max_context_len < 0 ||
        num_workers < 0 || num_workers > PKV_MAX_WORKERS || !std::isfinite(scale))
        return PKV_EINVAL;
    if (num_seqs > PKV_MAX_SEQS) return PKV_EUNSUPPORTED;
    if (head_dim != 64 && head_dim != 128) return PKV_EUNSUPPORTED;
    const int G = num_q_heads / num_kv_heads;
    if (G > 8) return PKV_EUNSUPPORTED;
    if (!is_pow2(block_size) || block_size < 8 || block_size > 1024) return PKV_EUNSUPPORTED;
    if (int64_t(num_blocks) * block_size > INT32_MAX) return PKV_EUNSUPPORTED;
    if (num_seqs == 0) return PKV_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out) return PKV_EINVAL;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out)) return PKV_EINVAL;
    const int64_t len_limit = std::min<int64_t>(max_context_len, int64_t(max_blocks_per_seq) * block_size);
    const int64_t max_tiles = int64_t(num_seqs) * ((len_limit + kTile - 1) / kTile);
    if (max_tiles > INT32_MAX) return PKV_EUNSUPPORTED;
    if (num_workers > 0 && int64_t(num_kv_heads) * max_tiles / num_workers + 1 > INT32_MAX) return PKV_EUNSUPPORTED;
    const WsLayout ws = ws_layout(num_seqs, G, num_kv_heads, head_dim);
    if (!workspace || workspace_bytes < ws.total || !aligned16(workspace)) return PKV_EWORKSPACE;

    DeviceInfo dev;
    if (!current_device_info(&dev)) return PKV_ECUDA;

    LaunchArgs a;
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
    p.num_workers = 0;
    p.scale_log2 = float(double(scale) * 1.4426950408889634);
    static std::atomic<uint32_t> generation{0};
    p.gen = generation.fetch_add(1u, std::memory_order_relaxed) + 1u;
    p.call = next_call_number(dev.device, workspace);
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.device = dev.device;
    a.sm_count = dev.sm_count;
    a.max_smem = dev.max_smem_optin;
    a.requested_workers = num_workers;
    a.stream = reinterpret_cast<cudaStream_t>(stream);

    LaunchFn fn = head_dim == 64 ? pick_group<64>(G) : pick_group<128>(G);
    if (!fn) return PKV_EUNSUPPORTED;
    return fn(a);
}

// ------------------------------------------------------------------ allocation-free variant
// Some callers cannot hand the library a workspace: an engine that gave
// (nearly) all free device memory to its KV block pool at start-up, or a host
// framework whose plugin interface passes only inputs and outputs and forbids
// device allocations while it runs.  For them the decode scratch lives in a
// fixed array owned by this library: kStaticScratchBytes on every device that
// loads it, held until the process exits.
#include <mutex>

namespace pkv {

constexpr size_t kStaticScratchBytes = size_t(PKV_NOALLOC_SCRATCH_BYTES);
static __device__ __align__(256) uint8_t g_decode_scratch[kStaticScratchBytes];

// Device address of g_decode_scratch on the current device.  The name of the
// array in host code is only a host-side stand-in, so the address is asked of
// the runtime once per device (with that device current) and cached.
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
    if (num_seqs == 0 || need == 0)  // nothing to do, or invalid sizes: the regular checks answer
        return pkv_paged_decode(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                                num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, max_context_len, scale,
                                out, nullptr, 0, num_workers, err_word, stream);
    pkv_status st = PKV_OK;
    void *scratch = static_scratch_address(&st);
    if (!scratch) return st;
    return pkv_paged_decode(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                            num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, max_context_len, scale, out,
                            scratch, kStaticScratchBytes, num_workers, err_word, stream);
}
