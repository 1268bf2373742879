// decode_attn.cu -- degree-aware decode attention over a (compressed) KV cache.
// [Chelsea §三 核心公式: O = softmax(q K^T / sqrt(d) + log N) V; CentroidKV 聚合]
//
// The log-degree bias is applied as a weight: e^(x + log n) = n e^x, so the
// online softmax keeps (m, l, acc) with p_t = n_t * 2^(x_t - m), x_t the
// base-2 scaled logit. No log is evaluated and integer degrees stay exact.
//
// Work split (bf16). Every unit's tokens are cut into fixed splits: a base
// length S (a multiple of the 64-token tile) chosen from the call's total so
// that an equal share of the GPU is about kItemsPerCta splits, longer for long
// units so no unit has more than kMaxSplitsPerUnit splits. The split boundaries
// depend only on the lengths. A persistent grid (two CTAs per SM) takes splits
// from one atomic ticket, units with many splits first, so the merges of the
// long units' partial states happen early and the last wave is made of short
// splits; SMs that stream faster simply take more splits. Inside a CTA one
// producer warp claims the next split while the current one streams and feeds
// K, V (128-byte swizzled, 2 boxes of 64 columns) and the degree tile into a
// 3-stage TMA/mbarrier ring, tagging every stage with its split. Four consumer
// warps each take 16 tokens of a tile and run S^T = K q^T and O^T += V^T P^T on
// mma.sync (bf16 in, fp32 accumulate), the G <= 8 query heads of the group in
// the N = 8 dimension, so each K/V byte is read once for the whole group. At a
// split's end the CTA merges its warps' states in shared memory (warp order)
// into one partial record per split. A second, small kernel (one CTA per unit
// and query head, launched to overlap the first one's end) merges every unit's
// records in split order into the output: records are indexed by split, so the
// result does not depend on which CTA ran which split, and no merge waits on a
// streaming CTA. The unit order and split offsets come from scans of the
// lengths inside every CTA (batches of up to kMaxScanUnits units), or from a
// one-CTA prologue for larger batches; while a CTA plans, its producer warp has
// L2 prefetch a slice of rows the call is sure to read (prefetch_piece), so HBM
// works from the first microsecond.
// After a device error the workspace must be zero-filled again before reuse.
#include <cuda_bf16.h>

#include <cmath>

#include "host_util.h"
#include "ptx.cuh"

namespace csmkv {

constexpr int kTile = 64;
constexpr int kConsumerWarps = 4;
constexpr int kDecThreads = (kConsumerWarps + 1) * 32;
constexpr int kStages = 3;
constexpr int kDecCtasPerSm = 2;
constexpr int kMaxScanUnits = 512;     // units whose plan a CTA computes itself
constexpr int kUnitBits = 9;           // scan tables pack (len << kUnitBits) | unit
#ifndef CSMKV_DEC_ITEMS
#define CSMKV_DEC_ITEMS 6
#endif
#ifndef CSMKV_DEC_MAX_SPLITS
#define CSMKV_DEC_MAX_SPLITS 40
#endif
constexpr int kItemsPerCta = CSMKV_DEC_ITEMS;           // splits per equal share of the GPU
#ifndef CSMKV_DEC_MIN_SPLIT
#define CSMKV_DEC_MIN_SPLIT 256
#endif
constexpr int kMinSplit = CSMKV_DEC_MIN_SPLIT;          // tokens (4 tiles: per-split costs stay small)
static_assert(kMinSplit % 64 == 0 && kMinSplit > 0, "the minimum split is a whole number of tiles");
constexpr int kMaxSplitsPerUnit = CSMKV_DEC_MAX_SPLITS;  // bounds the records one unit's merge reads
#ifndef CSMKV_DEC_PREFETCH_DIV
#define CSMKV_DEC_PREFETCH_DIV 4
#endif
#ifndef CSMKV_DEC_PREFETCH_MAX
#define CSMKV_DEC_PREFETCH_MAX 1024
#endif
// rows a CTA pulls into L2 while the call is planned: 1/kPrefetchDiv of its share
// of the call, in [64, kPrefetchMax] (0: none)
constexpr int kPrefetchDiv = CSMKV_DEC_PREFETCH_DIV;
constexpr int kPrefetchMax = CSMKV_DEC_PREFETCH_MAX;
constexpr uint32_t kFirst = 1u, kLast = 2u;
constexpr int kSlotHeads = 8;          // query heads of a group the MMA covers (N = 8)
#ifndef CSMKV_DEC_CLAIM_EARLY
#define CSMKV_DEC_CLAIM_EARLY 0
#endif

// Base split length for `total` tokens on n CTAs: about kItemsPerCta splits per
// CTA, a multiple of the tile, at least kMinSplit. Since S >= total / (n *
// kItemsPerCta), a call has at most n * kItemsPerCta + units splits.
__host__ __device__ __forceinline__ int split_base(int total, int n) {
    const unsigned per = (unsigned)n * kItemsPerCta;
    unsigned s = ((unsigned)total + per - 1u) / per;
    s = (s + kTile - 1u) / kTile * kTile;
    return (int)(s > (unsigned)kMinSplit ? s : (unsigned)kMinSplit);
}
// Split length of a unit of `len` rows (of `total` over n CTAs): the base S, or
// longer for a long unit, so that it has at most kMaxSplitsPerUnit splits -- or,
// if it alone is a large part of the call, about one split per CTA of its share.
// (The share is taken in fp32: the same operations give the same result in
// every CTA and in the prologue.)
__device__ __forceinline__ int unit_split(int len, int S, int total, int n) {
    int cap = total > 0 ? (int)((float)n * ((float)len / (float)total)) : 0;
    if (cap < kMaxSplitsPerUnit) cap = kMaxSplitsPerUnit;
    unsigned su = ((unsigned)len + (unsigned)cap - 1u) / (unsigned)cap;
    su = (su + kTile - 1u) / kTile * kTile;
    return (int)su > S ? (int)su : S;
}
__device__ __forceinline__ int unit_nsplit(int len, int su) { return (len + su - 1) / su; }
// Ticket order: units whose splits were lengthened first (long units: the
// longest splits and merges), then units with many splits, then the rest.
__device__ __forceinline__ int unit_class(int n, int su, int S) {
    return su > S ? 0 : (n >= 16 ? 1 : (n >= 4 ? 2 : 3));
}

// At most total / S <= nCTA * kItemsPerCta splits plus one per unit.
__host__ __device__ __forceinline__ int dec_max_splits(int nCTA, int BH) { return nCTA * kItemsPerCta + BH; }

struct DecParams {
    const void* q;
    const int32_t* len;
    // fused append (k_new != NULL): every unit's new token is written at row len and
    // attended, and len grows by one at the end of the call
    const void* k_new;    // [BH][D]
    const void* v_new;    // [BH][D]
    void* K;
    void* V;
    int32_t* N;
    int32_t* len_rw;      // the same array as len
    void* out;
    WsHeader* hdr;
    int32_t* g_first;     // [BH] first split of every unit (written by the plan)
    int32_t* g_n;         // [BH] splits of every unit
    int32_t* g_len;       // prologue path: [BH] rows attended per unit
    int32_t* g_unit;      // prologue path: [max splits] unit of every split
    float* pm;            // [splits][G] running max (base-2 domain)
    float* pl;            // [splits][G] running sum
    float* pacc;          // [splits][G][D] unnormalised output
    RowMap rm;            // logical row -> pool row (dense, or through a block table)
    int32_t pool_rows;    // rows of the K / V / N tensors the TMA maps cover
    int32_t BH, Hkv, Hq, G, cap, D, nCTA, max_splits;
    float scale_log2;     // scale * log2(e)
    float scale;          // natural-log scale (fp32 path)
};

// Rows of unit u this call attends: len, plus the appended token in fused-append
// mode (a full unit records CSMKV_ERR_CAPACITY and is attended as it is).
__device__ __forceinline__ int eff_len(const DecParams& p, int u, bool record) {
    int v = p.len[u];
    if (v < 0 || v > p.cap) {
        if (record) record_status(&p.hdr->status, CSMKV_ERR_ARG);
        return 0;
    }
    if (p.k_new) {
        if (v < p.cap) ++v;
        else if (record) record_status(&p.hdr->status, CSMKV_ERR_CAPACITY);
    }
    return v;
}

// Exclusive scan of 8 counters per thread over the block (threads in index
// order); tot gets the block totals. scratch: one row of 8 per warp.
__device__ __forceinline__ void block_scan8(int (&v)[8], int (&tot)[8], int (*scratch)[8]) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int incl[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        incl[i] = v[i];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int x = __shfl_up_sync(0xffffffffu, incl[i], o);
            if (lane >= o) incl[i] += x;
        }
        if (lane == 31) scratch[warp][i] = incl[i];
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        int base = 0, t = 0;
        for (int w = 0; w < nw; ++w) {
            const int x = scratch[w][i];
            if (w < warp) base += x;
            t += x;
        }
        v[i] = base + incl[i] - v[i];
        tot[i] = t;
    }
    __syncthreads();  // scratch may be reused
}

// ----------------------------------------------------------------------------
// Prologue (one CTA, batches of more than kMaxScanUnits units): rows per unit,
// the base split length, every unit's first split and split count (units in
// index order) and the unit of every split.
__global__ void __launch_bounds__(1024) decode_prologue_kernel(const DecParams p) {
    griddep_launch_dependents();  // the main kernel may set itself up meanwhile
    __shared__ int scratch[32][8];
    __shared__ int carry_s[2];
    const int tid = threadIdx.x;
    long long total = 0;
    for (int base = 0; base < p.BH; base += 1024) {
        const int u = base + tid;
        int v[8] = {u < p.BH ? eff_len(p, u, true) : 0, 0, 0, 0, 0, 0, 0, 0}, t[8];
        if (u < p.BH) p.g_len[u] = v[0];
        block_scan8(v, t, scratch);
        total += t[0];
    }
    const int S = split_base((int)total, p.nCTA);
    if (tid == 0) {
        carry_s[1] = 0;
        p.hdr->dec_total = (int32_t)total;
    }
    const int total32 = (int)total;
    __syncthreads();
    for (int base = 0; base < p.BH; base += 1024) {
        const int u = base + tid;
        const int len = u < p.BH ? p.g_len[u] : 0;
        const int n = len > 0 ? unit_nsplit(len, unit_split(len, S, total32, p.nCTA)) : 0;
        int w[8] = {n, 0, 0, 0, 0, 0, 0, 0}, t2[8];
        block_scan8(w, t2, scratch);
        const int first = carry_s[1] + w[0];
        if (u < p.BH) {
            p.g_first[u] = first;
            p.g_n[u] = n;
            for (int k = 0; k < n; ++k) p.g_unit[first + k] = u;
        }
        __syncthreads();
        if (tid == 0) carry_s[1] += t2[0];
        __syncthreads();
    }
    if (tid == 0) {
        p.hdr->dec_nsplits = carry_s[1];
        p.hdr->dec_split = S;
    }
}

// ----------------------------------------------------------------------------
template <int D>
struct DecGeom {
    static constexpr int kBoxes = D / 64;
    static constexpr int kBoxBytes = kTile * 128;              // 64 rows x 128 B
    static constexpr int kKOff = 0;
    static constexpr int kVOff = kBoxes * kBoxBytes;
    static constexpr int kStageBytes = 2 * kBoxes * kBoxBytes;  // K and V boxes; 1024-aligned
    static constexpr int kNBytes = (kTile / 4 + 1) * 16;       // 68 degrees (row rounded down to 4)
    static constexpr int kNStride = 384;                       // degree tiles after the ring
    static constexpr uint32_t kTxBytes = kStageBytes + kNBytes;
    static constexpr int kQBytes = kSlotHeads * D * 2;          // the group's query rows (first tile of a split)
    static constexpr int kQOff = kStages * kStageBytes + kStages * kNStride;
    static constexpr int kSmallOff = kQOff + kStages * kQBytes;
};

// Shared scratch for merging partial softmax states: per-warp head maxima and
// sums, and one fp32 row per head. The head stride of 132 floats puts the
// fragment stores of a warp (lanes 4g + t4 -> head 2 t4 or 2 t4 + 1, dim g) on
// 32 distinct banks.
constexpr int kRedStride = 132;
struct CombineScratch {
    float m[kConsumerWarps][kSlotHeads];
    float l[kConsumerWarps][kSlotHeads];
    float acc[kSlotHeads][kRedStride];
};

// What a stage holds: which split, which unit, where in the unit.
struct StageMeta {
    int32_t t;      // split (ticket); < 0: no more work
    int32_t unit;
    int32_t k;      // split index within the unit
    int32_t n;      // splits of the unit
    int32_t tok;    // first token of the tile within the unit
    int32_t nv;     // valid tokens in the tile
    uint32_t flags; // kFirst / kLast tile of the split
    int32_t pad;
};

// Scratch of the main kernel after the stage ring.
struct DecSmall {
    CombineScratch cs;
    StageMeta meta[kStages];
    uint64_t full[kStages];
    uint64_t empty[kStages];
    int scan[kDecThreads / 32][8];
    int abort_flag;
    int nsplits;
    int S;
    int total;
};

// One split, resolved from its ticket.
struct Split {
    int t, u, k, n, len, su;
    int tok0, ntok;  // the split's rows within the unit
};

__device__ __forceinline__ void consumer_barrier() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

// Barrier over the consumer warps that also ORs a predicate: every consumer
// thread gets the same answer, so all of them take the same branch after it.
__device__ __forceinline__ bool consumer_any(bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n"
        " setp.ne.u32 q, %1, 0;\n"
        " bar.red.or.pred p, 1, %2, q;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(kConsumerWarps * 32)
        : "memory");
    return r != 0;
}

// Ticket -> split. SCAN: the CTA's own tables (positions in ticket order: sp =
// first split, ulen = len << kUnitBits | unit); otherwise the prologue's global
// tables (units in index order, g_unit maps a split to its unit).
template <bool SCAN>
__device__ __forceinline__ Split resolve_split(const DecParams& p, int t, int nsplits, int S, int total,
                                               const int* sp, const uint32_t* ulen) {
    Split r;
    r.t = -1;
    if (t < 0 || t >= nsplits) return r;
    int first;
    if constexpr (SCAN) {
        int lo = 0, hi = p.BH;  // last position with first split <= t
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (sp[mid] <= t) lo = mid; else hi = mid;
        }
        const uint32_t x = ulen[lo];
        r.u = (int)(x & ((1u << kUnitBits) - 1u));
        r.len = (int)(x >> kUnitBits);
        first = sp[lo];
        r.n = sp[lo + 1] - first;
    } else {
        r.u = __ldcg(p.g_unit + t);
        r.len = __ldcg(p.g_len + r.u);
        first = __ldcg(p.g_first + r.u);
        r.n = __ldcg(p.g_n + r.u);
    }
    r.t = t;
    r.k = t - first;
    r.su = unit_split(r.len, S, total, p.nCTA);
    r.tok0 = r.k * r.su;
    r.ntok = min(r.su, r.len - r.tok0);
    return r;
}

// Merges the split records of every unit into the output, one CTA per (unit,
// query head of the group). Each thread owns 4 output columns and every RL-th
// record of the unit; it loads up to kCombBatch of its records at once (all
// loads in flight before any arithmetic: the records sit in L2, possibly on the
// other die, so a dependent chain would pay the full latency per record), folds
// them in split order with a running maximum, and the RL partial states are
// merged in a fixed order (deterministic). Empty units get a zero output. After
// its merge, the CTA for (0, 0) resets the split ticket for the next call and,
// with a fused append, moves every length past its new token: the main kernel,
// which read the lengths, has completed when griddepcontrol.wait returns.
constexpr int kCombThreads = 256;
constexpr int kCombBatch = 8;
template <int D>
__global__ void __launch_bounds__(kCombThreads) decode_combine_kernel(const DecParams p) {
    constexpr int C4 = D / 4;              // float4 columns of one head
    constexpr int RL = kCombThreads / C4;  // record lanes: 8 (D = 128) or 16 (D = 64)
    __shared__ float sm_m[RL], sm_l[RL];
    __shared__ float4 sm_acc[RL][C4];
    griddep_launch_dependents();  // the next kernel may set itself up meanwhile
    griddep_wait();
    const int u = blockIdx.x, g = blockIdx.y, tid = threadIdx.x;
    const int first = p.g_first[u], n = p.g_n[u];
    const int b = u / p.Hkv, kv = u - b * p.Hkv;
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out) + ((size_t)b * p.Hq + (size_t)kv * p.G + g) * D;
    if (n <= 0) {
        for (int i = tid; i < D / 8; i += kCombThreads) reinterpret_cast<uint4*>(o)[i] = make_uint4(0u, 0u, 0u, 0u);
    } else {
        const int c = tid % C4, rl = tid / C4;
        float m = -INFINITY, l = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int r0 = rl; r0 < n; r0 += RL * kCombBatch) {
            float pmv[kCombBatch], plv[kCombBatch];
            float4 v[kCombBatch];
#pragma unroll
            for (int j = 0; j < kCombBatch; ++j) {
                const int r = r0 + j * RL;
                pmv[j] = -INFINITY;
                plv[j] = 0.f;
                v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (r < n) {
                    const size_t rec = (size_t)(first + r) * p.G + g;
                    pmv[j] = __ldcg(p.pm + rec);
                    plv[j] = __ldcg(p.pl + rec);
                    v[j] = __ldcg(reinterpret_cast<const float4*>(p.pacc + rec * D) + c);
                }
            }
#pragma unroll
            for (int j = 0; j < kCombBatch; ++j) {
                // a record of a head that saw no token holds m = -inf, l = 0, acc = 0
                if (pmv[j] == -INFINITY) continue;
                const float mn = fmaxf(m, pmv[j]);
                const float a = (m == -INFINITY) ? 0.f : exp2f(m - mn);
                const float f = exp2f(pmv[j] - mn);
                l = fmaf(f, plv[j], l * a);
                acc.x = fmaf(f, v[j].x, acc.x * a);
                acc.y = fmaf(f, v[j].y, acc.y * a);
                acc.z = fmaf(f, v[j].z, acc.z * a);
                acc.w = fmaf(f, v[j].w, acc.w * a);
                m = mn;
            }
        }
        if (c == 0) {
            sm_m[rl] = m;
            sm_l[rl] = l;
        }
        sm_acc[rl][c] = acc;
        __syncthreads();
        if (rl == 0) {
            float M = sm_m[0];
#pragma unroll
            for (int k = 1; k < RL; ++k) M = fmaxf(M, sm_m[k]);
            float L = 0.f;
            float4 A = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k = 0; k < RL; ++k) {
                if (sm_m[k] == -INFINITY) continue;
                const float f = exp2f(sm_m[k] - M);
                const float4 x = sm_acc[k][c];
                L = fmaf(f, sm_l[k], L);
                A.x = fmaf(f, x.x, A.x);
                A.y = fmaf(f, x.y, A.y);
                A.z = fmaf(f, x.z, A.z);
                A.w = fmaf(f, x.w, A.w);
            }
            const float inv = 1.0f / L;
            *reinterpret_cast<uint2*>(o + 4 * c) =
                make_uint2(pack_bf16x2(A.x * inv, A.y * inv), pack_bf16x2(A.z * inv, A.w * inv));
        }
    }
    if (u == 0 && g == 0) {
        if (tid == 0) p.hdr->ticket = 0;
        if (p.k_new) {
            for (int x = tid; x < p.BH; x += kCombThreads) {
                const int v = p.len[x];
                if (v >= 0 && v < p.cap) p.len_rw[x] = v + 1;
            }
        }
    }
}

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}
// Exclusive prefix sum over the warp's lanes.
__device__ __forceinline__ int warp_excl(int v) {
    const int lane = threadIdx.x & 31;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += x;
    }
    return incl - v;
}
// The plan's per-unit scratch lives in the merge scratch's accumulator rows.
static_assert(kMaxScanUnits <= kSlotHeads * kRedStride, "one int per unit fits the merge scratch");

// While one warp plans the call, HBM would sit idle. Every row below a unit's
// length is read by the call, so the producer warp of CTA b asks L2 for the first
// rows of K and V of piece b / BH of unit b % BH (each unit's rows cut into as many
// pieces as there are CTAs per unit): 1/kPrefetchDiv of a CTA's share of the call's
// rows, in [64, kPrefetchMax]. The split that reads those rows later finds them in
// L2. rows[u] are the rows unit u attends. Paged layout: one prefetch per page the
// rows touch, lanes over the pages; a table entry outside the pool is skipped.
template <int D>
__device__ __forceinline__ void prefetch_piece(const DecParams& p, const int* rows, int lane) {
    long long t = 0;
    for (int u = lane; u < p.BH; u += 32) t += rows[u];
#pragma unroll
    for (int o = 16; o; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    const int b = (int)blockIdx.x, nb = (int)gridDim.x;
    const long long share = t / ((long long)nb * kPrefetchDiv);
    const int want = (int)min((long long)kPrefetchMax, max(64ll, share & ~63ll));
    const int u = b % p.BH, j = b / p.BH;
    const int pieces = (nb + p.BH - 1) / p.BH;
    const int len = rows[u];
    const int piece = (len + pieces - 1) / pieces;
    const int r0 = j * piece;
    const int nr = min(min(want, piece), len - r0);
    if (nr <= 0) return;
    constexpr int kRowBytes = D * 2;
    if (!p.rm.table) {
        if (lane > 1) return;
        const size_t off = ((size_t)u * p.cap + r0) * kRowBytes;
        bulk_prefetch_l2(static_cast<const uint8_t*>(lane ? p.V : p.K) + off, (uint32_t)nr * kRowBytes);
        return;
    }
    const int P = p.rm.P, pg0 = r0 / P, pg1 = (r0 + nr - 1) / P;
    for (int pi = pg0 + lane; pi <= pg1 && pi < p.rm.maxp; pi += 32) {
        const int pg = __ldg(p.rm.table + (size_t)u * p.rm.maxp + pi);
        if (pg < 0 || pg >= p.rm.npages) continue;
        const int a = max(r0, pi * P), e = min(r0 + nr, (pi + 1) * P);
        const size_t off = ((size_t)pg * P + (a - pi * P)) * kRowBytes;
        bulk_prefetch_l2(static_cast<const uint8_t*>(p.K) + off, (uint32_t)(e - a) * kRowBytes);
        bulk_prefetch_l2(static_cast<const uint8_t*>(p.V) + off, (uint32_t)(e - a) * kRowBytes);
    }
}

// SCAN: the CTA computes the unit order and split offsets itself (units <=
// kMaxScanUnits, kept in shared memory); otherwise decode_prologue_kernel has
// written them to the workspace.
template <int D, bool SCAN>
__global__ void __launch_bounds__(kDecThreads, kDecCtasPerSm)
    decode_main_kernel(const __grid_constant__ DecParams p, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmN) {
    using Geo = DecGeom<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* const sbase =
        reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* const nbase = sbase + kStages * Geo::kStageBytes;
    DecSmall& sm = *reinterpret_cast<DecSmall*>(sbase + Geo::kSmallOff);
    int* const sp = reinterpret_cast<int*>(&sm + 1);                      // [kMaxScanUnits + 1]
    uint32_t* const ulen = reinterpret_cast<uint32_t*>(sp + kMaxScanUnits + 1);  // [kMaxScanUnits]
    uint64_t* const full = sm.full;
    uint64_t* const empty = sm.empty;
    volatile int* const abort_flag = &sm.abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint64_t budget_ns = 2000000000ull;

    // Private setup first; then wait for the previous kernel in the stream (its
    // lengths, cache rows and workspace state) before reading anything.
    if (tid == 0) {
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        prefetch_tmap(&tmN);
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    griddep_launch_dependents();
    griddep_wait();

    // ---------------------------------------------------------------- split plan
    if constexpr (SCAN) {
        // Every thread loads some units' rows into sp[] (indexed by unit for now);
        // then one warp plans the call with rolled loops and shuffles. The code is
        // kept short on purpose: a call streams more than L2 holds, so this code is
        // fetched cold on every call.
#pragma unroll 4
        for (int u = tid; u < p.BH; u += kDecThreads) sp[u] = eff_len(p, u, true);
        __syncthreads();
        if (kPrefetchDiv > 0 && warp == kConsumerWarps) prefetch_piece<D>(p, sp, lane);
        if (warp == 0) {
            const int per = (p.BH + 31) / 32;
            const int ub = min(p.BH, lane * per), ue = min(p.BH, ub + per);
            int total = 0;
#pragma unroll 1
            for (int u = ub; u < ue; ++u) total += sp[u];
            total = warp_sum(total);
            const int S = split_base(total, (int)gridDim.x);
            // every unit's split count and class, computed once (the divisions are the
            // bulk of this code, fetched cold) and kept in the merge scratch, which is
            // first written at the end of a split: nsc[u] = splits << 2 | class
            int* const nsc = reinterpret_cast<int*>(&sm.cs.acc[0][0]);
            // positions: classes in order, units in index order inside a class; the
            // four class counts (each <= kMaxScanUnits < 2^16) travel packed in two ints
            int c01 = 0, c23 = 0;
#pragma unroll 1
            for (int u = ub; u < ue; ++u) {
                const int len = sp[u];
                int ns = 0, cls = 3;
                if (len > 0) {
                    const int su = unit_split(len, S, total, p.nCTA);
                    ns = unit_nsplit(len, su);
                    cls = unit_class(ns, su, S);
                }
                nsc[u] = (ns << 2) | cls;
                c01 += cls == 0 ? 1 : (cls == 1 ? 0x10000 : 0);
                c23 += cls == 2 ? 1 : (cls == 3 ? 0x10000 : 0);
            }
            const int e01 = warp_excl(c01), e23 = warp_excl(c23);
            const int t01 = __shfl_sync(0xffffffffu, e01 + c01, 31), t23 = __shfl_sync(0xffffffffu, e23 + c23, 31);
            int pos0 = e01 & 0xFFFF;
            int pos1 = (t01 & 0xFFFF) + (e01 >> 16);
            int pos2 = (t01 & 0xFFFF) + (t01 >> 16) + (e23 & 0xFFFF);
            int pos3 = (t01 & 0xFFFF) + (t01 >> 16) + (t23 & 0xFFFF) + (e23 >> 16);
#pragma unroll 1
            for (int u = ub; u < ue; ++u) {
                const int cls = nsc[u] & 3;
                const int pos = cls == 0 ? pos0++ : (cls == 1 ? pos1++ : (cls == 2 ? pos2++ : pos3++));
                ulen[pos] = ((uint32_t)sp[u] << kUnitBits) | (uint32_t)u;
            }
            __syncwarp();
            // in ticket order: every position's splits and its first split
            constexpr uint32_t kUnitMask = (1u << kUnitBits) - 1u;
            int ns = 0;
#pragma unroll 1
            for (int q = ub; q < ue; ++q) ns += nsc[ulen[q] & kUnitMask] >> 2;
            int first = warp_excl(ns);
            const int nsplits_all = __shfl_sync(0xffffffffu, first + ns, 31);
#pragma unroll 1
            for (int q = ub; q < ue; ++q) {
                const int u = (int)(ulen[q] & kUnitMask);
                const int n = nsc[u] >> 2;
                sp[q] = first;
                if (blockIdx.x == 0) {  // for the merge kernel
                    p.g_first[u] = first;
                    p.g_n[u] = n;
                }
                first += n;
            }
            if (lane == 0) {
                sp[p.BH] = nsplits_all;
                sm.nsplits = nsplits_all;
                sm.S = S;
                sm.total = total;
            }
        }
    } else {
        if (tid == 0) {
            sm.nsplits = p.hdr->dec_nsplits;
            sm.S = p.hdr->dec_split;
            sm.total = p.hdr->dec_total;
        }
    }
    __syncthreads();
    const int nsplits = sm.nsplits, S = sm.S, total = sm.total;

    if (warp == kConsumerWarps) {
        // ============================================================ producer
        int issued = 0;
        bool ok = true;
        // K and V are read once per call: their lines go first when L2 needs room, so the
        // kernel's code, the lengths, q and the split records stay resident
        const uint64_t pol = l2_policy_evict_first();
        // split blockIdx.x first; later splits come from the ticket, from gridDim.x on
        Split cur = resolve_split<SCAN>(p, (int)blockIdx.x, nsplits, S, total, sp, ulen);
        while (cur.t >= 0) {
            int tn = 0;
            const int tok0 = cur.tok0;
            const int ntok = cur.ntok;
            const int ntiles = (ntok + kTile - 1) / kTile;
            const long long row_base = (long long)cur.u * p.cap;
            // paged layout: the ids of the pages from pg_base on, one per lane (the
            // window moves when a tile runs past it); every lane calls pool_row
            int pg_base = 0, pg_id = -1;
            auto load_pages = [&](int first_page) {
                pg_base = first_page;
                const int pi = first_page + lane;
                pg_id = pi < p.rm.maxp ? __ldg(p.rm.table + (size_t)cur.u * p.rm.maxp + pi) : -1;
            };
            if (p.rm.table) load_pages(tok0 / p.rm.P);
            auto pool_row = [&](int t) -> long long {  // -1: a block-table entry outside the pool
                if (!p.rm.table) return row_base + t;
                const int pi = t / p.rm.P;
                if (pi - pg_base >= 32) load_pages(pi);
                const int pg = __shfl_sync(0xffffffffu, pg_id, pi - pg_base);
                return (pg < 0 || pg >= p.rm.npages) ? -1 : (long long)pg * p.rm.P + t % p.rm.P;
            };
            int arow = -1;  // fused append: the unit's new row, held by its last split
            long long arow_p = -1;
            if (p.k_new && cur.k == cur.n - 1) {
                const int old = p.len[cur.u];
                if (old >= 0 && old < p.cap) arow = old;
                if (arow >= 0) {
                    arow_p = pool_row(arow);
                    if (arow_p < 0 && lane == 0) record_status(&p.hdr->status, CSMKV_ERR_ARG);
                }
            }
            for (int i = 0; i < ntiles; ++i) {
                const int s = issued % kStages;
                // the next split is claimed with the last tile of this one: the ring
                // still holds up to kStages tiles of work while the ticket and its
                // plan resolve, and no split is held longer than that before it starts
#if CSMKV_DEC_CLAIM_EARLY
                if (i == 0 && lane == 0) tn = (int)gridDim.x + atomicAdd(&p.hdr->ticket, 1);
#else
                if (i == ntiles - 1 && lane == 0) tn = (int)gridDim.x + atomicAdd(&p.hdr->ticket, 1);
#endif
                if (issued >= kStages) {
                    int w = 1;
                    if (lane == 0)
                        w = mbar_wait(&empty[s], ((issued / kStages) - 1) & 1, globaltimer() + budget_ns) && !*abort_flag;
                    if (!__shfl_sync(0xffffffffu, w, 0)) {
                        ok = false;
                        break;
                    }
                }
                const int tok = tok0 + i * kTile;
                const int nv = min(kTile, ntok - i * kTile);
                const long long prow = pool_row(tok);
                if (arow >= tok && arow < tok + nv && arow_p >= 0) {
                    // the new token's K, V row and degree, written before the TMA reads the
                    // tile (one 16-byte piece per lane; the fence orders each lane's writes
                    // before the async-proxy reads that follow the warp sync)
                    constexpr int PPR = D / 8;
                    if (lane < 2 * PPR) {
                        const bool isv = lane >= PPR;
                        const int kk = isv ? lane - PPR : lane;
                        const uint4* src = static_cast<const uint4*>(isv ? p.v_new : p.k_new) + (size_t)cur.u * PPR + kk;
                        uint4* dst = static_cast<uint4*>(isv ? p.V : p.K) + (size_t)arow_p * PPR + kk;
                        *dst = *src;
                        if (lane == 0) p.N[arow_p] = 1;
                        fence_proxy_async_global();
                    }
                    __syncwarp();
                }
                if (lane == 0) {
                    StageMeta& mt = sm.meta[s];
                    mt.t = cur.t;
                    mt.unit = cur.u;
                    mt.k = cur.k;
                    mt.n = cur.n;
                    mt.tok = tok;
                    mt.nv = nv;
                    mt.flags = (i == 0 ? kFirst : 0u) | (i == ntiles - 1 ? kLast : 0u);
                    // a tile whose page entry is outside the pool reads the fill value (zeros)
                    if (prow < 0) record_status(&p.hdr->status, CSMKV_ERR_ARG);
                    const int row = prow < 0 ? p.pool_rows : (int)prow;
                    uint8_t* st = sbase + s * Geo::kStageBytes;
                    // the first tile of a split also brings the group's query rows
                    const uint32_t qbytes = i == 0 ? (uint32_t)(p.G * D * 2) : 0u;
                    mbar_expect_tx(&full[s], Geo::kTxBytes + qbytes);
                    if (i == 0) {
                        const int b = cur.u / p.Hkv, kv = cur.u - b * p.Hkv;
                        bulk_load(sbase + Geo::kQOff + s * Geo::kQBytes,
                                  static_cast<const __nv_bfloat16*>(p.q) + ((size_t)b * p.Hq + (size_t)kv * p.G) * D,
                                  qbytes, &full[s]);
                    }
#pragma unroll
                    for (int bx = 0; bx < Geo::kBoxes; ++bx) {
                        tma_load_2d_hint(st + Geo::kKOff + bx * Geo::kBoxBytes, &tmK, &full[s], bx * 64, row, pol);
                        tma_load_2d_hint(st + Geo::kVOff + bx * Geo::kBoxBytes, &tmV, &full[s], bx * 64, row, pol);
                    }
                    tma_load_2d(nbase + s * Geo::kNStride, &tmN, &full[s], 0, row >> 2);
                }
                ++issued;
            }
            if (!ok) break;
            tn = __shfl_sync(0xffffffffu, tn, 0);
            cur = resolve_split<SCAN>(p, tn, nsplits, S, total, sp, ulen);
        }
        if (ok) {
            // stop marker for the consumers, in the stage after the last one issued
            if (lane == 0) {
                const int s = issued % kStages;
                if (issued >= kStages)
                    ok = mbar_wait(&empty[s], ((issued / kStages) - 1) & 1, globaltimer() + budget_ns);
                sm.meta[s].t = -1;
                if (ok) mbar_arrive(&full[s]);
            }
            ok = __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
        }
        if (!ok && lane == 0) {
            record_status(&p.hdr->status, CSMKV_ERR_TIMEOUT);
            *abort_flag = 1;
            // the consumers may stop early: every issued stage must land before the CTA exits
            for (int i = max(0, issued - kStages); i < issued; ++i)
                (void)mbar_wait(&full[i % kStages], (i / kStages) & 1, globaltimer() + budget_ns);
        }
        __syncwarp();
    } else {
        // ============================================================ consumers
        const int g = lane >> 2, t4 = lane & 3;
        const int tok_lo = warp * 16;
        uint32_t qf[D / 16][2];
        float oacc[D / 16][4];
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
        int consumed = 0;
        bool ok = true;
        for (;;) {
            const int s = consumed % kStages;
            const bool got = mbar_wait(&full[s], (consumed / kStages) & 1, globaltimer() + budget_ns);
            if (consumer_any(!got || *abort_flag)) {
                ok = false;
                break;
            }
            const StageMeta mt = sm.meta[s];
            if (mt.t < 0) break;
            if (mt.flags & kFirst) {  // the split's query rows came with this tile
                const __nv_bfloat16* qrow =
                    reinterpret_cast<const __nv_bfloat16*>(sbase + Geo::kQOff + s * Geo::kQBytes) + g * D;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    if (g < p.G) {
                        qf[ks][0] = *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * t4);
                        qf[ks][1] = *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 8 + 2 * t4);
                    } else {
                        qf[ks][0] = 0u;
                        qf[ks][1] = 0u;
                    }
                }
#pragma unroll
                for (int mb = 0; mb < D / 16; ++mb) oacc[mb][0] = oacc[mb][1] = oacc[mb][2] = oacc[mb][3] = 0.f;
                m0 = m1 = -INFINITY;
                l0 = l1 = 0.f;
            }
            const int nv = mt.nv;
            uint8_t* st = sbase + s * Geo::kStageBytes;
            const int noff = (int)(((long long)mt.unit * p.cap + mt.tok) & 3);
            const int* sN = reinterpret_cast<const int*>(nbase + s * Geo::kNStride) + noff;
            if (tok_lo < nv) {
                // ---- S^T = K q^T (16 tokens x 8 heads)
                float sacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const int row = tok_lo + (lane & 7) + ((lane >> 3) & 1) * 8;
                    const int col = 16 * ks + (lane >> 4) * 8;
                    uint32_t a0, a1, a2, a3;
                    ldmatrix_x4(smem_u32(st + Geo::kKOff + (col >> 6) * Geo::kBoxBytes) + sw128_off(row, (col & 63) >> 3),
                                a0, a1, a2, a3);
                    mma_bf16_16816(sacc, a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
                }
                const int tA = tok_lo + g, tB = tA + 8;
                const bool vA = tA < nv, vB = tB < nv;
                const float x0 = vA ? sacc[0] * p.scale_log2 : -INFINITY;
                const float x1 = vA ? sacc[1] * p.scale_log2 : -INFINITY;
                const float x2 = vB ? sacc[2] * p.scale_log2 : -INFINITY;
                const float x3 = vB ? sacc[3] * p.scale_log2 : -INFINITY;
                float mh0 = fmaxf(x0, x2), mh1 = fmaxf(x1, x3);
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) {
                    mh0 = fmaxf(mh0, __shfl_xor_sync(0xffffffffu, mh0, o));
                    mh1 = fmaxf(mh1, __shfl_xor_sync(0xffffffffu, mh1, o));
                }
                const float mn0 = fmaxf(m0, mh0), mn1 = fmaxf(m1, mh1);
                const float al0 = (mn0 == -INFINITY) ? 1.f : exp2f(m0 - mn0);
                const float al1 = (mn1 == -INFINITY) ? 1.f : exp2f(m1 - mn1);
                const float nA = vA ? (float)sN[tA] : 0.f, nB = vB ? (float)sN[tB] : 0.f;
                const float p0 = vA ? nA * exp2f(x0 - mn0) : 0.f;
                const float p1 = vA ? nA * exp2f(x1 - mn1) : 0.f;
                const float p2 = vB ? nB * exp2f(x2 - mn0) : 0.f;
                const float p3 = vB ? nB * exp2f(x3 - mn1) : 0.f;
                const uint32_t rowA = pack_bf16x2(p0, p1), rowB = pack_bf16x2(p2, p3);
                // the denominator sums the same bf16-rounded weights the MMA sees
                l0 = l0 * al0 + bf16lo(rowA) + bf16lo(rowB);
                l1 = l1 * al1 + bf16hi(rowA) + bf16hi(rowB);
                if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
                    for (int mb = 0; mb < D / 16; ++mb) {
                        oacc[mb][0] *= al0;
                        oacc[mb][1] *= al1;
                        oacc[mb][2] *= al0;
                        oacc[mb][3] *= al1;
                    }
                }
                m0 = mn0;
                m1 = mn1;
                const uint32_t b0 = movmatrix_trans(rowA), b1 = movmatrix_trans(rowB);
                if (tok_lo + 16 > nv) {
                    // rows past the end may hold anything (NaN included): zero them so 0 * V stays 0
                    for (int i = lane; i < 16 * 8 * Geo::kBoxes; i += 32) {
                        const int r = tok_lo + i / (8 * Geo::kBoxes);
                        const int rem = i % (8 * Geo::kBoxes);
                        if (r >= nv)
                            *reinterpret_cast<uint4*>(st + Geo::kVOff + (rem >> 3) * Geo::kBoxBytes + sw128_off(r, rem & 7)) =
                                make_uint4(0u, 0u, 0u, 0u);
                    }
                    __syncwarp();
                }
                // ---- O^T += V^T P^T (16 dims x 8 heads per m-block)
#pragma unroll
                for (int mb = 0; mb < D / 16; ++mb) {
                    const int row = tok_lo + (lane & 7) + (lane >> 4) * 8;
                    const int col = 16 * mb + ((lane >> 3) & 1) * 8;
                    uint32_t a0, a1, a2, a3;
                    ldmatrix_x4_trans(smem_u32(st + Geo::kVOff + (col >> 6) * Geo::kBoxBytes) + sw128_off(row, (col & 63) >> 3),
                                      a0, a1, a2, a3);
                    mma_bf16_16816(oacc[mb], a0, a1, a2, a3, b0, b1);
                }
                if (tok_lo + 16 > nv) fence_proxy_async_smem();  // generic zeroing before the next TMA into this stage
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            ++consumed;
            if (!(mt.flags & kLast)) continue;

            // ---- end of a split: the 4 warps' states merged in shared memory, in warp
            //      order (deterministic), then written as the split's record
            float lt0 = l0, lt1 = l1;
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                lt0 += __shfl_xor_sync(0xffffffffu, lt0, o);
                lt1 += __shfl_xor_sync(0xffffffffu, lt1, o);
            }
            CombineScratch& cs = sm.cs;
            const int h0 = 2 * t4, h1 = 2 * t4 + 1;
            if (g == 0) {
                cs.m[warp][h0] = m0;
                cs.m[warp][h1] = m1;
                cs.l[warp][h0] = lt0;
                cs.l[warp][h1] = lt1;
            }
            consumer_barrier();
            {
                const float M0 = fmaxf(fmaxf(cs.m[0][h0], cs.m[1][h0]), fmaxf(cs.m[2][h0], cs.m[3][h0]));
                const float M1 = fmaxf(fmaxf(cs.m[0][h1], cs.m[1][h1]), fmaxf(cs.m[2][h1], cs.m[3][h1]));
                const float f0 = m0 == -INFINITY ? 0.f : exp2f(m0 - M0);
                const float f1 = m1 == -INFINITY ? 0.f : exp2f(m1 - M1);
                for (int w = 0; w < kConsumerWarps; ++w) {
                    if (warp == w) {
#pragma unroll
                        for (int mb = 0; mb < D / 16; ++mb) {
                            float* r0 = &cs.acc[h0][16 * mb + g];
                            float* r1 = &cs.acc[h1][16 * mb + g];
                            if (w == 0) {
                                r0[0] = f0 * oacc[mb][0];
                                r1[0] = f1 * oacc[mb][1];
                                r0[8] = f0 * oacc[mb][2];
                                r1[8] = f1 * oacc[mb][3];
                            } else {
                                r0[0] = fmaf(f0, oacc[mb][0], r0[0]);
                                r1[0] = fmaf(f1, oacc[mb][1], r1[0]);
                                r0[8] = fmaf(f0, oacc[mb][2], r0[8]);
                                r1[8] = fmaf(f1, oacc[mb][3], r1[8]);
                            }
                        }
                    }
                    consumer_barrier();
                }
            }
            const size_t rec = (size_t)mt.t * p.G;
            for (int i = tid; i < p.G * (D / 4); i += kConsumerWarps * 32) {
                const int h = i / (D / 4), d = (i - h * (D / 4)) * 4;
                __stcg(reinterpret_cast<float4*>(p.pacc + (rec + h) * D + d), *reinterpret_cast<const float4*>(&cs.acc[h][d]));
            }
            if (tid < p.G) {
                const float M = fmaxf(fmaxf(cs.m[0][tid], cs.m[1][tid]), fmaxf(cs.m[2][tid], cs.m[3][tid]));
                float L = 0.f;
                for (int w = 0; w < kConsumerWarps; ++w)
                    if (cs.m[w][tid] != -INFINITY) L = fmaf(exp2f(cs.m[w][tid] - M), cs.l[w][tid], L);
                p.pm[rec + tid] = M;
                p.pl[rec + tid] = L;
            }
            // the merge scratch is next written at the end of a later split, after at
            // least one more consumer barrier
        }
        if (!ok && tid == 0) {
            record_status(&p.hdr->status, CSMKV_ERR_TIMEOUT);
            *abort_flag = 1;
        }
    }
}

// ----------------------------------------------------------------------------
// fp32 path (exactness first): one CTA per (sequence, query head), four warps
// over the tokens, lanes over the head dimension, fp32 online softmax.
__global__ void __launch_bounds__(128) decode_f32_kernel(const DecParams p, const float* K, const float* V,
                                                         const int32_t* N) {
    const int bh = blockIdx.x;  // b * Hq + h
    const int b = bh / p.Hq, h = bh - b * p.Hq, kv = h / p.G;
    const int unit = b * p.Hkv + kv;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int D = p.D;
    int s = p.len[unit];
    if (s < 0 || s > p.cap) {
        if (threadIdx.x == 0) record_status(&p.hdr->status, CSMKV_ERR_ARG);
        s = 0;
    }
    const float* q = static_cast<const float*>(p.q) + (size_t)bh * D;
    float qv[4], acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 4; ++i) qv[i] = (lane + 32 * i < D) ? q[lane + 32 * i] : 0.f;
    float m = -INFINITY, l = 0.f;
    const size_t base = (size_t)unit * p.cap;
    for (int t = warp; t < s; t += 4) {
        const float* k = K + (base + t) * D;
        float dot = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (lane + 32 * i < D) dot = fmaf(qv[i], k[lane + 32 * i], dot);
        for (int o = 16; o; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        const float x = dot * p.scale;
        const float mn = fmaxf(m, x);
        const float al = expf(m - mn);  // m = -inf on the first token -> 0
        const float w = (float)N[base + t] * expf(x - mn);
        l = l * al + w;
        const float* v = V + (base + t) * D;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (lane + 32 * i < D) acc[i] = fmaf(w, v[lane + 32 * i], acc[i] * al);
        m = mn;
    }
    __shared__ float sm[4], sl[4], sacc[4][128];
    if (lane == 0) { sm[warp] = m; sl[warp] = l; }
#pragma unroll
    for (int i = 0; i < 4; ++i)
        if (lane + 32 * i < D) sacc[warp][lane + 32 * i] = acc[i];
    __syncthreads();
    if (warp == 0) {
        float M = fmaxf(fmaxf(sm[0], sm[1]), fmaxf(sm[2], sm[3]));
        float L = 0.f, f[4];
        for (int w = 0; w < 4; ++w) {
            f[w] = (sm[w] == -INFINITY) ? 0.f : expf(sm[w] - M);
            L += f[w] * sl[w];
        }
        float* out = static_cast<float*>(p.out) + (size_t)bh * D;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int d = lane + 32 * i;
            if (d < D) {
                float a = 0.f;
                for (int w = 0; w < 4; ++w) a = fmaf(f[w], sacc[w][d], a);
                out[d] = (s > 0) ? a / L : 0.f;
            }
        }
    }
}

static size_t dec_layout(const csmkv_cache* cache, int32_t h_q, int nCTA, size_t* o_first, size_t* o_n,
                         size_t* o_len, size_t* o_unit, size_t* o_pm, size_t* o_pl, size_t* o_pacc) {
    const size_t BH = (size_t)cache->batch * cache->h_kv;
    const size_t G = (size_t)h_q / cache->h_kv;
    const size_t splits = (size_t)dec_max_splits(nCTA, (int)BH);  // one record per split
    size_t off = kHeaderBytes;
    *o_first = off;
    off = align_up(off + BH * 4, 256);
    *o_n = off;
    off = align_up(off + BH * 4, 256);
    *o_len = off;
    off = align_up(off + BH * 4, 256);
    *o_unit = off;
    off = align_up(off + splits * 4, 256);
    *o_pm = off;
    off = align_up(off + splits * G * 4, 256);
    *o_pl = off;
    off = align_up(off + splits * G * 4, 256);
    *o_pacc = off;
    off = align_up(off + splits * G * (size_t)cache->head_dim * 4, 256);
    return off;
}

template <int D, bool SCAN>
static int launch_decode_bf16(const DecParams& P, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& tn, cudaStream_t st) {
    constexpr int smem = DecGeom<D>::kSmallOff + (int)sizeof(DecSmall) + (SCAN ? (2 * kMaxScanUnits + 1) * 4 : 0) +
                         1024;
    static_assert(kDecCtasPerSm * (smem + 1024) <= 228 * 1024, "two CTAs per SM must fit in shared memory");
    auto kern = decode_main_kernel<D, SCAN>;
    if (set_kernel_smem((const void*)kern, smem) != CSMKV_OK) return CSMKV_ERR_CUDA;
    if (launch_overlapped(kern, dim3(P.nCTA), dim3(kDecThreads), (size_t)smem, st, P, tk, tv, tn) != cudaSuccess)
        return CSMKV_ERR_CUDA;
    if (launch_overlapped(decode_combine_kernel<D>, dim3(P.BH, P.G), dim3(kCombThreads), 0, st, P) != cudaSuccess)
        return CSMKV_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? CSMKV_OK : CSMKV_ERR_CUDA;
}

int decode_attn_check_args(const void* q, const void* K, const void* V, const int32_t* N, const int32_t* len,
                           const void* k_new, const void* v_new, const csmkv_cache* cache, int32_t h_q, float scale,
                           const void* out) {
    int rc = check_cache(cache);
    if (rc != CSMKV_OK) return rc;
    if (!q || !K || !V || !N || !len || !out) return CSMKV_ERR_ARG;
    if ((k_new == nullptr) != (v_new == nullptr)) return CSMKV_ERR_ARG;
    if (k_new && (!aligned16(k_new) || !aligned16(v_new))) return CSMKV_ERR_ALIGN;
    if (h_q < 1 || (h_q % cache->h_kv) != 0) return CSMKV_ERR_ARG;
    if (!(scale > 0.f) || !std::isfinite(scale)) return CSMKV_ERR_ARG;
    if (!aligned16(K) || !aligned16(V) || !aligned16(N) || !aligned16(q) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(len) & 3u))
        return CSMKV_ERR_ALIGN;
    const int G = h_q / cache->h_kv;
    const int D = cache->head_dim;
    if (cache->dtype == CSMKV_BF16 && (G > 8 || (D != 64 && D != 128))) return CSMKV_ERR_UNSUPPORTED;
    return CSMKV_OK;
}

}  // namespace csmkv

using namespace csmkv;

extern "C" size_t decode_attn_workspace_bytes(const csmkv_cache* cache, int32_t h_q) {
    if (check_cache(cache) != CSMKV_OK || h_q < 1 || (h_q % cache->h_kv) != 0) return 0;
    const int nCTA = sm_count() * kDecCtasPerSm;
    if (nCTA <= 0) return 0;
    size_t a, b, c, d, e, f, g;
    return dec_layout(cache, h_q, nCTA, &a, &b, &c, &d, &e, &f, &g);
}

// Attention over the cache, optionally with the step's new token appended first
// (k_new != NULL: bf16 fuses the append into the attention kernel).
static int decode_attn_impl(const void* q, const void* K, const void* V, const int32_t* N, const int32_t* len,
                            const void* k_new, const void* v_new, const csmkv_cache* cache, const csmkv_pages* pages,
                            int32_t h_q, float scale, void* out, void* workspace, size_t ws_bytes, void* stream) {
    int rc = decode_attn_check_args(q, K, V, N, len, k_new, v_new, cache, h_q, scale, out);
    if (rc != CSMKV_OK) return rc;
    if (pages) {
        rc = check_pages(cache, pages);
        if (rc != CSMKV_OK) return rc;
        if (cache->dtype != CSMKV_BF16) return CSMKV_ERR_UNSUPPORTED;
    }
    const int G = h_q / cache->h_kv;
    const int D = cache->head_dim;
    const bool bf16 = cache->dtype == CSMKV_BF16;
    const int nCTA = sm_count() * kDecCtasPerSm;
    if (nCTA <= 0) return CSMKV_ERR_CUDA;
    size_t o_first, o_n, o_len, o_unit, o_pm, o_pl, o_pacc;
    const size_t need = dec_layout(cache, h_q, nCTA, &o_first, &o_n, &o_len, &o_unit, &o_pm, &o_pl, &o_pacc);
    if (!workspace || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return CSMKV_ERR_WORKSPACE;

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    DecParams P{};
    P.q = q;
    P.len = len;
    P.k_new = k_new;
    P.v_new = v_new;
    P.K = const_cast<void*>(K);
    P.V = const_cast<void*>(V);
    P.N = const_cast<int32_t*>(N);
    P.len_rw = const_cast<int32_t*>(len);
    P.out = out;
    P.hdr = reinterpret_cast<WsHeader*>(ws);
    P.g_first = reinterpret_cast<int32_t*>(ws + o_first);
    P.g_n = reinterpret_cast<int32_t*>(ws + o_n);
    P.g_len = reinterpret_cast<int32_t*>(ws + o_len);
    P.g_unit = reinterpret_cast<int32_t*>(ws + o_unit);
    P.pm = reinterpret_cast<float*>(ws + o_pm);
    P.pl = reinterpret_cast<float*>(ws + o_pl);
    P.pacc = reinterpret_cast<float*>(ws + o_pacc);
    P.BH = cache->batch * cache->h_kv;
    P.Hkv = cache->h_kv;
    P.Hq = h_q;
    P.G = G;
    P.cap = cache->cap;
    P.D = D;
    P.nCTA = nCTA;
    P.max_splits = dec_max_splits(nCTA, P.BH);
    P.rm = row_map(cache, pages);
    P.scale = scale;
    P.scale_log2 = scale * 1.4426950408889634f;
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    if (!bf16 && k_new) {  // fp32: the append kernel, then attention (status in this workspace)
        rc = csm_append(const_cast<void*>(K), const_cast<void*>(V), const_cast<int32_t*>(N), const_cast<int32_t*>(len),
                        cache, k_new, v_new, nullptr, workspace, ws_bytes, stream);
        if (rc != CSMKV_OK) return rc;
        P.k_new = P.v_new = nullptr;
    }
    if (!bf16) {
        decode_f32_kernel<<<cache->batch * h_q, 128, 0, st>>>(P, static_cast<const float*>(K),
                                                              static_cast<const float*>(V), N);
        return cudaGetLastError() == cudaSuccess ? CSMKV_OK : CSMKV_ERR_CUDA;
    }

    const uint64_t rows =
        pages ? (uint64_t)pages->num_pages * pages->page_rows : (uint64_t)cache->batch * cache->h_kv * cache->cap;
    P.pool_rows = (int32_t)rows;
    CUtensorMap tk{}, tv{}, tn{};
    {
        const uint64_t dims[2] = {(uint64_t)D, rows};
        const uint64_t strides[1] = {(uint64_t)D * 2};
        const uint32_t box[2] = {64, (uint32_t)kTile};
        if (!encode_tiled(&tk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(K), dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_tiled(&tv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(V), dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B))
            return CSMKV_ERR_CUDA;
        const uint64_t ndims[2] = {4, rows / 4};
        const uint64_t nstr[1] = {16};
        const uint32_t nbox[2] = {4, (uint32_t)(kTile / 4 + 1)};
        if (!encode_tiled(&tn, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, const_cast<int32_t*>(N), ndims, nstr, nbox,
                          CU_TENSOR_MAP_SWIZZLE_NONE))
            return CSMKV_ERR_CUDA;
    }
    // The in-CTA plan packs (len << kUnitBits) | unit into 32 bits.
    const bool scan = P.BH <= kMaxScanUnits && cache->cap < (1 << (32 - kUnitBits));
    if (scan)
        return D == 128 ? launch_decode_bf16<128, true>(P, tk, tv, tn, st) : launch_decode_bf16<64, true>(P, tk, tv, tn, st);
    decode_prologue_kernel<<<1, 1024, 0, st>>>(P);
    if (cudaGetLastError() != cudaSuccess) return CSMKV_ERR_CUDA;
    return D == 128 ? launch_decode_bf16<128, false>(P, tk, tv, tn, st) : launch_decode_bf16<64, false>(P, tk, tv, tn, st);
}

extern "C" int decode_attn_logn(const void* q, const void* K, const void* V, const int32_t* N, const int32_t* len,
                                const csmkv_cache* cache, int32_t h_q, float scale, void* out, void* workspace,
                                size_t ws_bytes, void* stream) {
    return decode_attn_impl(q, K, V, N, len, nullptr, nullptr, cache, nullptr, h_q, scale, out, workspace, ws_bytes,
                            stream);
}

extern "C" int decode_attn_logn_paged(const void* q, const void* K, const void* V, const int32_t* N,
                                      const int32_t* len, const csmkv_cache* cache, const csmkv_pages* pages,
                                      int32_t h_q, float scale, void* out, void* workspace, size_t ws_bytes,
                                      void* stream) {
    if (!pages) return CSMKV_ERR_ARG;
    return decode_attn_impl(q, K, V, N, len, nullptr, nullptr, cache, pages, h_q, scale, out, workspace, ws_bytes,
                            stream);
}

extern "C" int decode_step_logn(const void* q, const void* k_new, const void* v_new, void* K, void* V, int32_t* N,
                                int32_t* len, const csmkv_cache* cache, int32_t h_q, float scale, void* out,
                                void* workspace, size_t ws_bytes, void* stream) {
    if (!k_new || !v_new) return CSMKV_ERR_ARG;
    return decode_attn_impl(q, K, V, N, len, k_new, v_new, cache, nullptr, h_q, scale, out, workspace, ws_bytes,
                            stream);
}

extern "C" int decode_step_logn_paged(const void* q, const void* k_new, const void* v_new, void* K, void* V,
                                      int32_t* N, int32_t* len, const csmkv_cache* cache, const csmkv_pages* pages,
                                      int32_t h_q, float scale, void* out, void* workspace, size_t ws_bytes,
                                      void* stream) {
    if (!k_new || !v_new || !pages) return CSMKV_ERR_ARG;
    return decode_attn_impl(q, K, V, N, len, k_new, v_new, cache, pages, h_q, scale, out, workspace, ws_bytes,
                            stream);
}
