// decode_attn.cu -- degree-aware decode attention over a (compressed) KV cache.
// [Chelsea §三 核心公式: O = softmax(q K^T / sqrt(d) + log N) V; CentroidKV 聚合]
//
// The log-degree bias is applied as a weight: e^(x + log n) = n e^x, so the
// online softmax keeps (m, l, acc) with p_t = n_t * 2^(x_t - m), x_t the
// base-2 scaled logit. No log is evaluated and integer degrees stay exact.
//
// Work split (bf16): all units' tokens are laid end to end and cut into one
// equal range per CTA, so ragged lengths (outlier heads, ragged batches) stay
// balanced over the whole GPU. A CTA walks its range unit by unit in 64-token
// tiles: one producer warp streams K, V (128-byte swizzled, 2 boxes of 64
// columns) and the degree tile into a 3-stage TMA/mbarrier ring; four consumer
// warps each take 16 tokens of a tile and run S^T = K q^T and O^T += V^T P^T on
// mma.sync (bf16 in, fp32 accumulate), the G <= 8 query heads of the group in
// the N = 8 dimension, so each K/V byte is read once for the whole group. The
// CTA merges its warps' states in shared memory and writes one partial
// (m, l, acc) per unit it touched; the last CTA to
// finish its part of a unit (a per-unit counter) merges the unit's partials into
// the output. Unit offsets come from a block-wide scan of the lengths inside
// every CTA (or, for batches of more than 2048 units, from a one-CTA prologue).
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
constexpr int kSlotHeads = 8;  // partial records are padded to 8 heads
constexpr int kMaxScanUnits = 2048;  // units whose offsets a CTA scans itself
constexpr int kMinTokensPerCta = 512;  // small calls use fewer CTAs (the rest exit at once)

// Tokens per CTA for `total` tokens on a grid of n CTAs: an equal share, but at
// least kMinTokensPerCta, so a small call does not spread a few tiles over
// hundreds of CTAs and then merge hundreds of partial records.
__host__ __device__ __forceinline__ int tokens_per_cta(int total, int n) {
    const int share = (total + n - 1) / n;
    return share > kMinTokensPerCta ? share : kMinTokensPerCta;
}

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
    int32_t* prefix;      // [BH + 1] token offset of every unit
    int32_t* cta_unit;    // [nCTA] first unit of every CTA's range (BH = none)
    float* pm;            // [slots][8] running max (base-2 domain)
    float* pl;            // [slots][8] running sum
    float* pacc;          // [slots][8][D] unnormalised output
    int32_t* counter;     // [BH] parts of a unit finished in this call; the last one resets it
    int32_t BH, Hkv, Hq, G, cap, D, nCTA;
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

// ----------------------------------------------------------------------------
// Prologue (one CTA): prefix sums of the lengths, tokens per CTA, first unit of
// every CTA's range.
__global__ void __launch_bounds__(1024) decode_prologue_kernel(const DecParams p) {
    griddep_launch_dependents();  // the main kernel may set itself up meanwhile
    __shared__ int wsum[32];
    __shared__ int carry_s;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) carry_s = 0;
    __syncthreads();
    for (int base = 0; base < p.BH; base += 1024) {
        const int u = base + tid;
        const int v = u < p.BH ? eff_len(p, u, true) : 0;
        int incl = v;
        for (int o = 1; o < 32; o <<= 1) {
            const int x = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += x;
        }
        if (lane == 31) wsum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int w = wsum[lane];
            for (int o = 1; o < 32; o <<= 1) {
                const int x = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += x;
            }
            wsum[lane] = w;  // inclusive over warps
        }
        __syncthreads();
        const int carry = carry_s;
        const int excl = carry + incl - v + (warp ? wsum[warp - 1] : 0);
        if (u < p.BH) p.prefix[u] = excl;
        __syncthreads();
        if (tid == 1023) carry_s = excl + v;
        __syncthreads();
    }
    const int total = carry_s;
    if (tid == 0) p.prefix[p.BH] = total;
    const int W = tokens_per_cta(total, p.nCTA);
    if (tid == 0) {
        p.hdr->total_tokens = total;
        p.hdr->tokens_per_cta = W;
    }
    __syncthreads();
    for (int c = tid; c < p.nCTA; c += 1024) {
        const long long start = (long long)c * W;
        int lo = 0, hi = p.BH;  // first unit with prefix[u+1] > start
        if (start >= total) {
            lo = p.BH;
        } else {
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (p.prefix[mid + 1] > start) hi = mid; else lo = mid + 1;
            }
        }
        p.cta_unit[c] = lo;
    }
}

// ----------------------------------------------------------------------------
template <int D>
struct DecGeom {
    static constexpr int kBoxes = D / 64;
    static constexpr int kBoxBytes = kTile * 128;              // 64 rows x 128 B
    static constexpr int kKOff = 0;
    static constexpr int kVOff = kBoxes * kBoxBytes;
    static constexpr int kNOff = 2 * kBoxes * kBoxBytes;
    static constexpr int kNBytes = (kTile + 4) * 4;            // 68 degrees (row rounded down to 4)
    static constexpr int kStageBytes = kNOff + 1024;           // keeps stages 1024-aligned
    static constexpr uint32_t kTxBytes = 2 * kBoxes * kBoxBytes + kNBytes;
};

// Walks a CTA's token range as (unit, first token, token count) segments.
struct RangeWalker {
    const int32_t* prefix;
    int BH, u, tok, end;
    __device__ bool next(int& unit, int& t0, int& n) {
        while (u < BH && prefix[u + 1] <= tok) ++u;
        if (tok >= end || u >= BH) return false;
        const int seg_end = min(end, prefix[u + 1]);
        unit = u;
        t0 = tok - prefix[u];
        n = seg_end - tok;
        tok = seg_end;
        return true;
    }
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

// Scratch of the main kernel after the stage ring.
struct DecSmall {
    CombineScratch cs;
    uint64_t full[kStages];
    uint64_t empty[kStages];
    int abort_flag;
    int last;      // this CTA is the last contributor of the unit being closed
    int bump;      // fused append: this CTA finished last and bumps the lengths
    int u0;        // first unit of the CTA's range
    int total;
    int warp_tot[kDecThreads / 32];
};

__device__ __forceinline__ int atom_add_acq_rel_gpu(int32_t* addr, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void consumer_barrier() {
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
}

// Merges the partials of `unit` -- one record per contributing CTA c0..c1, a
// contiguous run -- into the output; run by the 4 consumer warps of the last
// contributing CTA, so it sits on the kernel's tail: records are spread over
// all 128 threads with several loads in flight per thread, and the cross-warp
// sums go through shared memory in warp order (deterministic).
template <int D>
__device__ void combine_unit(const DecParams& p, int unit, int c0, int c1, int warp, int lane, CombineScratch& cs) {
    constexpr int PER = D / 32;  // dims per lane
    const int tid = warp * 32 + lane;
    const int G = p.G;
    const int nrec = c1 - c0 + 1;
    const size_t rec0 = (size_t)c0 + unit;

    // pass 1: per-head maximum over the records
    float mx[kSlotHeads];
#pragma unroll
    for (int g = 0; g < kSlotHeads; ++g) mx[g] = -INFINITY;
    for (int r = tid; r < nrec; r += kConsumerWarps * 32) {
        const float4 a = __ldcg(reinterpret_cast<const float4*>(p.pm + (rec0 + r) * kSlotHeads));
        const float4 b = __ldcg(reinterpret_cast<const float4*>(p.pm + (rec0 + r) * kSlotHeads + 4));
        const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
        for (int g = 0; g < kSlotHeads; ++g)
            if (g < G) mx[g] = fmaxf(mx[g], v[g]);
    }
#pragma unroll
    for (int g = 0; g < kSlotHeads; ++g) {
#pragma unroll
        for (int o = 16; o; o >>= 1) mx[g] = fmaxf(mx[g], __shfl_xor_sync(0xffffffffu, mx[g], o));
    }
    if (lane == 0) {
#pragma unroll
        for (int g = 0; g < kSlotHeads; ++g) cs.m[warp][g] = mx[g];
    }
    consumer_barrier();
    float M[kSlotHeads];
#pragma unroll
    for (int g = 0; g < kSlotHeads; ++g) M[g] = fmaxf(fmaxf(cs.m[0][g], cs.m[1][g]), fmaxf(cs.m[2][g], cs.m[3][g]));

    // pass 2: warp w folds records w, w+4, ...; lane covers PER dims of every head
    float acc[kSlotHeads][PER], L[kSlotHeads];
#pragma unroll
    for (int g = 0; g < kSlotHeads; ++g) {
        L[g] = 0.f;
#pragma unroll
        for (int i = 0; i < PER; ++i) acc[g][i] = 0.f;
    }
#pragma unroll 4
    for (int r = warp; r < nrec; r += kConsumerWarps) {
        const size_t rec = rec0 + r;
        const float4 ma = __ldcg(reinterpret_cast<const float4*>(p.pm + rec * kSlotHeads));
        const float4 mb = __ldcg(reinterpret_cast<const float4*>(p.pm + rec * kSlotHeads + 4));
        const float4 la = __ldcg(reinterpret_cast<const float4*>(p.pl + rec * kSlotHeads));
        const float4 lb = __ldcg(reinterpret_cast<const float4*>(p.pl + rec * kSlotHeads + 4));
        const float mv[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
        const float lv[8] = {la.x, la.y, la.z, la.w, lb.x, lb.y, lb.z, lb.w};
#pragma unroll
        for (int g = 0; g < kSlotHeads; ++g) {
            if (g < G) {
                // a CTA that saw no token of a head left m = -inf, l = 0, acc = 0
                const float f = mv[g] == -INFINITY ? 0.f : exp2f(mv[g] - M[g]);
                L[g] = fmaf(f, lv[g], L[g]);
                const float* a = p.pacc + (rec * kSlotHeads + g) * D + lane * PER;
                if constexpr (PER == 4) {
                    const float4 v = __ldcg(reinterpret_cast<const float4*>(a));
                    acc[g][0] = fmaf(f, v.x, acc[g][0]);
                    acc[g][1] = fmaf(f, v.y, acc[g][1]);
                    acc[g][2] = fmaf(f, v.z, acc[g][2]);
                    acc[g][3] = fmaf(f, v.w, acc[g][3]);
                } else {
                    const float2 v = __ldcg(reinterpret_cast<const float2*>(a));
                    acc[g][0] = fmaf(f, v.x, acc[g][0]);
                    acc[g][1] = fmaf(f, v.y, acc[g][1]);
                }
            }
        }
    }

    // cross-warp sums in warp order
    for (int w = 0; w < kConsumerWarps; ++w) {
        if (warp == w) {
#pragma unroll
            for (int g = 0; g < kSlotHeads; ++g) {
                if (g < G) {
                    float* row = &cs.acc[g][lane * PER];
#pragma unroll
                    for (int i = 0; i < PER; ++i) row[i] = (w == 0) ? acc[g][i] : row[i] + acc[g][i];
                    if (lane == 0) cs.l[w][g] = L[g];
                }
            }
        }
        consumer_barrier();
    }
    const int b = unit / p.Hkv, kv = unit - b * p.Hkv;
    for (int i = tid; i < G * (D / 4); i += kConsumerWarps * 32) {
        const int g = i / (D / 4), d = (i - g * (D / 4)) * 4;
        const float inv = 1.0f / ((cs.l[0][g] + cs.l[1][g]) + (cs.l[2][g] + cs.l[3][g]));
        const float4 v = *reinterpret_cast<const float4*>(&cs.acc[g][d]);
        __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out) + ((size_t)b * p.Hq + (size_t)kv * G + g) * D + d;
        *reinterpret_cast<uint2*>(o) = make_uint2(pack_bf16x2(v.x * inv, v.y * inv), pack_bf16x2(v.z * inv, v.w * inv));
    }
}

// SCAN: the CTA computes the unit offsets itself (units <= kMaxScanUnits, kept in
// shared memory); otherwise decode_prologue_kernel has written them to the workspace.
template <int D, bool SCAN>
__global__ void __launch_bounds__(kDecThreads, kDecCtasPerSm)
    decode_main_kernel(const __grid_constant__ DecParams p, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmN) {
    using Geo = DecGeom<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* const sbase =
        reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    DecSmall& sm = *reinterpret_cast<DecSmall*>(sbase + kStages * Geo::kStageBytes);
    int* const sPrefix = reinterpret_cast<int*>(&sm + 1);
    uint64_t* const full = sm.full;
    uint64_t* const empty = sm.empty;
    volatile int* const abort_flag = &sm.abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // Private setup first; then wait for the previous kernel in the stream (its
    // lengths, cache rows and workspace state) before reading anything.
    if (tid == 0) {
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        prefetch_tmap(&tmN);
    }
    griddep_launch_dependents();
    griddep_wait();

    // ---------------------------------------------------------------- unit offsets
    const int* pre;
    int total, W;
    if constexpr (SCAN) {
        const int per = (p.BH + kDecThreads - 1) / kDecThreads;
        const int ub = tid * per;
        int local = 0;
        for (int i = 0; i < per; ++i) {
            const int u = ub + i;
            if (u < p.BH) local += eff_len(p, u, true);
        }
        int incl = local;
        for (int o = 1; o < 32; o <<= 1) {
            const int x = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += x;
        }
        if (lane == 31) sm.warp_tot[warp] = incl;
        __syncthreads();
        if (tid == 0) {
            int run = 0;
            for (int w = 0; w < kDecThreads / 32; ++w) {
                const int t = sm.warp_tot[w];
                sm.warp_tot[w] = run;
                run += t;
            }
            sm.total = run;
            sPrefix[p.BH] = run;
        }
        __syncthreads();
        int run = sm.warp_tot[warp] + incl - local;
        for (int i = 0; i < per; ++i) {
            const int u = ub + i;
            if (u < p.BH) {
                sPrefix[u] = run;
                run += eff_len(p, u, false);
            }
        }
        __syncthreads();
        pre = sPrefix;
        total = sm.total;
        W = tokens_per_cta(total, (int)gridDim.x);
    } else {
        pre = p.prefix;
        total = p.hdr->total_tokens;
        W = p.hdr->tokens_per_cta;
    }

    // Empty units get a zero output from the CTA whose range starts at their offset.
    for (int u = tid; u < p.BH; u += kDecThreads) {
        if (pre[u + 1] != pre[u]) continue;
        if (min(pre[u] / W, (int)gridDim.x - 1) != (int)blockIdx.x) continue;
        const int b = u / p.Hkv, kv = u - b * p.Hkv;
        __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out) + ((size_t)b * p.Hq + (size_t)kv * p.G) * D;
        for (int i = 0; i < p.G * D / 8; ++i) reinterpret_cast<uint4*>(o)[i] = make_uint4(0u, 0u, 0u, 0u);
    }

    const int r0 = blockIdx.x * W;
    const int r1 = min(total, r0 + W);
    // Fused append: once every CTA is done (and so done reading len), the last one
    // moves every unit's length past its new token.
    auto finish_append = [&](int nthr, bool block_sync) {
        if (!p.k_new) return;
        if (tid == 0) sm.bump = atomicAdd(&p.hdr->ctas_done, 1) == (int)gridDim.x - 1;
        if (block_sync) __syncthreads(); else consumer_barrier();
        if (!sm.bump) return;
        for (int u = tid; u < p.BH; u += nthr) {
            const int v = p.len[u];
            if (v >= 0 && v < p.cap) p.len_rw[u] = v + 1;
        }
        if (tid == 0) p.hdr->ctas_done = 0;
    };
    if (r0 >= r1) {
        finish_append(kDecThreads, true);
        return;
    }
    int u0;
    if constexpr (SCAN) {
        if (tid == 0) sm.u0 = p.BH;
        __syncthreads();
        for (int u = tid; u < p.BH; u += kDecThreads)
            if (pre[u] <= r0 && r0 < pre[u + 1]) sm.u0 = u;
        __syncthreads();
        u0 = sm.u0;
    } else {
        u0 = p.cta_unit[blockIdx.x];
    }
    int u0_last = u0;  // unit holding the range's last token
    if (p.k_new)
        while (u0_last + 1 < p.BH && pre[u0_last + 1] < r1) ++u0_last;

    // Fused append: the CTA whose range holds a unit's last row (the new token)
    // writes that row before any of its loads, 2 * D / 8 sixteen-byte pieces per
    // unit spread over the block; the fence orders the writes before the TMA reads.
    if (p.k_new) {
        constexpr int PPR = D / 8;  // 16-byte pieces per row
        for (int i = tid; i < (u0_last - u0 + 1) * 2 * PPR; i += kDecThreads) {
            const int u = u0 + i / (2 * PPR), k = i % (2 * PPR);
            const int old = p.len[u];
            if (old < 0 || old >= p.cap || pre[u + 1] - 1 < r0 || pre[u + 1] - 1 >= r1) continue;
            const size_t r = (size_t)u * p.cap + old;
            const bool isv = k >= PPR;
            const uint4* src = static_cast<const uint4*>(isv ? p.v_new : p.k_new) + (size_t)u * PPR + (k % PPR);
            uint4* dst = static_cast<uint4*>(isv ? p.V : p.K) + r * PPR + (k % PPR);
            *dst = *src;
            if (k == 0) p.N[r] = 1;
            fence_proxy_async_global();
        }
    }
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        prefetch_tmap(&tmN);
    }
    __syncthreads();
    const uint64_t budget_ns = 2000000000ull;

    if (warp == kConsumerWarps) {
        // ============================================================ producer
        if (lane == 0) {
            int issued = 0;
            RangeWalker rw{pre, p.BH, u0, r0, r1};
            int unit, t0, n;
            bool ok = true;
            while (ok && rw.next(unit, t0, n)) {
                const long long row_base = (long long)unit * p.cap;
                for (int t = 0; t < n; t += kTile) {
                    const int s = issued % kStages;
                    if (issued >= kStages) {
                        ok = mbar_wait(&empty[s], ((issued / kStages) - 1) & 1, globaltimer() + budget_ns);
                        if (!ok || *abort_flag) { ok = false; break; }
                    }
                    const int row = (int)(row_base + t0 + t);
                    uint8_t* st = sbase + s * Geo::kStageBytes;
                    mbar_expect_tx(&full[s], Geo::kTxBytes);
#pragma unroll
                    for (int bx = 0; bx < Geo::kBoxes; ++bx) {
                        tma_load_2d(st + Geo::kKOff + bx * Geo::kBoxBytes, &tmK, &full[s], bx * 64, row);
                        tma_load_2d(st + Geo::kVOff + bx * Geo::kBoxBytes, &tmV, &full[s], bx * 64, row);
                    }
                    tma_load_2d(st + Geo::kNOff, &tmN, &full[s], 0, row >> 2);
                    ++issued;
                }
            }
            if (!ok) {
                record_status(&p.hdr->status, CSMKV_ERR_TIMEOUT);
                *abort_flag = 1;
            }
            // Drain: every issued stage must land before the CTA may exit.
            for (int i = max(0, issued - kStages); i < issued; ++i)
                (void)mbar_wait(&full[i % kStages], (i / kStages) & 1, globaltimer() + budget_ns);
        }
        __syncwarp();
        return;
    }

    // ================================================================ consumers
    const int g = lane >> 2, t4 = lane & 3;
    const int tok_lo = warp * 16;
    const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(p.q);
    uint32_t qf[D / 16][2];
    float oacc[D / 16][4];
    float m0, m1, l0, l1;

    RangeWalker rw{pre, p.BH, u0, r0, r1};
    int unit, t0, n;
    int consumed = 0;
    bool ok = true;
    while (rw.next(unit, t0, n)) {
        const int b = unit / p.Hkv, kv = unit - b * p.Hkv;
        const __nv_bfloat16* qrow = qg + ((size_t)b * p.Hq + (size_t)kv * p.G + g) * D;
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
        const long long row_base = (long long)unit * p.cap;

        for (int t = 0; t < n; t += kTile) {
            const int s = consumed % kStages;
            if (!mbar_wait(&full[s], (consumed / kStages) & 1, globaltimer() + budget_ns) || *abort_flag) {
                ok = false;
                break;
            }
            const int nv = min(kTile, n - t);  // valid tokens in this tile
            uint8_t* st = sbase + s * Geo::kStageBytes;
            const int noff = (int)((row_base + t0 + t) & 3);
            const int* sN = reinterpret_cast<const int*>(st + Geo::kNOff) + noff;
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
        }
        // ---- every consumer warp reaches the barriers below, aborted or not
        if (!ok) *abort_flag = 1;
        consumer_barrier();
        if (*abort_flag) {
            ok = false;
            break;
        }
        // ---- one partial per (CTA, unit): the 4 warps' states merged in shared memory,
        //      in warp order (deterministic), then written as one record
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
        const size_t slot = (size_t)blockIdx.x + unit;
        for (int i = tid; i < p.G * (D / 4); i += kConsumerWarps * 32) {
            const int h = i / (D / 4), d = (i - h * (D / 4)) * 4;
            __stcg(reinterpret_cast<float4*>(p.pacc + (slot * kSlotHeads + h) * D + d),
                   *reinterpret_cast<const float4*>(&cs.acc[h][d]));
        }
        if (tid < p.G) {
            const float M = fmaxf(fmaxf(cs.m[0][tid], cs.m[1][tid]), fmaxf(cs.m[2][tid], cs.m[3][tid]));
            float L = 0.f;
            for (int w = 0; w < kConsumerWarps; ++w)
                if (cs.m[w][tid] != -INFINITY) L = fmaf(exp2f(cs.m[w][tid] - M), cs.l[w][tid], L);
            p.pm[slot * kSlotHeads + tid] = M;
            p.pl[slot * kSlotHeads + tid] = L;
        }
        // ---- the last CTA to finish its part of the unit merges every part. One
        //      acq_rel atomic both publishes this CTA's record (its stores are ordered
        //      before it by the barrier) and, for the last CTA, acquires the others'.
        consumer_barrier();
        const int c0 = pre[unit] / W, c1 = (pre[unit + 1] - 1) / W;
        if (tid == 0) {
            const int prev = atom_add_acq_rel_gpu(p.counter + unit, 1);
            const int last = prev == c1 - c0;
            if (last) p.counter[unit] = 0;  // ready for the next call
            sm.last = last;
        }
        consumer_barrier();
        if (sm.last) combine_unit<D>(p, unit, c0, c1, warp, lane, sm.cs);
        consumer_barrier();  // sm.last is rewritten for the next unit
    }
    if (!ok && tid == 0) record_status(&p.hdr->status, CSMKV_ERR_TIMEOUT);
    finish_append(kConsumerWarps * 32, false);
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

static size_t dec_layout(const csmkv_cache* cache, int nCTA, size_t* o_prefix, size_t* o_cta, size_t* o_cnt,
                         size_t* o_pm, size_t* o_pl, size_t* o_pacc) {
    const size_t BH = (size_t)cache->batch * cache->h_kv;
    const size_t slots = (size_t)nCTA + BH;  // one record per (CTA, unit it touches)
    size_t off = kHeaderBytes;
    *o_prefix = off;
    off = align_up(off + (BH + 1) * 4, 256);
    *o_cta = off;
    off = align_up(off + (size_t)nCTA * 4, 256);
    *o_cnt = off;
    off = align_up(off + BH * 4, 256);
    *o_pm = off;
    off = align_up(off + slots * kSlotHeads * 4, 256);
    *o_pl = off;
    off = align_up(off + slots * kSlotHeads * 4, 256);
    *o_pacc = off;
    off = align_up(off + slots * kSlotHeads * (size_t)cache->head_dim * 4, 256);
    return off;
}

template <int D, bool SCAN>
static int launch_decode_bf16(const DecParams& P, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& tn, cudaStream_t st) {
    constexpr int smem = kStages * DecGeom<D>::kStageBytes + (int)sizeof(DecSmall) +
                         (SCAN ? (kMaxScanUnits + 1) * 4 : 0) + 1024;
    static_assert(kDecCtasPerSm * (smem + 1024) <= 228 * 1024, "two CTAs per SM must fit in shared memory");
    auto kern = decode_main_kernel<D, SCAN>;
    if (set_kernel_smem((const void*)kern, smem) != CSMKV_OK) return CSMKV_ERR_CUDA;
    if (launch_overlapped(kern, dim3(P.nCTA), dim3(kDecThreads), (size_t)smem, st, P, tk, tv, tn) != cudaSuccess)
        return CSMKV_ERR_CUDA;
    return cudaGetLastError() == cudaSuccess ? CSMKV_OK : CSMKV_ERR_CUDA;
}

}  // namespace csmkv

using namespace csmkv;

extern "C" size_t decode_attn_workspace_bytes(const csmkv_cache* cache, int32_t h_q) {
    if (check_cache(cache) != CSMKV_OK || h_q < 1) return 0;
    const int nCTA = sm_count() * kDecCtasPerSm;
    if (nCTA <= 0) return 0;
    size_t a, b, c, d, e, f;
    return dec_layout(cache, nCTA, &a, &b, &c, &d, &e, &f);
}

namespace csmkv {
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

// Attention over the cache, optionally with the step's new token appended first
// (k_new != NULL: bf16 fuses the append into the attention kernel).
static int decode_attn_impl(const void* q, const void* K, const void* V, const int32_t* N, const int32_t* len,
                            const void* k_new, const void* v_new, const csmkv_cache* cache, int32_t h_q, float scale,
                            void* out, void* workspace, size_t ws_bytes, void* stream) {
    int rc = decode_attn_check_args(q, K, V, N, len, k_new, v_new, cache, h_q, scale, out);
    if (rc != CSMKV_OK) return rc;
    const int G = h_q / cache->h_kv;
    const int D = cache->head_dim;
    const bool bf16 = cache->dtype == CSMKV_BF16;
    const int nCTA = sm_count() * kDecCtasPerSm;
    if (nCTA <= 0) return CSMKV_ERR_CUDA;
    size_t o_prefix, o_cta, o_cnt, o_pm, o_pl, o_pacc;
    const size_t need = dec_layout(cache, nCTA, &o_prefix, &o_cta, &o_cnt, &o_pm, &o_pl, &o_pacc);
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
    P.prefix = reinterpret_cast<int32_t*>(ws + o_prefix);
    P.cta_unit = reinterpret_cast<int32_t*>(ws + o_cta);
    P.pm = reinterpret_cast<float*>(ws + o_pm);
    P.pl = reinterpret_cast<float*>(ws + o_pl);
    P.pacc = reinterpret_cast<float*>(ws + o_pacc);
    P.counter = reinterpret_cast<int32_t*>(ws + o_cnt);
    P.BH = cache->batch * cache->h_kv;
    P.Hkv = cache->h_kv;
    P.Hq = h_q;
    P.G = G;
    P.cap = cache->cap;
    P.D = D;
    P.nCTA = nCTA;
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

    const uint64_t rows = (uint64_t)cache->batch * cache->h_kv * cache->cap;
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
    if (P.BH <= kMaxScanUnits)
        return D == 128 ? launch_decode_bf16<128, true>(P, tk, tv, tn, st) : launch_decode_bf16<64, true>(P, tk, tv, tn, st);
    decode_prologue_kernel<<<1, 1024, 0, st>>>(P);
    if (cudaGetLastError() != cudaSuccess) return CSMKV_ERR_CUDA;
    return D == 128 ? launch_decode_bf16<128, false>(P, tk, tv, tn, st) : launch_decode_bf16<64, false>(P, tk, tv, tn, st);
}

extern "C" int decode_attn_logn(const void* q, const void* K, const void* V, const int32_t* N, const int32_t* len,
                                const csmkv_cache* cache, int32_t h_q, float scale, void* out, void* workspace,
                                size_t ws_bytes, void* stream) {
    return decode_attn_impl(q, K, V, N, len, nullptr, nullptr, cache, h_q, scale, out, workspace, ws_bytes, stream);
}

extern "C" int decode_step_logn(const void* q, const void* k_new, const void* v_new, void* K, void* V, int32_t* N,
                                int32_t* len, const csmkv_cache* cache, int32_t h_q, float scale, void* out,
                                void* workspace, size_t ws_bytes, void* stream) {
    if (!k_new || !v_new) return CSMKV_ERR_ARG;
    return decode_attn_impl(q, K, V, N, len, k_new, v_new, cache, h_q, scale, out, workspace, ws_bytes, stream);
}
