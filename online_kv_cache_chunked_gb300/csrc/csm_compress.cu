// csm_compress.cu -- one Chunked Soft Matching round on every (sequence, KV head)
// of a cache, compacted in place. [Chelsea §三 分块软匹配算法 steps 1-4;
// CentroidKV 分块软匹配 (CSM), 聚合]
//
// Work decomposition
//   A unit is one (sequence, KV head) cache. Its work items are its full chunks
//   (c rows each, from row n1) followed by "tail pieces" of up to 64 rows that
//   carry the unprocessed remainder and the recent window down by ch*m rows.
//   Items are handed out by an atomic ticket in level-major order (level j =
//   chunk j of every unit, then the tail pieces), to a persistent grid.
//
// In-place compaction
//   Chunk j writes its c-m survivors to rows [n1 + j(c-m), n1 + (j+1)(c-m)),
//   which overlap the *source* rows of at most two earlier chunks (or its own).
//   Each item publishes a "loaded" flag per array (K+N, and V) once it holds its
//   source rows on chip; an item writes an array only after every earlier item
//   whose source it overwrites has published that flag. Tickets are claimed in
//   increasing order, so every item waited on belongs to a running CTA whose
//   loads do not wait on anything: no deadlock. Each wait is bounded in time;
//   on expiry the kernel records CSMKV_ERR_TIMEOUT and stops.
//
// Similarity tile
//   bf16, c = 256, d in {64, 128}: the K chunk is split by TMA into the A rows
//   (even offsets) and B rows (odd offsets), each a 128 x d K-major operand in
//   the 128-byte swizzle layout; one thread issues d/16 tcgen05.mma (M = N =
//   128, fp32 accumulate in 128 TMEM columns); 8 warps read the 128 x 128 dot
//   products back with tcgen05.ld, scale them by fp32 inverse norms and take the
//   row argmax. Other shapes and fp32 use a CUDA-core fp32 tile.
#include <cuda_bf16.h>

#include <climits>

#include "host_util.h"
#include "ptx.cuh"

namespace csmkv {

constexpr int kCsmThreads = 256;
constexpr int kTailRows = 64;

struct CsmParams {
    void* K;
    void* V;
    int32_t* N;
    int32_t* len;
    int32_t* match_out;
    WsHeader* hdr;
    int32_t* snap;     // [BH] len at call start
    int32_t* unit_ch;  // [BH] full chunks to process (0 = untouched)
    int32_t* unit_tp;  // [BH] tail pieces to move
    int32_t* flag_kn;  // [BH][L] epoch when the item's K and N source rows are on chip
    int32_t* flag_v;   // [BH][L] epoch when the item's V source rows are on chip
    const uint8_t* head_mask;
    const uint8_t* seq_mask;
    int32_t BH, h_kv, cap, D, n1, n2, c, m, maxch, L;
    int64_t timeout_ns;
    int32_t withhold;
};

// ----------------------------------------------------------------------------
// Prologue: snapshot lengths, count the items of every unit, advance the epoch.
__global__ void __launch_bounds__(1024) csm_prologue_kernel(const CsmParams p) {
    __shared__ int red[2][32];
    int mch = 0, mtp = 0;
    for (int u = threadIdx.x; u < p.BH; u += blockDim.x) {
        const int s = p.len[u];
        p.snap[u] = s;
        bool active = true;
        if (p.head_mask && p.head_mask[u % p.h_kv]) active = false;
        if (p.seq_mask && !p.seq_mask[u / p.h_kv]) active = false;
        if (s < 0 || s > p.cap) {
            record_status(&p.hdr->status, CSMKV_ERR_ARG);
            active = false;
        }
        int ch = 0, tp = 0;
        if (active) {
            const int mid = s - p.n1 - p.n2;
            ch = mid > 0 ? mid / p.c : 0;
            if (ch > 0) tp = (s - (p.n1 + ch * p.c) + kTailRows - 1) / kTailRows;
        }
        p.unit_ch[u] = ch;
        p.unit_tp[u] = tp;
        mch = max(mch, ch);
        mtp = max(mtp, tp);
    }
    for (int o = 16; o; o >>= 1) {
        mch = max(mch, __shfl_xor_sync(0xffffffffu, mch, o));
        mtp = max(mtp, __shfl_xor_sync(0xffffffffu, mtp, o));
    }
    if ((threadIdx.x & 31) == 0) {
        red[0][threadIdx.x >> 5] = mch;
        red[1][threadIdx.x >> 5] = mtp;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w) {
            mch = max(mch, red[0][w]);
            mtp = max(mtp, red[1][w]);
        }
        p.hdr->levels_ch = mch;
        p.hdr->levels_tail = mtp;
        p.hdr->ticket = 0;
        p.hdr->epoch = p.hdr->epoch + 1;
    }
}

// ----------------------------------------------------------------------------
template <typename T>
struct Elem;
template <>
struct Elem<__nv_bfloat16> {
    static constexpr int kPer = 8;  // elements per 16-byte piece
    __device__ static void unpack(const uint4& v, float (&f)[8]) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = bf16lo(w[i]);
            f[2 * i + 1] = bf16hi(w[i]);
        }
    }
    __device__ static uint4 pack(const float (&f)[8]) {
        return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                          pack_bf16x2(f[6], f[7]));
    }
};
template <>
struct Elem<float> {
    static constexpr int kPer = 4;
    __device__ static void unpack(const uint4& v, float (&f)[4]) {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
    __device__ static uint4 pack(const float (&f)[4]) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
};

// Stage-buffer geometry. TC: [operand A|B][box of 64 columns][128 rows][128 B],
// 128-byte swizzled, as TMA writes it. SIMT: plain rows with a 16-byte pad.
template <typename T, bool TC>
struct Stage {
    uint8_t* base;
    int RB;  // row bytes
    int nbox;
    __device__ __forceinline__ uint8_t* piece(int q, int cc) const {
        if constexpr (TC) {
            const int op = q & 1, idx = q >> 1, box = cc >> 3, ch = cc & 7;
            return base + (op * nbox + box) * 16384 + sw128_off(idx, ch);
        } else {
            return base + q * (RB + 16) + cc * 16;
        }
    }
};

template <int D>
struct TcGeom {
    static constexpr int kBoxes = D / 64;
    static constexpr int kStageBytes = 2 * kBoxes * 16384;
};

// Small shared arrays after the stage buffer.
struct CsmSmall {
    float inv[256];       // inverse key norm per chunk row
    int32_t n[256];       // chunk degrees (tail items: row degrees)
    float best[256];      // per-group best similarity, then final per A row
    int32_t bestb[256];   // per-group argmax, then final per A row
    int32_t match[128];   // B index for selected A rows, else -1
    int32_t cnt[128];     // incoming edges per B row
    int32_t off[128];     // CSR offsets per B row
    int32_t nsum[128];    // merged degree per B row
    int32_t pre[132];     // selected A rows before index a (pre[H] = m)
    int16_t src[256];     // output row -> chunk row
    uint8_t list[128];    // CSR member list (A indices)
    int32_t misc[8];      // [0] ticket, [1] tmem base, [2] flag vote, [3..6] warp counts
    uint64_t bars[2];     // [0] TMA, [1] MMA
};

__host__ __device__ constexpr int csm_stage_bytes_simt(int c, int RB) {
    return (c * (RB + 16)) > (2 * kTailRows * RB) ? (c * (RB + 16)) : (2 * kTailRows * RB);
}

template <typename T, int DT, bool TC>
__global__ void __launch_bounds__(kCsmThreads, TC ? 3 : 1)
    csm_main_kernel(const __grid_constant__ CsmParams p, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV) {
    using E = Elem<T>;
    constexpr int EPP = E::kPer;
    const int D = TC ? DT : p.D;
    const int RB = D * (int)sizeof(T);
    const int PR = RB / 16;
    const int c = p.c, H = c / 2, m = p.m;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* stage_base =
        reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int stage_bytes = TC ? TcGeom<(DT > 0 ? DT : 64)>::kStageBytes : csm_stage_bytes_simt(c, RB);
    CsmSmall& sm = *reinterpret_cast<CsmSmall*>(stage_base + stage_bytes);
    Stage<T, TC> stg{stage_base, RB, TC ? (D / 64) : 0};

    T* const Kg = static_cast<T*>(p.K);
    T* const Vg = static_cast<T*>(p.V);
    int32_t* const status = &p.hdr->status;

    if (tid == 0) {
        mbar_init(&sm.bars[0], 1);
        mbar_init(&sm.bars[1], 1);
        fence_mbar_init();
        if constexpr (TC) {
            prefetch_tmap(&tmK);
            prefetch_tmap(&tmV);
        }
    }
    if constexpr (TC) {
        if (warp == 0) {
            tmem_alloc(reinterpret_cast<uint32_t*>(&sm.misc[1]), 128);
            tmem_relinquish();
        }
    }
    __syncthreads();
    if constexpr (TC) tc_fence_after();
    const uint32_t tmem = TC ? static_cast<uint32_t>(sm.misc[1]) : 0u;

    const int32_t epoch = p.hdr->epoch;
    const int levels_ch = p.hdr->levels_ch, levels_tail = p.hdr->levels_tail;
    const long long total = (long long)(levels_ch + levels_tail) * p.BH;
    uint32_t tma_phase = 0, mma_phase = 0;
    bool inflight_tma = false, inflight_mma = false;

    // Copies one 16-byte piece of output row p from the stage, merging when the
    // source row is a B token with incoming edges.
    auto emit_piece = [&](T* dst_rows, int pidx, int cc) {
        const int q = sm.src[pidx];
        uint4 val;
        if ((q & 1) && sm.cnt[q >> 1] > 0) {
            const int b = q >> 1;
            float acc[EPP], f[EPP];
            E::unpack(*reinterpret_cast<const uint4*>(stg.piece(q, cc)), f);
            const float nb = (float)sm.n[q];
#pragma unroll
            for (int e = 0; e < EPP; ++e) acc[e] = nb * f[e];
            const int o0 = sm.off[b], o1 = o0 + sm.cnt[b];
            for (int k = o0; k < o1; ++k) {
                const int qa = 2 * (int)sm.list[k];
                E::unpack(*reinterpret_cast<const uint4*>(stg.piece(qa, cc)), f);
                const float na = (float)sm.n[qa];
#pragma unroll
                for (int e = 0; e < EPP; ++e) acc[e] = fmaf(na, f[e], acc[e]);
            }
            const float ns = (float)sm.nsum[b];
#pragma unroll
            for (int e = 0; e < EPP; ++e) acc[e] = acc[e] / ns;
            val = E::pack(acc);
        } else {
            val = *reinterpret_cast<const uint4*>(stg.piece(q, cc));
        }
        *reinterpret_cast<uint4*>(dst_rows + (size_t)pidx * D + cc * EPP) = val;
    };

    // Bounded wait by thread 0 on a run of item flags; result broadcast to the block.
    auto wait_items = [&](const int32_t* flags, int lo, int hi, uint64_t deadline) -> bool {
        bool ok = true;
        if (tid == 0)
            for (int k = lo; k <= hi && ok; ++k) ok = wait_flag(flags + k, epoch, deadline);
        return __syncthreads_and(ok) != 0;
    };

    for (;;) {
        if (tid == 0) {
            int t = atomicAdd(&p.hdr->ticket, 1);
            if (ld_volatile(status) != 0) t = INT_MAX;  // another CTA failed: stop early
            sm.misc[0] = t;
        }
        __syncthreads();
        const long long t = sm.misc[0];
        if (t >= total) break;
        const int lev = (int)(t / p.BH);
        const int u = (int)(t % p.BH);
        const int ch = p.unit_ch[u];
        const int s = p.snap[u];
        const size_t urow = (size_t)u * p.cap;
        int32_t* const fkn = p.flag_kn + (size_t)u * p.L;
        int32_t* const fv = p.flag_v + (size_t)u * p.L;
        bool ok = true;

        if (lev < levels_ch && lev < ch) {
            // ================================================================ chunk item
            const int j = lev;
            const int src_row = p.n1 + j * c;
            const int dst_row = p.n1 + j * (c - m);
            const long long g0 = (long long)urow + src_row;

            // (1) stage K, read N
            if constexpr (TC) {
                if (tid == 0) {
                    mbar_expect_tx(&sm.bars[0], (uint32_t)stage_bytes);
                    const int ya = (int)(g0 & 1), za = (int)(g0 >> 1);
                    const int yb = (int)((g0 + 1) & 1), zb = (int)((g0 + 1) >> 1);
#pragma unroll
                    for (int bx = 0; bx < D / 64; ++bx) {
                        tma_load_3d(stage_base + (0 * (D / 64) + bx) * 16384, &tmK, &sm.bars[0], bx * 64, ya, za);
                        tma_load_3d(stage_base + (1 * (D / 64) + bx) * 16384, &tmK, &sm.bars[0], bx * 64, yb, zb);
                    }
                }
                inflight_tma = true;
            } else {
                const uint4* src = reinterpret_cast<const uint4*>(Kg + (urow + src_row) * D);
                for (int i = tid; i < c * PR; i += kCsmThreads) {
                    const int q = i / PR, cc = i - q * PR;
                    *reinterpret_cast<uint4*>(stg.piece(q, cc)) = src[(size_t)q * PR + cc];
                }
            }
            for (int q = tid; q < c; q += kCsmThreads) sm.n[q] = p.N[urow + src_row + q];
            if constexpr (TC) {
                ok = mbar_wait(&sm.bars[0], tma_phase, globaltimer() + p.timeout_ns);
                tma_phase ^= 1u;
            }
            ok = __syncthreads_and(ok) != 0;
            if (!ok) { record_status(status, CSMKV_ERR_TIMEOUT); break; }
            inflight_tma = false;
            if (tid == 0 && !p.withhold) {
                __threadfence();
                st_release(fkn + j, epoch);
            }

            // (2) inverse norms of every chunk row
            for (int q = tid; q < c; q += kCsmThreads) {
                float ss = 0.f;
                for (int cc = 0; cc < PR; ++cc) {
                    float f[EPP];
                    E::unpack(*reinterpret_cast<const uint4*>(stg.piece(q, cc)), f);
#pragma unroll
                    for (int e = 0; e < EPP; ++e) ss = fmaf(f[e], f[e], ss);
                }
                sm.inv[q] = ss > 0.f ? 1.0f / sqrtf(ss) : 0.0f;
            }
            __syncthreads();

            // (3) similarity tile and per-A argmax over groups of B columns
            int ngroups;
            if constexpr (TC) {
                ngroups = 2;
                if (tid == 0) {
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const int box = ks >> 2, koff = (ks & 3) * 32;
                        const uint64_t ad = smem_desc_sw128(smem_u32(stage_base + (0 * (D / 64) + box) * 16384 + koff));
                        const uint64_t bd = smem_desc_sw128(smem_u32(stage_base + (1 * (D / 64) + box) * 16384 + koff));
                        tc_mma_bf16(tmem, ad, bd, idesc_bf16_f32(128, 128), ks > 0 ? 1u : 0u);
                    }
                    tc_commit(&sm.bars[1]);
                }
                inflight_mma = true;
                ok = mbar_wait(&sm.bars[1], mma_phase, globaltimer() + p.timeout_ns);
                mma_phase ^= 1u;
                ok = __syncthreads_and(ok) != 0;
                if (!ok) { record_status(status, CSMKV_ERR_TIMEOUT); break; }
                inflight_mma = false;
                tc_fence_after();
                const int qtr = warp & 3, half = warp >> 2;
                const int a = qtr * 32 + lane;
                const float inv_a = sm.inv[2 * a];
                float best = -INFINITY;
                int bb = half * 64;
#pragma unroll
                for (int cb = 0; cb < 2; ++cb) {
                    float v[32];
                    const int col0 = half * 64 + cb * 32;
                    tmem_ld_32x32b_x32(tmem + ((uint32_t)(qtr * 32) << 16) + (uint32_t)col0, v);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float cs = v[i] * inv_a * sm.inv[2 * (col0 + i) + 1];
                        if (cs > best) { best = cs; bb = col0 + i; }
                    }
                }
                sm.best[half * 128 + a] = best;
                sm.bestb[half * 128 + a] = bb;
                tc_fence_before();
            } else {
                ngroups = kCsmThreads / H;
                const int per = (H + ngroups - 1) / ngroups;
                const int a = tid % H, g = tid / H;
                if (g < ngroups) {
                    const int b0 = g * per, b1 = min(H, b0 + per);
                    const float inv_a = sm.inv[2 * a];
                    float best = -INFINITY;
                    int bb = b0;
                    for (int b = b0; b < b1; ++b) {
                        float dot = 0.f;
                        for (int cc = 0; cc < PR; ++cc) {
                            float fa[EPP], fb[EPP];
                            E::unpack(*reinterpret_cast<const uint4*>(stg.piece(2 * a, cc)), fa);
                            E::unpack(*reinterpret_cast<const uint4*>(stg.piece(2 * b + 1, cc)), fb);
#pragma unroll
                            for (int e = 0; e < EPP; ++e) dot = fmaf(fa[e], fb[e], dot);
                        }
                        const float cs = dot * inv_a * sm.inv[2 * b + 1];
                        if (cs > best) { best = cs; bb = b; }
                    }
                    sm.best[g * H + a] = best;
                    sm.bestb[g * H + a] = bb;
                }
            }
            __syncthreads();
            if (tid < H) {  // combine groups in column order: later group wins only if strictly better
                float best = sm.best[tid];
                int bb = sm.bestb[tid];
                for (int g = 1; g < ngroups; ++g) {
                    const float v = sm.best[g * H + tid];
                    if (v > best) { best = v; bb = sm.bestb[g * H + tid]; }
                }
                sm.best[tid] = (best == best) ? best : -INFINITY;  // a NaN key ranks last
                sm.bestb[tid] = bb;
                sm.cnt[tid] = 0;
            }
            __syncthreads();

            // (4) top-m edges by (similarity desc, A index asc), exactly m of them
            bool sel = false;
            if (tid < H) {
                const float key = sm.best[tid];
                int rank = 0;
                for (int a2 = 0; a2 < H; ++a2) {
                    const float k2 = sm.best[a2];
                    rank += (k2 > key) || (k2 == key && a2 < tid);
                }
                sel = rank < m;
                sm.match[tid] = sel ? sm.bestb[tid] : -1;
                if (sel) atomicAdd(&sm.cnt[sm.bestb[tid]], 1);
            }
            {   // exclusive prefix of the selection over A (H <= 128 -> warps 0..3)
                const unsigned bal = __ballot_sync(0xffffffffu, sel);
                if (lane == 0 && warp < 4) sm.misc[3 + warp] = __popc(bal);
                __syncthreads();
                if (tid < H) {
                    int before = __popc(bal & ((1u << lane) - 1u));
                    for (int w = 0; w < warp; ++w) before += sm.misc[3 + w];
                    sm.pre[tid] = before;
                }
                if (tid == 0) sm.pre[H] = m;
            }
            if (warp == 0) {  // CSR offsets of incoming edges per B row (H <= 128: 4 per lane)
                int v[4], run = 0;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int b = lane * 4 + i;
                    v[i] = b < H ? sm.cnt[b] : 0;
                    run += v[i];
                }
                int incl = run;
                for (int o = 1; o < 32; o <<= 1) {
                    const int x = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += x;
                }
                int ex = incl - run;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int b = lane * 4 + i;
                    if (b < H) sm.off[b] = ex;
                    ex += v[i];
                }
            }
            __syncthreads();
            // output row of every kept chunk row; members of every merged B row
            for (int q = tid; q < c; q += kCsmThreads) {
                if ((q & 1) == 0) {
                    if (sm.match[q >> 1] < 0) sm.src[q - sm.pre[q >> 1]] = (int16_t)q;
                } else {
                    sm.src[q - sm.pre[(q >> 1) + 1]] = (int16_t)q;
                }
            }
            if (tid < H && sel) {
                const int b = sm.match[tid];
                int r = 0;
                for (int a2 = 0; a2 < tid; ++a2) r += (sm.match[a2] == b);
                sm.list[sm.off[b] + r] = (uint8_t)tid;
            }
            if (p.match_out && tid < H) p.match_out[((size_t)u * p.maxch + j) * H + tid] = sm.match[tid];
            __syncthreads();
            if (tid < H) {
                int ns = sm.n[2 * tid + 1];
                const int o0 = sm.off[tid], o1 = o0 + sm.cnt[tid];
                for (int k = o0; k < o1; ++k) ns += sm.n[2 * (int)sm.list[k]];
                sm.nsum[tid] = ns;
            }
            if (j == 0 && tid == 0) p.len[u] = s - ch * m;

            // (5) K and N: wait for the items whose sources we overwrite, then write
            const int lo = (j * (c - m)) / c, hi = min(((j + 1) * (c - m) - 1) / c, j - 1);
            ok = wait_items(fkn, lo, hi, globaltimer() + p.timeout_ns);
            if (!ok) { record_status(status, CSMKV_ERR_TIMEOUT); break; }
            {
                T* const dstK = Kg + (urow + dst_row) * D;
                const int npieces = (c - m) * PR;
                for (int i = tid; i < npieces; i += kCsmThreads) {
                    const int pr = i / PR;
                    emit_piece(dstK, pr, i - pr * PR);
                }
                int32_t* const dstN = p.N + urow + dst_row;
                for (int pr = tid; pr < c - m; pr += kCsmThreads) {
                    const int q = sm.src[pr];
                    dstN[pr] = ((q & 1) && sm.cnt[q >> 1] > 0) ? sm.nsum[q >> 1] : sm.n[q];
                }
            }

            // (6) stage V into the same buffer, publish, wait, write
            if constexpr (TC) fence_proxy_async_smem();
            __syncthreads();
            if constexpr (TC) {
                if (tid == 0) {
                    mbar_expect_tx(&sm.bars[0], (uint32_t)stage_bytes);
                    const int ya = (int)(g0 & 1), za = (int)(g0 >> 1);
                    const int yb = (int)((g0 + 1) & 1), zb = (int)((g0 + 1) >> 1);
#pragma unroll
                    for (int bx = 0; bx < D / 64; ++bx) {
                        tma_load_3d(stage_base + (0 * (D / 64) + bx) * 16384, &tmV, &sm.bars[0], bx * 64, ya, za);
                        tma_load_3d(stage_base + (1 * (D / 64) + bx) * 16384, &tmV, &sm.bars[0], bx * 64, yb, zb);
                    }
                }
                inflight_tma = true;
                ok = mbar_wait(&sm.bars[0], tma_phase, globaltimer() + p.timeout_ns);
                tma_phase ^= 1u;
            } else {
                const uint4* src = reinterpret_cast<const uint4*>(Vg + (urow + src_row) * D);
                for (int i = tid; i < c * PR; i += kCsmThreads) {
                    const int q = i / PR, cc = i - q * PR;
                    *reinterpret_cast<uint4*>(stg.piece(q, cc)) = src[(size_t)q * PR + cc];
                }
            }
            ok = __syncthreads_and(ok) != 0;
            if (!ok) { record_status(status, CSMKV_ERR_TIMEOUT); break; }
            inflight_tma = false;
            if (tid == 0 && !p.withhold) {
                __threadfence();
                st_release(fv + j, epoch);
            }
            ok = wait_items(fv, lo, hi, globaltimer() + p.timeout_ns);
            if (!ok) { record_status(status, CSMKV_ERR_TIMEOUT); break; }
            {
                T* const dstV = Vg + (urow + dst_row) * D;
                const int npieces = (c - m) * PR;
                for (int i = tid; i < npieces; i += kCsmThreads) {
                    const int pr = i / PR;
                    emit_piece(dstV, pr, i - pr * PR);
                }
            }
        } else if (lev >= levels_ch && lev - levels_ch < p.unit_tp[u]) {
            // ================================================================ tail piece
            const int piece = lev - levels_ch;
            const int T0 = p.n1 + ch * c;
            const int shift = ch * m;
            const int r0 = T0 + piece * kTailRows;
            const int nrows = min(kTailRows, s - r0);
            uint8_t* const sK = stage_base;
            uint8_t* const sV = stage_base + kTailRows * RB;
            {
                const uint4* srcK = reinterpret_cast<const uint4*>(Kg + (urow + r0) * D);
                const uint4* srcV = reinterpret_cast<const uint4*>(Vg + (urow + r0) * D);
                for (int i = tid; i < nrows * PR; i += kCsmThreads) {
                    reinterpret_cast<uint4*>(sK)[i] = srcK[i];
                    reinterpret_cast<uint4*>(sV)[i] = srcV[i];
                }
                for (int q = tid; q < nrows; q += kCsmThreads) sm.n[q] = p.N[urow + r0 + q];
            }
            __syncthreads();
            if (tid == 0 && !p.withhold) {
                __threadfence();
                st_release(fkn + p.maxch + piece, epoch);
                st_release(fv + p.maxch + piece, epoch);
            }
            const int d0 = r0 - shift, d1 = d0 + nrows;
            bool okw = true;
            if (tid == 0) {
                const uint64_t deadline = globaltimer() + p.timeout_ns;
                if (d0 < T0) {  // chunks whose sources lie under our destination
                    const int klo = (d0 - p.n1) / c;
                    const int khi = (min(d1, T0) - 1 - p.n1) / c;
                    for (int k = klo; k <= khi && okw; ++k)
                        okw = wait_flag(fkn + k, epoch, deadline) && wait_flag(fv + k, epoch, deadline);
                }
                if (d1 > T0) {  // earlier tail pieces under our destination
                    const int plo = d0 > T0 ? (d0 - T0) / kTailRows : 0;
                    const int phi = min(piece - 1, (d1 - 1 - T0) / kTailRows);
                    for (int q = plo; q <= phi && okw; ++q) okw = wait_flag(fkn + p.maxch + q, epoch, deadline);
                }
            }
            ok = __syncthreads_and(okw) != 0;
            if (!ok) { record_status(status, CSMKV_ERR_TIMEOUT); break; }
            {
                uint4* dstK = reinterpret_cast<uint4*>(Kg + (urow + d0) * D);
                uint4* dstV = reinterpret_cast<uint4*>(Vg + (urow + d0) * D);
                for (int i = tid; i < nrows * PR; i += kCsmThreads) {
                    dstK[i] = reinterpret_cast<const uint4*>(sK)[i];
                    dstV[i] = reinterpret_cast<const uint4*>(sV)[i];
                }
                for (int q = tid; q < nrows; q += kCsmThreads) p.N[urow + d0 + q] = sm.n[q];
            }
        }
        if constexpr (TC) fence_proxy_async_smem();  // the next TMA overwrites the stage
        __syncthreads();
    }

    // Teardown: after an abort, give in-flight copies and MMAs a bounded chance to land.
    if constexpr (TC) {
        if (inflight_tma) (void)mbar_wait(&sm.bars[0], tma_phase, globaltimer() + p.timeout_ns);
        if (inflight_mma) (void)mbar_wait(&sm.bars[1], mma_phase, globaltimer() + p.timeout_ns);
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (warp == 0) tmem_dealloc(tmem, 128);
    }
}

// ----------------------------------------------------------------------------
template <typename T, int DT, bool TC>
static int launch_main(const CsmParams& P, const CUtensorMap& tmK, const CUtensorMap& tmV, int smem,
                       int ctas_per_sm, cudaStream_t st) {
    auto kern = csm_main_kernel<T, DT, TC>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
        return CSMKV_ERR_CUDA;
    const int grid = sm_count() * ctas_per_sm;
    if (grid <= 0) return CSMKV_ERR_CUDA;
    kern<<<grid, kCsmThreads, smem, st>>>(P, tmK, tmV);
    return cudaGetLastError() == cudaSuccess ? CSMKV_OK : CSMKV_ERR_CUDA;
}

static size_t csm_layout(const csmkv_cache* cache, int32_t n1, int32_t n2, int32_t c, size_t* off_snap,
                         size_t* off_ch, size_t* off_tp, size_t* off_fkn, size_t* off_fv, int32_t* L_out) {
    const size_t BH = (size_t)cache->batch * cache->h_kv;
    const int32_t maxch = csm_max_chunks(cache, n1, n2, c);
    const int32_t tail = (c - 1 + n2 + kTailRows - 1) / kTailRows;
    const int32_t L = maxch + tail;
    size_t off = kHeaderBytes;
    *off_snap = off;
    off = align_up(off + BH * 4, 256);
    *off_ch = off;
    off = align_up(off + BH * 4, 256);
    *off_tp = off;
    off = align_up(off + BH * 4, 256);
    *off_fkn = off;
    off = align_up(off + BH * (size_t)L * 4, 256);
    *off_fv = off;
    off = align_up(off + BH * (size_t)L * 4, 256);
    *L_out = L;
    return off;
}

}  // namespace csmkv

using namespace csmkv;

extern "C" int32_t csm_max_chunks(const csmkv_cache* cache, int32_t n1, int32_t n2, int32_t c) {
    if (!cache || c <= 0) return 0;
    const int32_t mid = cache->cap - n1 - n2;
    return mid > 0 ? mid / c : 0;
}

extern "C" size_t csm_workspace_bytes(const csmkv_cache* cache, int32_t n1, int32_t n2, int32_t c) {
    if (check_cache(cache) != CSMKV_OK || n1 < 0 || n2 < 0 || c < 2 || (c & 1)) return 0;
    size_t a, b, d, e, f;
    int32_t L;
    return csm_layout(cache, n1, n2, c, &a, &b, &d, &e, &f, &L);
}

extern "C" int csm_compress_ex(void* K, void* V, int32_t* N, int32_t* len, const csmkv_cache* cache,
                               int32_t n1, int32_t n2, int32_t c, double r, const uint8_t* head_mask,
                               const uint8_t* seq_mask, int32_t* match_out, const csm_options* opts,
                               void* workspace, size_t ws_bytes, void* stream) {
    int rc = check_cache(cache);
    if (rc != CSMKV_OK) return rc;
    if (!K || !V || !N || !len) return CSMKV_ERR_ARG;
    if (!aligned16(K) || !aligned16(V) || !aligned16(N) || (reinterpret_cast<uintptr_t>(len) & 3u))
        return CSMKV_ERR_ALIGN;
    if (n1 < 0 || n2 < 0 || c < 2 || c > 256 || (c & 1)) return CSMKV_ERR_ARG;
    if (!(r >= 0.0 && r <= 0.5)) return CSMKV_ERR_ARG;  // also rejects NaN
    const int32_t m = csm_edges_per_chunk(r, c);
    if (m < 0 || m > c / 2) return CSMKV_ERR_ARG;
    size_t o_snap, o_ch, o_tp, o_fkn, o_fv;
    int32_t L;
    const size_t need = csm_layout(cache, n1, n2, c, &o_snap, &o_ch, &o_tp, &o_fkn, &o_fv, &L);
    if (!workspace || ws_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u)) return CSMKV_ERR_WORKSPACE;
    const int32_t maxch = csm_max_chunks(cache, n1, n2, c);
    if (m == 0 || maxch == 0) return CSMKV_OK;  // nothing can merge

    uint8_t* ws = static_cast<uint8_t*>(workspace);
    CsmParams P{};
    P.K = K;
    P.V = V;
    P.N = N;
    P.len = len;
    P.match_out = match_out;
    P.hdr = reinterpret_cast<WsHeader*>(ws);
    P.snap = reinterpret_cast<int32_t*>(ws + o_snap);
    P.unit_ch = reinterpret_cast<int32_t*>(ws + o_ch);
    P.unit_tp = reinterpret_cast<int32_t*>(ws + o_tp);
    P.flag_kn = reinterpret_cast<int32_t*>(ws + o_fkn);
    P.flag_v = reinterpret_cast<int32_t*>(ws + o_fv);
    P.head_mask = head_mask;
    P.seq_mask = seq_mask;
    P.BH = cache->batch * cache->h_kv;
    P.h_kv = cache->h_kv;
    P.cap = cache->cap;
    P.D = cache->head_dim;
    P.n1 = n1;
    P.n2 = n2;
    P.c = c;
    P.m = m;
    P.maxch = maxch;
    P.L = L;
    P.timeout_ns = (opts && opts->wait_timeout_ns > 0) ? opts->wait_timeout_ns : 2000000000LL;
    P.withhold = opts ? opts->withhold_signals : 0;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    csm_prologue_kernel<<<1, 1024, 0, st>>>(P);
    if (cudaGetLastError() != cudaSuccess) return CSMKV_ERR_CUDA;

    const int D = cache->head_dim;
    const bool tc = cache->dtype == CSMKV_BF16 && c == 256 && (D == 64 || D == 128) && !(opts && opts->force_simt);
    CUtensorMap tmK{}, tmV{};
    if (tc) {
        const uint64_t rows = (uint64_t)cache->batch * cache->h_kv * cache->cap;
        const uint64_t dims[3] = {(uint64_t)D, 2, rows / 2};
        const uint64_t strides[2] = {(uint64_t)D * 2, (uint64_t)D * 4};
        const uint32_t box[3] = {64, 1, 128};
        if (!encode_tiled(&tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, K, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B) ||
            !encode_tiled(&tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, V, dims, strides, box,
                          CU_TENSOR_MAP_SWIZZLE_128B))
            return CSMKV_ERR_CUDA;
        const int smem = (D == 128 ? TcGeom<128>::kStageBytes : TcGeom<64>::kStageBytes) + (int)sizeof(CsmSmall) + 1024;
        return D == 128 ? launch_main<__nv_bfloat16, 128, true>(P, tmK, tmV, smem, 3, st)
                        : launch_main<__nv_bfloat16, 64, true>(P, tmK, tmV, smem, 3, st);
    }
    const int RB = D * (int)dtype_bytes(cache->dtype);
    const int smem = csm_stage_bytes_simt(c, RB) + (int)sizeof(CsmSmall) + 1024;
    if (smem > 227 * 1024) return CSMKV_ERR_UNSUPPORTED;
    return cache->dtype == CSMKV_BF16 ? launch_main<__nv_bfloat16, 0, false>(P, tmK, tmV, smem, 1, st)
                                      : launch_main<float, 0, false>(P, tmK, tmV, smem, 1, st);
}

extern "C" int csm_compress(void* K, void* V, int32_t* N, int32_t* len, const csmkv_cache* cache, int32_t n1,
                            int32_t n2, int32_t c, double r, const uint8_t* head_mask, const uint8_t* seq_mask,
                            void* workspace, size_t ws_bytes, void* stream) {
    return csm_compress_ex(K, V, N, len, cache, n1, n2, c, r, head_mask, seq_mask, nullptr, nullptr, workspace,
                           ws_bytes, stream);
}
