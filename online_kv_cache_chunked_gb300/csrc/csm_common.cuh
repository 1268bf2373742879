// csm_common.cuh -- parts of one Chunked Soft Matching round shared by the
// tensor-core kernel (csm_tc3.cu) and the CUDA-core kernel (csm_compress.cu):
// work-item bookkeeping, the top-m selection and compaction tables, the
// degree-weighted merge of output rows and the tail move.
// [Chelsea §三 分块软匹配算法 steps 1-4; CentroidKV 分块软匹配 (CSM), 聚合]
#pragma once
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
    const int32_t* seq_limit;  // [batch] or NULL: at most this many chunks of sequence b (<= 0: all)
    RowMap rm;                 // logical row -> pool row (a paged layout's block table)
    int32_t BH, h_kv, cap, D, n1, n2, c, m, maxch, L;
    int64_t timeout_ns;
    int32_t withhold;
    int32_t paged_tma;  // block-table layout: chunk rows by TMA in 16-row groups (n1 a multiple of 16)
};

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

// Shared-memory tables of one chunk's decisions. 16-byte aligned and sized, so
// whatever follows it in shared memory (mbarriers included) stays aligned.
struct alignas(16) CsmTables {
    float invA[128];        // inverse key norm of A row a (chunk offset 2a)
    float invB[128];        // inverse key norm of B row b (chunk offset 2b+1)
    float best[512];        // per-group best similarity, then final per A row
    uint8_t bestb[512];     // per-group argmax, then final per A row
    int16_t match[128];     // B index for selected A rows, else -1
    uint32_t mask[128][4];  // bit a set: A row a merges into this B row
    int32_t nsum[128];      // degree of B row b after the round
    float ninv[128];        // 1 / nsum for B rows with incoming edges, 0 otherwise
    int16_t pre[136];       // selected A rows before index a (pre[H] = m)
    int16_t src[256];       // output row -> chunk row (only when m < H)
    uint8_t mlist[128];     // B rows with incoming edges, ascending
    int32_t nmerged;        // their count
    int32_t misc[8];        // [3..6] warp counts
};
static_assert(sizeof(CsmTables) % 16 == 0, "tables keep what follows them aligned");

// First non-empty work item at or after ticket t (claiming further tickets past
// empty ones), or INT_MAX when the work is done or a CTA has failed.
__device__ __forceinline__ int claim_from(const CsmParams& p, int t, int levels_ch, long long total) {
    for (;;) {
        if (t >= total || ld_volatile(&p.hdr->status) != 0) return INT_MAX;
        const int lev = t / p.BH, u = t - lev * p.BH;
        if (lev < levels_ch ? lev < p.unit_ch[u] : (lev - levels_ch) < p.unit_tp[u]) return t;
        t = atomicAdd(&p.hdr->ticket, 1);
    }
}

__device__ __forceinline__ int claim_item(const CsmParams& p, int levels_ch, long long total) {
    return claim_from(p, atomicAdd(&p.hdr->ticket, 1), levels_ch, total);
}

// Bounded wait by thread 0 on a run of item flags; the result is broadcast to the block.
__device__ __forceinline__ bool wait_items(const int32_t* flags, int lo, int hi, int32_t epoch, uint64_t deadline) {
    bool ok = true;
    if (threadIdx.x == 0)
        for (int k = lo; k <= hi && ok; ++k) ok = wait_flag(flags + k, epoch, deadline);
    return __syncthreads_and(ok) != 0;
}

__device__ __forceinline__ void publish(int32_t* flag, int32_t epoch, int withhold) {
    if (!withhold) {
        __threadfence();
        st_release(flag, epoch);
    }
}

// From per-group (best, argmax) records to the chunk's merge plan: exactly m
// selected A rows (similarity desc, A index asc), for every B row the set of A
// rows merging into it (a bit mask: atomicOr makes it independent of thread
// order, so the merge sums run in A order on every run), the merged degrees and,
// when m < H, the output row -> chunk row map. With m == H every A row is
// selected and the output rows are exactly the B rows. All threads call.
// With H = 128 and 256 or 512 threads, R = blockDim / 128 consecutive threads
// share one A row's rank count.
__device__ inline void chunk_tables(CsmTables& sm, const int32_t* sN, int c, int m, int ngroups) {
    const int H = c / 2;
    const bool all = (m == H);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int R = (H == 128 && blockDim.x >= 256) ? (int)blockDim.x / 128 : 1;  // 1, 2 or 4
    const int ra = tid / R, rp = tid - ra * R, span = H / R;
    if (tid < H) {  // combine groups in column order: a later group wins only if strictly better
        float best = sm.best[tid];
        int bb = sm.bestb[tid];
        for (int g = 1; g < ngroups; ++g) {
            const float v = sm.best[g * H + tid];
            if (v > best) { best = v; bb = sm.bestb[g * H + tid]; }
        }
        sm.best[tid] = (best == best) ? best : -INFINITY;  // a NaN key ranks last
        sm.bestb[tid] = (uint8_t)bb;
        sm.mask[tid][0] = sm.mask[tid][1] = sm.mask[tid][2] = sm.mask[tid][3] = 0u;
    }
    __syncthreads();
    if (all) {
        if (tid < H) {
            const int b = sm.bestb[tid];
            sm.match[tid] = (int16_t)b;
            atomicOr(&sm.mask[b][tid >> 5], 1u << (tid & 31));
        }
    } else if (ra < H) {  // rank of A row ra among all A rows, counted over R parts
        const float key = sm.best[ra];
        int rank = 0;
        const int a0 = rp * span;
#pragma unroll 8
        for (int i = 0; i < span; ++i) {
            const int a2 = a0 + i;
            const float k2 = sm.best[a2];
            rank += (k2 > key) || (k2 == key && a2 < ra);
        }
        for (int o = 1; o < R; o <<= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
        if (rp == 0) {
            const bool sel = rank < m;
            const int b = sm.bestb[ra];
            sm.match[ra] = (int16_t)(sel ? b : -1);
            if (sel) atomicOr(&sm.mask[b][ra >> 5], 1u << (ra & 31));
        }
    }
    __syncthreads();
    if (!all) {  // exclusive prefix of the selection over A (H <= 128 -> warps 0..3)
        const bool sel = tid < H && sm.match[tid] >= 0;
        const unsigned bal = __ballot_sync(0xffffffffu, sel);
        if (lane == 0 && warp < 4) sm.misc[3 + warp] = __popc(bal);
        __syncthreads();
        if (tid < H) {
            int before = __popc(bal & ((1u << lane) - 1u));
            for (int w = 0; w < warp; ++w) before += sm.misc[3 + w];
            sm.pre[tid] = (int16_t)before;
        }
        if (tid == 0) sm.pre[H] = (int16_t)m;
        __syncthreads();
        for (int q = tid; q < c; q += blockDim.x) {
            if ((q & 1) == 0) {
                if (sm.match[q >> 1] < 0) sm.src[q - sm.pre[q >> 1]] = (int16_t)q;
            } else {
                sm.src[q - sm.pre[(q >> 1) + 1]] = (int16_t)q;
            }
        }
    }
    if (tid < H) {
        int ns = sN[2 * tid + 1];
        bool any = false;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            uint32_t bits = sm.mask[tid][w];
            any |= bits != 0u;
            while (bits) {
                ns += sN[2 * (w * 32 + __ffs(bits) - 1)];
                bits &= bits - 1u;
            }
        }
        sm.nsum[tid] = ns;
        sm.ninv[tid] = any ? 1.0f / (float)ns : 0.0f;
    }
    {   // list of the merged B rows (H <= 128 -> warps 0..3)
        const bool any = tid < H && sm.ninv[tid] != 0.0f;
        const unsigned bal = __ballot_sync(0xffffffffu, any);
        __syncthreads();  // misc is reused; also orders the ninv writes above
        if (lane == 0 && warp < 4) sm.misc[3 + warp] = __popc(bal);
        __syncthreads();
        if (any) {
            int pos = __popc(bal & ((1u << lane) - 1u));
            for (int w = 0; w < warp; ++w) pos += sm.misc[3 + w];
            sm.mlist[pos] = (uint8_t)tid;
        }
        if (tid == 0) sm.nmerged = sm.misc[3] + sm.misc[4] + sm.misc[5] + sm.misc[6];
    }
    __syncthreads();
}

// Writes the c - m output rows of one array of a chunk: copies, or degree-
// weighted means for B rows with incoming edges (fp32 sums in A order, scaled
// by the reciprocal of the degree sum, rounded once to the cache dtype).
// piece(q, cc) gives the 16-byte piece cc of chunk row q in shared memory.
template <typename T, typename PieceFn>
__device__ __forceinline__ void emit_rows(T* dst_rows, int rows_out, int D, int m, const CsmTables& sm,
                                          const int32_t* sN, PieceFn piece) {
    using E = Elem<T>;
    constexpr int EPP = E::kPer;
    const int PR = D * (int)sizeof(T) / 16;
    const bool all = (rows_out == m);  // c - m == m exactly when m == H: the output rows are the B rows
    const int npieces = rows_out * PR;
    for (int i = threadIdx.x; i < npieces; i += blockDim.x) {
        const int pr = i / PR, cc = i - pr * PR;
        const int q = all ? 2 * pr + 1 : sm.src[pr];
        uint4 val = *reinterpret_cast<const uint4*>(piece(q, cc));
        if (q & 1) {
            const int b = q >> 1;
            const float inv = sm.ninv[b];
            if (inv != 0.0f) {
                float acc[EPP], f[EPP];
                E::unpack(val, f);
                const float nb = (float)sN[q];
#pragma unroll
                for (int e = 0; e < EPP; ++e) acc[e] = nb * f[e];
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    uint32_t bits = sm.mask[b][w];
                    while (bits) {
                        const int qa = 2 * (w * 32 + __ffs(bits) - 1);
                        bits &= bits - 1u;
                        E::unpack(*reinterpret_cast<const uint4*>(piece(qa, cc)), f);
                        const float na = (float)sN[qa];
#pragma unroll
                        for (int e = 0; e < EPP; ++e) acc[e] = fmaf(na, f[e], acc[e]);
                    }
                }
#pragma unroll
                for (int e = 0; e < EPP; ++e) acc[e] *= inv;
                val = E::pack(acc);
            }
        }
        *reinterpret_cast<uint4*>(dst_rows + (size_t)pr * D + cc * EPP) = val;
    }
}

__device__ __forceinline__ void emit_degrees(int32_t* dstN, int rows_out, int m, const CsmTables& sm,
                                             const int32_t* sN) {
    const bool all = (rows_out == m);
    for (int pr = threadIdx.x; pr < rows_out; pr += blockDim.x) {
        const int q = all ? 2 * pr + 1 : sm.src[pr];
        dstN[pr] = (q & 1) ? sm.nsum[q >> 1] : sN[q];
    }
}

// Chunks whose source rows the destination of chunk j overlaps (earlier than j).
__device__ __forceinline__ void chunk_deps(int j, int c, int m, int& lo, int& hi) {
    lo = (j * (c - m)) / c;
    hi = min(((j + 1) * (c - m) - 1) / c, j - 1);
}

// One tail piece: up to 64 rows of the remainder + recent window moved down by
// ch*m rows, staged through `stage` (>= 2 * 64 * row bytes), degrees through sN.
// PAGED: every row goes through the block table (rows whose entry is outside the
// pool are skipped and CSMKV_ERR_ARG recorded).
template <typename T, bool PAGED = false>
__device__ bool tail_piece(const CsmParams& p, int u, int piece, int32_t epoch, uint8_t* stage, int32_t* sN) {
    const int tid = threadIdx.x;
    const int c = p.c, m = p.m, D = p.D;
    const int ch = p.unit_ch[u];
    const int s = p.snap[u];
    const size_t urow = (size_t)u * p.cap;
    const int RB = D * (int)sizeof(T), PR = RB / 16;
    const int T0 = p.n1 + ch * c;
    const int shift = ch * m;
    const int r0 = T0 + piece * kTailRows;
    const int nrows = min(kTailRows, s - r0);
    int32_t* const fkn = p.flag_kn + (size_t)u * p.L;
    int32_t* const fv = p.flag_v + (size_t)u * p.L;
    T* const Kg = static_cast<T*>(p.K);
    T* const Vg = static_cast<T*>(p.V);
    uint8_t* const sK = stage;
    uint8_t* const sV = stage + kTailRows * RB;
    if constexpr (PAGED) {
        for (int i = tid; i < nrows * PR; i += blockDim.x) {
            const int q = i / PR, k = i - q * PR;
            const long long pr = map_row(p.rm, u, r0 + q);
            if (pr < 0) {
                if (k == 0) record_status(&p.hdr->status, CSMKV_ERR_ARG);
                continue;
            }
            reinterpret_cast<uint4*>(sK)[i] = reinterpret_cast<const uint4*>(Kg + pr * D)[k];
            reinterpret_cast<uint4*>(sV)[i] = reinterpret_cast<const uint4*>(Vg + pr * D)[k];
        }
        for (int q = tid; q < nrows; q += blockDim.x) {
            const long long pr = map_row(p.rm, u, r0 + q);
            sN[q] = pr < 0 ? 0 : p.N[pr];
        }
    } else {
        const uint4* srcK = reinterpret_cast<const uint4*>(Kg + (urow + r0) * D);
        const uint4* srcV = reinterpret_cast<const uint4*>(Vg + (urow + r0) * D);
        for (int i = tid; i < nrows * PR; i += blockDim.x) {
            reinterpret_cast<uint4*>(sK)[i] = srcK[i];
            reinterpret_cast<uint4*>(sV)[i] = srcV[i];
        }
        for (int q = tid; q < nrows; q += blockDim.x) sN[q] = p.N[urow + r0 + q];
    }
    __syncthreads();
    if (tid == 0) {
        publish(fkn + p.maxch + piece, epoch, p.withhold);
        publish(fv + p.maxch + piece, epoch, p.withhold);
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
    if (!__syncthreads_and(okw)) return false;
    if constexpr (PAGED) {
        for (int i = tid; i < nrows * PR; i += blockDim.x) {
            const int q = i / PR, k = i - q * PR;
            const long long pr = map_row(p.rm, u, d0 + q);
            if (pr < 0) {
                if (k == 0) record_status(&p.hdr->status, CSMKV_ERR_ARG);
                continue;
            }
            reinterpret_cast<uint4*>(Kg + pr * D)[k] = reinterpret_cast<const uint4*>(sK)[i];
            reinterpret_cast<uint4*>(Vg + pr * D)[k] = reinterpret_cast<const uint4*>(sV)[i];
        }
        for (int q = tid; q < nrows; q += blockDim.x) {
            const long long pr = map_row(p.rm, u, d0 + q);
            if (pr >= 0) p.N[pr] = sN[q];
        }
    } else {
        uint4* dstK = reinterpret_cast<uint4*>(Kg + (urow + d0) * D);
        uint4* dstV = reinterpret_cast<uint4*>(Vg + (urow + d0) * D);
        for (int i = tid; i < nrows * PR; i += blockDim.x) {
            dstK[i] = reinterpret_cast<const uint4*>(sK)[i];
            dstV[i] = reinterpret_cast<const uint4*>(sV)[i];
        }
        for (int q = tid; q < nrows; q += blockDim.x) p.N[urow + d0 + q] = sN[q];
    }
    return true;
}

// Tensor-core launcher: three CTAs per SM with one slot each (csm_tc3.cu);
// paged: the block-table variant.
int launch_csm_tc3(const CsmParams& P, int D, void* K, void* V, int32_t* N, uint64_t rows, bool paged, cudaStream_t st);

}  // namespace csmkv
