// csm_common.cuh -- parts of one Chunked Soft Matching round shared by the
// tensor-core kernel (csm_tc.cu) and the CUDA-core kernel (csm_compress.cu):
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
    int32_t BH, h_kv, cap, D, n1, n2, c, m, maxch, L;
    int64_t timeout_ns;
    int32_t withhold;
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

// Shared-memory tables of one chunk's decisions.
struct CsmTables {
    float inv[256];       // inverse key norm per chunk row
    float best[512];      // per-group best similarity, then final per A row
    int32_t bestb[512];   // per-group argmax, then final per A row
    int32_t match[128];   // B index for selected A rows, else -1
    int32_t cnt[128];     // incoming edges per B row
    int32_t off[128];     // CSR offsets per B row
    int32_t nsum[128];    // merged degree per B row
    float ninv[128];      // 1 / nsum
    int32_t pre[132];     // selected A rows before index a (pre[H] = m)
    int16_t src[256];     // output row -> chunk row
    uint8_t list[128];    // CSR member list (A indices)
    int32_t misc[8];      // [3..6] warp selection counts
};

// Non-empty work item at or after a ticket, or INT_MAX. Thread 0 only.
__device__ __forceinline__ int claim_item(const CsmParams& p, int levels_ch, long long total) {
    for (;;) {
        int t = atomicAdd(&p.hdr->ticket, 1);
        if (t >= total || ld_volatile(&p.hdr->status) != 0) return INT_MAX;
        const int lev = t / p.BH, u = t - lev * p.BH;
        if (lev < levels_ch ? lev < p.unit_ch[u] : (lev - levels_ch) < p.unit_tp[u]) return t;
    }
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
// selected A rows (similarity desc, A index asc), the output row -> chunk row
// map, and the CSR list of A rows merging into every B row. All threads call.
// With H = 128 and 256 or 512 threads, R = blockDim / 128 consecutive threads
// share one A row's rank count and list position.
__device__ inline void chunk_tables(CsmTables& sm, const int32_t* sN, int c, int m, int ngroups) {
    const int H = c / 2;
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
        sm.bestb[tid] = bb;
        sm.cnt[tid] = 0;
    }
    __syncthreads();
    if (ra < H) {  // rank of A row ra among all A rows, counted over R parts
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
            sm.match[ra] = sel ? sm.bestb[ra] : -1;
            if (sel) atomicAdd(&sm.cnt[sm.bestb[ra]], 1);
        }
    }
    __syncthreads();
    const bool sel = tid < H && sm.match[tid] >= 0;
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
    for (int q = tid; q < c; q += blockDim.x) {
        if ((q & 1) == 0) {
            if (sm.match[q >> 1] < 0) sm.src[q - sm.pre[q >> 1]] = (int16_t)q;
        } else {
            sm.src[q - sm.pre[(q >> 1) + 1]] = (int16_t)q;
        }
    }
    if (ra < H) {  // position of a selected A row in its target's list: earlier A rows with the same target
        const int b = sm.match[ra];
        int r = 0;
        if (b >= 0) {
            const int a0 = rp * span, a1 = min(a0 + span, ra);
            for (int a2 = a0; a2 < a1; ++a2) r += (sm.match[a2] == b);
        }
        for (int o = 1; o < R; o <<= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
        if (b >= 0 && rp == 0) sm.list[sm.off[b] + r] = (uint8_t)ra;
    }
    __syncthreads();
    if (tid < H) {
        int ns = sN[2 * tid + 1];
        const int o0 = sm.off[tid], o1 = o0 + sm.cnt[tid];
        for (int k = o0; k < o1; ++k) ns += sN[2 * (int)sm.list[k]];
        sm.nsum[tid] = ns;
        sm.ninv[tid] = 1.0f / (float)ns;
    }
    __syncthreads();
}

// Writes the c - m output rows of one array of a chunk: copies, or degree-
// weighted means for B rows with incoming edges (fp32 sums scaled by the reciprocal
// of the degree sum, rounded once to the cache dtype).
// piece(q, cc) gives the 16-byte piece cc of chunk row q in shared memory.
template <typename T, typename PieceFn>
__device__ __forceinline__ void emit_rows(T* dst_rows, int rows_out, int D, const CsmTables& sm,
                                          const int32_t* sN, PieceFn piece) {
    using E = Elem<T>;
    constexpr int EPP = E::kPer;
    const int PR = D * (int)sizeof(T) / 16;
    const int npieces = rows_out * PR;
    for (int i = threadIdx.x; i < npieces; i += blockDim.x) {
        const int pr = i / PR, cc = i - pr * PR;
        const int q = sm.src[pr];
        uint4 val;
        if ((q & 1) && sm.cnt[q >> 1] > 0) {
            const int b = q >> 1;
            float acc[EPP], f[EPP];
            E::unpack(*reinterpret_cast<const uint4*>(piece(q, cc)), f);
            const float nb = (float)sN[q];
#pragma unroll
            for (int e = 0; e < EPP; ++e) acc[e] = nb * f[e];
            const int o0 = sm.off[b], o1 = o0 + sm.cnt[b];
            for (int k = o0; k < o1; ++k) {
                const int qa = 2 * (int)sm.list[k];
                E::unpack(*reinterpret_cast<const uint4*>(piece(qa, cc)), f);
                const float na = (float)sN[qa];
#pragma unroll
                for (int e = 0; e < EPP; ++e) acc[e] = fmaf(na, f[e], acc[e]);
            }
            const float inv = sm.ninv[b];  // one reciprocal per merged row
#pragma unroll
            for (int e = 0; e < EPP; ++e) acc[e] *= inv;
            val = E::pack(acc);
        } else {
            val = *reinterpret_cast<const uint4*>(piece(q, cc));
        }
        *reinterpret_cast<uint4*>(dst_rows + (size_t)pr * D + cc * EPP) = val;
    }
}

__device__ __forceinline__ void emit_degrees(int32_t* dstN, int rows_out, const CsmTables& sm, const int32_t* sN) {
    for (int pr = threadIdx.x; pr < rows_out; pr += blockDim.x) {
        const int q = sm.src[pr];
        dstN[pr] = ((q & 1) && sm.cnt[q >> 1] > 0) ? sm.nsum[q >> 1] : sN[q];
    }
}

// Chunks whose source rows the destination of chunk j overlaps (earlier than j).
__device__ __forceinline__ void chunk_deps(int j, int c, int m, int& lo, int& hi) {
    lo = (j * (c - m)) / c;
    hi = min(((j + 1) * (c - m) - 1) / c, j - 1);
}

// One tail piece: up to 64 rows of the remainder + recent window moved down by
// ch*m rows, staged through `stage` (>= 2 * 64 * row bytes), degrees through sN.
template <typename T>
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
    {
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
    uint4* dstK = reinterpret_cast<uint4*>(Kg + (urow + d0) * D);
    uint4* dstV = reinterpret_cast<uint4*>(Vg + (urow + d0) * D);
    for (int i = tid; i < nrows * PR; i += blockDim.x) {
        dstK[i] = reinterpret_cast<const uint4*>(sK)[i];
        dstV[i] = reinterpret_cast<const uint4*>(sV)[i];
    }
    for (int q = tid; q < nrows; q += blockDim.x) p.N[urow + d0 + q] = sN[q];
    return true;
}

// Tensor-core path launcher (csm_tc.cu).
int launch_csm_tc(const CsmParams& P, int D, void* K, void* V, int32_t* N, uint64_t rows, cudaStream_t st);

}  // namespace csmkv
