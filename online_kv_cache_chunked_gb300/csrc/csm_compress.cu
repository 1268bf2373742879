// csm_compress.cu -- one Chunked Soft Matching round on every (sequence, KV head)
// of a cache, compacted in place: the C entry points, the per-call prologue,
// the choice of kernel, and the CUDA-core kernel (fp32 caches and the shapes the
// tensor-core kernel in csm_tc3.cu, the default, does not cover). [Chelsea §三 分块软匹配算法 steps 1-4;
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
#include "csm_common.cuh"

namespace csmkv {

// ----------------------------------------------------------------------------
// Prologue: snapshot lengths, count the items of every unit, advance the epoch.
__global__ void __launch_bounds__(1024) csm_prologue_kernel(const CsmParams p) {
    griddep_launch_dependents();  // the main kernel may set itself up meanwhile
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
            if (p.seq_limit) {  // budget-exact: only the oldest chunks; the rest moves as tail
                const int lim = p.seq_limit[u / p.h_kv];
                if (lim > 0 && lim < ch) ch = lim;
            }
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
// CUDA-core kernel: chunk rows staged in shared memory with a 16-byte row pad,
// fp32 dot products; K first, then V through the same buffer.
__host__ __device__ constexpr int csm_stage_bytes_simt(int c, int RB) {
    return (c * (RB + 16)) > (2 * kTailRows * RB) ? (c * (RB + 16)) : (2 * kTailRows * RB);
}

template <typename T>
__global__ void __launch_bounds__(kCsmThreads, 1) csm_simt_kernel(const CsmParams p) {
    using E = Elem<T>;
    constexpr int EPP = E::kPer;
    const int D = p.D, RB = D * (int)sizeof(T), PR = RB / 16;
    const int c = p.c, H = c / 2, m = p.m;
    const int tid = threadIdx.x;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* const stage =
        reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    CsmTables& sm = *reinterpret_cast<CsmTables*>(stage + csm_stage_bytes_simt(c, RB));
    int32_t* const sN = reinterpret_cast<int32_t*>(&sm + 1);  // [256]
    volatile int* const sTicket = sN + 256;
    auto piece = [&](int q, int cc) { return stage + q * (RB + 16) + cc * 16; };
    T* const Kg = static_cast<T*>(p.K);
    T* const Vg = static_cast<T*>(p.V);
    int32_t* const status = &p.hdr->status;
    const int32_t epoch = p.hdr->epoch;
    const int levels_ch = p.hdr->levels_ch, levels_tail = p.hdr->levels_tail;
    const long long total = (long long)(levels_ch + levels_tail) * p.BH;

    for (;;) {
        if (tid == 0) *sTicket = claim_item(p, levels_ch, total);
        __syncthreads();
        const int t = *sTicket;
        if (t == INT_MAX) break;
        const int lev = t / p.BH, u = t - lev * p.BH;
        if (lev < levels_ch) {
            const int j = lev, ch = p.unit_ch[u], s = p.snap[u];
            const size_t urow = (size_t)u * p.cap;
            const int src_row = p.n1 + j * c, dst_row = p.n1 + j * (c - m);
            int32_t* const fkn = p.flag_kn + (size_t)u * p.L;
            int32_t* const fv = p.flag_v + (size_t)u * p.L;
            auto stage_rows = [&](const T* base) {
                const uint4* src = reinterpret_cast<const uint4*>(base + (urow + src_row) * D);
                for (int i = tid; i < c * PR; i += kCsmThreads) {
                    const int q = i / PR, cc = i - q * PR;
                    *reinterpret_cast<uint4*>(piece(q, cc)) = src[(size_t)q * PR + cc];
                }
            };
            stage_rows(Kg);
            for (int q = tid; q < c; q += kCsmThreads) sN[q] = p.N[urow + src_row + q];
            __syncthreads();
            if (tid == 0) publish(fkn + j, epoch, p.withhold);
            for (int q = tid; q < c; q += kCsmThreads) {
                float ss = 0.f;
                for (int cc = 0; cc < PR; ++cc) {
                    float f[EPP];
                    E::unpack(*reinterpret_cast<const uint4*>(piece(q, cc)), f);
#pragma unroll
                    for (int e = 0; e < EPP; ++e) ss = fmaf(f[e], f[e], ss);
                }
                const float inv = ss > 0.f ? 1.0f / sqrtf(ss) : 0.0f;
                if (q & 1) sm.invB[q >> 1] = inv; else sm.invA[q >> 1] = inv;
            }
            __syncthreads();
            // groups of B columns per A row; a later group wins only if strictly better
            const int ngroups = kCsmThreads / H;
            const int per = (H + ngroups - 1) / ngroups;
            {
                const int a = tid % H, g = tid / H;
                if (g < ngroups) {
                    const int b0 = g * per, b1 = min(H, b0 + per);
                    const float inv_a = sm.invA[a];
                    float best = -INFINITY;
                    int bb = b0;
                    for (int b = b0; b < b1; ++b) {
                        float dot = 0.f;
                        for (int cc = 0; cc < PR; ++cc) {
                            float fa[EPP], fb[EPP];
                            E::unpack(*reinterpret_cast<const uint4*>(piece(2 * a, cc)), fa);
                            E::unpack(*reinterpret_cast<const uint4*>(piece(2 * b + 1, cc)), fb);
#pragma unroll
                            for (int e = 0; e < EPP; ++e) dot = fmaf(fa[e], fb[e], dot);
                        }
                        const float cs = dot * inv_a * sm.invB[b];
                        if (cs > best) { best = cs; bb = b; }
                    }
                    sm.best[g * H + a] = best;
                    sm.bestb[g * H + a] = (uint8_t)bb;
                }
            }
            __syncthreads();
            chunk_tables(sm, sN, c, m, ngroups);
            if (p.match_out && tid < H) p.match_out[((size_t)u * p.maxch + j) * H + tid] = (int32_t)sm.match[tid];
            if (j == 0 && tid == 0) p.len[u] = s - ch * m;
            int lo, hi;
            chunk_deps(j, c, m, lo, hi);
            if (!wait_items(fkn, lo, hi, epoch, globaltimer() + p.timeout_ns)) {
                record_status(status, CSMKV_ERR_TIMEOUT);
                break;
            }
            emit_rows<T>(Kg + (urow + dst_row) * D, c - m, D, m, sm, sN, piece);
            emit_degrees(p.N + urow + dst_row, c - m, m, sm, sN);
            __syncthreads();
            stage_rows(Vg);
            __syncthreads();
            if (tid == 0) publish(fv + j, epoch, p.withhold);
            if (!wait_items(fv, lo, hi, epoch, globaltimer() + p.timeout_ns)) {
                record_status(status, CSMKV_ERR_TIMEOUT);
                break;
            }
            emit_rows<T>(Vg + (urow + dst_row) * D, c - m, D, m, sm, sN, piece);
        } else if (!tail_piece<T>(p, u, lev - levels_ch, epoch, stage, sN)) {
            record_status(status, CSMKV_ERR_TIMEOUT);
            break;
        }
        __syncthreads();
    }
}

// ----------------------------------------------------------------------------
static size_t csm_layout(const csmkv_cache* cache, int32_t n1, int32_t n2, int32_t c, size_t* off_snap,
                         size_t* off_ch, size_t* off_tp, size_t* off_fkn, size_t* off_fv, int32_t* L_out) {
    const size_t BH = (size_t)cache->batch * cache->h_kv;
    const int32_t maxch = csm_max_chunks(cache, n1, n2, c);
    // tail pieces: the remainder and recent window, or (budget-exact rounds) every
    // row after the processed chunks, at most the whole cache
    const int32_t tail = (cache->cap + kTailRows - 1) / kTailRows;
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

static int compress_impl(void* K, void* V, int32_t* N, int32_t* len, const csmkv_cache* cache,
                         const csmkv_pages* pages, int32_t n1, int32_t n2, int32_t c, double r,
                         const uint8_t* head_mask, const uint8_t* seq_mask, int32_t* match_out,
                         const csm_options* opts, void* workspace, size_t ws_bytes, void* stream) {
    int rc = check_cache(cache);
    if (rc != CSMKV_OK) return rc;
    if (pages) {
        rc = check_pages(cache, pages);
        if (rc != CSMKV_OK) return rc;
    }
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
    const int want = pages ? CSM_KERNEL_TC_SPLIT : (opts ? opts->kernel : CSM_KERNEL_AUTO);
    if (want != CSM_KERNEL_AUTO && want != CSM_KERNEL_SIMT && want != CSM_KERNEL_TC_SPLIT) return CSMKV_ERR_ARG;
    const bool tc_shape = cache->dtype == CSMKV_BF16 && c == 256 && (cache->head_dim == 64 || cache->head_dim == 128);
    if (pages && !tc_shape) return CSMKV_ERR_UNSUPPORTED;  // the block-table variant is the tensor-core kernel
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
    P.seq_limit = opts ? opts->seq_max_chunks : nullptr;
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
    P.rm = row_map(cache, pages);
    P.paged_tma = (pages && n1 % 16 == 0) ? 1 : 0;  // 16-row groups then never straddle a page
    P.timeout_ns = (opts && opts->wait_timeout_ns > 0) ? opts->wait_timeout_ns : 2000000000LL;
    P.withhold = opts ? opts->withhold_signals : 0;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    csm_prologue_kernel<<<1, 1024, 0, st>>>(P);
    if (cudaGetLastError() != cudaSuccess) return CSMKV_ERR_CUDA;

    const int D = cache->head_dim;
    const bool tc = cache->dtype == CSMKV_BF16 && c == 256 && (D == 64 || D == 128) && want != CSM_KERNEL_SIMT;
    const uint64_t rows =
        pages ? (uint64_t)pages->num_pages * pages->page_rows : (uint64_t)cache->batch * cache->h_kv * cache->cap;
    if (tc) return launch_csm_tc3(P, D, K, V, N, rows, pages != nullptr, st);
    const int RB = D * (int)dtype_bytes(cache->dtype);
    const int smem = csm_stage_bytes_simt(c, RB) + (int)sizeof(CsmTables) + 257 * 4 + 1024;
    if (smem > 227 * 1024) return CSMKV_ERR_UNSUPPORTED;
    if (cache->dtype == CSMKV_BF16) {
        if (set_kernel_smem((const void*)csm_simt_kernel<__nv_bfloat16>, smem) != CSMKV_OK) return CSMKV_ERR_CUDA;
        csm_simt_kernel<__nv_bfloat16><<<sm_count(), kCsmThreads, smem, st>>>(P);
    } else {
        if (set_kernel_smem((const void*)csm_simt_kernel<float>, smem) != CSMKV_OK) return CSMKV_ERR_CUDA;
        csm_simt_kernel<float><<<sm_count(), kCsmThreads, smem, st>>>(P);
    }
    return cudaGetLastError() == cudaSuccess ? CSMKV_OK : CSMKV_ERR_CUDA;
}

extern "C" int csm_compress_ex(void* K, void* V, int32_t* N, int32_t* len, const csmkv_cache* cache,
                               int32_t n1, int32_t n2, int32_t c, double r, const uint8_t* head_mask,
                               const uint8_t* seq_mask, int32_t* match_out, const csm_options* opts,
                               void* workspace, size_t ws_bytes, void* stream) {
    return compress_impl(K, V, N, len, cache, nullptr, n1, n2, c, r, head_mask, seq_mask, match_out, opts, workspace,
                         ws_bytes, stream);
}

extern "C" int csm_compress_paged(void* K, void* V, int32_t* N, int32_t* len, const csmkv_cache* cache,
                                  const csmkv_pages* pages, int32_t n1, int32_t n2, int32_t c, double r,
                                  const uint8_t* head_mask, const uint8_t* seq_mask, int32_t* match_out,
                                  const csm_options* opts, void* workspace, size_t ws_bytes, void* stream) {
    if (!pages) return CSMKV_ERR_ARG;
    return compress_impl(K, V, N, len, cache, pages, n1, n2, c, r, head_mask, seq_mask, match_out, opts, workspace,
                         ws_bytes, stream);
}

extern "C" int csm_compress(void* K, void* V, int32_t* N, int32_t* len, const csmkv_cache* cache, int32_t n1,
                            int32_t n2, int32_t c, double r, const uint8_t* head_mask, const uint8_t* seq_mask,
                            void* workspace, size_t ws_bytes, void* stream) {
    return csm_compress_ex(K, V, N, len, cache, n1, n2, c, r, head_mask, seq_mask, nullptr, nullptr, workspace,
                           ws_bytes, stream);
}
