// append.cu -- decode append K=[K,k], V=[V,v], N=[N,1], s=s+1 for every
// (sequence, KV head). [Chelsea §三 算法流程, Algorithm 1 decode update]
// One warp per unit; lanes move 16-byte pieces of the new K and V rows.
#include "host_util.h"
#include "ptx.cuh"

namespace csmkv {

struct AppendParams {
    uint8_t* K;
    uint8_t* V;
    int32_t* N;
    int32_t* len;
    const uint8_t* k_new;
    const uint8_t* v_new;
    const uint8_t* seq_mask;
    int32_t* status;
    RowMap rm;                 // logical row -> pool row (dense, or through a block table)
    int32_t BH, Hkv, cap, RB;  // RB = row bytes
};

__global__ void __launch_bounds__(256) append_kernel(const AppendParams p) {
    const int u = blockIdx.x * 8 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (u >= p.BH) return;
    if (p.seq_mask && !p.seq_mask[u / p.Hkv]) return;
    const int s = p.len[u];
    __syncwarp();
    if (s < 0 || s >= p.cap) {
        if (lane == 0) record_status(p.status, CSMKV_ERR_CAPACITY);
        return;
    }
    const int pieces = p.RB / 16;
    const long long prow = map_row(p.rm, u, s);
    if (prow < 0) {  // a block-table entry outside the pool: nothing is written
        if (lane == 0) record_status(p.status, CSMKV_ERR_ARG);
        return;
    }
    const size_t row = (size_t)prow;
    for (int i = lane; i < pieces; i += 32) {
        reinterpret_cast<uint4*>(p.K + row * p.RB)[i] = reinterpret_cast<const uint4*>(p.k_new + (size_t)u * p.RB)[i];
        reinterpret_cast<uint4*>(p.V + row * p.RB)[i] = reinterpret_cast<const uint4*>(p.v_new + (size_t)u * p.RB)[i];
    }
    if (lane == 0) {
        p.N[row] = 1;
        p.len[u] = s + 1;
    }
}

}  // namespace csmkv

using namespace csmkv;

extern "C" size_t csm_append_workspace_bytes(void) { return kHeaderBytes; }

static int append_impl(void* K, void* V, int32_t* N, int32_t* len, const csmkv_cache* cache, const csmkv_pages* pages,
                       const void* k_new, const void* v_new, const uint8_t* seq_mask, void* workspace, size_t ws_bytes,
                       void* stream) {
    int rc = check_cache(cache);
    if (rc != CSMKV_OK) return rc;
    if (pages) {
        rc = check_pages(cache, pages);
        if (rc != CSMKV_OK) return rc;
    }
    if (!K || !V || !N || !len || !k_new || !v_new) return CSMKV_ERR_ARG;
    if (!aligned16(K) || !aligned16(V) || !aligned16(k_new) || !aligned16(v_new) ||
        (reinterpret_cast<uintptr_t>(N) & 3u) || (reinterpret_cast<uintptr_t>(len) & 3u))
        return CSMKV_ERR_ALIGN;
    if (!workspace || ws_bytes < kHeaderBytes) return CSMKV_ERR_WORKSPACE;
    AppendParams P{};
    P.K = static_cast<uint8_t*>(K);
    P.V = static_cast<uint8_t*>(V);
    P.N = N;
    P.len = len;
    P.k_new = static_cast<const uint8_t*>(k_new);
    P.v_new = static_cast<const uint8_t*>(v_new);
    P.seq_mask = seq_mask;
    P.status = reinterpret_cast<int32_t*>(workspace);
    P.BH = cache->batch * cache->h_kv;
    P.Hkv = cache->h_kv;
    P.cap = cache->cap;
    P.rm = row_map(cache, pages);
    P.RB = cache->head_dim * (int)dtype_bytes(cache->dtype);
    append_kernel<<<(P.BH + 7) / 8, 256, 0, static_cast<cudaStream_t>(stream)>>>(P);
    return cudaGetLastError() == cudaSuccess ? CSMKV_OK : CSMKV_ERR_CUDA;
}

extern "C" int csm_append(void* K, void* V, int32_t* N, int32_t* len, const csmkv_cache* cache, const void* k_new,
                          const void* v_new, const uint8_t* seq_mask, void* workspace, size_t ws_bytes,
                          void* stream) {
    return append_impl(K, V, N, len, cache, nullptr, k_new, v_new, seq_mask, workspace, ws_bytes, stream);
}

extern "C" int csm_append_paged(void* K, void* V, int32_t* N, int32_t* len, const csmkv_cache* cache,
                                const csmkv_pages* pages, const void* k_new, const void* v_new,
                                const uint8_t* seq_mask, void* workspace, size_t ws_bytes, void* stream) {
    if (!pages) return CSMKV_ERR_ARG;
    return append_impl(K, V, N, len, cache, pages, k_new, v_new, seq_mask, workspace, ws_bytes, stream);
}
