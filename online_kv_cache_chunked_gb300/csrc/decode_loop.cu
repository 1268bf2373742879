// decode_loop.cu -- the decode phase of the serving loop, issued from native code.
// [Chelsea §三 算法流程, Algorithm 1 (decode phase); CentroidKV 技术摘要: 推理流水线]
//
// Per step: append the new token's k, v (degree 1), attend over the whole
// cache with log-N weights, then run the compression rounds the caller planned
// for that step. Everything is enqueued on one stream without host/device
// synchronisation; the per-step host cost is a few launches, so the GPU runs
// ahead of the host even when a step's attention is a few tens of
// microseconds.
#include <cuda_runtime.h>

#include "host_util.h"

namespace {

// Reads a buffer once, 16 bytes per thread per step, so that its lines replace
// whatever L2 held; nothing is written (an impossible-value check keeps the
// loads alive), so no dirty lines are left for the next kernel to write back.
__global__ void __launch_bounds__(256) l2_evict_kernel(const uint4* buf, size_t n16, unsigned int* sink) {
    unsigned int x = 0;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n16; i += (size_t)gridDim.x * blockDim.x) {
        const uint4 v = __ldcg(buf + i);
        x ^= v.x ^ v.y ^ v.z ^ v.w;
    }
    if (x == 0x9e3779b9u && threadIdx.x == 1023u) *sink = x;  // threadIdx.x < 256: never taken
}

size_t cache_elem_bytes(const csmkv_cache& c) { return c.dtype == CSMKV_BF16 ? 2 : 4; }

int record(void* const* evs, int k, cudaStream_t st) {
    if (!evs) return CSMKV_OK;
    return cudaEventRecord(static_cast<cudaEvent_t>(evs[k]), st) == cudaSuccess ? CSMKV_OK : CSMKV_ERR_CUDA;
}

}  // namespace

extern "C" int csm_decode_run(const csm_decode_loop* L, int32_t first_step, int32_t steps, void* stream) {
    if (!L || first_step < 1 || steps < 0) return CSMKV_ERR_ARG;
    if (steps == 0) return CSMKV_OK;
    if (!L->q || !L->k_new || !L->v_new || !L->out) return CSMKV_ERR_ARG;
    if (L->n_rounds < 0 || (L->n_rounds > 0 && !L->rounds)) return CSMKV_ERR_ARG;
    for (int k = 1; k < L->n_rounds; ++k)
        if (L->rounds[k].step < L->rounds[k - 1].step) return CSMKV_ERR_ARG;
    int rc = csmkv::check_cache(&L->cache);
    if (rc != CSMKV_OK) return rc;
    if ((L->l2_flush == nullptr) != (L->l2_flush_bytes == 0)) return CSMKV_ERR_ARG;
    if (L->l2_flush && (!csmkv::aligned16(L->l2_flush) || L->l2_flush_bytes % 16 != 0)) return CSMKV_ERR_ALIGN;
    const csmkv_pages* const pg = L->pages;  // block-table layout: the paged entry points, fused steps
    if (pg) {
        if (!L->fused_append) return CSMKV_ERR_ARG;
        if ((rc = csmkv::check_pages(&L->cache, pg)) != CSMKV_OK) return rc;
    }

    const csmkv_cache& C = L->cache;
    const size_t eb = cache_elem_bytes(C);
    const size_t kv_step = (size_t)C.batch * C.h_kv * C.head_dim * eb;  // one step of k_new / v_new
    const size_t q_step = (size_t)C.batch * L->h_q * C.head_dim * eb;   // one step of q / out
    const cudaStream_t st = static_cast<cudaStream_t>(stream);
    csm_options opts{};
    opts.kernel = L->csm_kernel;

    int ri = 0;
    while (ri < L->n_rounds && L->rounds[ri].step < first_step) ++ri;
    int attn_k = 0, csm_k = 0;
    for (int i = first_step; i < first_step + steps; ++i) {
        const size_t s = (size_t)(i - 1);
        const uint8_t* const kn = static_cast<const uint8_t*>(L->k_new) + s * kv_step;
        const uint8_t* const vn = static_cast<const uint8_t*>(L->v_new) + s * kv_step;
        if (!L->fused_append) {
            rc = csm_append(L->K, L->V, L->N, L->len, &C, kn, vn, nullptr, L->ws_append, L->ws_append_bytes, stream);
            if (rc != CSMKV_OK) return rc;
        }
        if (L->l2_flush) {
            l2_evict_kernel<<<4 * csmkv::sm_count(), 256, 0, st>>>(static_cast<const uint4*>(L->l2_flush),
                                                                   L->l2_flush_bytes / 16,
                                                                   static_cast<unsigned int*>(L->l2_flush));
            if (cudaGetLastError() != cudaSuccess) return CSMKV_ERR_CUDA;
        }
        if ((rc = record(L->attn_events, 2 * attn_k, st)) != CSMKV_OK) return rc;
        const uint8_t* const qs = static_cast<const uint8_t*>(L->q) + s * q_step;
        uint8_t* const os = static_cast<uint8_t*>(L->out) + s * q_step;
        if (pg)
            rc = decode_step_logn_paged(qs, kn, vn, L->K, L->V, L->N, L->len, &C, pg, L->h_q, L->scale, os,
                                        L->ws_attn, L->ws_attn_bytes, stream);
        else
            rc = L->fused_append
                     ? decode_step_logn(qs, kn, vn, L->K, L->V, L->N, L->len, &C, L->h_q, L->scale, os, L->ws_attn,
                                        L->ws_attn_bytes, stream)
                     : decode_attn_logn(qs, L->K, L->V, L->N, L->len, &C, L->h_q, L->scale, os, L->ws_attn,
                                        L->ws_attn_bytes, stream);
        if (rc != CSMKV_OK) return rc;
        if ((rc = record(L->attn_events, 2 * attn_k + 1, st)) != CSMKV_OK) return rc;
        ++attn_k;
        for (; ri < L->n_rounds && L->rounds[ri].step == i; ++ri) {
            const csm_round_plan& R = L->rounds[ri];
            if ((rc = record(L->csm_events, 2 * csm_k, st)) != CSMKV_OK) return rc;
            opts.seq_max_chunks = R.seq_max_chunks;
            rc = pg ? csm_compress_paged(L->K, L->V, L->N, L->len, &C, pg, L->n1, L->n2, L->c, R.r, L->head_mask,
                                         R.seq_mask, nullptr, &opts, L->ws_csm, L->ws_csm_bytes, stream)
                    : csm_compress_ex(L->K, L->V, L->N, L->len, &C, L->n1, L->n2, L->c, R.r, L->head_mask, R.seq_mask,
                                      nullptr, &opts, L->ws_csm, L->ws_csm_bytes, stream);
            if (rc != CSMKV_OK) return rc;
            if ((rc = record(L->csm_events, 2 * csm_k + 1, st)) != CSMKV_OK) return rc;
            ++csm_k;
        }
    }
    return CSMKV_OK;
}
