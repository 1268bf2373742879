// host.cpp -- host-only parts of the C ABI: schedule helpers, status words,
// status strings, tensor-map encoding and device queries.
#include <cmath>
#include <cstdio>
#include <mutex>

#include "host_util.h"

namespace csmkv {

int sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev] = n;
    }
    return cache[dev];
}

namespace {
struct SmemSetting {
    int dev;
    const void* fn;
    int bytes;
};
std::mutex g_smem_mu;
SmemSetting g_smem[256];
int g_smem_n = 0;
}  // namespace

int set_kernel_smem(const void* fn, int bytes, bool max_carveout) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CSMKV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_smem_mu);
    int k = 0;
    while (k < g_smem_n && !(g_smem[k].dev == dev && g_smem[k].fn == fn)) ++k;
    if (k < g_smem_n && g_smem[k].bytes >= bytes) return CSMKV_OK;
    if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
        return CSMKV_ERR_CUDA;
    if (max_carveout && cudaFuncSetAttribute(fn, cudaFuncAttributePreferredSharedMemoryCarveout, 100) != cudaSuccess)
        return CSMKV_ERR_CUDA;
    if (k < g_smem_n) {
        g_smem[k].bytes = bytes;
    } else if (g_smem_n < 256) {  // a full table only means the attribute is set again on later calls
        g_smem[g_smem_n++] = SmemSetting{dev, fn, bytes};
    }
    return CSMKV_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

const void* encode_fn() {
    static void* fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = p;
    });
    return fn;
}

bool encode_tiled(CUtensorMap* map, CUtensorMapDataType dt, uint32_t rank, void* base, const uint64_t* dims,
                  const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swizzle) {
    auto fn = reinterpret_cast<EncodeTiledFn>(const_cast<void*>(encode_fn()));
    if (!fn) return false;
    cuuint64_t d[5], s[4];
    cuuint32_t b[5], e[5];
    for (uint32_t i = 0; i < rank; ++i) {
        d[i] = dims[i];
        b[i] = box[i];
        e[i] = 1;
        if (i + 1 < rank) s[i] = strides_bytes[i];
    }
    CUresult r = fn(map, dt, rank, base, d, s, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace csmkv

extern "C" {

double csm_budget(int64_t n, double R, int64_t Gamma) { return R * ((double)n + (double)Gamma); }

int csm_should_trigger(int64_t s, double B, int32_t g) { return (double)s >= B + (double)g ? 1 : 0; }

double csm_ratio(int32_t j, double r_init, double dr, double r_min) {
    const double r = r_init - (double)j * dr;
    return r > r_min ? r : r_min;
}

int32_t csm_edges_per_chunk(double r, int32_t c) { return (int32_t)std::floor(r * (double)c + 1e-9); }

int64_t csm_num_chunks(int64_t s, int32_t n1, int32_t n2, int32_t c) {
    if (c <= 0) return 0;
    const int64_t mid = s - n1 - n2;
    return mid > 0 ? mid / c : 0;
}

int64_t csm_len_after(int64_t s, int32_t n1, int32_t n2, int32_t c, int32_t m) {
    return s - csm_num_chunks(s, n1, n2, c) * (int64_t)m;
}

int32_t csm_chunks_to_budget(int64_t s, double B, int32_t n1, int32_t n2, int32_t c, int32_t m) {
    if (m <= 0 || !((double)s > B)) return 0;
    const double need = std::ceil(((double)s - B) / (double)m);
    const int64_t have = csm_num_chunks(s, n1, n2, c);
    return (int32_t)(need < (double)have ? (int64_t)need : have);
}

int csmkv_device_status(const void* workspace, void* stream) {
    if (!workspace) return CSMKV_ERR_WORKSPACE;
    int32_t v = 0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess) return CSMKV_ERR_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return CSMKV_ERR_CUDA;
    return v;
}

int csmkv_clear_status(void* workspace, void* stream) {
    if (!workspace) return CSMKV_ERR_WORKSPACE;
    if (cudaMemsetAsync(workspace, 0, sizeof(int32_t), static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return CSMKV_ERR_CUDA;
    return CSMKV_OK;
}

const char* csmkv_status_str(int status) {
    switch (status) {
        case CSMKV_OK: return "ok";
        case CSMKV_ERR_ARG: return "argument out of range";
        case CSMKV_ERR_DTYPE: return "unknown dtype";
        case CSMKV_ERR_ALIGN: return "pointer or size misaligned";
        case CSMKV_ERR_CAPACITY: return "cache full (len == cap) on append";
        case CSMKV_ERR_WORKSPACE: return "workspace missing or too small";
        case CSMKV_ERR_TIMEOUT: return "a bounded device wait ran out";
        case CSMKV_ERR_CUDA: return "CUDA runtime error";
        case CSMKV_ERR_UNSUPPORTED: return "shape not covered by a kernel";
        default: return "unknown status";
    }
}

}  // extern "C"
