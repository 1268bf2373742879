// decode_attn_noalloc.cu -- degree-aware decode attention for callers that cannot
// allocate device memory.
//
// decode_attn_logn needs a workspace (unit offsets, per-unit counters and the
// partial softmax states of the split). Some callers cannot provide one: code
// that runs after a host application has reserved all device memory up front,
// plugins that do not own the CUDA allocator, or deployments whose memory
// budget is fixed before the first request. This entry point keeps that scratch
// in a fixed array in the library's own device memory instead, so the caller
// passes only inputs and outputs.
//
// The array lives as long as the library stays loaded, on every GPU that loads
// it (kNoAllocScratchBytes each). In host code its name is only a stand-in for
// the symbol, not a device address: the address is looked up once per device
// with cudaGetSymbolAddress and cached.
#include <mutex>

#include "host_util.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB per device

static __device__ __align__(256) unsigned char g_attn_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device (looked up on first use).
int scratch_for_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CSMKV_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || p == nullptr) return CSMKV_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return CSMKV_OK;
}

}  // namespace

extern "C" int decode_attn_logn_noalloc(const void* q, const void* K, const void* V, const int32_t* N,
                                        const int32_t* len, const csmkv_cache* cache, int32_t h_q, float scale,
                                        void* out, void* stream) {
    // Every argument check runs before the shared array is touched, so a rejected
    // call leaves it (and any call still running on it) alone.
    int rc = csmkv::decode_attn_check_args(q, K, V, N, len, nullptr, nullptr, cache, h_q, scale, out);
    if (rc != CSMKV_OK) return rc;
    const size_t need = decode_attn_workspace_bytes(cache, h_q);
    if (need == 0) return CSMKV_ERR_CUDA;
    if (need > kNoAllocScratchBytes) return CSMKV_ERR_WORKSPACE;  // batch too large for the fixed scratch
    void* scratch = nullptr;
    rc = scratch_for_current_device(&scratch);
    if (rc != CSMKV_OK) return rc;
    // The previous call's contents stay in the array: start from zero as a new workspace would.
    if (cudaMemsetAsync(scratch, 0, need, static_cast<cudaStream_t>(stream)) != cudaSuccess) return CSMKV_ERR_CUDA;
    return decode_attn_logn(q, K, V, N, len, cache, h_q, scale, out, scratch, kNoAllocScratchBytes, stream);
}
