// host_util.h -- host-side helpers shared by the library's translation units:
// tensor-map encoding (driver entry point fetched through the runtime, so the
// library needs no -lcuda), per-device SM count, and argument checks.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <utility>

#include "../../include/csmkv.h"

namespace csmkv {

// Launches a kernel that may overlap its setup with the tail of the previous
// kernel in the stream (programmatic dependent launch); the kernel must call
// griddep_wait() before it touches memory that earlier work writes.
template <typename... ExpTypes, typename... ActTypes>
inline cudaError_t launch_overlapped(void (*kern)(ExpTypes...), dim3 grid, dim3 block, size_t smem,
                                     cudaStream_t st, ActTypes&&... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<ActTypes>(args)...);
}

constexpr size_t kHeaderBytes = 256;  // every workspace starts with this header

// Layout of the workspace header (offset 0). Only `status` is part of the public contract.
struct WsHeader {
    int32_t status;       // first device-side error (csmkv_status), sticky
    int32_t ticket;       // work-ticket counter of the current call
    int32_t epoch;        // call sequence number; flags equal to it are "set"
    int32_t levels_ch;    // CSM: max full chunks over active units
    int32_t levels_tail;  // CSM: max tail pieces over active units
    int32_t dec_nsplits;  // decode (prologue path): token splits of the call
    int32_t dec_split;    // decode (prologue path): base split length in tokens
    int32_t ctas_done;    // decode: CTAs finished; the last one resets the ticket (and bumps lengths)
    int32_t dec_total;    // decode (prologue path): rows attended over all units
    int32_t pad[55];
};
static_assert(sizeof(WsHeader) == kHeaderBytes, "header size");

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline size_t dtype_bytes(int32_t dt) { return dt == CSMKV_BF16 ? 2 : (dt == CSMKV_F32 ? 4 : 0); }

// Validates the cache descriptor itself; returns CSMKV_OK or the error.
inline int check_cache(const csmkv_cache* c) {
    if (!c) return CSMKV_ERR_ARG;
    if (c->dtype != CSMKV_BF16 && c->dtype != CSMKV_F32) return CSMKV_ERR_DTYPE;
    if (c->batch < 1 || c->h_kv < 1 || c->cap < 8 || (c->cap % 8) != 0) return CSMKV_ERR_ARG;
    if (c->head_dim < 8 || c->head_dim > 128 || (c->head_dim % 8) != 0) return CSMKV_ERR_ARG;
    const long long rows = (long long)c->batch * c->h_kv * c->cap;
    if (rows > 0x7FFFFFFFLL) return CSMKV_ERR_ARG;  // row coordinates are int32
    return CSMKV_OK;
}

// Validates a paged layout against the logical cache descriptor.
inline int check_pages(const csmkv_cache* c, const csmkv_pages* pg) {
    if (!pg || !pg->table) return CSMKV_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(pg->table) & 3u) return CSMKV_ERR_ALIGN;
    if (pg->page_rows < 64 || (pg->page_rows % 64) != 0 || pg->max_pages < 1 || pg->num_pages < 1)
        return CSMKV_ERR_ARG;
    if ((long long)pg->max_pages * pg->page_rows != c->cap) return CSMKV_ERR_ARG;
    if ((long long)pg->num_pages * pg->page_rows > 0x7FFFFFFFLL) return CSMKV_ERR_ARG;  // pool rows are int32
    return CSMKV_OK;
}

// Logical row -> pool row of a cache: unit-major dense rows (table == nullptr),
// or a paged layout's block table. Plain data, passed to kernels by value.
struct RowMap {
    const int32_t* table;
    int32_t P, maxp, npages, cap;
};

inline RowMap row_map(const csmkv_cache* c, const csmkv_pages* pg) {
    RowMap m{};
    m.cap = c->cap;
    if (pg) {
        m.table = pg->table;
        m.P = pg->page_rows;
        m.maxp = pg->max_pages;
        m.npages = pg->num_pages;
    }
    return m;
}

int sm_count();                 // SMs of the current device (cached per device)
// Raises a kernel's dynamic shared-memory limit on the current device (and, if
// asked, prefers the largest shared-memory carveout). The setting is remembered
// per (device, kernel), so repeated launches cost no runtime call.
int set_kernel_smem(const void* fn, int bytes, bool max_carveout = false);
const void* encode_fn();        // cuTensorMapEncodeTiled, or nullptr

// Argument checks of decode attention (everything but the workspace): the
// status decode_attn_logn / decode_step_logn would return before launching.
int decode_attn_check_args(const void* q, const void* K, const void* V, const int32_t* N, const int32_t* len,
                           const void* k_new, const void* v_new, const csmkv_cache* cache, int32_t h_q, float scale,
                           const void* out);

// Encodes a tiled tensor map; returns false on failure.
bool encode_tiled(CUtensorMap* map, CUtensorMapDataType dt, uint32_t rank, void* base, const uint64_t* dims,
                  const uint64_t* strides_bytes /* rank-1 entries */, const uint32_t* box,
                  CUtensorMapSwizzle swizzle);

}  // namespace csmkv
