// csm_tc.cu -- Chunked Soft Matching on the tensor cores (bf16, c = 256,
// d in {64, 128}). [Chelsea §三 分块软匹配算法 steps 1-4; CentroidKV 分块软匹配 (CSM), 聚合]
//
// One persistent CTA per SM walks work tickets (level-major: chunk j of every
// unit, then the tail pieces) through a ring of three 64 KB shared-memory slots
// filled by TMA. While chunk i is decided and written, the slots hold K(i),
// V(i) and K(i+1); when K(i)'s slot frees, V(i+1) is loaded into it, and when
// V(i)'s slot frees, K(i+2) is. Degrees come with K through a second tensor
// map. Each slot is a [A rows | B rows] x [64-column boxes] x 128 rows x 128 B
// layout with the 128-byte swizzle: the A rows (even chunk offsets) and B rows
// (odd offsets) land as two K-major MMA operands.
//
// Per chunk: fp32 inverse key norms; one thread issues d/16 tcgen05.mma
// (M = N = 128, fp32 accumulate in 128 TMEM columns) for the 128 x 128 dot
// products; sixteen warps read them back with tcgen05.ld, scale by the norms and
// take the per-A argmax; then the shared top-m selection, merge and compaction.
// The "loaded" flag of an item is published as soon as its slot's TMA lands, so
// items that overwrite its source rows wait as little as possible.
#include "csm_common.cuh"

namespace csmkv {

template <int D>
struct TcRing {
    static constexpr int kBoxes = D / 64;
    static constexpr int kSlotBytes = 2 * kBoxes * 16384;  // A and B rows of one chunk of one array
    static constexpr int kSlots = 3;
    static constexpr int kNRows = 65;                      // degree tile: 65 x 4 int32 covers 256 rows
    static constexpr int kNBytes = kNRows * 16;
    static constexpr int kNStride = 1152;                  // per-slot degree buffer
    static constexpr int kSmem = kSlots * kSlotBytes + kSlots * kNStride + (int)sizeof(CsmTables) + 64 + 1024;
};

constexpr int kTcThreads = 512;  // 16 warps: 4 TMEM lane quarters x 4 column groups

struct TcState {
    uint64_t bar[3];  // one per ring slot
    uint64_t mma_bar;
    int32_t tk[3];    // tickets: current item, next, the one after
    uint32_t tmem;
};

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    csm_tc_kernel(const __grid_constant__ CsmParams p, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmN) {
    using R = TcRing<D>;
    using T = __nv_bfloat16;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* const ring =
        reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* const nbuf = ring + R::kSlots * R::kSlotBytes;
    CsmTables& sm = *reinterpret_cast<CsmTables*>(nbuf + R::kSlots * R::kNStride);
    TcState& st = *reinterpret_cast<TcState*>(&sm + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = p.c, m = p.m, BH = p.BH;
    T* const Kg = static_cast<T*>(p.K);
    T* const Vg = static_cast<T*>(p.V);
    int32_t* const status = &p.hdr->status;

    if (tid == 0) {
        for (int s = 0; s < R::kSlots; ++s) mbar_init(&st.bar[s], 1);
        mbar_init(&st.mma_bar, 1);
        fence_mbar_init();
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        prefetch_tmap(&tmN);
    }
    if (warp == 0) {
        tmem_alloc(&st.tmem, 128);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = st.tmem;

    const int32_t epoch = p.hdr->epoch;
    const int levels_ch = p.hdr->levels_ch, levels_tail = p.hdr->levels_tail;
    const long long total = (long long)(levels_ch + levels_tail) * BH;

    uint32_t phase_bits = 0u;  // bit s: next phase of slot s to complete (all threads agree)
    uint32_t mma_phase = 0;
    uint32_t pend_bits = 0u;   // thread 0, bit s: slot s has a load in flight
    bool mma_pend = false;

    auto is_chunk = [&](int t) { return t != INT_MAX && t / BH < levels_ch; };
    auto chunk_row0 = [&](int t) {  // global row of a chunk ticket's first row
        const int j = t / BH, u = t - j * BH;
        return (long long)u * p.cap + p.n1 + (long long)j * c;
    };
    auto issue_k = [&](int t, int slot) {  // thread 0: K and degrees of chunk t
        const long long g0 = chunk_row0(t);
        uint8_t* dst = ring + slot * R::kSlotBytes;
        mbar_expect_tx(&st.bar[slot], (uint32_t)(R::kSlotBytes + R::kNBytes));
        const int ya = (int)(g0 & 1), za = (int)(g0 >> 1);
        const int yb = (int)((g0 + 1) & 1), zb = (int)((g0 + 1) >> 1);
#pragma unroll
        for (int bx = 0; bx < R::kBoxes; ++bx) {
            tma_load_3d(dst + bx * 16384, &tmK, &st.bar[slot], bx * 64, ya, za);
            tma_load_3d(dst + (R::kBoxes + bx) * 16384, &tmK, &st.bar[slot], bx * 64, yb, zb);
        }
        tma_load_2d(nbuf + slot * R::kNStride, &tmN, &st.bar[slot], 0, (int)(g0 >> 2));
        pend_bits |= 1u << slot;
    };
    auto issue_v = [&](int t, int slot) {  // thread 0: V of chunk t
        const long long g0 = chunk_row0(t);
        uint8_t* dst = ring + slot * R::kSlotBytes;
        mbar_expect_tx(&st.bar[slot], (uint32_t)R::kSlotBytes);
        const int ya = (int)(g0 & 1), za = (int)(g0 >> 1);
        const int yb = (int)((g0 + 1) & 1), zb = (int)((g0 + 1) >> 1);
#pragma unroll
        for (int bx = 0; bx < R::kBoxes; ++bx) {
            tma_load_3d(dst + bx * 16384, &tmV, &st.bar[slot], bx * 64, ya, za);
            tma_load_3d(dst + (R::kBoxes + bx) * 16384, &tmV, &st.bar[slot], bx * 64, yb, zb);
        }
        pend_bits |= 1u << slot;
    };
    // Thread 0: publish a prefetched item's flag as soon as its slot has landed.
    auto poll_publish = [&](int t, int slot, int32_t* flags_base, bool& done) {
        if (done || !is_chunk(t) || !((pend_bits >> slot) & 1u)) return;
        if (mbar_try_wait(&st.bar[slot], ((phase_bits >> slot) & 1u))) {
            const int j = t / BH, u = t - j * BH;
            publish(flags_base + (size_t)u * p.L + j, epoch, p.withhold);
            done = true;
        }
    };

    if (tid == 0) {
        const int t0 = claim_item(p, levels_ch, total);
        const int t1 = claim_item(p, levels_ch, total);
        if (is_chunk(t0)) {
            issue_k(t0, 0);
            issue_v(t0, 1);
        }
        if (is_chunk(t1)) issue_k(t1, 2);
        st.tk[0] = t0;
        st.tk[1] = t1;
    }
    __syncthreads();
    int kslot = 0, vslot = 1, nkslot = 2;
    bool kn_next_done = false, v_next_done = false;  // thread 0: early publication of the next item

    for (;;) {
        const int t = st.tk[0], tn = st.tk[1];
        if (t == INT_MAX) break;
        const int lev = t / BH, u = t - lev * BH;
        const bool kn_done_now = kn_next_done, v_done_now = v_next_done;
        kn_next_done = v_next_done = false;
        bool ok = true;

        if (lev < levels_ch) {
            // ================================================================ chunk item
            const int j = lev;
            const int ch = p.unit_ch[u];
            const int s = p.snap[u];
            const size_t urow = (size_t)u * p.cap;
            const int dst_row = p.n1 + j * (c - m);
            const long long g0 = (long long)urow + p.n1 + (long long)j * c;
            uint8_t* const kb = ring + kslot * R::kSlotBytes;
            uint8_t* const vb = ring + vslot * R::kSlotBytes;
            const int32_t* const sN = reinterpret_cast<const int32_t*>(nbuf + kslot * R::kNStride) + (int)(g0 & 3);
            int32_t* const fkn = p.flag_kn + (size_t)u * p.L;
            int32_t* const fv = p.flag_v + (size_t)u * p.L;
            auto kpiece = [&](int q, int cc) {
                return kb + ((q & 1) * R::kBoxes + (cc >> 3)) * 16384 + sw128_off((uint32_t)(q >> 1), (uint32_t)(cc & 7));
            };
            auto vpiece = [&](int q, int cc) {
                return vb + ((q & 1) * R::kBoxes + (cc >> 3)) * 16384 + sw128_off((uint32_t)(q >> 1), (uint32_t)(cc & 7));
            };

            // (1) K and degrees on chip
            ok = mbar_wait(&st.bar[kslot], ((phase_bits >> kslot) & 1u), globaltimer() + p.timeout_ns);
            phase_bits ^= 1u << kslot;
            if (!__syncthreads_and(ok)) { record_status(status, CSMKV_ERR_TIMEOUT); break; }
            if (tid == 0) {
                pend_bits &= ~(1u << kslot);
                if (!kn_done_now) publish(fkn + j, epoch, p.withhold);
            }

            // (2) inverse key norms, two threads per chunk row (c = 256 rows, 512 threads)
            {
                const int q = tid >> 1, h = tid & 1;
                float ss = 0.f;
#pragma unroll
                for (int i = 0; i < D / 16; ++i) {
                    float f[8];
                    Elem<T>::unpack(*reinterpret_cast<const uint4*>(kpiece(q, h * (D / 16) + i)), f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
                }
                ss += __shfl_xor_sync(0xffffffffu, ss, 1);
                if (h == 0) sm.inv[q] = ss > 0.f ? 1.0f / sqrtf(ss) : 0.0f;
            }
            __syncthreads();

            // (3) 128 x 128 dot products on the tensor cores, read back by 8 warps
            if (tid == 0) {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const int box = ks >> 2, koff = (ks & 3) * 32;
                    const uint64_t ad = smem_desc_sw128(smem_u32(kb + box * 16384 + koff));
                    const uint64_t bd = smem_desc_sw128(smem_u32(kb + (R::kBoxes + box) * 16384 + koff));
                    tc_mma_bf16(tmem, ad, bd, idesc_bf16_f32(128, 128), ks > 0 ? 1u : 0u);
                }
                tc_commit(&st.mma_bar);
                mma_pend = true;
                poll_publish(tn, nkslot, p.flag_kn, kn_next_done);
            }
            ok = mbar_wait(&st.mma_bar, mma_phase, globaltimer() + p.timeout_ns);
            mma_phase ^= 1u;
            if (!__syncthreads_and(ok)) { record_status(status, CSMKV_ERR_TIMEOUT); break; }
            if (tid == 0) mma_pend = false;
            tc_fence_after();
            {   // warp w reads TMEM lanes 32(w%4).. (its A rows) and 32 columns 32(w/4)..
                const int qtr = warp & 3, grp = warp >> 2;
                const int a = qtr * 32 + lane;
                const int col0 = grp * 32;
                float v[32];
                tmem_ld_32x32b_x32(tmem + ((uint32_t)(qtr * 32) << 16) + (uint32_t)col0, v);
                const float inv_a = sm.inv[2 * a];
                float best = -INFINITY;
                int bb = col0;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float cs = v[i] * inv_a * sm.inv[2 * (col0 + i) + 1];
                    if (cs > best) { best = cs; bb = col0 + i; }
                }
                sm.best[grp * 128 + a] = best;
                sm.bestb[grp * 128 + a] = bb;
            }
            tc_fence_before();
            __syncthreads();

            // (4) selection, merge plan, compaction map
            chunk_tables(sm, sN, c, m, 4);
            if (p.match_out && tid < 128) p.match_out[((size_t)u * p.maxch + j) * 128 + tid] = sm.match[tid];
            if (j == 0 && tid == 0) p.len[u] = s - ch * m;
            if (tid == 0) poll_publish(tn, nkslot, p.flag_kn, kn_next_done);

            // (5) K and degrees: wait for the items whose sources we overwrite, then write
            int lo, hi;
            chunk_deps(j, c, m, lo, hi);
            if (!wait_items(fkn, lo, hi, epoch, globaltimer() + p.timeout_ns)) {
                record_status(status, CSMKV_ERR_TIMEOUT);
                break;
            }
            emit_rows<T>(Kg + (urow + dst_row) * D, c - m, D, sm, sN, kpiece);
            emit_degrees(p.N + urow + dst_row, c - m, sm, sN);

            // (6) K's slot is free: start V of the next item there
            fence_proxy_async_smem();
            __syncthreads();
            if (tid == 0 && is_chunk(tn)) issue_v(tn, kslot);

            // (7) V on chip, publish, wait, write
            ok = mbar_wait(&st.bar[vslot], ((phase_bits >> vslot) & 1u), globaltimer() + p.timeout_ns);
            phase_bits ^= 1u << vslot;
            if (!__syncthreads_and(ok)) { record_status(status, CSMKV_ERR_TIMEOUT); break; }
            if (tid == 0) {
                pend_bits &= ~(1u << vslot);
                if (!v_done_now) publish(fv + j, epoch, p.withhold);
                poll_publish(tn, nkslot, p.flag_kn, kn_next_done);
            }
            if (!wait_items(fv, lo, hi, epoch, globaltimer() + p.timeout_ns)) {
                record_status(status, CSMKV_ERR_TIMEOUT);
                break;
            }
            emit_rows<T>(Vg + (urow + dst_row) * D, c - m, D, sm, sN, vpiece);
            if (tid == 0) {
                poll_publish(tn, nkslot, p.flag_kn, kn_next_done);
                poll_publish(tn, kslot, p.flag_v, v_next_done);
            }
        } else {
            // ================================================================ tail piece
            ok = tail_piece<T>(p, u, lev - levels_ch, epoch, ring + kslot * R::kSlotBytes,
                               reinterpret_cast<int32_t*>(nbuf + kslot * R::kNStride));
            if (!ok) { record_status(status, CSMKV_ERR_TIMEOUT); break; }
            fence_proxy_async_smem();
            __syncthreads();
            if (tid == 0 && is_chunk(tn)) issue_v(tn, kslot);
        }

        // (8) V's slot is free: claim the item after next and start its K there
        fence_proxy_async_smem();
        __syncthreads();
        if (tid == 0) {
            const int t2 = claim_item(p, levels_ch, total);
            if (is_chunk(t2)) issue_k(t2, vslot);
            st.tk[0] = tn;
            st.tk[1] = t2;
        }
        __syncthreads();
        const int nk = nkslot;
        nkslot = vslot;
        vslot = kslot;
        kslot = nk;
    }

    // Teardown: loads or MMAs still in flight (after an abort) get a bounded chance to land.
    if (tid == 0) {
        for (int s = 0; s < R::kSlots; ++s)
            if ((pend_bits >> s) & 1u) (void)mbar_wait(&st.bar[s], ((phase_bits >> s) & 1u), globaltimer() + p.timeout_ns);
        if (mma_pend) (void)mbar_wait(&st.mma_bar, mma_phase, globaltimer() + p.timeout_ns);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

int launch_csm_tc(const CsmParams& P, int D, void* K, void* V, int32_t* N, uint64_t rows, cudaStream_t st) {
    CUtensorMap tmK{}, tmV{}, tmN{};
    const uint64_t dims[3] = {(uint64_t)D, 2, rows / 2};
    const uint64_t strides[2] = {(uint64_t)D * 2, (uint64_t)D * 4};
    const uint32_t box[3] = {64, 1, 128};
    const uint64_t ndims[2] = {4, rows / 4};
    const uint64_t nstr[1] = {16};
    const uint32_t nbox[2] = {4, (uint32_t)TcRing<128>::kNRows};
    if (!encode_tiled(&tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, K, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tiled(&tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, V, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tiled(&tmN, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, N, ndims, nstr, nbox, CU_TENSOR_MAP_SWIZZLE_NONE))
        return CSMKV_ERR_CUDA;
    const int grid = sm_count();
    if (grid <= 0) return CSMKV_ERR_CUDA;
    if (D == 128) {
        auto kern = csm_tc_kernel<128>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, TcRing<128>::kSmem) != cudaSuccess)
            return CSMKV_ERR_CUDA;
        kern<<<grid, kTcThreads, TcRing<128>::kSmem, st>>>(P, tmK, tmV, tmN);
    } else {
        auto kern = csm_tc_kernel<64>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, TcRing<64>::kSmem) != cudaSuccess)
            return CSMKV_ERR_CUDA;
        kern<<<grid, kTcThreads, TcRing<64>::kSmem, st>>>(P, tmK, tmV, tmN);
    }
    return cudaGetLastError() == cudaSuccess ? CSMKV_OK : CSMKV_ERR_CUDA;
}

}  // namespace csmkv
