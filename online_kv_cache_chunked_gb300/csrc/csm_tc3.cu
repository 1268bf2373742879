// csm_tc3.cu -- Chunked Soft Matching on the tensor cores, three CTAs per SM
// (bf16, c = 256, d in {64, 128}). [Chelsea §三 分块软匹配算法 steps 1-4;
// CentroidKV 分块软匹配 (CSM), 聚合]
//
// Each CTA (8 warps) owns one 64 KB shared-memory slot and walks work tickets
// (level-major: chunk j of every unit, then the tail pieces). Per chunk:
//   K by TMA through a 3-D view (column, row parity, row pair) of the cache, so
//   the A rows (even offsets) and B rows (odd offsets) land as two K-major MMA
//   operands in the 128-byte swizzle layout, with the degree tile by a 2-D map;
//   one thread issues d/16 tcgen05.mma (M = N = 128, fp32 accumulate in 128
//   TMEM columns) while the CUDA cores take fp32 inverse norms; 8 warps read
//   the dot products back with tcgen05.ld and take per-A argmaxes; then the
//   shared selection tables; then the K output; then V through the same slot.
// Output: when m = c/2 every A row merges and the output rows are exactly the
// B rows, already in shared memory in the layout a 2-D TMA store takes, so the
// merged rows are rewritten in place and two TMA stores write the block; for
// other m the output rows (copies and merges) are written straight to global
// memory. Three independent CTAs per SM
// overlap one another's loads, barriers and compute.
// In-place safety: every item publishes an epoch-tagged "loaded" flag per array
// once its TMA lands; an item writes an array only after the items whose source
// rows it overwrites have published (see csm_compress.cu).
// PAGED (block-table layout): a chunk's rows come through the unit's block table --
// when n1 is a multiple of 16, by TMA in 16-row groups (each inside one page) through
// the pool's parity view; otherwise row by row with 16-byte cp.async -- into the
// same swizzled operand layout,
// and every output row is stored through the table; the flags and the order of
// the in-place writes are those of the dense layout, in logical rows.
#include "csm_common.cuh"

namespace csmkv {

constexpr int kTc3Threads = 256;

struct alignas(16) Tc3State {
    uint64_t bar;      // slot loads
    uint64_t mma_bar;  // MMA completion
    int32_t tk;        // current ticket
    uint32_t tmem;
    int32_t dep_ok[2];  // the flags this chunk waits on were already set (K+N, V)
};

template <int D>
struct Tc3 {
    static constexpr int kBoxes = D / 64;
    static constexpr int kSlotBytes = 2 * kBoxes * 16384;
    static constexpr int kNRows = 65;  // degree tile: 65 x 4 int32 covers 256 rows from any start
    static constexpr int kNBytes = kNRows * 16;
    static constexpr int kNStride = 1088;
    static constexpr int kSmem = kSlotBytes + kNStride + (int)sizeof(CsmTables) + (int)sizeof(Tc3State) + 1024;
};

template <int D, bool PAGED>
__global__ void __launch_bounds__(kTc3Threads, 3)
    csm_tc3_kernel(const __grid_constant__ CsmParams p, const __grid_constant__ CUtensorMap tmK,
                   const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmN,
                   const __grid_constant__ CUtensorMap tmKs, const __grid_constant__ CUtensorMap tmVs) {
    using R = Tc3<D>;
    using T = __nv_bfloat16;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* const slot =
        reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    int32_t* const nbuf = reinterpret_cast<int32_t*>(slot + R::kSlotBytes);
    CsmTables& sm = *reinterpret_cast<CsmTables*>(slot + R::kSlotBytes + R::kNStride);
    Tc3State& st = *reinterpret_cast<Tc3State*>(&sm + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = p.c, m = p.m, BH = p.BH;
    T* const Kg = static_cast<T*>(p.K);
    T* const Vg = static_cast<T*>(p.V);
    int32_t* const status = &p.hdr->status;
    // Flags are published by a thread that writes no global memory on the m == H
    // path (degrees are written by threads 0..127), so release stores never wait
    // behind output writes.
    const bool publisher = (tid == 128);

    if (tid == 0) {
        mbar_init(&st.bar, 1);
        mbar_init(&st.mma_bar, 1);
        fence_mbar_init();
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        prefetch_tmap(&tmN);
        prefetch_tmap(&tmKs);
        prefetch_tmap(&tmVs);
    }
    if (warp == 0) {
        tmem_alloc(&st.tmem, 128);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = st.tmem;

    // Everything above is private setup; from here on the prologue's tables and the
    // cache are read, so wait for the prologue (launched just before) to complete.
    griddep_launch_dependents();
    griddep_wait();
    const int32_t epoch = p.hdr->epoch;
    const int levels_ch = p.hdr->levels_ch, levels_tail = p.hdr->levels_tail;
    const long long total = (long long)(levels_ch + levels_tail) * BH;
    const bool all = (m == 128);  // every A row merges: the output rows are the B rows, in order
    uint32_t phase = 0, mma_phase = 0;
    bool load_pend = false, mma_pend = false, stores_pend = false;  // thread 0

    auto load_slot = [&](const CUtensorMap* map, long long g0, bool with_degrees) {  // thread 0
        mbar_expect_tx(&st.bar, (uint32_t)(R::kSlotBytes + (with_degrees ? R::kNBytes : 0)));
        const int ya = (int)(g0 & 1), za = (int)(g0 >> 1);
        const int yb = (int)((g0 + 1) & 1), zb = (int)((g0 + 1) >> 1);
#pragma unroll
        for (int bx = 0; bx < R::kBoxes; ++bx) {
            tma_load_3d(slot + bx * 16384, map, &st.bar, bx * 64, ya, za);
            tma_load_3d(slot + (R::kBoxes + bx) * 16384, map, &st.bar, bx * 64, yb, zb);
        }
        if (with_degrees) tma_load_2d(nbuf, &tmN, &st.bar, 0, (int)(g0 >> 2));
        load_pend = true;
    };
    // m == H: every merged B row replaces its own shared-memory row (same arithmetic
    // as emit_rows: fp32 sums in A order, scaled by 1 / degree sum, rounded once).
    // Four threads per 64-column box of a row, two 16-byte pieces each, so the
    // per-row work (row lookup, member scan, swizzle terms) is paid once per 32
    // bytes; threads of the second box take their two pieces in the other order,
    // so a quarter warp (one row) reads 8 distinct bank groups at every step.
    auto merge_inplace = [&](const int32_t* sN) {
        constexpr int TPR = 4 * R::kBoxes;  // threads per row; divides the block size
        const int sub = tid % TPR;
        const int box = sub >> 2;
        const uint32_t c0 = (uint32_t)((sub & 3) * 2 + (box & 1)), c1 = c0 ^ 1u;
        uint8_t* const abox = slot + box * 16384;
        uint8_t* const bbox = slot + (R::kBoxes + box) * 16384;
        const int n = sm.nmerged * TPR;
        for (int i = tid; i < n; i += kTc3Threads) {
            const int b = sm.mlist[i / TPR];
            const uint32_t xb = (uint32_t)(b & 7);
            uint4* const d0 = reinterpret_cast<uint4*>(bbox + b * 128 + ((c0 ^ xb) << 4));
            uint4* const d1 = reinterpret_cast<uint4*>(bbox + b * 128 + ((c1 ^ xb) << 4));
            float acc0[8], acc1[8], f[8];
            const float nb = (float)sN[2 * b + 1];
            Elem<T>::unpack(*d0, f);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc0[e] = nb * f[e];
            Elem<T>::unpack(*d1, f);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc1[e] = nb * f[e];
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                uint32_t bits = sm.mask[b][w];
                while (bits) {
                    const int a = w * 32 + __ffs(bits) - 1;
                    bits &= bits - 1u;
                    const uint8_t* const arow = abox + a * 128;
                    const uint32_t xa = (uint32_t)(a & 7);
                    const float na = (float)sN[2 * a];
                    Elem<T>::unpack(*reinterpret_cast<const uint4*>(arow + ((c0 ^ xa) << 4)), f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc0[e] = fmaf(na, f[e], acc0[e]);
                    Elem<T>::unpack(*reinterpret_cast<const uint4*>(arow + ((c1 ^ xa) << 4)), f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc1[e] = fmaf(na, f[e], acc1[e]);
                }
            }
            const float inv = sm.ninv[b];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                acc0[e] *= inv;
                acc1[e] *= inv;
            }
            *d0 = Elem<T>::pack(acc0);
            *d1 = Elem<T>::pack(acc1);
        }
    };
    // m < H: the c - m output rows (copies, or merged B rows) written straight to
    // global memory; as merge_inplace, two 16-byte pieces per thread in a
    // bank-distinct order, so the per-row lookups are paid once per 32 bytes.
    auto emit_rows2 = [&](auto rowptr, const int32_t* sN) {  // rowptr(output row) -> T*, or nullptr: skip
        constexpr int TPR = 4 * R::kBoxes;
        const int sub = tid % TPR;
        const int box = sub >> 2;
        const uint32_t c0 = (uint32_t)((sub & 3) * 2 + (box & 1)), c1 = c0 ^ 1u;
        uint8_t* const abox = slot + box * 16384;
        const int n = (c - m) * TPR;
        for (int i = tid; i < n; i += kTc3Threads) {
            const int pr = i / TPR;
            const int q = sm.src[pr], row = q >> 1;
            const uint8_t* const src = slot + ((q & 1) * R::kBoxes + box) * 16384 + row * 128;
            const uint32_t x = (uint32_t)(row & 7);
            uint4 v0 = *reinterpret_cast<const uint4*>(src + ((c0 ^ x) << 4));
            uint4 v1 = *reinterpret_cast<const uint4*>(src + ((c1 ^ x) << 4));
            if (q & 1) {
                const float inv = sm.ninv[row];
                if (inv != 0.0f) {  // a B row with incoming edges: degree-weighted mean
                    float acc0[8], acc1[8], f[8];
                    const float nb = (float)sN[q];
                    Elem<T>::unpack(v0, f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc0[e] = nb * f[e];
                    Elem<T>::unpack(v1, f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc1[e] = nb * f[e];
#pragma unroll
                    for (int w = 0; w < 4; ++w) {
                        uint32_t bits = sm.mask[row][w];
                        while (bits) {
                            const int a = w * 32 + __ffs(bits) - 1;
                            bits &= bits - 1u;
                            const uint8_t* const arow = abox + a * 128;
                            const uint32_t xa = (uint32_t)(a & 7);
                            const float na = (float)sN[2 * a];
                            Elem<T>::unpack(*reinterpret_cast<const uint4*>(arow + ((c0 ^ xa) << 4)), f);
#pragma unroll
                            for (int e = 0; e < 8; ++e) acc0[e] = fmaf(na, f[e], acc0[e]);
                            Elem<T>::unpack(*reinterpret_cast<const uint4*>(arow + ((c1 ^ xa) << 4)), f);
#pragma unroll
                            for (int e = 0; e < 8; ++e) acc1[e] = fmaf(na, f[e], acc1[e]);
                        }
                    }
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        acc0[e] *= inv;
                        acc1[e] *= inv;
                    }
                    v0 = Elem<T>::pack(acc0);
                    v1 = Elem<T>::pack(acc1);
                }
            }
            T* const rp = rowptr(pr);
            if (!rp) continue;
            uint4* const drow = reinterpret_cast<uint4*>(rp) + box * 8;
            drow[c0] = v0;
            drow[c1] = v1;
        }
    };
    auto store_b_rows = [&](const CUtensorMap* map, long long row) {  // thread 0
#pragma unroll
        for (int bx = 0; bx < R::kBoxes; ++bx) tma_store_2d(map, slot + (R::kBoxes + bx) * 16384, bx * 64, (int)row);
        bulk_commit();
        stores_pend = true;
    };
    // PAGED: chunk row tid (c == 256 rows, one per thread) of unit u from logical row
    // base, through the block table, into the swizzled A / B operand layout; its
    // degree into nbuf[tid]. Completed by cp_async_wait_all.
    auto gather_slot = [&](const T* arr, int u, int base, bool with_degrees) {  // all threads
        const int q = tid, op = q & 1, r2 = q >> 1;
        const long long pr = map_row(p.rm, u, base + q);
        if (pr < 0) {
            record_status(status, CSMKV_ERR_ARG);
            if (with_degrees) nbuf[q] = 0;
            return;
        }
        const uint8_t* src = reinterpret_cast<const uint8_t*>(arr + pr * D);
#pragma unroll
        for (int k = 0; k < D / 8; ++k) {
            const int bx = k >> 3, c16 = k & 7;
            cp_async16(slot + (op * R::kBoxes + bx) * 16384 + r2 * 128 + ((c16 ^ (r2 & 7)) << 4), src + k * 16);
        }
        if (with_degrees) cp_async4(nbuf + q, p.N + pr);
    };
    // PAGED, n1 a multiple of 16: the chunk's rows from logical row base as 16 groups of
    // 16 rows, each inside one page, by TMA through the 3-D parity view of the pool (a
    // box of 8 rows of one parity): lane 2 g + op loads group g's A (op 0) or B rows into
    // rows 8 g .. 8 g + 7 of that operand's boxes. A block-table entry outside the pool
    // gets an out-of-range coordinate (zeros land) and CSMKV_ERR_ARG. Completes on st.bar.
    auto tma_gather_slot = [&](const CUtensorMap* map, int u, int base) {  // warp 0
        if (lane == 0) {
            mbar_expect_tx(&st.bar, (uint32_t)R::kSlotBytes);
            load_pend = true;
        }
        __syncwarp();
        const int g = lane >> 1, op = lane & 1;
        const long long pr = map_row(p.rm, u, base + 16 * g);
        int y = 0, z = -16;
        if (pr < 0) {
            record_status(status, CSMKV_ERR_ARG);
        } else {
            y = (int)((pr + op) & 1);
            z = (int)((pr + op) >> 1);
        }
#pragma unroll
        for (int bx = 0; bx < R::kBoxes; ++bx)
            tma_load_3d(slot + (op * R::kBoxes + bx) * 16384 + g * 1024, map, &st.bar, bx * 64, y, z);
    };
    // PAGED, n1 a multiple of 16: the 128 output rows held in the B boxes (every A row
    // merged) stored by TMA in 16-row groups through the table to logical rows drow ..
    // drow + 127 (drow is then a multiple of 16: no group straddles a page); a group
    // whose entry lies outside the pool is not stored and CSMKV_ERR_ARG is recorded.
    auto store_b_rows_paged_tma = [&](const CUtensorMap* map, int u, int drow) {  // thread 0
        for (int g = 0; g < 8; ++g) {
            const long long pr = map_row(p.rm, u, drow + 16 * g);
            if (pr < 0) {
                record_status(status, CSMKV_ERR_ARG);
                continue;
            }
#pragma unroll
            for (int bx = 0; bx < R::kBoxes; ++bx)
                tma_store_2d(map, slot + (R::kBoxes + bx) * 16384 + g * 2048, bx * 64, (int)pr);
        }
        bulk_commit();
        stores_pend = true;
    };
    // PAGED: the degrees of the chunk's rows, one per thread, by cp.async (completed by
    // cp_async_wait_all).
    auto gather_degrees = [&](int u, int base) {  // all threads
        const long long pr = map_row(p.rm, u, base + tid);
        if (pr < 0) nbuf[tid] = 0; else cp_async4(nbuf + tid, p.N + pr);
    };
    // PAGED: the 128 B rows of the slot (the output when every A row merges) stored
    // through the block table to logical rows drow .. drow + 127.
    auto store_b_rows_paged = [&](T* arr, int u, int drow) {  // all threads
        constexpr int PPR = D / 8;
        for (int i = tid; i < 128 * PPR; i += kTc3Threads) {
            const int b = i / PPR, k = i - (i / PPR) * PPR, bx = k >> 3, c16 = k & 7;
            const long long pr = map_row(p.rm, u, drow + b);
            if (pr < 0) {
                record_status(status, CSMKV_ERR_ARG);
                continue;
            }
            reinterpret_cast<uint4*>(arr + pr * D)[k] =
                *reinterpret_cast<const uint4*>(slot + (R::kBoxes + bx) * 16384 + b * 128 + ((c16 ^ (b & 7)) << 4));
        }
    };

    for (;;) {
        if (tid == 0) {
            const int t = claim_item(p, levels_ch, total);
            st.tk = t;
            if (stores_pend) {  // the previous item's V store must have left the slot
                bulk_wait_read_all();
                stores_pend = false;
            }
            if (!PAGED && t != INT_MAX && t / BH < levels_ch) {
                const int j = t / BH, u = t - j * BH;
                load_slot(&tmK, (long long)u * p.cap + p.n1 + (long long)j * c, true);
            }
        }
        __syncthreads();
        const int t = st.tk;
        if (t == INT_MAX) break;
        const int lev = t / BH, u = t - lev * BH;
        bool ok = true;
        if constexpr (PAGED) {
            if (lev < levels_ch) {
                if (p.paged_tma) {
                    gather_degrees(u, p.n1 + lev * c);
                    if (warp == 0) tma_gather_slot(&tmK, u, p.n1 + lev * c);
                } else {
                    gather_slot(Kg, u, p.n1 + lev * c, true);
                }
            }
        }

        if (lev < levels_ch) {
            // ================================================================ chunk item
            const int j = lev, ch = p.unit_ch[u], s = p.snap[u];
            const size_t urow = (size_t)u * p.cap;
            const int dst_row = p.n1 + j * (c - m);
            const long long g0 = (long long)urow + p.n1 + (long long)j * c;
            const int32_t* const sN = PAGED ? nbuf : nbuf + (int)(g0 & 3);
            int32_t* const fkn = p.flag_kn + (size_t)u * p.L;
            int32_t* const fv = p.flag_v + (size_t)u * p.L;
            int lo, hi;
            chunk_deps(j, c, m, lo, hi);
            // thread 64 peeks at the flags this chunk will wait on (relaxed; compared later)
            int32_t pk0 = epoch, pk1 = epoch, pv0 = epoch, pv1 = epoch;
            if (tid == 64) {
                if (lo <= hi) {
                    pk0 = ld_volatile(fkn + lo);
                    pv0 = ld_volatile(fv + lo);
                }
                if (lo < hi) {
                    pk1 = ld_volatile(fkn + hi);
                    pv1 = ld_volatile(fv + hi);
                }
            }

            // (1) K and degrees on chip
            if constexpr (PAGED) {
                cp_async_wait_all();
                fence_proxy_async_smem();  // the gathered operands before the MMA reads them
                if (p.paged_tma) {
                    ok = mbar_wait(&st.bar, phase, globaltimer() + p.timeout_ns);
                    phase ^= 1u;
                }
            } else {
                ok = mbar_wait(&st.bar, phase, globaltimer() + p.timeout_ns);
                phase ^= 1u;
            }
            if (!__syncthreads_and(ok)) { record_status(status, CSMKV_ERR_TIMEOUT); break; }
            if (tid == 0) load_pend = false;
            if (publisher) publish(fkn + j, epoch, p.withhold);

            // (2) the dot products start on the tensor cores; the norms run meanwhile
            if (tid == 0) {
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const int box = ks >> 2, koff = (ks & 3) * 32;
                    const uint64_t ad = smem_desc_sw128(smem_u32(slot + box * 16384 + koff));
                    const uint64_t bd = smem_desc_sw128(smem_u32(slot + (R::kBoxes + box) * 16384 + koff));
                    tc_mma_bf16(tmem, ad, bd, idesc_bf16_f32(128, 128), ks > 0 ? 1u : 0u);
                }
                tc_commit(&st.mma_bar);
                mma_pend = true;
            }
            {   // one thread per chunk row; a quarter warp covers 8 consecutive rows of one
                // operand and reads physical 16-byte chunks in swizzled order: distinct banks
                const int op = (tid >> 3) & 1;
                const int idx = (tid & 7) | ((tid >> 4) << 3);
                const uint8_t* row = slot + op * R::kBoxes * 16384 + idx * 128;
                float ss = 0.f;
#pragma unroll
                for (int bx = 0; bx < R::kBoxes; ++bx) {
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        float f[8];
                        Elem<T>::unpack(*reinterpret_cast<const uint4*>(row + bx * 16384 + ((i ^ (idx & 7)) << 4)), f);
#pragma unroll
                        for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
                    }
                }
                const float inv = ss > 0.f ? 1.0f / sqrtf(ss) : 0.0f;
                if (op) sm.invB[idx] = inv; else sm.invA[idx] = inv;
                if (tid == 64) {
                    const int ok_k = pk0 == epoch && pk1 == epoch, ok_v = pv0 == epoch && pv1 == epoch;
                    if (ok_k || ok_v) __threadfence();  // acquire side of the flags seen set
                    st.dep_ok[0] = ok_k;
                    st.dep_ok[1] = ok_v;
                }
            }
            __syncthreads();

            // (3) 8 warps read the 128 x 128 dot products: TMEM lane quarter w % 4, 64 columns per half
            ok = mbar_wait(&st.mma_bar, mma_phase, globaltimer() + p.timeout_ns);
            mma_phase ^= 1u;
            if (!__syncthreads_and(ok)) { record_status(status, CSMKV_ERR_TIMEOUT); break; }
            if (tid == 0) mma_pend = false;
            tc_fence_after();
            {
                const int qtr = warp & 3, half = warp >> 2;
                const int a = qtr * 32 + lane;
                const float inv_a = sm.invA[a];
                float best = -INFINITY;
                int bb = half * 64;
#pragma unroll
                for (int cb = 0; cb < 2; ++cb) {
                    const int col0 = half * 64 + cb * 32;
                    float v[32];
                    tmem_ld_32x32b_x32(tmem + ((uint32_t)(qtr * 32) << 16) + (uint32_t)col0, v);
                    // argmax_b of dot * invB[b] (invA[a] > 0 does not move it), scaled once
                    const float4* ib = reinterpret_cast<const float4*>(sm.invB + col0);
#pragma unroll
                    for (int i4 = 0; i4 < 8; ++i4) {
                        const float4 w4 = ib[i4];
                        const float wv[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float cs = v[4 * i4 + e] * wv[e];
                            if (cs > best) { best = cs; bb = col0 + 4 * i4 + e; }
                        }
                    }
                }
                if (inv_a == 0.0f) {  // a zero key has cosine 0 to every B row: lowest index
                    best = 0.0f;
                    bb = half * 64;
                }
                sm.best[half * 128 + a] = best * inv_a;
                sm.bestb[half * 128 + a] = (uint8_t)bb;
            }
            tc_fence_before();
            __syncthreads();

            // (4) selection, merge plan, compaction map
            chunk_tables(sm, sN, c, m, 2);
            if (p.match_out && tid < 128) p.match_out[((size_t)u * p.maxch + j) * 128 + tid] = (int32_t)sm.match[tid];
            if (j == 0 && tid == 0) p.len[u] = s - ch * m;

            // (5) K and degrees out, after the items whose sources they overwrite
            if (!st.dep_ok[0] && !wait_items(fkn, lo, hi, epoch, globaltimer() + p.timeout_ns)) {
                record_status(status, CSMKV_ERR_TIMEOUT);
                break;
            }
            if (all) {
                merge_inplace(sN);
                if constexpr (PAGED) {
                    if (p.paged_tma) {
                        fence_proxy_async_smem();
                        __syncthreads();
                        if (tid == 0) store_b_rows_paged_tma(&tmKs, u, dst_row);
                    } else {
                        __syncthreads();
                        store_b_rows_paged(Kg, u, dst_row);
                    }
                } else {
                    fence_proxy_async_smem();
                    __syncthreads();
                    if (tid == 0) store_b_rows(&tmKs, (long long)urow + dst_row);
                }
            } else if constexpr (PAGED) {
                emit_rows2([&](int pr) -> T* {
                    const long long r = map_row(p.rm, u, dst_row + pr);
                    if (r < 0) record_status(status, CSMKV_ERR_ARG);
                    return r < 0 ? nullptr : Kg + r * D;
                }, sN);
            } else {
                emit_rows2([&](int pr) -> T* { return Kg + (urow + dst_row + pr) * D; }, sN);
            }
            if constexpr (PAGED) {
                for (int pr = tid; pr < c - m; pr += kTc3Threads) {
                    const int q = all ? 2 * pr + 1 : sm.src[pr];
                    const long long r = map_row(p.rm, u, dst_row + pr);
                    if (r >= 0) p.N[r] = (q & 1) ? sm.nsum[q >> 1] : sN[q];
                }
            } else {
                emit_degrees(p.N + urow + dst_row, c - m, m, sm, sN);
            }

            // (6) V through the same slot once the K output has left it
            fence_proxy_async_smem();
            __syncthreads();
            if constexpr (PAGED) {
                if (p.paged_tma) {
                    if (warp == 0) {
                        if (tid == 0 && stores_pend) {  // the K rows' stores have left the slot
                            bulk_wait_read_all();
                            stores_pend = false;
                        }
                        __syncwarp();
                        tma_gather_slot(&tmV, u, p.n1 + j * c);
                    }
                    ok = mbar_wait(&st.bar, phase, globaltimer() + p.timeout_ns);
                    phase ^= 1u;
                } else {
                    gather_slot(Vg, u, p.n1 + j * c, false);
                    cp_async_wait_all();
                }
            } else {
                if (tid == 0) {
                    if (stores_pend) {
                        bulk_wait_read_all();
                        stores_pend = false;
                    }
                    load_slot(&tmV, g0, false);
                }
                ok = mbar_wait(&st.bar, phase, globaltimer() + p.timeout_ns);
                phase ^= 1u;
            }
            if (!__syncthreads_and(ok)) { record_status(status, CSMKV_ERR_TIMEOUT); break; }
            if (tid == 0) load_pend = false;
            if (publisher) publish(fv + j, epoch, p.withhold);
            if (!st.dep_ok[1] && !wait_items(fv, lo, hi, epoch, globaltimer() + p.timeout_ns)) {
                record_status(status, CSMKV_ERR_TIMEOUT);
                break;
            }
            if (all) {
                merge_inplace(sN);
                if constexpr (PAGED) {
                    if (p.paged_tma) {
                        fence_proxy_async_smem();
                        __syncthreads();
                        if (tid == 0) store_b_rows_paged_tma(&tmVs, u, dst_row);
                    } else {
                        __syncthreads();
                        store_b_rows_paged(Vg, u, dst_row);
                    }
                } else {
                    fence_proxy_async_smem();
                    __syncthreads();
                    if (tid == 0) store_b_rows(&tmVs, (long long)urow + dst_row);
                }
            } else if constexpr (PAGED) {
                emit_rows2([&](int pr) -> T* {
                    const long long r = map_row(p.rm, u, dst_row + pr);
                    return r < 0 ? nullptr : Vg + r * D;
                }, sN);
            } else {
                emit_rows2([&](int pr) -> T* { return Vg + (urow + dst_row + pr) * D; }, sN);
            }
        } else {
            // ================================================================ tail piece
            ok = tail_piece<T, PAGED>(p, u, lev - levels_ch, epoch, slot, nbuf);
            if (!ok) { record_status(status, CSMKV_ERR_TIMEOUT); break; }
        }
        fence_proxy_async_smem();  // the next TMA overwrites the slot
        __syncthreads();
    }

    // Teardown: stores, loads or MMAs still in flight get a bounded chance to land.
    if (tid == 0) {
        bulk_wait_all();
        if (load_pend) (void)mbar_wait(&st.bar, phase, globaltimer() + p.timeout_ns);
        if (mma_pend) (void)mbar_wait(&st.mma_bar, mma_phase, globaltimer() + p.timeout_ns);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 128);
}

int launch_csm_tc3(const CsmParams& P, int D, void* K, void* V, int32_t* N, uint64_t rows, bool paged, cudaStream_t st) {
    CUtensorMap tmK{}, tmV{}, tmN{}, tmKs{}, tmVs{};
    const uint64_t dims[3] = {(uint64_t)D, 2, rows / 2};
    const uint64_t strides[2] = {(uint64_t)D * 2, (uint64_t)D * 4};
    const uint32_t box[3] = {64, 1, paged ? 8u : 128u};  // paged: 16-row groups, 8 rows of one parity
    const uint64_t ndims[2] = {4, rows / 4};
    const uint64_t nstr[1] = {16};
    const uint32_t nbox[2] = {4, (uint32_t)Tc3<128>::kNRows};
    const uint64_t sdims[2] = {(uint64_t)D, rows};
    const uint64_t sstr[1] = {(uint64_t)D * 2};
    const uint32_t sbox[2] = {64, paged ? 16u : 128u};  // paged: 16-row groups
    if (!encode_tiled(&tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, K, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tiled(&tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, V, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tiled(&tmN, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, N, ndims, nstr, nbox, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_tiled(&tmKs, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, K, sdims, sstr, sbox, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tiled(&tmVs, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, V, sdims, sstr, sbox, CU_TENSOR_MAP_SWIZZLE_128B))
        return CSMKV_ERR_CUDA;
    const int grid = 3 * sm_count();
    if (grid <= 0) return CSMKV_ERR_CUDA;
    auto run = [&](auto kern, int smem) {
        if (set_kernel_smem((const void*)kern, smem, true) != CSMKV_OK) return (int)CSMKV_ERR_CUDA;
        if (launch_overlapped(kern, dim3(grid), dim3(kTc3Threads), (size_t)smem, st, P, tmK, tmV, tmN, tmKs,
                              tmVs) != cudaSuccess)
            return (int)CSMKV_ERR_CUDA;
        return cudaGetLastError() == cudaSuccess ? (int)CSMKV_OK : (int)CSMKV_ERR_CUDA;
    };
    if (paged)
        return D == 128 ? run(csm_tc3_kernel<128, true>, Tc3<128>::kSmem) : run(csm_tc3_kernel<64, true>, Tc3<64>::kSmem);
    return D == 128 ? run(csm_tc3_kernel<128, false>, Tc3<128>::kSmem) : run(csm_tc3_kernel<64, false>, Tc3<64>::kSmem);
}

}  // namespace csmkv
