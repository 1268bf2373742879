// csm_tc.cu -- Chunked Soft Matching on the tensor cores (bf16, c = 256,
// d in {64, 128}), one 16-warp CTA per SM with a slot ring: the alternative to
// the three-CTAs-per-SM kernel in csm_tc3.cu (the default), selected with
// CSM_KERNEL_TC_RING. [Chelsea §三 分块软匹配算法 steps 1-4; CentroidKV 分块软匹配 (CSM), 聚合]
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

constexpr int kTcThreads = 512;  // 16 warps: 4 TMEM lane quarters x 4 column groups

struct alignas(16) TcState {
    uint64_t bar[3];  // one per ring slot
    uint64_t mma_bar;
    int32_t tk[3];    // tickets: current item, next, the one after
    uint32_t tmem;
    int32_t raw_tk;   // ticket fetched early in the iteration, checked at its end
    int32_t raw_ok;   // that ticket is a non-empty item
    int32_t mma_early;  // the MMA of the next item was issued at the end of this one
    int32_t defer_k;    // chunk whose K load waits for the last V store to leave its slot
    int32_t dep_ok[2];  // flags this chunk waits on were already set (K+N, V)
};

template <int D>
struct TcRing {
    static constexpr int kBoxes = D / 64;
    static constexpr int kSlotBytes = 2 * kBoxes * 16384;  // A and B rows of one chunk of one array
    static constexpr int kSlots = 3;
    static constexpr int kNRows = 65;                      // degree tile: 65 x 4 int32 covers 256 rows
    static constexpr int kNBytes = kNRows * 16;
    static constexpr int kNStride = 1152;                  // per-slot degree buffer
    static constexpr int kSmem = kSlots * kSlotBytes + kSlots * kNStride + (int)sizeof(CsmTables) + (int)sizeof(TcState) + 1024;
    static_assert((kSlots * kSlotBytes + kSlots * kNStride) % 16 == 0, "tables start 16-byte aligned");
};

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1)
    csm_tc_kernel(const __grid_constant__ CsmParams p, const __grid_constant__ CUtensorMap tmK,
                  const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmN,
                  const __grid_constant__ CUtensorMap tmKs, const __grid_constant__ CUtensorMap tmVs) {
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
        bulk_wait_all();  // output stores complete before the CTA exits
        for (int s = 0; s < R::kSlots; ++s) mbar_init(&st.bar[s], 1);
        mbar_init(&st.mma_bar, 1);
        fence_mbar_init();
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        prefetch_tmap(&tmN);
        prefetch_tmap(&tmKs);
        prefetch_tmap(&tmVs);
        st.mma_early = 0;
        st.defer_k = INT_MAX;
    }
    if (warp == 0) {
        tmem_alloc(&st.tmem, 128);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = st.tmem;

    const int32_t epoch = p.hdr->epoch;
    const bool all = (m == 128);  // every A row merges: the output rows are the B rows, in order
    bool stores_pending = false;  // thread 0: TMA stores committed since the last read-wait
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
    // Flags are published by one thread that writes no global memory on the m == H
    // path, so its release stores never wait behind output writes. Polling a slot
    // whose load is not issued yet finds its next phase incomplete and does nothing.
    const bool publisher = (tid == 256);
    auto poll_publish = [&](int t, int slot, int32_t* flags_base, bool& done) {
        if (done || !is_chunk(t)) return;
        if (mbar_test(&st.bar[slot], ((phase_bits >> slot) & 1u))) {
            const int j = t / BH, u = t - j * BH;
            publish(flags_base + (size_t)u * p.L + j, epoch, p.withhold);
            done = true;
        }
    };

    // m == H: every merged B row replaces its own shared-memory row (same arithmetic
    // as emit_rows: fp32 sums in A order, scaled by 1 / degree sum, rounded once).
    auto merge_inplace = [&](auto piece, const int32_t* sN) {
        constexpr int PR = D / 8;
        const int n = sm.nmerged * PR;
        for (int i = tid; i < n; i += kTcThreads) {
            const int k = i / PR, cc = i - k * PR;
            const int b = sm.mlist[k], q = 2 * b + 1;
            uint4* dst = reinterpret_cast<uint4*>(piece(q, cc));
            float acc[8], f[8];
            Elem<T>::unpack(*dst, f);
            const float nb = (float)sN[q];
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = nb * f[e];
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                uint32_t bits = sm.mask[b][w];
                while (bits) {
                    const int qa = 2 * (w * 32 + __ffs(bits) - 1);
                    bits &= bits - 1u;
                    Elem<T>::unpack(*reinterpret_cast<const uint4*>(piece(qa, cc)), f);
                    const float na = (float)sN[qa];
#pragma unroll
                    for (int e = 0; e < 8; ++e) acc[e] = fmaf(na, f[e], acc[e]);
                }
            }
            const float inv = sm.ninv[b];
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] *= inv;
            *dst = Elem<T>::pack(acc);
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
        // Off the critical path: thread 32 fetches the ticket after next and thread 64
        // peeks at the flags this chunk will wait on; both results are used much later.
        int raw_ticket = INT_MAX, raw_uch = 0;
        if (tid == 32) raw_ticket = atomicAdd(&p.hdr->ticket, 1);
        // relaxed loads of at most two K and two V flags; compared (and fenced) later
        int32_t pk0 = epoch, pk1 = epoch, pv0 = epoch, pv1 = epoch;
        if (tid == 64 && lev < levels_ch) {
            int lo, hi;
            chunk_deps(lev, c, p.m, lo, hi);
            const int32_t* fk = p.flag_kn + (size_t)u * p.L;
            const int32_t* fw = p.flag_v + (size_t)u * p.L;
            if (lo <= hi) {
                pk0 = ld_volatile(fk + lo);
                pv0 = ld_volatile(fw + lo);
            }
            if (lo < hi) {
                pk1 = ld_volatile(fk + hi);
                pv1 = ld_volatile(fw + hi);
            }
        }

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
                if (st.defer_k != INT_MAX) {  // K two items ahead, once the last V store left its slot
                    bulk_wait_read_all();
                    stores_pending = false;
                    issue_k(st.defer_k, nkslot);
                    st.defer_k = INT_MAX;
                }
            }
            if (publisher && !kn_done_now) publish(fkn + j, epoch, p.withhold);
            // (2) the 128 x 128 dot products start on the tensor cores now; the norms
            // below run on the CUDA cores meanwhile
            if (tid == 0 && !st.mma_early) {
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
            }
            if (publisher) poll_publish(tn, nkslot, p.flag_kn, kn_next_done);

            // (2b) inverse key norms, two threads per chunk row. A quarter warp covers 8
            // consecutive rows of one operand, reading physical 16-byte chunks in swizzled
            // order, so its loads hit distinct banks; the row's two halves meet by shuffle.
            {
                const int h = (tid >> 3) & 1, op = (tid >> 4) & 1;
                const int idx = (tid & 7) | ((tid >> 5) << 3);  // row within its operand
                const uint8_t* row = kb + op * R::kBoxes * 16384 + idx * 128;
                float ss = 0.f;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int box = R::kBoxes == 2 ? h : 0;
                    const int chk = R::kBoxes == 2 ? i : (h * 4 + (i & 3));
                    if (R::kBoxes == 1 && i >= 4) break;
                    float f[8];
                    Elem<T>::unpack(*reinterpret_cast<const uint4*>(row + box * 16384 + ((chk ^ (idx & 7)) << 4)), f);
#pragma unroll
                    for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
                }
                ss += __shfl_xor_sync(0xffffffffu, ss, 8);
                if (h == 0) {
                    const float inv = ss > 0.f ? 1.0f / sqrtf(ss) : 0.0f;
                    if (op) sm.invB[idx] = inv; else sm.invA[idx] = inv;
                }
                if (tid == 32) raw_uch = raw_ticket < total ? (raw_ticket / BH < levels_ch ? p.unit_ch[raw_ticket % BH]
                                                                                          : p.unit_tp[raw_ticket % BH])
                                                             : 0;
                if (tid == 64) {
                    const int ok_k = pk0 == epoch && pk1 == epoch, ok_v = pv0 == epoch && pv1 == epoch;
                    if (ok_k || ok_v) __threadfence();  // acquire side of the flags seen set
                    st.dep_ok[0] = ok_k;
                    st.dep_ok[1] = ok_v;
                }
            }
            __syncthreads();

            // (3) the dot products, read back by 16 warps
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
                // argmax_b of dot * invB[b] (invA[a] > 0 does not move it), scaled once
                const float inv_a = sm.invA[a];
                const float4* ib = reinterpret_cast<const float4*>(sm.invB + col0);
                float best = -INFINITY;
                int bb = col0;
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
                if (inv_a == 0.0f) {  // a zero key has cosine 0 to every B row: lowest index
                    best = 0.0f;
                    bb = col0;
                }
                sm.best[grp * 128 + a] = best * inv_a;
                sm.bestb[grp * 128 + a] = (uint8_t)bb;
            }
            tc_fence_before();
            __syncthreads();

            // (4) selection, merge plan, compaction map
            chunk_tables(sm, sN, c, m, 4);
            if (p.match_out && tid < 128) p.match_out[((size_t)u * p.maxch + j) * 128 + tid] = (int32_t)sm.match[tid];
            if (j == 0 && tid == 0) p.len[u] = s - ch * m;
            if (publisher) poll_publish(tn, nkslot, p.flag_kn, kn_next_done);

            // (5) K and degrees: wait for the items whose sources we overwrite, then write
            int lo, hi;
            chunk_deps(j, c, m, lo, hi);
            if (!st.dep_ok[0] && !wait_items(fkn, lo, hi, epoch, globaltimer() + p.timeout_ns)) {
                record_status(status, CSMKV_ERR_TIMEOUT);
                break;
            }
            if (all) {  // merged B rows in place, then the B boxes go out by TMA
                merge_inplace(kpiece, sN);
                fence_proxy_async_smem();
                __syncthreads();
                if (tid == 0) {
#pragma unroll
                    for (int bx = 0; bx < R::kBoxes; ++bx)
                        tma_store_2d(&tmKs, kb + (R::kBoxes + bx) * 16384, bx * 64, (int)(urow + dst_row));
                    bulk_commit();
                    stores_pending = true;
                }
            } else {
                emit_rows<T>(Kg + (urow + dst_row) * D, c - m, D, m, sm, sN, kpiece);
            }
            emit_degrees(p.N + urow + dst_row, c - m, m, sm, sN);

            // (6) K's slot is free: start V of the next item there
            fence_proxy_async_smem();
            __syncthreads();
            if (tid == 0 && is_chunk(tn) && !all) issue_v(tn, kslot);  // m == H: after the V store, below

            // (7) V on chip, publish, wait, write
            ok = mbar_wait(&st.bar[vslot], ((phase_bits >> vslot) & 1u), globaltimer() + p.timeout_ns);
            phase_bits ^= 1u << vslot;
            if (!__syncthreads_and(ok)) { record_status(status, CSMKV_ERR_TIMEOUT); break; }
            if (tid == 0) pend_bits &= ~(1u << vslot);
            if (publisher) {
                if (!v_done_now) publish(fv + j, epoch, p.withhold);
                poll_publish(tn, nkslot, p.flag_kn, kn_next_done);
            }
            if (!st.dep_ok[1] && !wait_items(fv, lo, hi, epoch, globaltimer() + p.timeout_ns)) {
                record_status(status, CSMKV_ERR_TIMEOUT);
                break;
            }
            if (all) {
                merge_inplace(vpiece, sN);
                fence_proxy_async_smem();
                __syncthreads();
                if (tid == 0) {
#pragma unroll
                    for (int bx = 0; bx < R::kBoxes; ++bx)
                        tma_store_2d(&tmVs, vb + (R::kBoxes + bx) * 16384, bx * 64, (int)(urow + dst_row));
                    bulk_commit();
                    stores_pending = true;
                    if (is_chunk(tn)) {  // K's slot is free once the K store has read it
                        bulk_wait_read_but_one();
                        issue_v(tn, kslot);
                    }
                }
            } else {
                emit_rows<T>(Vg + (urow + dst_row) * D, c - m, D, m, sm, sN, vpiece);
            }
            if (publisher) {
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
            if (tid == 0) {
                if (stores_pending) {
                    bulk_wait_read_all();
                    stores_pending = false;
                }
                if (st.defer_k != INT_MAX) {
                    issue_k(st.defer_k, nkslot);
                    st.defer_k = INT_MAX;
                }
                if (is_chunk(tn)) issue_v(tn, kslot);
            }
        }

        // (8) V's slot is free: claim the item after next and start its K there
        fence_proxy_async_smem();
        if (tid == 32) {
            st.raw_tk = raw_ticket;
            st.raw_ok = raw_uch > (raw_ticket / BH < levels_ch ? raw_ticket / BH : raw_ticket / BH - levels_ch);
        }
        __syncthreads();
        if (tid == 0) {
            const int t2 = (st.raw_ok && ld_volatile(status) == 0) ? st.raw_tk : claim_from(p, st.raw_tk, levels_ch, total);
            if (is_chunk(t2)) {
                if (stores_pending) st.defer_k = t2;  // the V store may still be reading this slot
                else issue_k(t2, vslot);
            }
            // the next chunk's MMA can start now if its K has landed (TMEM is free)
            st.mma_early = 0;
            if (is_chunk(tn) && mbar_test(&st.bar[nkslot], (phase_bits >> nkslot) & 1u)) {
                const uint8_t* nkb = ring + nkslot * R::kSlotBytes;
                tc_fence_after();
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const int box = ks >> 2, koff = (ks & 3) * 32;
                    const uint64_t ad = smem_desc_sw128(smem_u32(nkb + box * 16384 + koff));
                    const uint64_t bd = smem_desc_sw128(smem_u32(nkb + (R::kBoxes + box) * 16384 + koff));
                    tc_mma_bf16(tmem, ad, bd, idesc_bf16_f32(128, 128), ks > 0 ? 1u : 0u);
                }
                tc_commit(&st.mma_bar);
                mma_pend = true;
                st.mma_early = 1;
            }
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
    CUtensorMap tmKs{}, tmVs{};
    const uint64_t sdims[2] = {(uint64_t)D, rows};
    const uint64_t sstr[1] = {(uint64_t)D * 2};
    const uint32_t sbox[2] = {64, 128};
    if (!encode_tiled(&tmKs, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, K, sdims, sstr, sbox, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tiled(&tmVs, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, V, sdims, sstr, sbox, CU_TENSOR_MAP_SWIZZLE_128B))
        return CSMKV_ERR_CUDA;
    if (!encode_tiled(&tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, K, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tiled(&tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, V, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tiled(&tmN, CU_TENSOR_MAP_DATA_TYPE_INT32, 2, N, ndims, nstr, nbox, CU_TENSOR_MAP_SWIZZLE_NONE))
        return CSMKV_ERR_CUDA;
    const int grid = sm_count();
    if (grid <= 0) return CSMKV_ERR_CUDA;
    if (D == 128) {
        auto kern = csm_tc_kernel<128>;
        if (set_kernel_smem((const void*)kern, TcRing<128>::kSmem) != CSMKV_OK) return CSMKV_ERR_CUDA;
        kern<<<grid, kTcThreads, TcRing<128>::kSmem, st>>>(P, tmK, tmV, tmN, tmKs, tmVs);
    } else {
        auto kern = csm_tc_kernel<64>;
        if (set_kernel_smem((const void*)kern, TcRing<64>::kSmem) != CSMKV_OK) return CSMKV_ERR_CUDA;
        kern<<<grid, kTcThreads, TcRing<64>::kSmem, st>>>(P, tmK, tmV, tmN, tmKs, tmVs);
    }
    return cudaGetLastError() == cudaSuccess ? CSMKV_OK : CSMKV_ERR_CUDA;
}

}  // namespace csmkv
