// prefill_attn.cu -- the prompt's causal attention on the tensor cores, with the
// first Chunked Soft Matching round fused into it (bf16, head_dim 128, chunks of
// 256 rows). [Chelsea §三 算法流程, Algorithm 1: 预填充 O = FlashAttn(Q,K,V), then
// the first Chelsea(K,V,N,s,...) round; §三 分块软匹配算法 steps 1-4]
//
// One CTA per (128-row query block, query head). Row tiles of 128 start at
// off = (n1 mod 128) - 128 (0 when 128 divides n1), so a chunk (256 rows from
// n1 + 256 j) is exactly two key tiles, and query block i and key tile i cover the
// same rows (the diagonal, where the causal mask cuts).
// Warp roles during the attention:
//   warp 0     TMA (two lanes): the query block once, then K tiles and V tiles through
//              2-stage rings released separately (K after Q K^T, V after P V);
//   warp 1     tcgen05.mma from one thread, by readiness: S = Q K^T into one of two
//              TMEM buffers (128 columns each) up to two tiles ahead of the softmax, and
//              O += P V into a third, P read from tensor memory; the warp's lanes zero
//              V rows past the prompt before they are used (they may hold anything);
//   warps 4-7  the online softmax, one thread per query row (its TMEM lane): one
//              128-column load of the row's scores, row max, P = 2^(x - m) packed as
//              bf16 pairs and stored over the first 64 columns of the same S buffer
//              (the A operand of P V), row sums; O is rescaled in TMEM only when the row
//              max has grown by more than 2^8 since the last rescale (until then
//              P <= 2^8, exact in bf16's range), and divided by the row sum at the end.
// The degrees of a prompt are all 1, so there is no log-degree term here.
// Cache output, by the CTA of query head h with h mod G == 0 of each KV head:
// when its diagonal tile is the second tile of chunk j it runs the chunk's CSM
// round on the two tiles still in its ring -- K copied into the A/B parity layout
// for the similarity MMA, merges read straight from the ring -- and writes the
// chunk's output rows to the second cache; sink, remainder and recent rows are
// copied there by the CTA whose diagonal tile holds them. The decisions and the
// merged rows are those of the standalone tensor-core round on the same rows.
#include "csm_common.cuh"

namespace csmkv {

constexpr int kPfThreads = 256;
constexpr int kPfTile = 128;      // query rows per block = key rows per tile
constexpr int kPfTileBytes = 32768;  // 128 rows x 128 bf16 (two 64-column boxes)
constexpr float kPfLazy = 8.0f;   // log2 of the growth of the row max tolerated before a rescale

constexpr int kOffQ = 0;                          // query block, later the CSM parity slot (with P0)
constexpr int kOffP = kOffQ + kPfTileBytes;       // the fused round's: with the query block, its parity slot,
constexpr int kOffK0 = kOffP + 2 * kPfTileBytes;  // rings: K0 V0 K1 V1
constexpr int kOffTables = kOffP + kPfTileBytes;  // then its tables and the prompt degrees
constexpr int kOffOnes = kOffTables + (int)sizeof(CsmTables);
constexpr int kOffBars = kOffK0 + 4 * kPfTileBytes;
static_assert(kOffOnes + 256 * 4 <= kOffK0, "CSM tables fit in the second P buffer");

struct PfParams {
    const int32_t* seq_len;  // [batch] prompt rows per sequence, or null (all n)
    int32_t n;               // rows of q per head
    int32_t batch, h_kv, h_q, G, cap;
    int32_t T;               // query blocks per head
    int32_t off;             // first row of tile 0 (<= 0)
    float scale_log2;        // softmax scale * log2(e)
    __nv_bfloat16* out;      // [batch][h_q][n][128]
    // the second cache (null Ko: attention only)
    __nv_bfloat16* Ko;
    __nv_bfloat16* Vo;
    int32_t* No;
    int32_t* leno;
    int32_t cap_out, n1, n2, c, m;  // m == 0: no round (every row copied)
    const uint8_t* head_mask;       // [h_kv] 1 = outlier head (copied), or null
    WsHeader* hdr;
    int64_t timeout_ns;
};

struct alignas(8) PfBars {
    uint64_t q_full;
    uint64_t k_full[2], v_full[2], k_empty[2], v_empty[2];
    uint64_t s_full[2], s_empty[2];
    uint64_t p_full[2], pv_done[2], csm_mma, drain;
    uint32_t tmem;
    int32_t err;
};

constexpr int kPfSmem = kOffBars + (int)sizeof(PfBars) + 1024;  // + alignment of the base to 1 KB
static_assert(kOffTables % 16 == 0 && kOffBars % 8 == 0, "shared-memory layout alignment");

// Shared-memory descriptor of an MN-major operand in the 128-byte swizzle layout:
// 64 contiguous elements (128 bytes) along M/N per row, rows consecutive along K
// in 8-row atoms 1024 bytes apart (SBO), the next 64 elements along M/N `lbo`
// bytes further (LBO).
__device__ __forceinline__ uint64_t smem_desc_mn_sw128(uint32_t saddr, uint32_t lbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFF);
    d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// 32 lanes x 32 consecutive fp32 columns written back to TMEM (thread i: lane base + i).
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const float (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// 32 lanes x 128 consecutive 32-bit columns (thread i: lane base + i), completed
// (tcgen05.wait::ld) inside the same statement, so no use can move above the wait.
__device__ __forceinline__ void tmem_ld_32x32b_x128(uint32_t taddr, uint32_t (&r)[128]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x128.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%128];\n"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
        : "r"(taddr)
        : "memory");
}

// 2^x on the MUFU unit (ex2.approx, flush-to-zero; 2^-inf = +0).
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 32 lanes x 64 consecutive 32-bit columns from r[0..63] (thread i: lane base + i),
// completed (tcgen05.wait::st) inside the same statement.
__device__ __forceinline__ void tmem_st_32x32b_x64(uint32_t taddr, const uint32_t (&r)[128]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64};\n"
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]), "r"(r[32]), "r"(r[33]), "r"(r[34]), "r"(r[35]), "r"(r[36]), "r"(r[37]), "r"(r[38]), "r"(r[39]), "r"(r[40]), "r"(r[41]), "r"(r[42]), "r"(r[43]), "r"(r[44]), "r"(r[45]), "r"(r[46]), "r"(r[47]), "r"(r[48]), "r"(r[49]), "r"(r[50]), "r"(r[51]), "r"(r[52]), "r"(r[53]), "r"(r[54]), "r"(r[55]), "r"(r[56]), "r"(r[57]), "r"(r[58]), "r"(r[59]), "r"(r[60]), "r"(r[61]), "r"(r[62]), "r"(r[63])
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]^T, kind::f16: A (M rows in TMEM lanes, two 16-bit
// elements per 32-bit column along K) is read from tensor memory.
__device__ __forceinline__ void tc_mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n"
        " setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Bounded mbarrier wait by a whole warp, with one outcome for all its lanes (the
// warp goes on to .sync.aligned tcgen05 instructions).
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, uint64_t deadline) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, deadline)) != 0;
}

// Byte offset of 16-byte piece k (0..15) of row r in a 128-row tile of two 64-column
// boxes in the 128-byte swizzle layout.
__device__ __forceinline__ int tile_piece(int r, int k) {
    return (k >> 3) * 16384 + r * 128 + (((k & 7) ^ (r & 7)) << 4);
}

__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_attn_kernel(const __grid_constant__ PfParams p, const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV) {
    using T = __nv_bfloat16;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* const sb = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* const sQ = sb + kOffQ;
    CsmTables& sm = *reinterpret_cast<CsmTables*>(sb + kOffTables);
    int32_t* const ones = reinterpret_cast<int32_t*>(sb + kOffOnes);
    PfBars& br = *reinterpret_cast<PfBars*>(sb + kOffBars);
    auto sK = [&](int st) { return sb + kOffK0 + st * 2 * kPfTileBytes; };
    auto sV = [&](int st) { return sb + kOffK0 + st * 2 * kPfTileBytes + kPfTileBytes; };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nqh = p.batch * p.h_q;
    const int i = p.T - 1 - (int)(blockIdx.x / (unsigned)nqh);  // longest query blocks first
    const int qh = (int)(blockIdx.x % (unsigned)nqh);
    const int b = qh / p.h_q, h = qh - b * p.h_q, kvh = h / p.G;
    const int u = b * p.h_kv + kvh;
    const int s = p.seq_len ? max(0, min(p.seq_len[b], p.n)) : p.n;  // prompt rows of this sequence
    const int row0 = p.off + i * kPfTile;  // first row of query block i and of key tile i
    int32_t* const status = &p.hdr->status;
    const bool writer = p.Ko != nullptr && h % p.G == 0;  // this CTA writes the second cache
    const bool active = p.m > 0 && !(p.head_mask && p.head_mask[kvh]);
    const int ch = active ? max(0, (s - p.n1 - p.n2) / p.c) : 0;  // full chunks of the round
    if (writer && i == 0 && tid == 0) p.leno[u] = s - ch * p.m;
    if (row0 >= s) return;  // no prompt row in this block

    if (tid == 0) {
        mbar_init(&br.q_full, 1);
        for (int k = 0; k < 2; ++k) {
            mbar_init(&br.k_full[k], 1);
            mbar_init(&br.v_full[k], 1);
            mbar_init(&br.k_empty[k], 1);
            mbar_init(&br.v_empty[k], 1);
            mbar_init(&br.s_full[k], 1);
            mbar_init(&br.s_empty[k], 4);
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(&br.p_full[k], 4);
            mbar_init(&br.pv_done[k], 1);
        }
        mbar_init(&br.csm_mma, 1);
        mbar_init(&br.drain, 1);
        br.err = 0;
        fence_mbar_init();
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
    }
    if (warp == 0) {
        tmem_alloc(&br.tmem, 512);
        tmem_relinquish();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = br.tmem;
    const uint32_t tO = tmem + 256;
    auto tS = [&](int st) { return tmem + (uint32_t)(st * 128); };
    const uint64_t deadline = globaltimer() + (uint64_t)p.timeout_ns;
    volatile int32_t* const err = &br.err;
    auto fail = [&]() {
        record_status(status, CSMKV_ERR_TIMEOUT);
        *err = 1;
    };
    int last_load[2] = {-1, -1};  // warp 0 lanes 0 (K) and 1 (V): last tile loaded into each stage

    if (warp == 0) {
        // ------------------------------------------------------------ loads
        // lane 0: the query block, then K tiles (a stage is free once S = Q K^T of the tile
        // two before has completed); lane 1: V tiles (free once that tile's P V has)
        if (lane < 2) {
            const bool is_k = lane == 0;
            if (is_k) {
                mbar_expect_tx(&br.q_full, kPfTileBytes);
                tma_load_3d(sQ, &tmQ, &br.q_full, 0, row0, qh);
                tma_load_3d(sQ + 16384, &tmQ, &br.q_full, 64, row0, qh);
            }
            uint64_t* const empty = is_k ? br.k_empty : br.v_empty;
            uint64_t* const full = is_k ? br.k_full : br.v_full;
            const CUtensorMap* const map = is_k ? &tmK : &tmV;
            for (int t = 0; t <= i; ++t) {
                const int st = t & 1;
                if (t >= 2 && !mbar_wait(&empty[st], ((t >> 1) - 1) & 1, deadline)) {
                    fail();
                    break;
                }
                if (*err) break;
                const int r = p.off + t * kPfTile;
                uint8_t* const dst = is_k ? sK(st) : sV(st);
                mbar_expect_tx(&full[st], kPfTileBytes);
                tma_load_3d(dst, map, &full[st], 0, r, u);
                tma_load_3d(dst + 16384, map, &full[st], 64, r, u);
                last_load[st] = t;
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMAs (lane 0 issues)
        const uint32_t idS = idesc_bf16_f32(128, 128);
        const uint32_t idPV = idesc_bf16_f32(128, 128) | (1u << 16);  // B (V) is MN-major
        auto issue_S = [&](int t) {
            const int st = t & 1;
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const int box = ks >> 2, koff = (ks & 3) * 32;
                const uint64_t ad = smem_desc_sw128(smem_u32(sQ + box * 16384 + koff));
                const uint64_t bd = smem_desc_sw128(smem_u32(sK(st) + box * 16384 + koff));
                tc_mma_bf16(tS(st), ad, bd, idS, ks > 0 ? 1u : 0u);
            }
            tc_commit(&br.s_full[st]);
            tc_commit(&br.k_empty[st]);
        };
        // Issue order follows readiness: S = Q K^T of tile ns as soon as its K has landed
        // and its S buffer has been read (so S runs up to two tiles ahead of the softmax),
        // P V of tile np as soon as its P and V are in shared memory. Tests are
        // non-blocking and taken by the whole warp, so lane 0 never waits on one
        // barrier while the other operation is ready.
        bool ok = warp_wait(&br.q_full, 0, deadline);
        int ns = 0, np = 0;  // next S and next P V to issue
        while (ok && np <= i) {
            if (!__all_sync(0xffffffffu, !*err)) {
                ok = false;
                break;
            }
            bool did = false;
            if (np < ns) {
                const int st = np & 1;
                const bool ready = __all_sync(0xffffffffu, mbar_test(&br.p_full[st], (np >> 1) & 1) &&
                                                               mbar_test(&br.v_full[st], (np >> 1) & 1));
                if (ready) {
                    const int rt = p.off + np * kPfTile;
                    if (rt + kPfTile > s) {  // rows at or past the prompt's end: their V may hold anything
                        const int z0 = s - rt;  // first such row of the tile (> 0: the tile holds row s - 1)
                        for (int x = lane; x < (kPfTile - z0) * 16; x += 32) {
                            const int r = z0 + (x >> 4), k = x & 15;
                            *reinterpret_cast<uint4*>(sV(st) + tile_piece(r, k)) = make_uint4(0u, 0u, 0u, 0u);
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                    }
                    if (lane == 0) {
                        tc_fence_after();
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks) {  // 16 keys per step
                            const uint64_t bd = smem_desc_mn_sw128(smem_u32(sV(st) + ks * 2048), 16384);
                            tc_mma_bf16_ta(tO, tS(st) + (uint32_t)(ks * 8), bd, idPV, (np > 0 || ks > 0) ? 1u : 0u);
                        }
                        tc_commit(&br.pv_done[st]);
                        tc_commit(&br.v_empty[st]);
                    }
                    __syncwarp();
                    ++np;
                    did = true;
                }
            }
            if (ns <= i) {
                const int st = ns & 1;
                const bool ready = __all_sync(0xffffffffu, mbar_test(&br.k_full[st], (ns >> 1) & 1) &&
                                                               (ns < 2 || np >= ns - 1));
                if (ready) {
                    if (lane == 0) issue_S(ns);
                    __syncwarp();
                    ++ns;
                    did = true;
                }
            }
            if (!did) {
                if (globaltimer() > deadline) ok = false;
                __nanosleep(20);  // leave the issue slots to the softmax warp sharing this sub-partition
            }
        }
        if (!ok && lane == 0) fail();
    } else if (warp >= 4) {
        // ------------------------------------------------------------ online softmax
        const int qtr = warp & 3;
        const int r = qtr * 32 + lane;  // query row of the block = TMEM lane
        const int qrow = row0 + r;      // prompt position
        const uint32_t lo = (uint32_t)(qtr * 32) << 16;
        float m_run = -INFINITY, l = 0.f;
        bool ok = true;
        for (int t = 0; t <= i; ++t) {
            const int st = t & 1;
            ok = warp_wait(&br.s_full[st], (t >> 1) & 1, deadline);
            if (!__all_sync(0xffffffffu, ok && !*err)) break;
            tc_fence_after();
            uint32_t sv[128];  // the row's 128 scores of this tile, one pass over TMEM
            tmem_ld_32x32b_x128(tS(st) + lo, sv);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&br.s_empty[st]);  // S buffer st may take the tile after next
            const int k0 = p.off + t * kPfTile;
            const int jlo = max(0, -k0), jhi = min(kPfTile - 1, qrow - k0);  // visible columns (inclusive)
            if (__any_sync(0xffffffffu, jlo > 0 || jhi < kPfTile - 1)) {  // first or diagonal tile
#pragma unroll
                for (int j = 0; j < kPfTile; ++j)
                    if (j < jlo || j > jhi) sv[j] = 0xff800000u;  // -inf: weight 0, never the max
            }
            float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int j = 0; j < kPfTile; ++j) mq[j & 3] = fmaxf(mq[j & 3], __uint_as_float(sv[j]));
            const float m_tile = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3])) * p.scale_log2;
            float m_use = m_run, factor = 1.f;
            bool rescale = false;
            if (m_tile > m_run + kPfLazy) {
                m_use = m_tile;
                if (m_run != -INFINITY) {
                    rescale = true;
                    factor = ex2_approx(m_run - m_tile);
                }
            }
            // P buffer t & 1 is free once tile t - 2's P V has completed; O may be rescaled
            // once tile t - 1's has (P V of tile t cannot start before this P is written)
            if (t >= 2 && !warp_wait(&br.pv_done[st], ((t - 2) >> 1) & 1, deadline)) {
                ok = false;
                break;
            }
            const bool any_rescale = __any_sync(0xffffffffu, rescale);
            if (any_rescale && t >= 1 && !warp_wait(&br.pv_done[st ^ 1], ((t - 1) >> 1) & 1, deadline)) {
                ok = false;
                break;
            }
            tc_fence_after();
            if (any_rescale) {  // the TMEM accesses are warp-wide; factor is 1 elsewhere
                l *= factor;
#pragma unroll 1
                for (int cb = 0; cb < 4; ++cb) {
                    float v[32];
                    tmem_ld_32x32b_x32(tO + lo + (uint32_t)(cb * 32), v);
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] *= factor;
                    tmem_st_32x32b_x32(tO + lo + (uint32_t)(cb * 32), v);
                }
                tmem_st_wait();
            }
            const float mneg = m_use == -INFINITY ? 0.f : -m_use;  // a row with nothing visible: all 0
            const float sl = p.scale_log2;
            float ls[2] = {0.f, 0.f};
#pragma unroll
            for (int k = 0; k < 64; ++k) {  // pair k of the row's P, packed in place (sv[k] is free)
                const float p0 = ex2_approx(fmaf(__uint_as_float(sv[2 * k]), sl, mneg));
                const float p1 = ex2_approx(fmaf(__uint_as_float(sv[2 * k + 1]), sl, mneg));
                ls[k & 1] += p0 + p1;
                sv[k] = pack_bf16x2(p0, p1);
            }
            l += ls[0] + ls[1];
            // P into the S buffer's first 64 columns: the A operand of P V, read from TMEM
            tmem_st_32x32b_x64(tS(st) + lo, sv);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&br.p_full[st]);
            m_run = m_use;
        }
        if (ok) ok = __all_sync(0xffffffffu, !*err) && warp_wait(&br.pv_done[i & 1], (i >> 1) & 1, deadline);
        if (ok) {
            tc_fence_after();
            const bool valid = qrow >= 0 && qrow < s;
            const float inv = l > 0.f ? 1.0f / l : 0.f;
            T* const orow = p.out + ((size_t)qh * p.n + (size_t)(valid ? qrow : 0)) * 128;
#pragma unroll 1
            for (int cb = 0; cb < 4; ++cb) {
                float v[32];
                tmem_ld_32x32b_x32(tO + lo + (uint32_t)(cb * 32), v);
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) pk[e >> 1] = pack_bf16x2(v[e] * inv, v[e + 1] * inv);
                if (valid) {
                    uint4* const d = reinterpret_cast<uint4*>(orow + cb * 32);
#pragma unroll
                    for (int k = 0; k < 4; ++k) d[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
                }
            }
        }
        if (!ok && lane == 0) fail();
    }
    tc_fence_before();
    __syncthreads();

    // ---------------------------------------------------------------- second cache
    if (writer && !*err) {
        const int t0 = (p.n1 - p.off) / kPfTile;  // first tile of chunk 0
        const int rel = i - t0;
        if (rel >= 0 && rel < 2 * ch) {
            if (rel & 1) {  // chunk j = tiles i - 1 and i, both still in the ring
                const int j = rel >> 1;
                const uint8_t* const kt0 = sK((i - 1) & 1);
                const uint8_t* const kt1 = sK(i & 1);
                const uint8_t* const vt0 = sV((i - 1) & 1);
                const uint8_t* const vt1 = sV(i & 1);
                // K into the A/B parity layout of the similarity MMA (query and P buffers,
                // free now): A = even chunk rows (boxes at 0 and 16 KB), B = odd rows (32, 48 KB)
                uint8_t* const slot = sQ;
                for (int x = tid; x < 256 * 16; x += kPfThreads) {
                    const int q = x >> 4, k = x & 15;
                    const uint4 v = *reinterpret_cast<const uint4*>((q < 128 ? kt0 : kt1) + tile_piece(q & 127, k));
                    *reinterpret_cast<uint4*>(slot + (q & 1) * 32768 + tile_piece(q >> 1, k)) = v;
                }
                ones[tid] = 1;  // prompt degrees
                fence_proxy_async_smem();
                __syncthreads();
                if (tid == 32) {
                    tc_fence_after();
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        const int box = ks >> 2, koff = (ks & 3) * 32;
                        const uint64_t ad = smem_desc_sw128(smem_u32(slot + box * 16384 + koff));
                        const uint64_t bd = smem_desc_sw128(smem_u32(slot + 32768 + box * 16384 + koff));
                        tc_mma_bf16(tmem, ad, bd, idesc_bf16_f32(128, 128), ks > 0 ? 1u : 0u);
                    }
                    tc_commit(&br.csm_mma);
                }
                {   // fp32 inverse norms, one thread per chunk row (the standalone round's order)
                    const int op = (tid >> 3) & 1;
                    const int idx = (tid & 7) | ((tid >> 4) << 3);
                    const uint8_t* row = slot + op * 32768 + idx * 128;
                    float ss = 0.f;
#pragma unroll
                    for (int bx = 0; bx < 2; ++bx) {
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            float f[8];
                            Elem<T>::unpack(*reinterpret_cast<const uint4*>(row + bx * 16384 + ((k ^ (idx & 7)) << 4)), f);
#pragma unroll
                            for (int e = 0; e < 8; ++e) ss = fmaf(f[e], f[e], ss);
                        }
                    }
                    const float inv = ss > 0.f ? 1.0f / sqrtf(ss) : 0.0f;
                    if (op) sm.invB[idx] = inv; else sm.invA[idx] = inv;
                }
                __syncthreads();
                const bool okm = mbar_wait(&br.csm_mma, 0, globaltimer() + (uint64_t)p.timeout_ns);
                if (!__syncthreads_and(okm)) {
                    if (tid == 0) fail();
                } else {
                    tc_fence_after();
                    {   // per-A argmax over B of dot * invB, two halves of the B columns
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
                    chunk_tables(sm, ones, p.c, p.m, 2);
                    const int dst = p.n1 + j * (p.c - p.m);
                    const size_t orow = (size_t)u * p.cap_out + (size_t)dst;
                    emit_rows(p.Ko + orow * 128, p.c - p.m, 128, p.m, sm, ones,
                              [&](int q, int cc) { return (q < 128 ? kt0 : kt1) + tile_piece(q & 127, cc); });
                    emit_degrees(p.No + orow, p.c - p.m, p.m, sm, ones);
                    emit_rows(p.Vo + orow * 128, p.c - p.m, 128, p.m, sm, ones,
                              [&](int q, int cc) { return (q < 128 ? vt0 : vt1) + tile_piece(q & 127, cc); });
                }
            }
        } else {  // sink, remainder or recent rows: copied (after the round's chunks, shifted down)
            const int rlo = max(row0, 0), rhi = min(row0 + kPfTile, s);
            const uint8_t* const kt = sK(i & 1);
            const uint8_t* const vt = sV(i & 1);
            for (int x = tid; x < (rhi - rlo) * 16; x += kPfThreads) {
                const int row = rlo + (x >> 4), k = x & 15, rr = row - row0;
                const int dst = row < p.n1 ? row : row - ch * p.m;
                const size_t o = ((size_t)u * p.cap_out + (size_t)dst) * 128 + (size_t)k * 8;
                *reinterpret_cast<uint4*>(p.Ko + o) = *reinterpret_cast<const uint4*>(kt + tile_piece(rr, k));
                *reinterpret_cast<uint4*>(p.Vo + o) = *reinterpret_cast<const uint4*>(vt + tile_piece(rr, k));
            }
            for (int row = rlo + tid; row < rhi; row += kPfThreads)
                p.No[(size_t)u * p.cap_out + (size_t)(row < p.n1 ? row : row - ch * p.m)] = 1;
        }
    }

    // ---------------------------------------------------------------- teardown
    __syncthreads();
    if (tid == 32) {  // every MMA (all issued by this thread) has completed before TMEM is freed
        tc_commit(&br.drain);
        (void)mbar_wait(&br.drain, 0, globaltimer() + (uint64_t)p.timeout_ns);
    }
    if (tid < 2) {  // after a timeout, loads still in flight land before the CTA leaves
        const uint64_t dl = globaltimer() + (uint64_t)p.timeout_ns;
        if (tid == 0) (void)mbar_wait(&br.q_full, 0, dl);
        uint64_t* const full = tid == 0 ? br.k_full : br.v_full;
        for (int st = 0; st < 2; ++st)
            if (last_load[st] >= 0) (void)mbar_wait(&full[st], (last_load[st] >> 1) & 1, dl);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace csmkv

using namespace csmkv;

extern "C" {

size_t prefill_workspace_bytes(void) { return kHeaderBytes; }

int prefill_attn_csm(const void* q, const void* K, const void* V, const csmkv_cache* cache, int32_t n,
                     const int32_t* seq_len, int32_t h_q, float scale, void* out, void* K_out, void* V_out,
                     int32_t* N_out, int32_t* len_out, const csmkv_cache* cache_out, int32_t n1, int32_t n2, int32_t c,
                     double r, const uint8_t* head_mask, void* workspace, size_t ws_bytes, void* stream) {
    int rc = check_cache(cache);
    if (rc != CSMKV_OK) return rc;
    if (!q || !K || !V || !out) return CSMKV_ERR_ARG;
    if (h_q <= 0 || h_q % cache->h_kv != 0 || n < 0 || n > cache->cap) return CSMKV_ERR_ARG;
    if (!(scale == scale)) return CSMKV_ERR_ARG;
    const bool write = K_out != nullptr;
    int32_t m = 0;
    if (write) {
        rc = check_cache(cache_out);
        if (rc != CSMKV_OK) return rc;
        if (!V_out || !N_out || !len_out) return CSMKV_ERR_ARG;
        if (cache_out->batch != cache->batch || cache_out->h_kv != cache->h_kv ||
            cache_out->head_dim != cache->head_dim || cache_out->dtype != cache->dtype || cache_out->cap < n)
            return CSMKV_ERR_ARG;
        if (n1 < 0 || n2 < 0 || !(r >= 0.0 && r <= 0.5) || c < 2 || (c & 1)) return CSMKV_ERR_ARG;
        m = csm_edges_per_chunk(r, c);
    }
    if (cache->dtype != CSMKV_BF16 || cache->head_dim != 128 || (write && c != 256)) return CSMKV_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(K) || !aligned16(V) || !aligned16(out)) return CSMKV_ERR_ALIGN;
    if (write && (!aligned16(K_out) || !aligned16(V_out) || !aligned16(N_out))) return CSMKV_ERR_ALIGN;
    if (!workspace || ws_bytes < kHeaderBytes) return CSMKV_ERR_WORKSPACE;
    if (!aligned16(workspace)) return CSMKV_ERR_ALIGN;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int32_t units = cache->batch * cache->h_kv;
    if (n == 0) {
        if (write && cudaMemsetAsync(len_out, 0, sizeof(int32_t) * (size_t)units, st) != cudaSuccess)
            return CSMKV_ERR_CUDA;
        return CSMKV_OK;
    }
    const int32_t off = (!write || n1 % 128 == 0) ? 0 : n1 % 128 - 128;
    const long long T = ((long long)n - off + 127) / 128;
    const long long grid = T * (long long)cache->batch * h_q;
    if (grid > 0x7FFFFFFFLL) return CSMKV_ERR_UNSUPPORTED;

    CUtensorMap tmQ{}, tmK{}, tmV{};
    const uint64_t qdims[3] = {128, (uint64_t)n, (uint64_t)cache->batch * (uint64_t)h_q};
    const uint64_t qstr[2] = {256, (uint64_t)n * 256};
    const uint64_t kdims[3] = {128, (uint64_t)cache->cap, (uint64_t)units};
    const uint64_t kstr[2] = {256, (uint64_t)cache->cap * 256};
    const uint32_t box[3] = {64, 128, 1};
    if (!encode_tiled(&tmQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), qdims, qstr, box,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tiled(&tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(K), kdims, kstr, box,
                      CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_tiled(&tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(V), kdims, kstr, box,
                      CU_TENSOR_MAP_SWIZZLE_128B))
        return CSMKV_ERR_CUDA;

    PfParams P{};
    P.seq_len = seq_len;
    P.n = n;
    P.batch = cache->batch;
    P.h_kv = cache->h_kv;
    P.h_q = h_q;
    P.G = h_q / cache->h_kv;
    P.cap = cache->cap;
    P.T = (int32_t)T;
    P.off = off;
    const float sc = scale > 0.f ? scale : 1.0f / sqrtf(128.0f);
    P.scale_log2 = sc * 1.4426950408889634f;
    P.out = static_cast<__nv_bfloat16*>(out);
    P.Ko = static_cast<__nv_bfloat16*>(K_out);
    P.Vo = static_cast<__nv_bfloat16*>(V_out);
    P.No = N_out;
    P.leno = len_out;
    P.cap_out = write ? cache_out->cap : 0;
    P.n1 = write ? n1 : 0;
    P.n2 = write ? n2 : 0;
    P.c = write ? c : 256;
    P.m = m;
    P.head_mask = head_mask;
    P.hdr = static_cast<WsHeader*>(workspace);
    P.timeout_ns = 2000000000LL;
    if (set_kernel_smem((const void*)prefill_attn_kernel, kPfSmem, true) != CSMKV_OK) return CSMKV_ERR_CUDA;
    prefill_attn_kernel<<<(unsigned)grid, kPfThreads, kPfSmem, st>>>(P, tmQ, tmK, tmV);
    return cudaGetLastError() == cudaSuccess ? CSMKV_OK : CSMKV_ERR_CUDA;
}

int prefill_attn(const void* q, const void* K, const void* V, const csmkv_cache* cache, int32_t n,
                 const int32_t* seq_len, int32_t h_q, float scale, void* out, void* workspace, size_t ws_bytes,
                 void* stream) {
    return prefill_attn_csm(q, K, V, cache, n, seq_len, h_q, scale, out, nullptr, nullptr, nullptr, nullptr,
                            nullptr, 0, 0, 256, 0.0, nullptr, workspace, ws_bytes, stream);
}

}  // extern "C"
