/*
 * csmkv.h -- C ABI of the GB300 (sm_103a) library for online KV-cache
 * clustering: Chunked Soft Matching (CSM) compression and degree-aware
 * ("log N") decode attention over the compressed cache.
 *
 * Defining sources (web pages on arXiv 2506.11418):
 *   [Chelsea]    "Chelsea: Efficient Long-Context LLM Inference via KV Cache
 *                Clustering" (xllm-io paper review): §三 核心公式 (attention with
 *                cluster degrees), §三 算法流程 (Algorithm 1, the inference
 *                pipeline), §三 分块软匹配算法 (CSM steps 1-4), §三 理论分析
 *                (Theorem 6.1), §三 Outlier Heads处理.
 *   [CentroidKV] "CentroidKV: Efficient Long-Context LLM Inference via KV Cache
 *                Clustering" (gist.science explainer), 技术摘要: 推理流水线,
 *                分块软匹配 (CSM) incl. 渐进式调度, 聚合.
 *
 * Conventions for every call below
 *   - Memory: the caller owns every buffer. Device pointers must come from
 *     device memory of the current CUDA device. The library never allocates.
 *   - Cache layout (csmkv_cache): K and V are [batch][h_kv][cap][head_dim]
 *     row-major in the cache dtype, N (cluster degrees) is int32
 *     [batch][h_kv][cap], len is int32 [batch][h_kv] (rows in use per
 *     (sequence, KV head)). A layer stack folds into batch. K, V, N bases must
 *     be 16-byte aligned; cap must be a multiple of 8 and head_dim a multiple
 *     of 8 with head_dim <= 128.
 *   - Execution: every device call is asynchronous on `stream` (a
 *     cudaStream_t; NULL is the legacy default stream). Nothing synchronises
 *     the host and nothing reads device memory back, so calls can be issued
 *     back to back or captured into a CUDA graph.
 *   - Errors: argument errors return a csmkv_status synchronously without
 *     launching anything. Errors found on the device (a full cache on append,
 *     a bounded wait that ran out) are recorded, first one wins, in the status
 *     word at offset 0 of the call's workspace; read it with
 *     csmkv_device_status(), reset it with csmkv_clear_status(). A new
 *     workspace must be zero-filled once before its first use. No kernel
 *     traps or spins without bound.
 *   - Workspaces: a workspace serves one call at a time; calls that share a
 *     workspace must be ordered on one stream.
 */
#ifndef CSMKV_H
#define CSMKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CSMKV_OK = 0,
    CSMKV_ERR_ARG = 1,         /* an argument is out of its documented range */
    CSMKV_ERR_DTYPE = 2,       /* unknown dtype */
    CSMKV_ERR_ALIGN = 3,       /* a pointer or a size breaks the alignment rules */
    CSMKV_ERR_CAPACITY = 4,    /* device: append into a cache with len == cap */
    CSMKV_ERR_WORKSPACE = 5,   /* workspace NULL or smaller than the query says */
    CSMKV_ERR_TIMEOUT = 6,     /* device: a bounded wait ran out; that work was skipped */
    CSMKV_ERR_CUDA = 7,        /* a CUDA runtime call failed */
    CSMKV_ERR_UNSUPPORTED = 8  /* valid arguments no kernel here covers (e.g. h_q/h_kv > 8 on bf16) */
} csmkv_status;

typedef enum { CSMKV_BF16 = 0, CSMKV_F32 = 1 } csmkv_dtype;

typedef struct {
    int32_t batch;    /* independent sequences (times layers, when a stack is folded in) */
    int32_t h_kv;     /* KV heads per sequence */
    int32_t head_dim; /* d */
    int32_t cap;      /* rows allocated per (sequence, KV head) */
    int32_t dtype;    /* csmkv_dtype of K, V, q, k_new, v_new and the attention output */
} csmkv_cache;

/* ------------------------------------------------------------------------
 * Chunked Soft Matching, one round   [Chelsea §三 分块软匹配算法 steps 1-4;
 *                                     CentroidKV 分块软匹配 (CSM), 聚合]
 *
 * For every (sequence b, KV head h) with head_mask[h] == 0 and (seq_mask ==
 * NULL or seq_mask[b] != 0), on its first s = len[b][h] rows:
 *   - rows [0, n1) (attention sinks) and the last n2 rows (recent tokens) are
 *     never merged; the middle [n1, s - n2) is cut into ch = floor((s-n1-n2)/c)
 *     full chunks starting at row n1; a shorter remainder is left as it is;
 *   - inside a chunk, A = even offsets, B = odd offsets (Theorem 6.1);
 *   - each A token takes argmax_b cos(k_a, k_b) over the B tokens of its
 *     chunk (keys only; cos = 0 for a zero key; ties -> lowest b);
 *   - the m = floor(r*c + 1e-9) edges with the largest similarity are
 *     selected (ties -> lowest a);
 *   - every B token with selected edges becomes the degree-weighted mean of
 *     itself and its A tokens, k = sum n_i k_i / sum n_i, likewise v,
 *     n = sum n_i (pre-round values, fp32 arithmetic, rounded once to the
 *     cache dtype); several A tokens may merge into one B;
 *   - the selected A rows are removed and K, V, N are compacted in place in
 *     original order (sinks, chunks, remainder, recent window);
 *   - len[b][h] -= ch * m.
 * Units that are masked, or have no full chunk, are untouched.
 *
 * K, V, N, len: device, in/out (layout above).
 * n1, n2 >= 0; c even with 2 <= c <= 256; 0 <= r <= 0.5 (at most half of a
 * chunk merges, as the pages state). r == 0 is a no-op.
 * head_mask: device uint8 [h_kv], 1 = outlier head (left uncompressed), or
 *   NULL (no outliers). The mask is a property of the layer's heads and is
 *   shared by every sequence of the batch [Chelsea §三 Outlier Heads处理].
 * seq_mask: device uint8 [batch], nonzero = compress this sequence in this
 *   call, or NULL (all). Lets a ragged batch compress only the sequences
 *   whose trigger fired.
 * workspace: device, >= csm_workspace_bytes(cache, n1, n2, c) bytes,
 *   zero-filled before its first use, not touched by anything else between
 *   calls except csmkv_clear_status.
 * bf16 with c == 256 and head_dim in {64, 128} runs the similarity tile on
 * the tensor cores (tcgen05, fp32 accumulate); every other shape, and f32,
 * runs it on fp32 CUDA cores.
 * ---------------------------------------------------------------------- */
size_t csm_workspace_bytes(const csmkv_cache* cache, int32_t n1, int32_t n2, int32_t c);

int csm_compress(void* K, void* V, int32_t* N, int32_t* len, const csmkv_cache* cache,
                 int32_t n1, int32_t n2, int32_t c, double r,
                 const uint8_t* head_mask, const uint8_t* seq_mask,
                 void* workspace, size_t ws_bytes, void* stream);

/* Extra controls for csm_compress_ex. Zero-initialise for the defaults. */
typedef struct {
    int64_t wait_timeout_ns;  /* bound on each device-side wait; <= 0 -> 2 s */
    int32_t withhold_signals; /* test hook: work items never publish their "loaded"
                                 flags, so every wait on another item runs into the
                                 timeout and reports CSMKV_ERR_TIMEOUT (the cache is
                                 then partly compacted and must be discarded) */
    int32_t kernel;           /* which compression kernel runs (CSM_KERNEL_*) */
    const int32_t* seq_max_chunks; /* device [batch] or NULL. Budget-exact rounds:
                                 entry b > 0 processes only the first (oldest)
                                 min(entry, full chunks) chunks of sequence b;
                                 every later row, unprocessed chunks included,
                                 moves down unchanged and len -= chunks * m.
                                 <= 0 or NULL: every full chunk (the pages'
                                 Algorithm 1). See csm_chunks_to_budget. */
} csm_options;

/* csm_options.kernel. AUTO picks a tensor-core kernel where the shape allows
 * one (bf16, c == 256, head_dim in {64, 128}) and the CUDA-core kernel
 * elsewhere; asking for a tensor-core kernel on another shape falls back to
 * the CUDA-core kernel. All choices give the same decisions and outputs up to
 * the order of fp32 rounding in the similarity scores. */
#define CSM_KERNEL_AUTO 0
#define CSM_KERNEL_SIMT 1    /* fp32 CUDA cores, one persistent CTA per SM */
/* (value 2 is not used: any value other than those listed is CSMKV_ERR_ARG) */
#define CSM_KERNEL_TC_SPLIT 3 /* tcgen05, three CTAs per SM with one slot each */

/* csm_compress plus two optional outputs/controls:
 * match_out: device int32 [batch*h_kv][csm_max_chunks(...)][c/2] or NULL.
 *   For every processed chunk j of unit u, entry [u][j][a] receives the B index
 *   (0..c/2-1) that A token a merged into, or -1. Entries of chunks that were
 *   not processed are left untouched.
 * opts: NULL for defaults. */
int csm_compress_ex(void* K, void* V, int32_t* N, int32_t* len, const csmkv_cache* cache,
                    int32_t n1, int32_t n2, int32_t c, double r,
                    const uint8_t* head_mask, const uint8_t* seq_mask,
                    int32_t* match_out, const csm_options* opts,
                    void* workspace, size_t ws_bytes, void* stream);

/* Full chunks that fit in cap: max(0, (cap - n1 - n2) / c). */
int32_t csm_max_chunks(const csmkv_cache* cache, int32_t n1, int32_t n2, int32_t c);

/* ------------------------------------------------------------------------
 * Decode append   [Chelsea §三 算法流程, Algorithm 1 decode update]
 * K=[K,k], V=[V,v], N=[N,1], s=s+1 for every (sequence, KV head) whose
 * sequence is selected (seq_mask NULL = all). k_new, v_new: device
 * [batch][h_kv][head_dim] in the cache dtype. A unit with len == cap is left
 * unchanged and CSMKV_ERR_CAPACITY is recorded in the workspace status word.
 * workspace: device, >= csm_append_workspace_bytes() bytes (status only).
 * ---------------------------------------------------------------------- */
size_t csm_append_workspace_bytes(void);

int csm_append(void* K, void* V, int32_t* N, int32_t* len, const csmkv_cache* cache,
               const void* k_new, const void* v_new, const uint8_t* seq_mask,
               void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Degree-aware decode attention   [Chelsea §三 核心公式; CentroidKV 聚合]
 *   o_h = softmax(scale * q_h K^T + log N) V
 *       = sum_t n_t exp(scale q_h.k_t) v_t / sum_t n_t exp(scale q_h.k_t)
 * over the first len rows of KV head floor(h / G) of the same sequence,
 * G = h_q / h_kv (contiguous query-head groups, GQA).
 * q: device [batch][h_q][head_dim]; out: device [batch][h_q][head_dim], both
 * in the cache dtype; K, V, N, len read only. A unit with len == 0 gives a
 * zero output. scale is normally 1/sqrt(head_dim).
 * h_q must be a positive multiple of h_kv; bf16 needs G <= 8 and head_dim in
 * {64, 128} (CSMKV_ERR_UNSUPPORTED otherwise).
 * workspace: device, >= decode_attn_workspace_bytes(cache, h_q) bytes.
 * Work: every unit's rows are cut into fixed splits (boundaries depend only on
 * the lengths) that a persistent grid takes from an atomic ticket, long units
 * first, so ragged lengths and uneven SM bandwidth stay balanced; a second
 * kernel merges each unit's per-split softmax states in split order. Results do
 * not depend on which CTA ran which split (repeated calls are bit-identical).
 * ---------------------------------------------------------------------- */
size_t decode_attn_workspace_bytes(const csmkv_cache* cache, int32_t h_q);

int decode_attn_logn(const void* q, const void* K, const void* V, const int32_t* N,
                     const int32_t* len, const csmkv_cache* cache, int32_t h_q, float scale,
                     void* out, void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * One fused decode step: append, then attend   [Chelsea §三 算法流程,
 *                                               Algorithm 1 decode update]
 * Equivalent to csm_append(k_new, v_new) followed by decode_attn_logn on the
 * same stream, with the same results bit for bit, in one kernel for bf16: the
 * new token's K, V row and degree 1 are written at row len of every unit by
 * the CTA whose share of the tokens holds that row (just before it loads the
 * row), the unit is attended with len + 1 rows, and the last CTA to finish
 * sets len += 1. A unit with len == cap is attended unchanged and
 * CSMKV_ERR_CAPACITY is recorded in the workspace status word. fp32 caches
 * run the two kernels back to back.
 * k_new, v_new: device [batch][h_kv][head_dim] in the cache dtype; K, V, N,
 * len: device, in/out; q, out, scale, workspace as for decode_attn_logn (the
 * same workspace size).
 * ---------------------------------------------------------------------- */
int decode_step_logn(const void* q, const void* k_new, const void* v_new, void* K, void* V, int32_t* N,
                     int32_t* len, const csmkv_cache* cache, int32_t h_q, float scale, void* out,
                     void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * Decode attention without a caller-provided workspace.
 * (The pages have no counterpart: this is a deployment convenience.)
 *
 * For callers that cannot allocate device memory -- code running after the
 * host application has reserved all device memory, plugins that do not own
 * the CUDA allocator, services whose memory budget is fixed before the first
 * request. Same computation, arguments and layouts as decode_attn_logn, minus
 * the workspace: the scratch is a fixed 16 MiB array inside the library, one
 * per GPU that loads it, held until the process exits.
 *  - Capacity: returns CSMKV_ERR_WORKSPACE when decode_attn_workspace_bytes(
 *    cache, h_q) exceeds 16 MiB (at head_dim 128 on 152 SMs: about 5500
 *    (sequence, KV head) units with 4 query heads per KV head, 1600 with 8).
 *    Nothing is launched then.
 *  - The first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress) and caches it; make that first call before any
 *    stream capture.
 *  - Every call zero-fills the part of the array it uses, asynchronously on
 *    `stream`, then runs decode_attn_logn on it. The library allocates
 *    nothing.
 *  - All calls on a device share the one array: calls that overlap on the GPU
 *    (different streams, no ordering between them) race and give wrong
 *    results. Device-side errors are recorded in the array's status word and
 *    cleared by the next call; use decode_attn_logn with a workspace when
 *    they must be read back.
 * ---------------------------------------------------------------------- */
int decode_attn_logn_noalloc(const void* q, const void* K, const void* V, const int32_t* N,
                             const int32_t* len, const csmkv_cache* cache, int32_t h_q, float scale,
                             void* out, void* stream);

/* ------------------------------------------------------------------------
 * Paged (block-table) cache layout   [CentroidKV 技术摘要, 结果: the method
 *                                     serving inside vLLM's paged KV cache]
 *
 * Pages of page_rows rows are taken from one pool per array: K and V are
 * [num_pages][page_rows][head_dim] in the cache dtype, N is int32
 * [num_pages][page_rows]. Every (sequence, KV head) unit u owns the pages its
 * block table lists: logical row r of unit u lives in pool row
 *     table[u * max_pages + r / page_rows] * page_rows + r % page_rows.
 * The csmkv_cache descriptor describes the logical cache as for the dense
 * layout, with cap = max_pages * page_rows; len stays [batch][h_kv]. A page
 * may belong to at most one (unit, logical page): compression compacts every
 * unit in place through its own pages. Pages past a unit's rows need not be
 * listed (any value); a listed page that the call touches must be in
 * [0, num_pages): an access through an entry outside it is skipped and
 * CSMKV_ERR_ARG recorded in the workspace status word.
 * page_rows: a multiple of 64, >= 64. Pools 16-byte aligned.
 * ---------------------------------------------------------------------- */
typedef struct {
    const int32_t* table; /* device int32 [batch * h_kv][max_pages] */
    int32_t page_rows;
    int32_t max_pages;
    int32_t num_pages;    /* pages in each pool */
} csmkv_pages;

/* csm_append on a paged cache (any dtype). */
int csm_append_paged(void* K, void* V, int32_t* N, int32_t* len, const csmkv_cache* cache, const csmkv_pages* pages,
                     const void* k_new, const void* v_new, const uint8_t* seq_mask, void* workspace, size_t ws_bytes,
                     void* stream);

/* csm_compress_ex on a paged cache: the same round, decisions and results (bit
 * for bit, given the same decisions) as on the dense layout. Tensor-core shapes
 * only (bf16, c == 256, head_dim in {64, 128}; CSMKV_ERR_UNSUPPORTED
 * otherwise); workspace as csm_workspace_bytes(cache, ...) with the logical
 * cap. match_out and opts as for csm_compress_ex (opts->kernel is ignored). */
int csm_compress_paged(void* K, void* V, int32_t* N, int32_t* len, const csmkv_cache* cache, const csmkv_pages* pages,
                       int32_t n1, int32_t n2, int32_t c, double r, const uint8_t* head_mask, const uint8_t* seq_mask,
                       int32_t* match_out, const csm_options* opts, void* workspace, size_t ws_bytes, void* stream);

/* decode_attn_logn / decode_step_logn on a paged cache (bf16 only;
 * CSMKV_ERR_UNSUPPORTED otherwise); workspace as decode_attn_workspace_bytes. */
int decode_attn_logn_paged(const void* q, const void* K, const void* V, const int32_t* N, const int32_t* len,
                           const csmkv_cache* cache, const csmkv_pages* pages, int32_t h_q, float scale, void* out,
                           void* workspace, size_t ws_bytes, void* stream);
int decode_step_logn_paged(const void* q, const void* k_new, const void* v_new, void* K, void* V, int32_t* N,
                           int32_t* len, const csmkv_cache* cache, const csmkv_pages* pages, int32_t h_q, float scale,
                           void* out, void* workspace, size_t ws_bytes, void* stream);

/* ------------------------------------------------------------------------
 * The decode loop, issued natively   [Chelsea §三 算法流程, Algorithm 1
 *                                     (decode phase); CentroidKV 技术摘要:
 *                                     推理流水线]
 *
 * Runs decode steps i = first_step .. first_step + steps - 1 (1-based) of the
 * serving loop back to back on one stream, each exactly as the separate calls
 * would:
 *     csm_append(k_new[i-1], v_new[i-1])           K=[K,k], V=[V,v], N=[N,1]
 *     decode_attn_logn(q[i-1]) -> out[i-1]
 *     csm_compress_ex(r) for every planned round with step == i, in order
 * The trigger test s >= B + g and the ratio schedule stay with the caller
 * (csm_should_trigger, csm_ratio): lengths after append and compression are
 * known on the host without reading the device, so the caller lists the
 * rounds up front. Issuing the loop from here keeps host time per step far
 * below the GPU time of the step, which a per-call binding from an
 * interpreter does not.
 *
 * q, out: device [steps_total][batch][h_q][head_dim]; k_new, v_new: device
 *   [steps_total][batch][h_kv][head_dim], all in the cache dtype; step i uses
 *   slice i-1.
 * rounds: host array of n_rounds entries with step >= 1, sorted by step;
 *   entries outside the steps run here are ignored. seq_mask as in
 *   csm_compress (device, or NULL).
 * Workspaces as for the separate calls, each zero-filled before first use.
 * attn_events / csm_events: NULL, or host arrays of cudaEvent_t (2 per
 *   attention call, 2 per round, in issue order; index 2k and 2k+1 for the
 *   k-th call of this invocation), recorded on `stream` right before and
 *   right after that call, for per-call device timing.
 * l2_flush, l2_flush_bytes: NULL/0, or a device buffer (16-byte aligned, size
 *   a multiple of 16) that is read in full before every attention call
 *   (outside the attention events), so that each call reads the cache from HBM
 *   rather than from the previous call's L2 residue; for cold-cache timing of
 *   caches smaller than about twice L2. The buffer is only read, so L2 holds
 *   no dirty lines afterwards.
 * Returns the first error of any call (nothing after it is issued).
 * Everything is enqueued on `stream` without host synchronisation, so a call
 * with attn_events, csm_events and l2_flush all NULL can be captured into a
 * CUDA graph (after one direct call has set the kernels' attributes) and the
 * graph replayed on the same buffers.
 * ---------------------------------------------------------------------- */
typedef struct {
    int32_t step;            /* decode step after whose attention the round runs (>= 1) */
    double r;                /* merge ratio of the round */
    const uint8_t* seq_mask; /* device [batch], nonzero = compress; NULL = all */
    const int32_t* seq_max_chunks; /* device [batch] or NULL: as csm_options.seq_max_chunks */
} csm_round_plan;

typedef struct {
    void* K;
    void* V;
    int32_t* N;
    int32_t* len;
    csmkv_cache cache;
    int32_t h_q;
    float scale;
    const void* q;
    const void* k_new;
    const void* v_new;
    void* out;
    int32_t n1, n2, c;
    const uint8_t* head_mask;
    int32_t csm_kernel; /* csm_options.kernel for every round */
    const csm_round_plan* rounds;
    int32_t n_rounds;
    void* ws_csm;
    size_t ws_csm_bytes;
    void* ws_append;
    size_t ws_append_bytes;
    void* ws_attn;
    size_t ws_attn_bytes;
    void* const* attn_events;
    void* const* csm_events;
    void* l2_flush;
    size_t l2_flush_bytes;
    int32_t fused_append; /* nonzero: each step's append and attention run as one
                             decode_step_logn (ws_append unused) */
    const csmkv_pages* pages; /* NULL: dense layout; else every call uses the paged
                             entry points (fused_append must then be nonzero) */
} csm_decode_loop;

int csm_decode_run(const csm_decode_loop* loop, int32_t first_step, int32_t steps, void* stream);

/* ------------------------------------------------------------------------
 * Prefill attention, with the first CSM round fused into it
 *   [Chelsea §三 算法流程, Algorithm 1: 预填充 O = FlashAttn(Q,K,V), every degree
 *    N = 1; then, if s >= B + g, the first Chelsea(K,V,N,s,n1,n2,r,c) round]
 *
 * prefill_attn: for every sequence b, query head h and prompt position i < s_b,
 *   out[b][h][i] = softmax_{t <= i}(q[b][h][i] . K[b][h / G][t] * scale) V[b][h / G][t]
 *   (causal; G = h_q / h_kv query heads per KV head; no log-degree term, since
 *   every prompt degree is 1). Positions i >= s_b of out are not written.
 * prefill_attn_csm: the same attention, and, from the same K/V tiles while
 *   they are on chip, a second cache (K_out, V_out, N_out, len_out, layout
 *   `cache_out`) holding the prompt after one CSM round with ratio r: exactly
 *   what csm_compress (the tensor-core kernel) leaves in place on a cache
 *   whose first s_b rows are the prompt with N = 1 and len = s_b -- sinks, the
 *   chunks' output rows, remainder and recent window, N and len -- written
 *   out of place, because later query blocks still read the prompt's rows.
 *   Units of an outlier head (head_mask[h] = 1), units without a full chunk,
 *   and every unit when r gives m = 0 get the prompt unchanged (N = 1,
 *   len = s_b). Rows of the second cache past len_out are not written.
 *
 * q: device bf16 [batch][h_q][n][128]; K, V: device, the prompt's rows
 *   [0, n) of a cache (layout `cache`; bf16, head_dim 128; read only).
 * n: prompt rows per sequence (0 <= n <= cache->cap); seq_len: device int32
 *   [batch] with the sequences' own prompt lengths s_b (clamped to [0, n]),
 *   or NULL (s_b = n for all).
 * scale: softmax scale; <= 0 -> 1/sqrt(128).
 * out: device bf16 [batch][h_q][n][128].
 * cache_out: batch, h_kv, head_dim and dtype as `cache`, cap >= n; K_out,
 *   V_out, N_out (16-byte aligned) and len_out [batch][h_kv] are device and
 *   written only. n1, n2 >= 0, 0 <= r <= 0.5 and c == 256 (other c:
 *   CSMKV_ERR_UNSUPPORTED), as csm_compress.
 * head_mask: device uint8 [h_kv] or NULL, as csm_compress.
 * workspace: device, >= prefill_workspace_bytes(), zero-filled once (its
 *   status word records a bounded wait that ran out: CSMKV_ERR_TIMEOUT).
 * Returns CSMKV_ERR_UNSUPPORTED for dtypes other than bf16 or head_dim != 128.
 * Work: one 256-thread CTA per (128-row query block, query head), tcgen05
 * MMAs with fp32 accumulation in TMEM, bf16 softmax probabilities.
 * ---------------------------------------------------------------------- */
size_t prefill_workspace_bytes(void);

int prefill_attn(const void* q, const void* K, const void* V, const csmkv_cache* cache, int32_t n,
                 const int32_t* seq_len, int32_t h_q, float scale, void* out, void* workspace, size_t ws_bytes,
                 void* stream);

int prefill_attn_csm(const void* q, const void* K, const void* V, const csmkv_cache* cache, int32_t n,
                     const int32_t* seq_len, int32_t h_q, float scale, void* out, void* K_out, void* V_out,
                     int32_t* N_out, int32_t* len_out, const csmkv_cache* cache_out, int32_t n1, int32_t n2,
                     int32_t c, double r, const uint8_t* head_mask, void* workspace, size_t ws_bytes,
                     void* stream);

/* ------------------------------------------------------------------------
 * Host-side schedule helpers   [Chelsea §三 算法流程, Algorithm 1;
 *                               CentroidKV 分块软匹配 (CSM), 渐进式调度]
 * Pure functions; no device work.
 * ---------------------------------------------------------------------- */
double csm_budget(int64_t n, double R, int64_t Gamma);            /* B = R (n + Gamma) */
int csm_should_trigger(int64_t s, double B, int32_t g);           /* s >= B + g */
double csm_ratio(int32_t j, double r_init, double dr, double r_min); /* max(r_init - j dr, r_min) */
int32_t csm_edges_per_chunk(double r, int32_t c);                 /* floor(r c + 1e-9) */
int64_t csm_num_chunks(int64_t s, int32_t n1, int32_t n2, int32_t c); /* floor(max(0, s-n1-n2) / c) */
int64_t csm_len_after(int64_t s, int32_t n1, int32_t n2, int32_t c, int32_t m); /* s - chunks * m */
/* Budget-exact compression (an extension; the pages' Algorithm 1 compresses
 * every full chunk): the fewest oldest chunks whose merge brings s to <= B,
 * k = ceil((s - B) / m), at most the full chunks there are; 0 when s <= B or
 * m <= 0. After a prefill-sized round the cache then sits just under the
 * budget, and the trigger fires again after about m appends. */
int32_t csm_chunks_to_budget(int64_t s, double B, int32_t n1, int32_t n2, int32_t c, int32_t m);

/* ------------------------------------------------------------------------
 * Device status word (offset 0 of every workspace)
 * ---------------------------------------------------------------------- */
/* Synchronises `stream`, then returns the recorded csmkv_status (CSMKV_OK if
 * none), or CSMKV_ERR_CUDA if the read itself failed. */
int csmkv_device_status(const void* workspace, void* stream);
/* Enqueues a reset of the status word to CSMKV_OK on `stream`. */
int csmkv_clear_status(void* workspace, void* stream);
/* Static description of a status code. */
const char* csmkv_status_str(int status);

#ifdef __cplusplus
}
#endif

#endif /* CSMKV_H */
