/*
 * fp.h -- C ABI of the GB300 (sm_103a) FlashPrefill V2 block-sparse prefill
 * attention library (libfp.so).
 *
 * Method: "FlashPrefill V2: Block-Sparse Prefill Attention for Long-Context
 * LLM Serving" (arXiv 2608.19758). One attention layer runs in two calls:
 *
 *   fp_select     Stage 1 / index stage (Sec.3.1, Sec.3.3 "Single-Pass Score
 *                 and Selection", Alg.1 steps 1-5): block means of K and V
 *                 (Eq.5), pooled-key energies of every packed query tile
 *                 (Eq.19), the max-based threshold with forced sink / window /
 *                 diagonal blocks (Eq.3, Eq.20), compacted into a CSR index.
 *   fp_attention  Stage 2 / attention stage (Sec.3.2, Sec.3.3, Alg.1 steps
 *                 6-11): exact attention over the selected blocks, one
 *                 mean-correction term per pruned causal block (Eq.6), online
 *                 softmax, epilogue normalisation; BF16 or FP8-E4M3 (Eq.15).
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers unless a name starts with
 *     `host_`. The caller owns and allocates every buffer, the workspace
 *     included; the library allocates nothing and keeps no state between
 *     calls. Inputs are read-only; outputs are fully overwritten.
 *   - Work is enqueued asynchronously on `stream`; no call synchronises the
 *     host except fp_device_status. Results are deterministic for fixed
 *     inputs (bit-identical across runs, page placements and request orders).
 *   - Host-detected errors return a negative fp_status and enqueue nothing.
 *     Device-detected errors (a page id out of range, a malformed CSR, an
 *     index capacity overflow, an expired bounded wait) are recorded in the
 *     workspace's status word; the kernels never trap. fp_device_status
 *     reads it back.
 *
 * Lengths (Sec.3.4, Alg.1 inputs): request b brings L_b^q = cu_seqlens[b+1] -
 * cu_seqlens[b] new query tokens against L_b^kv >= L_b^q keys/values in the
 * paged cache (seqlens_kv; L_b^kv = L_b^q without a cached prefix). The new
 * tokens are the last L_b^q positions: query i of request b sits at absolute
 * position L_b^kv - L_b^q + i and attends causally to keys 0 .. that position
 * (chunked prefill, or prefill after a prefix-cache hit). Pooling, scoring and
 * the correction cover the whole KV.
 *
 * Layouts (row-major, innermost last)
 *   q          [T, Hq, 128] elements of `dtype`; T = cu_seqlens[batch]
 *   k_pages,   [num_pages, page_size, Hkv, 128] elements of `dtype`; token j
 *   v_pages      of request b lives in page page_table[b * stride + j / page_size]
 *                at slot j % page_size (Sec.3.3 "Paged and Variable-Length
 *                Execution", Eq.22), 0 <= j < L_b^kv. Slots past a request's KV
 *                length must hold finite values (they are multiplied by zero,
 *                never selected).
 *   out        [T, Hq, 128] bf16
 *   lse        [T, Hq] fp32, natural-log softmax denominator (optional)
 * q, k_pages, v_pages, kbar_op, vbar_op and out start on 16-byte boundaries
 * (TMA reads, 16-byte stores); lse, the means, the CSR arrays, the other
 * int32 outputs and the description's device int32 arrays on 4-byte ones. A
 * misaligned pointer is rejected with FP_ERR_INVALID_ARG before anything is
 * enqueued.
 *   kbar, vbar [num_blocks, Hkv, 128] fp32 block means; request b's blocks
 *                are rows blk_base(b) .. blk_base(b) + ceil(L_b^kv/128) - 1,
 *                blk_base(b) = sum_{b' < b} ceil(L_b'^kv/128)
 *   kbar_op,   [num_blocks, Hkv, 128] the same means in the operand format:
 *   vbar_op      bf16, or E4M3 of mean / c_k (resp. mean / c_v) for FP8
 *   CSR        one segment per (request b, KV head h, packed tile t), in that
 *                order (Sec.3.3 "Index-Driven Sparse Traversal"). Packed row
 *                r of Q' = PackGQA(Q) is absolute position floor(r/g) of query
 *                head h*g + r mod g (Eq.12-13); tiles are 128 rows on that
 *                absolute grid, so none straddles two blocks, and request b's
 *                tiles are those holding a query row r in
 *                [g (L_b^kv - L_b^q), g L_b^kv): tile t of the request is
 *                absolute tile t0(b) + t, t0(b) = floor(g (L_b^kv - L_b^q) /
 *                128) (t0 = 0 without a prefix). Its diagonal block is
 *                D = floor((t0(b) + t) / g). csr_cu [num_segments + 1] int32
 *                are offsets into csr_idx [capacity] int32, which lists each
 *                segment's selected 128-token block ids (relative to the
 *                request) ascending.
 *
 * Limits: head_dim = block_size = 128; g = Hq / Hkv a power of two <= 16;
 * page_size a power of two in [8, 128]; 0 <= L_b^q <= L_b^kv <= 1,048,576.
 */
#ifndef FP_H_
#define FP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The CUDA runtime's stream handle (cudaStream_t); NULL is the legacy stream. */
typedef struct CUstream_st *fp_stream_t;

typedef enum {
    FP_OK = 0,
    /* detected on the host: nothing was enqueued */
    FP_ERR_INVALID_ARG = -1,      /* null or misaligned pointer, negative size, inconsistent description */
    FP_ERR_UNSUPPORTED = -2,      /* outside the limits listed above */
    FP_ERR_WORKSPACE = -3,        /* workspace smaller than fp_workspace_bytes() */
    FP_ERR_CUDA = -4,             /* a CUDA runtime call or kernel launch failed */
    FP_ERR_CAPACITY = -5,         /* CSR index capacity smaller than required */
    /* detected on the device: recorded in the workspace status word */
    FP_ERR_DEVICE_PAGE = -16,     /* a page id outside [0, num_pages) was needed */
    FP_ERR_DEVICE_CSR = -17,      /* CSR segment malformed (ids outside [0, D] or not ascending) */
    FP_ERR_DEVICE_OVERFLOW = -18, /* selected blocks exceed the CSR index capacity */
    FP_ERR_DEVICE_TIMEOUT = -19,  /* a bounded pipeline wait expired */
    FP_ERR_DEVICE_SEQLEN = -20    /* device cu_seqlens / seqlens_kv differ from their host copies */
} fp_status;

typedef enum { FP_DTYPE_BF16 = 0, FP_DTYPE_E4M3 = 1 } fp_dtype;

/* fp_attention flags */
#define FP_MEAN_CORRECTION 1 /* add the Eq.6 surrogate of every pruned causal block (off: Eq.4) */
#define FP_DENSE 2           /* ignore the CSR: every causal block is exact, no correction (alpha = 0) */

/* Description of one attention layer's batch (Alg.1 inputs: packed queries,
 * paged KV with page table, lengths {(L_b^q, L_b^kv)}). */
typedef struct {
    int32_t batch;                  /* number of requests (continuous batching) */
    int32_t num_q_heads;            /* Hq */
    int32_t num_kv_heads;           /* Hkv; g = Hq / Hkv (Eq.12) */
    int32_t head_dim;               /* d, must be 128 */
    int32_t block_size;             /* B, must be 128 */
    int32_t page_size;              /* p of Eq.22 */
    int32_t dtype;                  /* fp_dtype of q, k_pages, v_pages */
    float c_q, c_k, c_v;            /* per-tensor dequantisation scales (Eq.15); ignored for BF16 */
    const int32_t *cu_seqlens;      /* device [batch + 1], cu_seqlens[0] = 0, nondecreasing */
    const int32_t *page_table;      /* device [batch * page_table_stride] */
    int32_t page_table_stride;      /* entries per request row, >= ceil(max L_b^kv / page_size) */
    int32_t num_pages;              /* pages in the K/V pool (bounds checks) */
    const int32_t *host_cu_seqlens; /* host copy of cu_seqlens, read for sizing only */
    const int32_t *seqlens_kv;      /* device [batch] L_b^kv >= L_b^q, or NULL: L_b^kv = L_b^q */
    const int32_t *host_seqlens_kv; /* host copy of seqlens_kv (sizing only); NULL iff seqlens_kv is NULL */
} fp_problem;

/* Sizing (host only, no device work, no synchronisation). Each returns a
 * negative value if the description is invalid or unsupported. */

/* Bytes of device workspace fp_select and fp_attention need (256-byte aligned
 * base). One workspace may serve both calls of a layer; calls that overlap on
 * the device must use distinct workspaces. It includes 21 MB for the partial
 * outputs of KV splits (320 slots of 128 x 128 fp32). */
int64_t fp_workspace_bytes(const fp_problem *p);

/* Number of CSR segments: sum_b Hkv * n_b, n_b = ceil(g L_b^kv / 128) - t0(b)
 * tiles (0 when L_b^q = 0); without a prefix n_b = ceil(g L_b / 128). */
int64_t fp_num_segments(const fp_problem *p);

/* Rows of the pooled-mean arrays: sum_b ceil(L_b^kv / 128). */
int64_t fp_num_blocks(const fp_problem *p);

/* Worst-case CSR index entries, sum over segments of (D + 1) where D is the
 * tile's diagonal block; passing this capacity can never overflow. */
int64_t fp_csr_capacity(const fp_problem *p);

/* Stage 1 (Alg.1 steps 1-5). Pools K/V block means (Eq.5; FP8 inputs
 * descaled first), scores every packed 128-row query tile against the pooled
 * keys of its causal blocks J <= D with logits q.kbar_J / sqrt(d) (Eq.19),
 * keeps block J iff E_J >= alpha * max_{J' <= D} E_J' or J < sink_blocks or
 * D - window_blocks <= J < D or J = D (Eq.20), and writes the CSR.
 *   alpha          >= 0; 0 selects every causal block
 *   sink_blocks    >= 0 leading blocks always kept
 *   window_blocks  >= 0 blocks just before the diagonal block always kept
 *   csr_cu         out [num_segments + 1]
 *   csr_idx        out [csr_idx_capacity]; entries past csr_cu[num_segments] undefined
 *   kbar, vbar     out fp32 means; kbar_op, vbar_op out operand-format means
 *   workspace      device scratch of at least fp_workspace_bytes(p) bytes */
fp_status fp_select(const fp_problem *p, const void *q, const void *k_pages, const void *v_pages, float alpha,
                    int32_t sink_blocks, int32_t window_blocks, int32_t *csr_cu, int32_t *csr_idx,
                    int64_t csr_idx_capacity, float *kbar, float *vbar, void *kbar_op, void *vbar_op,
                    void *workspace, size_t workspace_bytes, fp_stream_t stream);

/* fp_select for one chunk of a chunked prefill (Sec.4.3 "Compatibility with
 * Chunked Prefill"): the same outputs as fp_select, bit for bit, when kbar,
 * vbar, kbar_op and vbar_op already hold the means that fp_select (or this
 * call) wrote for the same request rows and the same keys and values, e.g.
 * from the previous chunk of the request. The means of every block lying
 * wholly in a request's cached prefix (blocks J with (J + 1) * 128 <=
 * L_b^kv - L_b^q) are then kept as they are, since those tokens did not
 * change; only the blocks holding new tokens are pooled from k_pages and
 * v_pages, and the kept blocks' rounding statistics (workspace) are derived
 * from the stored means. Each request's block rows sit at blk_base(b) as for
 * fp_select, so the rows must hold that request's prefix means at this call's
 * row positions (for example, a request that stays first in its batch). A
 * request without a prefix is pooled in full. Arguments are fp_select's. */
fp_status fp_select_chunk(const fp_problem *p, const void *q, const void *k_pages, const void *v_pages,
                          float alpha, int32_t sink_blocks, int32_t window_blocks, int32_t *csr_cu, int32_t *csr_idx,
                          int64_t csr_idx_capacity, float *kbar, float *vbar, void *kbar_op, void *vbar_op,
                          void *workspace, size_t workspace_bytes, fp_stream_t stream);

/* Stage 2 (Alg.1 steps 6-11). For every segment, walks its selected blocks in
 * descending order (Eq.17) with exact Q'K^T and PV (token-causal mask on the
 * diagonal block), then, with FP_MEAN_CORRECTION, one term per pruned block
 * J < D with logit q.kbar_J / sqrt(d) + ln 128 and value vbar_J (Eq.6, Sec.3.2
 * "Implementation"), all in one online softmax; the epilogue divides by the
 * accumulated denominator. FP8 computes S = c_q c_k (Q~K~^T), quantises
 * P~ = e4m3(256 exp(S - m)) and O = c_v sum P~V~ / sum P~ (Eq.15).
 * When the problem has fewer packed tiles than four times the GPU's SMs, a
 * tile of n > C* iterations (selected blocks, then correction chunks) is cut
 * into U = ceil(n / C*) contiguous runs of ceil(n / U) iterations
 * (count-balanced KV splits, Sec.3.3 Eq.18), C* = max(8, ceil(total
 * iterations / min(SMs, 160))); each run writes a normalised fp32 partial
 * output and its LSE to the workspace, and a combine kernel merges them:
 * lse = ln sum_u e^{lse_u}, O = sum_u e^{lse_u - lse} O_u. The result equals
 * the unsplit one up to rounding.
 *   csr_cu, csr_idx   a CSR in fp_select's format (ignored with FP_DENSE); every
 *                     segment is checked (ids in [0, D], ascending, within
 *                     csr_idx_capacity) and a malformed one is skipped and
 *                     reported as FP_ERR_DEVICE_CSR
 *   kbar_op, vbar_op  operand-format means from fp_select (ignored without correction)
 *   out               out [T, Hq, 128] bf16
 *   lse               out [T, Hq] fp32 natural-log denominator, or NULL */
fp_status fp_attention(const fp_problem *p, const void *q, const void *k_pages, const void *v_pages,
                       const int32_t *csr_cu, const int32_t *csr_idx, int64_t csr_idx_capacity,
                       const void *kbar_op, const void *vbar_op, int32_t flags, void *out, float *lse,
                       void *workspace, size_t workspace_bytes, fp_stream_t stream);

/* fp_attention that also records the attention kernel's integer work, so that
 * it can be checked against a host recomputation from the same CSR: the
 * scheduler's work list (heaviest tiles first, Sec.3.3 "Sparsity-Aware Load
 * Balancing"), each tile's visit sequence (selected blocks in descending order,
 * Eq.17, then correction chunks in descending order), each correction chunk's
 * mask (todo = valid & ~selected, Sec.3.2 "Implementation") and the page-table
 * rows each block is read from (Eq.22). It computes the same outputs as
 * fp_attention, a little more slowly. Arguments are fp_attention's, plus:
 *   trace        device int32 [trace_words], 16-byte aligned, overwritten:
 *                  words 0..7: header {words used after the header, 1 if the
 *                    trace ran out of room (records past that point are
 *                    dropped) else 0, number of work items, 0, 0, 0, 0, 0}
 *                  then one record per work item, in no particular order:
 *                    8 words {w, b, h, T, D, it_lo, it_hi, n_exact}: the item's
 *                    position w in the work list, request, KV head, absolute
 *                    packed tile, diagonal block, the item's iterations
 *                    [it_lo, it_hi) of the tile's sequence (a whole tile: 0 and
 *                    its iteration count; a run of a split tile, Eq.18, its
 *                    contiguous slice; 0 and 0 for an item with no work) and
 *                    the tile's selected-block count (-1 for a malformed segment);
 *                    then it_hi - it_lo entries of 8 words
 *                    {J, flags, m0, m1, m2, m3, r0, r1} in visit order:
 *                      J >= 0  a selected block; r0, r1 = pool rows (page *
 *                              page_size + slot) of its first and last page
 *                              chunk of min(page_size, 128) tokens, or
 *                              num_pages * page_size past the request's end
 *                      J < 0   correction chunk c = -1 - J; m0..m3 = the mask of
 *                              its blocks 128c .. 128c + 127 (bit i of mk = block
 *                              128c + 32k + i); r0 = its first pooled-mean row
 *                      flags   bit 0: first iteration of the item, bit 1: last
 *   trace_words  capacity in int32 words (at most 2^31 - 1): 8 + 8 x (items +
 *                iterations) always suffices */
fp_status fp_attention_trace(const fp_problem *p, const void *q, const void *k_pages, const void *v_pages,
                             const int32_t *csr_cu, const int32_t *csr_idx, int64_t csr_idx_capacity,
                             const void *kbar_op, const void *vbar_op, int32_t flags, void *out, float *lse,
                             void *workspace, size_t workspace_bytes, fp_stream_t stream, int32_t *trace,
                             int64_t trace_words);

/* fp_select without a caller-provided workspace, for callers that cannot
 * allocate device memory (for example a plugin that receives only its input
 * and output tensors, or code on a path where cudaMalloc's implicit
 * synchronisation is not allowed). The paper has no counterpart: it is a
 * packaging variant of fp_select that computes the same outputs, bit for bit.
 * Scratch comes from a fixed 16 MiB device array inside the library, which
 * every GPU that loads the library holds until the process exits.
 *   - Problems whose fp_select scratch (fp_workspace_bytes less the 21 MB of
 *     split partial outputs that only fp_attention uses) exceeds 16 MiB are
 *     rejected with FP_ERR_WORKSPACE before anything is enqueued.
 *   - It calls no allocator. The first call in each CUDA context (the first
 *     on each device, and the first after a device reset, which moves the
 *     array) looks up the array's device address in that context; make that
 *     first call before any stream capture.
 *   - All calls share the array and it keeps the previous call's contents:
 *     calls whose work overlaps on the GPU race and must be serialised.
 *   - device_status (device int32, nullable) receives the call's device
 *     status code (FP_OK or a device error) when the work completes; the
 *     workspace-based fp_device_status cannot see this call.
 * Other arguments are those of fp_select. */
fp_status fp_select_noalloc(const fp_problem *p, const void *q, const void *k_pages, const void *v_pages,
                            float alpha, int32_t sink_blocks, int32_t window_blocks, int32_t *csr_cu,
                            int32_t *csr_idx, int64_t csr_idx_capacity, float *kbar, float *vbar, void *kbar_op,
                            void *vbar_op, int32_t *device_status, fp_stream_t stream);

/* Expands a CSR of 128-token blocks (fp_select's format) into the same CSR over
 * 64-token physical KV tiles, the unit the serving integration's page table
 * and attention backend index (Sec.3.4 "Serving Integration", Alg.1 step 5):
 * block J of a request becomes tiles 2J and 2J + 1, the second only when the
 * request holds a token at position (2J + 1) * 64, i.e. when
 * (2J + 1) * 64 < L_b^kv. Segments keep their order and each stays ascending.
 *   csr_cu, csr_idx    a CSR from fp_select (block ids must lie in [0, ceil(L_b^kv / 128));
 *                      an id outside is skipped and reported as FP_ERR_DEVICE_CSR)
 *   tile_cu            out [num_segments + 1]
 *   tile_idx           out [tile_idx_capacity]; 2 * csr_cu[num_segments] always suffices;
 *                      a larger result is cut off and reported as FP_ERR_DEVICE_OVERFLOW
 *   workspace          as for fp_select (its status word and request table are used) */
fp_status fp_csr_expand64(const fp_problem *p, const int32_t *csr_cu, const int32_t *csr_idx, int32_t *tile_cu,
                          int32_t *tile_idx, int64_t tile_idx_capacity, void *workspace, size_t workspace_bytes,
                          fp_stream_t stream);

/* Waits for `stream`, then returns the device-detected error recorded in
 * `workspace` by the most recent fp_select or fp_attention on it (each call
 * clears the status word when it starts), FP_OK if none, or FP_ERR_CUDA if
 * the stream reported an error. */
fp_status fp_device_status(const void *workspace, fp_stream_t stream);

/* Counters of the most recent fp_select on `workspace`, for tests and
 * monitoring. The scoring kernel settles most blocks with bounds on their
 * low-precision energies and recomputes the few it cannot settle in fp32
 * (the exact path); these counters say how often that happened. */
typedef struct {
    int32_t status;       /* the device status code, as fp_device_status returns it */
    int32_t exact_tiles;  /* packed query tiles whose selection took the fp32 recomputation */
    int32_t exact_blocks; /* blocks those tiles recomputed in fp32 */
} fp_select_stats;

/* Waits for `stream`, then copies the counters that the most recent fp_select
 * on `workspace` left there. A later fp_attention or fp_csr_expand64 on the
 * same workspace clears them. Returns FP_OK, FP_ERR_INVALID_ARG for a null
 * pointer, or FP_ERR_CUDA if the stream reported an error. */
fp_status fp_read_select_stats(const void *workspace, fp_select_stats *stats, fp_stream_t stream);

/* Static, human-readable name of a status code. */
const char *fp_status_string(fp_status s);

#ifdef __cplusplus
}
#endif

#endif /* FP_H_ */
