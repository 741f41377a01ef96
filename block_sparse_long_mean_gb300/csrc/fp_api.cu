// Host side of the C ABI declared in include/fp.h: argument validation,
// sizing, workspace layout and the launch sequence of each stage.
#include <stdio.h>
#include <string.h>

#include "fp_internal.cuh"

namespace fp {
namespace {

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

int64_t align256(int64_t x) { return (x + 255) & ~int64_t(255); }

}  // namespace

// Validates the description; fills the sizes from host_cu_seqlens and host_seqlens_kv.
fp_status describe(const fp_problem *p, Sizes *s) {
    if (!p || !p->host_cu_seqlens) return FP_ERR_INVALID_ARG;
    if (p->batch < 0 || p->num_q_heads <= 0 || p->num_kv_heads <= 0) return FP_ERR_INVALID_ARG;
    if (p->num_kv_heads > 64) return FP_ERR_UNSUPPORTED;
    if (p->num_q_heads % p->num_kv_heads) return FP_ERR_UNSUPPORTED;
    int g = p->num_q_heads / p->num_kv_heads;
    if (!is_pow2(g) || g > 16) return FP_ERR_UNSUPPORTED;
    if (p->head_dim != kHeadDim || p->block_size != kBlock) return FP_ERR_UNSUPPORTED;
    if (!is_pow2(p->page_size) || p->page_size < 8 || p->page_size > 128) return FP_ERR_UNSUPPORTED;
    if (p->dtype != FP_DTYPE_BF16 && p->dtype != FP_DTYPE_E4M3) return FP_ERR_UNSUPPORTED;
    if (p->dtype == FP_DTYPE_E4M3 && !(p->c_q > 0.f && p->c_k > 0.f && p->c_v > 0.f)) return FP_ERR_INVALID_ARG;
    if (p->num_pages < 0 || p->page_table_stride < 0) return FP_ERR_INVALID_ARG;
    if (p->host_cu_seqlens[0] != 0) return FP_ERR_INVALID_ARG;
    if ((p->seqlens_kv == nullptr) != (p->host_seqlens_kv == nullptr)) return FP_ERR_INVALID_ARG;
    // the device int32 arrays are read with 4-byte loads
    if ((reinterpret_cast<uintptr_t>(p->cu_seqlens) | reinterpret_cast<uintptr_t>(p->seqlens_kv) |
         reinterpret_cast<uintptr_t>(p->page_table)) & 3)
        return FP_ERR_INVALID_ARG;
    Sizes r;
    r.g = g;
    for (int b = 0; b < p->batch; ++b) {
        int64_t L = (int64_t)p->host_cu_seqlens[b + 1] - p->host_cu_seqlens[b];
        int64_t Lkv = p->host_seqlens_kv ? (int64_t)p->host_seqlens_kv[b] : L;
        if (L < 0 || Lkv < L) return FP_ERR_INVALID_ARG;
        if (Lkv > kMaxLen) return FP_ERR_UNSUPPORTED;
        // tiles on the absolute packed-row grid that hold one of the request's g L query rows
        int64_t t0 = g * (Lkv - L) / kTileRows;
        int64_t nb = (Lkv + kBlock - 1) / kBlock;
        int64_t nt = L > 0 ? (g * Lkv + kTileRows - 1) / kTileRows - t0 : 0;
        int64_t words = (nb + 31) / 32;
        if ((Lkv + p->page_size - 1) / p->page_size > p->page_table_stride) return FP_ERR_INVALID_ARG;
        r.nseg += p->num_kv_heads * nt;
        r.nblocks += nb;
        r.mask_words += p->num_kv_heads * nt * words;
        // sum over the request's tiles of (D + 1), D = floor(128 T / g / 128) = floor(T / g), T = t0 + t
        for (int64_t t = 0; t < nt; ++t) r.capacity += p->num_kv_heads * ((t0 + t) / g + 1);
        r.total_tokens += L;
        r.kv_tokens += Lkv;
        if (Lkv > r.max_len) r.max_len = (int32_t)Lkv;
        if (nb > r.max_blocks) r.max_blocks = (int32_t)nb;
    }
    if (r.nseg >= INT32_MAX || r.nblocks >= INT32_MAX || r.mask_words >= INT32_MAX || r.total_tokens >= INT32_MAX)
        return FP_ERR_UNSUPPORTED;
    if (r.kv_tokens >= INT32_MAX) return FP_ERR_UNSUPPORTED;
    if ((r.total_tokens > 0 || r.kv_tokens > 0) && (!p->cu_seqlens || !p->page_table)) return FP_ERR_INVALID_ARG;
    *s = r;
    return FP_OK;
}

WsLayout layout(const fp_problem *p, const Sizes &s) {
    WsLayout w;
    int64_t o = 0;
    w.status = o; o = align256(o + 64 * 4);
    w.req = o; o = align256(o + (int64_t)sizeof(ReqInfo) * (p->batch + 1));
    w.seg_count = o; o = align256(o + 4 * (s.nseg + 1));
    w.mask = o; o = align256(o + 4 * (s.mask_words + 1));
    w.work = o; o = align256(o + (int64_t)sizeof(TileTask) * (s.nseg + kMaxSlots + 1));
    w.hist = o; o = align256(o + 4 * (int64_t)(kCostBuckets + 2));
    w.counters = o; o = align256(o + 4 * 64);
    w.kstat = o; o = align256(o + 8 * (s.nblocks * p->num_kv_heads + 1));
    w.meta = o; o = align256(o + (int64_t)sizeof(SegMeta) * (s.nseg + 1));
    w.splits = o; o = align256(o + (int64_t)sizeof(SplitRec) * kMaxSlots);
    // partial outputs of split tiles (fp_attention only; the last region, so fp_select's scratch ends here)
    w.part_lse = o; o = align256(o + 4 * (int64_t)kMaxSlots * kTileRows);
    w.part_o = o; o = align256(o + 4 * (int64_t)kMaxSlots * kTileRows * kHeadDim);
    w.total = o;
    return w;
}

namespace {

using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The driver's tensor-map encoder, fetched through the runtime once.
EncodeTiled encoder() {
    static EncodeTiled fn = [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            ptr = nullptr;
        return reinterpret_cast<EncodeTiled>(ptr);
    }();
    return fn;
}

}  // namespace

bool make_tmap(CUtensorMap *map, const void *base, bool u8, int rank, const uint64_t *dims, const uint64_t *strides,
               const uint32_t *box) {
    EncodeTiled fn = encoder();
    if (!fn) {
        fprintf(stderr, "libfp: cuTensorMapEncodeTiled unavailable\n");
        return false;
    }
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    const CUresult r = fn(map, u8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank,
                          const_cast<void *>(base), reinterpret_cast<const cuuint64_t *>(dims),
                          reinterpret_cast<const cuuint64_t *>(strides), box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) fprintf(stderr, "libfp: cuTensorMapEncodeTiled failed (%d)\n", (int)r);
    return r == CUDA_SUCCESS;
}

int num_sms() {
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (!cached[dev]) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cached[dev] = n;
    }
    return cached[dev];
}

namespace {

fp_status make_ctx(const fp_problem *p, void *workspace, size_t ws_bytes, fp_stream_t stream, Ctx *c) {
    Sizes s;
    fp_status st = describe(p, &s);
    if (st != FP_OK) return st;
    if (!workspace) return FP_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) % 256) return FP_ERR_INVALID_ARG;
    WsLayout w = layout(p, s);
    if ((int64_t)ws_bytes < w.total) return FP_ERR_WORKSPACE;
    c->p = *p;
    c->s = s;
    c->ws = w;
    c->wsbase = static_cast<char *>(workspace);
    c->stream = reinterpret_cast<cudaStream_t>(stream);
    return FP_OK;
}

// A null pointer, or one on an a-byte boundary (a a power of two).
bool aligned(const void *ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) == 0; }

fp_status launched(cudaError_t e) {
    if (e != cudaSuccess) {
        fprintf(stderr, "libfp: CUDA error: %s\n", cudaGetErrorString(e));
        return FP_ERR_CUDA;
    }
    return FP_OK;
}

}  // namespace
}  // namespace fp

using namespace fp;

extern "C" {

int64_t fp_workspace_bytes(const fp_problem *p) {
    Sizes s;
    fp_status st = describe(p, &s);
    if (st != FP_OK) return st;
    return layout(p, s).total;
}

int64_t fp_num_segments(const fp_problem *p) {
    Sizes s;
    fp_status st = describe(p, &s);
    return st != FP_OK ? st : s.nseg;
}

int64_t fp_num_blocks(const fp_problem *p) {
    Sizes s;
    fp_status st = describe(p, &s);
    return st != FP_OK ? st : s.nblocks;
}

int64_t fp_csr_capacity(const fp_problem *p) {
    Sizes s;
    fp_status st = describe(p, &s);
    return st != FP_OK ? st : s.capacity;
}

}  // extern "C"

namespace {

fp_status select_impl(const fp_problem *p, const void *q, const void *k_pages, const void *v_pages, float alpha,
                      int32_t sink_blocks, int32_t window_blocks, int32_t *csr_cu, int32_t *csr_idx,
                      int64_t csr_idx_capacity, float *kbar, float *vbar, void *kbar_op, void *vbar_op,
                      void *workspace, size_t workspace_bytes, fp_stream_t stream, bool reuse_prefix) {
    Ctx c;
    fp_status st = make_ctx(p, workspace, workspace_bytes, stream, &c);
    if (st != FP_OK) return st;
    if (!(alpha >= 0.f) || sink_blocks < 0 || window_blocks < 0 || csr_idx_capacity < 0) return FP_ERR_INVALID_ARG;
    if (!csr_cu) return FP_ERR_INVALID_ARG;
    if ((c.s.total_tokens > 0 && !q) ||
        (c.s.nblocks > 0 && (!k_pages || !v_pages || !kbar || !vbar || !kbar_op || !vbar_op)))
        return FP_ERR_INVALID_ARG;
    if (c.s.nseg > 0 && !csr_idx) return FP_ERR_INVALID_ARG;
    // tensors read through TMA start on 16-byte boundaries; the int32 / fp32 outputs on 4-byte ones
    if (!aligned(q, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(kbar_op, 16) ||
        !aligned(vbar_op, 16) || !aligned(csr_cu, 4) || !aligned(csr_idx, 4) || !aligned(kbar, 4) ||
        !aligned(vbar, 4))
        return FP_ERR_INVALID_ARG;
    cudaError_t e = cudaMemsetAsync(c.status(), 0, 64 * 4, c.stream);
    if (e == cudaSuccess) e = launch_prep(c);
    if (e == cudaSuccess && c.s.nblocks > 0)
        e = launch_pool(c, k_pages, v_pages, kbar, vbar, kbar_op, vbar_op, reuse_prefix);
    if (e == cudaSuccess && c.s.nseg > 0)
        e = launch_score(c, q, kbar, kbar_op, alpha, sink_blocks, window_blocks);
    if (e == cudaSuccess) e = launch_csr(c, csr_cu, csr_idx, csr_idx_capacity);
    return launched(e);
}

}  // namespace

extern "C" {

fp_status fp_select(const fp_problem *p, const void *q, const void *k_pages, const void *v_pages, float alpha,
                    int32_t sink_blocks, int32_t window_blocks, int32_t *csr_cu, int32_t *csr_idx,
                    int64_t csr_idx_capacity, float *kbar, float *vbar, void *kbar_op, void *vbar_op,
                    void *workspace, size_t workspace_bytes, fp_stream_t stream) {
    return select_impl(p, q, k_pages, v_pages, alpha, sink_blocks, window_blocks, csr_cu, csr_idx, csr_idx_capacity,
                       kbar, vbar, kbar_op, vbar_op, workspace, workspace_bytes, stream, false);
}

fp_status fp_select_chunk(const fp_problem *p, const void *q, const void *k_pages, const void *v_pages,
                          float alpha, int32_t sink_blocks, int32_t window_blocks, int32_t *csr_cu, int32_t *csr_idx,
                          int64_t csr_idx_capacity, float *kbar, float *vbar, void *kbar_op, void *vbar_op,
                          void *workspace, size_t workspace_bytes, fp_stream_t stream) {
    return select_impl(p, q, k_pages, v_pages, alpha, sink_blocks, window_blocks, csr_cu, csr_idx, csr_idx_capacity,
                       kbar, vbar, kbar_op, vbar_op, workspace, workspace_bytes, stream, true);
}

fp_status fp_csr_expand64(const fp_problem *p, const int32_t *csr_cu, const int32_t *csr_idx, int32_t *tile_cu,
                          int32_t *tile_idx, int64_t tile_idx_capacity, void *workspace, size_t workspace_bytes,
                          fp_stream_t stream) {
    Ctx c;
    fp_status st = make_ctx(p, workspace, workspace_bytes, stream, &c);
    if (st != FP_OK) return st;
    if (tile_idx_capacity < 0 || !tile_cu) return FP_ERR_INVALID_ARG;
    if (c.s.nseg > 0 && (!csr_cu || !csr_idx || (tile_idx_capacity > 0 && !tile_idx))) return FP_ERR_INVALID_ARG;
    if (!aligned(csr_cu, 4) || !aligned(csr_idx, 4) || !aligned(tile_cu, 4) || !aligned(tile_idx, 4))
        return FP_ERR_INVALID_ARG;
    cudaError_t e = cudaMemsetAsync(c.status(), 0, 64 * 4, c.stream);
    if (e == cudaSuccess) e = launch_prep(c);
    if (e == cudaSuccess) e = launch_expand64(c, csr_cu, csr_idx, tile_cu, tile_idx, tile_idx_capacity);
    return launched(e);
}

}  // extern "C"

namespace {

fp_status attention_impl(const fp_problem *p, const void *q, const void *k_pages, const void *v_pages,
                         const int32_t *csr_cu, const int32_t *csr_idx, int64_t csr_idx_capacity,
                         const void *kbar_op, const void *vbar_op, int32_t flags, void *out, float *lse,
                         void *workspace, size_t workspace_bytes, fp_stream_t stream, int32_t *trace,
                         int64_t trace_words) {
    Ctx c;
    fp_status st = make_ctx(p, workspace, workspace_bytes, stream, &c);
    if (st != FP_OK) return st;
    if (flags & ~(FP_MEAN_CORRECTION | FP_DENSE)) return FP_ERR_INVALID_ARG;
    bool dense = flags & FP_DENSE;
    bool corr = (flags & FP_MEAN_CORRECTION) && !dense;
    if (csr_idx_capacity < 0) return FP_ERR_INVALID_ARG;
    if (c.s.total_tokens > 0 && (!q || !k_pages || !v_pages || !out)) return FP_ERR_INVALID_ARG;
    if (c.s.nseg > 0 && !dense && (!csr_cu || !csr_idx)) return FP_ERR_INVALID_ARG;
    if (c.s.nseg > 0 && corr && (!kbar_op || !vbar_op)) return FP_ERR_INVALID_ARG;
    // TMA-read tensors and the 16-byte output stores start on 16-byte boundaries; lse takes fp32 stores
    if (!aligned(q, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(kbar_op, 16) ||
        !aligned(vbar_op, 16) || !aligned(out, 16) || !aligned(lse, 4) || !aligned(csr_cu, 4) ||
        !aligned(csr_idx, 4))
        return FP_ERR_INVALID_ARG;
    cudaError_t e = cudaMemsetAsync(c.status(), 0, 64 * 4, c.stream);
    if (e == cudaSuccess) e = launch_prep(c);
    if (e == cudaSuccess && c.s.nseg > 0)
        e = launch_attention(c, q, k_pages, v_pages, csr_cu, csr_idx, csr_idx_capacity, kbar_op, vbar_op,
                             (corr ? FP_MEAN_CORRECTION : 0) | (dense ? FP_DENSE : 0), out, lse, trace,
                             (int32_t)trace_words);
    else if (e == cudaSuccess && trace)
        e = cudaMemsetAsync(trace, 0, 8 * sizeof(int32_t), c.stream);  // an empty trace
    return launched(e);
}

}  // namespace

extern "C" {

fp_status fp_attention(const fp_problem *p, const void *q, const void *k_pages, const void *v_pages,
                       const int32_t *csr_cu, const int32_t *csr_idx, int64_t csr_idx_capacity,
                       const void *kbar_op, const void *vbar_op, int32_t flags, void *out, float *lse,
                       void *workspace, size_t workspace_bytes, fp_stream_t stream) {
    return attention_impl(p, q, k_pages, v_pages, csr_cu, csr_idx, csr_idx_capacity, kbar_op, vbar_op, flags, out,
                          lse, workspace, workspace_bytes, stream, nullptr, 0);
}

fp_status fp_attention_trace(const fp_problem *p, const void *q, const void *k_pages, const void *v_pages,
                             const int32_t *csr_cu, const int32_t *csr_idx, int64_t csr_idx_capacity,
                             const void *kbar_op, const void *vbar_op, int32_t flags, void *out, float *lse,
                             void *workspace, size_t workspace_bytes, fp_stream_t stream, int32_t *trace,
                             int64_t trace_words) {
    // the trace is written in 16-byte pieces and counted in int32 words
    if (!trace || !aligned(trace, 16) || trace_words < 8 || trace_words > INT32_MAX) return FP_ERR_INVALID_ARG;
    return attention_impl(p, q, k_pages, v_pages, csr_cu, csr_idx, csr_idx_capacity, kbar_op, vbar_op, flags, out,
                          lse, workspace, workspace_bytes, stream, trace, trace_words);
}

fp_status fp_device_status(const void *workspace, fp_stream_t stream) {
    if (!workspace) return FP_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int32_t code = 0;
    cudaError_t e = cudaMemcpyAsync(&code, workspace, sizeof code, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
        fprintf(stderr, "libfp: CUDA error: %s\n", cudaGetErrorString(e));
        return FP_ERR_CUDA;
    }
    return (fp_status)code;
}

fp_status fp_read_select_stats(const void *workspace, fp_select_stats *stats, fp_stream_t stream) {
    if (!workspace || !stats) return FP_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int32_t words[4] = {0, 0, 0, 0};
    cudaError_t e = cudaMemcpyAsync(words, workspace, sizeof words, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
        fprintf(stderr, "libfp: CUDA error: %s\n", cudaGetErrorString(e));
        return FP_ERR_CUDA;
    }
    stats->status = words[kStatusCode];
    stats->exact_tiles = words[kStatusExactTiles];
    stats->exact_blocks = words[kStatusExactBlocks];
    return FP_OK;
}

const char *fp_status_string(fp_status s) {
    switch (s) {
        case FP_OK: return "ok";
        case FP_ERR_INVALID_ARG: return "invalid argument";
        case FP_ERR_UNSUPPORTED: return "unsupported problem";
        case FP_ERR_WORKSPACE: return "workspace too small";
        case FP_ERR_CUDA: return "CUDA error";
        case FP_ERR_CAPACITY: return "CSR capacity too small";
        case FP_ERR_DEVICE_PAGE: return "device: page id out of range";
        case FP_ERR_DEVICE_CSR: return "device: malformed CSR segment";
        case FP_ERR_DEVICE_OVERFLOW: return "device: CSR index capacity exceeded";
        case FP_ERR_DEVICE_TIMEOUT: return "device: bounded wait expired";
        case FP_ERR_DEVICE_SEQLEN: return "device: cu_seqlens or seqlens_kv differ from host copy";
    }
    return "unknown status";
}

}  // extern "C"
