// Internal declarations of libfp: workspace layout, per-request tables, device
// helpers and the launchers each translation unit provides to fp_api.cu.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "../../include/fp.h"

namespace fp {

constexpr int kHeadDim = 128;     // d
constexpr int kBlock = 128;       // B, tokens per selection block
constexpr int kTileRows = 128;    // packed query rows per tile (PackGQA M-tile)
constexpr int kMaxLen = 1 << 20;  // longest request
constexpr int kMaxBlocks = kMaxLen / kBlock;
constexpr int kMaxChunks = kMaxBlocks / 128;          // 128-block correction chunks per tile (64)
constexpr int kCostBuckets = kMaxBlocks + kMaxChunks + 2;

// Per-segment Stage 2 schedule entry: iterations and correction chunks.
struct SegMeta {
    int32_t n_exact;      // selected blocks walked exactly, -1 if the segment's CSR is malformed
    int32_t n_chunks;     // correction chunks holding at least one pruned block
    uint32_t chunk_lo;    // bit c: chunk c (blocks 128c .. 128c+127) needs correction, c < 32
    uint32_t chunk_hi;    // same for c in [32, 64)
};

// One entry of the Stage 2 work list (heaviest first): everything the
// attention kernel needs about a segment, in one 64-byte record.
struct alignas(16) TileTask {
    int32_t n_exact;    // selected blocks walked exactly, -1 if the CSR is malformed
    int32_t n_chunks;   // correction chunks
    uint32_t chunk_lo, chunk_hi;
    int32_t csr_end;    // CSR offset one past the segment's last entry
    int32_t b, h, t;    // request, KV head, tile
    int32_t D;          // diagonal block of the tile
    int32_t rows;       // valid packed rows (<= 128)
    int32_t q_start;    // first token of the request
    int32_t len;        // request length
    int32_t blk_base;   // first pooled-mean row of the request
    int32_t pad;
    int64_t todo;       // first word of the segment's correction bitmap
};
static_assert(sizeof(TileTask) == 64, "TileTask is one 64-byte record");

// Per-request table, built on the device from cu_seqlens at the start of each
// call (the host mirrors it from host_cu_seqlens only to size buffers).
struct ReqInfo {
    int32_t q_start;    // cu_seqlens[b]
    int32_t len;        // L_b
    int32_t nblocks;    // ceil(L_b / 128)
    int32_t ntiles;     // ceil(g L_b / 128) packed tiles per KV head
    int32_t blk_base;   // first row of this request in the pooled-mean arrays
    int32_t seg_base;   // first CSR segment of this request (segments: h-major, then t)
    int32_t mask_base;  // first selection-mask word of this request
    int32_t words;      // selection-mask words per segment: ceil(nblocks / 32)
};

// Status word slots in the workspace (int32 each).
enum StatusSlot { kStatusCode = 0, kStatusDetail = 1 };

// Byte offsets of the workspace regions, derived on the host from the sizes.
struct WsLayout {
    int64_t status, req, seg_count, mask, work, hist, counters, kstat, meta, total;
};

struct Sizes {
    int64_t nseg = 0, nblocks = 0, capacity = 0, mask_words = 0, total_tokens = 0;
    int32_t max_len = 0, max_blocks = 0, g = 1;
};

// Everything a launcher needs, resolved on the host.
struct Ctx {
    fp_problem p;
    Sizes s;
    WsLayout ws;
    char *wsbase;
    cudaStream_t stream;
    int32_t *status() const { return reinterpret_cast<int32_t *>(wsbase + ws.status); }
    ReqInfo *req() const { return reinterpret_cast<ReqInfo *>(wsbase + ws.req); }
    int32_t *seg_count() const { return reinterpret_cast<int32_t *>(wsbase + ws.seg_count); }
    uint32_t *mask() const { return reinterpret_cast<uint32_t *>(wsbase + ws.mask); }
    TileTask *tasks() const { return reinterpret_cast<TileTask *>(wsbase + ws.work); }
    int32_t *hist() const { return reinterpret_cast<int32_t *>(wsbase + ws.hist); }
    int32_t *counters() const { return reinterpret_cast<int32_t *>(wsbase + ws.counters); }
    // per (pooled block, KV head): {|kbar - operand-format kbar|_2, |kbar|_2}
    float2 *kstat() const { return reinterpret_cast<float2 *>(wsbase + ws.kstat); }
    SegMeta *meta() const { return reinterpret_cast<SegMeta *>(wsbase + ws.meta); }
};

// ----------------------------------------------------------------- device helpers

// Records the first device-detected error; later errors keep the first code.
__device__ __forceinline__ void set_status(int32_t *status, int32_t code, int32_t detail = 0) {
    if (atomicCAS(status + kStatusCode, 0, code) == 0) status[kStatusDetail] = detail;
}

__device__ __forceinline__ bool status_bad(const int32_t *status) {
    return *reinterpret_cast<const volatile int32_t *>(status + kStatusCode) == FP_ERR_DEVICE_SEQLEN;
}

// Request holding segment `seg` (binary search over seg_base).
__device__ __forceinline__ int find_req_by_seg(const ReqInfo *req, int batch, int64_t seg) {
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (req[mid].seg_base <= seg) lo = mid; else hi = mid - 1;
    }
    // skip empty requests sharing the same base
    while (lo + 1 < batch && req[lo + 1].seg_base <= seg) ++lo;
    return lo;
}

__device__ __forceinline__ int find_req_by_block(const ReqInfo *req, int batch, int64_t gb) {
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (req[mid].blk_base <= gb) lo = mid; else hi = mid - 1;
    }
    while (lo + 1 < batch && req[lo + 1].blk_base <= gb) ++lo;
    return lo;
}

// Decoded coordinates of a CSR segment.
struct SegCoord {
    int b, h, t, D, rows;  // rows: valid packed rows of the tile (<= 128)
};

// Coordinates of segment `seg` of request b, whose record is r.
__device__ __forceinline__ SegCoord coord_in_req(const ReqInfo &r, int b, int g, int64_t seg) {
    SegCoord c;
    c.b = b;
    int rem = (int)(seg - r.seg_base);
    c.h = rem / r.ntiles;
    c.t = rem - c.h * r.ntiles;
    int r0 = c.t * kTileRows;
    int total_rows = g * r.len;
    c.rows = min(kTileRows, total_rows - r0);
    c.D = (r0 / g) / kBlock;
    return c;
}

__device__ __forceinline__ SegCoord decode_seg(const ReqInfo *req, int batch, int g, int64_t seg) {
    SegCoord c;
    c.b = find_req_by_seg(req, batch, seg);
    const ReqInfo r = req[c.b];
    int rem = (int)(seg - r.seg_base);
    c.h = rem / r.ntiles;
    c.t = rem - c.h * r.ntiles;
    int r0 = c.t * kTileRows;
    int total_rows = g * r.len;
    c.rows = min(kTileRows, total_rows - r0);
    c.D = (r0 / g) / kBlock;
    return c;
}

template <int kDtype> struct Elem;
template <> struct Elem<FP_DTYPE_BF16> {
    using T = __nv_bfloat16;
    static constexpr int kBytes = 2;
    __device__ __forceinline__ static float to_float(T x) { return __bfloat162float(x); }
};
template <> struct Elem<FP_DTYPE_E4M3> {
    using T = __nv_fp8_e4m3;
    static constexpr int kBytes = 1;
    __device__ __forceinline__ static float to_float(T x) { return float(x); }
};

// Number of SMs of the current device (cached per device).
int num_sms();

// Encodes a tiled TMA descriptor with 128-byte swizzling over a row-major
// tensor: dims innermost first, strides in bytes for dims 1..rank-1, box in
// elements. Element type bf16, or 8-bit when u8. Returns false on failure.
bool make_tmap(CUtensorMap *map, const void *base, bool u8, int rank, const uint64_t *dims, const uint64_t *strides,
               const uint32_t *box);

// Host sizing shared by the entry points (fp_api.cu).
fp_status describe(const fp_problem *p, Sizes *s);
WsLayout layout(const fp_problem *p, const Sizes &s);

// ---------------------------------------------------------------------- launchers
// Each returns cudaSuccess or the launch error.
cudaError_t launch_prep(const Ctx &c);
cudaError_t launch_pool(const Ctx &c, const void *k_pages, const void *v_pages, float *kbar, float *vbar,
                        void *kbar_op, void *vbar_op);
cudaError_t launch_score(const Ctx &c, const void *q, const float *kbar, const void *kbar_op, float alpha, int sink,
                         int window);
cudaError_t launch_csr(const Ctx &c, int32_t *csr_cu, int32_t *csr_idx, int64_t capacity);
cudaError_t launch_expand64(const Ctx &c, const int32_t *csr_cu, const int32_t *csr_idx, int32_t *tile_cu,
                            int32_t *tile_idx, int64_t capacity);
cudaError_t launch_attention(const Ctx &c, const void *q, const void *k_pages, const void *v_pages,
                             const int32_t *csr_cu, const int32_t *csr_idx, int64_t capacity, const void *kbar_op,
                             const void *vbar_op, int flags, void *out, float *lse);

}  // namespace fp
