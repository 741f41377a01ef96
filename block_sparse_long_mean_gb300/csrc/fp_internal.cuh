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

// KV splits (count-balanced, FlashPrefill V2 Eq.18): a tile whose iteration count exceeds the per-CTA
// share C* = max(kMinSplitIters, ceil(total iterations / P)) is cut into U = ceil(n / C*) contiguous runs
// of ceil(n / U) iterations, each run computed by its own work item into a partial-output slot and merged
// by log-sum-exp. With P <= kSplitCtas CTAs the split tiles need at most 2 P slots.
constexpr int kSplitCtas = 160;
constexpr int kMaxSlots = 2 * kSplitCtas;
constexpr int kMinSplitIters = 8;  // a run below 8 iterations costs more in pipeline fill and merge than it saves
constexpr int kSplitTilesPerSm = 4;  // splits are enabled while tiles < 4 x SMs

// Slots of the workspace counter array.
enum CounterSlot { kCntSplitTarget = 0, kCntSlots = 1, kCntSplits = 2, kCntItems = 3 };

// One split tile: its runs' partial outputs are in slots slot0 .. slot0 + nsplit - 1; the rest places
// its rows in the output (as in TileTask).
struct SplitRec {
    int32_t slot0, nsplit;
    int32_t t, h, q_start, lo, rows, pad;
};

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
    int32_t b, h;       // request, KV head
    int32_t t;          // absolute packed tile: the tile's row i is absolute packed row 128 t + i
    int32_t D;          // diagonal block of the tile
    int32_t rows;       // query rows of the tile are [lo, rows) (rows <= 128)
    int32_t q_start;    // token of q holding absolute position 0 (cu_seqlens[b] - (L^kv - L^q); may be < 0)
    int32_t len;        // KV length L^kv
    int32_t blk_base;   // first pooled-mean row of the request
    int32_t lo;         // first query row of the tile (> 0 only in a chunk's first tile)
    int32_t it_lo, it_hi;  // this work item's iterations [it_lo, it_hi) of the tile's sequence (Eq.18)
    int32_t slot;       // partial-output slot of a split tile's run, -1 for a whole tile
    int32_t split;      // the split tile's SplitRec, -1 for a whole tile
    int64_t todo;       // first word of the segment's correction bitmap
};
static_assert(sizeof(TileTask) == 80, "TileTask is five 16-byte words");

// Per-request table, built on the device from cu_seqlens and seqlens_kv at the
// start of each call (the host mirrors it from the host copies only to size
// buffers). The request's L^q new tokens are the last of its L^kv positions;
// packed rows are numbered by absolute position (r = g pos + head mod g) and
// tiled 128 at a time from r = 0, so no tile straddles two blocks.
struct ReqInfo {
    int32_t q_start;    // cu_seqlens[b]: token of q holding the first new query
    int32_t len;        // L^q, new query tokens
    int32_t kv_len;     // L^kv >= L^q: keys and values (cached prefix + new tokens)
    int32_t t0;         // absolute tile of the request's first tile: floor(g (L^kv - L^q) / 128)
    int32_t nblocks;    // ceil(L^kv / 128)
    int32_t ntiles;     // packed tiles per KV head: ceil(g L^kv / 128) - t0, 0 if L^q = 0
    int32_t blk_base;   // first row of this request in the pooled-mean arrays
    int32_t seg_base;   // first CSR segment of this request (segments: h-major, then t)
    int32_t mask_base;  // first selection-mask word of this request
    int32_t words;      // selection-mask words per segment: ceil(nblocks / 32)
    int32_t pad[2];
};
static_assert(sizeof(ReqInfo) == 48, "ReqInfo is three 16-byte words");

// Status word slots in the workspace (int32 each). The slots after the code are counters of the last
// fp_select, cleared with the status word when a call starts.
enum StatusSlot { kStatusCode = 0, kStatusDetail = 1, kStatusExactTiles = 2, kStatusExactBlocks = 3 };

// Byte offsets of the workspace regions, derived on the host from the sizes.
struct WsLayout {
    int64_t status, req, seg_count, mask, work, hist, counters, kstat, meta, splits, part_lse, part_o, total;
};

struct Sizes {
    int64_t nseg = 0, nblocks = 0, capacity = 0, mask_words = 0, total_tokens = 0, kv_tokens = 0;
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
    SplitRec *splits() const { return reinterpret_cast<SplitRec *>(wsbase + ws.splits); }
    float *part_lse() const { return reinterpret_cast<float *>(wsbase + ws.part_lse); }  // [kMaxSlots, 128]
    float *part_o() const { return reinterpret_cast<float *>(wsbase + ws.part_o); }      // [kMaxSlots, 128, 128]
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
    int b, h, t, D;  // request, KV head, tile within the request, diagonal block
    int lo, rows;    // query rows of the tile: [lo, rows), rows <= 128
    int row0;        // absolute packed row of the tile's row 0 (128 (t0 + t))
    int q_pos;       // token of q holding the position of row 0 (below cu_seqlens[b] when lo > 0)
};

// Coordinates of segment `seg` of request b, whose record is r.
__device__ __forceinline__ SegCoord coord_in_req(const ReqInfo &r, int b, int g, int64_t seg) {
    SegCoord c;
    c.b = b;
    int rem = (int)(seg - r.seg_base);
    c.h = rem / r.ntiles;
    c.t = rem - c.h * r.ntiles;
    const int shift = r.kv_len - r.len;
    c.row0 = (r.t0 + c.t) * kTileRows;
    c.lo = max(0, g * shift - c.row0);
    c.rows = min(kTileRows, g * r.kv_len - c.row0);
    c.D = (c.row0 / g) / kBlock;
    c.q_pos = r.q_start - shift + c.row0 / g;
    return c;
}

__device__ __forceinline__ SegCoord decode_seg(const ReqInfo *req, int batch, int g, int64_t seg) {
    const int b = find_req_by_seg(req, batch, seg);
    return coord_in_req(req[b], b, g, seg);
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
                        void *kbar_op, void *vbar_op, bool reuse_prefix = false);
cudaError_t launch_score(const Ctx &c, const void *q, const float *kbar, const void *kbar_op, float alpha, int sink,
                         int window);
cudaError_t launch_csr(const Ctx &c, int32_t *csr_cu, int32_t *csr_idx, int64_t capacity);
cudaError_t launch_expand64(const Ctx &c, const int32_t *csr_cu, const int32_t *csr_idx, int32_t *tile_cu,
                            int32_t *tile_idx, int64_t capacity);
cudaError_t launch_attention(const Ctx &c, const void *q, const void *k_pages, const void *v_pages,
                             const int32_t *csr_cu, const int32_t *csr_idx, int64_t capacity, const void *kbar_op,
                             const void *vbar_op, int flags, void *out, float *lse, int32_t *trace = nullptr,
                             int32_t trace_words = 0);

}  // namespace fp
