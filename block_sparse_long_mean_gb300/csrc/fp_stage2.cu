// Stage 2 of FlashPrefill V2 (Alg.1 steps 6-11) on tcgen05 / TMEM / TMA.
//
// Scheduling (Sec.3.3 "Sparsity-Aware Load Balancing"): a prep kernel reads
// each segment's CSR once, validates it, derives the correction chunks that
// hold a pruned block (the paper's todo = valid & ~selected, Sec.3.2
// "Implementation") and orders the segments by descending work
// |S| + #chunks with a counting sort. A persistent CTA per SM then walks that
// list round-robin.
//
// Per segment (one 128-row packed query tile, Eq.12-13) the CTA runs one
// pipeline iteration per selected block, in descending block order (Eq.17),
// then one per correction chunk of 128 pooled means (Eq.6): TMA producers
// bring the Q tile, the block's K and V pages through the page table (Eq.22)
// or the chunk's means; one thread issues S = Q K^T and O += P V on tcgen05;
// softmax warps keep half a row per thread (online softmax in the base-2
// domain, row maxima returned by the TMEM load, causal mask on the diagonal
// block, the log2|B_J| = 7 shift and the correction mask on mean chunks, lazy
// rescaling of O); epilogue warps divide by the denominator and write bf16 O
// and the LSE.
// FP8 (Eq.15): Q, K, V and the means are E4M3, S = c_q c_k (Q~ K~^T),
// P~ = e4m3(256 * 2^(x - m)) with the denominator summing P~, O = c_v ... / l.
#include <math.h>

#include "fp_internal.cuh"
#include "sm100_ptx.cuh"

namespace fp {
namespace {

using namespace sm100;

// ------------------------------------------------------------ schedule prep

// One warp per segment (a CTA takes 32, four per warp): validates its CSR,
// counts selected blocks per 128-block chunk, and records the iteration
// counts and chunk mask. The CTA's 32 costs enter the histogram with one
// atomic per distinct cost: most tiles share a handful of costs, and
// same-address atomics from every segment would serialise.
constexpr int kMetaSegs = 32;
__global__ void __launch_bounds__(256) attn_meta_kernel(const ReqInfo *__restrict__ req, int batch, int g,
                                                        int32_t nseg, const int32_t *__restrict__ cu,
                                                        const int32_t *__restrict__ idx, int64_t capacity, int flags,
                                                        SegMeta *__restrict__ meta, uint32_t *__restrict__ todo,
                                                        int32_t *__restrict__ hist, int32_t *__restrict__ status) {
    __shared__ int cnt[8][kMaxChunks];
    __shared__ int scost[kMetaSegs];
    if (status_bad(status)) return;  // the same outcome in every thread (only the prep kernel sets that code)
    const int lane = threadIdx.x & 31, wl = threadIdx.x >> 5;
    for (int k = 0; k < kMetaSegs / 8; ++k) {
        const int64_t seg = (int64_t)blockIdx.x * kMetaSegs + 8 * k + wl;
        int cost = -1;
        if (seg < nseg) {
            const SegCoord sc = decode_seg(req, batch, g, seg);
            const bool dense = flags & FP_DENSE;
            const bool corr = (flags & FP_MEAN_CORRECTION) && !dense;
            SegMeta m = {0, 0, 0u, 0u};
            if (dense) {
                m.n_exact = sc.D + 1;
            } else {
                const int64_t beg = cu[seg], end = cu[seg + 1];
                int bad = (beg < 0 || end < beg || end > capacity) ? 1 : 0;
                for (int c = lane; c < kMaxChunks; c += 32) cnt[wl][c] = 0;
                __syncwarp();
                if (!bad)
                    for (int64_t i = beg + lane; i < end; i += 32) {
                        const int J = idx[i];
                        if (J < 0 || J > sc.D || (i > beg && idx[i - 1] >= J)) bad = 1;
                        else if (J < sc.D) atomicAdd(&cnt[wl][J >> 7], 1);
                    }
                bad = __any_sync(0xffffffffu, bad);
                __syncwarp();
                if (bad) {
                    m.n_exact = -1;
                    if (lane == 0) set_status(status, FP_ERR_DEVICE_CSR, (int32_t)seg);
                } else {
                    m.n_exact = (int)(end - beg);
                    if (corr) {
                        // correction bitmap over [0, D): every causal block fully visible to the tile, minus the
                        // selected ones (todo = valid & ~selected); read by the attention kernel per chunk
                        const ReqInfo r = req[sc.b];
                        uint32_t *tw = todo + (int64_t)r.mask_base + (int64_t)(sc.h * r.ntiles + sc.t) * r.words;
                        const int nw = (sc.D + 31) / 32;
                        for (int wd = lane; wd < nw; wd += 32) {
                            const int left = sc.D - 32 * wd;
                            tw[wd] = left >= 32 ? 0xffffffffu : ((1u << left) - 1u);
                        }
                        __syncwarp();
                        __threadfence_block();
                        for (int64_t i = beg + lane; i < end; i += 32) {
                            const int J = idx[i];
                            if (J < sc.D) atomicAnd(&tw[J >> 5], ~(1u << (J & 31)));
                        }
                        const int nch = (sc.D + 127) / 128;
                        for (int c0 = 0; c0 < kMaxChunks; c0 += 32) {
                            const int c = c0 + lane;
                            const bool need = c < nch && cnt[wl][c] < min(128, sc.D - 128 * c);
                            const unsigned bal = __ballot_sync(0xffffffffu, need);
                            if (c0 == 0) m.chunk_lo = bal; else m.chunk_hi = bal;
                        }
                        m.n_chunks = __popc(m.chunk_lo) + __popc(m.chunk_hi);
                    }
                }
            }
            if (lane == 0) meta[seg] = m;
            cost = m.n_exact < 0 ? 0 : min(m.n_exact + m.n_chunks, kCostBuckets - 1);
            __syncwarp();
        }
        if (lane == 0) scost[8 * k + wl] = cost;
    }
    __syncthreads();
    if (wl == 0) {
        const int c = scost[lane];
        const unsigned peers = __match_any_sync(0xffffffffu, c);
        if (c >= 0 && lane == __ffs(peers) - 1) atomicAdd(&hist[c], __popc(peers));
        // the largest cost, so that the bucket scan covers only [0, max]
        int mx = c;
        for (int o = 16; o; o >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0 && mx > 0) atomicMax(&hist[kCostBuckets], mx);
    }
}

// Number of runs a tile of `cost` iterations is cut into (count-balanced KV splits, Eq.18).
__device__ __forceinline__ int num_splits(int cost, int target) { return cost > target ? (cost + target - 1) / target : 1; }

// Turns the cost histogram into descending-cost offsets of the work list (one CTA). With splits
// (ctas > 0) it first sums the iterations of all tiles and fixes the split target
// C* = max(kMinSplitIters, ceil(total / ctas)); a bucket of cost c then takes num_splits(c, C*) work
// items per tile. Without, every tile is one item.
__global__ void __launch_bounds__(1024) attn_bucket_kernel(int32_t *__restrict__ hist, int32_t *__restrict__ counters,
                                                           int ctas, int32_t *__restrict__ status) {
    __shared__ int32_t warp_sums[32];
    __shared__ long long warp_tot[32];
    __shared__ int32_t carry, target;
    if (status_bad(status)) return;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nb = hist[kCostBuckets] + 1;  // buckets 0 .. the largest cost
    long long tot = 0;
    if (ctas > 0) {
        for (int c = threadIdx.x; c < nb; c += 1024) tot += (long long)c * hist[c];
        for (int o = 16; o; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
        if (lane == 0) warp_tot[warp] = tot;
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        long long all = 0;
        if (ctas > 0)
            for (int i = 0; i < 32; ++i) all += warp_tot[i];
        const long long per = ctas > 0 ? (all + ctas - 1) / ctas : (long long)kCostBuckets;
        target = (int)max((long long)kMinSplitIters, min(per, (long long)kCostBuckets));
        counters[kCntSplitTarget] = target;
        counters[kCntSlots] = 0;
        counters[kCntSplits] = 0;
        carry = 0;
    }
    __syncthreads();
    const int tgt = target;
    for (int base = 0; base < nb; base += 1024) {
        const int i = base + threadIdx.x;
        const int bucket = nb - 1 - i;  // descending cost
        int32_t v = i < nb ? hist[bucket] * num_splits(bucket, tgt) : 0;
        const int32_t own = v;
        for (int o = 1; o < 32; o <<= 1) {
            int32_t n = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += n;
        }
        if (lane == 31) warp_sums[warp] = v;
        __syncthreads();
        if (warp == 0) {
            int32_t s = warp_sums[lane];
            for (int o = 1; o < 32; o <<= 1) {
                int32_t n = __shfl_up_sync(0xffffffffu, s, o);
                if (lane >= o) s += n;
            }
            warp_sums[lane] = s;
        }
        __syncthreads();
        const int32_t excl = carry + (warp ? warp_sums[warp - 1] : 0) + v - own;
        const int32_t total = warp_sums[31];
        __syncthreads();
        if (i < nb) hist[bucket] = excl;
        if (threadIdx.x == 0) carry += total;
        __syncthreads();
    }
    if (threadIdx.x == 0) counters[kCntItems] = carry;  // length of the work list
}

// Places every segment in the work list (descending cost) as one TileTask, or as one per run when the
// tile is split; a split tile also takes consecutive partial-output slots and a SplitRec.
__global__ void __launch_bounds__(256) attn_scatter_kernel(const ReqInfo *__restrict__ req, int batch, int g,
                                                           const SegMeta *__restrict__ meta, int32_t nseg,
                                                           const int32_t *__restrict__ cu, int flags,
                                                           int32_t *__restrict__ hist, int32_t *__restrict__ counters,
                                                           SplitRec *__restrict__ splits, TileTask *__restrict__ tasks,
                                                           int32_t *__restrict__ status) {
    if (status_bad(status)) return;
    const int64_t seg = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (seg >= nseg) return;
    const SegMeta m = meta[seg];
    const int cost = m.n_exact < 0 ? 0 : min(m.n_exact + m.n_chunks, kCostBuckets - 1);
    const int nsplit = num_splits(cost, counters[kCntSplitTarget]);
    const SegCoord sc = decode_seg(req, batch, g, seg);
    const ReqInfo r = req[sc.b];
    TileTask t;
    t.n_exact = m.n_exact;
    t.n_chunks = m.n_chunks;
    t.chunk_lo = m.chunk_lo;
    t.chunk_hi = m.chunk_hi;
    t.csr_end = (flags & FP_DENSE) ? 0 : cu[seg + 1];
    t.b = sc.b;
    t.h = sc.h;
    t.t = sc.row0 / kTileRows;
    t.D = sc.D;
    t.rows = sc.rows;
    t.q_start = r.q_start - (r.kv_len - r.len);
    t.len = r.kv_len;
    t.blk_base = r.blk_base;
    t.lo = sc.lo;
    t.it_lo = 0;
    t.it_hi = m.n_exact < 0 ? 0 : m.n_exact + m.n_chunks;
    t.slot = -1;
    t.split = -1;
    t.todo = (int64_t)r.mask_base + (int64_t)(sc.h * r.ntiles + sc.t) * r.words;
    // one atomic per distinct cost in the warp (equal costs take equal run counts)
    const unsigned peers = __match_any_sync(__activemask(), cost);
    const int lane = threadIdx.x & 31, leader = __ffs(peers) - 1;
    int base = 0;
    if (lane == leader) base = atomicAdd(&hist[cost], nsplit * __popc(peers));
    const int pos = __shfl_sync(peers, base, leader) + nsplit * __popc(peers & ((1u << lane) - 1));
    if (nsplit == 1) {
        tasks[pos] = t;
        return;
    }
    const int slot0 = atomicAdd(&counters[kCntSlots], nsplit);
    const bool room = slot0 + nsplit <= kMaxSlots;  // always, by the choice of the split target
    if (room) {
        t.split = atomicAdd(&counters[kCntSplits], 1);
        splits[t.split] = SplitRec{slot0, nsplit, t.t, t.h, t.q_start, t.lo, t.rows, 0};
    } else {
        set_status(status, FP_ERR_DEVICE_OVERFLOW, (int32_t)seg);
        t.n_exact = -2;  // not run
    }
    const int per = (cost + nsplit - 1) / nsplit;
    for (int u = 0; u < nsplit; ++u) {
        t.it_lo = u * per;
        t.it_hi = min(cost, (u + 1) * per);
        t.slot = slot0 + u;
        tasks[pos + u] = t;
    }
}

// ------------------------------------------------------------ split combine

// Merges the runs of every split tile (the LSE combine of split-KV attention): per query row,
// lse = ln sum_u e^{lse_u} and O = sum_u e^{lse_u - lse} O_u over its runs' normalised outputs. CTA
// 4 k + q takes rows 32 q .. 32 q + 31 of split tile k; thread i of it row 32 q + i / 32 and columns
// 4 (i % 32) .. + 3, so a warp reads one 512-byte row of a run's partial output and every thread has only
// its runs' loads to wait for. The grid is small (an empty launch costs little) and strides over the tiles.
constexpr int kCombineThreads = 1024, kCombineTiles = 40;
__global__ void __launch_bounds__(kCombineThreads) attn_combine_kernel(const SplitRec *__restrict__ splits,
                                                                       const int32_t *__restrict__ counters,
                                                                       const float *__restrict__ part_o,
                                                                       const float *__restrict__ part_lse,
                                                                       __nv_bfloat16 *__restrict__ out,
                                                                       float *__restrict__ lse, int hq, int g,
                                                                       const int32_t *__restrict__ status) {
    const int nsplit_tiles = counters[kCntSplits];
    if (status_bad(status)) return;
    const int j = 32 * (blockIdx.x & 3) + (threadIdx.x >> 5), cg = threadIdx.x & 31;
    for (int k = blockIdx.x >> 2; k < nsplit_tiles; k += gridDim.x >> 2) {
        const SplitRec sr = splits[k];
        if (j < sr.lo || j >= sr.rows) continue;
        const float *lp = part_lse + (int64_t)sr.slot0 * kTileRows + j;
        const float4 *op = reinterpret_cast<const float4 *>(part_o + ((int64_t)sr.slot0 * kTileRows + j) * kHeadDim) + cg;
        constexpr int64_t kRunStride4 = (int64_t)kTileRows * kHeadDim / 4;  // float4s between runs
        float m = -INFINITY;
#pragma unroll 4
        for (int u = 0; u < sr.nsplit; ++u) m = fmaxf(m, lp[u * kTileRows]);
        float sum = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 4
        for (int u = 0; u < sr.nsplit; ++u) {
            const float w = expf(lp[u * kTileRows] - m);
            const float4 x = op[u * kRunStride4];
            sum += w;
            acc.x = fmaf(w, x.x, acc.x);
            acc.y = fmaf(w, x.y, acc.y);
            acc.z = fmaf(w, x.z, acc.z);
            acc.w = fmaf(w, x.w, acc.w);
        }
        const float rs = 1.f / sum;
        const int gr = sr.t * kTileRows + j;
        const int64_t rowi = (int64_t)(sr.q_start + gr / g) * hq + sr.h * g + gr % g;
        const __nv_bfloat162 lo2 = __floats2bfloat162_rn(acc.x * rs, acc.y * rs);
        const __nv_bfloat162 hi2 = __floats2bfloat162_rn(acc.z * rs, acc.w * rs);
        uint2 pk;
        pk.x = *reinterpret_cast<const uint32_t *>(&lo2);
        pk.y = *reinterpret_cast<const uint32_t *>(&hi2);
        reinterpret_cast<uint2 *>(out + rowi * kHeadDim)[cg] = pk;
        if (lse && cg == 0) lse[rowi] = m + logf(sum);
    }
}

// --------------------------------------------------------------- attention

// Warp roles (four warpgroups; registers rebalanced with setmaxnreg):
//   warp 0      walker: walks the CTA's tiles, looks up the CSR, the page table
//               and the correction masks in batches, and publishes one record
//               per iteration in a shared-memory ring, up to kRing ahead
//   warp 1      MMA issue + TMEM owner: one wait per MMA group, then issue
//   warp 2      loader: Q, K and V tiles by TMA, as stages free up
//   warp 3      group scheduler: reads the records, waits for each MMA
//               group's inputs and publishes the group for the MMA warp
//   warps 4-11  softmax: each warp owns 16 rows of the tile, each row spread
//               over two threads (64 consecutive keys each)
//   warps 12-15 epilogue: O / l to bf16, LSE
// The softmax of an iteration is its critical chain: its exponentials (one
// per score, 512 cycles of MUFU for a 128 x 128 tile) run on both softmax
// warps of a scheduler at once, and the loads, maxima and handoffs around
// them are latency; together they take longer than the iteration's two MMAs.
// TMEM: two S buffers (P of an iteration is written over its S), one O
// buffer and two Q buffers (E4M3: and the 16 columns of its row sums). Each
// tile's Q is copied from shared memory into TMEM once (tcgen05.cp), at its
// first QK^T: that frees the one shared-memory Q buffer, so the next tile's Q
// loads a whole tile ahead, and both MMAs then take A from TMEM.
// The iterations of all the CTA's tiles form one stream. MMA group g issues
// PV(g - 2) then QK^T(g), so the tensor core computes the next scores while
// the softmax works on these. Every tcgen05 operation of the CTA comes from
// one thread and executes in issue order, so QK^T(g) may write the columns
// PV(g - 2) reads P from. The epilogue drains O while the next tile's first
// QK^T and softmax run.
constexpr int kAWarps = 16;
constexpr int kAThreads = 32 * kAWarps;
constexpr int kKStages = 3, kVStages = 3;
constexpr int kRing = 8;                    // iteration records in flight
constexpr int kRingUsers = 10;              // group scheduler, 8 softmax warps, loader
constexpr int kGroupRing = 4;               // MMA groups published ahead by the scheduler
constexpr int32_t kRecEnd = -0x7fffffff;    // record after the CTA's last iteration
constexpr uint32_t kColS = 0, kColO = 256, kColQ = 384;  // S_b at 128 b, O at 256, Q_b at 384 + 64 b
// FP8 only, where a Q buffer takes 32 columns: the Eq.15 denominator sum P~ 1, 16 equal columns accumulated by
// the tensor core next to O (between the two Q buffers)
constexpr uint32_t kColL = 416;
constexpr int kRegsProducer = 80, kRegsSoftmax = 160, kRegsEpilogue = 112;  // 128 x (80 + 2 x 160 + 112) = 64K

template <int kDtype>
struct ACfg {
    static constexpr int kEb = Elem<kDtype>::kBytes;
    static constexpr int kTile = 128 * 128 * kEb;  // Q tile, K block, V block, mean chunk
    static constexpr int kBoxElems = 128 / kEb;     // elements per 128-byte row of a TMA box
    static constexpr int kBoxes = 128 / kBoxElems;  // boxes along d
    static constexpr int kKStep = 32 / kEb;         // MMA K per instruction (32 bytes)
    static constexpr int kNumK = 128 / kKStep;
    static constexpr uint32_t kFmt = kDtype == FP_DTYPE_BF16 ? 1u : 0u;
    static constexpr uint32_t kIdescQK = instr_desc(kFmt, kFmt, false, false, 128, 128);
    static constexpr uint32_t kIdescPV = instr_desc(kFmt, kFmt, false, true, 128, 128);
};

// FP8: P~ (from TMEM) times a 128 x 16 tile of ones (K-major): the row sums of P~ in 16 columns
constexpr uint32_t kIdescL8 = instr_desc(0, 0, false, false, 128, 16);

// The B operand of the FP8 row-sum MMA: 16 rows of 128 E4M3 ones (two 8-row groups of the 128-byte swizzle
// atom; every byte is 1.0, so the swizzle does not matter). BF16 keeps its row sums on the softmax warps.
template <int kDtype> struct OnesTile {};
template <> struct OnesTile<FP_DTYPE_E4M3> {
    alignas(1024) uint32_t w[512];
};

// One pipeline iteration as the walker publishes it.
struct alignas(16) IterRec {
    int32_t J;      // block id; -1 - c for correction chunk c; kRecEnd after the last iteration
    int32_t tile;   // the CTA's tile counter (selects the Q buffers)
    int32_t flags;  // bit 0: first iteration of its tile, bit 1: last
    int32_t row0;   // absolute packed row of the tile's row 0 (t * 128)
    int32_t D;      // diagonal block of the tile
    int32_t h;      // KV head
    int32_t q_pos;  // token of q holding row 0's position (Q rows, for its first iteration)
    int32_t len;    // KV length of the request
    union {
        int32_t rows[16];  // block: pool row of each page chunk
        struct {
            int32_t mrow;      // chunk: first pooled-mean row
            int32_t pad[3];
            uint32_t mask[4];  // chunk: which of its 128 means are corrected
        } c;
    } u;
};

// One MMA group as the scheduler warp publishes it: what the MMA warp issues for group g.
struct GroupRec {
    int32_t pv;  // PV(g - 2): -1 none, else bit 0 the tile's first PV (overwrites O), bit 1 its last (O complete)
    int32_t qk;  // QK^T(g): -1 none, else bit 0 the tile's first (copies Q into TMEM), bit 1 its last
    int32_t qb;  // TMEM Q buffer of QK^T(g)
    int32_t end; // 1: no more groups
};

// MMA group g: PV(g - 2) (when g >= 2 and that iteration exists) followed by
// QK^T(g) (when iteration g exists), closed by one commit to grp[g % 4]; its
// completion means S(g) is ready, K stage g % 3 and V stage (g - 2) % 3 are
// free and O holds PV(g - 2).

template <int kDtype>
struct AttnSmem {
    alignas(1024) uint8_t q[ACfg<kDtype>::kTile];
    alignas(1024) uint8_t k[kKStages][ACfg<kDtype>::kTile];
    alignas(1024) uint8_t v[kVStages][ACfg<kDtype>::kTile];
    OnesTile<kDtype> ones;
    float stat_m[128], stat_l[128];    // a finished tile's running max (log2) and denominator per row
    IterRec ring[kRing];
    uint8_t chunk_list[kMaxChunks];  // walker scratch: a tile's correction chunks, descending
    GroupRec group[kGroupRing];
    uint64_t q_full, q_empty, k_full[kKStages], v_full[kVStages], grp[4], go[2], qk_done[2], o_full, o_empty,
        st_full, rec_full[kRing], rec_empty[kRing];
    uint32_t tmem_base;
    int abort, skip, nitems;
};

static_assert(sizeof(AttnSmem<FP_DTYPE_BF16>) <= 232448, "attention shared memory exceeds the 227 KB opt-in limit");

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Registers per thread at launch: 64K over the CTA's threads, rounded down to a multiple of 8.
constexpr int kRegsLaunch = (65536 / kAThreads) & ~7;
static_assert(kRegsProducer + 2 * kRegsSoftmax + kRegsEpilogue <= 4 * kRegsLaunch, "register split exceeds the launch");

// Sets this warpgroup's register count: setmaxnreg.inc to grow, .dec to shrink
// (a .dec to a larger count is not allowed), chosen at compile time.
template <int kRegs>
__device__ __forceinline__ void regs_set() {
    static_assert(kRegs % 8 == 0 && kRegs >= 24 && kRegs <= 256, "setmaxnreg range");
    if constexpr (kRegs > kRegsLaunch)
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegs));
    else if constexpr (kRegs < kRegsLaunch)
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegs));
}

// Kernel arguments besides the tensor maps (read from the constant bank).
struct AttnParams {
    const int32_t *pt;  // page table
    int pt_stride, num_pages, page_size;
    const int32_t *csr_idx;
    const uint32_t *todo;    // per-segment correction bitmaps
    const TileTask *tasks;   // work list, heaviest first
    __nv_bfloat16 *out;
    float *lse;
    int hq, g, flags;
    float c_q, c_k, c_v;
    int32_t nseg;              // segments
    const int32_t *nitems;     // work-list length with splits (written by the bucket kernel)
    float *part_o, *part_lse;  // partial outputs of split tiles' runs
    uint32_t smem_bytes;
    int32_t *status;
    int32_t *trace;      // integer-work trace (fp_attention_trace), or null
    int32_t trace_cap;   // its capacity in words
};

// Words of the trace header, of an item header and of one iteration entry (fp.h, fp_attention_trace).
constexpr int kTraceHeader = 8, kTraceItem = 8, kTraceEntry = 8;

template <bool kSplit>
__device__ __forceinline__ bool task_live(const TileTask &t) {
    return t.n_exact >= 0 && (kSplit ? t.it_hi > t.it_lo : t.n_exact + t.n_chunks > 0);
}

template <int kDtype, bool kSplit, bool kTrace>
__global__ void __launch_bounds__(kAThreads, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_kb,
                   const __grid_constant__ CUtensorMap tm_vb, const __grid_constant__ AttnParams P) {
    using C = ACfg<kDtype>;
    extern __shared__ uint8_t smem_raw[];
    const uintptr_t base = (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023);
    AttnSmem<kDtype> &sm = *reinterpret_cast<AttnSmem<kDtype> *>(base);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (base + sizeof(AttnSmem<kDtype>) > reinterpret_cast<uintptr_t>(smem_raw) + P.smem_bytes) {
        if (threadIdx.x == 0) set_status(P.status, FP_ERR_DEVICE_TIMEOUT, -1);
        return;
    }
    int32_t *const status = P.status;
    const int g = P.g;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            // group 2 k + i may issue: 8 softmax arrivals (P of iteration 2 k + i - 2) and the scheduler's
            mbar_init(&sm.go[i], 9);
            mbar_init(&sm.qk_done[i], 1);
        }
        for (int i = 0; i < 4; ++i) mbar_init(&sm.grp[i], 1);
        mbar_init(&sm.q_full, 1);
        mbar_init(&sm.q_empty, 1);
        mbar_init(&sm.o_full, 1);
        mbar_init(&sm.o_empty, 4);
        mbar_init(&sm.st_full, 8);
        for (int i = 0; i < kKStages; ++i) mbar_init(&sm.k_full[i], 1);
        for (int i = 0; i < kVStages; ++i) mbar_init(&sm.v_full[i], 1);
        for (int i = 0; i < kRing; ++i) {
            mbar_init(&sm.rec_full[i], 1);
            mbar_init(&sm.rec_empty[i], kRingUsers);
        }
        sm.abort = 0;
        if (kSplit) sm.nitems = *P.nitems;
        // an earlier stage failed: every warp skips its role (one read, so the CTA agrees)
        sm.skip = status_bad(P.status) ? 1 : 0;
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(&sm.tmem_base, 512);
    if constexpr (kDtype == FP_DTYPE_E4M3) {
        // the ones tile of the row-sum MMA, made visible to the tensor core (async proxy)
        static_assert(kAThreads == 512, "one word of the ones tile per thread");
        sm.ones.w[threadIdx.x] = 0x38383838u;  // E4M3 1.0 in every byte
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const Abort ab{&sm.abort};
    const uint32_t tmem = sm.tmem_base;
    const int ps_eff = min(P.page_size, 128);
    const int npc = 128 / ps_eff;  // page chunks per 128-token block (<= 16 as page_size >= 8)
    const int oob_row = P.num_pages * P.page_size;  // first row past the pool: TMA fills zeros
    const bool dense = P.flags & FP_DENSE;

    if (sm.skip) {
    } else if (warp < 4) {
        regs_set<kRegsProducer>();
        if (warp == 0) {
            // ------------------------------------------------------------------------ walker
            uint32_t gi = 0;
            bool ok = true;
            // the trace entry of the next iteration (fp_attention_trace only; warp-uniform)
            int32_t *tr = nullptr;
            // publishes iteration gi; `row` is this lane's page-chunk row (lane % npc) for a block
            auto emit = [&](int J, int flags, int tile, const TileTask &tk, uint4 mk, int row) -> bool {
                if (kTrace && tr && J != kRecEnd) {
                    const int row_last = __shfl_sync(0xffffffffu, row, npc - 1);
                    if (lane == 0) {
                        const int4 a = make_int4(J, flags, (int)mk.x, (int)mk.y);
                        const int4 b = J >= 0 ? make_int4(0, 0, row, row_last)
                                              : make_int4((int)mk.z, (int)mk.w, tk.blk_base + 128 * (-1 - J), 0);
                        reinterpret_cast<int4 *>(tr)[0] = a;
                        reinterpret_cast<int4 *>(tr)[1] = b;
                    }
                    tr += kTraceEntry;
                }
                const int slot = gi % kRing;
                if (!mbar_wait(&sm.rec_empty[slot], ((gi / kRing) & 1) ^ 1, ab)) return false;
                IterRec &rc = sm.ring[slot];
                if (J >= 0 && J != kRecEnd && lane < 16) rc.u.rows[lane] = row;
                if (lane == 0) {
                    rc.J = J;
                    rc.tile = tile;
                    rc.flags = flags;
                    rc.row0 = tk.t * kTileRows;
                    rc.D = tk.D;
                    rc.h = tk.h;
                    rc.q_pos = tk.q_start + (tk.t * kTileRows) / g;
                    rc.len = tk.len;
                    if (J < 0 && J != kRecEnd) {
                        rc.u.c.mrow = tk.blk_base + 128 * (-1 - J);
                        rc.u.c.mask[0] = mk.x;
                        rc.u.c.mask[1] = mk.y;
                        rc.u.c.mask[2] = mk.z;
                        rc.u.c.mask[3] = mk.w;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.rec_full[slot]);
                ++gi;
                return true;
            };
            const int per = 32 / npc;  // block lookups per batch
            uint32_t ti = 0;
            int w = blockIdx.x;
            const int nitems = kSplit ? sm.nitems : P.nseg;
            TileTask cur;
            if (w < nitems) cur = P.tasks[w];
            if (kTrace && blockIdx.x == 0 && lane == 0) P.trace[2] = nitems;
            while (w < nitems && ok) {
                const int wn = w + gridDim.x;
                TileTask nxt;
                if (wn < nitems) nxt = P.tasks[wn];  // overlaps this tile
                if (kTrace) {
                    // the item's header, then one entry per iteration as emit publishes it
                    const bool live = task_live<kSplit>(cur);
                    const int lo = kSplit ? cur.it_lo : 0, hi = kSplit ? cur.it_hi : cur.n_exact + cur.n_chunks;
                    const int n = live ? hi - lo : 0;
                    const int words = kTraceItem + kTraceEntry * n;
                    int off = 0;
                    if (lane == 0) off = atomicAdd(P.trace, words);
                    off = __shfl_sync(0xffffffffu, off, 0);
                    tr = nullptr;
                    if (off < 0 || (int64_t)off + words > (int64_t)P.trace_cap - kTraceHeader) {
                        if (lane == 0) P.trace[1] = 1;
                    } else {
                        tr = P.trace + kTraceHeader + off;
                        if (lane == 0) {
                            reinterpret_cast<int4 *>(tr)[0] = make_int4(w, cur.b, cur.h, cur.t);
                            reinterpret_cast<int4 *>(tr)[1] = make_int4(cur.D, live ? lo : 0, live ? hi : 0, cur.n_exact);
                        }
                        tr += kTraceItem;
                    }
                }
                if (task_live<kSplit>(cur)) {
                    // this item's iterations [it_lo, it_hi) of the tile's sequence: the selected blocks
                    // (iterations 0 .. n_exact - 1), then the correction chunks
                    const int it_lo = kSplit ? cur.it_lo : 0, it_hi = kSplit ? cur.it_hi : cur.n_exact + cur.n_chunks;
                    const int e_hi = min(it_hi, cur.n_exact);
                    int it = it_lo;
                    // selected blocks, descending (Eq.17): lane l looks up block base + l / npc, page chunk l % npc
                    for (int bs = it_lo; bs < e_hi && ok; bs += per) {
                        const int my = bs + lane / npc, pc = lane % npc;
                        int Jl = 0, rowl = oob_row;
                        if (my < e_hi) {
                            Jl = dense ? cur.D - my : __ldg(P.csr_idx + cur.csr_end - 1 - my);
                            const int tok = Jl * kBlock + pc * ps_eff;
                            if (tok < cur.len) {
                                const int page = __ldg(P.pt + (int64_t)cur.b * P.pt_stride + tok / P.page_size);
                                if (page >= 0 && page < P.num_pages)
                                    rowl = page * P.page_size + tok % P.page_size;
                                else
                                    set_status(status, FP_ERR_DEVICE_PAGE, page);
                            }
                        }
                        const int cnt = min(per, e_hi - bs);
                        for (int i = 0; i < cnt; ++i, ++it) {
                            const int J = __shfl_sync(0xffffffffu, Jl, i * npc);
                            const int row = __shfl_sync(0xffffffffu, rowl, i * npc + pc);
                            const int fl = (it == it_lo ? 1 : 0) | (it == it_hi - 1 ? 2 : 0);
                            if (!(ok = emit(J, fl, (int)ti, cur, make_uint4(0, 0, 0, 0), row))) break;
                        }
                    }
                    // correction chunks, descending: list them, then look up 32 masks at a time
                    const int c_lo = max(it_lo - cur.n_exact, 0), c_hi = it_hi - cur.n_exact;
                    if (c_hi > c_lo && ok) {
                        const uint32_t hi = cur.chunk_hi, lo = cur.chunk_lo;
                        const unsigned below = (1u << lane) - 1u;
                        const bool in_hi = (hi >> (31 - lane)) & 1u, in_lo = (lo >> (31 - lane)) & 1u;
                        const unsigned bhi = __ballot_sync(0xffffffffu, in_hi), blo = __ballot_sync(0xffffffffu, in_lo);
                        // lane l stands for bits 31 - l: its rank counts the set bits above it
                        if (in_hi) sm.chunk_list[__popc(bhi & below)] = (uint8_t)(63 - lane);
                        if (in_lo) sm.chunk_list[__popc(hi) + __popc(blo & below)] = (uint8_t)(31 - lane);
                        __syncwarp();
                        const int nw = (cur.D + 31) / 32;
                        for (int bs = c_lo; bs < c_hi && ok; bs += 32) {
                            int cl = 0;
                            uint4 ml = make_uint4(0, 0, 0, 0);
                            if (bs + lane < c_hi) {
                                cl = sm.chunk_list[bs + lane];
                                const uint32_t *tw = P.todo + cur.todo + 4 * cl;
                                ml.x = 4 * cl + 0 < nw ? __ldg(tw + 0) : 0u;
                                ml.y = 4 * cl + 1 < nw ? __ldg(tw + 1) : 0u;
                                ml.z = 4 * cl + 2 < nw ? __ldg(tw + 2) : 0u;
                                ml.w = 4 * cl + 3 < nw ? __ldg(tw + 3) : 0u;
                            }
                            const int cnt = min(32, c_hi - bs);
                            for (int i = 0; i < cnt; ++i, ++it) {
                                const int c = __shfl_sync(0xffffffffu, cl, i);
                                uint4 mk;
                                mk.x = __shfl_sync(0xffffffffu, ml.x, i);
                                mk.y = __shfl_sync(0xffffffffu, ml.y, i);
                                mk.z = __shfl_sync(0xffffffffu, ml.z, i);
                                mk.w = __shfl_sync(0xffffffffu, ml.w, i);
                                const int fl = (it == it_lo ? 1 : 0) | (it == it_hi - 1 ? 2 : 0);
                                if (!(ok = emit(-1 - c, fl, (int)ti, cur, mk, 0))) break;
                            }
                        }
                        __syncwarp();
                    }
                    ++ti;
                }
                cur = nxt;
                w = wn;
            }
            if (ok) emit(kRecEnd, 0, 0, cur, make_uint4(0, 0, 0, 0), 0);
        } else if (warp == 2) {
            // ------------------------------------------------------------------------ loader
            if (lane == 0) {
                tma_prefetch_desc(&tm_q);
                tma_prefetch_desc(&tm_k);
                tma_prefetch_desc(&tm_v);
                tma_prefetch_desc(&tm_kb);
                tma_prefetch_desc(&tm_vb);
            }
            // a block (J >= 0: lane L < kBoxes npc copies d box L / npc of page chunk L % npc) or 128 means
            auto load = [&](const CUtensorMap *tm_pages, const CUtensorMap *tm_means, uint8_t *dst, uint64_t *bar,
                            int J, int h, int row) {
                if (lane == 0) mbar_arrive_expect_tx(bar, C::kTile);
                __syncwarp();
                if (J >= 0) {
                    if (lane < C::kBoxes * npc)
                        tma_load_3d(dst + (lane / npc) * 16384 + (lane % npc) * ps_eff * 128, tm_pages, bar,
                                    (lane / npc) * C::kBoxElems, h, row);
                } else if (lane < C::kBoxes) {
                    tma_load_3d(dst + lane * 16384, tm_means, bar, lane * C::kBoxElems, h, row);
                }
            };
            // V of the previous iteration, issued one step behind K (V is needed one MMA group later)
            int pJ = kRecEnd, ph = 0, prow = 0;
            for (uint32_t gi = 0;; ++gi) {
                const int slot = gi % kRing;
                if (!mbar_wait(&sm.rec_full[slot], (gi / kRing) & 1, ab)) break;
                const IterRec &rc = sm.ring[slot];
                const int J = rc.J, h = rc.h, fl = rc.flags, tile = rc.tile, q_pos = rc.q_pos;
                const int row = J >= 0 ? rc.u.rows[lane % npc] : rc.u.c.mrow;
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.rec_empty[slot]);
                if (J != kRecEnd) {
                    if (fl & 1) {
                        // the shared Q buffer is free once the previous tile's Q was copied into TMEM
                        if (!mbar_wait(&sm.q_empty, (tile & 1) ^ 1, ab)) break;
                        if (lane == 0) {
                            mbar_arrive_expect_tx(&sm.q_full, C::kTile);
                            for (int i = 0; i < C::kBoxes; ++i)
                                tma_load_4d(sm.q + i * 16384, &tm_q, &sm.q_full, i * C::kBoxElems, 0, h, q_pos);
                        }
                    }
                    // K stage gi % 3 was last read by QK^T(gi - 3), closed by group gi - 3
                    if (gi >= kKStages && !mbar_wait(&sm.grp[(gi - 3) & 3], ((gi - 3) >> 2) & 1, ab)) break;
                    load(&tm_k, &tm_kb, sm.k[gi % kKStages], &sm.k_full[gi % kKStages], J, h, row);
                }
                if (gi >= 1 && pJ != kRecEnd) {
                    // V stage vi % kVStages was last read by PV(vi - kVStages), closed by group vi - kVStages + 2
                    const uint32_t vi = gi - 1, gv = vi + 2 - kVStages;
                    if (vi >= kVStages && !mbar_wait(&sm.grp[gv & 3], (gv >> 2) & 1, ab)) break;
                    load(&tm_v, &tm_vb, sm.v[vi % kVStages], &sm.v_full[vi % kVStages], pJ, ph, prow);
                }
                if (J == kRecEnd) break;
                pJ = J;
                ph = h;
                prow = row;
            }
        } else if (warp == 3) {
            // --------------------------------------------------------------------- group scheduler
            // Group g = PV(g - 2) then QK^T(g). For each group this warp reads the records, waits for every
            // input except the softmax's P(g - 2) (V and K stages, O free for a tile's first PV, Q loaded and
            // its TMEM buffer free for a tile's first QK^T), then publishes the group and arrives on go[g % 2],
            // which the softmax warps complete with P. The MMA warp thus has one wait per group: the tensor
            // core holds about one queued MMA, so any bookkeeping between groups would leave it idle.
            struct It {
                int tile, fl;
                bool valid;
            };
            uint32_t nrec = 0;
            auto fetch = [&](It &x) -> bool {
                const int slot = nrec % kRing;
                if (!mbar_wait(&sm.rec_full[slot], (nrec / kRing) & 1, ab)) return false;
                const int4 hd = *reinterpret_cast<const int4 *>(&sm.ring[slot]);  // J, tile, flags, row0
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.rec_empty[slot]);
                x.tile = hd.y;
                x.fl = hd.z;
                x.valid = hd.x != kRecEnd;
                if (x.valid) ++nrec;
                return true;
            };
            It a, b, c;  // iterations g - 2, g - 1 and g
            a.valid = b.valid = false;
            bool more = true;  // records not yet exhausted
            for (uint32_t g = 0;; ++g) {
                // at most three groups ahead of the tensor core: the slot of group g - 4 is free once group g - 3
                // has completed (group g - 4 was issued before it)
                if (g >= 3 && !mbar_wait(&sm.grp[(g - 3) & 3], ((g - 3) >> 2) & 1, ab)) break;
                c.valid = false;
                if (more) {
                    if (!fetch(c)) break;
                    more = c.valid;
                }
                GroupRec gr{-1, -1, 0, 0};
                bool ok = true;
                if (a.valid) {
                    // V(g - 2) loaded; O released by the epilogue before a tile's first PV
                    ok = mbar_wait(&sm.v_full[(g - 2) % kVStages], ((g - 2) / kVStages) & 1, ab);
                    if (ok && (a.fl & 1)) ok = mbar_wait(&sm.o_empty, (a.tile & 1) ^ 1, ab);
                    gr.pv = a.fl & 3;
                }
                if (ok && c.valid) {
                    if (c.fl & 1) {
                        // a new tile: its Q in shared memory, and TMEM Q buffer tile % 2 done with tile - 2
                        ok = mbar_wait(&sm.q_full, c.tile & 1, ab);
                        if (ok) ok = mbar_wait(&sm.qk_done[c.tile & 1], ((c.tile >> 1) & 1) ^ 1, ab);
                    }
                    if (ok) ok = mbar_wait(&sm.k_full[g % kKStages], (g / kKStages) & 1, ab);
                    gr.qk = c.fl & 3;
                    gr.qb = c.tile & 1;
                }
                // go[g % 2] takes this group's arrivals once its phase for group g - 2 has completed. A group
                // without a PV completes its phase by this warp's arrival alone, so it also waits until the MMA
                // warp has passed the phase of group g - 2 (that group has completed): a barrier two phases ahead
                // of its waiter would read as not yet complete
                if (ok && g >= 2) ok = mbar_wait(&sm.go[g & 1], ((g - 2) >> 1) & 1, ab);
                if (ok && g >= 2 && !a.valid) ok = mbar_wait(&sm.grp[(g - 2) & 3], ((g - 2) >> 2) & 1, ab);
                if (!ok) break;
                const bool last = !a.valid && !c.valid && !b.valid;
                gr.end = last ? 1 : 0;
                if (lane == 0) {
                    sm.group[g % kGroupRing] = gr;
                    // a group without a PV (the first two, an empty one, the end marker) has no P to wait for:
                    // the scheduler's arrival completes its phase alone
                    mbar_arrive_cnt(&sm.go[g & 1], a.valid ? 1u : 9u);
                }
                __syncwarp();
                if (last) break;
                a = b;
                b = c;
            }
        } else if (warp == 1) {
            // ------------------------------------------------------------------------- MMA
            // Per group: one wait (go: the scheduler's inputs and the softmax's P), then the group's MMAs and
            // one commit. The whole warp runs the loop (operands stay warp-uniform); one elected lane issues.
            auto issue_qk = [&](uint32_t gi, int fl, int qb) {
                const int ks = gi % kKStages, sb = gi & 1;
                const uint32_t tq = tmem + kColQ + qb * 64;
                if (fl & 1) {
                    // a new tile: copy its Q into TMEM buffer qb (last read by the QK^Ts of tile - 2)
                    const uint32_t qbase = smem_addr(sm.q);
#pragma unroll
                    for (int k = 0; k < C::kNumK; ++k)
                        tmem_cp_128x256b(tq + k * 8, sw128_desc(qbase + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024));
                    umma_commit(&sm.q_empty);
                }
                const uint32_t kbase = smem_addr(sm.k[ks]);
#pragma unroll
                for (int k = 0; k < C::kNumK; ++k) {
                    // A = Q from TMEM (K step k: 32 bytes = 8 columns), B = K rows in shared memory
                    const uint64_t bd = sw128_desc(kbase + (k >> 2) * 16384 + (k & 3) * 32, 16, 1024);
                    if (kDtype == FP_DTYPE_BF16)
                        umma_f16_ts(tmem + kColS + sb * 128, tq + k * 8, bd, C::kIdescQK, k > 0);
                    else
                        umma_f8_ts(tmem + kColS + sb * 128, tq + k * 8, bd, C::kIdescQK, k > 0);
                }
                if (fl & 2) umma_commit(&sm.qk_done[qb]);
            };
            // O (+)= P(i) V(i); a tile's first PV overwrites O
            auto issue_pv = [&](uint32_t i, int fl) {
                const int vs = i % kVStages, pb = i & 1;
                const bool first = fl & 1;
                const uint32_t vbase = smem_addr(sm.v[vs]);
#pragma unroll
                for (int k = 0; k < C::kNumK; ++k) {
                    // B = V, MN-major: 8-key row groups 1024 B apart, 64-element d atoms 16 KB apart
                    const uint64_t bd = sw128_desc(vbase + k * C::kKStep * 128, 16384, 1024);
                    const uint32_t a = tmem + kColS + pb * 128 + k * (C::kKStep * C::kEb / 4);
                    const uint32_t acc = (!first || k > 0) ? 1u : 0u;
                    if (kDtype == FP_DTYPE_BF16)
                        umma_f16_ts(tmem + kColO, a, bd, C::kIdescPV, acc);
                    else
                        umma_f8_ts(tmem + kColO, a, bd, C::kIdescPV, acc);
                }
                if constexpr (kDtype == FP_DTYPE_E4M3) {
                    // Eq.15's denominator: sum of the quantised P~ per row, accumulated like O (N = 16)
                    const uint32_t obase = smem_addr(sm.ones.w);
#pragma unroll
                    for (int k = 0; k < C::kNumK; ++k)
                        umma_f8_ts(tmem + kColL, tmem + kColS + pb * 128 + k * (C::kKStep * C::kEb / 4),
                                   sw128_desc(obase + k * 32, 16, 1024), kIdescL8, (!first || k > 0) ? 1u : 0u);
                }
                if (fl & 2) umma_commit(&sm.o_full);
            };
            for (uint32_t g = 0;; ++g) {
                // a wait whose outcome is the same in every lane, so the warp stays converged for elect.sync. It
                // probes once, then blocks in try_wait rather than spinning: the warp shares its scheduler with
                // two softmax warps, and the softmax is what this wait is usually for
                if (!__all_sync(0xffffffffu, mbar_wait(&sm.go[g & 1], (g >> 1) & 1, ab))) break;
                const int4 gr = *reinterpret_cast<const int4 *>(&sm.group[g % kGroupRing]);  // pv, qk, qb, end
                if (gr.w) break;
                if (elect_one()) {
                    tc_fence_after();
                    if (gr.x >= 0) issue_pv(g - 2, gr.x);
                    if (gr.y >= 0) issue_qk(g, gr.y, gr.z);
                    umma_commit(&sm.grp[g & 3]);
                }
                __syncwarp();
            }
        }
    } else if (warp < 12) {
        regs_set<kRegsSoftmax>();
        // -------------------------------------------------------------------------- softmax
        // Warp w owns 16 rows of the tile: TMEM lanes 32 (w % 4) + 16 sub .. + 15 (TMEM lane = packed row).
        // Thread t holds row 32 (w % 4) + 16 sub + t % 16 and the half t / 16 of its 128 keys, 64 consecutive
        // ones (the .16x32bx2 shapes: the two half-warps read the same lanes at column offsets 0 and 64). The
        // TMEM load returns the thread's maximum with the scores, and a row's two threads (t, t ^ 16) combine
        // maxima and sums with one shuffle.
        const int quarter = warp & 3, sub = (warp - 4) >> 2;
        const int half = lane >> 4;
        const int row = 32 * quarter + 16 * sub + (lane & 15);  // row of the tile
        const uint32_t tlane = static_cast<uint32_t>(32 * quarter + 16 * sub) << 16;
        const float LOG2E = 1.4426950408889634f;
        const float sl2 = P.c_q * P.c_k * LOG2E * rsqrtf((float)kHeadDim);
        // lazy rescale slack (log2 units): bf16 P may reach 2^8; FP8 P~ must stay within [0, 256]
        const float tau = kDtype == FP_DTYPE_E4M3 ? 0.f : 8.f;
        const float pshift = kDtype == FP_DTYPE_E4M3 ? 8.f : 0.f;  // FP8 probabilities in [0, 256] (Eq.15)
        const int gshift = __ffs(g) - 1;                            // g is a power of two
        float mx = -INFINITY, l = 0.f;  // the row's running maximum (log2 units); l: this thread's half of the sum
        for (uint32_t gi = 0;; ++gi) {
            const int slot = gi % kRing;
            if (!mbar_wait(&sm.rec_full[slot], (gi / kRing) & 1, ab)) break;
            const IterRec &rc = sm.ring[slot];
            const int J = rc.J, fl = rc.flags, D = rc.D, tile = rc.tile, row0 = rc.row0;
            uint4 mw = make_uint4(0, 0, 0, 0);
            if (J < 0) mw = make_uint4(rc.u.c.mask[0], rc.u.c.mask[1], rc.u.c.mask[2], rc.u.c.mask[3]);
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.rec_empty[slot]);
            if (J == kRecEnd) break;
            const int sb = gi & 1;
            const uint32_t tS = tmem + tlane + kColS + sb * 128;
            const uint32_t tO = tmem + tlane + kColO;
            const bool first = fl & 1;
            if (first) {
                mx = -INFINITY;
                l = 0.f;
            }
            if (!mbar_wait(&sm.grp[gi & 3], (gi >> 2) & 1, ab)) break;  // group gi computed S(gi)
            tc_fence_after();
            // v[j]: key 64 half + j of the thread's row; rmax their maximum
            const float shift = J < 0 ? 7.f : 0.f;  // log2 |B_J| of a full 128-token block for means
            const bool plain = J >= 0 ? J != D : (mw.x & mw.y & mw.z & mw.w) == 0xffffffffu;
            uint32_t v[64];
            float rmax;
            if (plain) {
                tmem_ld_16x32bx2_x64_max<64>(tS, v, rmax);
                tmem_ld_wait();
                reg_fence64(v);
                asm volatile("" : "+f"(rmax));
            } else {
                // Masked keys become -inf and the maximum is taken over the rest. The thread's 64 keys load as
                // four groups of 16, each with its maximum: a group whose keys are all kept keeps that maximum,
                // and only a group the mask cuts through is masked key by key.
                float gm[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) tmem_ld_16x32bx2_x16_max<64>(tS + 16 * q, v + 16 * q, gm[q]);
                tmem_ld_wait();
                reg_fence64(v);
                asm volatile("" : "+f"(gm[0]), "+f"(gm[1]), "+f"(gm[2]), "+f"(gm[3]));
                // kept keys of the thread's half: bit j of kw[j / 32] for key 64 half + j
                uint32_t kw0, kw1;
                if (J >= 0) {
                    // causal mask on the diagonal block: key <= position - 128 J
                    const int lim = ((row0 + row) >> gshift) - J * kBlock - 64 * half;
                    kw0 = lim >= 31 ? 0xffffffffu : lim < 0 ? 0u : (2u << lim) - 1u;
                    kw1 = lim >= 63 ? 0xffffffffu : lim < 32 ? 0u : (2u << (lim - 32)) - 1u;
                } else {
                    // correction chunk: keep the means of pruned blocks only (bit k & 31 of word k / 32)
                    kw0 = half ? mw.z : mw.x;
                    kw1 = half ? mw.w : mw.y;
                }
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const uint32_t b = ((q < 2 ? kw0 : kw1) >> (16 * (q & 1))) & 0xffffu;
                    if (b == 0u) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) v[16 * q + i] = __float_as_uint(-INFINITY);
                        gm[q] = -INFINITY;
                    } else if (b != 0xffffu) {
                        float p0 = -INFINITY, p1 = -INFINITY;
#pragma unroll
                        for (int i = 0; i < 16; i += 2) {
                            const float x0 = (b >> i) & 1u ? __uint_as_float(v[16 * q + i]) : -INFINITY;
                            const float x1 = (b >> (i + 1)) & 1u ? __uint_as_float(v[16 * q + i + 1]) : -INFINITY;
                            v[16 * q + i] = __float_as_uint(x0);
                            v[16 * q + i + 1] = __float_as_uint(x1);
                            p0 = fmaxf(p0, x0);
                            p1 = fmaxf(p1, x1);
                        }
                        gm[q] = fmaxf(p0, p1);
                    }
                }
                rmax = fmaxf(fmaxf(gm[0], gm[1]), fmaxf(gm[2], gm[3]));
            }
            rmax = fmaxf(rmax, __shfl_xor_sync(0xffffffffu, rmax, 16));
            const float tm = fmaf(rmax, sl2, shift);
            // online softmax with lazy rescaling of O
            const bool grow = first || tm > mx + tau;
            const float mn = grow ? fmaxf(mx, tm) : mx;
            const bool need_o = !first && grow;
            const float fo = need_o ? ex2(mx - mn) : 1.f;  // O's rescale factor
            if (!first) l *= ex2(mx - mn);
            mx = mn;
            // pass 2: p = 2^(x - m) (FP8: 2^(x - m + 8)), this thread's part of the row sum, P packed and written
            // over the S columns the PV MMA reads it from
            const float off = shift - mx + pshift;
            const uint64_t sl2x2 = f2pack(sl2, sl2), off2 = f2pack(off, off);
            uint64_t acc = f2pack(0.f, 0.f);
            if (kDtype == FP_DTYPE_BF16) {
                // P column 32 half + i holds keys 64 half + 2 i, + 1 as two bf16
                uint32_t pw[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    float y0, y1;
                    f2unpack(ffma2(f2pack(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])), sl2x2, off2), y0,
                             y1);
                    const float p0 = ex2(y0), p1 = ex2(y1);
                    acc = fadd2(acc, f2pack(p0, p1));
                    const __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
                    pw[i] = *reinterpret_cast<const uint32_t *>(&b2);
                }
                tmem_st_16x32bx2_x32<32>(tS, pw);
            } else {
                // P column 16 half + i holds keys 64 half + 4 i .. + 3 as four e4m3; Eq.15's denominator (the sum
                // of these quantised values) is accumulated by the tensor core next to O
                uint32_t pw[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int k = 4 * i;
                    float y0, y1, y2, y3;
                    f2unpack(ffma2(f2pack(__uint_as_float(v[k]), __uint_as_float(v[k + 1])), sl2x2, off2), y0, y1);
                    f2unpack(ffma2(f2pack(__uint_as_float(v[k + 2]), __uint_as_float(v[k + 3])), sl2x2, off2), y2, y3);
                    const __nv_fp8x2_e4m3 qa(make_float2(ex2(y0), ex2(y1))), qb(make_float2(ex2(y2), ex2(y3)));
                    pw[i] = (uint32_t)qa.__x | ((uint32_t)qb.__x << 16);
                }
                tmem_st_16x32bx2_x16<16>(tS, pw);
            }
            if constexpr (kDtype == FP_DTYPE_BF16) {
                float s0, s1;
                f2unpack(acc, s0, s1);
                l += s0 + s1;
            }
            if (__any_sync(0xffffffffu, need_o)) {
                // O holds the sum up to iteration gi-1 of this tile: wait for that PV (in group gi + 1),
                // then rescale this thread's half of its row in TMEM. Done after P is written, while the
                // scores are no longer live; the PV of this iteration waits for the arrival below.
                if (!mbar_wait(&sm.grp[(gi + 1) & 3], ((gi + 1) >> 2) & 1, ab)) break;
                tc_fence_after();
                const uint64_t f2 = f2pack(fo, fo);
                // 16 columns at a time
#pragma unroll
                for (int c = 0; c < 64; c += 16) {
                    uint32_t ov[16];
                    tmem_ld_16x32bx2_x16<64>(tO + c, ov);
                    tmem_ld_wait();
                    reg_fence16(ov);
#pragma unroll
                    for (int k = 0; k < 16; k += 2) {
                        float x0, x1;
                        f2unpack(fmul2(f2pack(__uint_as_float(ov[k]), __uint_as_float(ov[k + 1])), f2), x0, x1);
                        ov[k] = __float_as_uint(x0);
                        ov[k + 1] = __float_as_uint(x1);
                    }
                    tmem_st_16x32bx2_x16<64>(tO + c, ov);
                }
                if constexpr (kDtype == FP_DTYPE_E4M3) {
                    // the row sum accumulated beside O takes the same factor (columns 0 and 8 of its 16)
                    uint32_t lw;
                    tmem_ld_16x32bx2_x1<8>(tmem + tlane + kColL, lw);
                    tmem_ld_wait();
                    tmem_st_16x32bx2_x1<8>(tmem + tlane + kColL, __float_as_uint(__uint_as_float(lw) * fo));
                }
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.go[sb]);  // P(gi) is ready for group gi + 2
            if (fl & 2) {
                // hand the row statistics to the epilogue once it has finished the previous tile
                const float lr = l + __shfl_xor_sync(0xffffffffu, l, 16);
                if (!mbar_wait(&sm.o_empty, (tile & 1) ^ 1, ab)) break;
                if (half == 0) {
                    sm.stat_m[row] = mx;
                    sm.stat_l[row] = lr;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.st_full);
            }
        }
    } else {
        regs_set<kRegsEpilogue>();
        // ------------------------------------------------------------------------- epilogue
        const int j = 32 * (warp & 3) + lane;
        const uint32_t tlane = static_cast<uint32_t>(32 * (warp & 3)) << 16;
        const float pshift = kDtype == FP_DTYPE_E4M3 ? 8.f : 0.f;
        bool ok = true;
        uint32_t ti = 0;
        int w = blockIdx.x;
        const int nitems = kSplit ? sm.nitems : P.nseg;
        TileTask cur;
        if (w < nitems) cur = P.tasks[w];
        while (w < nitems && ok) {
            const int wn = w + gridDim.x;
            TileTask nxt;
            if (wn < nitems) nxt = P.tasks[wn];
            const int gr = cur.t * kTileRows + j;
            const int64_t rowi = (int64_t)(cur.q_start + gr / g) * P.hq + cur.h * g + gr % g;
            const bool valid = j >= cur.lo && j < cur.rows;
            if (task_live<kSplit>(cur)) {
                if (!(ok = mbar_wait(&sm.o_full, ti & 1, ab))) break;
                if (!(ok = mbar_wait(&sm.st_full, ti & 1, ab))) break;
                tc_fence_after();
                float l;
                if constexpr (kDtype == FP_DTYPE_E4M3) {
                    // Eq.15's denominator from the tensor core (read before O is released below)
                    uint32_t lw;
                    tmem_ld_32x32b_x1(tmem + tlane + kColL, lw);
                    tmem_ld_wait();
                    l = __uint_as_float(lw);
                } else {
                    l = sm.stat_l[j];
                }
                const float mx = sm.stat_m[j];
                const float inv = l > 0.f ? P.c_v / l : 0.f;
                const bool part = kSplit && cur.slot >= 0;  // one run of a split tile: fp32 partial output
                __nv_bfloat16 *orow = P.out + rowi * kHeadDim;
                float *prow = P.part_o + ((int64_t)cur.slot * kTileRows + j) * kHeadDim;
#pragma unroll
                for (int q2 = 0; q2 < 2; ++q2) {
                    uint32_t ov[2][32];
                    tmem_ld32(tmem + tlane + kColO + q2 * 64, ov[0]);
                    tmem_ld32(tmem + tlane + kColO + q2 * 64 + 32, ov[1]);
                    tmem_ld_wait();
                    reg_fence32(ov[0]);
                    reg_fence32(ov[1]);
                    if (q2 == 1) {
                        // O is in registers: the next tile's PVs may overwrite it
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&sm.o_empty);
                    }
                    if (valid && !part) {
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
#pragma unroll
                            for (int e = 0; e < 32; e += 8) {
                                uint4 pk;
                                uint32_t *pw = reinterpret_cast<uint32_t *>(&pk);
#pragma unroll
                                for (int u = 0; u < 4; ++u) {
                                    const __nv_bfloat162 b2 =
                                        __floats2bfloat162_rn(__uint_as_float(ov[hh][e + 2 * u]) * inv,
                                                              __uint_as_float(ov[hh][e + 2 * u + 1]) * inv);
                                    pw[u] = *reinterpret_cast<const uint32_t *>(&b2);
                                }
                                *reinterpret_cast<uint4 *>(orow + q2 * 64 + hh * 32 + e) = pk;
                            }
                        }
                    } else if (valid) {
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
                            for (int e = 0; e < 32; e += 4)
                                *reinterpret_cast<float4 *>(prow + q2 * 64 + hh * 32 + e) =
                                    make_float4(__uint_as_float(ov[hh][e]) * inv, __uint_as_float(ov[hh][e + 1]) * inv,
                                                __uint_as_float(ov[hh][e + 2]) * inv,
                                                __uint_as_float(ov[hh][e + 3]) * inv);
                    }
                }
                if (!part) {
                    if (valid && P.lse) P.lse[rowi] = (mx + log2f(l) - pshift) * 0.6931471805599453f;
                } else {
                    if (valid)
                        P.part_lse[cur.slot * kTileRows + j] =
                            l > 0.f ? (mx + log2f(l) - pshift) * 0.6931471805599453f : -INFINITY;
                }
                ++ti;
            } else if (cur.n_exact == 0 && cur.n_chunks == 0 && valid) {
                // a well-formed segment with nothing to attend: zero rows
                for (int e = 0; e < kHeadDim; e += 8)
                    *reinterpret_cast<uint4 *>(P.out + rowi * kHeadDim + e) = make_uint4(0, 0, 0, 0);
                if (P.lse) P.lse[rowi] = -INFINITY;
            }
            cur = nxt;
            w = wn;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (sm.abort && threadIdx.x == 0) set_status(status, FP_ERR_DEVICE_TIMEOUT, blockIdx.x);
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Dynamic shared memory to request: the layout plus slack for 1024-byte
// alignment, capped at the device's opt-in maximum (the kernel checks that
// its aligned layout fits and reports an error otherwise).
size_t smem_request(size_t layout) {
    int dev = 0, cap = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&cap, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess || cap <= 0)
        cap = 232448;
    return layout + 1024 <= (size_t)cap ? layout + 1024 : (size_t)cap;
}

}  // namespace

cudaError_t launch_attention(const Ctx &c, const void *q, const void *k_pages, const void *v_pages,
                             const int32_t *csr_cu, const int32_t *csr_idx, int64_t capacity, const void *kbar_op,
                             const void *vbar_op, int flags, void *out, float *lse, int32_t *trace,
                             int32_t trace_words) {
    const int32_t nseg = (int32_t)c.s.nseg;
    // the histogram and, past it, the largest cost
    cudaError_t e = cudaMemsetAsync(c.hist(), 0, sizeof(int32_t) * (kCostBuckets + 1), c.stream);
    if (e != cudaSuccess) return e;
    attn_meta_kernel<<<(nseg + kMetaSegs - 1) / kMetaSegs, 256, 0, c.stream>>>(c.req(), c.p.batch, c.s.g, nseg, csr_cu, csr_idx,
                                                            capacity, flags, c.meta(), c.mask(), c.hist(),
                                                            c.status());
    // KV splits pay off only when the tiles do not fill the GPU several times over; larger problems run the
    // kernel without the split path (every tile one work item)
    const bool split = nseg < kSplitTilesPerSm * num_sms();
    const int split_ctas = !split ? 0 : num_sms() < kSplitCtas ? num_sms() : kSplitCtas;
    attn_bucket_kernel<<<1, 1024, 0, c.stream>>>(c.hist(), c.counters(), split_ctas, c.status());
    attn_scatter_kernel<<<(nseg + 255) / 256, 256, 0, c.stream>>>(c.req(), c.p.batch, c.s.g, c.meta(), nseg, csr_cu,
                                                                   flags, c.hist(), c.counters(), c.splits(),
                                                                   c.tasks(), c.status());
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    const bool fp8 = c.p.dtype == FP_DTYPE_E4M3;
    const int eb = fp8 ? 1 : 2;
    const int g = c.s.g, hkv = c.p.num_kv_heads, hq = c.p.num_q_heads;
    const int ps_eff = c.p.page_size < 128 ? c.p.page_size : 128;
    CUtensorMap tm_q, tm_k, tm_v, tm_kb, tm_vb;
    {
        const uint64_t dims[4] = {128, (uint64_t)g, (uint64_t)hkv, (uint64_t)c.s.total_tokens};
        const uint64_t strides[3] = {(uint64_t)128 * eb, (uint64_t)g * 128 * eb, (uint64_t)hq * 128 * eb};
        const uint32_t box[4] = {(uint32_t)(128 / eb), (uint32_t)g, 1, (uint32_t)(kTileRows / g)};
        if (!make_tmap(&tm_q, q, fp8, 4, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t dims[3] = {128, (uint64_t)hkv, (uint64_t)c.p.num_pages * c.p.page_size};
        const uint64_t strides[2] = {(uint64_t)128 * eb, (uint64_t)hkv * 128 * eb};
        const uint32_t box[3] = {(uint32_t)(128 / eb), 1, (uint32_t)ps_eff};
        if (!make_tmap(&tm_k, k_pages, fp8, 3, dims, strides, box)) return cudaErrorInvalidValue;
        if (!make_tmap(&tm_v, v_pages, fp8, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    const bool corr = (flags & FP_MEAN_CORRECTION) && !(flags & FP_DENSE);
    {
        // means: the caller's arrays when the correction is on, else any valid mapping (never read)
        const void *kb = corr ? kbar_op : k_pages, *vb = corr ? vbar_op : v_pages;
        const uint64_t rows = corr ? (uint64_t)c.s.nblocks : (uint64_t)c.p.num_pages * c.p.page_size;
        const uint64_t dims[3] = {128, (uint64_t)hkv, rows};
        const uint64_t strides[2] = {(uint64_t)128 * eb, (uint64_t)hkv * 128 * eb};
        const uint32_t box[3] = {(uint32_t)(128 / eb), 1, 128};
        if (!make_tmap(&tm_kb, kb, fp8, 3, dims, strides, box)) return cudaErrorInvalidValue;
        if (!make_tmap(&tm_vb, vb, fp8, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    // with splits every SM: the work list may hold more runs than segments
    const int grid = split || nseg > num_sms() ? num_sms() : nseg;
    AttnParams prm;
    prm.pt = c.p.page_table;
    prm.pt_stride = c.p.page_table_stride;
    prm.num_pages = c.p.num_pages;
    prm.page_size = c.p.page_size;
    prm.csr_idx = csr_idx;
    prm.todo = c.mask();
    prm.tasks = c.tasks();
    prm.out = (__nv_bfloat16 *)out;
    prm.lse = lse;
    prm.hq = hq;
    prm.g = g;
    prm.flags = flags;
    prm.c_q = fp8 ? c.p.c_q : 1.f;
    prm.c_k = fp8 ? c.p.c_k : 1.f;
    prm.c_v = fp8 ? c.p.c_v : 1.f;
    prm.nseg = nseg;
    prm.nitems = c.counters() + kCntItems;
    prm.part_o = c.part_o();
    prm.part_lse = c.part_lse();
    prm.status = c.status();
    prm.trace = trace;
    prm.trace_cap = trace_words;
    if (trace && (e = cudaMemsetAsync(trace, 0, kTraceHeader * sizeof(int32_t), c.stream)) != cudaSuccess) return e;
    auto launch = [&](auto kernel, size_t layout) -> cudaError_t {
        const size_t smem = smem_request(layout);
        prm.smem_bytes = (uint32_t)smem;
        cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        kernel<<<grid, kAThreads, smem, c.stream>>>(tm_q, tm_k, tm_v, tm_kb, tm_vb, prm);
        return cudaSuccess;
    };
    // the traced variants differ only in the walker's recording of its records
    const size_t lay = fp8 ? sizeof(AttnSmem<FP_DTYPE_E4M3>) : sizeof(AttnSmem<FP_DTYPE_BF16>);
    if (trace) {
        if (fp8)
            e = split ? launch(attn_tc_kernel<FP_DTYPE_E4M3, true, true>, lay)
                      : launch(attn_tc_kernel<FP_DTYPE_E4M3, false, true>, lay);
        else
            e = split ? launch(attn_tc_kernel<FP_DTYPE_BF16, true, true>, lay)
                      : launch(attn_tc_kernel<FP_DTYPE_BF16, false, true>, lay);
    } else if (fp8) {
        e = split ? launch(attn_tc_kernel<FP_DTYPE_E4M3, true, false>, lay)
                  : launch(attn_tc_kernel<FP_DTYPE_E4M3, false, false>, lay);
    } else {
        e = split ? launch(attn_tc_kernel<FP_DTYPE_BF16, true, false>, lay)
                  : launch(attn_tc_kernel<FP_DTYPE_BF16, false, false>, lay);
    }
    if (e != cudaSuccess) return e;
    if (split)
        attn_combine_kernel<<<4 * kCombineTiles, kCombineThreads, 0, c.stream>>>(
            c.splits(), c.counters(), c.part_o(), c.part_lse(), (__nv_bfloat16 *)out, lse, hq, g, c.status());
    return cudaGetLastError();
}

}  // namespace fp
