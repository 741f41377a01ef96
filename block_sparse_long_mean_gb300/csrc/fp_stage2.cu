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
// softmax warps keep one row per thread (online softmax in the base-2
// domain, causal mask on the diagonal block, the log2|B_J| = 7 shift and the
// correction mask on mean chunks, lazy rescaling of O); epilogue warps divide
// by the denominator and write bf16 O and the LSE.
// FP8 (Eq.15): Q, K, V and the means are E4M3, S = c_q c_k (Q~ K~^T),
// P~ = e4m3(256 * 2^(x - m)) with the denominator summing P~, O = c_v ... / l.
#include <math.h>

#include "fp_internal.cuh"
#include "sm100_ptx.cuh"

namespace fp {
namespace {

using namespace sm100;

// ------------------------------------------------------------ schedule prep

// One warp per segment: validates its CSR, counts selected blocks per
// 128-block chunk, and records the iteration counts and chunk mask.
__global__ void __launch_bounds__(256) attn_meta_kernel(const ReqInfo *__restrict__ req, int batch, int g,
                                                        int32_t nseg, const int32_t *__restrict__ cu,
                                                        const int32_t *__restrict__ idx, int64_t capacity, int flags,
                                                        SegMeta *__restrict__ meta, uint32_t *__restrict__ todo,
                                                        int32_t *__restrict__ hist, int32_t *__restrict__ status) {
    __shared__ int cnt[8][kMaxChunks];
    if (status_bad(status)) return;
    const int lane = threadIdx.x & 31, wl = threadIdx.x >> 5;
    const int64_t seg = (int64_t)blockIdx.x * 8 + wl;
    if (seg >= nseg) return;
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
    if (lane == 0) {
        meta[seg] = m;
        const int cost = m.n_exact < 0 ? 0 : min(m.n_exact + m.n_chunks, kCostBuckets - 1);
        atomicAdd(&hist[cost], 1);
    }
}

// Turns the cost histogram into descending-cost bucket offsets (one CTA).
__global__ void __launch_bounds__(1024) attn_bucket_kernel(int32_t *__restrict__ hist, int32_t *__restrict__ status) {
    __shared__ int32_t warp_sums[32];
    __shared__ int32_t carry;
    if (status_bad(status)) return;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int base = 0; base < kCostBuckets; base += 1024) {
        const int i = base + threadIdx.x;
        const int bucket = kCostBuckets - 1 - i;  // descending cost
        int32_t v = i < kCostBuckets ? hist[bucket] : 0;
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
        if (i < kCostBuckets) hist[bucket] = excl;
        if (threadIdx.x == 0) carry += total;
        __syncthreads();
    }
}

__global__ void __launch_bounds__(256) attn_scatter_kernel(const SegMeta *__restrict__ meta, int32_t nseg,
                                                           int32_t *__restrict__ hist, int32_t *__restrict__ work,
                                                           int32_t *__restrict__ status) {
    if (status_bad(status)) return;
    const int64_t seg = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (seg >= nseg) return;
    const SegMeta m = meta[seg];
    const int cost = m.n_exact < 0 ? 0 : min(m.n_exact + m.n_chunks, kCostBuckets - 1);
    work[atomicAdd(&hist[cost], 1)] = (int32_t)seg;
}

// --------------------------------------------------------------- attention

// Warp roles (three warpgroups; registers rebalanced with setmaxnreg):
//   warp 0      Q and K producer (TMA)     warp 1   MMA issuer + TMEM owner
//   warp 2      V producer (TMA)           warp 3   idle
//   warps 4-7   softmax, one thread per packed row
//   warps 8-11  epilogue: O / l to bf16, LSE
// TMEM: two S buffers (P of an iteration is written over its S), two O buffers.
// The MMA warp issues QK^T of iteration i+1 before PV of iteration i, so the
// tensor core computes the next scores while the softmax works on these.
// Every tcgen05.mma of the CTA comes from one thread and executes in issue
// order, so QK^T(i+2) may be issued right after PV(i), which read P(i) from
// the same columns. O is double-buffered so one tile's epilogue overlaps the
// next tile's PVs.
constexpr int kAWarps = 12;
constexpr int kAThreads = 32 * kAWarps;
constexpr int kKStages = 3, kVStages = 2;
constexpr uint32_t kColS = 0, kColO = 256;  // S_b at 128 b, O_o at 256 + 128 o
constexpr int kRegsProducer = 56, kRegsSoftmax = 232, kRegsEpilogue = 160;  // 128 x (56 + 232 + 160) <= 384 x 168

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

template <int kDtype>
struct AttnSmem {
    alignas(1024) uint8_t q[2][ACfg<kDtype>::kTile];
    alignas(1024) uint8_t k[kKStages][ACfg<kDtype>::kTile];
    alignas(1024) uint8_t v[kVStages][ACfg<kDtype>::kTile];
    float stat_m[2][128], stat_l[2][128];  // per O buffer: running max (log2) and denominator of each row
    uint64_t q_full[2], q_empty[2], k_full[kKStages], k_empty[kKStages], v_full[kVStages], v_empty[kVStages],
        s_full[2], p_full[2], pv_done[2], o_full[2], o_empty[2], st_full[2];
    uint32_t tmem_base;
    int abort, skip;
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <uint32_t kRegs>
__device__ __forceinline__ void regs_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegs));
}
template <uint32_t kRegs>
__device__ __forceinline__ void regs_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegs));
}

// Kernel arguments besides the tensor maps (read from the constant bank).
struct AttnParams {
    const int32_t *pt;  // page table
    int pt_stride, num_pages, page_size;
    const int32_t *csr_cu, *csr_idx;
    const SegMeta *meta;
    const uint32_t *todo;  // per-segment correction bitmaps
    const int32_t *work;   // segments, heaviest first
    __nv_bfloat16 *out;
    float *lse;
    const ReqInfo *req;
    int batch, hq, g, flags;
    float c_q, c_k, c_v;
    int32_t nseg;
    uint32_t smem_bytes;
    int32_t *status;
};

// Walk over this CTA's tiles (work items blockIdx.x + k gridDim.x, skipping
// empty or malformed segments) and each tile's iterations: the selected blocks
// in descending order (Eq.17), then the correction chunks.
struct TileWalk {
    int w, seg, n, it, n_exact;
    SegCoord sc;
    int32_t end;
    uint64_t chunks;
    bool live;
    __device__ __forceinline__ void start(const AttnParams &a) {
        w = (int)blockIdx.x - (int)gridDim.x;
        n = it = 0;
        live = true;
        next_tile(a);
    }
    // moves to the next tile holding at least one iteration; live = false when none is left
    __device__ __forceinline__ void next_tile(const AttnParams &a) {
        for (;;) {
            w += gridDim.x;
            if (w >= a.nseg) {
                live = false;
                return;
            }
            seg = a.work[w];
            const SegMeta m = a.meta[seg];
            if (m.n_exact < 0 || m.n_exact + m.n_chunks == 0) continue;
            sc = decode_seg(a.req, a.batch, a.g, seg);
            n_exact = m.n_exact;
            n = m.n_exact + m.n_chunks;
            it = 0;
            end = (a.flags & FP_DENSE) ? 0 : (int32_t)a.csr_cu[seg + 1];
            chunks = ((uint64_t)m.chunk_hi << 32) | m.chunk_lo;
            return;
        }
    }
    // block id (>= 0) or correction chunk (-1 - c) of iteration `it`, then advances
    __device__ __forceinline__ int take(const AttnParams &a) {
        int J;
        if (it < n_exact) {
            J = (a.flags & FP_DENSE) ? sc.D - it : a.csr_idx[end - 1 - it];
        } else {
            const int c = 63 - __clzll((long long)chunks);
            chunks &= ~(1ull << c);
            J = -1 - c;
        }
        ++it;
        return J;
    }
};

template <int kDtype>
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
            mbar_init(&sm.q_full[i], 1);
            mbar_init(&sm.q_empty[i], 1);
            mbar_init(&sm.s_full[i], 1);
            mbar_init(&sm.p_full[i], 4);
            mbar_init(&sm.pv_done[i], 1);
            mbar_init(&sm.o_full[i], 1);
            mbar_init(&sm.o_empty[i], 4);
            mbar_init(&sm.st_full[i], 4);
        }
        for (int i = 0; i < kKStages; ++i) {
            mbar_init(&sm.k_full[i], 1);
            mbar_init(&sm.k_empty[i], 1);
        }
        for (int i = 0; i < kVStages; ++i) {
            mbar_init(&sm.v_full[i], 1);
            mbar_init(&sm.v_empty[i], 1);
        }
        sm.abort = 0;
        // an earlier stage failed: every warp skips its role (one read, so the CTA agrees)
        sm.skip = status_bad(P.status) ? 1 : 0;
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(&sm.tmem_base, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const Abort ab{&sm.abort};
    const uint32_t tmem = sm.tmem_base;

    if (sm.skip) {
    } else if (warp < 4) {
        regs_dec<kRegsProducer>();
        if (warp == 0 || warp == 2) {
            // ------------------------------------------------ Q + K (warp 0) / V (warp 2) producer
            const bool is_k = warp == 0;
            if (lane == 0) {
                if (is_k) tma_prefetch_desc(&tm_q);
                tma_prefetch_desc(is_k ? &tm_k : &tm_v);
                tma_prefetch_desc(is_k ? &tm_kb : &tm_vb);
            }
            const int ps_eff = min(P.page_size, 128);
            const int npc = 128 / ps_eff;                   // page chunks per 128-token block
            const int oob_row = P.num_pages * P.page_size;  // first row past the pool: TMA fills zeros
            const int nst = is_k ? kKStages : kVStages;
            uint64_t *fullb = is_k ? sm.k_full : sm.v_full;
            uint64_t *emptyb = is_k ? sm.k_empty : sm.v_empty;
            TileWalk s;
            s.start(P);
            uint32_t gi = 0;
            bool ok = true;
            for (uint32_t ti = 0; s.live && ok; ++ti) {
                const ReqInfo r = P.req[s.sc.b];
                const int h = s.sc.h, b = s.sc.b;
                if (is_k) {
                    const int qb = ti & 1;
                    if (!(ok = mbar_wait(&sm.q_empty[qb], ((ti >> 1) & 1) ^ 1, ab))) break;
                    if (lane == 0) {
                        mbar_arrive_expect_tx(&sm.q_full[qb], C::kTile);
                        const int pos0 = r.q_start + (s.sc.t * kTileRows) / g;
                        for (int i = 0; i < C::kBoxes; ++i)
                            tma_load_4d(sm.q[qb] + i * 16384, &tm_q, &sm.q_full[qb], i * C::kBoxElems, 0, h, pos0);
                    }
                }
                const int n = s.n;
                for (int it = 0; it < n; ++it, ++gi) {
                    const int J = s.take(P);
                    // lane l < kBoxes * npc (<= 32 as page_size >= 8) copies page chunk l % npc of d box l / npc;
                    // its page row is looked up before waiting for the slot
                    int row = oob_row;
                    if (J >= 0 && lane < C::kBoxes * npc) {
                        const int tok = J * kBlock + (lane % npc) * ps_eff;
                        if (tok < r.len) {
                            const int page = P.pt[(int64_t)b * P.pt_stride + tok / P.page_size];
                            if (page >= 0 && page < P.num_pages)
                                row = page * P.page_size + tok % P.page_size;
                            else
                                set_status(status, FP_ERR_DEVICE_PAGE, page);
                        }
                    }
                    const int st = gi % nst;
                    if (!(ok = mbar_wait(&emptyb[st], ((gi / nst) & 1) ^ 1, ab))) break;
                    if (lane == 0) mbar_arrive_expect_tx(&fullb[st], C::kTile);
                    __syncwarp();
                    uint8_t *dst = is_k ? sm.k[st] : sm.v[st];
                    if (J >= 0) {
                        if (lane < C::kBoxes * npc) {
                            const int box = lane / npc, pc = lane % npc;
                            tma_load_3d(dst + box * 16384 + pc * ps_eff * 128, is_k ? &tm_k : &tm_v, &fullb[st],
                                        box * C::kBoxElems, h, row);
                        }
                    } else if (lane < C::kBoxes) {
                        tma_load_3d(dst + lane * 16384, is_k ? &tm_kb : &tm_vb, &fullb[st], lane * C::kBoxElems, h,
                                    r.blk_base + 128 * (-1 - J));
                    }
                }
                s.next_tile(P);
            }
        } else if (warp == 1 && lane == 0) {
            // ------------------------------------------------------------------ MMA issue
            TileWalk s;
            s.start(P);
            uint32_t gi = 0;
            bool ok = true;
            // O_ob (+)= P(i) V(i); the first PV of a tile overwrites O_ob once its previous epilogue read it
            auto issue_pv = [&](uint32_t i, bool first, int ob, uint32_t ti) -> bool {
                const int vs = i % kVStages, pb = i & 1;
                if (first && !mbar_wait(&sm.o_empty[ob], ((ti >> 1) & 1) ^ 1, ab)) return false;
                if (!mbar_wait(&sm.v_full[vs], (i / kVStages) & 1, ab)) return false;
                if (!mbar_wait(&sm.p_full[pb], (i >> 1) & 1, ab)) return false;
                tc_fence_after();
                const uint32_t vbase = smem_addr(sm.v[vs]);
#pragma unroll
                for (int k = 0; k < C::kNumK; ++k) {
                    // B = V, MN-major: 8-key row groups 1024 B apart, 64-element d atoms 16 KB apart
                    const uint64_t bd = sw128_desc(vbase + k * C::kKStep * 128, 16384, 1024);
                    const uint32_t a = tmem + kColS + pb * 128 + k * (C::kKStep * C::kEb / 4);
                    const uint32_t acc = (!first || k > 0) ? 1u : 0u;
                    if (kDtype == FP_DTYPE_BF16)
                        umma_f16_ts(tmem + kColO + ob * 128, a, bd, C::kIdescPV, acc);
                    else
                        umma_f8_ts(tmem + kColO + ob * 128, a, bd, C::kIdescPV, acc);
                }
                umma_commit(&sm.v_empty[vs]);
                umma_commit(&sm.pv_done[pb]);
                return true;
            };
            for (uint32_t ti = 0; s.live && ok; ++ti) {
                const int qb = ti & 1, ob = ti & 1;
                const int n = s.n;
                if (!(ok = mbar_wait(&sm.q_full[qb], (ti >> 1) & 1, ab))) break;
                const uint32_t qbase = smem_addr(sm.q[qb]);
                for (int it = 0; it < n; ++it, ++gi) {
                    const int ks = gi % kKStages, sb = gi & 1;
                    if (!(ok = mbar_wait(&sm.k_full[ks], (gi / kKStages) & 1, ab))) break;
                    tc_fence_after();
                    const uint32_t kbase = smem_addr(sm.k[ks]);
#pragma unroll
                    for (int k = 0; k < C::kNumK; ++k) {
                        const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
                        const uint64_t ad = sw128_desc(qbase + off, 16, 1024);
                        const uint64_t bd = sw128_desc(kbase + off, 16, 1024);
                        if (kDtype == FP_DTYPE_BF16)
                            umma_f16_ss(tmem + kColS + sb * 128, ad, bd, C::kIdescQK, k > 0);
                        else
                            umma_f8_ss(tmem + kColS + sb * 128, ad, bd, C::kIdescQK, k > 0);
                    }
                    umma_commit(&sm.k_empty[ks]);
                    umma_commit(&sm.s_full[sb]);
                    if (it == n - 1) umma_commit(&sm.q_empty[qb]);
                    if (it >= 1 && !(ok = issue_pv(gi - 1, it == 1, ob, ti))) break;
                }
                if (!ok) break;
                if (!(ok = issue_pv(gi - 1, n == 1, ob, ti))) break;
                umma_commit(&sm.o_full[ob]);
                s.next_tile(P);
            }
        }
    } else if (warp < 8) {
        regs_inc<kRegsSoftmax>();
        // -------------------------------------------------------------------------- softmax
        const int j = 32 * (warp & 3) + lane;  // TMEM lane = packed row of the tile
        const uint32_t tlane = static_cast<uint32_t>(32 * (warp & 3)) << 16;
        const float LOG2E = 1.4426950408889634f;
        const float sl2 = P.c_q * P.c_k * LOG2E * rsqrtf((float)kHeadDim);
        // lazy rescale slack (log2 units): bf16 P may reach 2^8; FP8 P~ must stay within [0, 256]
        const float tau = kDtype == FP_DTYPE_E4M3 ? 0.f : 8.f;
        const float pshift = kDtype == FP_DTYPE_E4M3 ? 8.f : 0.f;  // FP8 probabilities in [0, 256] (Eq.15)
        TileWalk s;
        s.start(P);
        uint32_t gi = 0;
        bool ok = true;
        for (uint32_t ti = 0; s.live && ok; ++ti) {
            const int ob = ti & 1;
            const SegCoord sc = s.sc;
            const ReqInfo r = P.req[sc.b];
            const int pos = (sc.t * kTileRows + j) / g;
            const uint32_t *tw = P.todo + (int64_t)r.mask_base + (int64_t)(sc.h * r.ntiles + sc.t) * r.words;
            const int nw = (sc.D + 31) / 32;
            const int n = s.n;
            const uint32_t tO = tmem + tlane + kColO + ob * 128;
            float mx = -INFINITY, l = 0.f;
            for (int it = 0; it < n; ++it, ++gi) {
                const int sb = gi & 1;
                const uint32_t tS = tmem + tlane + kColS + sb * 128;
                const int J = s.take(P);
                uint4 mv = make_uint4(0, 0, 0, 0);  // correction-chunk key mask
                if (J < 0) {
                    const int c = -1 - J;
                    uint32_t wv[4];
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) wv[q4] = (4 * c + q4 < nw) ? __ldg(tw + 4 * c + q4) : 0u;
                    mv = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                }
                if (!(ok = mbar_wait(&sm.s_full[sb], (gi >> 1) & 1, ab))) break;
                tc_fence_after();
                uint32_t sv[4][32];
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) tmem_ld32(tS + q4 * 32, sv[q4]);
                tmem_ld_wait();
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) reg_fence32(sv[q4]);
                // pass 1: mask and row maximum of the raw dot products
                float pm[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) pm[u] = -INFINITY;
                const float shift = J < 0 ? 7.f : 0.f;  // log2 |B_J| of a full 128-token block for means
                const bool plain = J >= 0 ? J != sc.D : (mv.x & mv.y & mv.z & mv.w) == 0xffffffffu;
                if (plain) {
                    // every key takes part (a block off the diagonal, or a chunk with no selected block)
#pragma unroll
                    for (int e = 0; e < 128; e += 2)
                        pm[(e >> 1) & 7] = fmax3(pm[(e >> 1) & 7], __uint_as_float(sv[e >> 5][e & 31]),
                                                 __uint_as_float(sv[e >> 5][(e & 31) + 1]));
                } else if (J >= 0) {
                    const int lim = pos - J * kBlock;  // causal mask on the diagonal block
#pragma unroll
                    for (int e = 0; e < 128; ++e) {
                        const float v = e <= lim ? __uint_as_float(sv[e >> 5][e & 31]) : -INFINITY;
                        sv[e >> 5][e & 31] = __float_as_uint(v);
                        pm[e & 7] = fmaxf(pm[e & 7], v);
                    }
                } else {
                    const uint32_t wv[4] = {mv.x, mv.y, mv.z, mv.w};
#pragma unroll
                    for (int e = 0; e < 128; ++e) {
                        const float v = (wv[e >> 5] >> (e & 31)) & 1u ? __uint_as_float(sv[e >> 5][e & 31]) : -INFINITY;
                        sv[e >> 5][e & 31] = __float_as_uint(v);
                        pm[e & 7] = fmaxf(pm[e & 7], v);
                    }
                }
                const float rmax = fmax3(fmax3(pm[0], pm[1], pm[2]), fmax3(pm[3], pm[4], pm[5]), fmaxf(pm[6], pm[7]));
                const float tmax = fmaf(rmax, sl2, shift);
                // online softmax with lazy rescaling of O
                const bool first = it == 0;
                const bool grow = first || tmax > mx + tau;
                const float m_new = grow ? fmaxf(mx, tmax) : mx;
                const bool need_o = !first && grow;
                if (__any_sync(0xffffffffu, need_o)) {
                    // O holds the sum up to iteration it-1: wait for that PV, then rescale it in TMEM
                    const uint32_t prev = gi - 1;
                    if (!(ok = mbar_wait(&sm.pv_done[prev & 1], (prev >> 1) & 1, ab))) break;
                    tc_fence_after();
                    const float f = need_o ? ex2(mx - m_new) : 1.f;
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint32_t ov[32];
                        tmem_ld32(tO + q4 * 32, ov);
                        tmem_ld_wait();
                        reg_fence32(ov);
#pragma unroll
                        for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * f);
                        tmem_st32(tO + q4 * 32, ov);
                    }
                }
                if (!first) l *= ex2(mx - m_new);
                mx = m_new;
                // pass 2: p = 2^(x - m) (FP8: 2^(x - m + 8)), row sum, P packed in place and written over S
                const float off = shift - mx + pshift;
                float ps4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint32_t *w32 = sv[q4];
                    if (kDtype == FP_DTYPE_BF16) {
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            const float p0 = ex2(fmaf(__uint_as_float(w32[2 * e]), sl2, off));
                            const float p1 = ex2(fmaf(__uint_as_float(w32[2 * e + 1]), sl2, off));
                            ps4[e & 3] += p0 + p1;
                            const __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
                            w32[e] = *reinterpret_cast<const uint32_t *>(&b2);
                        }
                        tmem_st16(tS + q4 * 16, w32);
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            uint32_t word = 0;
#pragma unroll
                            for (int b4 = 0; b4 < 4; b4 += 2) {
                                const float p0 = ex2(fmaf(__uint_as_float(w32[4 * e + b4]), sl2, off));
                                const float p1 = ex2(fmaf(__uint_as_float(w32[4 * e + b4 + 1]), sl2, off));
                                const __nv_fp8x2_e4m3 q2(make_float2(p0, p1));
                                const float2 back = float2(q2);  // Eq.15: the denominator sums the quantised values
                                ps4[e & 3] += back.x + back.y;
                                word |= (uint32_t)(*reinterpret_cast<const uint16_t *>(&q2)) << (8 * b4);
                            }
                            w32[e] = word;
                        }
                        tmem_st8(tS + q4 * 8, w32);
                    }
                }
                l += (ps4[0] + ps4[1]) + (ps4[2] + ps4[3]);
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.p_full[sb]);
            }
            if (!ok) break;
            // hand the row statistics to the epilogue (its previous use of this buffer must be done)
            if (!(ok = mbar_wait(&sm.o_empty[ob], ((ti >> 1) & 1) ^ 1, ab))) break;
            sm.stat_m[ob][j] = mx;
            sm.stat_l[ob][j] = l;
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.st_full[ob]);
            s.next_tile(P);
        }
    } else {
        regs_dec<kRegsEpilogue>();
        // ------------------------------------------------------------------------- epilogue
        const int j = 32 * (warp & 3) + lane;
        const uint32_t tlane = static_cast<uint32_t>(32 * (warp & 3)) << 16;
        const float pshift = kDtype == FP_DTYPE_E4M3 ? 8.f : 0.f;
        TileWalk s;
        s.start(P);
        bool ok = true;
        for (uint32_t ti = 0; s.live && ok; ++ti) {
            const int ob = ti & 1;
            const SegCoord sc = s.sc;
            const ReqInfo r = P.req[sc.b];
            const int gr = sc.t * kTileRows + j;
            const int pos = gr / g, head = sc.h * g + gr % g;
            const bool valid = j < sc.rows;
            if (!(ok = mbar_wait(&sm.o_full[ob], (ti >> 1) & 1, ab))) break;
            if (!(ok = mbar_wait(&sm.st_full[ob], (ti >> 1) & 1, ab))) break;
            tc_fence_after();
            const float mx = sm.stat_m[ob][j], l = sm.stat_l[ob][j];
            uint32_t ov[4][32];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) tmem_ld32(tmem + tlane + kColO + ob * 128 + q4 * 32, ov[q4]);
            tmem_ld_wait();
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) reg_fence32(ov[q4]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.o_empty[ob]);
            if (valid) {
                const float inv = l > 0.f ? P.c_v / l : 0.f;
                __nv_bfloat16 *orow = P.out + ((int64_t)(r.q_start + pos) * P.hq + head) * kHeadDim;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        uint4 pk;
                        uint32_t *pw = reinterpret_cast<uint32_t *>(&pk);
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const __nv_bfloat162 b2 = __floats2bfloat162_rn(
                                __uint_as_float(ov[q4][e + 2 * u]) * inv, __uint_as_float(ov[q4][e + 2 * u + 1]) * inv);
                            pw[u] = *reinterpret_cast<const uint32_t *>(&b2);
                        }
                        *reinterpret_cast<uint4 *>(orow + q4 * 32 + e) = pk;
                    }
                }
                if (P.lse)
                    P.lse[(int64_t)(r.q_start + pos) * P.hq + head] = (mx + log2f(l) - pshift) * 0.6931471805599453f;
            }
            s.next_tile(P);
        }
        // empty (but well-formed) segments of this CTA get zero rows
        for (int w = blockIdx.x; w < P.nseg; w += gridDim.x) {
            const int seg = P.work[w];
            const SegMeta m = P.meta[seg];
            if (m.n_exact != 0 || m.n_chunks != 0) continue;
            const SegCoord sc = decode_seg(P.req, P.batch, g, seg);
            const ReqInfo r = P.req[sc.b];
            const int gr = sc.t * kTileRows + j;
            if (j < sc.rows) {
                const int64_t rowi = (int64_t)(r.q_start + gr / g) * P.hq + sc.h * g + gr % g;
                for (int e = 0; e < kHeadDim; e += 8)
                    *reinterpret_cast<uint4 *>(P.out + rowi * kHeadDim + e) = make_uint4(0, 0, 0, 0);
                if (P.lse) P.lse[rowi] = -INFINITY;
            }
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
                             const void *vbar_op, int flags, void *out, float *lse) {
    const int32_t nseg = (int32_t)c.s.nseg;
    cudaError_t e = cudaMemsetAsync(c.hist(), 0, sizeof(int32_t) * kCostBuckets, c.stream);
    if (e != cudaSuccess) return e;
    attn_meta_kernel<<<(nseg + 7) / 8, 256, 0, c.stream>>>(c.req(), c.p.batch, c.s.g, nseg, csr_cu, csr_idx,
                                                            capacity, flags, c.meta(), c.mask(), c.hist(),
                                                            c.status());
    attn_bucket_kernel<<<1, 1024, 0, c.stream>>>(c.hist(), c.status());
    attn_scatter_kernel<<<(nseg + 255) / 256, 256, 0, c.stream>>>(c.meta(), nseg, c.hist(), c.work(), c.status());
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
    const int grid = nseg < num_sms() ? nseg : num_sms();
    AttnParams prm;
    prm.pt = c.p.page_table;
    prm.pt_stride = c.p.page_table_stride;
    prm.num_pages = c.p.num_pages;
    prm.page_size = c.p.page_size;
    prm.csr_cu = csr_cu;
    prm.csr_idx = csr_idx;
    prm.meta = c.meta();
    prm.todo = c.mask();
    prm.work = c.work();
    prm.out = (__nv_bfloat16 *)out;
    prm.lse = lse;
    prm.req = c.req();
    prm.batch = c.p.batch;
    prm.hq = hq;
    prm.g = g;
    prm.flags = flags;
    prm.c_q = fp8 ? c.p.c_q : 1.f;
    prm.c_k = fp8 ? c.p.c_k : 1.f;
    prm.c_v = fp8 ? c.p.c_v : 1.f;
    prm.nseg = nseg;
    prm.status = c.status();
    if (fp8) {
        const size_t smem = smem_request(sizeof(AttnSmem<FP_DTYPE_E4M3>));
        prm.smem_bytes = (uint32_t)smem;
        e = cudaFuncSetAttribute(attn_tc_kernel<FP_DTYPE_E4M3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        attn_tc_kernel<FP_DTYPE_E4M3><<<grid, kAThreads, smem, c.stream>>>(tm_q, tm_k, tm_v, tm_kb, tm_vb, prm);
    } else {
        const size_t smem = smem_request(sizeof(AttnSmem<FP_DTYPE_BF16>));
        prm.smem_bytes = (uint32_t)smem;
        e = cudaFuncSetAttribute(attn_tc_kernel<FP_DTYPE_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        attn_tc_kernel<FP_DTYPE_BF16><<<grid, kAThreads, smem, c.stream>>>(tm_q, tm_k, tm_v, tm_kb, tm_vb, prm);
    }
    return cudaGetLastError();
}

}  // namespace fp
