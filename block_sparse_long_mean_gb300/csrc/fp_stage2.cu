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
// then one per correction chunk of 128 pooled means (Eq.6):
//   warp 0      TMA producer: Q tile once; per iteration the block's K and V
//               pages through the page table (Eq.22) or the chunk's means
//   warp 1      MMA issuer (one thread): S = Q K^T into TMEM, then O += P V
//               with P read from TMEM
//   warps 2-5   softmax / epilogue, one thread per row: online softmax in the
//               base-2 domain (causal mask on the diagonal block; the log2|B_J|
//               = 7 shift and the todo mask on mean chunks), P written to TMEM,
//               lazy rescaling of O, final O / l and the LSE
// TMEM columns: S0 [0,128) S1 [128,256) O [256,384) P0 [384,448) P1 [448,512).
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
//   warp 0  K producer      warp 1  MMA issuer + TMEM owner
//   warp 2  V producer      warp 3  Q producer (lane 0: slot 0, lane 1: slot 1)
//   warps 4-7   softmax + epilogue of tile slot 0
//   warps 8-11  softmax + epilogue of tile slot 1
// Two query tiles ("slots") are in flight per CTA: while one slot's softmax
// runs, the tensor core works on the other slot's QK^T and PV (ping-pong).
constexpr int kAWarps = 12;
constexpr int kAThreads = 32 * kAWarps;
constexpr int kKStages = 3, kVStages = 2;
// TMEM columns: S_X (P_X aliased on its first columns) at 128 X, O_X at 256 + 128 X
constexpr uint32_t kColS = 0, kColO = 256;
constexpr int kRegsProducer = 56, kRegsSoftmax = 224;  // 128 x 56 + 256 x 224 = 384 x 168

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
    uint64_t q_full[2], q_empty[2], k_full[kKStages], k_empty[kKStages], v_full[kVStages], v_empty[kVStages],
        s_full[2], p_full[2], o_full[2], o_empty[2];
    uint32_t tmem_base;
    int abort;
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

__device__ __forceinline__ void tma_prefetch_l2_4d(const CUtensorMap *map, int c0, int c1, int c2, int c3) {
    asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2), "r"(c3)
                 : "memory");
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

// One slot's walk over its tiles (work items blockIdx.x + (2k + slot) * gridDim.x,
// skipping empty or malformed segments) and over each tile's iterations: the
// selected blocks in descending order (Eq.17), then the correction chunks.
struct SlotWalk {
    int w, seg, n, it, n_exact;
    SegCoord sc;
    int32_t end;
    uint64_t chunks;
    bool live;
    __device__ __forceinline__ void start(const AttnParams &a, int slot) {
        w = blockIdx.x + slot * gridDim.x - 2 * gridDim.x;
        n = it = 0;
        live = true;
        next_tile(a);
    }
    // moves to the next tile holding at least one iteration; live = false when none is left
    __device__ __forceinline__ void next_tile(const AttnParams &a) {
        for (;;) {
            w += 2 * gridDim.x;
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
    if (status_bad(P.status)) return;
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
            mbar_init(&sm.o_full[i], 1);
            mbar_init(&sm.o_empty[i], 4);
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
        fence_barrier_init();
    }
    if (warp == 1) tmem_alloc(&sm.tmem_base, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const Abort ab{&sm.abort};
    const uint32_t tmem = sm.tmem_base;

    if (warp < 4) {
        regs_dec<kRegsProducer>();
        if (warp == 0 || warp == 2) {
            // ------------------------------------------------ K (warp 0) / V (warp 2) producer
            const bool is_k = warp == 0;
            if (lane == 0) {
                tma_prefetch_desc(is_k ? &tm_k : &tm_v);
                tma_prefetch_desc(is_k ? &tm_kb : &tm_vb);
            }
            const int ps_eff = min(P.page_size, 128);
            const int npc = 128 / ps_eff;               // page chunks per 128-token block
            const int oob_row = P.num_pages * P.page_size;  // first row past the pool: TMA fills zeros
            const int nst = is_k ? kKStages : kVStages;
            uint64_t *fullb = is_k ? sm.k_full : sm.v_full;
            uint64_t *emptyb = is_k ? sm.k_empty : sm.v_empty;
            SlotWalk sw[2];
            sw[0].start(P, 0);
            sw[1].start(P, 1);
            int turn = 0;
            for (uint32_t i = 0;; ++i) {
                // the tensor core consumes K (QK^T) and V (PV) tiles alternating between the slots
                int x = turn;
                if (!sw[x].live) x ^= 1;
                if (!sw[x].live) break;
                turn = x ^ 1;
                SlotWalk &s = sw[x];
                const ReqInfo r = P.req[s.sc.b];
                const int J = s.take(P);
                const int h = s.sc.h;
                // lane l < kBoxes * npc (<= 32 as page_size >= 8) copies page chunk l % npc of d box l / npc;
                // its page row is looked up before waiting for the slot
                int row = oob_row;
                if (J >= 0 && lane < C::kBoxes * npc) {
                    const int tok = J * kBlock + (lane % npc) * ps_eff;
                    if (tok < r.len) {
                        const int page = P.pt[(int64_t)s.sc.b * P.pt_stride + tok / P.page_size];
                        if (page >= 0 && page < P.num_pages)
                            row = page * P.page_size + tok % P.page_size;
                        else
                            set_status(status, FP_ERR_DEVICE_PAGE, page);
                    }
                }
                if (s.it == s.n) s.next_tile(P);
                const int st = i % nst;
                if (!mbar_wait(&emptyb[st], ((i / nst) & 1) ^ 1, ab)) break;
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
        } else if (warp == 3) {
            // ------------------------------------------------------ Q producer, one lane per slot
            if (lane < 2) {
                const int x = lane;
                if (x == 0) tma_prefetch_desc(&tm_q);
                SlotWalk s;
                s.start(P, x);
                for (uint32_t t = 0; s.live; ++t) {
                    const ReqInfo r = P.req[s.sc.b];
                    const int pos0 = r.q_start + (s.sc.t * kTileRows) / g;
                    const int h = s.sc.h;
                    if (!mbar_wait(&sm.q_empty[x], (t & 1) ^ 1, ab)) break;
                    mbar_arrive_expect_tx(&sm.q_full[x], C::kTile);
                    for (int i = 0; i < C::kBoxes; ++i)
                        tma_load_4d(sm.q[x] + i * 16384, &tm_q, &sm.q_full[x], i * C::kBoxElems, 0, h, pos0);
                    s.next_tile(P);
                    if (s.live) {
                        // warm L2 with the slot's next tile while this one runs
                        const ReqInfo rn = P.req[s.sc.b];
                        const int p1 = rn.q_start + (s.sc.t * kTileRows) / g;
                        for (int i = 0; i < C::kBoxes; ++i) tma_prefetch_l2_4d(&tm_q, i * C::kBoxElems, 0, s.sc.h, p1);
                    }
                }
            }
        } else if (lane == 0) {
            // ------------------------------------------------------------------ MMA issue
            SlotWalk sw[2];
            sw[0].start(P, 0);
            sw[1].start(P, 1);
            uint32_t ki = 0, vi = 0;
            uint32_t qt[2] = {0, 0};    // tiles whose Q was consumed, per slot
            uint32_t pt_[2] = {0, 0};   // PVs issued per slot
            uint32_t ot[2] = {0, 0};    // tiles whose O was started, per slot
            bool pv_pending[2] = {false, false}, pv_first[2] = {false, false}, pv_last[2] = {false, false};
            bool ok = true;
            // QK^T of slot x's next iteration into S_x
            auto issue_qk = [&](int x) -> bool {
                SlotWalk &s = sw[x];
                const bool first = s.it == 0;
                if (first && !mbar_wait(&sm.q_full[x], qt[x] & 1, ab)) return false;
                s.take(P);
                const bool last = s.it == s.n;
                const int ks = ki % kKStages;
                if (!mbar_wait(&sm.k_full[ks], (ki / kKStages) & 1, ab)) return false;
                tc_fence_after();
                const uint32_t qbase = smem_addr(sm.q[x]), kbase = smem_addr(sm.k[ks]);
#pragma unroll
                for (int k = 0; k < C::kNumK; ++k) {
                    const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
                    const uint64_t ad = sw128_desc(qbase + off, 16, 1024);
                    const uint64_t bd = sw128_desc(kbase + off, 16, 1024);
                    if (kDtype == FP_DTYPE_BF16)
                        umma_f16_ss(tmem + kColS + x * 128, ad, bd, C::kIdescQK, k > 0);
                    else
                        umma_f8_ss(tmem + kColS + x * 128, ad, bd, C::kIdescQK, k > 0);
                }
                umma_commit(&sm.k_empty[ks]);
                umma_commit(&sm.s_full[x]);
                ++ki;
                pv_pending[x] = true;
                pv_first[x] = first;
                pv_last[x] = last;
                if (last) {
                    umma_commit(&sm.q_empty[x]);
                    ++qt[x];
                    s.next_tile(P);
                }
                return true;
            };
            // O_x (+)= P_x V of slot x's pending iteration
            auto issue_pv = [&](int x) -> bool {
                if (pv_first[x] && !mbar_wait(&sm.o_empty[x], (ot[x] & 1) ^ 1, ab)) return false;
                const int vs = vi % kVStages;
                if (!mbar_wait(&sm.v_full[vs], (vi / kVStages) & 1, ab)) return false;
                if (!mbar_wait(&sm.p_full[x], pt_[x] & 1, ab)) return false;
                tc_fence_after();
                const uint32_t vbase = smem_addr(sm.v[vs]);
#pragma unroll
                for (int k = 0; k < C::kNumK; ++k) {
                    // B = V, MN-major: 8-key row groups 1024 B apart, 64-element d atoms 16 KB apart
                    const uint64_t bd = sw128_desc(vbase + k * C::kKStep * 128, 16384, 1024);
                    const uint32_t a = tmem + kColS + x * 128 + k * (C::kKStep * C::kEb / 4);
                    const uint32_t acc = (!pv_first[x] || k > 0) ? 1u : 0u;
                    if (kDtype == FP_DTYPE_BF16)
                        umma_f16_ts(tmem + kColO + x * 128, a, bd, C::kIdescPV, acc);
                    else
                        umma_f8_ts(tmem + kColO + x * 128, a, bd, C::kIdescPV, acc);
                }
                umma_commit(&sm.v_empty[vs]);
                ++vi;
                ++pt_[x];
                if (pv_first[x]) ++ot[x];
                if (pv_last[x]) umma_commit(&sm.o_full[x]);
                pv_pending[x] = false;
                return true;
            };
            for (int x = 0; x < 2 && ok; ++x)
                if (sw[x].live) ok = issue_qk(x);
            for (int x = 0; ok; x ^= 1) {
                if (!pv_pending[0] && !pv_pending[1]) break;
                if (pv_pending[x]) {
                    if (!(ok = issue_pv(x))) break;
                    if (sw[x].live && !(ok = issue_qk(x))) break;
                }
            }
        }
    } else {
        regs_inc<kRegsSoftmax>();
        // ---------------------------------------------------- softmax / epilogue of one slot
        const int x = (warp - 4) >> 2;          // slot
        const int j = 32 * (warp & 3) + lane;   // TMEM lane = packed row of the tile
        const uint32_t tlane = static_cast<uint32_t>(32 * (warp & 3)) << 16;
        const uint32_t tS = tmem + tlane + kColS + x * 128, tO = tmem + tlane + kColO + x * 128;
        const float LOG2E = 1.4426950408889634f;
        const float sl2 = (kDtype == FP_DTYPE_E4M3 ? P.c_q * P.c_k : 1.f) * LOG2E * rsqrtf((float)kHeadDim);
        // lazy rescale slack (log2 units): bf16 P may reach 2^8; FP8 P~ must stay within [0, 256]
        const float tau = kDtype == FP_DTYPE_E4M3 ? 0.f : 8.f;
        const float pshift = kDtype == FP_DTYPE_E4M3 ? 8.f : 0.f;  // FP8 probabilities in [0, 256] (Eq.15)
        uint32_t si = 0, ti = 0;
        bool ok = true;
        SlotWalk s;
        s.start(P, x);
        // empty (but well-formed) segments of this slot get zero rows
        for (int w = blockIdx.x + x * gridDim.x; w < P.nseg; w += 2 * gridDim.x) {
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
        while (s.live && ok) {
            const SegCoord sc = s.sc;
            const ReqInfo r = P.req[sc.b];
            const int gr = sc.t * kTileRows + j;
            const int pos = gr / g, head = sc.h * g + gr % g;
            const bool valid = j < sc.rows;
            const uint32_t *tw = P.todo + (int64_t)r.mask_base + (int64_t)(sc.h * r.ntiles + sc.t) * r.words;
            const int nw = (sc.D + 31) / 32;
            const int n = s.n;
            float mx = -INFINITY, l = 0.f;
            for (int it = 0; it < n; ++it, ++si) {
                const int J = s.take(P);
                uint4 mv = make_uint4(0, 0, 0, 0);  // correction-chunk key mask
                if (J < 0) {
                    const int c = -1 - J;
                    uint32_t wv[4];
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) wv[q4] = (4 * c + q4 < nw) ? __ldg(tw + 4 * c + q4) : 0u;
                    mv = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                }
                if (!(ok = mbar_wait(&sm.s_full[x], si & 1, ab))) break;
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
                    for (int e = 0; e < 128; ++e) pm[e & 7] = fmaxf(pm[e & 7], __uint_as_float(sv[e >> 5][e & 31]));
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
                const float rmax = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])),
                                         fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7])));
                const float tmax = fmaf(rmax, sl2, shift);
                // online softmax with lazy rescaling of O (PV of the previous iteration is complete:
                // it was issued before this iteration's QK^T, whose completion s_full signalled)
                const bool first = it == 0;
                const bool grow = first || tmax > mx + tau;
                const float m_new = grow ? fmaxf(mx, tmax) : mx;
                const bool need_o = !first && grow;
                if (__any_sync(0xffffffffu, need_o)) {
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
                // pass 2: p = 2^(x - m) (FP8: 2^(x - m + 8)), row sum, P written over S_x
                // (packed in place over the consumed scores, 32 keys at a time)
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
                if (lane == 0) mbar_arrive(&sm.p_full[x]);
            }
            if (!ok) break;
            s.next_tile(P);
            // epilogue: wait for the tile's last PV, O / l to bf16, release O_x
            if (!(ok = mbar_wait(&sm.o_full[x], ti & 1, ab))) break;
            tc_fence_after();
            const float inv = l > 0.f ? (kDtype == FP_DTYPE_E4M3 ? P.c_v : 1.f) / l : 0.f;
            uint32_t ov[4][32];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) tmem_ld32(tO + q4 * 32, ov[q4]);
            tmem_ld_wait();
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) reg_fence32(ov[q4]);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.o_empty[x]);
            if (valid) {
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
                if (P.lse) P.lse[(int64_t)(r.q_start + pos) * P.hq + head] = (mx + log2f(l) - pshift) * 0.6931471805599453f;
            }
            ++ti;
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
    // two tile slots per CTA: enough CTAs to give every slot work, at most one per SM
    const int grid = (nseg + 1) / 2 < num_sms() ? (nseg + 1) / 2 : num_sms();
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
