// Stage 1 scoring + selection on the tensor cores (FlashPrefill V2 Sec.3.3
// "Single-Pass Score and Selection", Eq.19-20; Sec.3.1 Eq.1-3).
//
// One persistent CTA per SM walks the packed query tiles. For a tile of
// (request b, KV head h, tile t) with diagonal block D it computes, chunk by
// chunk of 128 pooled keys, S[J][r] = kbar_J . q_r on tcgen05 (pooled keys on
// the 128 TMEM lanes, the tile's 128 packed rows on 128 columns), so each
// reduction thread owns one block J and reduces its row of S without any
// cross-thread traffic:
//     lE_J = ln sum_r exp(s_rJ),   s_rJ = kbar_J . q_r / sqrt(d)
// (Eq.19's E_J up to the common factor exp(-M), which cancels in Eq.20).
// Block J is kept iff lE_J >= ln(alpha) + max_J' lE_J' or J is forced.
//
// Exactness. The tensor core sees kbar rounded to the operand format (bf16 or
// e4m3). Per (block, head) the pooling kernel records |kbar - kbar_op|_2 and
// |kbar|_2, so |s_rJ(screen) - s_rJ(exact)| <= eps_J = max_r |q_r| (|kbar -
// kbar_op| + 2^-12 |kbar|) / sqrt(d) + 2e-4 (Cauchy-Schwarz; the second term
// covers fp32 accumulation and the exp/log approximations), hence
// |lE_J(screen) - lE_J| <= eps_J. max_r |q_r| is bounded by sqrt(d) max |q_ri|
// for bf16 and by the rows' own norms for e4m3, whose coarser means make the
// bound weigh more. Every block whose decision (or whose claim
// to the maximum) is not settled by these bounds is recomputed in fp32 from
// the fp32 means, so the CSR matches an exact evaluation except for blocks
// within fp32 rounding of the threshold.
//
// Exponentials are computed only for blocks that can matter. A block's
// maximum logit ms_J over the tile's rows (for a full tile, returned by the
// TMEM load itself: tcgen05.ld.red.max) bounds its log-energy from both
// sides, ms_J <= lE_J <= ms_J + ln(rows); the first chunk processed holds the
// diagonal block, and one block-wide maximum there gives a proven lower bound
// of max_J lE_J. A later block whose upper bound lies below ln(alpha) plus that
// bound is certainly pruned and certainly not the maximum, so it needs no
// exponentials.
#include <math.h>

#include "fp_internal.cuh"
#include "sm100_ptx.cuh"

namespace fp {
namespace {

using namespace sm100;

// Two independent pipelines ("sets") take the CTA's tiles alternately, so that one tile's selection overlaps
// the other set's scores and neither set's pace holds up the other. Set s: warp 2 s loads its Q tiles
// (lane 1) and pooled-key chunks (lane 0) by TMA, warp 2 s + 1 issues its MMAs into its own TMEM columns,
// and warps 4 + 4 s .. 7 + 4 s reduce and select. Warp 1 also owns the TMEM allocation.
constexpr int kSWarps = 12;
constexpr int kSThreads = 32 * kSWarps;
// registers per thread: 64K over the CTA at launch, then 48 for the TMA/MMA warpgroup and 224 for each set
constexpr int kSRegsLaunch = (65536 / kSThreads) & ~7;
constexpr int kSRegsProducer = 48, kSRegsReduce = 224;
static_assert(kSRegsProducer + 2 * kSRegsReduce <= 3 * kSRegsLaunch, "register split exceeds the launch");
constexpr int kRedThreads = 128;
constexpr int kRefineList = 256;
constexpr int kCand = 128;  // candidates per tile settled without the exact path

enum ScoreMode { kModeScore = 0, kModeAll = 1, kModeForced = 2 };

template <int kDtype>
struct SCfg {
    static constexpr int kEb = Elem<kDtype>::kBytes;
    static constexpr int kTile = 128 * 128 * kEb;  // bytes of a Q tile or of a chunk of 128 pooled keys
    static constexpr int kKStep = 32 / kEb;         // K elements per MMA (32 bytes)
    static constexpr int kNumK = 128 / kKStep;      // MMAs per chunk
    static constexpr int kBoxElems = 128 / kEb;     // elements per 128-byte TMA box row
    static constexpr int kBoxes = 128 / kBoxElems;  // boxes along d
    static constexpr uint32_t kIdesc =
        instr_desc(kDtype == FP_DTYPE_BF16 ? 1u : 0u, kDtype == FP_DTYPE_BF16 ? 1u : 0u, false, false, 128, 128);
};

// Fixed-size scratch of one reduction set.
struct RedFixed {
    float4 dbuf[32];  // the diagonal block's 128 logits: rows r, r + 32, r + 64, r + 96 at [r]
    int32_t list[kRefineList];
    int32_t cand[kCand];  // blocks with a screened log-energy
    float red[2][4];
    float red3[3][4];
    int nlist, ncand, nsel;
    int any2[2];  // per tile of the set, alternately: some candidate was left open (read after the tile's last barrier)
};

// Barriers of the two sets (index [set][Q buffer / stage / S buffer]).
struct ScoreBars {
    uint64_t q_full[2][2], q_empty[2][2], k_full[2][2], k_empty[2][2], s_full[2][2], s_empty[2][2];
    uint32_t tmem_base;
    int abort;
};

// Shared-memory layout (byte offsets from a 1024-byte aligned base): nq Q buffers per set, nst chunk stages per
// set, the barriers, then each set's scratch with per-block arrays for nb blocks (a multiple of 128). With two
// Q buffers a set loads its next tile's Q while the current tile's MMAs still read the other.
struct SLayout {
    uint32_t q, k, bars, fixed[2], lE[2], words[2], state[2], total;
};
__host__ __device__ inline SLayout score_layout(int tile, int nq, int nst, int nb) {
    SLayout L;
    uint32_t o = 0;
    L.q = o;
    o += 2 * nq * tile;
    L.k = o;
    o += 2 * nst * tile;
    L.bars = o;
    o += (sizeof(ScoreBars) + 15) & ~15u;
    for (int s = 0; s < 2; ++s) {
        L.fixed[s] = o;
        o += (sizeof(RedFixed) + 15) & ~15u;
        L.lE[s] = o;
        o += 4 * nb;
        L.words[s] = o;
        o += nb / 8;
        L.state[s] = o;
        o += (nb + 15) & ~15;
    }
    L.total = o;
    return L;
}

// state bits
constexpr uint8_t kStBound = 1;      // lE holds only an upper bound (block certainly pruned)
constexpr uint8_t kStUncertain = 2;  // decision not settled by the bounds
constexpr uint8_t kStMaxCand = 4;    // may hold the maximum
constexpr uint8_t kStRefined = 8;    // lE is the fp32 recomputation
constexpr uint8_t kStSelected = 0x80;

// Named barrier of one reduction set (ids 1 and 2; 128 threads each).
__device__ __forceinline__ void red_bar(int set) { asm volatile("bar.sync %0, 128;" ::"r"(1 + set) : "memory"); }

template <int kRegs>
__device__ __forceinline__ void sregs_set() {
    static_assert(kRegs % 8 == 0 && kRegs >= 24 && kRegs <= 256, "setmaxnreg range");
    if constexpr (kRegs > kSRegsLaunch)
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegs));
    else if constexpr (kRegs < kSRegsLaunch)
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegs));
}

// tcgen05.ld of 128 columns (.32x32b.x128) that also returns the largest of the 128 values this thread loads
// (.red.max, sm_103a); r[q][i] is column 32 q + i. Like the loaded registers, the maximum is valid once
// tcgen05.wait::ld has returned.
__device__ __forceinline__ void tmem_ld128_max(uint32_t taddr, uint32_t (&r)[4][32], float &mx) {
    asm volatile(
        "tcgen05.ld.red.sync.aligned.32x32b.x128.max.f32 "
        "{"
        "%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, "
        "%32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
        "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63, "
        "%64, %65, %66, %67, %68, %69, %70, %71, %72, %73, %74, %75, %76, %77, %78, %79, "
        "%80, %81, %82, %83, %84, %85, %86, %87, %88, %89, %90, %91, %92, %93, %94, %95, "
        "%96, %97, %98, %99, %100, %101, %102, %103, %104, %105, %106, %107, %108, %109, %110, %111, "
        "%112, %113, %114, %115, %116, %117, %118, %119, %120, %121, %122, %123, %124, %125, %126, %127"
        "}, %128, [%129];"
        : "=r"(r[0][0]), "=r"(r[0][1]), "=r"(r[0][2]), "=r"(r[0][3]), "=r"(r[0][4]), "=r"(r[0][5]), "=r"(r[0][6]), "=r"(r[0][7]),
          "=r"(r[0][8]), "=r"(r[0][9]), "=r"(r[0][10]), "=r"(r[0][11]), "=r"(r[0][12]), "=r"(r[0][13]), "=r"(r[0][14]), "=r"(r[0][15]),
          "=r"(r[0][16]), "=r"(r[0][17]), "=r"(r[0][18]), "=r"(r[0][19]), "=r"(r[0][20]), "=r"(r[0][21]), "=r"(r[0][22]), "=r"(r[0][23]),
          "=r"(r[0][24]), "=r"(r[0][25]), "=r"(r[0][26]), "=r"(r[0][27]), "=r"(r[0][28]), "=r"(r[0][29]), "=r"(r[0][30]), "=r"(r[0][31]),
          "=r"(r[1][0]), "=r"(r[1][1]), "=r"(r[1][2]), "=r"(r[1][3]), "=r"(r[1][4]), "=r"(r[1][5]), "=r"(r[1][6]), "=r"(r[1][7]),
          "=r"(r[1][8]), "=r"(r[1][9]), "=r"(r[1][10]), "=r"(r[1][11]), "=r"(r[1][12]), "=r"(r[1][13]), "=r"(r[1][14]), "=r"(r[1][15]),
          "=r"(r[1][16]), "=r"(r[1][17]), "=r"(r[1][18]), "=r"(r[1][19]), "=r"(r[1][20]), "=r"(r[1][21]), "=r"(r[1][22]), "=r"(r[1][23]),
          "=r"(r[1][24]), "=r"(r[1][25]), "=r"(r[1][26]), "=r"(r[1][27]), "=r"(r[1][28]), "=r"(r[1][29]), "=r"(r[1][30]), "=r"(r[1][31]),
          "=r"(r[2][0]), "=r"(r[2][1]), "=r"(r[2][2]), "=r"(r[2][3]), "=r"(r[2][4]), "=r"(r[2][5]), "=r"(r[2][6]), "=r"(r[2][7]),
          "=r"(r[2][8]), "=r"(r[2][9]), "=r"(r[2][10]), "=r"(r[2][11]), "=r"(r[2][12]), "=r"(r[2][13]), "=r"(r[2][14]), "=r"(r[2][15]),
          "=r"(r[2][16]), "=r"(r[2][17]), "=r"(r[2][18]), "=r"(r[2][19]), "=r"(r[2][20]), "=r"(r[2][21]), "=r"(r[2][22]), "=r"(r[2][23]),
          "=r"(r[2][24]), "=r"(r[2][25]), "=r"(r[2][26]), "=r"(r[2][27]), "=r"(r[2][28]), "=r"(r[2][29]), "=r"(r[2][30]), "=r"(r[2][31]),
          "=r"(r[3][0]), "=r"(r[3][1]), "=r"(r[3][2]), "=r"(r[3][3]), "=r"(r[3][4]), "=r"(r[3][5]), "=r"(r[3][6]), "=r"(r[3][7]),
          "=r"(r[3][8]), "=r"(r[3][9]), "=r"(r[3][10]), "=r"(r[3][11]), "=r"(r[3][12]), "=r"(r[3][13]), "=r"(r[3][14]), "=r"(r[3][15]),
          "=r"(r[3][16]), "=r"(r[3][17]), "=r"(r[3][18]), "=r"(r[3][19]), "=r"(r[3][20]), "=r"(r[3][21]), "=r"(r[3][22]), "=r"(r[3][23]),
          "=r"(r[3][24]), "=r"(r[3][25]), "=r"(r[3][26]), "=r"(r[3][27]), "=r"(r[3][28]), "=r"(r[3][29]), "=r"(r[3][30]), "=r"(r[3][31]),
          "=f"(mx)
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float warp_max(float v) {
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Max over the 128 threads of reduction set `set`; slot selects the smem buffer.
__device__ __forceinline__ float red_max(RedFixed &rs, int set, float v, int slot) {
    v = warp_max(v);
    const int w = (threadIdx.x >> 5) & 3;
    if ((threadIdx.x & 31) == 0) rs.red[slot][w] = v;
    red_bar(set);
    const float r = fmaxf(fmaxf(rs.red[slot][0], rs.red[slot][1]), fmaxf(rs.red[slot][2], rs.red[slot][3]));
    return r;
}
__device__ __forceinline__ float red_sum(RedFixed &rs, int set, float v, int slot) {
    v = warp_sum(v);
    const int w = (threadIdx.x >> 5) & 3;
    if ((threadIdx.x & 31) == 0) rs.red[slot][w] = v;
    red_bar(set);
    return (rs.red[slot][0] + rs.red[slot][1]) + (rs.red[slot][2] + rs.red[slot][3]);
}

template <int kDtype>
__global__ void __launch_bounds__(kSThreads, 1)
    score_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const float *__restrict__ kbar, const float2 *__restrict__ kstat,
                    const ReqInfo *__restrict__ req, int batch, int hkv, int g, int mode, float log_alpha, int sink,
                    int window, float qscale, float kscale, int32_t nseg, int32_t *__restrict__ seg_count,
                    uint32_t *__restrict__ mask, const uint8_t *__restrict__ qg, int hq, int nq, int nst, int nb,
                    int32_t *__restrict__ status) {
    using C = SCfg<kDtype>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *const base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const SLayout L = score_layout(C::kTile, nq, nst, nb);
    ScoreBars &sm = *reinterpret_cast<ScoreBars *>(base + L.bars);
    uint8_t *const qbase = base + L.q, *const kbase = base + L.k;
    auto qbuf = [=](int set, int qi) { return qbase + (set * nq + qi) * C::kTile; };
    auto kbuf = [=](int set, int st) { return kbase + (set * nst + st) * C::kTile; };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (status_bad(status)) return;

    if (threadIdx.x == 0) {
        for (int i = 0; i < 2; ++i) {
            for (int qi = 0; qi < 2; ++qi) {
                mbar_init(&sm.q_full[i][qi], 1);
                mbar_init(&sm.q_empty[i][qi], 2);  // MMA commit + reduction set done with Q
            }
            for (int b = 0; b < 2; ++b) {
                mbar_init(&sm.s_full[i][b], 1);
                mbar_init(&sm.s_empty[i][b], 4);  // one arrival per warp of the set
                mbar_init(&sm.k_full[i][b], 1);
                mbar_init(&sm.k_empty[i][b], 1);
            }
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
    const bool scoring = mode == kModeScore;

    if (warp < 4 && (warp & 1) == 0) {
        sregs_set<kSRegsProducer>();
        // ------------------------------------------------------------ TMA producers of set warp / 2
        // lane 0: the set's pooled-key chunks; lane 1: its Q tiles, each as soon as the tile nq before it is done
        // with that Q buffer (its MMAs complete and its reduction past the Q maximum)
        const int set = warp >> 1;
        if (lane < 2 && scoring) {
            if (lane == 0) {
                tma_prefetch_desc(&tm_q);
                tma_prefetch_desc(&tm_k);
            }
            uint32_t tile_it = 0, chunk_it = 0;  // this set's tiles and chunks
            for (int w = blockIdx.x + set * gridDim.x; w < nseg; w += 2 * gridDim.x, ++tile_it) {
                const SegCoord sc = decode_seg(req, batch, g, nseg - 1 - w);
                if (lane == 1) {
                    const int qi = tile_it & (nq - 1);
                    if (!mbar_wait(&sm.q_empty[set][qi], ((tile_it >> (nq - 1)) & 1) ^ 1, ab)) break;
                    mbar_arrive_expect_tx(&sm.q_full[set][qi], C::kTile);
                    // rows before sc.lo (a chunk's first tile) read other tokens or the zero fill; they are masked
                    for (int i = 0; i < C::kBoxes; ++i)
                        tma_load_4d(qbuf(set, qi) + i * 16384, &tm_q, &sm.q_full[set][qi], i * C::kBoxElems, 0, sc.h,
                                    sc.q_pos);
                    continue;
                }
                const int blk_base = req[sc.b].blk_base;
                const int nch = sc.D / 128 + 1;
                bool ok = true;
                for (int cc = 0; cc < nch && ok; ++cc, ++chunk_it) {
                    const int c = nch - 1 - cc;
                    const int st = chunk_it % nst;
                    if (!(ok = mbar_wait(&sm.k_empty[set][st], ((chunk_it / nst) & 1) ^ 1, ab))) break;
                    mbar_arrive_expect_tx(&sm.k_full[set][st], C::kTile);
                    for (int i = 0; i < C::kBoxes; ++i)
                        tma_load_3d(kbuf(set, st) + i * 16384, &tm_k, &sm.k_full[set][st], i * C::kBoxElems, sc.h,
                                    blk_base + 128 * c);
                }
                if (!ok) break;
            }
        }
    } else if (warp < 4) {
        sregs_set<kSRegsProducer>();
        // --------------------------------------------------------------- MMA issue of set warp / 2
        // The whole warp runs the loop (descriptors stay warp-uniform) and one elected lane issues:
        // issued from a lone lane, every MMA costs tens of cycles more. Waits end alike in all lanes.
        const int set = warp >> 1;
        if (scoring) {
            auto wait_w = [&](uint64_t *bar, uint32_t parity) -> bool {
                return __all_sync(0xffffffffu, mbar_wait(bar, parity, ab));
            };
            uint32_t tile_it = 0, chunk_it = 0;
            for (int w = blockIdx.x + set * gridDim.x; w < nseg; w += 2 * gridDim.x, ++tile_it) {
                const SegCoord sc = decode_seg(req, batch, g, nseg - 1 - w);
                const int qi = tile_it & (nq - 1);
                if (!wait_w(&sm.q_full[set][qi], (tile_it >> (nq - 1)) & 1)) break;
                const int nch = sc.D / 128 + 1;
                bool ok = true;
                for (int cc = 0; cc < nch; ++cc, ++chunk_it) {
                    const int st = chunk_it % nst, sb = chunk_it & 1;
                    if (!(ok = wait_w(&sm.k_full[set][st], (chunk_it / nst) & 1))) break;
                    if (!(ok = wait_w(&sm.s_empty[set][sb], ((chunk_it >> 1) & 1) ^ 1))) break;
                    if (elect_one()) {
                        tc_fence_after();
                        const uint32_t abase = smem_addr(kbuf(set, st)), bbase = smem_addr(qbuf(set, qi));
#pragma unroll
                        for (int k = 0; k < C::kNumK; ++k) {
                            const uint32_t off = (k >> 2) * 16384 + (k & 3) * 32;
                            const uint64_t ad = sw128_desc(abase + off, 16, 1024);
                            const uint64_t bd = sw128_desc(bbase + off, 16, 1024);
                            if (kDtype == FP_DTYPE_BF16)
                                umma_f16_ss(tmem + set * 256 + sb * 128, ad, bd, C::kIdesc, k > 0);
                            else
                                umma_f8_ss(tmem + set * 256 + sb * 128, ad, bd, C::kIdesc, k > 0);
                        }
                        umma_commit(&sm.k_empty[set][st]);
                        umma_commit(&sm.s_full[set][sb]);
                        if (cc == nch - 1) umma_commit(&sm.q_empty[set][qi]);
                    }
                    __syncwarp();
                }
                if (!ok) break;
            }
        }
    } else {
        sregs_set<kSRegsReduce>();
        // --------------------------------------------------- reduction / selection
        // Thread j owns block J = 128 c + j of each chunk c. Its screened maximum logit ms_J bounds the
        // block's log-energy, ms_J - eps_J <= lE_J <= ms_J + ln(rows) + eps_J. Blocks whose upper bound
        // falls below ln(alpha) plus a proven lower bound of the maximum are certainly pruned; the few
        // others ("candidates") get a screened log-energy and are settled at the end of the tile against
        // the threshold interval, and any candidate the interval cannot settle sends the tile through the
        // exact fp32 path. Mask words start from the forced blocks (sink, window, diagonal).
        const int set = (warp - 4) >> 2;               // this set takes the CTA's tiles k with k % 2 == set
        // the set's scratch: the fixed part and per-block arrays for the longest request
        // (selects rather than indexes L, so that L stays in registers)
        RedFixed &rs = *reinterpret_cast<RedFixed *>(base + (set ? L.fixed[1] : L.fixed[0]));
        float *const blE = reinterpret_cast<float *>(base + (set ? L.lE[1] : L.lE[0]));  // log-energy, bound or refined
        uint8_t *const bstate = base + (set ? L.state[1] : L.state[0]);                 // kSt* bits per block
        uint32_t *const words = reinterpret_cast<uint32_t *>(base + (set ? L.words[1] : L.words[0]));  // tile's mask
        const int rt = (threadIdx.x - 128) & 127;     // 0..127 within the set
        const int j = 32 * (warp & 3) + lane;         // TMEM lane = block in chunk = tile row
        const uint32_t tlane = (static_cast<uint32_t>(32 * (warp & 3)) << 16) + set * 256;
        const float inv_sqrt_d = rsqrtf((float)kHeadDim);
        const float scale = qscale * kscale * inv_sqrt_d;  // raw MMA dot -> logit
        const float LOG2E = 1.4426950408889634f, LN2 = 0.6931471805599453f;
        // bits of the blocks [lo, hi) that fall in mask word k
        auto range_bits = [](int k, int lo, int hi) -> uint32_t {
            lo = max(lo - 32 * k, 0);
            hi = min(hi - 32 * k, 32);
            if (hi <= lo) return 0u;
            const uint32_t up = hi >= 32 ? 0xffffffffu : ((1u << hi) - 1u);
            return up & ~((1u << lo) - 1u);
        };
        uint32_t tile_it = set, chunk_it = 0;  // tile_it: the CTA's tile counter; chunk_it: this set's chunks
        bool ok = true;
        const int wstep = 2 * (int)gridDim.x;
        // the next tile's coordinates and request record are fetched a tile ahead
        const int w0 = (int)blockIdx.x + set * (int)gridDim.x;
        int b_next = find_req_by_seg(req, batch, nseg - 1 - min(w0, nseg - 1));
        ReqInfo r_next = req[b_next];
        for (int w = w0; w < nseg && ok; w += wstep, tile_it += 2) {
            const int seg = nseg - 1 - w;
            // this tile's coordinates from the request record loaded a tile ago (no load to wait for here);
            // the next tile's record is loaded now and used a tile later
            const ReqInfo r = r_next;
            const SegCoord sc = coord_in_req(r, b_next, g, seg);
            if (w + wstep < nseg) {
                b_next = find_req_by_seg(req, batch, nseg - 1 - (w + wstep));
                r_next = req[b_next];
            }
            const int ap = (tile_it >> 1) & 1;  // alternates between this set's consecutive tiles
            const int D = sc.D;
            // query rows of the tile: [lo, rows) packed as rows | lo << 8 (128 for a full tile); the packed
            // value, unpacked at each use, keeps the chunk loop within its registers
            const int row_span = sc.rows | (sc.lo << 8);
            const int qi = (tile_it >> 1) & (nq - 1);  // the set's Q buffer of this tile (nq is 1 or 2)
            const int nch = D / 128 + 1;
            const float2 *ks_base = kstat + (int64_t)r.blk_base * hkv + sc.h;
            const float lnrows = logf((float)(sc.rows - sc.lo));
            const int s_end = min(sink, D + 1), w_lo = max(D - window, 0);
            // mask words of this tile start as the forced set; thread k owns word k
            for (int k = rt; k < r.words; k += kRedThreads)
                words[k] = range_bits(k, 0, s_end) | range_bits(k, w_lo, D) | range_bits(k, D, D + 1);
            if (rt == 0) {
                rs.ncand = 0;
                rs.nsel = 0;
                rs.any2[ap] = 0;
            }
            float eps_tile = 0.f;                    // largest per-block logit error bound of the tile
            float mlo = -INFINITY, mhi = -INFINITY;  // this thread's bounds of max_J lE_J
            float m_run = -INFINITY;                 // proven lower bound of max_J lE_J
            if (scoring) {
                if (!(ok = mbar_wait(&sm.q_full[set][qi], ((tile_it >> 1) >> (nq - 1)) & 1, ab))) break;
                // a bound of |q_r|_2 over the tile's rows. BF16: sqrt(d) max_i |q_ri|, the largest element
                // magnitude of this thread's row (an integer maximum over the magnitude bits of the 16-byte chunks
                // of the swizzled tile). E4M3, whose operand-format means round coarsely and so weigh the bound
                // more: the row's own norm, from the squares of its elements (exact products of the exactly
                // widened values, summed in fp32), raised by 2^-12 to cover the rounding of the sum and the root.
                float qbound = 0.f;
                if (j >= (row_span >> 8) && j < (row_span & 255)) {
                    if (kDtype == FP_DTYPE_BF16) {
                        uint32_t mx = 0;
#pragma unroll
                        for (int ch = 0; ch < 16; ++ch) {
                            const int atom = ch >> 3, c16 = ch & 7;
                            const uint4 u = *reinterpret_cast<const uint4 *>(qbuf(set, qi) + atom * 16384 + j * 128 +
                                                                             ((c16 ^ (j & 7)) << 4));
                            mx = __vmaxu2(mx, __vmaxu2(u.x & 0x7fff7fffu, u.y & 0x7fff7fffu));
                            mx = __vmaxu2(mx, __vmaxu2(u.z & 0x7fff7fffu, u.w & 0x7fff7fffu));
                        }
                        qbound = __uint_as_float(max(mx & 0xffffu, mx >> 16) << 16) * sqrtf((float)kHeadDim);
                    } else {
                        uint64_t ss2 = f2pack(0.f, 0.f);
#pragma unroll
                        for (int ch = 0; ch < 8; ++ch) {
                            const uint4 u = *reinterpret_cast<const uint4 *>(qbuf(set, qi) + j * 128 + ((ch ^ (j & 7)) << 4));
                            const uint32_t uw[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                            for (int q = 0; q < 4; ++q)
#pragma unroll
                                for (int hh = 0; hh < 2; ++hh) {
                                    const float2 f = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(
                                        (__nv_fp8x2_storage_t)(uw[q] >> (16 * hh)), __NV_E4M3)));
                                    const uint64_t x2 = f2pack(f.x, f.y);
                                    ss2 = ffma2(x2, x2, ss2);
                                }
                        }
                        float s0, s1;
                        f2unpack(ss2, s0, s1);
                        qbound = sqrtf(s0 + s1) * 1.000244140625f;
                    }
                }
                const float qmax = red_max(rs, set, qbound, 0) * qscale;  // bounds |q_r|_2 (real units), every row
                // the set is done with the Q tile in shared memory (the rare exact path reads Q from global
                // memory): once the tile's MMAs are complete too, the next tile's Q may load into the buffer
                if (rt == 0) mbar_arrive(&sm.q_empty[set][qi]);
                // rounding statistics of this thread's block, loaded one chunk ahead
                float2 ks_next = (128 * (nch - 1) + j <= D) ? __ldg(ks_base + (int64_t)(128 * (nch - 1) + j) * hkv)
                                                            : make_float2(0.f, 0.f);
                for (int cc = 0; cc < nch; ++cc, ++chunk_it) {
                    const int c = nch - 1 - cc;
                    const int sb = chunk_it & 1;
                    const int J = 128 * c + j;
                    const bool valid = J <= D;
                    const float2 ks = ks_next;
                    if (c > 0) ks_next = __ldg(ks_base + (int64_t)(J - 128) * hkv);
                    if (!(ok = mbar_wait(&sm.s_full[set][sb], (chunk_it >> 1) & 1, ab))) break;
                    tc_fence_after();
                    uint32_t v[4][32];
                    float m = -INFINITY;  // full tiles: the block's maximum, taken by the load itself
                    if (row_span == 128) {
                        tmem_ld128_max(tmem + tlane + sb * 128, v, m);
                    } else {
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) tmem_ld32(tmem + tlane + sb * 128 + q4 * 32, v[q4]);
                    }
                    tmem_ld_wait();
                    asm volatile("" : "+f"(m));
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) reg_fence32(v[q4]);
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sm.s_empty[set][sb]);
                    if (row_span != 128) {
                        // a partial tile: only the rows [lo, rows) count
                        float pm[8];
#pragma unroll
                        for (int u = 0; u < 8; ++u) pm[u] = -INFINITY;
#pragma unroll
                        for (int x = 0; x < 128; ++x)
                            pm[x & 7] = fmaxf(pm[x & 7], x >= (row_span >> 8) && x < (row_span & 255)
                                                             ? __uint_as_float(v[x >> 5][x & 31]) : -INFINITY);
                        m = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])),
                                  fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7])));
                    }
                    const float eps = valid ? qmax * (ks.x + 2.44140625e-4f * ks.y) * inv_sqrt_d + 2e-4f : 0.f;
                    const float ms = m * scale;
                    // the first chunk holds the diagonal block (usually the maximum): one block-wide max of the
                    // lower bounds there gives m_run, a proven lower bound of max_J lE_J for the whole tile. The
                    // diagonal block contributes its screened log-energy less eps, which exceeds its maximum
                    // logit by up to ln(rows); computed first, by its whole warp (its lane stages the 128 logits
                    // in shared memory, each lane takes four rows), it leaves few candidates in any chunk.
                    float lE_diag = 0.f;  // the diagonal block's screened log-energy (its own thread)
                    if (cc == 0) {
                        const int dj = D & 127;  // thread of the diagonal block within the set
                        if ((dj >> 5) == (warp & 3)) {
                            const int dl = dj & 31;
                            if (lane == dl) {
#pragma unroll
                                for (int i = 0; i < 32; ++i)
                                    rs.dbuf[i] = make_float4(__uint_as_float(v[0][i]), __uint_as_float(v[1][i]),
                                                             __uint_as_float(v[2][i]), __uint_as_float(v[3][i]));
                            }
                            __syncwarp();
                            // 2^(x k2 - m k2) for rows lane + 32 u; the rounding of m k2 (|logit| 2^-24) lies far
                            // inside the bound's relative term (2^-12 |q||kbar| >= 2^-12 |logit|)
                            const float k2 = scale * LOG2E;
                            const float mk2 = -__shfl_sync(0xffffffffu, m, dl) * k2;
                            const float4 x = rs.dbuf[lane];
                            const float xs[4] = {x.x, x.y, x.z, x.w};
                            float e = 0.f;
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const int r = lane + 32 * u;
                                if (r >= (row_span >> 8) && r < (row_span & 255)) e += ex2(fmaf(xs[u], k2, mk2));
                            }
                            e = warp_sum(e);
                            lE_diag = ms + log2f(e) * LN2;
                        }
                        m_run = red_max(rs, set, J == D ? lE_diag - eps : (valid ? ms - eps : -INFINITY), 1);
                    }
                    if (valid) {
                        eps_tile = fmaxf(eps_tile, eps);
                        const float hi = ms + lnrows + eps;
                        if (hi >= log_alpha + m_run) {
                            // a candidate: screened log-energy (operand-format kbar, fp32 sums); the diagonal
                            // block's is already known
                            const float k2 = scale * LOG2E;
                            float ps[4] = {0.f, 0.f, 0.f, 0.f};
                            if (J == D) {
                            } else if (row_span == 128) {
                                // 2^(v k2 - m k2) with packed FMAs and sums; the rounding of m k2 (|logit| 2^-24)
                                // lies far inside the bound's relative term (2^-12 |q||kbar| >= 2^-12 |logit|)
                                const uint64_t k2x2 = f2pack(k2, k2), mk2 = f2pack(-m * k2, -m * k2);
                                uint64_t acc2[2] = {f2pack(0.f, 0.f), f2pack(0.f, 0.f)};
#pragma unroll
                                for (int x = 0; x < 128; x += 2) {
                                    float y0, y1;
                                    f2unpack(ffma2(f2pack(__uint_as_float(v[x >> 5][x & 31]),
                                                          __uint_as_float(v[x >> 5][(x & 31) + 1])),
                                                   k2x2, mk2),
                                             y0, y1);
                                    acc2[(x >> 1) & 1] = fadd2(acc2[(x >> 1) & 1], f2pack(ex2(y0), ex2(y1)));
                                }
                                f2unpack(acc2[0], ps[0], ps[1]);
                                f2unpack(acc2[1], ps[2], ps[3]);
                            } else {
#pragma unroll
                                for (int x = 0; x < 128; ++x)
                                    if (x >= (row_span >> 8) && x < (row_span & 255))
                                        ps[x & 3] += ex2((__uint_as_float(v[x >> 5][x & 31]) - m) * k2);
                            }
                            const float lE = J == D ? lE_diag : ms + log2f((ps[0] + ps[1]) + (ps[2] + ps[3])) * LN2;
                            blE[J] = lE;
                            bstate[J] = 0;
                            mlo = fmaxf(mlo, lE - eps);
                            mhi = fmaxf(mhi, lE + eps);
                            const int slot = atomicAdd(&rs.ncand, 1);
                            if (slot < kCand) rs.cand[slot] = J;
                        } else {
                            // certainly pruned and certainly not the maximum: hi < ln(alpha) + m_run
                            blE[J] = hi;
                            bstate[J] = kStBound;
                            mhi = fmaxf(mhi, hi);
                        }
                    }
                }
                if (!ok) break;
            }
            // ------------------------------------------------------------ selection
            const int64_t wbase = (int64_t)r.mask_base + (int64_t)(sc.h * r.ntiles + sc.t) * r.words;
            float thr_lo = 0.f, thr_hi = 0.f;
            if (scoring) {
                // one barrier for the three tile-wide maxima
                float e3[3] = {eps_tile, mlo, mhi};
#pragma unroll
                for (int o = 16; o; o >>= 1)
#pragma unroll
                    for (int q = 0; q < 3; ++q) e3[q] = fmaxf(e3[q], __shfl_xor_sync(0xffffffffu, e3[q], o));
                if (lane == 0)
                    for (int q = 0; q < 3; ++q) rs.red3[q][warp & 3] = e3[q];
                red_bar(set);
#pragma unroll
                for (int q = 0; q < 3; ++q)
                    e3[q] = fmaxf(fmaxf(rs.red3[q][0], rs.red3[q][1]), fmaxf(rs.red3[q][2], rs.red3[q][3]));
                eps_tile = e3[0];
                mlo = e3[1];
                mhi = e3[2];
                thr_lo = log_alpha + mlo;
                thr_hi = log_alpha + mhi;
                // settle the candidates against the threshold interval
                const int nc = rs.ncand;
                if (nc > kCand) {
                    if (rt == 0) rs.any2[ap] = 1;
                } else {
                    for (int i = rt; i < nc; i += kRedThreads) {
                        const int J = rs.cand[i];
                        const bool forced = J < sink || (J >= D - window && J < D) || J == D;
                        if (forced) continue;
                        const float lE = blE[J];
                        if (lE - eps_tile >= thr_hi) {
                            atomicOr(&words[J >> 5], 1u << (J & 31));
                            atomicAdd(&rs.nsel, 1);
                        } else if (lE + eps_tile >= thr_lo) {
                            rs.any2[ap] = 1;
                        }
                    }
                }
                red_bar(set);
            }
            if (scoring && rs.any2[ap]) {
                // fp32 recomputation of every unsettled block and every candidate for the maximum
                if (rt == 0) atomicAdd(status + kStatusExactTiles, 1);
                int nrefined = 0;
                for (int J = rt; J <= D; J += kRedThreads) {
                    const bool forced = J < sink || (J >= D - window && J < D) || J == D;
                    const bool bound = bstate[J] & kStBound;
                    const float lo = bound ? -INFINITY : blE[J] - eps_tile;
                    const float hi = bound ? blE[J] : blE[J] + eps_tile;
                    uint8_t st = 0;
                    if (forced || lo >= thr_hi) st |= kStSelected;
                    else if (!(hi < thr_lo)) st |= kStUncertain;
                    if (hi >= mlo) st |= kStMaxCand;
                    bstate[J] = st;
                }
                float qr[kHeadDim];
                if (j >= (row_span >> 8) && j < (row_span & 255)) {
                    // row j of the tile: position q_pos + j / g, query head h g + j % g
                    const uint4 *src = reinterpret_cast<const uint4 *>(
                        qg + (((int64_t)(sc.q_pos + j / g) * hq + sc.h * g + j % g) * kHeadDim) * SCfg<kDtype>::kEb);
                    constexpr int kPer = 16 / SCfg<kDtype>::kEb;
#pragma unroll
                    for (int v = 0; v < kHeadDim / kPer; ++v) {
                        const uint4 x = __ldg(src + v);
                        const uint8_t *b = reinterpret_cast<const uint8_t *>(&x);
#pragma unroll
                        for (int e = 0; e < kPer; ++e) {
                            float f;
                            if (kDtype == FP_DTYPE_BF16)
                                f = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(b + 2 * e));
                            else
                                f = float(*reinterpret_cast<const __nv_fp8_e4m3 *>(b + e));
                            qr[v * kPer + e] = f * qscale;
                        }
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < kHeadDim; ++c) qr[c] = 0.f;
                }
                for (;;) {
                    if (rt == 0) rs.nlist = 0;
                    red_bar(set);
                    // collect up to kRefineList pending candidates, in order
                    for (int J0 = 0; J0 <= D; J0 += kRedThreads) {
                        const int J = J0 + rt;
                        const bool need = J <= D && (bstate[J] & (kStUncertain | kStMaxCand)) &&
                                          !(bstate[J] & kStRefined);
                        const unsigned bal = __ballot_sync(0xffffffffu, need);
                        int base = 0;
                        if (lane == 0 && bal) base = atomicAdd(&rs.nlist, __popc(bal));
                        base = __shfl_sync(0xffffffffu, base, 0);
                        if (need) {
                            const int slot = base + __popc(bal & ((1u << lane) - 1u));
                            if (slot < kRefineList) rs.list[slot] = J;
                        }
                        red_bar(set);
                        if (rs.nlist >= kRefineList) break;
                    }
                    const int n = min(rs.nlist, kRefineList);
                    if (n == 0) break;
                    nrefined += n;
                    for (int i = 0; i < n; ++i) {
                        const int J = rs.list[i];
                        const float *kb = kbar + ((int64_t)(r.blk_base + J) * hkv + sc.h) * kHeadDim;
                        float dot = 0.f;
#pragma unroll
                        for (int c = 0; c < kHeadDim; c += 4) {
                            const float4 k4 = __ldg(reinterpret_cast<const float4 *>(kb + c));
                            dot = fmaf(qr[c], k4.x, dot);
                            dot = fmaf(qr[c + 1], k4.y, dot);
                            dot = fmaf(qr[c + 2], k4.z, dot);
                            dot = fmaf(qr[c + 3], k4.w, dot);
                        }
                        const float s = j >= (row_span >> 8) && j < (row_span & 255) ? dot * inv_sqrt_d : -INFINITY;
                        const float mxs = red_max(rs, set, s, 0);
                        const float e = j >= (row_span >> 8) && j < (row_span & 255) ? expf(s - mxs) : 0.f;
                        const float sum = red_sum(rs, set, e, 1);
                        if (rt == 0) {
                            blE[J] = mxs + logf(sum);
                            bstate[J] |= kStRefined;
                        }
                        red_bar(set);
                    }
                    red_bar(set);
                }
                if (rt == 0) atomicAdd(status + kStatusExactBlocks, nrefined);
                // every candidate for the maximum is now exact
                float mex = -INFINITY;
                for (int J = rt; J <= D; J += kRedThreads)
                    if (bstate[J] & kStMaxCand) mex = fmaxf(mex, blE[J]);
                mex = red_max(rs, set, mex, 0);
                const float thr = log_alpha + mex;
                for (int J = rt; J <= D; J += kRedThreads) {
                    const uint8_t st = bstate[J];
                    if ((st & kStUncertain) && blE[J] >= thr) bstate[J] = st | kStSelected;
                }
                red_bar(set);
                // rebuild the mask words from the final states
                int cnt = 0;
                for (int J0 = 32 * (warp & 3); J0 < 32 * r.words; J0 += kRedThreads) {
                    const int J = J0 + lane;
                    const bool sel = J <= D && (bstate[J] & kStSelected);
                    const unsigned bits = __ballot_sync(0xffffffffu, sel);
                    if (lane == 0) mask[wbase + (J0 >> 5)] = bits;
                    cnt += __popc(bits);
                }
                cnt = (int)red_sum(rs, set, lane == 0 ? (float)cnt : 0.f, 0);
                if (rt == 0) seg_count[seg] = cnt;
                red_bar(set);
            } else {
                // settled by bounds: forced blocks plus the selected candidates
                if (!scoring) red_bar(set);  // the forced words are complete
                for (int k = rt; k < r.words; k += kRedThreads) {
                    uint32_t wv = words[k];
                    if (mode == kModeAll) wv = range_bits(k, 0, D + 1);
                    mask[wbase + k] = wv;
                }
                if (rt == 0) {
                    const int forced_cnt = s_end + max(0, D - max(w_lo, s_end)) + (D >= sink ? 1 : 0);
                    seg_count[seg] = mode == kModeAll ? D + 1 : forced_cnt + (scoring ? rs.nsel : 0);
                }
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

}  // namespace

cudaError_t launch_score(const Ctx &c, const void *q, const float *kbar, const void *kbar_op, float alpha, int sink,
                         int window) {
    const int mode = alpha == 0.f ? kModeAll : (alpha > 1.f ? kModeForced : kModeScore);
    const float log_alpha = alpha > 0.f ? logf(alpha) : -INFINITY;
    const bool fp8 = c.p.dtype == FP_DTYPE_E4M3;
    const int eb = fp8 ? 1 : 2;
    const int g = c.s.g, hkv = c.p.num_kv_heads, hq = c.p.num_q_heads;
    CUtensorMap tm_q, tm_k;
    {
        const uint64_t dims[4] = {128, (uint64_t)g, (uint64_t)hkv, (uint64_t)c.s.total_tokens};
        const uint64_t strides[3] = {(uint64_t)128 * eb, (uint64_t)g * 128 * eb, (uint64_t)hq * 128 * eb};
        const uint32_t box[4] = {(uint32_t)(128 / eb), (uint32_t)g, 1, (uint32_t)(kTileRows / g)};
        if (!make_tmap(&tm_q, q, fp8, 4, dims, strides, box)) return cudaErrorInvalidValue;
    }
    {
        const uint64_t dims[3] = {128, (uint64_t)hkv, (uint64_t)c.s.nblocks};
        const uint64_t strides[2] = {(uint64_t)128 * eb, (uint64_t)hkv * 128 * eb};
        const uint32_t box[3] = {(uint32_t)(128 / eb), 1, 128};
        if (!make_tmap(&tm_k, kbar_op, fp8, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    const int grid = (int)(c.s.nseg < num_sms() ? c.s.nseg : num_sms());
    // per-block scratch for the longest request; two chunk stages per set when they fit, else one
    const int nb = ((c.s.max_blocks > 0 ? c.s.max_blocks : 1) + 127) / 128 * 128;
    const int tile = fp8 ? SCfg<FP_DTYPE_E4M3>::kTile : SCfg<FP_DTYPE_BF16>::kTile;
    int dev = 0, cap = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&cap, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess || cap <= 0)
        cap = 232448;
    // two Q buffers per set (the next tile's Q loads during this tile) only beside two chunk stages: a second
    // chunk stage is worth more than a second Q buffer (BF16 128K: 0.650 ms with 1 + 2, 0.685 ms with 2 + 1;
    // E4M3, where 2 + 2 fit: 0.591 -> 0.582 ms)
    int nq = 2, nst = 2;
    if (score_layout(tile, nq, nst, nb).total + 1024 > (uint32_t)cap) nq = 1;
    if (score_layout(tile, nq, nst, nb).total + 1024 > (uint32_t)cap) nst = 1;
    const size_t smem = score_layout(tile, nq, nst, nb).total + 1024;
    if (smem > (size_t)cap) return cudaErrorInvalidConfiguration;
    cudaError_t e;
    if (fp8) {
        e = cudaFuncSetAttribute(score_tc_kernel<FP_DTYPE_E4M3>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        score_tc_kernel<FP_DTYPE_E4M3><<<grid, kSThreads, smem, c.stream>>>(
            tm_q, tm_k, kbar, c.kstat(), c.req(), c.p.batch, hkv, g, mode, log_alpha, sink, window, c.p.c_q,
            c.p.c_k, (int32_t)c.s.nseg, c.seg_count(), c.mask(), (const uint8_t *)q, hq, nq, nst, nb, c.status());
    } else {
        e = cudaFuncSetAttribute(score_tc_kernel<FP_DTYPE_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
        if (e != cudaSuccess) return e;
        score_tc_kernel<FP_DTYPE_BF16><<<grid, kSThreads, smem, c.stream>>>(
            tm_q, tm_k, kbar, c.kstat(), c.req(), c.p.batch, hkv, g, mode, log_alpha, sink, window, 1.f, 1.f,
            (int32_t)c.s.nseg, c.seg_count(), c.mask(), (const uint8_t *)q, hq, nq, nst, nb, c.status());
    }
    return cudaGetLastError();
}

}  // namespace fp
