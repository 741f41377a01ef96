// Stage 1 of FlashPrefill V2 (Alg.1 steps 1-5): request tables, block mean
// pooling (Eq.5), pooled-key scoring (Eq.19), max-based thresholding with
// forced blocks (Eq.20) and CSR assembly (Sec.3.3 "Index-Driven Sparse
// Traversal").
#include <math.h>

#include "fp_internal.cuh"

namespace fp {
namespace {

// ------------------------------------------------------------ block scan helper

// Inclusive scan of three int32 lanes across a CTA of blockDim.x threads
// (a multiple of 32). Returns the inclusive values; totals go to `tot`.
__device__ void block_scan3(int32_t v[3], int32_t tot[3]) {
    __shared__ int32_t warp_sums[32][3];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
#pragma unroll
    for (int k = 0; k < 3; ++k) {
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int32_t n = __shfl_up_sync(0xffffffffu, v[k], o);
            if (lane >= o) v[k] += n;
        }
    }
    if (lane == 31)
        for (int k = 0; k < 3; ++k) warp_sums[warp][k] = v[k];
    __syncthreads();
    if (warp == 0) {
        for (int k = 0; k < 3; ++k) {
            int32_t s = lane < nwarps ? warp_sums[lane][k] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                int32_t n = __shfl_up_sync(0xffffffffu, s, o);
                if (lane >= o) s += n;
            }
            if (lane < nwarps) warp_sums[lane][k] = s;
        }
    }
    __syncthreads();
    for (int k = 0; k < 3; ++k) {
        if (warp > 0) v[k] += warp_sums[warp - 1][k];
        tot[k] = warp_sums[nwarps - 1][k];
    }
    __syncthreads();
}

// ------------------------------------------------------------------ prep kernel

// Builds the per-request table from the device cu_seqlens and seqlens_kv and
// checks it against the totals the host derived from the host copies.
__global__ void __launch_bounds__(1024) prep_kernel(const int32_t *__restrict__ cu, const int32_t *__restrict__ kv,
                                                    int batch, int hkv, int g, int64_t want_nseg,
                                                    int64_t want_blocks, int64_t want_words, int64_t want_tokens,
                                                    int64_t want_kv_tokens, ReqInfo *__restrict__ req,
                                                    int32_t *__restrict__ status) {
    __shared__ int32_t carry[3];
    __shared__ int bad;
    __shared__ unsigned long long kv_sum;
    if (threadIdx.x == 0) {
        carry[0] = carry[1] = carry[2] = 0;
        bad = 0;
        kv_sum = 0ull;
    }
    __syncthreads();
    for (int base = 0; base < batch; base += blockDim.x) {
        const int b = base + threadIdx.x;
        ReqInfo r = {};
        int32_t v[3] = {0, 0, 0};
        if (b < batch) {
            int32_t q0 = cu[b], q1 = cu[b + 1];
            int32_t L = q1 - q0;
            int32_t Lkv = kv ? kv[b] : L;
            if (q0 < 0 || L < 0 || Lkv < L || Lkv > kMaxLen || q1 > want_tokens) {
                bad = 1;
                L = Lkv = 0;
            }
            atomicAdd(&kv_sum, (unsigned long long)Lkv);
            r.q_start = q0;
            r.len = L;
            r.kv_len = Lkv;
            r.t0 = (g * (Lkv - L)) / kTileRows;
            r.nblocks = (Lkv + kBlock - 1) / kBlock;
            r.ntiles = L > 0 ? (g * Lkv + kTileRows - 1) / kTileRows - r.t0 : 0;
            r.words = (r.nblocks + 31) / 32;
            v[0] = r.nblocks;
            v[1] = hkv * r.ntiles;
            v[2] = hkv * r.ntiles * r.words;
        }
        int32_t own[3] = {v[0], v[1], v[2]};
        int32_t tot[3];
        block_scan3(v, tot);
        if (b < batch) {
            r.blk_base = carry[0] + v[0] - own[0];
            r.seg_base = carry[1] + v[1] - own[1];
            r.mask_base = carry[2] + v[2] - own[2];
            req[b] = r;
        }
        __syncthreads();
        if (threadIdx.x == 0)
            for (int k = 0; k < 3; ++k) carry[k] += tot[k];
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        ReqInfo s = {};
        s.blk_base = carry[0];
        s.seg_base = carry[1];
        s.mask_base = carry[2];
        req[batch] = s;
        if (bad || carry[0] != want_blocks || carry[1] != want_nseg || carry[2] != want_words ||
            cu[batch] != want_tokens || kv_sum != (unsigned long long)want_kv_tokens)
            set_status(status, FP_ERR_DEVICE_SEQLEN);
    }
}

// ----------------------------------------------------------------- pool kernel

// One CTA per (request, block): the means of its <= 128 tokens for every KV
// head (Eq.5). Each thread accumulates one 16-byte column vector of the
// token rows over a strided subset of tokens in fp32; a shared-memory pass
// sums the token groups. FP8 elements are descaled before summing. The
// block's page ids are looked up once per CTA, and the per-head rounding
// statistics are reduced within each warp before their shared atomics.
// With reuse_prefix, a block lying wholly in the request's cached prefix
// keeps the means already in the arrays (an earlier chunk's pooling of the
// same keys and values) and only its rounding statistics are recomputed.
template <int kDtype>
__global__ void __launch_bounds__(256) pool_kernel(const uint8_t *__restrict__ kp, const uint8_t *__restrict__ vp,
                                                   const int32_t *__restrict__ page_table, int pt_stride,
                                                   int num_pages, int page_size, const ReqInfo *__restrict__ req,
                                                   int batch, int hkv, float c_k, float c_v,
                                                   float *__restrict__ kbar, float *__restrict__ vbar,
                                                   void *__restrict__ kbar_op, void *__restrict__ vbar_op,
                                                   float2 *__restrict__ kstat, int reuse_prefix,
                                                   int32_t *__restrict__ status) {
    using E = Elem<kDtype>;
    constexpr int kEb = E::kBytes;
    constexpr int kEpv = 16 / kEb;  // elements per 16-byte vector
    __shared__ float red[2][256 * kEpv];
    __shared__ float kst[2][64];  // per KV head: squared rounding error and squared norm of kbar
    __shared__ int32_t pages[kBlock / 8];  // the block's page ids (page_size >= 8), -1 if out of range
    if (status_bad(status)) return;
    if (threadIdx.x < 64) kst[0][threadIdx.x] = kst[1][threadIdx.x] = 0.f;
    const int gb = blockIdx.x;
    const int b = find_req_by_block(req, batch, gb);
    const ReqInfo r = req[b];
    const int J = gb - r.blk_base;
    if (reuse_prefix && (J + 1) * kBlock <= r.kv_len - r.len) {
        // every token of the block precedes the new ones: its means are kept; the rounding statistics of the
        // operand-format key mean go to this call's workspace, reduced in the same warp grouping as below
        const int64_t base = (int64_t)gb * hkv * kHeadDim;
        __syncthreads();
        for (int x = threadIdx.x; x < hkv * kHeadDim; x += 256) {
            const float mk = kbar[base + x];
            const float kq = kDtype == FP_DTYPE_E4M3
                                 ? float(reinterpret_cast<const __nv_fp8_e4m3 *>(kbar_op)[base + x]) * c_k
                                 : __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(kbar_op)[base + x]);
            float e2 = (mk - kq) * (mk - kq), n2 = mk * mk;
#pragma unroll
            for (int o = 16; o; o >>= 1) {
                e2 += __shfl_xor_sync(0xffffffffu, e2, o);
                n2 += __shfl_xor_sync(0xffffffffu, n2, o);
            }
            if ((threadIdx.x & 31) == 0) {
                atomicAdd(&kst[0][x / kHeadDim], e2);
                atomicAdd(&kst[1][x / kHeadDim], n2);
            }
        }
        __syncthreads();
        if (threadIdx.x < hkv)
            kstat[(int64_t)gb * hkv + threadIdx.x] =
                make_float2(sqrtf(kst[0][threadIdx.x]), sqrtf(kst[1][threadIdx.x]));
        return;
    }
    const int n = min(kBlock, r.kv_len - J * kBlock);
    const int npg = (n + page_size - 1) / page_size;  // pages holding the block's tokens (blocks start on a page)
    if (threadIdx.x < npg) {
        const int page = page_table[(int64_t)b * pt_stride + (J * kBlock) / page_size + threadIdx.x];
        const bool ok = page >= 0 && page < num_pages;
        if (!ok) set_status(status, FP_ERR_DEVICE_PAGE, page);
        pages[threadIdx.x] = ok ? page : -1;
    }
    __syncthreads();
    const int row_bytes = hkv * kHeadDim * kEb;
    const int nvec = row_bytes / 16;
    const int TG = nvec >= 256 ? 1 : 256 / nvec;
    const int cols = 256 / TG;
    const float sk = kDtype == FP_DTYPE_E4M3 ? c_k : 1.f;
    const float sv = kDtype == FP_DTYPE_E4M3 ? c_v : 1.f;
    for (int c0 = 0; c0 < nvec; c0 += cols) {
        const int col = c0 + threadIdx.x % cols;
        const int tg = threadIdx.x / cols;
        float ak[kEpv], av[kEpv];
#pragma unroll
        for (int e = 0; e < kEpv; ++e) ak[e] = av[e] = 0.f;
        if (col < nvec && tg < TG) {
            for (int j = tg; j < n; j += TG) {
                const int page = pages[j / page_size];
                if (page < 0) continue;
                const int64_t off = ((int64_t)page * page_size + j % page_size) * row_bytes + (int64_t)col * 16;
                const uint4 kraw = __ldg(reinterpret_cast<const uint4 *>(kp + off));
                const uint4 vraw = __ldg(reinterpret_cast<const uint4 *>(vp + off));
                const typename E::T *ke = reinterpret_cast<const typename E::T *>(&kraw);
                const typename E::T *ve = reinterpret_cast<const typename E::T *>(&vraw);
#pragma unroll
                for (int e = 0; e < kEpv; ++e) {
                    ak[e] += E::to_float(ke[e]) * sk;
                    av[e] += E::to_float(ve[e]) * sv;
                }
            }
        }
#pragma unroll
        for (int e = 0; e < kEpv; ++e) {
            red[0][threadIdx.x * kEpv + e] = ak[e];
            red[1][threadIdx.x * kEpv + e] = av[e];
        }
        __syncthreads();
        const float inv_n = 1.f / (float)n;
        for (int x = threadIdx.x; x < cols * kEpv; x += 256) {
            const int lc = x / kEpv, e = x % kEpv;
            const int colx = c0 + lc;
            // element c0 kEpv + x: the bound hkv * 128 is a multiple of 32, so whole warps skip together
            if (colx >= nvec) continue;
            float sk_ = 0.f, sv_ = 0.f;
            for (int t = 0; t < TG; ++t) {
                sk_ += red[0][(t * cols + lc) * kEpv + e];
                sv_ += red[1][(t * cols + lc) * kEpv + e];
            }
            const float mk = sk_ * inv_n, mv = sv_ * inv_n;
            const int64_t oi = (int64_t)gb * hkv * kHeadDim + (int64_t)colx * kEpv + e;
            kbar[oi] = mk;
            vbar[oi] = mv;
            float kq;  // the operand-format value as the tensor core sees it, in real units
            if (kDtype == FP_DTYPE_E4M3) {
                const __nv_fp8_e4m3 k8(mk / c_k);
                reinterpret_cast<__nv_fp8_e4m3 *>(kbar_op)[oi] = k8;
                reinterpret_cast<__nv_fp8_e4m3 *>(vbar_op)[oi] = __nv_fp8_e4m3(mv / c_v);
                kq = float(k8) * c_k;
            } else {
                const __nv_bfloat16 k16 = __float2bfloat16_rn(mk);
                reinterpret_cast<__nv_bfloat16 *>(kbar_op)[oi] = k16;
                reinterpret_cast<__nv_bfloat16 *>(vbar_op)[oi] = __float2bfloat16_rn(mv);
                kq = __bfloat162float(k16);
            }
            // a warp's 32 consecutive elements lie in one head: reduce them before the shared atomics
            float e2 = (mk - kq) * (mk - kq), n2 = mk * mk;
#pragma unroll
            for (int o = 16; o; o >>= 1) {
                e2 += __shfl_xor_sync(0xffffffffu, e2, o);
                n2 += __shfl_xor_sync(0xffffffffu, n2, o);
            }
            if ((threadIdx.x & 31) == 0) {
                const int head = (colx * kEpv + e) / kHeadDim;
                atomicAdd(&kst[0][head], e2);
                atomicAdd(&kst[1][head], n2);
            }
        }
        __syncthreads();
    }
    if (threadIdx.x < hkv)
        kstat[(int64_t)gb * hkv + threadIdx.x] = make_float2(sqrtf(kst[0][threadIdx.x]), sqrtf(kst[1][threadIdx.x]));
}

// ------------------------------------------------------------------ CSR kernels

// Exclusive scan of the per-segment counts into csr_cu (one CTA). In rounds of
// 32 warps x 1024 counts, warp w scans its own 1024 consecutive counts, 32 at
// a time with coalesced loads and stores, and the CTA offsets the warps by a
// scan of their totals.
__global__ void __launch_bounds__(1024) csr_scan_kernel(const int32_t *__restrict__ count, int32_t nseg,
                                                        int64_t capacity, int32_t *__restrict__ cu,
                                                        int32_t *__restrict__ status) {
    constexpr int kRows = 32;  // rows of 32 counts per warp and round
    __shared__ int32_t wsum[32];
    __shared__ int32_t carry;
    if (status_bad(status)) {
        if (threadIdx.x == 0) cu[0] = 0;
        return;
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) carry = 0;
    for (int base = 0; base < nseg; base += 32 * 32 * kRows) {
        const int cs = base + warp * 32 * kRows;
        int32_t v[kRows];
#pragma unroll
        for (int q = 0; q < kRows; ++q) {
            const int i = cs + 32 * q + lane;
            v[q] = i < nseg ? count[i] : 0;
        }
        int32_t run = 0;  // the warp's running total; v[q] becomes the exclusive prefix within the warp's counts
#pragma unroll
        for (int q = 0; q < kRows; ++q) {
            int32_t x = v[q];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t n = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += n;
            }
            const int32_t own = v[q];
            v[q] = run + x - own;
            run += __shfl_sync(0xffffffffu, x, 31);
        }
        if (lane == 0) wsum[warp] = run;
        __syncthreads();
        if (warp == 0) {
            int32_t w = wsum[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t n = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += n;
            }
            wsum[lane] = w;
        }
        __syncthreads();
        const int32_t off = carry + (warp ? wsum[warp - 1] : 0);
#pragma unroll
        for (int q = 0; q < kRows; ++q) {
            const int i = cs + 32 * q + lane;
            if (i < nseg) cu[i] = off + v[q];
        }
        __syncthreads();
        if (threadIdx.x == 0) carry += wsum[31];
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        cu[nseg] = carry;
        if (carry > capacity) set_status(status, FP_ERR_DEVICE_OVERFLOW, carry);
    }
}

// One warp per segment: expands the selection bitmask into ascending block ids.
__global__ void __launch_bounds__(256) csr_expand_kernel(const uint32_t *__restrict__ mask,
                                                         const ReqInfo *__restrict__ req, int batch, int g,
                                                         int32_t nseg, const int32_t *__restrict__ cu,
                                                         int64_t capacity, int32_t *__restrict__ idx,
                                                         int32_t *__restrict__ status) {
    if (status_bad(status)) return;
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t seg = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); seg < nseg; seg += warps) {
        const SegCoord sc = decode_seg(req, batch, g, seg);
        const ReqInfo r = req[sc.b];
        const int64_t wbase = (int64_t)r.mask_base + (int64_t)(sc.h * r.ntiles + sc.t) * r.words;
        const int nw = (sc.D + 1 + 31) / 32;
        int64_t pos = cu[seg];
        for (int w0 = 0; w0 < nw; w0 += 32) {
            const int w = w0 + lane;
            uint32_t word = w < nw ? mask[wbase + w] : 0u;
            const int c = __popc(word);
            int incl = c;
            for (int o = 1; o < 32; o <<= 1) {
                int n = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += n;
            }
            int64_t p = pos + incl - c;
            while (word) {
                const int bit = __ffs(word) - 1;
                if (p < capacity) idx[p] = 32 * w + bit;
                ++p;
                word &= word - 1;
            }
            pos += __shfl_sync(0xffffffffu, incl, 31);
        }
    }
}

}  // namespace

cudaError_t launch_prep(const Ctx &c) {
    const int threads = 1024;
    prep_kernel<<<1, threads, 0, c.stream>>>(c.p.cu_seqlens, c.p.seqlens_kv, c.p.batch, c.p.num_kv_heads, c.s.g,
                                             c.s.nseg, c.s.nblocks, c.s.mask_words, c.s.total_tokens,
                                             c.s.kv_tokens, c.req(), c.status());
    return cudaGetLastError();
}

cudaError_t launch_pool(const Ctx &c, const void *k_pages, const void *v_pages, float *kbar, float *vbar,
                        void *kbar_op, void *vbar_op, bool reuse_prefix) {
    const dim3 grid((unsigned)c.s.nblocks);
    if (c.p.dtype == FP_DTYPE_E4M3)
        pool_kernel<FP_DTYPE_E4M3><<<grid, 256, 0, c.stream>>>(
            (const uint8_t *)k_pages, (const uint8_t *)v_pages, c.p.page_table, c.p.page_table_stride,
            c.p.num_pages, c.p.page_size, c.req(), c.p.batch, c.p.num_kv_heads, c.p.c_k, c.p.c_v, kbar, vbar,
            kbar_op, vbar_op, c.kstat(), reuse_prefix ? 1 : 0, c.status());
    else
        pool_kernel<FP_DTYPE_BF16><<<grid, 256, 0, c.stream>>>(
            (const uint8_t *)k_pages, (const uint8_t *)v_pages, c.p.page_table, c.p.page_table_stride,
            c.p.num_pages, c.p.page_size, c.req(), c.p.batch, c.p.num_kv_heads, 1.f, 1.f, kbar, vbar, kbar_op,
            vbar_op, c.kstat(), reuse_prefix ? 1 : 0, c.status());
    return cudaGetLastError();
}

// ---------------------------------------------------- 64-token tile expansion

// Tiles block J of a request of length len covers: 2J, and 2J + 1 when (2J + 1) * 64 < len.
__device__ __forceinline__ int tiles_of_block(int J, int len) { return 1 + ((2 * J + 1) * 64 < len ? 1 : 0); }

// One warp per segment: the number of 64-token tiles its selected blocks cover.
__global__ void __launch_bounds__(256) tile_count_kernel(const ReqInfo *__restrict__ req, int batch, int g,
                                                         int32_t nseg, const int32_t *__restrict__ cu,
                                                         const int32_t *__restrict__ idx, int32_t *__restrict__ count,
                                                         int32_t *__restrict__ status) {
    if (status_bad(status)) return;
    const int lane = threadIdx.x & 31;
    const int64_t seg = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (seg >= nseg) return;
    const int b = find_req_by_seg(req, batch, seg);
    const ReqInfo r = req[b];
    int n = 0;
    for (int64_t i = cu[seg] + lane; i < cu[seg + 1]; i += 32) {
        const int J = idx[i];
        if (J < 0 || J >= r.nblocks) set_status(status, FP_ERR_DEVICE_CSR, (int32_t)seg);
        else n += tiles_of_block(J, r.kv_len);
    }
    for (int o = 16; o; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
    if (lane == 0) count[seg] = n;
}

// One warp per segment: writes the tiles in order (a warp-wide exclusive scan of the per-entry counts).
__global__ void __launch_bounds__(256) tile_expand_kernel(const ReqInfo *__restrict__ req, int batch, int32_t nseg,
                                                          const int32_t *__restrict__ cu,
                                                          const int32_t *__restrict__ idx,
                                                          const int32_t *__restrict__ tile_cu, int64_t capacity,
                                                          int32_t *__restrict__ tile_idx, int32_t *__restrict__ status) {
    if (status_bad(status)) return;
    const int lane = threadIdx.x & 31;
    const int64_t seg = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
    if (seg >= nseg) return;
    const ReqInfo r = req[find_req_by_seg(req, batch, seg)];
    int64_t out = tile_cu[seg];
    for (int64_t i0 = cu[seg]; i0 < cu[seg + 1]; i0 += 32) {
        const int64_t i = i0 + lane;
        int J = -1, n = 0;
        if (i < cu[seg + 1]) {
            J = idx[i];
            if (J >= 0 && J < r.nblocks) n = tiles_of_block(J, r.kv_len);
        }
        int incl = n;
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += v;
        }
        const int64_t at = out + incl - n;
        for (int k = 0; k < n; ++k)
            if (at + k < capacity) tile_idx[at + k] = 2 * J + k;
        out += __shfl_sync(0xffffffffu, incl, 31);
    }
}

cudaError_t launch_expand64(const Ctx &c, const int32_t *csr_cu, const int32_t *csr_idx, int32_t *tile_cu,
                            int32_t *tile_idx, int64_t capacity) {
    const int64_t nseg = c.s.nseg;
    const unsigned blocks = (unsigned)((nseg + 7) / 8);
    if (nseg > 0) {
        tile_count_kernel<<<blocks, 256, 0, c.stream>>>(c.req(), c.p.batch, c.s.g, (int32_t)nseg, csr_cu, csr_idx,
                                                        c.seg_count(), c.status());
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    csr_scan_kernel<<<1, 1024, 0, c.stream>>>(c.seg_count(), (int32_t)nseg, capacity, tile_cu, c.status());
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || nseg == 0) return e;
    tile_expand_kernel<<<blocks, 256, 0, c.stream>>>(c.req(), c.p.batch, (int32_t)nseg, csr_cu, csr_idx, tile_cu,
                                                     capacity, tile_idx, c.status());
    return cudaGetLastError();
}

cudaError_t launch_csr(const Ctx &c, int32_t *csr_cu, int32_t *csr_idx, int64_t capacity) {
    csr_scan_kernel<<<1, 1024, 0, c.stream>>>(c.seg_count(), (int32_t)c.s.nseg, capacity, csr_cu, c.status());
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || c.s.nseg == 0) return e;
    const int64_t warps = c.s.nseg;
    const unsigned blocks = (unsigned)((warps + 7) / 8 < 65535 * 8 ? (warps + 7) / 8 : 65535 * 8);
    csr_expand_kernel<<<blocks, 256, 0, c.stream>>>(c.mask(), c.req(), c.p.batch, c.s.g, (int32_t)c.s.nseg, csr_cu,
                                                    capacity, csr_idx, c.status());
    return cudaGetLastError();
}

}  // namespace fp
