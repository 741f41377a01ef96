// Stage 2 of FlashPrefill V2 (Alg.1 steps 6-11): exact attention over each
// segment's selected blocks walked in descending order (Eq.17), one
// mean-correction term per pruned causal block (Eq.6, Sec.3.2
// "Implementation"), online softmax and the epilogue division; FP8 follows
// Eq.15.
#include <math.h>

#include "fp_internal.cuh"

namespace fp {
namespace {

constexpr int kAttnThreads = 256;  // two threads per packed row, 64 dims each
constexpr int kChunk = 16;         // keys per online-softmax update

template <int kDtype>
struct AttnSmem {
    using T = typename Elem<kDtype>::T;
    T k[kBlock][kHeadDim];
    T v[kBlock][kHeadDim];
    uint32_t todo[kMaxBlocks / 32];
    int flag;
};

// Copies the 128 key and value rows of block J of (request b, KV head h) into
// shared memory through the page table (Eq.22); rows past the request are zero.
template <int kDtype>
__device__ void load_kv_block(AttnSmem<kDtype> &sm, const uint8_t *kp, const uint8_t *vp, const int32_t *pt,
                              int pt_stride, int num_pages, int page_size, int b, int hkv, int h, int L, int J,
                              int32_t *status) {
    constexpr int kEb = Elem<kDtype>::kBytes;
    constexpr int kVecs = kHeadDim * kEb / 16;  // 16-byte vectors per row
    for (int x = threadIdx.x; x < kBlock * kVecs; x += kAttnThreads) {
        const int row = x / kVecs, v = x % kVecs;
        const int tok = J * kBlock + row;
        uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
        if (tok < L) {
            const int page = pt[(int64_t)b * pt_stride + tok / page_size];
            if (page >= 0 && page < num_pages) {
                const int64_t off = (((int64_t)page * page_size + tok % page_size) * hkv + h) * kHeadDim * kEb;
                kv = *reinterpret_cast<const uint4 *>(kp + off + v * 16);
                vv = *reinterpret_cast<const uint4 *>(vp + off + v * 16);
            } else {
                set_status(status, FP_ERR_DEVICE_PAGE, page);
            }
        }
        reinterpret_cast<uint4 *>(&sm.k[row][0])[v] = kv;
        reinterpret_cast<uint4 *>(&sm.v[row][0])[v] = vv;
    }
}

// Pooled-mean rows of correction chunk c (blocks 128c .. 128c+127).
template <int kDtype>
__device__ void load_mean_chunk(AttnSmem<kDtype> &sm, const uint8_t *kbar_op, const uint8_t *vbar_op,
                                int blk_base, int hkv, int h, int D, int c) {
    constexpr int kEb = Elem<kDtype>::kBytes;
    constexpr int kVecs = kHeadDim * kEb / 16;
    for (int x = threadIdx.x; x < kBlock * kVecs; x += kAttnThreads) {
        const int row = x / kVecs, v = x % kVecs;
        const int J = c * kBlock + row;
        uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
        if (J < D) {
            const int64_t off = ((int64_t)(blk_base + J) * hkv + h) * kHeadDim * kEb;
            kv = *reinterpret_cast<const uint4 *>(kbar_op + off + v * 16);
            vv = *reinterpret_cast<const uint4 *>(vbar_op + off + v * 16);
        }
        reinterpret_cast<uint4 *>(&sm.k[row][0])[v] = kv;
        reinterpret_cast<uint4 *>(&sm.v[row][0])[v] = vv;
    }
}

// Online-softmax state of one half row (64 of the 128 output dims).
struct RowState {
    float m, l, o[64];
};

// Folds 128 staged keys into the row state. `key_ok(i)` says whether staged
// row i takes part; `shift` is added to every logit (ln|B_J| for means).
template <int kDtype, typename KeyOk>
__device__ void fold_block(const AttnSmem<kDtype> &sm, const float (&qh)[64], int half, float scale, float shift,
                           KeyOk key_ok, RowState &st) {
    using E = Elem<kDtype>;
    for (int k0 = 0; k0 < kBlock; k0 += kChunk) {
        float s[kChunk];
        float cmax = -INFINITY;
#pragma unroll
        for (int kk = 0; kk < kChunk; ++kk) {
            const typename E::T *kr = &sm.k[k0 + kk][half * 64];
            float part = 0.f;
#pragma unroll
            for (int e = 0; e < 64; ++e) part = fmaf(qh[e], E::to_float(kr[e]), part);
            const float full = part + __shfl_xor_sync(0xffffffffu, part, 1);
            s[kk] = key_ok(k0 + kk) ? fmaf(full, scale, shift) : -INFINITY;
            cmax = fmaxf(cmax, s[kk]);
        }
        const float m_new = fmaxf(st.m, cmax);
        if (m_new == -INFINITY) continue;
        const float corr = expf(st.m - m_new);
        st.l *= corr;
#pragma unroll
        for (int e = 0; e < 64; ++e) st.o[e] *= corr;
        st.m = m_new;
#pragma unroll
        for (int kk = 0; kk < kChunk; ++kk) {
            float p = expf(s[kk] - st.m);
            float pw;
            if (kDtype == FP_DTYPE_E4M3) {
                // Eq.15: probabilities shifted into [0, 256] and quantised to E4M3;
                // the denominator sums the quantised values.
                p = float(__nv_fp8_e4m3(256.f * p));
                pw = p;
            } else {
                pw = __bfloat162float(__float2bfloat16_rn(p));
            }
            st.l += p;
            const typename E::T *vr = &sm.v[k0 + kk][half * 64];
#pragma unroll
            for (int e = 0; e < 64; ++e) st.o[e] = fmaf(pw, E::to_float(vr[e]), st.o[e]);
        }
    }
}

template <int kDtype>
__global__ void __launch_bounds__(kAttnThreads) attn_kernel(
    const typename Elem<kDtype>::T *__restrict__ q, const uint8_t *__restrict__ kp, const uint8_t *__restrict__ vp,
    const int32_t *__restrict__ pt, int pt_stride, int num_pages, int page_size, const int32_t *__restrict__ csr_cu,
    const int32_t *__restrict__ csr_idx, int64_t capacity, const uint8_t *__restrict__ kbar_op,
    const uint8_t *__restrict__ vbar_op, int flags, __nv_bfloat16 *__restrict__ out, float *__restrict__ lse,
    const ReqInfo *__restrict__ req, int batch, int hq, int hkv, int g, float c_q, float c_k, float c_v,
    int32_t nseg, int32_t *__restrict__ status) {
    using E = Elem<kDtype>;
    extern __shared__ __align__(16) uint8_t smem_raw[];
    AttnSmem<kDtype> &sm = *reinterpret_cast<AttnSmem<kDtype> *>(smem_raw);
    if (status_bad(status)) return;
    const int seg = nseg - 1 - blockIdx.x;
    const SegCoord sc = decode_seg(req, batch, g, seg);
    const ReqInfo r = req[sc.b];
    const bool dense = flags & FP_DENSE;
    const bool corr = (flags & FP_MEAN_CORRECTION) && !dense;
    const int row = threadIdx.x >> 1, half = threadIdx.x & 1;
    const bool valid = row < sc.rows;
    const int gr = sc.t * kTileRows + row;
    const int pos = gr / g, head = sc.h * g + gr % g;

    float qh[64];
#pragma unroll
    for (int e = 0; e < 64; ++e)
        qh[e] = valid ? E::to_float(q[((int64_t)(r.q_start + pos) * hq + head) * kHeadDim + half * 64 + e]) : 0.f;

    // segment bounds and CSR validation (ids in [0, D], strictly ascending)
    int beg = 0, end = 0;
    if (!dense) {
        beg = csr_cu[seg];
        end = csr_cu[seg + 1];
        int bad = (beg < 0 || end < beg || end > capacity) ? 1 : 0;
        if (!bad)
            for (int i = beg + threadIdx.x; i < end; i += kAttnThreads) {
                const int J = csr_idx[i];
                if (J < 0 || J > sc.D || (i > beg && csr_idx[i - 1] >= J)) bad = 1;
            }
        if (__syncthreads_or(bad)) {
            if (threadIdx.x == 0) set_status(status, FP_ERR_DEVICE_CSR, seg);
            return;
        }
    }
    const int nwords = (sc.D + 31) / 32;
    if (corr) {
        for (int w = threadIdx.x; w < nwords; w += kAttnThreads) {
            const int left = sc.D - 32 * w;
            sm.todo[w] = left >= 32 ? 0xffffffffu : ((1u << left) - 1u);
        }
        __syncthreads();
        for (int i = beg + threadIdx.x; i < end; i += kAttnThreads) {
            const int J = csr_idx[i];
            if (J < sc.D) atomicAnd(&sm.todo[J >> 5], ~(1u << (J & 31)));
        }
    }

    RowState st;
    st.m = -INFINITY;
    st.l = 0.f;
#pragma unroll
    for (int e = 0; e < 64; ++e) st.o[e] = 0.f;
    const float scale = (kDtype == FP_DTYPE_E4M3 ? c_q * c_k : 1.f) / sqrtf((float)kHeadDim);

    const int nexact = dense ? sc.D + 1 : end - beg;
    for (int it = 0; it < nexact; ++it) {
        const int J = dense ? sc.D - it : csr_idx[end - 1 - it];  // descending (Eq.17)
        __syncthreads();
        load_kv_block<kDtype>(sm, kp, vp, pt, pt_stride, num_pages, page_size, sc.b, hkv, sc.h, r.len, J, status);
        __syncthreads();
        const bool diag = J == sc.D;
        fold_block<kDtype>(sm, qh, half, scale, 0.f,
                           [&](int i) { return valid && (!diag || J * kBlock + i <= pos); }, st);
    }
    if (corr) {
        const float shift = logf((float)kBlock);  // ln|B_J|, every corrected block is full
        for (int c = 0; c * kBlock < sc.D; ++c) {
            __syncthreads();
            uint32_t any = 0;
            for (int w = 4 * c; w < min(4 * c + 4, nwords); ++w) any |= sm.todo[w];
            if (!any) continue;  // every block of the chunk was selected
            load_mean_chunk<kDtype>(sm, kbar_op, vbar_op, r.blk_base, hkv, sc.h, sc.D, c);
            __syncthreads();
            fold_block<kDtype>(sm, qh, half, scale, shift,
                               [&](int i) {
                                   const int J = c * kBlock + i;
                                   return valid && J < sc.D && ((sm.todo[J >> 5] >> (J & 31)) & 1u);
                               },
                               st);
        }
    }
    if (!valid) return;
    const float inv = st.l > 0.f ? (kDtype == FP_DTYPE_E4M3 ? c_v : 1.f) / st.l : 0.f;
    __nv_bfloat16 *orow = out + ((int64_t)(r.q_start + pos) * hq + head) * kHeadDim + half * 64;
#pragma unroll
    for (int e = 0; e < 64; e += 2)
        *reinterpret_cast<__nv_bfloat162 *>(orow + e) = __floats2bfloat162_rn(st.o[e] * inv, st.o[e + 1] * inv);
    if (lse && half == 0)
        lse[(int64_t)(r.q_start + pos) * hq + head] =
            st.m + logf(st.l) - (kDtype == FP_DTYPE_E4M3 ? logf(256.f) : 0.f);
}

}  // namespace

cudaError_t launch_attention(const Ctx &c, const void *q, const void *k_pages, const void *v_pages,
                             const int32_t *csr_cu, const int32_t *csr_idx, int64_t capacity, const void *kbar_op,
                             const void *vbar_op, int flags, void *out, float *lse) {
    const dim3 grid((unsigned)c.s.nseg);
    cudaError_t e;
    if (c.p.dtype == FP_DTYPE_E4M3) {
        const size_t smem = sizeof(AttnSmem<FP_DTYPE_E4M3>);
        e = cudaFuncSetAttribute(attn_kernel<FP_DTYPE_E4M3>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attn_kernel<FP_DTYPE_E4M3><<<grid, kAttnThreads, smem, c.stream>>>(
            (const __nv_fp8_e4m3 *)q, (const uint8_t *)k_pages, (const uint8_t *)v_pages, c.p.page_table,
            c.p.page_table_stride, c.p.num_pages, c.p.page_size, csr_cu, csr_idx, capacity,
            (const uint8_t *)kbar_op, (const uint8_t *)vbar_op, flags, (__nv_bfloat16 *)out, lse, c.req(),
            c.p.batch, c.p.num_q_heads, c.p.num_kv_heads, c.s.g, c.p.c_q, c.p.c_k, c.p.c_v, (int32_t)c.s.nseg,
            c.status());
    } else {
        const size_t smem = sizeof(AttnSmem<FP_DTYPE_BF16>);
        e = cudaFuncSetAttribute(attn_kernel<FP_DTYPE_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        attn_kernel<FP_DTYPE_BF16><<<grid, kAttnThreads, smem, c.stream>>>(
            (const __nv_bfloat16 *)q, (const uint8_t *)k_pages, (const uint8_t *)v_pages, c.p.page_table,
            c.p.page_table_stride, c.p.num_pages, c.p.page_size, csr_cu, csr_idx, capacity,
            (const uint8_t *)kbar_op, (const uint8_t *)vbar_op, flags, (__nv_bfloat16 *)out, lse, c.req(),
            c.p.batch, c.p.num_q_heads, c.p.num_kv_heads, c.s.g, 1.f, 1.f, 1.f, (int32_t)c.s.nseg, c.status());
    }
    return cudaGetLastError();
}

}  // namespace fp
