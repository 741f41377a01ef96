/*
 * fp_oracle.c -- plain, slow, fp64 CPU oracle for FlashPrefill V2 causal
 * block-sparse prefill attention with mean correction.
 *
 * TEST INFRASTRUCTURE ONLY. The test-suite, the smoke check and the
 * benchmark's CPU-baseline leg are the only callers. The product path (the
 * CUDA library) never loads, links or calls this file, and this file shares
 * no code, header, table or constant with it.
 *
 * Source: "FlashPrefill V2: Block-Sparse Prefill Attention for Long-Context
 * LLM Serving" (arXiv 2608.19758), referred to below as [V2], and the summary
 * page of its predecessor "FlashPrefill" (arXiv 2603.06199), referred to as
 * [V1]. Every step follows the definitions in the order the paper gives them;
 * no blocking, fusion or reordering beyond what the definitions state.
 *
 * Readings taken where the paper is silent or ambiguous (each one is listed in
 * the design notes of the repository):
 *   - logits carry 1/sqrt(d) everywhere ([V2] Eq.5 and Eq.19; Eq.1 omits it);
 *   - a query tile is 128 packed rows of Q' ([V2] Sec.3.3 "PackGQA", Eq.12-13),
 *     so one tile holds 128/g positions of all g heads of one KV head;
 *   - the maximum in the threshold runs over the causal blocks J <= D of the
 *     tile, forced blocks included ([V2] Eq.20, [V1] Sec.3.4);
 *   - scoring uses the whole-block mean of the diagonal block (no token mask);
 *   - the comparison is ">=" ([V2] Eq.3, Eq.20);
 *   - epsilon of Eq.2 cancels in the comparison and is taken as 0;
 *   - forced set = first `sink` blocks, `window` blocks just before the
 *     diagonal block D, and D itself ([V2] Eq.20);
 *   - corrected blocks are C = {J < D} \ S, the causal blocks fully visible to
 *     the whole tile that were not selected ([V2] Sec.3.2 "Implementation");
 *   - the logit shift of a corrected block is the natural log ln|B_J|;
 *   - with a cached prefix (L^kv > L^q, [V2] Sec.3.4), the new queries are the
 *     last L^q positions, pooling and selection cover all L^kv keys, and tiles
 *     sit on the grid of absolute packed rows (a chunk whose first row is off
 *     that grid starts with a partial tile), so no tile straddles two blocks.
 *
 * Element formats: bf16 (bit pattern, exactly widened), and OCP FP8 E4M3
 * ("fn": no infinities, S.1111.111 is NaN, max 448) multiplied by its
 * per-tensor scale ([V2] Sec.3.3 "FP8 Execution", Eq.15), so the oracle works
 * on exactly the values the GPU receives, in fp64.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_EINVAL (-1)
#define ORC_ENOMEM (-2)
#define ORC_EPAGE (-3)

typedef struct {
    int32_t batch, hq, hkv, d, block, page_size, tile_rows, dtype; /* dtype: 0 bf16, 1 e4m3 */
    double c_q, c_k, c_v;           /* dequantisation scales; ignored for bf16 */
    const int32_t *cu_seqlens;      /* [batch+1] token offsets of the requests in q */
    const int32_t *page_table;      /* [batch * pt_stride] page ids */
    int32_t pt_stride;
    int32_t num_pages;
    const void *q;                  /* [T, hq, d] elements */
    const void *k_pages, *v_pages;  /* [num_pages, page_size, hkv, d] elements */
    const int32_t *seqlens_kv;      /* [batch] KV lengths L_b^kv >= L_b^q, or NULL for L_b^kv = L_b^q */
} orc_problem;

/* ------------------------------------------------------------------ decode */

double orc_decode_bf16(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP 8-bit floating point, E4M3 variant: bias 7, 3 mantissa bits,
 * subnormals at exponent field 0, only S.1111.111 encodes NaN. */
double orc_decode_e4m3(uint8_t x) {
    int sign = x >> 7, e = (x >> 3) & 15, m = x & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);            /* (m/8) * 2^(1-7) */
    else
        v = ldexp((double)(8 + m), e - 10);  /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

/* The E4M3 value nearest to x, ties to even, saturating at +-448 (the same
 * format: 3 mantissa bits, so within the binade [2^e, 2^(e+1)) the spacing is
 * 2^(e-3); below 2^-6 the subnormal spacing 2^-9 continues the lowest binade's).
 * The division by the spacing is exact, and nearbyint rounds ties to even in
 * the default rounding mode. */
double orc_round_e4m3(double x) {
    double a = fabs(x);
    if (a == 0.0 || isnan(x)) return x;
    int e;
    frexp(a, &e); /* a = f 2^e with f in [0.5, 1): a lies in [2^(e-1), 2^e) */
    int lo = e - 1 < -6 ? -6 : e - 1;
    double spacing = ldexp(1.0, lo - 3);
    double r = nearbyint(a / spacing) * spacing;
    if (r > 448.0) r = 448.0;
    return copysign(r, x);
}

void orc_round_e4m3_n(const double *x, double *y, int64_t n) {
    for (int64_t i = 0; i < n; ++i) y[i] = orc_round_e4m3(x[i]);
}

static double elem(const orc_problem *p, const void *base, size_t i, double scale) {
    if (p->dtype == 0) return orc_decode_bf16(((const uint16_t *)base)[i]);
    return scale * orc_decode_e4m3(((const uint8_t *)base)[i]);
}

/* --------------------------------------------------------------- geometry */

/* Request b brings L^q new query tokens against L^kv cached keys/values, the
 * new tokens last ([V2] Sec.3.4 and Alg.1 inputs: lengths (L_b^q, L_b^kv)):
 * query i sits at absolute position L^kv - L^q + i, and attends causally to
 * the keys at positions 0 .. L^kv - L^q + i. L^kv = L^q is a plain prefill;
 * L^kv > L^q is a chunk of a chunked prefill after a cached prefix. */
static int q_len(const orc_problem *p, int b) { return p->cu_seqlens[b + 1] - p->cu_seqlens[b]; }
static int kv_len(const orc_problem *p, int b) { return p->seqlens_kv ? p->seqlens_kv[b] : q_len(p, b); }
static int q_shift(const orc_problem *p, int b) { return kv_len(p, b) - q_len(p, b); }
static int group(const orc_problem *p) { return p->hq / p->hkv; }
int orc_req_blocks(const orc_problem *p, int b) { return (kv_len(p, b) + p->block - 1) / p->block; }

/* Packed rows ([V2] Eq.12-13) are numbered by absolute position,
 * r = g pos + (head mod g), and tiled 128 at a time from r = 0, so every tile
 * lies inside one block. The tiles of request b under one KV head are those
 * holding one of its query rows r in [g (L^kv - L^q), g L^kv); local tile t is
 * absolute tile first_tile + t. Without a prefix this is the usual tiling from
 * the request's first row. */
static long first_tile(const orc_problem *p, int b) { return (long)group(p) * q_shift(p, b) / p->tile_rows; }
int orc_req_tiles(const orc_problem *p, int b) {
    if (q_len(p, b) <= 0) return 0;
    long end = ((long)group(p) * kv_len(p, b) + p->tile_rows - 1) / p->tile_rows;
    return (int)(end - first_tile(p, b));
}

/* Absolute packed rows [*r0, *r1) of local tile t of request b that are query rows. */
static void tile_rows(const orc_problem *p, int b, int t, long *r0, long *r1) {
    long g = group(p), lo = (first_tile(p, b) + t) * p->tile_rows, hi = lo + p->tile_rows;
    if (lo < g * q_shift(p, b)) lo = g * q_shift(p, b);
    if (hi > g * kv_len(p, b)) hi = g * kv_len(p, b);
    *r0 = lo;
    *r1 = hi;
}

/* Diagonal block of local tile t of request b: the block holding the tile's
 * positions, pos(r) = floor(r / g) ([V2] Eq.13). */
int orc_tile_diag(const orc_problem *p, int b, int t) {
    long first_row = (first_tile(p, b) + t) * p->tile_rows;
    return (int)((first_row / group(p)) / p->block);
}

/* Element offset of key/value token j of request b, KV head h, through the
 * page table: addr(b, j) = page_table[b, floor(j/p)] * p + (j mod p)
 * ([V2] Sec.3.3 "Paged and Variable-Length Execution", Eq.22). */
static size_t kv_offset(const orc_problem *p, int b, int j, int h) {
    int32_t page = p->page_table[(size_t)b * p->pt_stride + j / p->page_size];
    size_t slot = (size_t)page * p->page_size + (size_t)(j % p->page_size);
    return (slot * p->hkv + h) * p->d;
}

/* Element offset of absolute packed row r of request b under KV head h:
 * pos(r) = floor(r/g), head(r) = h*g + (r mod g) ([V2] Eq.12-13); the query of
 * position pos is token cu_seqlens[b] + pos - (L^kv - L^q) of q. */
static size_t q_offset(const orc_problem *p, int b, long r, int h) {
    int g = group(p);
    long pos = r / g;
    int head = h * g + (int)(r % g);
    return ((size_t)(p->cu_seqlens[b] + pos - q_shift(p, b)) * p->hq + head) * p->d;
}

/* Checks the description and every page id a request can touch. */
int orc_validate(const orc_problem *p) {
    if (p->batch < 0 || p->hq <= 0 || p->hkv <= 0 || p->hq % p->hkv) return ORC_EINVAL;
    if (p->d <= 0 || p->block <= 0 || p->page_size <= 0 || p->tile_rows <= 0) return ORC_EINVAL;
    /* every tile must lie inside one block: (tile_rows / g) divides block */
    if (p->tile_rows % group(p)) return ORC_EINVAL;
    if (p->block % (p->tile_rows / group(p))) return ORC_EINVAL;
    for (int b = 0; b < p->batch; ++b) {
        int L = kv_len(p, b);
        if (q_len(p, b) < 0 || L < q_len(p, b)) return ORC_EINVAL;
        int npg = (L + p->page_size - 1) / p->page_size;
        if (npg > p->pt_stride) return ORC_EINVAL;
        for (int i = 0; i < npg; ++i) {
            int32_t pg = p->page_table[(size_t)b * p->pt_stride + i];
            if (pg < 0 || pg >= p->num_pages) return ORC_EPAGE;
        }
    }
    return ORC_OK;
}

/* ---------------------------------------------------------------- pooling */

/* Block means of one (request, KV head) over all L^kv keys ([V2] Sec.3.2 Eq.5):
 *   kbar_J = (1/|B_J|) sum_{i in B_J} k_i,  vbar_J = (1/|B_J|) sum_{i in B_J} v_i,
 * with |B_J| = min(B, L^kv - J*B) for the ragged last block. FP8 inputs are
 * descaled before pooling ([V2] Alg.1 step 2). Outputs are [nb, d] and [nb]. */
int orc_pool(const orc_problem *p, int b, int h, double *kbar, double *vbar, int32_t *cnt) {
    int L = kv_len(p, b), B = p->block, d = p->d, nb = orc_req_blocks(p, b);
    for (int J = 0; J < nb; ++J) {
        int n = L - J * B < B ? L - J * B : B;
        double *kb = kbar + (size_t)J * d, *vb = vbar + (size_t)J * d;
        for (int c = 0; c < d; ++c) kb[c] = vb[c] = 0.0;
        for (int j = J * B; j < J * B + n; ++j) {
            size_t off = kv_offset(p, b, j, h);
            for (int c = 0; c < d; ++c) {
                kb[c] += elem(p, p->k_pages, off + c, p->c_k);
                vb[c] += elem(p, p->v_pages, off + c, p->c_v);
            }
        }
        for (int c = 0; c < d; ++c) {
            kb[c] /= n;
            vb[c] /= n;
        }
        cnt[J] = n;
    }
    return ORC_OK;
}

/* ---------------------------------------------------------------- scoring */

/* Block energies of packed tile t of (b, h) against the pooled keys
 * ([V2] Sec.3.3 "Single-Pass Score and Selection", Eq.19, which equals the
 * rescaled numerator of Eq.1-2 up to one common factor):
 *   s_rJ = q_r . kbar_J / sqrt(d)       for the tile's rows r, blocks J <= D
 *   M    = max_{r,J} s_rJ
 *   E_J  = sum_r exp(s_rJ - M).
 * E must hold D+1 entries. Returns D (the diagonal block) or a negative code. */
int orc_energies(const orc_problem *p, const double *kbar, long kstride, int b, int h, int t, double *E,
                 double *M_out) {
    int d = p->d;
    long r0, r1;
    tile_rows(p, b, t, &r0, &r1);
    int D = orc_tile_diag(p, b, t);
    long nr = r1 - r0;
    double *s = (double *)malloc(sizeof(double) * (size_t)nr * (size_t)(D + 1));
    double *q = (double *)malloc(sizeof(double) * (size_t)d);
    if (!s || !q) {
        free(s);
        free(q);
        return ORC_ENOMEM;
    }
    double inv_sqrt_d = 1.0 / sqrt((double)d);
    double M = -INFINITY;
    for (long r = r0; r < r1; ++r) {
        size_t qo = q_offset(p, b, r, h);
        for (int c = 0; c < d; ++c) q[c] = elem(p, p->q, qo + c, p->c_q);
        for (int J = 0; J <= D; ++J) {
            double acc = 0.0;
            const double *kb = kbar + (size_t)J * kstride;
            for (int c = 0; c < d; ++c) acc += q[c] * kb[c];
            double v = acc * inv_sqrt_d;
            s[(r - r0) * (D + 1) + J] = v;
            if (v > M) M = v;
        }
    }
    for (int J = 0; J <= D; ++J) {
        double e = 0.0;
        for (long r = 0; r < nr; ++r) e += exp(s[r * (D + 1) + J] - M);
        E[J] = e;
    }
    if (M_out) *M_out = M;
    free(s);
    free(q);
    return D;
}

/* -------------------------------------------------------------- selection */

/* Max-based dynamic threshold with forced blocks ([V2] Sec.3.1 Eq.3, Sec.3.3
 * Eq.20, Alg.1 step 4):
 *   thr = alpha * max_{J <= D} E_J
 *   J in S  <=>  E_J >= thr  or  J < sink  or  D - window <= J < D  or  J == D.
 * near[J] flags non-forced blocks with |E_J - thr| <= 1e-3 * thr, whose
 * decision a lower-precision implementation may legitimately flip.
 * Returns |S|. */
int orc_select(const double *E, int D, double alpha, int sink, int window, uint8_t *sel, uint8_t *near) {
    double emax = 0.0;
    for (int J = 0; J <= D; ++J)
        if (E[J] > emax) emax = E[J];
    double thr = alpha * emax;
    int n = 0;
    for (int J = 0; J <= D; ++J) {
        int forced = (J < sink) || (J >= D - window && J < D) || (J == D);
        sel[J] = (uint8_t)(forced || E[J] >= thr);
        if (near) near[J] = (uint8_t)(!forced && fabs(E[J] - thr) <= 1e-3 * thr);
        n += sel[J];
    }
    return n;
}

/* -------------------------------------------------------------- attention */

#define ORC_CORRECTION 1 /* add mean-correction terms for pruned blocks */
#define ORC_DENSE 2      /* ignore `sel`: every causal block is exact */
#define ORC_EQ15 4       /* E4M3 problems: quantised probabilities of Eq.15 (below) */

/* [V2] Sec.3.3 "FP8 Execution", Eq.15, taken literally: the online softmax
 * runs over the iterations of Eq.17 (the selected blocks J = D .. 0 in
 * descending order, each one iteration; then, by Alg.1 step 9, the correction
 * terms appended as chunks of 128 consecutive blocks, chunk c covering blocks
 * 128c .. 128c + 127, in descending order). m is the running row maximum after
 * each iteration; when it grows, the running numerator and denominator are
 * multiplied by e^{m_old - m}; then every term of the iteration adds
 * P~ = e4m3(2^8 e^{s - m}) to the denominator and P~ v to the numerator. The
 * 2^8 offset leaves O unchanged and is taken out of the LSE. The means enter
 * as the tensor cores read them (reading of the design notes): the mean of
 * the block's E4M3 codes, kbar / c_k (exactly: sums of E4M3 values are exact
 * in fp64, and a full block divides by 128), rounded to E4M3, times c_k; the
 * same for the values with c_v. */
static void eq15_step(const double *s, const double *const *v, int n, int d, double *m, double *l, double *o) {
    double mi = *m;
    for (int i = 0; i < n; ++i)
        if (s[i] > mi) mi = s[i];
    if (mi > *m) {
        double f = *m == -INFINITY ? 0.0 : exp(*m - mi);
        *l *= f;
        for (int c = 0; c < d; ++c) o[c] *= f;
        *m = mi;
    }
    for (int i = 0; i < n; ++i) {
        double w = orc_round_e4m3(256.0 * exp(s[i] - *m));
        *l += w;
        for (int c = 0; c < d; ++c) o[c] += w * v[i][c];
    }
}

static int attend_tile_eq15(const orc_problem *p, const int32_t *cnt, int b, int h, int t, const uint8_t *sel,
                            int flags, double *O, double *lse) {
    int g = group(p), d = p->d, B = p->block, L = kv_len(p, b);
    long r0, r1;
    tile_rows(p, b, t, &r0, &r1);
    long row_base = (first_tile(p, b) + t) * p->tile_rows;
    int D = orc_tile_diag(p, b, t);
    double inv_sqrt_d = 1.0 / sqrt((double)d);
    /* one iteration holds at most B keys or B means */
    double *s = (double *)malloc(sizeof(double) * (size_t)B);
    const double **v = (const double **)malloc(sizeof(double *) * (size_t)B);
    double *vals = (double *)malloc(sizeof(double) * (size_t)B * d);   /* values of exact keys */
    double *kop = (double *)malloc(sizeof(double) * (size_t)(D + 1) * d); /* operand-format means */
    double *vop = (double *)malloc(sizeof(double) * (size_t)(D + 1) * d);
    double *q = (double *)malloc(sizeof(double) * (size_t)d);
    int rc = ORC_OK;
    if (!s || !v || !vals || !kop || !vop || !q) {
        rc = ORC_ENOMEM;
        goto done;
    }
    for (int J = 0; J < D; ++J) { /* the correction blocks are full and lie below the diagonal */
        if (sel[J] || !(flags & ORC_CORRECTION) || (flags & ORC_DENSE)) continue;
        double *kj = kop + (size_t)J * d, *vj = vop + (size_t)J * d;
        for (int c = 0; c < d; ++c) kj[c] = vj[c] = 0.0;
        for (int j = J * B; j < (J + 1) * B; ++j) {
            size_t ko = kv_offset(p, b, j, h);
            for (int c = 0; c < d; ++c) {
                kj[c] += elem(p, p->k_pages, ko + c, 1.0);
                vj[c] += elem(p, p->v_pages, ko + c, 1.0);
            }
        }
        for (int c = 0; c < d; ++c) {
            kj[c] = p->c_k * orc_round_e4m3(kj[c] / cnt[J]);
            vj[c] = p->c_v * orc_round_e4m3(vj[c] / cnt[J]);
        }
    }
    memset(O, 0, sizeof(double) * (size_t)p->tile_rows * d);
    for (int i = 0; i < p->tile_rows; ++i) lse[i] = 0.0;
    for (long r = r0; r < r1; ++r) {
        long pos = r / g;
        size_t qo = q_offset(p, b, r, h);
        for (int c = 0; c < d; ++c) q[c] = elem(p, p->q, qo + c, p->c_q);
        double m = -INFINITY, l = 0.0;
        double *o = O + (size_t)(r - row_base) * d;
        for (int J = D; J >= 0; --J) {
            if (!((flags & ORC_DENSE) || sel[J])) continue;
            int n = 0;
            int jend = (J + 1) * B < L ? (J + 1) * B : L;
            for (int j = J * B; j < jend && j <= pos; ++j, ++n) {
                size_t ko = kv_offset(p, b, j, h);
                double acc = 0.0;
                for (int c = 0; c < d; ++c) acc += q[c] * elem(p, p->k_pages, ko + c, p->c_k);
                s[n] = acc * inv_sqrt_d;
                for (int c = 0; c < d; ++c) vals[(size_t)n * d + c] = elem(p, p->v_pages, ko + c, p->c_v);
                v[n] = vals + (size_t)n * d;
            }
            eq15_step(s, v, n, d, &m, &l, o);
        }
        if ((flags & ORC_CORRECTION) && !(flags & ORC_DENSE) && D > 0) {
            for (int ch = (D - 1) / B; ch >= 0; --ch) {
                int n = 0;
                for (int J = ch * B; J < (ch + 1) * B && J < D; ++J) {
                    if (sel[J]) continue;
                    const double *kb = kop + (size_t)J * d;
                    double acc = 0.0;
                    for (int c = 0; c < d; ++c) acc += q[c] * kb[c];
                    s[n] = acc * inv_sqrt_d + log((double)cnt[J]);
                    v[n++] = vop + (size_t)J * d;
                }
                if (n) eq15_step(s, v, n, d, &m, &l, o);
            }
        }
        for (int c = 0; c < d; ++c) o[c] /= l;
        lse[r - row_base] = m + log(l) - log(256.0);
    }
done:
    free(s);
    free(v);
    free(vals);
    free(kop);
    free(vop);
    free(q);
    return rc;
}

/* Output of packed tile t of (b, h) given its selected set sel[0..D]
 * ([V2] Sec.3.2 Eq.6; Eq.4 when the correction is off). For each row r at
 * position pos and head hq:
 *   exact terms       (q.k_j/sqrt(d), v_j)               j in B_J, J in S, j <= pos
 *   correction terms  (q.kbar_J/sqrt(d) + ln|B_J|, vbar_J) J in C = {J < D} \ S
 *   O = sum e^{s-m} v / sum e^{s-m},  LSE = m + ln sum e^{s-m},  m = max s.
 * O is [tile_rows, d] and lse is [tile_rows], row i holding absolute packed
 * row 128 (first tile + t) + i; rows that are not query rows stay 0. */
int orc_attend_tile(const orc_problem *p, const double *kbar, const double *vbar, long kstride, const int32_t *cnt,
                    int b, int h, int t, const uint8_t *sel, int flags, double *O, double *lse) {
    if (flags & ORC_EQ15) {
        if (p->dtype != 1) return ORC_EINVAL;
        return attend_tile_eq15(p, cnt, b, h, t, sel, flags, O, lse);
    }
    int g = group(p), d = p->d, B = p->block, L = kv_len(p, b);
    long r0, r1;
    tile_rows(p, b, t, &r0, &r1);
    long row_base = (first_tile(p, b) + t) * p->tile_rows; /* absolute row of the tile's row 0 */
    int D = orc_tile_diag(p, b, t);
    int nb = orc_req_blocks(p, b);
    size_t maxterms = (size_t)(D + 1) * B + (size_t)nb;
    double *s = (double *)malloc(sizeof(double) * maxterms);
    int32_t *who = (int32_t *)malloc(sizeof(int32_t) * maxterms); /* token j, or -1-J for a mean */
    double *q = (double *)malloc(sizeof(double) * (size_t)d);
    if (!s || !who || !q) {
        free(s);
        free(who);
        free(q);
        return ORC_ENOMEM;
    }
    double inv_sqrt_d = 1.0 / sqrt((double)d);
    memset(O, 0, sizeof(double) * (size_t)p->tile_rows * d);
    for (int i = 0; i < p->tile_rows; ++i) lse[i] = 0.0;
    for (long r = r0; r < r1; ++r) {
        long pos = r / g;
        size_t qo = q_offset(p, b, r, h);
        for (int c = 0; c < d; ++c) q[c] = elem(p, p->q, qo + c, p->c_q);
        size_t n = 0;
        for (int J = 0; J <= D; ++J) {
            int exact = (flags & ORC_DENSE) ? 1 : sel[J];
            if (exact) {
                int jend = (J + 1) * B < L ? (J + 1) * B : L;
                for (int j = J * B; j < jend && j <= pos; ++j) {
                    size_t ko = kv_offset(p, b, j, h);
                    double acc = 0.0;
                    for (int c = 0; c < d; ++c) acc += q[c] * elem(p, p->k_pages, ko + c, p->c_k);
                    s[n] = acc * inv_sqrt_d;
                    who[n++] = j;
                }
            } else if ((flags & ORC_CORRECTION) && J < D) {
                const double *kb = kbar + (size_t)J * kstride;
                double acc = 0.0;
                for (int c = 0; c < d; ++c) acc += q[c] * kb[c];
                s[n] = acc * inv_sqrt_d + log((double)cnt[J]);
                who[n++] = -1 - J;
            }
        }
        double m = -INFINITY;
        for (size_t i = 0; i < n; ++i)
            if (s[i] > m) m = s[i];
        double den = 0.0;
        double *o = O + (size_t)(r - row_base) * d;
        for (size_t i = 0; i < n; ++i) {
            double w = exp(s[i] - m);
            den += w;
            if (who[i] >= 0) {
                size_t vo = kv_offset(p, b, who[i], h);
                for (int c = 0; c < d; ++c) o[c] += w * elem(p, p->v_pages, vo + c, p->c_v);
            } else {
                const double *vb = vbar + (size_t)(-1 - who[i]) * kstride;
                for (int c = 0; c < d; ++c) o[c] += w * vb[c];
            }
        }
        for (int c = 0; c < d; ++c) o[c] /= den;
        lse[r - row_base] = m + log(den);
    }
    free(s);
    free(who);
    free(q);
    return ORC_OK;
}

/* --------------------------------------------------- whole-problem driver */

/* Segment ids run over (request b, KV head h, tile t) in that order
 * ([V2] Sec.3.3 "Index-Driven Sparse Traversal": one CSR segment per
 * (batch, head, tile), the head being the KV head under PackGQA). */
typedef struct {
    const orc_problem *p;
    const int64_t *seg_ids;  /* segments to process */
    int64_t nseg;
    const int32_t *seg_b, *seg_h, *seg_t; /* decoded segment coordinates (all segments) */
    const int64_t *blk_base;              /* first pooled row of request b */
    const double *kbar, *vbar;            /* [total_blocks, hkv, d] */
    const int32_t *cnt;                   /* [total_blocks] */
    /* selection */
    int do_select;
    double alpha;
    int sink, window;
    const int64_t *full_off;              /* [nseg_all] offset of segment's [0..D] entries */
    uint8_t *sel_full, *near_full;        /* selection / near flags over [0..D] per segment */
    double *energy_full;                  /* optional energies over [0..D] per segment */
    /* attention */
    int do_attend, flags;
    const uint8_t *sel_in;                /* selection used by attention ([0..D] per segment) */
    double *O, *lse;                      /* [nseg_listed, tile_rows, d] / [nseg_listed, tile_rows] */
    int64_t next;
    pthread_mutex_t mu;
    int err;
} orc_job;

static void *orc_worker(void *arg) {
    orc_job *job = (orc_job *)arg;
    const orc_problem *p = job->p;
    for (;;) {
        pthread_mutex_lock(&job->mu);
        int64_t i = job->next++;
        pthread_mutex_unlock(&job->mu);
        if (i >= job->nseg) break;
        int64_t sg = job->seg_ids[i];
        int b = job->seg_b[sg], h = job->seg_h[sg], t = job->seg_t[sg];
        int D = orc_tile_diag(p, b, t);
        size_t d = (size_t)p->d;
        /* pooled rows of this (b, h): row J lives at (blk_base[b] + J) * hkv + h */
        long kstride = (long)p->hkv * p->d;
        const double *kb = job->kbar + ((size_t)job->blk_base[b] * p->hkv + h) * d;
        const double *vb = job->vbar + ((size_t)job->blk_base[b] * p->hkv + h) * d;
        const int32_t *cb = job->cnt + job->blk_base[b];
        double *E = (double *)malloc(sizeof(double) * (size_t)(D + 1));
        if (!E) {
            job->err = ORC_ENOMEM;
            break;
        }
        if (job->do_select) {
            int rc = orc_energies(p, kb, kstride, b, h, t, E, NULL);
            if (rc < 0) job->err = rc;
            int64_t off = job->full_off[sg];
            orc_select(E, D, job->alpha, job->sink, job->window, job->sel_full + off, job->near_full + off);
            if (job->energy_full) memcpy(job->energy_full + off, E, sizeof(double) * (size_t)(D + 1));
        }
        if (job->do_attend) {
            const uint8_t *sel = job->sel_in ? job->sel_in + job->full_off[sg] : job->sel_full + job->full_off[sg];
            int rc = orc_attend_tile(p, kb, vb, kstride, cb, b, h, t, sel, job->flags,
                                     job->O + (size_t)i * p->tile_rows * d,
                                     job->lse + (size_t)i * p->tile_rows);
            if (rc < 0) job->err = rc;
        }
        free(E);
    }
    return NULL;
}

/* Pools every (request, KV head) into kbar/vbar [total_blocks, hkv, d] and
 * cnt [total_blocks], where request b's blocks start at row blk_base[b]. */
int orc_pool_all(const orc_problem *p, const int64_t *blk_base, double *kbar, double *vbar, int32_t *cnt) {
    int rc = orc_validate(p);
    if (rc) return rc;
    size_t d = (size_t)p->d;
    for (int b = 0; b < p->batch; ++b) {
        int nb = orc_req_blocks(p, b);
        double *kb = (double *)malloc(sizeof(double) * (size_t)(nb ? nb : 1) * d);
        double *vb = (double *)malloc(sizeof(double) * (size_t)(nb ? nb : 1) * d);
        int32_t *cb = (int32_t *)malloc(sizeof(int32_t) * (size_t)(nb ? nb : 1));
        if (!kb || !vb || !cb) {
            free(kb); free(vb); free(cb);
            return ORC_ENOMEM;
        }
        for (int h = 0; h < p->hkv; ++h) {
            orc_pool(p, b, h, kb, vb, cb);
            for (int J = 0; J < nb; ++J) {
                size_t row = (size_t)(blk_base[b] + J) * p->hkv + h;
                memcpy(kbar + row * d, kb + J * d, sizeof(double) * d);
                memcpy(vbar + row * d, vb + J * d, sizeof(double) * d);
                cnt[blk_base[b] + J] = cb[J];
            }
        }
        free(kb); free(vb); free(cb);
    }
    return ORC_OK;
}

/* Runs selection and/or attention for the listed segments on `nthreads`
 * POSIX threads. `seg_b/h/t` decode every segment id; `full_off` gives each
 * segment's offset into the per-block arrays (D+1 entries per segment).
 * With do_select, sel_full/near_full (and energy_full if non-NULL) receive the
 * decisions. With do_attend, O/lse receive [nseg, tile_rows, d]/[nseg,
 * tile_rows] for the listed segments, using sel_in if non-NULL (a selection
 * supplied by the caller, e.g. another implementation's CSR), else sel_full. */
int orc_run_segments(const orc_problem *p, const int64_t *seg_ids, int64_t nseg, const int32_t *seg_b,
                     const int32_t *seg_h, const int32_t *seg_t, const int64_t *blk_base, const double *kbar,
                     const double *vbar, const int32_t *cnt, const int64_t *full_off, int do_select, double alpha,
                     int sink, int window, uint8_t *sel_full, uint8_t *near_full, double *energy_full, int do_attend,
                     int flags, const uint8_t *sel_in, double *O, double *lse, int nthreads) {
    int rc = orc_validate(p);
    if (rc) return rc;
    orc_job job;
    memset(&job, 0, sizeof job);
    job.p = p;
    job.seg_ids = seg_ids;
    job.nseg = nseg;
    job.seg_b = seg_b;
    job.seg_h = seg_h;
    job.seg_t = seg_t;
    job.blk_base = blk_base;
    job.kbar = kbar;
    job.vbar = vbar;
    job.cnt = cnt;
    job.full_off = full_off;
    job.do_select = do_select;
    job.alpha = alpha;
    job.sink = sink;
    job.window = window;
    job.sel_full = sel_full;
    job.near_full = near_full;
    job.energy_full = energy_full;
    job.do_attend = do_attend;
    job.flags = flags;
    job.sel_in = sel_in;
    job.O = O;
    job.lse = lse;
    pthread_mutex_init(&job.mu, NULL);
    if (nthreads < 1) nthreads = 1;
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    if (!th) return ORC_ENOMEM;
    for (int i = 0; i < nthreads; ++i) pthread_create(&th[i], NULL, orc_worker, &job);
    for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
    free(th);
    pthread_mutex_destroy(&job.mu);
    return job.err;
}
