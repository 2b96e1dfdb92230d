/*
 * mla_oracle.c -- plain fp64 CPU oracle for absorbed MLA decode over a paged latent cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or call this file:
 * only the tests, the package smoke check and the benchmark's CPU-baseline leg use it.  It
 * shares no code, header, table or constant generator with the CUDA library.
 *
 * Sources (web pages; section / figure named in each function):
 *   [KV]  "DeepSeek's KV Cache: From 3.9 MB to 890 B per Token" (ai-systems-engineering.com)
 *   [MLA] "What attention stores, and what DeepSeek changed" (yashdatta.dev)
 *   [SKV] "Shared KV Memory: From Transformers to DeepSeek" (nilsonchapagain.com.np)
 *   [OCP] OCP 8-bit Floating Point Specification (OFP8), format E4M3 -- the FP8 code the
 *         [KV] page's "Calculating V3.2's KV cache" section stores C^KV in.
 *
 * Every floating-point step is done in double precision.  Inputs are bf16 bit patterns
 * (uint16) and fp32 scales, widened exactly; the FP8 encoder works on fp32 as the cache
 * format prescribes.  Nothing is blocked, fused or reordered beyond the plain definitions.
 *
 * Parity status: every function is pinned by a test under tests/ (worked example, expanded
 * brute force, closed forms, codec properties, special cases); none is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_DC 512      /* latent width d_c of C^KV  ([KV] Fig. 3, "Shared KV path")      */
#define ORACLE_DR 64       /* rotary key width d_R of K^R ([KV] Fig. 3, "Shared rotary key") */
#define ORACLE_DK (ORACLE_DC + ORACLE_DR)
#define ORACLE_PAGE 64     /* tokens per cache page (paged-pool layout of this library)     */
#define ORACLE_FP8_GROUP 128 /* one fp32 scale per 128 latent dims ([KV] "Calculating V3.2") */

enum { ORACLE_BF16 = 0, ORACLE_FP8_MIXED = 1 };

/* ---------------------------------------------------------------------------------------- */
/* Scalar codecs                                                                             */
/* ---------------------------------------------------------------------------------------- */

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
double oracle_bf16_to_f64(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* [OCP] E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits, no infinities,
 * S.1111.111 is NaN.  Normal: 2^(E-7) * (1 + M/8) for E in 1..15; subnormal (E = 0):
 * 2^-6 * M/8.  Decoding is exact in double. */
double oracle_e4m3_decode(uint8_t code) {
    int s = (code >> 7) & 1;
    int e = (code >> 3) & 15;
    int m = code & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);
    else        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* [OCP] E4M3 encoding of an fp32 value, round-to-nearest-even, saturating to the largest
 * finite magnitude (448) instead of producing NaN ("satfinite").  Written from the
 * definition: the non-negative finite codes 0x00..0x7E are strictly increasing in value,
 * so the result is the code nearest to |x|, and on an exact tie the code whose lowest
 * mantissa bit is 0 (the "even" one).  NaN input maps to the NaN code 0x7F. */
uint8_t oracle_e4m3_encode(float x) {
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0) return sign | 0x7E;
    /* binary search for the largest code lo with value(lo) <= a */
    int lo = 0, hi = 0x7E;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (oracle_e4m3_decode((uint8_t)mid) <= a) lo = mid; else hi = mid - 1;
    }
    if (lo == 0x7E) return sign | 0x7E;
    double vlo = oracle_e4m3_decode((uint8_t)lo);
    double vhi = oracle_e4m3_decode((uint8_t)(lo + 1));
    int code;
    if (a - vlo < vhi - a) code = lo;
    else if (a - vlo > vhi - a) code = lo + 1;
    else code = (lo & 1) ? lo + 1 : lo;   /* tie: even mantissa */
    return sign | (uint8_t)code;
}

/* Bulk wrappers for the exhaustive codec sweep in the tests. */
void oracle_e4m3_encode_array(const float* x, uint8_t* codes, int64_t n, int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static)
#endif
    for (int64_t i = 0; i < n; ++i) codes[i] = oracle_e4m3_encode(x[i]);
}

/* ---------------------------------------------------------------------------------------- */
/* Attention core                                                                            */
/* ---------------------------------------------------------------------------------------- */

/* Scaled dot-product attention of one query over n keys/values ([MLA] "The four numbers
 * attention works with"; [SKV] section 1 "Attention reads a set of vectors"):
 *   s_t   = scale * (q . K_t)
 *   lse   = ln sum_t exp(s_t)          (computed as m + ln sum exp(s_t - m), m = max s_t)
 *   out   = sum_t exp(s_t - lse) * V_t
 * K rows have dk entries at stride ldk, V rows dv entries at stride ldv (V may alias K).
 * n == 0: out = 0 and lse = -inf (nothing visible).  The scores are returned when s != NULL. */
void oracle_attend(const double* q, const double* K, int64_t ldk, const double* V, int64_t ldv,
                   int64_t n, int dk, int dv, double scale, double* out, double* lse, double* s_out) {
    double* s = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    for (int j = 0; j < dv; ++j) out[j] = 0.0;
    if (n == 0) {
        *lse = -INFINITY;
        free(s);
        return;
    }
    double m = -INFINITY;
    for (int64_t t = 0; t < n; ++t) {
        double dot = 0.0;
        for (int k = 0; k < dk; ++k) dot += q[k] * K[t * ldk + k];
        s[t] = scale * dot;
        if (s[t] > m) m = s[t];
    }
    double l = 0.0;
    for (int64_t t = 0; t < n; ++t) l += exp(s[t] - m);
    double L = m + log(l);
    for (int64_t t = 0; t < n; ++t) {
        double p = exp(s[t] - L);
        for (int j = 0; j < dv; ++j) out[j] += p * V[t * ldv + j];
    }
    *lse = L;
    if (s_out) memcpy(s_out, s, sizeof(double) * (size_t)n);
    free(s);
}

/* ---------------------------------------------------------------------------------------- */
/* Cache record format                                                                       */
/* ---------------------------------------------------------------------------------------- */

/* Bytes of one token's record in one layer.
 *   BF16: (C^KV 512 + K^R 64) x 2 B = 1,152 B        ([KV] "Calculating V2's KV cache")
 *   FP8 mixed: 512 B e4m3 + 4 x 4 B fp32 scales + 64 x 2 B bf16 rope = 656 B
 *              ([KV] "Calculating V3.2's KV cache"; field order as in FlashMLA's FP8 format,
 *               listed in the page's "Cache formats used for storage", no padding). */
int64_t oracle_record_bytes(int fmt) {
    if (fmt == ORACLE_BF16) return (ORACLE_DC + ORACLE_DR) * 2;
    if (fmt == ORACLE_FP8_MIXED) return ORACLE_DC + (ORACLE_DC / ORACLE_FP8_GROUP) * 4 + ORACLE_DR * 2;
    return -1;
}

/* Write T new tokens into their slots (slot = page * 64 + row; slot < 0 skips the row).
 * BF16: the 576 bf16 values are stored as they are.
 * FP8 mixed, per 128-dim group g of the latent (the scale rule is absmax / 448, so that the
 * largest magnitude maps onto the largest finite E4M3 value):
 *     amax = max |x| (fp32),  s_g = fl32(amax / 448),  code = E4M3_RNE_satfinite(fl32(x / s_g)),
 *     amax == 0 gives s_g = 0 and all-zero codes;  the 64 rope values stay bf16.
 * Returns the number of rows whose slot is outside the pool (those rows are not written).
 * Rows are independent; with nthreads > 1 they are written by that many threads, which the
 * caller may ask for only when no two rows share a slot (the row order then cannot matter). */
int64_t oracle_cache_append(int fmt, uint8_t* pool, int64_t num_pages, const uint16_t* c_kv,
                            const uint16_t* k_rope, const int32_t* slot, int64_t T, int nthreads) {
    int64_t rb = oracle_record_bytes(fmt);
    int64_t bad = 0;
#ifdef _OPENMP
    if (nthreads > 1) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static) reduction(+ : bad) if (nthreads > 1)
#endif
    for (int64_t i = 0; i < T; ++i) {
        int64_t sl = slot[i];
        if (sl < 0) continue;
        if (sl >= num_pages * ORACLE_PAGE) { ++bad; continue; }
        uint8_t* rec = pool + sl * rb;
        const uint16_t* c = c_kv + i * ORACLE_DC;
        const uint16_t* r = k_rope + i * ORACLE_DR;
        if (fmt == ORACLE_BF16) {
            memcpy(rec, c, ORACLE_DC * 2);
            memcpy(rec + ORACLE_DC * 2, r, ORACLE_DR * 2);
        } else {
            for (int g = 0; g < ORACLE_DC / ORACLE_FP8_GROUP; ++g) {
                float amax = 0.0f;
                for (int k = 0; k < ORACLE_FP8_GROUP; ++k) {
                    float v = fabsf((float)oracle_bf16_to_f64(c[g * ORACLE_FP8_GROUP + k]));
                    if (v > amax) amax = v;
                }
                float sg = amax / 448.0f;
                for (int k = 0; k < ORACLE_FP8_GROUP; ++k) {
                    float v = (float)oracle_bf16_to_f64(c[g * ORACLE_FP8_GROUP + k]);
                    rec[g * ORACLE_FP8_GROUP + k] = (amax == 0.0f) ? 0 : oracle_e4m3_encode(v / sg);
                }
                memcpy(rec + ORACLE_DC + 4 * g, &sg, 4);
            }
            memcpy(rec + ORACLE_DC + 16, r, ORACLE_DR * 2);
        }
    }
    return bad;
}

/* Read one record back as exact doubles: c[512], kr[64].
 * FP8 mixed: c[k] = e4m3_value(code[k]) * s_{k / 128}, exact in double (at most 4 + 24
 * significant bits); multiplying by the scale restores the magnitude that the low-precision
 * codes were divided down from ([KV] "KV cache per token at a glance"). */
void oracle_read_record(int fmt, const uint8_t* pool, int64_t slot, double* c, double* kr) {
    int64_t rb = oracle_record_bytes(fmt);
    const uint8_t* rec = pool + slot * rb;
    if (fmt == ORACLE_BF16) {
        for (int k = 0; k < ORACLE_DC; ++k) {
            uint16_t b;
            memcpy(&b, rec + 2 * k, 2);
            c[k] = oracle_bf16_to_f64(b);
        }
        for (int r = 0; r < ORACLE_DR; ++r) {
            uint16_t b;
            memcpy(&b, rec + 2 * ORACLE_DC + 2 * r, 2);
            kr[r] = oracle_bf16_to_f64(b);
        }
    } else {
        float sc[ORACLE_DC / ORACLE_FP8_GROUP];
        memcpy(sc, rec + ORACLE_DC, sizeof sc);
        for (int k = 0; k < ORACLE_DC; ++k)
            c[k] = oracle_e4m3_decode(rec[k]) * (double)sc[k / ORACLE_FP8_GROUP];
        for (int r = 0; r < ORACLE_DR; ++r) {
            uint16_t b;
            memcpy(&b, rec + ORACLE_DC + 16 + 2 * r, 2);
            kr[r] = oracle_bf16_to_f64(b);
        }
    }
}

/* ---------------------------------------------------------------------------------------- */
/* Absorbed MLA decode                                                                       */
/* ---------------------------------------------------------------------------------------- */

/* Absorbed MLA decode for a list of (request b, head h) pairs.
 *
 * Per request b the visible set is every cached position t = 0 .. seq_lens[b]-1, the newest
 * token included ([KV] "The score that picks positions": "itself included"; [SKV] causal
 * mask M_tj = 0 for j <= t).  With topk_idx != NULL it is instead the listed entries
 * topk_idx[b][j] with 0 <= idx < seq_lens[b], each taken once as listed ([KV] Fig. 10:
 * the selection mask M keeps probability only at picked positions, and the softmax
 * renormalises over them).
 *
 * Position t lives at page block_table[b][t / 64], row t % 64.  For each visible t the
 * record gives c_t (512) and k^R_t (64), and for head h
 *     s_t = scale * ( q_lat[b,h,:] . c_t + q_rope[b,h,:] . k^R_t )
 * which is the absorbed content score (Q^C_h (W^UK_h)^T) (C^KV)^T plus the rotary score
 * Q^R_h (K^R)^T, divided by sqrt(d_k + d_r) ([KV] Fig. 4 (1) and Fig. 5 (2)).  The output is
 * the absorbed value path U_h = sum_t P_t c_t ([KV] Fig. 6 (2)), i.e. attention with
 * K_t = [c_t | k^R_t] and V_t = c_t, plus lse = ln sum_t exp(s_t).
 *
 * out: double[n_pairs][512], lse: double[n_pairs].
 * Returns 0, or -1 if a visible position's page lies outside the pool or a page index is
 * negative (nothing is computed for that pair then; its lse is NaN). */
int oracle_mla_decode(int fmt, const uint8_t* pool, int64_t num_pages,
                      const uint16_t* q_lat, const uint16_t* q_rope,
                      const int32_t* block_table, int32_t max_pages, const int32_t* seq_lens,
                      const int32_t* topk_idx, int32_t topk, int32_t B, int32_t H, float scale,
                      const int32_t* pairs, int64_t n_pairs, double* out, double* lse,
                      int nthreads) {
    int rc = 0;
    (void)B;
    /* Group pairs by request so each request's K rows are gathered once. */
    for (int64_t i0 = 0; i0 < n_pairs;) {
        int32_t b = pairs[2 * i0];
        int64_t i1 = i0;
        while (i1 < n_pairs && pairs[2 * i1] == b) ++i1;

        int64_t N = seq_lens[b];
        int64_t n = 0;
        int64_t* pos = (int64_t*)malloc(sizeof(int64_t) * (size_t)((topk_idx ? topk : N) + 1));
        if (topk_idx) {
            for (int32_t j = 0; j < topk; ++j) {
                int64_t t = topk_idx[(int64_t)b * topk + j];
                if (t >= 0 && t < N) pos[n++] = t;
            }
        } else {
            for (int64_t t = 0; t < N; ++t) pos[n++] = t;
        }
        double* K = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * ORACLE_DK);
        int bad = 0;
        /* each row of K is read on its own: threads split the rows, nothing else */
#ifdef _OPENMP
        if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static) reduction(| : bad)
#endif
        for (int64_t j = 0; j < n; ++j) {
            int64_t t = pos[j];
            int64_t pg = t / ORACLE_PAGE;
            if (pg >= max_pages) { bad = 1; continue; }
            int64_t page = block_table[(int64_t)b * max_pages + pg];
            if (page < 0 || page >= num_pages) { bad = 1; continue; }
            oracle_read_record(fmt, pool, page * ORACLE_PAGE + t % ORACLE_PAGE,
                               K + j * ORACLE_DK, K + j * ORACLE_DK + ORACLE_DC);
        }
        if (bad) {
            rc = -1;
            for (int64_t i = i0; i < i1; ++i) lse[i] = NAN;
        } else {
#ifdef _OPENMP
            if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic)
#endif
            for (int64_t i = i0; i < i1; ++i) {
                int32_t h = pairs[2 * i + 1];
                double q[ORACLE_DK];
                for (int k = 0; k < ORACLE_DC; ++k)
                    q[k] = oracle_bf16_to_f64(q_lat[((int64_t)b * H + h) * ORACLE_DC + k]);
                for (int r = 0; r < ORACLE_DR; ++r)
                    q[ORACLE_DC + r] = oracle_bf16_to_f64(q_rope[((int64_t)b * H + h) * ORACLE_DR + r]);
                oracle_attend(q, K, ORACLE_DK, K, ORACLE_DK, n, ORACLE_DK, ORACLE_DC,
                              (double)scale, out + i * ORACLE_DC, lse + i, NULL);
            }
        }
        free(K);
        free(pos);
        i0 = i1;
    }
    return rc;
}

/* ---------------------------------------------------------------------------------------- */
/* Split-KV merge                                                                            */
/* ---------------------------------------------------------------------------------------- */

/* Merge S partial results of the same query over disjoint position sets.  Partial i holds the
 * normalised output o_i over its positions and lse_i = ln sum exp(s_t) over them.  Then, with
 * lse = ln sum_i exp(lse_i), the whole-set output is sum_i exp(lse_i - lse) o_i: the softmax
 * over the union renormalises each part by its share of the mass (the same renormalisation
 * [KV] Fig. 10 applies to a subset).  Partials with lse_i = -inf (no positions) contribute
 * nothing; if all are empty, out = 0 and lse = -inf. */
void oracle_combine(const float* o_part, const float* lse_part, int32_t S, int64_t D,
                    double* out, double* lse) {
    double m = -INFINITY;
    for (int32_t i = 0; i < S; ++i)
        if ((double)lse_part[i] > m) m = lse_part[i];
    for (int64_t j = 0; j < D; ++j) out[j] = 0.0;
    if (m == -INFINITY) { *lse = -INFINITY; return; }
    double l = 0.0;
    for (int32_t i = 0; i < S; ++i) l += exp((double)lse_part[i] - m);
    double L = m + log(l);
    for (int32_t i = 0; i < S; ++i) {
        double w = exp((double)lse_part[i] - L);
        if (w == 0.0) continue;
        for (int64_t j = 0; j < D; ++j) out[j] += w * (double)o_part[(int64_t)i * D + j];
    }
    *lse = L;
}

/* ---------------------------------------------------------------------------------------- */
/* Value up-projection and output projection ([KV] "Computing without expanding Key and      */
/* Value", Fig. 6)                                                                           */
/* ---------------------------------------------------------------------------------------- */

/* Fig. 6 (2), "Absorb": the decode output U_h of head h (the probability-weighted sum of the
 * cached latent rows, dc wide) is multiplied by W^UV_h, which gives head h's value output
 * Z_h = U_h W^UV_h (dv wide), and then by W^O_h, the block of dv rows of the output weight W^O
 * that belongs to head h; the heads' contributions Y_h = Z_h W^O_h add up to the layer output
 * Y (Fig. 4 (2): the heads' outputs, concatenated, times W^O).
 *   u    [B][H][dc]
 *   w_uv [H][dc][dv]   W^UV_h as in the figure: dc rows, dv columns
 *   w_o  [H*dv][D]     W^O; row h*dv + j is row j of W^O_h
 *   z    [B][H][dv]    out: Z_h
 *   y    [B][D]        out: Y = sum_h Z_h W^O_h
 * Threads (nthreads > 0) split the requests b; each output element is one plain sum. */
void oracle_value_project(const double* u, const double* w_uv, const double* w_o, int B, int H, int dc,
                          int dv, int D, double* z, double* y, int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic)
#endif
    for (int b = 0; b < B; ++b) {
        for (int h = 0; h < H; ++h)
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int k = 0; k < dc; ++k)
                    acc += u[((int64_t)b * H + h) * dc + k] * w_uv[((int64_t)h * dc + k) * dv + j];
                z[((int64_t)b * H + h) * dv + j] = acc;
            }
        for (int n = 0; n < D; ++n) {
            double acc = 0.0;
            for (int h = 0; h < H; ++h)
                for (int j = 0; j < dv; ++j)
                    acc += z[((int64_t)b * H + h) * dv + j] * w_o[((int64_t)h * dv + j) * D + n];
            y[(int64_t)b * D + n] = acc;
        }
    }
}

/* Fig. 6 (3), "Pre-merge the weights": W^UV_h and W^O_h are merged ahead of time into
 * What^O_h = W^UV_h W^O_h (dc rows, D columns).   w_hat [H][dc][D]. */
void oracle_merge_value_output(const double* w_uv, const double* w_o, int H, int dc, int dv, int D,
                               double* w_hat, int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic)
#endif
    for (int h = 0; h < H; ++h)
        for (int k = 0; k < dc; ++k)
            for (int n = 0; n < D; ++n) {
                double acc = 0.0;
                for (int j = 0; j < dv; ++j)
                    acc += w_uv[((int64_t)h * dc + k) * dv + j] * w_o[((int64_t)h * dv + j) * D + n];
                w_hat[((int64_t)h * dc + k) * D + n] = acc;
            }
}

/* Y = sum_h U_h What^O_h with the pre-merged weight (Fig. 6 (3)).  u [B][H][dc],
 * w_hat [H][dc][D], y [B][D]. */
void oracle_project_merged(const double* u, const double* w_hat, int B, int H, int dc, int D, double* y,
                           int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for collapse(2) schedule(static)
#endif
    for (int b = 0; b < B; ++b)
        for (int n = 0; n < D; ++n) {
            double acc = 0.0;
            for (int h = 0; h < H; ++h)
                for (int k = 0; k < dc; ++k)
                    acc += u[((int64_t)b * H + h) * dc + k] * w_hat[((int64_t)h * dc + k) * D + n];
            y[(int64_t)b * D + n] = acc;
        }
}

/* ---------------------------------------------------------------------------------------- */
/* Shared K = V decode over V4 / V4.1 main-KV entries ([KV] "HCA: 128 tokens into one",       */
/* Fig. 15; "Calculating V4-Flash's KV cache"; "Calculating V4.1-Flash's KV cache")          */
/* ---------------------------------------------------------------------------------------- */

#define ORACLE_E 512          /* entry width c: one entry serves as Key and Value            */
#define ORACLE_E_NOPE 448     /* V4: non-RoPE dims stored as E4M3                               */
#define ORACLE_E_ROPE 64      /* the last 64 dims carry RoPE                                    */
#define ORACLE_V4_GROUP 64    /* V4: one UE8M0 scale per 64 channels (7 scales + 1 pad byte)   */
#define ORACLE_V41_GROUP 16   /* V4.1: one E4M3 scale per 16 channels                           */
enum { ORACLE_V4_FP8 = 2, ORACLE_V41_FP4 = 3 };

/* [OCP MX] E2M1: 1 sign bit, 2 exponent bits (bias 1), 1 mantissa bit, no infinities or NaN.
 * Normal (E > 0): 2^(E-1) * (1 + M/2); subnormal (E = 0): M/2.  Magnitudes 0, 0.5, 1, 1.5, 2,
 * 3, 4, 6. */
double oracle_e2m1_decode(uint8_t code) {
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -v : v;
}

/* E2M1 of an fp32 value, round to nearest with ties to the even mantissa bit, saturating to 6.
 * The non-negative codes 0..7 increase in value, so this is the nearest-code search of the E4M3
 * encoder over eight codes. */
uint8_t oracle_e2m1_encode(float x) {
    uint8_t sign = signbit(x) ? 0x8 : 0x0;
    double a = fabs((double)x);
    if (a >= 6.0) return sign | 0x7;
    int lo = 0;
    while (lo < 7 && oracle_e2m1_decode((uint8_t)(lo + 1)) <= a) ++lo;
    if (lo == 7) return sign | 0x7;
    double vlo = oracle_e2m1_decode((uint8_t)lo), vhi = oracle_e2m1_decode((uint8_t)(lo + 1));
    int code;
    if (a - vlo < vhi - a) code = lo;
    else if (a - vlo > vhi - a) code = lo + 1;
    else code = (lo & 1) ? lo + 1 : lo;
    return sign | (uint8_t)code;
}

/* Bytes of one entry: V4 448 x 1 B (E4M3) + 64 x 2 B (bf16 RoPE) + 7 x 1 B (UE8M0) + 1 B pad =
 * 584; V4.1 512 x 0.5 B (E2M1) + 32 x 1 B (E4M3 scales) = 288. */
int64_t oracle_shared_record_bytes(int fmt) {
    if (fmt == ORACLE_V4_FP8) return ORACLE_E_NOPE + 2 * ORACLE_E_ROPE + ORACLE_E_NOPE / ORACLE_V4_GROUP + 1;
    if (fmt == ORACLE_V41_FP4) return ORACLE_E / 2 + ORACLE_E / ORACLE_V41_GROUP;
    return -1;
}

/* Where each field of slot s lives.  V4 (this library's page layout; the pages give only the
 * sizes): a 64-entry page holds all its entries' codes [64][448], then their RoPE dims [64][64]
 * bf16, then their scale bytes [64][8] (7 UE8M0 + 1 pad), so that every field starts on a 16-byte
 * boundary.  V4.1: entries one after another, [256 B of E2M1 pairs | 32 E4M3 scales]. */
static void v4_fields(const uint8_t* pool, int64_t slot, const uint8_t** codes, const uint8_t** rope,
                      const uint8_t** scales) {
    const int64_t page = slot / ORACLE_PAGE, row = slot % ORACLE_PAGE;
    const uint8_t* base = pool + page * ORACLE_PAGE * 584;
    *codes = base + row * ORACLE_E_NOPE;
    *rope = base + ORACLE_PAGE * ORACLE_E_NOPE + row * 2 * ORACLE_E_ROPE;
    *scales = base + ORACLE_PAGE * (ORACLE_E_NOPE + 2 * ORACLE_E_ROPE) + row * 8;
}

/* Write T entries (bf16 bits [T][512]) at `slot` (< 0 skips; beyond the pool: counted, not
 * written).
 * V4 ("Calculating V4-Flash's KV cache": 448 non-RoPE dims in FP8 E4M3 with one UE8M0 scale per
 * 64 channels, 64 RoPE dims in BF16): per group g of 64 non-RoPE dims, amax = max |x|; the scale
 * is the power of two 2^e with the smallest integer e such that 448 * 2^e >= amax (so that no code
 * saturates), stored as the byte e + 127 (e clamped to [-127, 127]; amax = 0 stores byte 0 and
 * zero codes); code = E4M3_RNE_satfinite(fl32(x / 2^e)).  The RoPE dims are copied, the pad byte
 * is 0.
 * V4.1 ("Calculating V4.1-Flash's KV cache": all 512 dims in FP4 E2M1, the RoPE part included,
 * one E4M3 scale per 16 channels): per group of 16 dims, s = E4M3_RNE_satfinite(fl32(amax / 6))
 * (6 is E2M1's largest magnitude); code = E2M1_RNE_satfinite(fl32(x / value(s))), all codes 0
 * when value(s) = 0.  Dims 2i and 2i + 1 share byte i, dim 2i in the low nibble. */
int64_t oracle_shared_append(int fmt, uint8_t* pool, int64_t num_pages, const uint16_t* entry,
                             const int32_t* slot, int64_t T) {
    int64_t rb = oracle_shared_record_bytes(fmt);
    int64_t bad = 0;
    for (int64_t i = 0; i < T; ++i) {
        int64_t sl = slot[i];
        if (sl < 0) continue;
        if (sl >= num_pages * ORACLE_PAGE) { ++bad; continue; }
        const uint16_t* x = entry + i * ORACLE_E;
        if (fmt == ORACLE_V4_FP8) {
            const uint8_t *c0, *r0, *s0;
            v4_fields(pool, sl, &c0, &r0, &s0);
            uint8_t* codes = (uint8_t*)c0;
            uint8_t* rope = (uint8_t*)r0;
            uint8_t* scales = (uint8_t*)s0;
            for (int g = 0; g < ORACLE_E_NOPE / ORACLE_V4_GROUP; ++g) {
                double amax = 0.0;
                for (int k = 0; k < ORACLE_V4_GROUP; ++k) {
                    double v = fabs(oracle_bf16_to_f64(x[g * ORACLE_V4_GROUP + k]));
                    if (v > amax) amax = v;
                }
                if (amax == 0.0) {
                    scales[g] = 0;
                    for (int k = 0; k < ORACLE_V4_GROUP; ++k) codes[g * ORACLE_V4_GROUP + k] = 0;
                    continue;
                }
                int e = -127;
                while (e < 127 && 448.0 * ldexp(1.0, e) < amax) ++e;
                scales[g] = (uint8_t)(e + 127);
                for (int k = 0; k < ORACLE_V4_GROUP; ++k) {
                    float v = (float)oracle_bf16_to_f64(x[g * ORACLE_V4_GROUP + k]);
                    codes[g * ORACLE_V4_GROUP + k] = oracle_e4m3_encode((float)((double)v / ldexp(1.0, e)));
                }
            }
            scales[7] = 0;
            memcpy(rope, x + ORACLE_E_NOPE, 2 * ORACLE_E_ROPE);
        } else {
            uint8_t* rec = pool + sl * rb;
            for (int g = 0; g < ORACLE_E / ORACLE_V41_GROUP; ++g) {
                float amax = 0.0f;
                for (int k = 0; k < ORACLE_V41_GROUP; ++k) {
                    float v = fabsf((float)oracle_bf16_to_f64(x[g * ORACLE_V41_GROUP + k]));
                    if (v > amax) amax = v;
                }
                uint8_t sc = oracle_e4m3_encode(amax / 6.0f);
                float sv = (float)oracle_e4m3_decode(sc);
                rec[ORACLE_E / 2 + g] = sc;
                for (int k = 0; k < ORACLE_V41_GROUP; k += 2) {
                    float v0 = (float)oracle_bf16_to_f64(x[g * ORACLE_V41_GROUP + k]);
                    float v1 = (float)oracle_bf16_to_f64(x[g * ORACLE_V41_GROUP + k + 1]);
                    uint8_t q0 = sv == 0.0f ? 0 : oracle_e2m1_encode(v0 / sv);
                    uint8_t q1 = sv == 0.0f ? 0 : oracle_e2m1_encode(v1 / sv);
                    rec[(g * ORACLE_V41_GROUP + k) / 2] = (uint8_t)(q0 | (q1 << 4));
                }
            }
        }
    }
    return bad;
}

/* One entry as exact doubles e[512]: V4 code * 2^(byte - 127) for the 448 non-RoPE dims, the
 * bf16 RoPE dims widened; V4.1 E2M1 value * E4M3 scale value. */
void oracle_shared_read(int fmt, const uint8_t* pool, int64_t slot, double* e) {
    if (fmt == ORACLE_V4_FP8) {
        const uint8_t *codes, *rope, *scales;
        v4_fields(pool, slot, &codes, &rope, &scales);
        for (int k = 0; k < ORACLE_E_NOPE; ++k)
            e[k] = oracle_e4m3_decode(codes[k]) * ldexp(1.0, (int)scales[k / ORACLE_V4_GROUP] - 127);
        for (int r = 0; r < ORACLE_E_ROPE; ++r) {
            uint16_t b;
            memcpy(&b, rope + 2 * r, 2);
            e[ORACLE_E_NOPE + r] = oracle_bf16_to_f64(b);
        }
    } else {
        const uint8_t* rec = pool + slot * oracle_shared_record_bytes(fmt);
        for (int k = 0; k < ORACLE_E; ++k) {
            uint8_t byte = rec[k / 2];
            uint8_t q = (k & 1) ? (byte >> 4) : (byte & 0xF);
            e[k] = oracle_e2m1_decode(q) * oracle_e4m3_decode(rec[ORACLE_E / 2 + k / ORACLE_V41_GROUP]);
        }
    }
}

/* Scaled dot-product attention of one query with a sink ([KV] Fig. 15 (2): the head adds
 * exp(z') to the softmax denominator, so the weights on the real entries may sum to less than 1):
 *   s_t = scale * (q . K_t);  L = sum_t exp(s_t) + exp(z');  out = sum_t (exp(s_t) / L) V_t;
 *   lse = ln L.
 * z' = -inf is no sink (plain attention).  n == 0: out = 0 and lse = z'.  Computed with
 * m = max(z', max_t s_t) subtracted inside every exponential. */
void oracle_attend_sink(const double* q, const double* K, int64_t ldk, const double* V, int64_t ldv, int64_t n,
                        int dk, int dv, double scale, double sink, double* out, double* lse) {
    double* s = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    for (int j = 0; j < dv; ++j) out[j] = 0.0;
    double m = sink;
    for (int64_t t = 0; t < n; ++t) {
        double dot = 0.0;
        for (int k = 0; k < dk; ++k) dot += q[k] * K[t * ldk + k];
        s[t] = scale * dot;
        if (s[t] > m) m = s[t];
    }
    if (m == -INFINITY) {   /* nothing visible and no sink */
        *lse = -INFINITY;
        free(s);
        return;
    }
    double l = exp(sink - m);
    for (int64_t t = 0; t < n; ++t) l += exp(s[t] - m);
    for (int64_t t = 0; t < n; ++t) {
        double p = exp(s[t] - m) / l;
        for (int j = 0; j < dv; ++j) out[j] += p * V[t * ldv + j];
    }
    *lse = m + log(l);
    free(s);
}

/* Inverse rotation of the last 64 dims of a head output by the query position ([KV] Fig. 15 (3):
 * E serves as the Value with RoPE still applied, so the output's RoPE dims are rotated back by
 * the current position t).  The rotation acts on the pairs (448 + 2i, 448 + 2i + 1), i < 32, by
 * the angle theta_i of position t, given as cos_sin[i] = cos(theta_i), cos_sin[32 + i] =
 * sin(theta_i); rotating back is rotating by -theta_i:
 *   y0 = x0 cos + x1 sin,   y1 = -x0 sin + x1 cos. */
void oracle_unrotate(double* o, const float* cos_sin) {
    for (int i = 0; i < ORACLE_E_ROPE / 2; ++i) {
        double c = cos_sin[i], sn = cos_sin[ORACLE_E_ROPE / 2 + i];
        double x0 = o[ORACLE_E_NOPE + 2 * i], x1 = o[ORACLE_E_NOPE + 2 * i + 1];
        o[ORACLE_E_NOPE + 2 * i] = x0 * c + x1 * sn;
        o[ORACLE_E_NOPE + 2 * i + 1] = -x0 * sn + x1 * c;
    }
}

/* Shared K = V decode ([KV] Fig. 15 (1)-(3)) for (request b, head h) pairs: the visible entries
 * (dense: positions 0 .. seq_lens[b]-1; with topk_idx: the listed ones, as in oracle_mla_decode)
 * serve as both Key and Value, E_t (512) read from the pool; s_t = scale * (q[b,h] . E_t); the
 * softmax adds the sink exp(sink[h]) to its denominator (sink NULL: none); the output's last 64
 * dims are rotated back by rope_cs[b] (NULL: not rotated).  lse = ln(sum_t exp(s_t) + exp(z')).
 * Returns -1 if a visible position maps outside the pool (that pair's lse is NaN). */
int oracle_shared_kv_decode(int fmt, const uint8_t* pool, int64_t num_pages, const uint16_t* q,
                            const int32_t* block_table, int32_t max_pages, const int32_t* seq_lens,
                            const int32_t* topk_idx, int32_t topk, int32_t B, int32_t H, float scale,
                            const float* sink, const float* rope_cs, const int32_t* pairs, int64_t n_pairs,
                            double* out, double* lse, int nthreads) {
    int rc = 0;
    (void)B;
    for (int64_t i0 = 0; i0 < n_pairs;) {
        int32_t b = pairs[2 * i0];
        int64_t i1 = i0;
        while (i1 < n_pairs && pairs[2 * i1] == b) ++i1;
        int64_t N = seq_lens[b], n = 0;
        int64_t* pos = (int64_t*)malloc(sizeof(int64_t) * (size_t)((topk_idx ? topk : N) + 1));
        if (topk_idx) {
            for (int32_t j = 0; j < topk; ++j) {
                int64_t t = topk_idx[(int64_t)b * topk + j];
                if (t >= 0 && t < N) pos[n++] = t;
            }
        } else {
            for (int64_t t = 0; t < N; ++t) pos[n++] = t;
        }
        double* E = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * ORACLE_E);
        int bad = 0;
#ifdef _OPENMP
        if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(static) reduction(| : bad)
#endif
        for (int64_t j = 0; j < n; ++j) {
            int64_t t = pos[j], pg = t / ORACLE_PAGE;
            if (pg >= max_pages) { bad = 1; continue; }
            int64_t page = block_table[(int64_t)b * max_pages + pg];
            if (page < 0 || page >= num_pages) { bad = 1; continue; }
            oracle_shared_read(fmt, pool, page * ORACLE_PAGE + t % ORACLE_PAGE, E + j * ORACLE_E);
        }
        if (bad) {
            rc = -1;
            for (int64_t i = i0; i < i1; ++i) lse[i] = NAN;
        } else {
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic)
#endif
            for (int64_t i = i0; i < i1; ++i) {
                int32_t h = pairs[2 * i + 1];
                double qd[ORACLE_E];
                for (int k = 0; k < ORACLE_E; ++k) qd[k] = oracle_bf16_to_f64(q[((int64_t)b * H + h) * ORACLE_E + k]);
                double z = sink ? (double)sink[h] : -INFINITY;
                oracle_attend_sink(qd, E, ORACLE_E, E, ORACLE_E, n, ORACLE_E, ORACLE_E, (double)scale, z,
                                   out + i * ORACLE_E, lse + i);
                if (rope_cs) oracle_unrotate(out + i * ORACLE_E, rope_cs + (int64_t)b * ORACLE_E_ROPE);
            }
        }
        free(E);
        free(pos);
        i0 = i1;
    }
    return rc;
}

/* ---------------------------------------------------------------------------------------- */
/* DSA lightning indexer and top-k selection                                                */
/* ([KV] "DSA: three things the indexer builds" (Fig. 8), "The score that picks positions"   */
/* (Fig. 9), "Calculating V3.2's KV cache" (search key, 132 B))                              */
/* ---------------------------------------------------------------------------------------- */

/* Index-key page of this library's pool: the 64 tokens' 128 E4M3 codes (token-major, 8,192 B)
 * followed by their 64 fp32 scales (256 B), 8,448 B per page = 64 x 132 B: a search key is 128
 * FP8 codes sharing a single fp32 scale, every dimension quantised, the rotary ones included
 * ([KV] "Calculating V3.2's KV cache").  The scale rule is the main cache's: absmax / 448. */
#define ORACLE_IDX_DIM 128
#define ORACLE_IDX_PAGE_BYTES (ORACLE_PAGE * (ORACLE_IDX_DIM + 4))

int64_t oracle_index_page_bytes(void) { return ORACLE_IDX_PAGE_BYTES; }

/* Write T search keys (bf16 bits k[T,128]) at `slot` (page * 64 + row; < 0 skipped).  Returns the
 * number of rows whose slot is outside the pool (not written). */
int64_t oracle_index_append(uint8_t* pool, int64_t num_pages, const uint16_t* k, const int32_t* slot,
                            int64_t T) {
    int64_t bad = 0;
    for (int64_t i = 0; i < T; ++i) {
        int64_t sl = slot[i];
        if (sl < 0) continue;
        if (sl >= num_pages * ORACLE_PAGE) { ++bad; continue; }
        uint8_t* page = pool + (sl / ORACLE_PAGE) * ORACLE_IDX_PAGE_BYTES;
        int64_t row = sl % ORACLE_PAGE;
        const uint16_t* x = k + i * ORACLE_IDX_DIM;
        float amax = 0.0f;
        for (int d = 0; d < ORACLE_IDX_DIM; ++d) {
            float v = fabsf((float)oracle_bf16_to_f64(x[d]));
            if (v > amax) amax = v;
        }
        float s = amax / 448.0f;
        for (int d = 0; d < ORACLE_IDX_DIM; ++d)
            page[row * ORACLE_IDX_DIM + d] = (amax == 0.0f) ? 0 : oracle_e4m3_encode((float)oracle_bf16_to_f64(x[d]) / s);
        memcpy(page + ORACLE_PAGE * ORACLE_IDX_DIM + 4 * row, &s, 4);
    }
    return bad;
}

/* The search key of one cached token as exact doubles: k[d] = e4m3_value(code[d]) * s. */
void oracle_index_read(const uint8_t* pool, int64_t slot, double* k) {
    const uint8_t* page = pool + (slot / ORACLE_PAGE) * ORACLE_IDX_PAGE_BYTES;
    int64_t row = slot % ORACLE_PAGE;
    float s;
    memcpy(&s, page + ORACLE_PAGE * ORACLE_IDX_DIM + 4 * row, 4);
    for (int d = 0; d < ORACLE_IDX_DIM; ++d) k[d] = oracle_e4m3_decode(page[row * ORACLE_IDX_DIM + d]) * (double)s;
}

/* Indexer score of one query (heads x dim, fp64) against one key (dim):
 *     I = sum_j w[j] * ReLU(q[j] . k)
 * ([KV] "The score that picks positions": per head, the query-key dot product goes through a
 * ReLU and is weighted by that head's weight; the weighted terms add up over the heads).  Written for any head count and width. */
double oracle_index_score(const double* q, const double* w, const double* k, int heads, int dim) {
    double I = 0.0;
    for (int j = 0; j < heads; ++j) {
        double dot = 0.0;
        for (int d = 0; d < dim; ++d) dot += q[(int64_t)j * dim + d] * k[d];
        I += w[j] * (dot > 0.0 ? dot : 0.0);
    }
    return I;
}

/* Scores of request b's query (q bf16 bits [B, heads, 128], w fp32 [B, heads]) at every visible
 * position t < seq_lens[b] (clamped to [0, ld]) of the paged index pool; scores[b * ld + t].
 * Positions from seq_lens[b] on are set to -inf (not visible).  Returns 1 if a visible position
 * maps outside the pool, else 0. */
int oracle_indexer_scores(const uint8_t* pool, int64_t num_pages, const uint16_t* q, const float* w,
                          int heads, const int32_t* block_table, int32_t max_pages, const int32_t* seq_lens,
                          int32_t B, int64_t ld, double* scores, int nthreads) {
    int err = 0;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic) reduction(| : err)
#endif
    for (int32_t b = 0; b < B; ++b) {
        int64_t n = seq_lens[b];
        if (n < 0) n = 0;
        if (n > ld) n = ld;
        double* qd = (double*)malloc(sizeof(double) * (size_t)heads * ORACLE_IDX_DIM);
        double* wd = (double*)malloc(sizeof(double) * (size_t)heads);
        double k[ORACLE_IDX_DIM];
        for (int64_t e = 0; e < (int64_t)heads * ORACLE_IDX_DIM; ++e)
            qd[e] = oracle_bf16_to_f64(q[(int64_t)b * heads * ORACLE_IDX_DIM + e]);
        for (int j = 0; j < heads; ++j) wd[j] = (double)w[(int64_t)b * heads + j];
        for (int64_t t = 0; t < ld; ++t) {
            if (t >= n) { scores[(int64_t)b * ld + t] = -INFINITY; continue; }
            int64_t page = block_table[(int64_t)b * max_pages + t / ORACLE_PAGE];
            if (page < 0 || page >= num_pages) { err = 1; scores[(int64_t)b * ld + t] = NAN; continue; }
            oracle_index_read(pool, page * ORACLE_PAGE + t % ORACLE_PAGE, k);
            scores[(int64_t)b * ld + t] = oracle_index_score(qd, wd, k, heads, ORACLE_IDX_DIM);
        }
        free(qd);
        free(wd);
    }
    return err;
}

/* Top-k selection of one row: among positions t < n, the K with the highest scores, a tie going
 * to the lower position; written to idx[0 .. K) in increasing position order, -1 past the
 * min(K, n) picks ([KV] "The score that picks positions": a query keeps at most 2,048 of the
 * positions it can see, those that score highest).  Plain selection: K passes
 * over the row, each taking the best position not taken yet (the tie rule is the order of the
 * comparison), then a sort of the picks. */
void oracle_topk_row(const double* scores, int64_t n, int32_t K, int32_t* idx) {
    int32_t m = (int32_t)(n < K ? n : K);
    unsigned char* taken = (unsigned char*)calloc((size_t)(n > 0 ? n : 1), 1);
    for (int32_t r = 0; r < m; ++r) {
        int64_t best = -1;
        for (int64_t t = 0; t < n; ++t) {
            if (taken[t]) continue;
            if (best < 0 || scores[t] > scores[best]) best = t;   /* strict: ties keep the lower t */
        }
        if (best >= 0) taken[best] = 1;
    }
    int32_t c = 0;
    for (int64_t t = 0; t < n; ++t)
        if (taken[t]) idx[c++] = (int32_t)t;
    for (; c < K; ++c) idx[c] = -1;
    free(taken);
}

void oracle_topk(const double* scores, int64_t ld, const int32_t* seq_lens, int32_t B, int32_t K, int32_t* idx,
                 int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic)
#endif
    for (int32_t b = 0; b < B; ++b) {
        int64_t n = seq_lens[b];
        if (n < 0) n = 0;
        if (n > ld) n = ld;
        oracle_topk_row(scores + (int64_t)b * ld, n, K, idx + (int64_t)b * K);
    }
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
