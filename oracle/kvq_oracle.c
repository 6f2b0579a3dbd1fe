/*
 * kvq_oracle.c -- plain CPU oracle for the quantized K/V cache path.
 *
 * TEST INFRASTRUCTURE ONLY (see kvq_oracle.h).  Scalar, no blocking, no
 * reordering beyond the definitions it restates.  Single-threaded, except
 * that a second build with -fopenmp runs the independent rows of the
 * decode attention on several threads (same arithmetic per row).
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -ffp-contract=off -fno-fast-math
 *        (no FMA contraction, IEEE float division and rint in the default
 *        rounding mode, which is round-to-nearest-even).
 */
#include "kvq_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* IEEE-754 binary16 (fp16) from its definition.                             */
/*                                                                           */
/* [kv-q8 PR, "Summary"]: the FP16 cache stores K/V as fp16 and the int8     */
/* cache keeps "one FP16 scale per 64 dims"; [kv-q8 PR, "What changed"]:     */
/* scale = fp16(max|x| / 127).  fp16() is read as IEEE round-to-nearest,     */
/* ties-to-even, with subnormals kept and overflow to infinity.             */
/* ------------------------------------------------------------------------ */

uint16_t kvo_fp16_from_float(float x)
{
    uint32_t bits;
    memcpy(&bits, &x, sizeof bits);
    const uint16_t sign = (bits >> 31) ? 0x8000u : 0u;

    if (isnan(x))
        return (uint16_t)(sign | 0x7e00u);
    if (isinf(x))
        return (uint16_t)(sign | 0x7c00u);

    const double a = fabs((double)x);
    /* Largest finite binary16 is 65504; the next grid point would be 65536.
     * Their midpoint 65520 ties to the even neighbour, which is 65536, i.e.
     * it overflows.  Everything at or above 65520 becomes infinity. */
    if (a >= 65520.0)
        return (uint16_t)(sign | 0x7c00u);

    /* Spacing of the binary16 grid around a: 2^-24 below the smallest normal
     * 2^-14, else 2^(e-10) for a in [2^e, 2^(e+1)). */
    double quantum;
    if (a < ldexp(1.0, -14)) {
        quantum = ldexp(1.0, -24);
    } else {
        int e2;
        (void)frexp(a, &e2); /* a in [2^(e2-1), 2^e2) */
        quantum = ldexp(1.0, (e2 - 1) - 10);
    }
    const double n = a / quantum;   /* exact: scaling by a power of two */
    const double r = nearbyint(n);  /* nearest, ties to even (default mode) */
    const double v = r * quantum;   /* the nearest binary16 value, exact   */

    if (v == 0.0)
        return sign;
    if (v < ldexp(1.0, -14)) /* subnormal: v = m * 2^-24 */
        return (uint16_t)(sign | (uint16_t)r);

    int e;
    const double f = frexp(v, &e); /* v = f * 2^e, f in [0.5, 1) */
    const uint32_t exp16 = (uint32_t)((e - 1) + 15);
    const uint32_t mant = (uint32_t)((f * 2.0 - 1.0) * 1024.0); /* exact */
    return (uint16_t)(sign | (exp16 << 10) | mant);
}

float kvo_fp16_to_float(uint16_t h)
{
    const int sign = h >> 15;
    const int e = (h >> 10) & 0x1f;
    const int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);               /* zero or subnormal */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp(1024.0 + (double)m, e - 25);   /* (1 + m/1024) 2^(e-15) */
    return (float)(sign ? -v : v);
}

void kvo_fp16_from_float_array(const float *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = kvo_fp16_from_float(x[i]);
}

void kvo_fp16_to_float_array(const uint16_t *h, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = kvo_fp16_to_float(h[i]);
}

/* All 65536 fp16 values as float, filled from kvo_fp16_to_float on first use
 * so that dequantization inside the attention loops is a lookup. */
static float g_fp16_table[65536];
static int g_fp16_table_ready = 0;

static void fp16_table_init(void)
{
    if (g_fp16_table_ready)
        return;
    for (int i = 0; i < 65536; ++i)
        g_fp16_table[i] = kvo_fp16_to_float((uint16_t)i);
    g_fp16_table_ready = 1;
}

/* ------------------------------------------------------------------------ */
/* Quantize-on-write.                                                        */
/*                                                                           */
/* [kv-q8 PR, "What changed"]: under --kv-q8 a row is quantized on write     */
/* with scale = fp16(max|x| / 127) and code = clamp(rint(x / scale), -127,   */
/* 127); [kv-q8 PR, "Summary"]: one scale per 64 dims.  The group maximum    */
/* covers the whole group before any code is formed (the same section's note */
/* on the barrier every thread must reach before the stores).                */
/*                                                                           */
/* Readings where the page gives only symbols:                               */
/*  - max|x|/127 and x/scale are IEEE fp32 divisions; x/scale divides by the */
/*    stored fp16 scale widened to fp32 (the same symbol on both sides).     */
/*  - rint rounds half to even.                                              */
/*  - a group whose scale is 0 (all zeros, or max|x|/127 below the fp16      */
/*    range) gets all-zero codes; an infinite scale gives x/inf = 0 codes.   */
/*  - NaN inputs are outside the domain; they give code 0 here.             */
/* ------------------------------------------------------------------------ */

int kvo_quantize_row_q8(const float *x, int hd, int8_t *codes, uint16_t *scales)
{
    if (hd <= 0 || hd % KVO_GROUP != 0)
        return -1;
    for (int g = 0; g < hd / KVO_GROUP; ++g) {
        const float *xg = x + (size_t)g * KVO_GROUP;
        float a = 0.0f;
        for (int i = 0; i < KVO_GROUP; ++i) {
            const float ax = fabsf(xg[i]);
            if (ax > a)
                a = ax;
        }
        const float t = a / 127.0f;
        const uint16_t s = kvo_fp16_from_float(t);
        const float sf = kvo_fp16_to_float(s);
        scales[g] = s;
        for (int i = 0; i < KVO_GROUP; ++i) {
            int c = 0;
            if (sf != 0.0f) {
                const float ratio = xg[i] / sf;
                if (ratio == ratio) { /* not NaN */
                    float rr = rintf(ratio);
                    if (rr > 127.0f)
                        rr = 127.0f;
                    if (rr < -127.0f)
                        rr = -127.0f;
                    c = (int)rr;
                }
            }
            codes[(size_t)g * KVO_GROUP + i] = (int8_t)c;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Paged addressing.                                                         */
/*                                                                           */
/* A block holds block_size consecutive cells of one sequence for every KV   */
/* head; codes and scales are separate runs ([k8v4 PR, "How"]: a block is a  */
/* list of byte runs, K codes then K scales).  Logical cell p of sequence b  */
/* is block table[b][p / block_size], slot p % block_size.                   */
/* ------------------------------------------------------------------------ */

static int64_t cell_row(const int32_t *block_table, int max_blocks_per_seq,
                        int n_blocks, int n_kv, int block_size,
                        int seq, int pos, int kvh)
{
    if (pos < 0)
        return -1;
    const int lb = pos / block_size;
    if (lb >= max_blocks_per_seq)
        return -1;
    const int32_t blk = block_table[(size_t)seq * max_blocks_per_seq + lb];
    if (blk < 0 || blk >= n_blocks)
        return -1;
    const int slot = pos % block_size;
    return ((int64_t)blk * n_kv + kvh) * block_size + slot;
}

static int check_geometry(int fmt, int n_kv, int hd, int block_size, int n_blocks)
{
    if (fmt != KVO_FMT_F16 && fmt != KVO_FMT_Q8 && fmt != KVO_FMT_K8V4)
        return -1;
    if (n_kv <= 0 || hd <= 0 || block_size <= 0 || n_blocks <= 0)
        return -1;
    if (fmt != KVO_FMT_F16 && hd % KVO_GROUP != 0)
        return -1;
    if (fmt == KVO_FMT_K8V4 && (hd & (hd - 1)) != 0) /* the rotation needs a power of two */
        return -1;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* K8V4: int8 K and rotated Q4_0 V ([k8v4 PR], "What": INT8 K + rotated Q4_0  */
/* V, 816 B/cell).  The page names the rotation but not which one: here the  */
/* Walsh-Hadamard transform (entries +-1, applied by butterflies in fp32),   */
/* which spreads a row's outliers over all its dims before 4-bit codes, and  */
/* whose inverse is itself divided by hd (a power of two, so exact).         */
/* ------------------------------------------------------------------------ */

void kvo_hadamard_f32(float *x, int n)
{
    for (int h = 1; h < n; h *= 2)
        for (int i = 0; i < n; i += 2 * h)
            for (int j = i; j < i + h; ++j) {
                const float a = x[j], b = x[j + h];
                x[j] = a + b;
                x[j + h] = a - b;
            }
}

int kvo_quantize_row_q4r(const float *x, int hd, uint8_t *codes, uint16_t *scales)
{
    if (hd <= 0 || hd % KVO_Q4_BLOCK != 0 || (hd & (hd - 1)) != 0 || hd > 4096)
        return -1;
    float y[4096];
    memcpy(y, x, sizeof(float) * (size_t)hd);
    kvo_hadamard_f32(y, hd);
    for (int b0 = 0; b0 < hd; b0 += KVO_Q4_BLOCK) {
        float m = 0.0f;
        for (int i = b0; i < b0 + KVO_Q4_BLOCK; ++i)
            if (fabsf(y[i]) > fabsf(m))
                m = y[i];
        const uint16_t d16 = kvo_fp16_from_float(m / -8.0f);
        const float d = kvo_fp16_to_float(d16);
        scales[b0 / KVO_Q4_BLOCK] = d16;
        for (int i = b0; i < b0 + KVO_Q4_BLOCK; i += 2) {
            int c[2];
            for (int e = 0; e < 2; ++e) {
                c[e] = 8;
                if (d != 0.0f) {
                    float r = rintf(y[i + e] / d);
                    if (!(r == r))
                        r = 0.0f;
                    if (r < -8.0f)
                        r = -8.0f;
                    if (r > 7.0f)
                        r = 7.0f;
                    c[e] = (int)r + 8;
                }
            }
            codes[i / 2] = (uint8_t)(c[0] | (c[1] << 4));
        }
    }
    return 0;
}

/* Store one row (one cell, one KV head) of K or V at pool row `row`. */
static int store_row(int fmt, int hd, void *data, uint16_t *scales, int64_t row,
                     const float *x, int is_v)
{
    if (fmt == KVO_FMT_K8V4 && is_v)
        return kvo_quantize_row_q4r(x, hd, (uint8_t *)data + (size_t)row * (hd / 2),
                                    scales + (size_t)row * (hd / KVO_Q4_BLOCK));
    if (fmt == KVO_FMT_F16) {
        uint16_t *dst = (uint16_t *)data + (size_t)row * hd;
        for (int d = 0; d < hd; ++d)
            dst[d] = kvo_fp16_from_float(x[d]);
        return 0;
    }
    int8_t *dst = (int8_t *)data + (size_t)row * hd;
    uint16_t *sdst = scales + (size_t)row * (hd / KVO_GROUP);
    return kvo_quantize_row_q8(x, hd, dst, sdst);
}

int kvo_append(int fmt, int n_kv, int hd, int block_size, int n_blocks,
               void *k_data, void *v_data, uint16_t *k_scales, uint16_t *v_scales,
               const float *k, const float *v, int n_tok,
               const int32_t *tok_seq, const int32_t *tok_pos,
               const int32_t *block_table, int max_blocks_per_seq)
{
    if (check_geometry(fmt, n_kv, hd, block_size, n_blocks) != 0)
        return -1;
    if (fmt != KVO_FMT_F16 && (k_scales == NULL || v_scales == NULL))
        return -2;
    for (int t = 0; t < n_tok; ++t) {
        for (int kvh = 0; kvh < n_kv; ++kvh) {
            const int64_t row = cell_row(block_table, max_blocks_per_seq, n_blocks,
                                         n_kv, block_size, tok_seq[t], tok_pos[t], kvh);
            if (row < 0)
                return -3;
            const size_t src = ((size_t)t * n_kv + kvh) * hd;
            if (store_row(fmt, hd, k_data, k_scales, row, k + src, 0) != 0)
                return -4;
            if (store_row(fmt, hd, v_data, v_scales, row, v + src, 1) != 0)
                return -4;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Dequantization: k_hat = code * scale.  A code has at most 8 significant   */
/* bits and an fp16 scale 11, so the product is exact in float and in       */
/* double.  The FP16 cache dequantizes to the stored fp16 value.             */
/* ------------------------------------------------------------------------ */

static double dequant(int fmt, int hd, const void *data, const uint16_t *scales,
                      int64_t row, int d)
{   /* K of every format, V of FP16 and int8 */
    if (fmt == KVO_FMT_F16)
        return (double)g_fp16_table[((const uint16_t *)data)[(size_t)row * hd + d]];
    const int8_t c = ((const int8_t *)data)[(size_t)row * hd + d];
    const uint16_t s = scales[(size_t)row * (hd / KVO_GROUP) + d / KVO_GROUP];
    return (double)c * (double)g_fp16_table[s];
}

/* V of any format: K8V4's V is dequantized in the rotated basis, (code - 8)
 * * d, exact in float and double; its attention output is rotated back. */
static double dequant_v(int fmt, int hd, const void *data, const uint16_t *scales,
                        int64_t row, int d)
{
    if (fmt != KVO_FMT_K8V4)
        return dequant(fmt, hd, data, scales, row, d);
    const uint8_t byte = ((const uint8_t *)data)[(size_t)row * (hd / 2) + d / 2];
    const int c = (d & 1) ? (byte >> 4) : (byte & 15);
    const uint16_t s = scales[(size_t)row * (hd / KVO_Q4_BLOCK) + d / KVO_Q4_BLOCK];
    return (double)(c - 8) * (double)g_fp16_table[s];
}

/* The inverse rotation of a K8V4 attention output row, in float64. */
static void unrotate_f64(double *o, int hd)
{
    for (int h = 1; h < hd; h *= 2)
        for (int i = 0; i < hd; i += 2 * h)
            for (int j = i; j < i + h; ++j) {
                const double a = o[j], b = o[j + h];
                o[j] = a + b;
                o[j + h] = a - b;
            }
    for (int d = 0; d < hd; ++d)
        o[d] /= (double)hd;
}

/* ------------------------------------------------------------------------ */
/* Decode attention, float64.                                                */
/*                                                                           */
/* [kv-q8 PR, "What changed" and "Extra Notes"]: the decode of the next      */
/* token reads the cache through a split-K partial kernel; the split-K      */
/* combine is an exact re-association of the plain softmax written here:    */
/*   z_c = sm_scale * sum_d q_d * k_hat_c,d        for visible cells c       */
/*   out_d = sum_c exp(z_c - max z) v_hat_c,d / sum_c exp(z_c - max z)       */
/* GQA: query head h reads KV head h / G, G = n_q / n_kv (consecutive query  */
/* heads share one KV head).  With W query tokens per sequence (a verify     */
/* window) the W queries are the last W cells already in the cache and token */
/* w sees cells [0, L - W + w].                                              */
/* ------------------------------------------------------------------------ */

/* One output row: sequence b, query token w, query head h.  z and rows are
 * scratch of at least L_b entries.  Returns 0, or -3 for a cell whose block
 * id is out of range. */
static int attend_row(int fmt, int n_kv, int hd, int block_size, int n_blocks,
                      const void *k_data, const void *v_data,
                      const uint16_t *k_scales, const uint16_t *v_scales,
                      const float *q, int W, int n_q, int G,
                      const int32_t *ctx_lens, const int32_t *block_table,
                      int max_blocks_per_seq, float sm_scale, int b, int w, int h,
                      double *out, double *z, int64_t *rows)
{
    const int L = ctx_lens[b];
    const int last = L - W + w; /* last visible cell */
    double *o = out + (((size_t)b * W + w) * n_q + h) * hd;
    const float *qv = q + (((size_t)b * W + w) * n_q + h) * hd;
    for (int d = 0; d < hd; ++d)
        o[d] = 0.0;
    if (last < 0)
        return 0;
    const int kvh = h / G;
    const int n_vis = last + 1;

    double zmax = -INFINITY;
    for (int c = 0; c < n_vis; ++c) {
        const int64_t row = cell_row(block_table, max_blocks_per_seq, n_blocks,
                                     n_kv, block_size, b, c, kvh);
        if (row < 0)
            return -3;
        rows[c] = row;
        double dot = 0.0;
        for (int d = 0; d < hd; ++d)
            dot += (double)qv[d] * dequant(fmt, hd, k_data, k_scales, row, d);
        z[c] = (double)sm_scale * dot;
        if (z[c] > zmax)
            zmax = z[c];
    }

    double den = 0.0;
    for (int c = 0; c < n_vis; ++c) {
        const double e = exp(z[c] - zmax);
        den += e;
        for (int d = 0; d < hd; ++d)
            o[d] += e * dequant_v(fmt, hd, v_data, v_scales, rows[c], d);
    }
    for (int d = 0; d < hd; ++d)
        o[d] /= den;
    if (fmt == KVO_FMT_K8V4)
        unrotate_f64(o, hd);
    return 0;
}

/* The rows are independent: a build with -fopenmp (the multi-core CPU
 * baseline) spreads them over threads; without it the pragmas are ignored
 * and the rows run in order on one thread.  Each row's arithmetic is the
 * same either way. */
int kvo_attention(int fmt, int n_kv, int hd, int block_size, int n_blocks,
                  const void *k_data, const void *v_data,
                  const uint16_t *k_scales, const uint16_t *v_scales,
                  const float *q, int n_seq, int W, int n_q,
                  const int32_t *ctx_lens, const int32_t *block_table,
                  int max_blocks_per_seq, float sm_scale, double *out)
{
    if (check_geometry(fmt, n_kv, hd, block_size, n_blocks) != 0)
        return -1;
    if (n_seq <= 0 || W <= 0 || n_q <= 0 || n_q % n_kv != 0)
        return -1;
    if (fmt != KVO_FMT_F16 && (k_scales == NULL || v_scales == NULL))
        return -2;
    fp16_table_init();
    const int G = n_q / n_kv;

    int max_len = 0;
    for (int b = 0; b < n_seq; ++b)
        if (ctx_lens[b] > max_len)
            max_len = ctx_lens[b];
    const long long n_rows = (long long)n_seq * W * n_q;

    int rc = 0;
#pragma omp parallel
    {
        double *z = (double *)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
        int64_t *rows = (int64_t *)malloc(sizeof(int64_t) * (size_t)(max_len > 0 ? max_len : 1));
        int my_rc = (z == NULL || rows == NULL) ? -5 : 0;
#pragma omp for schedule(dynamic)
        for (long long i = 0; i < n_rows; ++i) {
            if (my_rc != 0)
                continue;
            const int h = (int)(i % n_q);
            const int w = (int)((i / n_q) % W);
            const int b = (int)(i / ((long long)n_q * W));
            my_rc = attend_row(fmt, n_kv, hd, block_size, n_blocks, k_data, v_data, k_scales,
                               v_scales, q, W, n_q, G, ctx_lens, block_table,
                               max_blocks_per_seq, sm_scale, b, w, h, out, z, rows);
        }
#pragma omp critical
        {
            if (my_rc != 0 && rc == 0)
                rc = my_rc;
        }
        free(z);
        free(rows);
    }
    return rc;
}

/* Threads the attention rows may use (1 unless built with -fopenmp). */
int kvo_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Ask for n threads (no effect unless built with -fopenmp). */
void kvo_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------------ */
/* FP16 compaction.                                                          */
/*                                                                           */
/* [kv-q8 PR, "What changed" and "Extra Notes"]: k_kv_f16 compacts           */
/* [kvh][ctx][HD] into the contiguous [kvh][P][HD] fp16 halves that the      */
/* prompt chunk's QK^T and PV products read; on the FP16 cache it is a pure  */
/* copy.  For the int8 cache each value is fp16(code * scale).               */
/* ------------------------------------------------------------------------ */

int kvo_compact_f16(int fmt, int n_kv, int hd, int block_size, int n_blocks,
                    const void *k_data, const void *v_data,
                    const uint16_t *k_scales, const uint16_t *v_scales,
                    const int32_t *block_table_row, int n_cells,
                    uint16_t *out_k, uint16_t *out_v)
{
    if (check_geometry(fmt, n_kv, hd, block_size, n_blocks) != 0)
        return -1;
    if (n_cells < 0)
        return -1;
    if (fmt != KVO_FMT_F16 && (k_scales == NULL || v_scales == NULL))
        return -2;
    if (hd > 4096)
        return -1;
    fp16_table_init();
    const int max_blocks = (n_cells + block_size - 1) / block_size;
    for (int kvh = 0; kvh < n_kv; ++kvh) {
        for (int p = 0; p < n_cells; ++p) {
            const int64_t row = cell_row(block_table_row, max_blocks, n_blocks, n_kv,
                                         block_size, 0, p, kvh);
            if (row < 0)
                return -3;
            uint16_t *dk = out_k + ((size_t)kvh * n_cells + p) * hd;
            uint16_t *dv = out_v + ((size_t)kvh * n_cells + p) * hd;
            for (int d = 0; d < hd; ++d) {
                if (fmt == KVO_FMT_F16) {
                    dk[d] = ((const uint16_t *)k_data)[(size_t)row * hd + d];
                    dv[d] = ((const uint16_t *)v_data)[(size_t)row * hd + d];
                } else {
                    dk[d] = kvo_fp16_from_float(
                        (float)dequant(fmt, hd, k_data, k_scales, row, d));
                    if (fmt == KVO_FMT_Q8)
                        dv[d] = kvo_fp16_from_float(
                            (float)dequant(fmt, hd, v_data, v_scales, row, d));
                }
            }
            if (fmt == KVO_FMT_K8V4) {
                /* V rotated back in fp32 (the transform's butterflies, then
                 * / hd, a power of two) and rounded to fp16 */
                float w[4096];
                for (int d = 0; d < hd; ++d)
                    w[d] = (float)dequant_v(fmt, hd, v_data, v_scales, row, d);
                kvo_hadamard_f32(w, hd);
                for (int d = 0; d < hd; ++d)
                    dv[d] = kvo_fp16_from_float(w[d] / (float)hd);
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Prompt-chunk attention over the fp16 staging.                             */
/*                                                                           */
/* [kv-q8 PR, "Extra Notes"]: the prompt chunk's Q K^T and P V products read  */
/* the contiguous [kvh][P][HD] fp16 halves k_kv_f16 writes.  The chunk's      */
/* tokens are the sequence's last T cells (appended before the attention),   */
/* each attending causally to every cell up to its own position.  Written    */
/* out as the softmax definition, float64, like kvo_attention.                */
/* ------------------------------------------------------------------------ */

int kvo_chunk_attention(int n_kv, int P, int hd, const uint16_t *k16, const uint16_t *v16,
                        const float *q, int T, int n_q, float sm_scale, double *out)
{
    if (n_kv <= 0 || P <= 0 || hd <= 0 || T <= 0 || T > P || n_q <= 0 || n_q % n_kv != 0)
        return -1;
    fp16_table_init();
    const int G = n_q / n_kv;
    double *z = (double *)malloc(sizeof(double) * (size_t)P);
    if (z == NULL)
        return -5;
    for (int t = 0; t < T; ++t) {
        const int last = P - T + t; /* last visible cell */
        for (int h = 0; h < n_q; ++h) {
            const int src_head = h / G; /* the KV head query head h reads */
            const float *qv = q + ((size_t)t * n_q + h) * hd;
            double *o = out + ((size_t)t * n_q + h) * hd;
            double zmax = -INFINITY;
            for (int c = 0; c <= last; ++c) {
                const uint16_t *kr = k16 + ((size_t)src_head * P + c) * hd;
                double dot = 0.0;
                for (int d = 0; d < hd; ++d)
                    dot += (double)qv[d] * (double)g_fp16_table[kr[d]];
                z[c] = dot * (double)sm_scale;
                if (z[c] > zmax)
                    zmax = z[c];
            }
            for (int d = 0; d < hd; ++d)
                o[d] = 0.0;
            double den = 0.0;
            for (int c = 0; c <= last; ++c) {
                const double e = exp(z[c] - zmax);
                const uint16_t *vr = v16 + ((size_t)src_head * P + c) * hd;
                den += e;
                for (int d = 0; d < hd; ++d)
                    o[d] += e * (double)g_fp16_table[vr[d]];
            }
            for (int d = 0; d < hd; ++d)
                o[d] = o[d] / den;
        }
    }
    free(z);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Persistence: gather a sequence's cells out of the pool and scatter them   */
/* back ([Path F v3], "Scope": the saved body is the used cells' K/V bytes   */
/* followed by their scales, token-major; [k8v4 PR, "How"]: a block's runs   */
/* are its codes, then its scales).  Int8 codes never move without their     */
/* scales ([Path F v3], "Why": int8 bytes without scales hydrate to garbage). */
/* ------------------------------------------------------------------------ */

static int64_t seq_row(const int32_t *block_table_row, int n_blocks, int n_kv, int block_size,
                       int pos, int kvh)
{
    const int32_t blk = block_table_row[pos / block_size];
    if (blk < 0 || blk >= n_blocks)
        return -1;
    return ((int64_t)blk * n_kv + kvh) * block_size + pos % block_size;
}

/* Bytes of one K or V row and fp16 scales per row, per format. */
static void row_sizes(int fmt, int hd, size_t *k_b, size_t *v_b, int *k_ng, int *v_ng)
{
    *k_b = fmt == KVO_FMT_F16 ? (size_t)hd * 2 : (size_t)hd;
    *v_b = fmt == KVO_FMT_F16 ? (size_t)hd * 2 : fmt == KVO_FMT_Q8 ? (size_t)hd : (size_t)hd / 2;
    *k_ng = fmt == KVO_FMT_F16 ? 0 : hd / KVO_GROUP;
    *v_ng = fmt == KVO_FMT_F16 ? 0 : fmt == KVO_FMT_Q8 ? hd / KVO_GROUP : hd / KVO_Q4_BLOCK;
}

int kvo_gather_cells(int fmt, int n_kv, int hd, int block_size, int n_blocks,
                     const void *k_data, const void *v_data,
                     const uint16_t *k_scales, const uint16_t *v_scales,
                     const int32_t *block_table_row, int n_cells,
                     void *codes_k, void *codes_v, uint16_t *scales_k, uint16_t *scales_v)
{
    if (check_geometry(fmt, n_kv, hd, block_size, n_blocks) != 0 || n_cells < 0)
        return -1;
    if (fmt != KVO_FMT_F16 && (k_scales == NULL || v_scales == NULL || scales_k == NULL ||
                               scales_v == NULL))
        return -2;
    size_t kb, vb;
    int kng, vng;
    row_sizes(fmt, hd, &kb, &vb, &kng, &vng);
    for (int p = 0; p < n_cells; ++p) {
        for (int kvh = 0; kvh < n_kv; ++kvh) {
            const int64_t row = seq_row(block_table_row, n_blocks, n_kv, block_size, p, kvh);
            if (row < 0)
                return -3;
            const size_t dst = (size_t)p * n_kv + kvh;
            memcpy((char *)codes_k + dst * kb, (const char *)k_data + (size_t)row * kb, kb);
            memcpy((char *)codes_v + dst * vb, (const char *)v_data + (size_t)row * vb, vb);
            for (int gi = 0; gi < kng; ++gi)
                scales_k[dst * kng + gi] = k_scales[(size_t)row * kng + gi];
            for (int gi = 0; gi < vng; ++gi)
                scales_v[dst * vng + gi] = v_scales[(size_t)row * vng + gi];
        }
    }
    return 0;
}

int kvo_scatter_cells(int fmt, int n_kv, int hd, int block_size, int n_blocks,
                      void *k_data, void *v_data, uint16_t *k_scales, uint16_t *v_scales,
                      const int32_t *block_table_row, int n_cells,
                      const void *codes_k, const void *codes_v,
                      const uint16_t *scales_k, const uint16_t *scales_v)
{
    if (check_geometry(fmt, n_kv, hd, block_size, n_blocks) != 0 || n_cells < 0)
        return -1;
    if (fmt != KVO_FMT_F16 && (k_scales == NULL || v_scales == NULL || scales_k == NULL ||
                               scales_v == NULL))
        return -2;
    size_t kb, vb;
    int kng, vng;
    row_sizes(fmt, hd, &kb, &vb, &kng, &vng);
    for (int p = 0; p < n_cells; ++p) {
        for (int kvh = 0; kvh < n_kv; ++kvh) {
            const int64_t row = seq_row(block_table_row, n_blocks, n_kv, block_size, p, kvh);
            if (row < 0)
                return -3;
            const size_t src = (size_t)p * n_kv + kvh;
            memcpy((char *)k_data + (size_t)row * kb, (const char *)codes_k + src * kb, kb);
            memcpy((char *)v_data + (size_t)row * vb, (const char *)codes_v + src * vb, vb);
            for (int gi = 0; gi < kng; ++gi)
                k_scales[(size_t)row * kng + gi] = scales_k[src * kng + gi];
            for (int gi = 0; gi < vng; ++gi)
                v_scales[(size_t)row * vng + gi] = scales_v[src * vng + gi];
        }
    }
    return 0;
}
