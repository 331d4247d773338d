/*
 * q4k_oracle.c -- plain, slow, obviously-correct CPU oracle for the Q4_K
 * quantized-weight projection path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or helper with the CUDA
 * path.
 *
 * What it follows:
 *  - "spec: specialized model runtimes", section "Architecture": tier T0 is the
 *    kernel tier (GEMM, quant/dequant ...); section "Kernel and portability
 *    contract", rule 1: every tuned kernel has a clear, slow reference that
 *    serves as its differential oracle.
 *  - "Layer Package Repository Spec", sections "Repository Identity" and
 *    "Manifest Schema": the weight artifact is a GGUF Q4_K ("UD-Q4_K_XL")
 *    distribution split into per-layer quantized tensors.
 *  - The pages name the Q4_K format but do not print its bytes.  The layout
 *    used here is the plain reading of "GGUF-style Q4_K" (the GGUF k-quant
 *    super-block), restated in the comments below.  Compatibility with real
 *    GGUF files is therefore parity unpinned; self-consistency is pinned by the
 *    tests (hand-built blocks, a pack/unpack round trip, exact brute force).
 *
 * Q4_K super-block (256 weights, 144 bytes, little-endian):
 *    bytes   0..1   d     (IEEE binary16)   super-block scale
 *    bytes   2..3   dmin  (IEEE binary16)   super-block min scale
 *    bytes   4..15  s[12] 8 six-bit sub-block scales sc_j and mins m_j
 *    bytes  16..143 qs[128] 256 four-bit quants
 *  Sub-block j (0..7) holds weights 32j .. 32j+31 and
 *      w = d * sc_j * q - dmin * m_j .
 *  Scale packing: for j < 4:  sc_j = s[j] & 63,  m_j = s[j+4] & 63;
 *                 for j >= 4: sc_j = (s[j+4] & 15) | ((s[j-4] >> 6) << 4),
 *                             m_j  = (s[j+4] >> 4) | ((s[j]   >> 6) << 4).
 *  Quants: value i lives in chunk c = i/64 (32 bytes, qs[32c .. 32c+31]);
 *  l = i % 32; the low nibble of qs[32c+l] is value 64c+l (sub-block 2c),
 *  the high nibble is value 64c+32+l (sub-block 2c+1).
 *
 * Arithmetic: every weight is computed exactly in fp64 (d*sc has at most 17
 * significant bits, times q at most 21; dmin*m likewise), products with the
 * activations and all sums are taken in fp64 in natural index order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define Q4K_VALUES 256
#define Q4K_BYTES 144

/* IEEE binary16 -> double, decoded from the bit fields (exact). */
double oracle_fp16_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 31;
    int frac = h & 1023;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24);               /* subnormal: frac * 2^-24 */
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + frac), expo - 25); /* (1 + frac/1024) 2^(e-15) */
    }
    return sign ? -v : v;
}

/* bfloat16 -> double, decoded from the bit fields (exact). */
double oracle_bf16_to_f64(uint16_t b) {
    int sign = (b >> 15) & 1;
    int expo = (b >> 7) & 255;
    int frac = b & 127;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -133);              /* subnormal: frac * 2^-133 */
    } else if (expo == 255) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(128 + frac), expo - 134); /* (1 + frac/128) 2^(e-127) */
    }
    return sign ? -v : v;
}

/* fp32 -> bfloat16, round to nearest, ties to even, written out explicitly:
 * keep the top 16 bits, look at the 16 dropped bits. */
uint16_t oracle_f32_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u) {          /* NaN stays NaN (quiet) */
        return (uint16_t)((u >> 16) | 0x0040u);
    }
    uint32_t kept = u >> 16;
    uint32_t dropped = u & 0xffffu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u))) {
        kept += 1u;                                  /* may carry into inf: correct */
    }
    return (uint16_t)kept;
}

/* The eight (sc_j, m_j) pairs of one super-block, from its 12 scale bytes. */
void oracle_unpack_scales(const uint8_t s[12], int sc[8], int m[8]) {
    for (int j = 0; j < 8; ++j) {
        if (j < 4) {
            sc[j] = s[j] & 63;
            m[j] = s[j + 4] & 63;
        } else {
            sc[j] = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
            m[j] = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
        }
    }
}

/* The 4-bit quant of value i (0..255) of one super-block. */
int oracle_quant(const uint8_t qs[128], int i) {
    int c = i / 64;
    int l = i % 32;
    int hi = (i % 64) >= 32;
    uint8_t byte = qs[32 * c + l];
    return hi ? (byte >> 4) : (byte & 15);
}

/* One super-block -> its 256 weights, exact, in fp64. */
void oracle_dequant_block_f64(const uint8_t *blk, double out[Q4K_VALUES]) {
    uint16_t dbits = (uint16_t)(blk[0] | (blk[1] << 8));
    uint16_t mbits = (uint16_t)(blk[2] | (blk[3] << 8));
    double d = oracle_fp16_to_f64(dbits);
    double dmin = oracle_fp16_to_f64(mbits);
    int sc[8], m[8];
    oracle_unpack_scales(blk + 4, sc, m);
    const uint8_t *qs = blk + 16;
    for (int i = 0; i < Q4K_VALUES; ++i) {
        int j = i / 32;
        int q = oracle_quant(qs, i);
        out[i] = d * sc[j] * q - dmin * m[j];
    }
}

/* Row r of an n x k Q4_K matrix (rows are contiguous runs of k/256 blocks). */
static const uint8_t *row_ptr(const uint8_t *w, int64_t k, int64_t r) {
    return w + (size_t)r * (size_t)(k / Q4K_VALUES) * Q4K_BYTES;
}

static void dequant_row_f64(const uint8_t *w, int64_t k, int64_t r, double *out) {
    const uint8_t *row = row_ptr(w, k, r);
    for (int64_t b = 0; b < k / Q4K_VALUES; ++b) {
        oracle_dequant_block_f64(row + b * Q4K_BYTES, out + b * Q4K_VALUES);
    }
}

/* Whole matrix -> exact weights (fp64), row-major n x k. */
void oracle_dequant_f64(const uint8_t *w, int64_t n, int64_t k, double *out) {
    for (int64_t r = 0; r < n; ++r) dequant_row_f64(w, k, r, out + r * k);
}

/* Whole matrix -> fp32: one round-to-nearest-even of the exact value. */
void oracle_dequant_f32(const uint8_t *w, int64_t n, int64_t k, float *out) {
    double *tmp = (double *)malloc(sizeof(double) * (size_t)k);
    for (int64_t r = 0; r < n; ++r) {
        dequant_row_f64(w, k, r, tmp);
        for (int64_t i = 0; i < k; ++i) out[r * k + i] = (float)tmp[i];
    }
    free(tmp);
}

/* Whole matrix -> bf16: the fp32 value, then round-to-nearest-even to bf16. */
void oracle_dequant_bf16(const uint8_t *w, int64_t n, int64_t k, uint16_t *out) {
    double *tmp = (double *)malloc(sizeof(double) * (size_t)k);
    for (int64_t r = 0; r < n; ++r) {
        dequant_row_f64(w, k, r, tmp);
        for (int64_t i = 0; i < k; ++i) out[r * k + i] = oracle_f32_to_bf16_rne((float)tmp[i]);
    }
    free(tmp);
}

/*
 * y[b, r] = sum_k w[r, k] * x[b, k]  (fp64, natural k order) and
 * s[b, r] = sum_k |w[r, k]| * |x[b, k]|  (the scale of the error bound),
 * for bf16 activations x (batch rows, row stride ldx elements).
 * Only the rows listed in `rows` (nrows of them) are computed when rows is not
 * NULL; outputs are then indexed [b * nrows + i].  y and s are [batch x n]
 * (or [batch x nrows]).  s may be NULL.
 */
void oracle_gemv_bf16(const uint8_t *w, int64_t n, int64_t k, const uint16_t *x, int64_t batch,
                      int64_t ldx, const int64_t *rows, int64_t nrows, double *y, double *s) {
    int64_t count = rows ? nrows : n;
    double *xd = (double *)malloc(sizeof(double) * (size_t)(batch * k));
    for (int64_t b = 0; b < batch; ++b)
        for (int64_t i = 0; i < k; ++i) xd[b * k + i] = oracle_bf16_to_f64(x[b * ldx + i]);
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t ri = 0; ri < count; ++ri) {
        int64_t r = rows ? rows[ri] : ri;
        double *wr = (double *)malloc(sizeof(double) * (size_t)k);
        dequant_row_f64(w, k, r, wr);
        for (int64_t b = 0; b < batch; ++b) {
            double acc = 0.0, mag = 0.0;
            for (int64_t i = 0; i < k; ++i) {
                acc += wr[i] * xd[b * k + i];
                mag += fabs(wr[i]) * fabs(xd[b * k + i]);
            }
            y[b * count + ri] = acc;
            if (s) s[b * count + ri] = mag;
        }
        free(wr);
    }
    free(xd);
}

/*
 * The same contraction for fp64 activations (used for the MoE down
 * projection, whose input is the fp64 hidden vector).  With use_abs != 0 the
 * weights enter as |w| (callers pass |x| to obtain sum |w||x|).
 * x is [batch x ldx], y is [batch x n].
 */
void oracle_gemv_f64(const uint8_t *w, int64_t n, int64_t k, const double *x, int64_t batch,
                     int64_t ldx, int use_abs, double *y) {
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < n; ++r) {
        double *wr = (double *)malloc(sizeof(double) * (size_t)k);
        dequant_row_f64(w, k, r, wr);
        for (int64_t b = 0; b < batch; ++b) {
            double acc = 0.0;
            for (int64_t i = 0; i < k; ++i) acc += (use_abs ? fabs(wr[i]) : wr[i]) * x[b * ldx + i];
            y[b * n + r] = acc;
        }
        free(wr);
    }
}

/*
 * Fused gate/up projection of a dense or shared-expert FFN ("Layer Package
 * Repository Spec", section "Policy Resolution": the merged shared gate/up and
 * the SwiGLU of the FFN; section "Execution Policy": merged shared gate/up):
 *     g = sum_k wg[r, k] x[b, k],  u = sum_k wu[r, k] x[b, k]   (fp64)
 *     h[b, r] = silu(g) * u,  silu(g) = g / (1 + exp(-g))
 * for bf16 activations x (batch rows, row stride ldx).  Outputs are
 * [batch x n]; g, u, sg = sum_k |wg||x| and su = sum_k |wu||x| may be NULL.
 */
void oracle_gemv_glu(const uint8_t *wg, const uint8_t *wu, int64_t n, int64_t k,
                     const uint16_t *x, int64_t batch, int64_t ldx, double *h, double *g_out,
                     double *u_out, double *sg_out, double *su_out) {
    double *xd = (double *)malloc(sizeof(double) * (size_t)(batch * k));
    for (int64_t b = 0; b < batch; ++b)
        for (int64_t i = 0; i < k; ++i) xd[b * k + i] = oracle_bf16_to_f64(x[b * ldx + i]);
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < n; ++r) {
        double *wgr = (double *)malloc(sizeof(double) * (size_t)k);
        double *wur = (double *)malloc(sizeof(double) * (size_t)k);
        dequant_row_f64(wg, k, r, wgr);
        dequant_row_f64(wu, k, r, wur);
        for (int64_t b = 0; b < batch; ++b) {
            double g = 0.0, u = 0.0, sg = 0.0, su = 0.0;
            for (int64_t i = 0; i < k; ++i) {
                g += wgr[i] * xd[b * k + i];
                u += wur[i] * xd[b * k + i];
                sg += fabs(wgr[i]) * fabs(xd[b * k + i]);
                su += fabs(wur[i]) * fabs(xd[b * k + i]);
            }
            h[b * n + r] = g / (1.0 + exp(-g)) * u;
            if (g_out) g_out[b * n + r] = g;
            if (u_out) u_out[b * n + r] = u;
            if (sg_out) sg_out[b * n + r] = sg;
            if (su_out) su_out[b * n + r] = su;
        }
        free(wgr);
        free(wur);
    }
    free(xd);
}

/*
 * Routed mixture-of-experts FFN for decode tokens ("Layer Package Repository
 * Spec", section "Policy Resolution": the routed gate/up/down expert matmuls,
 * the fused SwiGLU and the route-weighted sum of a routed FFN decode layer).
 *
 * For token t and slot j with expert e = ids[t*top_k + j]:
 *     g = Wg_e x_t,  u = Wu_e x_t            (ffn values each)
 *     h = silu(g) * u,  silu(g) = g / (1 + exp(-g))
 *     p = Wd_e h                             (hidden values)
 *     y_t = sum_j wts[t*top_k + j] * p       (slots in order j = 0 .. top_k-1)
 * With weighted_down set, the route weight moves ahead of the down projection
 * ("Layer Package Repository Spec", section "Execution Policy",
 * experimental.moe_weighted_down):
 *     p = Wd_e (wts[t*top_k + j] * h),  y_t = sum_j p   (same slot order)
 * which equals the plain form in exact arithmetic (Wd is linear).
 * Expert e's matrices start at byte e * expert_stride of each weight array;
 * gate/up are ffn x hidden, down is hidden x ffn.  A slot whose id is outside
 * [0, n_experts) contributes nothing.  x is [n_tokens x ldx] bf16, y is
 * [n_tokens x hidden] fp64.  g, u, h (each [n_tokens*top_k x ffn], slot-major
 * within a token; h before any route weight) may be NULL.
 */
void oracle_moe(const uint8_t *wg, const uint8_t *wu, const uint8_t *wd, int64_t expert_stride,
                int32_t n_experts, int64_t hidden, int64_t ffn, const uint16_t *x, int32_t n_tokens,
                int64_t ldx, const int32_t *ids, const float *wts, int32_t top_k, double *y,
                double *g_out, double *u_out, double *h_out, int weighted_down) {
    double *g = (double *)malloc(sizeof(double) * (size_t)ffn);
    double *u = (double *)malloc(sizeof(double) * (size_t)ffn);
    double *h = (double *)malloc(sizeof(double) * (size_t)ffn);
    double *p = (double *)malloc(sizeof(double) * (size_t)hidden);
    for (int32_t t = 0; t < n_tokens; ++t) {
        for (int64_t i = 0; i < hidden; ++i) y[t * hidden + i] = 0.0;
        for (int32_t j = 0; j < top_k; ++j) {
            int64_t slot = (int64_t)t * top_k + j;
            int32_t e = ids[slot];
            if (e < 0 || e >= n_experts) {
                for (int64_t f = 0; f < ffn; ++f) {
                    if (g_out) g_out[slot * ffn + f] = 0.0;
                    if (u_out) u_out[slot * ffn + f] = 0.0;
                    if (h_out) h_out[slot * ffn + f] = 0.0;
                }
                continue;
            }
            const uint8_t *ge = wg + (size_t)e * (size_t)expert_stride;
            const uint8_t *ue = wu + (size_t)e * (size_t)expert_stride;
            const uint8_t *de = wd + (size_t)e * (size_t)expert_stride;
            oracle_gemv_bf16(ge, ffn, hidden, x + (size_t)t * ldx, 1, ldx, NULL, 0, g, NULL);
            oracle_gemv_bf16(ue, ffn, hidden, x + (size_t)t * ldx, 1, ldx, NULL, 0, u, NULL);
            for (int64_t f = 0; f < ffn; ++f) {
                h[f] = g[f] / (1.0 + exp(-g[f])) * u[f];
                if (g_out) g_out[slot * ffn + f] = g[f];
                if (u_out) u_out[slot * ffn + f] = u[f];
                if (h_out) h_out[slot * ffn + f] = h[f];
            }
            double r = (double)wts[slot];
            if (weighted_down) {
                for (int64_t f = 0; f < ffn; ++f) h[f] *= r;
                oracle_gemv_f64(de, hidden, ffn, h, 1, ffn, 0, p);
                for (int64_t i = 0; i < hidden; ++i) y[t * hidden + i] += p[i];
            } else {
                oracle_gemv_f64(de, hidden, ffn, h, 1, ffn, 0, p);
                for (int64_t i = 0; i < hidden; ++i) y[t * hidden + i] += r * p[i];
            }
        }
    }
    free(g);
    free(u);
    free(h);
    free(p);
}

/*
 * Quantized projection of RMS-normalised activations ("spec: specialized model
 * runtimes", section "Feasibility gate": one quantized GEMM plus fused
 * RMSNorm; the norm is the prologue of the projection).  For each token b:
 *     rinv_b  = 1 / sqrt( (1/k) sum_i x[b,i]^2 + eps )
 *     xh[b,i] = x[b,i] * rinv_b * gamma[i]
 *     y[b,r]  = sum_i w[r,i] xh[b,i],   s[b,r] = sum_i |w[r,i]| |xh[b,i]|
 * in fp64 throughout (x bf16, gamma and eps fp32 as given).  y and s are
 * [batch x n]; rinv_out ([batch]) may be NULL.
 */
void oracle_rmsnorm_gemv(const uint8_t *w, int64_t n, int64_t k, const uint16_t *x, int64_t batch,
                         int64_t ldx, const float *gamma, float eps, double *y, double *s,
                         double *rinv_out) {
    double *xh = (double *)malloc(sizeof(double) * (size_t)(batch * k));
    double *axh = (double *)malloc(sizeof(double) * (size_t)(batch * k));
    for (int64_t b = 0; b < batch; ++b) {
        double ss = 0.0;
        for (int64_t i = 0; i < k; ++i) {
            double v = oracle_bf16_to_f64(x[b * ldx + i]);
            ss += v * v;
        }
        double rinv = 1.0 / sqrt(ss / (double)k + (double)eps);
        if (rinv_out) rinv_out[b] = rinv;
        for (int64_t i = 0; i < k; ++i) {
            xh[b * k + i] = oracle_bf16_to_f64(x[b * ldx + i]) * rinv * (double)gamma[i];
            axh[b * k + i] = fabs(xh[b * k + i]);
        }
    }
    oracle_gemv_f64(w, n, k, xh, batch, k, 0, y);
    oracle_gemv_f64(w, n, k, axh, batch, k, 1, s);
    free(xh);
    free(axh);
}

/*
 * Other k-quant formats ("Layer Package Repository Spec", section "Policy
 * Resolution": the q2_K / q3_K routed-down recipes; "UD-Q4_K_XL" mixes also
 * carry Q5_K and Q6_K tensors).  The pages name these formats and print none of
 * their bytes; the layouts below are the plain reading of the GGUF k-quant
 * super-blocks (256 weights each), restated here.  Compatibility with real
 * GGUF files is parity unpinned; the tests pin each layout against an
 * independent packer, Q5_K against Q4_K, and the weight positions by probes.
 * Every weight is exact in fp64 (at most 11 + 8 + 6 significant bits).
 *
 * q2_K, 84 bytes:  sc[16] | qs[64] | d (binary16) | dmin (binary16)
 *   16 sub-blocks of 16 weights; byte sc[j]: scale = low nibble, min = high
 *   nibble.  Weight i: half h = i/128, r = i%128, group g = r/32, l = r%32:
 *   q = (qs[32h + l] >> 2g) & 3, sub-block j = 8h + 2g + (l >= 16);
 *   w = d * scale_j * q - dmin * min_j.
 * q3_K, 110 bytes: hmask[32] | qs[64] | s[12] | d (binary16)
 *   16 six-bit scales: low 4 bits of scale j are the low nibble of s[j]
 *   (j < 8) or the high nibble of s[j-8] (j >= 8); its top 2 bits are bits
 *   2(j/4), 2(j/4)+1 of s[8 + j%4].  Weight i (h, g, l, j as for q2_K):
 *   q = ((qs[32h + l] >> 2g) & 3) - (bit (4h + g) of hmask[l] ? 0 : 4),
 *   w = d * (scale_j - 32) * q.
 * Q5_K, 176 bytes: d | dmin | s[12] (as Q4_K) | qh[32] | qs[128]
 *   as Q4_K with a fifth bit: weight i in chunk c = i/64, l = i%32, high
 *   half (i%64 >= 32) or low: q = nibble of qs[32c + l] + 16 * bit (2c + high)
 *   of qh[l];  w = d * sc_j * q - dmin * m_j, j = i/32.
 * Q6_K, 210 bytes: ql[128] | qh[64] | sc[16] (int8) | d (binary16)
 *   weight i: half h = i/128, r = i%128, quarter u = r/32, l = r%32:
 *   low 4 bits: ql[64h + l + 32(u & 1)], low nibble for u < 2, high for u >= 2;
 *   high 2 bits: bits 2u, 2u+1 of qh[32h + l];  q = that 6-bit value - 32;
 *   w = d * sc[8h + 2u + l/16] * q.
 */
int oracle_kq_block_bytes(int fmt) {
    switch (fmt) {
        case 2: return 84;
        case 3: return 110;
        case 4: return Q4K_BYTES;
        case 5: return 176;
        case 6: return 210;
        default: return 0;
    }
}

static double half_at(const uint8_t *p) {
    return oracle_fp16_to_f64((uint16_t)(p[0] | (p[1] << 8)));
}

static void dequant_q2k_block(const uint8_t *b, double out[256]) {
    const uint8_t *sc = b, *qs = b + 16;
    double d = half_at(b + 80), dmin = half_at(b + 82);
    for (int i = 0; i < 256; ++i) {
        int h = i / 128, r = i % 128, g = r / 32, l = r % 32;
        int q = (qs[32 * h + l] >> (2 * g)) & 3;
        int j = 8 * h + 2 * g + (l >= 16);
        out[i] = d * (sc[j] & 15) * q - dmin * (sc[j] >> 4);
    }
}

static int q3k_scale(const uint8_t s[12], int j) {
    int lo = j < 8 ? (s[j] & 15) : (s[j - 8] >> 4);
    int hi = (s[8 + j % 4] >> (2 * (j / 4))) & 3;
    return lo | (hi << 4);
}

static void dequant_q3k_block(const uint8_t *b, double out[256]) {
    const uint8_t *hm = b, *qs = b + 32, *s = b + 96;
    double d = half_at(b + 108);
    for (int i = 0; i < 256; ++i) {
        int h = i / 128, r = i % 128, g = r / 32, l = r % 32;
        int q = ((qs[32 * h + l] >> (2 * g)) & 3) - (((hm[l] >> (4 * h + g)) & 1) ? 0 : 4);
        int j = 8 * h + 2 * g + (l >= 16);
        out[i] = d * (q3k_scale(s, j) - 32) * q;
    }
}

static void dequant_q5k_block(const uint8_t *b, double out[256]) {
    double d = half_at(b), dmin = half_at(b + 2);
    int sc[8], m[8];
    oracle_unpack_scales(b + 4, sc, m);
    const uint8_t *qh = b + 16, *qs = b + 48;
    for (int i = 0; i < 256; ++i) {
        int c = i / 64, l = i % 32, high = (i % 64) >= 32;
        int nib = high ? (qs[32 * c + l] >> 4) : (qs[32 * c + l] & 15);
        int q = nib + 16 * ((qh[l] >> (2 * c + high)) & 1);
        out[i] = d * sc[i / 32] * q - dmin * m[i / 32];
    }
}

static void dequant_q6k_block(const uint8_t *b, double out[256]) {
    const uint8_t *ql = b, *qh = b + 128;
    const int8_t *sc = (const int8_t *)(b + 192);
    double d = half_at(b + 208);
    for (int i = 0; i < 256; ++i) {
        int h = i / 128, r = i % 128, u = r / 32, l = r % 32;
        uint8_t lb = ql[64 * h + l + 32 * (u & 1)];
        int lo = u < 2 ? (lb & 15) : (lb >> 4);
        int hi = (qh[32 * h + l] >> (2 * u)) & 3;
        int q = (lo | (hi << 4)) - 32;
        out[i] = d * sc[8 * h + 2 * u + l / 16] * q;
    }
}

/* One super-block of format fmt -> its 256 weights, exact, in fp64. */
void oracle_kq_dequant_block_f64(int fmt, const uint8_t *blk, double out[256]) {
    switch (fmt) {
        case 2: dequant_q2k_block(blk, out); break;
        case 3: dequant_q3k_block(blk, out); break;
        case 4: oracle_dequant_block_f64(blk, out); break;
        case 5: dequant_q5k_block(blk, out); break;
        case 6: dequant_q6k_block(blk, out); break;
        default: memset(out, 0, sizeof(double) * 256);
    }
}

static void kq_row_f64(int fmt, const uint8_t *w, int64_t k, int64_t r, double *out) {
    int bb = oracle_kq_block_bytes(fmt);
    const uint8_t *row = w + (size_t)r * (size_t)(k / 256) * (size_t)bb;
    for (int64_t b = 0; b < k / 256; ++b) oracle_kq_dequant_block_f64(fmt, row + b * bb, out + b * 256);
}

void oracle_kq_dequant_f64(int fmt, const uint8_t *w, int64_t n, int64_t k, double *out) {
    for (int64_t r = 0; r < n; ++r) kq_row_f64(fmt, w, k, r, out + r * k);
}

/* fp32: one round-to-nearest-even of the exact value; bf16: that, then RNE. */
void oracle_kq_dequant_f32(int fmt, const uint8_t *w, int64_t n, int64_t k, float *out) {
    double *tmp = (double *)malloc(sizeof(double) * (size_t)k);
    for (int64_t r = 0; r < n; ++r) {
        kq_row_f64(fmt, w, k, r, tmp);
        for (int64_t i = 0; i < k; ++i) out[r * k + i] = (float)tmp[i];
    }
    free(tmp);
}

void oracle_kq_dequant_bf16(int fmt, const uint8_t *w, int64_t n, int64_t k, uint16_t *out) {
    double *tmp = (double *)malloc(sizeof(double) * (size_t)k);
    for (int64_t r = 0; r < n; ++r) {
        kq_row_f64(fmt, w, k, r, tmp);
        for (int64_t i = 0; i < k; ++i) out[r * k + i] = oracle_f32_to_bf16_rne((float)tmp[i]);
    }
    free(tmp);
}

/* y = W x and s = |W| |x| (fp64, natural k order) for bf16 activations
 * [batch x k], row stride ldx; y and s are [batch x n]. */
void oracle_kq_gemv_bf16(int fmt, const uint8_t *w, int64_t n, int64_t k, const uint16_t *x,
                         int64_t batch, int64_t ldx, double *y, double *s) {
    double *xd = (double *)malloc(sizeof(double) * (size_t)(batch * k));
    for (int64_t b = 0; b < batch; ++b)
        for (int64_t i = 0; i < k; ++i) xd[b * k + i] = oracle_bf16_to_f64(x[b * ldx + i]);
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t r = 0; r < n; ++r) {
        double *wr = (double *)malloc(sizeof(double) * (size_t)k);
        kq_row_f64(fmt, w, k, r, wr);
        for (int64_t b = 0; b < batch; ++b) {
            double acc = 0.0, mag = 0.0;
            for (int64_t i = 0; i < k; ++i) {
                acc += wr[i] * xd[b * k + i];
                mag += fabs(wr[i]) * fabs(xd[b * k + i]);
            }
            y[b * n + r] = acc;
            if (s) s[b * n + r] = mag;
        }
        free(wr);
    }
    free(xd);
}

/* Threads the parallel loops above use (1 without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
