/*
 * qvg_oracle.c -- plain, slow CPU oracle for 2-bit / 4-bit video KV-cache
 * compression (Quant VideoGen "QVG" / "QVG-Pro") and the QuantWM extensions
 * (QSAC weighting, PSAC rank-r key-error correction), plus attention over
 * the reconstructed cache.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or helper with the CUDA library; both sides read the same
 * seeded synthetic inputs and nothing else.
 *
 * Precision: fp64 wherever the pages leave precision open (k-means
 * distances, means, attention, second moments, Jacobi).  The integer
 * decisions of the quantisers (codes) are taken in fp32 with IEEE division
 * and round-half-to-even, the arithmetic the GPU kernels use, so that codes
 * can be compared bit for bit.
 *
 * Sources, by page and section:
 *   [QVG]  "Quant VideoGen: Auto-Regressive Long Video Generation via 2-Bit
 *          KV-Cache Quantization" (papernotes.org, ICML 2026 notes):
 *          "core tension" (quantiser S = max|X|/(2^{b-1}-1), X_INT = round(X/S)),
 *          "overall framework" (chunk-wise k-means, residual, dequant
 *          S*X_INT + C_i, BF16 centroids), "Semantic-Aware Smoothing",
 *          "Progressive Residual Quantization", "algorithm-system co-design"
 *          (packed INT2).
 *   [P1]   "The 2-bit quantisation trap in video generation"
 *          (cloud.baidu.com), section 2: toy per-group 2-bit quantiser with
 *          scale = amax/2 and clamp to [-2, 1]; section 1: KV size formula.
 *   [QWM]  QuantWM write-up (loncent.com): QSAC (query-activity-weighted
 *          clustering) and PSAC (top-8 eigenvectors of the history-query
 *          second moment, projected key error, quantised, added back to the
 *          logits).
 *   [P2]   Temporally stable 2-bit KV-cache compression for video world models, in practice (hmyw.cn), section 3.4 (outlier separation).
 *
 * Readings of points the pages leave open are stated where they are used.
 *
 * Parity status: every function here is pinned by a CPU test against a
 * worked example, a closed form, an invariant or brute force, except the
 * absolute quality figures of the pages (PSNR, shift rates), which need the
 * pages' models and are out of reach ("parity unpinned" for those only).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* Number formats.                                                     */
/* ------------------------------------------------------------------ */

/* bf16 -> fp32: the bf16 pattern is the top half of the fp32 pattern. */
static float bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* fp32 -> bf16 with round-to-nearest-even (finite inputs). */
static uint16_t f32_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

static float bf16_round(float f) { return bf16_to_f32(f32_to_bf16(f)); }

/* fp32 <-> IEEE binary16, round-to-nearest-even (compiler conversion). */
static uint16_t f32_to_f16(float f) {
    _Float16 h = (_Float16)f;
    uint16_t b;
    memcpy(&b, &h, 2);
    return b;
}

static float f16_to_f32(uint16_t b) {
    _Float16 h;
    memcpy(&h, &b, 2);
    return (float)h;
}

/* ------------------------------------------------------------------ */
/* Per-group symmetric quantiser.                                      */
/* ------------------------------------------------------------------ */

/*
 * [QVG] "core tension": S = max|X| / (2^{b-1} - 1), X_INT = round(X / S).
 * [P1] section 2 variant (mode 1): scale = amax / 2, q = clamp(round(x/scale), -2, 1).
 *
 * Readings: the scale is stored as fp16 (round-to-nearest-even, saturated at
 * the fp16 maximum 65504) and the codes are computed with the stored value,
 * so encoder and decoder agree; round() is half-to-even (torch.round in the
 * P1 listing is half-to-even); codes are clamped to the signed b-bit range
 * [-2^{b-1}, 2^{b-1}-1] (for b = 2 that is the P1 clamp [-2, 1]); a group
 * whose stored scale is 0 gets all-zero codes.  Dequantisation is S' * q.
 */
void orc_quant_group(const float *r, int G, int bits, int mode,
                     uint16_t *scale_f16, int32_t *q, float *rhat) {
    float amax = 0.0f;
    for (int j = 0; j < G; ++j) {
        float a = fabsf(r[j]);
        if (a > amax) amax = a;
    }
    const int qmax = (1 << (bits - 1)) - 1;
    const int qmin = -(1 << (bits - 1));
    float S = (mode == 0) ? amax / (float)qmax : amax / 2.0f;
    if (S > 65504.0f) S = 65504.0f;
    *scale_f16 = f32_to_f16(S);
    const float Sp = f16_to_f32(*scale_f16);
    for (int j = 0; j < G; ++j) {
        int qi = 0;
        if (Sp > 0.0f) {
            float t = rintf(r[j] / Sp);
            if (t < (float)qmin) t = (float)qmin;
            if (t > (float)qmax) t = (float)qmax;
            qi = (int)t;
        }
        q[j] = qi;
        rhat[j] = Sp * (float)qi;
    }
}

/*
 * Outlier split ([P2] section 3.4, "outlier separation"): before a block is
 * quantised, each value whose magnitude is above the block's 99th
 * percentile is taken out of the block and kept in fp16; the block's scale
 * and codes come from the values that remain, so one large value no longer
 * widens the step of all the others.  Readings:
 *   - the block is the quantisation group (G consecutive channels of one
 *     token's residual);
 *   - the percentile is the linear-interpolation one: with the magnitudes
 *     sorted ascending, a_0 <= ... <= a_{G-1}, position p = 0.99 (G - 1),
 *     T = a_k + (p - k)(a_{k+1} - a_k), k = floor(p) (numpy's default);
 *     a value is an outlier when |r| > T, strictly;
 *   - the fp16 copy saturates at +-65504 (like the scales);
 *   - an outlier's code is 0 and it is rebuilt as its fp16 value (plus the
 *     centroid), its channel index within the group kept as a uint8;
 *   - the side list holds one (value, index) pair per group, index 0xFF
 *     meaning "none": for G <= 100, p > G - 2, so at most the largest value
 *     can lie above T.  Larger groups are refused (return -1).
 * The page's companion "dynamic clipping" (an adaptive per-block range) is
 * what the per-group scale of the remaining values already is; it gives no
 * formula for a clip below their maximum, so none is applied.
 */
static int cmp_double(const void *a, const void *b) {
    const double x = *(const double *)a, y = *(const double *)b;
    return (x > y) - (x < y);
}

int orc_quant_group_outlier(const float *r, int G, int bits, int mode,
                            uint16_t *scale_f16, int32_t *q, float *rhat,
                            uint16_t *outl_f16, uint8_t *outl_idx) {
    if (G < 2 || G > 100) return -1;
    double a[100];
    for (int j = 0; j < G; ++j) a[j] = fabs((double)r[j]);
    qsort(a, (size_t)G, sizeof(double), cmp_double);
    const double p = 0.99 * (double)(G - 1);
    const int k = (int)floor(p);
    const double T = a[k] + (p - (double)k) * (a[k + 1] - a[k]);
    int out = -1, count = 0;
    for (int j = 0; j < G; ++j)
        if (fabs((double)r[j]) > T) { out = j; ++count; }
    if (count > 1) return -1;
    /* quantise the remaining values (the outlier's slot holds 0) */
    float rest[100];
    for (int j = 0; j < G; ++j) rest[j] = (j == out) ? 0.0f : r[j];
    orc_quant_group(rest, G, bits, mode, scale_f16, q, rhat);
    if (out < 0) {
        *outl_f16 = 0;
        *outl_idx = 0xFF;
        return 0;
    }
    float o = r[out];
    if (o > 65504.0f) o = 65504.0f;
    if (o < -65504.0f) o = -65504.0f;
    *outl_f16 = f32_to_f16(o);
    *outl_idx = (uint8_t)out;
    q[out] = 0;
    rhat[out] = f16_to_f32(*outl_f16);
    return 0;
}

/*
 * Packing ([QVG] "algorithm-system co-design": 2-bit codes are stored as a
 * packed integer representation).  Reading: offset-binary u = q + 2^{b-1};
 * element j of a row occupies bits [(j*b) mod 8, +b) of byte (j*b)/8.
 */
void orc_pack_row(const int32_t *q, int d, int bits, uint8_t *out) {
    const int nbytes = d * bits / 8;
    memset(out, 0, (size_t)nbytes);
    for (int j = 0; j < d; ++j) {
        uint32_t u = (uint32_t)(q[j] + (1 << (bits - 1)));
        out[(j * bits) / 8] |= (uint8_t)(u << ((j * bits) % 8));
    }
}

void orc_unpack_row(const uint8_t *in, int d, int bits, int32_t *q) {
    const uint32_t mask = (1u << bits) - 1u;
    for (int j = 0; j < d; ++j) {
        uint32_t u = ((uint32_t)in[(j * bits) / 8] >> ((j * bits) % 8)) & mask;
        q[j] = (int32_t)u - (1 << (bits - 1));
    }
}

/* ------------------------------------------------------------------ */
/* k-means (Semantic-Aware Smoothing).                                 */
/* ------------------------------------------------------------------ */

/* SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
 * generators", OOPSLA 2014): one output for a given state. */
static uint64_t splitmix64_next(uint64_t *state) {
    uint64_t z = (*state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/*
 * Initial centroids.  The pages do not say how k-means starts.  Reading: a
 * seeded systematic sample of C distinct tokens -- one random 32-bit offset
 * u per (chunk, head, stage) and token index
 *   idx_c = floor((c * 2^32 + u) * N / (C * 2^32)),  c = 0..C-1,
 * i.e. one pick in each of C equal strata of the chunk's raster order.
 * u is the top 32 bits of the first SplitMix64 output from state
 * seed ^ (chunk << 40) ^ (head << 20) ^ stage.  Requires C <= N.
 */
void orc_init_picks(int N, int C, uint64_t seed, int chunk, int head,
                    int stage, int32_t *idx) {
    uint64_t st = seed ^ ((uint64_t)chunk << 40) ^ ((uint64_t)head << 20) ^
                  (uint64_t)stage;
    const uint64_t u = splitmix64_next(&st) >> 32;
    for (int c = 0; c < C; ++c) {
        const uint64_t num = (((uint64_t)c << 32) + u) * (uint64_t)N;
        idx[c] = (int32_t)(num / ((uint64_t)C << 32));
    }
}

/*
 * Assignment step: id(n) = argmin_c sum_j w_j (x_nj - c_j)^2, fp64, from the
 * bf16-valued operands the clustering sees; ties go to the lowest c.
 * w == NULL means w = 1 (plain QVG); otherwise w is the QSAC per-channel
 * query activity ([QWM] QSAC: weight the quantisation error of channels by
 * how active history queries are on them).
 * Optional outputs for the near-tie analysis: best and second-best
 * distance, and ||x||_w^2 + ||c_best||_w^2.
 */
void orc_assign(const float *g, int N, int d, const float *cent, int C,
                const float *w, int32_t *ids, double *best, double *second,
                double *denom) {
    for (int n = 0; n < N; ++n) {
        const float *x = g + (size_t)n * d;
        double b1 = INFINITY, b2 = INFINITY;
        int arg = 0;
        for (int c = 0; c < C; ++c) {
            const float *cc = cent + (size_t)c * d;
            double s = 0.0;
            for (int j = 0; j < d; ++j) {
                const double diff = (double)x[j] - (double)cc[j];
                const double wj = w ? (double)w[j] : 1.0;
                s += wj * diff * diff;
            }
            if (s < b1) {
                b2 = b1;
                b1 = s;
                arg = c;
            } else if (s < b2) {
                b2 = s;
            }
        }
        ids[n] = arg;
        if (best) best[n] = b1;
        if (second) second[n] = b2;
        if (denom) {
            const float *cc = cent + (size_t)arg * d;
            double nx = 0.0, nc = 0.0;
            for (int j = 0; j < d; ++j) {
                const double wj = w ? (double)w[j] : 1.0;
                nx += wj * (double)x[j] * (double)x[j];
                nc += wj * (double)cc[j] * (double)cc[j];
            }
            denom[n] = nx + nc;
        }
    }
}

/*
 * Update step: each centroid becomes the mean of its members' fp32 stage
 * input (summed in fp64, token order), held as fp32 and stored as bf16
 * ([QVG] "overall framework": centroids are kept in BF16).  A cluster with
 * no member keeps its previous centroid.  A diagonal weight does not move
 * the minimiser of a weighted squared distance, so the update is the plain
 * mean for QSAC too.  cent is updated in place (bf16-valued floats);
 * mean32 (optional) receives the fp32 means (previous centroid for empty
 * clusters); counts (optional) receives member counts.
 */
void orc_update(const float *xin, int N, int d, const int32_t *ids, int C,
                float *cent, float *mean32, int32_t *counts) {
    double *sum = (double *)calloc((size_t)C * d, sizeof(double));
    int32_t *cnt = (int32_t *)calloc((size_t)C, sizeof(int32_t));
    for (int n = 0; n < N; ++n) {
        const int c = ids[n];
        cnt[c] += 1;
        for (int j = 0; j < d; ++j)
            sum[(size_t)c * d + j] += (double)xin[(size_t)n * d + j];
    }
    for (int c = 0; c < C; ++c) {
        for (int j = 0; j < d; ++j) {
            float m = cent[(size_t)c * d + j];
            if (cnt[c] > 0) m = (float)(sum[(size_t)c * d + j] / (double)cnt[c]);
            if (mean32) mean32[(size_t)c * d + j] = m;
            cent[(size_t)c * d + j] = bf16_round(m);
        }
        if (counts) counts[c] = cnt[c];
    }
    free(sum);
    free(cnt);
}

/* Weighted inertia sum_n sum_j w_j (x_nj - c_{id(n),j})^2 in fp64. */
double orc_inertia(const float *g, int N, int d, const float *cent,
                   const int32_t *ids, const float *w) {
    double s = 0.0;
    for (int n = 0; n < N; ++n)
        for (int j = 0; j < d; ++j) {
            const double diff = (double)g[(size_t)n * d + j] -
                                (double)cent[(size_t)ids[n] * d + j];
            s += (w ? (double)w[j] : 1.0) * diff * diff;
        }
    return s;
}

/* ------------------------------------------------------------------ */
/* PSAC encode / decode of one token ([QWM] PSAC).                      */
/* ------------------------------------------------------------------ */

/*
 * P = E U projects the token's remaining key error E (d values) on the r
 * basis vectors (U is d x r, row-major).  Reading: "quantised and stored"
 * is INT8, one symmetric fp16 scale per token, S = amax/127, codes clamped
 * to [-127, 127], the quantiser rules as above.  The projection is
 * accumulated in fp32 by fused multiply-add in ascending channel order, so
 * the INT8 decision is taken in the same arithmetic on every side.
 */
void orc_psac_encode_token(const float *E, const float *U, int d, int r,
                           int8_t *p, uint16_t *s_f16) {
    float P[64];
    float amax = 0.0f;
    for (int k = 0; k < r; ++k) {
        float acc = 0.0f;
        for (int j = 0; j < d; ++j) acc = fmaf(E[j], U[(size_t)j * r + k], acc);
        P[k] = acc;
        if (fabsf(acc) > amax) amax = fabsf(acc);
    }
    float S = amax / 127.0f;
    if (S > 65504.0f) S = 65504.0f;
    *s_f16 = f32_to_f16(S);
    const float Sp = f16_to_f32(*s_f16);
    for (int k = 0; k < r; ++k) {
        int qi = 0;
        if (Sp > 0.0f) {
            float t = rintf(P[k] / Sp);
            if (t < -127.0f) t = -127.0f;
            if (t > 127.0f) t = 127.0f;
            qi = (int)t;
        }
        p[k] = (int8_t)qi;
    }
}

/* ------------------------------------------------------------------ */
/* Compression of one chunk (all heads, all stages).                   */
/* ------------------------------------------------------------------ */

typedef struct {
    int C, L, bits, group, iters, mode, outlier;
    uint64_t seed;
} orc_params;

typedef struct {
    const float *x;      /* [N][H][d] bf16-valued input */
    int N, H, d, chunk;
    orc_params p;
    const float *qsac_w; /* [H][d] or NULL */
    const float *psac_U; /* [H][d][r] or NULL */
    int psac_r;
    const float *cent_in; /* [L][H][C][d] given centroids or NULL */
    uint8_t *codes;       /* [L][H][N][d*bits/8] */
    uint16_t *scales;     /* [L][H][N][d/G] fp16 */
    uint8_t *ids;         /* [L][H][N] */
    uint16_t *cent;       /* [L][H][C][d] bf16 */
    float *means;         /* [L][H][C][d] fp32 or NULL */
    int8_t *psac_p;       /* [H][N][r] */
    uint16_t *psac_s;     /* [H][N] */
    float *xhat;          /* [N][H][d] or NULL: sum over stages of dequant */
    float *resid;         /* [N][H][d] or NULL: residual after the last stage */
    uint16_t *outl_val;   /* [L][H][N][d/G] fp16 (outlier split) */
    uint8_t *outl_idx;    /* [L][H][N][d/G] channel within the group, 0xFF none */
} compress_job;

/*
 * One head, all stages ([QVG] "Semantic-Aware Smoothing" and "Progressive
 * Residual Quantization"):
 *   stage input X_1 = X (fp32 values of the bf16 chunk), X_{l+1} = X_l - deq_l;
 *   clustering operand = X_1 (stage 1) or bf16(X_l) (later stages, reading);
 *   k-means: init, `iters` x (assign, update), one final assign;
 *   residual R = X_l - C_id (fp32), per-group quantisation (with the
 *   outlier split when p->outlier), deq_l = S'q + C_id (fp16 outlier + C_id
 *   at an outlier's channel);
 *   reconstruction = deq_1 + deq_2 + ... (fp32, stage order).
 * C = 0 is plain per-group quantisation (RTN): no centroid.
 * C > N clusters with C_eff = N; centroid rows C_eff..C-1 are stored as 0.
 */
static void compress_head(const compress_job *J, int h) {
    const int N = J->N, H = J->H, d = J->d;
    const orc_params *p = &J->p;
    const int C = p->C, L = p->L, G = p->group, bits = p->bits;
    const int Ce = (C < N) ? C : N;
    const int nb = d * bits / 8, ng = d / G;
    const float *w = J->qsac_w ? J->qsac_w + (size_t)h * d : NULL;

    float *xin = (float *)malloc(sizeof(float) * (size_t)N * d);
    float *g = (float *)malloc(sizeof(float) * (size_t)N * d);
    float *xh = (float *)calloc((size_t)N * d, sizeof(float));
    float *cent = (float *)calloc((size_t)(C > 0 ? C : 1) * d, sizeof(float));
    int32_t *ids = (int32_t *)calloc((size_t)N, sizeof(int32_t));
    int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * (size_t)(C > 0 ? C : 1));
    int32_t q[1024];
    float rr[1024], rh[1024], deq[1024];

    for (int n = 0; n < N; ++n)
        for (int j = 0; j < d; ++j)
            xin[(size_t)n * d + j] = J->x[((size_t)n * H + h) * d + j];

    for (int l = 0; l < L; ++l) {
        for (size_t i = 0; i < (size_t)N * d; ++i)
            g[i] = (l == 0) ? xin[i] : bf16_round(xin[i]);
        const size_t lh = (size_t)l * H + h;
        if (C > 0) {
            memset(cent, 0, sizeof(float) * (size_t)C * d);
            if (J->cent_in) {
                for (int c = 0; c < Ce; ++c)
                    for (int j = 0; j < d; ++j)
                        cent[(size_t)c * d + j] =
                            J->cent_in[(lh * C + c) * d + j];
            } else {
                orc_init_picks(N, Ce, p->seed, J->chunk, h, l, idx);
                for (int c = 0; c < Ce; ++c)
                    for (int j = 0; j < d; ++j)
                        cent[(size_t)c * d + j] = g[(size_t)idx[c] * d + j];
            }
            float *mean = J->means ? J->means + lh * C * d : NULL;
            if (mean)
                for (size_t i = 0; i < (size_t)C * d; ++i) mean[i] = cent[i];
            for (int it = 0; it < p->iters; ++it) {
                orc_assign(g, N, d, cent, Ce, w, ids, NULL, NULL, NULL);
                orc_update(xin, N, d, ids, Ce, cent, mean, NULL);
            }
            orc_assign(g, N, d, cent, Ce, w, ids, NULL, NULL, NULL);
            for (int c = 0; c < C; ++c)
                for (int j = 0; j < d; ++j)
                    J->cent[(lh * C + c) * d + j] =
                        f32_to_bf16(cent[(size_t)c * d + j]);
        }
        for (int n = 0; n < N; ++n) {
            const float *xr = xin + (size_t)n * d;
            const float *cr = cent + (size_t)ids[n] * d;
            J->ids[lh * N + n] = (uint8_t)ids[n];
            for (int j = 0; j < d; ++j) rr[j] = (C > 0) ? xr[j] - cr[j] : xr[j];
            for (int gi = 0; gi < ng; ++gi) {
                const size_t gidx = (lh * N + n) * ng + gi;
                if (p->outlier)
                    orc_quant_group_outlier(rr + gi * G, G, bits, p->mode, &J->scales[gidx],
                                            q + gi * G, rh + gi * G, &J->outl_val[gidx],
                                            &J->outl_idx[gidx]);
                else
                    orc_quant_group(rr + gi * G, G, bits, p->mode, &J->scales[gidx], q + gi * G,
                                    rh + gi * G);
            }
            orc_pack_row(q, d, bits, &J->codes[(lh * N + n) * nb]);
            for (int j = 0; j < d; ++j) deq[j] = (C > 0) ? rh[j] + cr[j] : rh[j];
            for (int j = 0; j < d; ++j) {
                xh[(size_t)n * d + j] = xh[(size_t)n * d + j] + deq[j];
                xin[(size_t)n * d + j] = xr[j] - deq[j];
            }
        }
    }

    if (J->psac_U) {
        const float *U = J->psac_U + (size_t)h * d * J->psac_r;
        for (int n = 0; n < N; ++n)
            orc_psac_encode_token(xin + (size_t)n * d, U, d, J->psac_r,
                                  J->psac_p + ((size_t)h * N + n) * J->psac_r,
                                  J->psac_s + (size_t)h * N + n);
    }
    for (int n = 0; n < N; ++n)
        for (int j = 0; j < d; ++j) {
            if (J->xhat) J->xhat[((size_t)n * H + h) * d + j] = xh[(size_t)n * d + j];
            if (J->resid) J->resid[((size_t)n * H + h) * d + j] = xin[(size_t)n * d + j];
        }
    free(xin); free(g); free(xh); free(cent); free(ids); free(idx);
}

/* ------------------------------------------------------------------ */
/* A tiny static thread pool over independent work units.              */
/* ------------------------------------------------------------------ */

typedef struct {
    void (*fn)(const void *ctx, int unit);
    const void *ctx;
    int units, nthreads, tid;
} pool_arg;

static void *pool_worker(void *a_) {
    const pool_arg *a = (const pool_arg *)a_;
    for (int u = a->tid; u < a->units; u += a->nthreads) a->fn(a->ctx, u);
    return NULL;
}

static void run_units(void (*fn)(const void *, int), const void *ctx,
                      int units, int nthreads) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > units) nthreads = units;
    if (nthreads <= 1) {
        for (int u = 0; u < units; ++u) fn(ctx, u);
        return;
    }
    pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    pool_arg *args = (pool_arg *)malloc(sizeof(pool_arg) * (size_t)nthreads);
    for (int t = 0; t < nthreads; ++t) {
        args[t] = (pool_arg){fn, ctx, units, nthreads, t};
        pthread_create(&th[t], NULL, pool_worker, &args[t]);
    }
    for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
    free(th);
    free(args);
}

static void compress_unit(const void *ctx, int h) {
    compress_head((const compress_job *)ctx, h);
}

/* Public entry: compress one chunk of N tokens, all H heads.  Returns 0 on
 * success, -1 on unsupported arguments. */
int orc_compress_chunk(const float *x, int N, int H, int d, int C, int L,
                       int bits, int group, int iters, int mode, uint64_t seed,
                       int chunk, const float *qsac_w, const float *psac_U,
                       int psac_r, const float *cent_in, uint8_t *codes,
                       uint16_t *scales, uint8_t *ids, uint16_t *cent,
                       float *means, int8_t *psac_p, uint16_t *psac_s,
                       float *xhat, float *resid, uint16_t *outl_val,
                       uint8_t *outl_idx, int nthreads) {
    const int outlier = outl_val != NULL;
    if (N < 1 || H < 1 || d < 1 || d > 1024 || L < 1 || group < 1 ||
        d % group != 0 || (bits != 2 && bits != 4) || (d * bits) % 8 != 0 ||
        C < 0 || C > 256 || iters < 0 || (mode == 1 && bits != 2) ||
        psac_r > 64 || (outlier && (!outl_idx || group < 2 || group > 100)))
        return -1;
    compress_job J = {x, N, H, d, chunk, {C, L, bits, group, iters, mode, outlier, seed},
                      qsac_w, psac_U, psac_r, cent_in, codes, scales, ids,
                      cent, means, psac_p, psac_s, xhat, resid, outl_val, outl_idx};
    run_units(compress_unit, &J, H, nthreads);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Reconstruction from the stored layout.                              */
/* ------------------------------------------------------------------ */

/*
 * Rebuild X_hat = sum_l (S'_l q_l + C_{l,id}) from stored codes, fp16
 * scales, ids and bf16 centroids ([QVG] "overall framework": dequant adds
 * S_X * X_INT + C_i back), fp32, in stage order; at a split-off outlier's
 * channel the stage's term is its fp16 value + C_{l,id} ([P2] section 3.4);
 * plus, when PSAC data are given, the correction P_hat U^T computed in
 * fp64.  Layouts as in orc_compress_chunk with N tokens.  out is [N][H][d].
 */
int orc_decompress(const uint8_t *codes, const uint16_t *scales,
                   const uint8_t *ids, const uint16_t *cent, int N, int H,
                   int d, int C, int L, int bits, int group,
                   const int8_t *psac_p, const uint16_t *psac_s,
                   const float *psac_U, int psac_r, const uint16_t *outl_val,
                   const uint8_t *outl_idx, float *out) {
    const int nb = d * bits / 8, ng = d / group;
    int32_t q[1024];
    for (int h = 0; h < H; ++h)
        for (int n = 0; n < N; ++n) {
            float acc[1024];
            for (int j = 0; j < d; ++j) acc[j] = 0.0f;
            for (int l = 0; l < L; ++l) {
                const size_t lh = (size_t)l * H + h;
                orc_unpack_row(&codes[(lh * N + n) * nb], d, bits, q);
                for (int j = 0; j < d; ++j) {
                    const size_t gidx = (lh * N + n) * ng + j / group;
                    const float S = f16_to_f32(scales[gidx]);
                    float v = S * (float)q[j];
                    if (outl_val && outl_idx[gidx] == j % group) v = f16_to_f32(outl_val[gidx]);
                    if (C > 0) v = v + bf16_to_f32(cent[(lh * C + ids[lh * N + n]) * d + j]);
                    acc[j] = acc[j] + v;
                }
            }
            if (psac_p) {
                const float Sp = f16_to_f32(psac_s[(size_t)h * N + n]);
                const float *U = psac_U + (size_t)h * d * psac_r;
                for (int j = 0; j < d; ++j) {
                    double corr = 0.0;
                    for (int k = 0; k < psac_r; ++k)
                        corr += (double)(Sp * (float)psac_p[((size_t)h * N + n) * psac_r + k]) *
                                (double)U[(size_t)j * psac_r + k];
                    acc[j] = (float)((double)acc[j] + corr);
                }
            }
            for (int j = 0; j < d; ++j) out[((size_t)n * H + h) * d + j] = acc[j];
        }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Attention over the reconstructed cache.                             */
/* ------------------------------------------------------------------ */

typedef struct {
    const float *q, *k, *v;
    int Nq, Hq, Nk, H, d;
    double scale;
    double *out, *lse;
    int32_t *argmax;
} attn_job;

/*
 * O = softmax(scale * q K^T) V for one query row of one query head, fp64,
 * max-subtracted ([QVG] "overall framework": the reconstructed K/V enter
 * attention; softmax scale 1/sqrt(d) and no mask are readings: the cache
 * holds only earlier tokens).  Query head hq reads KV head hq / (Hq/H).
 * Also the log-sum-exp (natural log) and the top-1 key (lowest index on ties).
 */
static void attn_unit(const void *ctx, int unit) {
    const attn_job *A = (const attn_job *)ctx;
    const int hq = unit / A->Nq, i = unit % A->Nq;
    const int h = hq / (A->Hq / A->H), d = A->d;
    const float *qr = A->q + ((size_t)i * A->Hq + hq) * d;
    double *s = (double *)malloc(sizeof(double) * (size_t)A->Nk);
    double mx = -INFINITY;
    int arg = 0;
    for (int t = 0; t < A->Nk; ++t) {
        const float *kr = A->k + ((size_t)t * A->H + h) * d;
        double dot = 0.0;
        for (int j = 0; j < d; ++j) dot += (double)qr[j] * (double)kr[j];
        s[t] = A->scale * dot;
        if (s[t] > mx) { mx = s[t]; arg = t; }
    }
    double den = 0.0;
    for (int t = 0; t < A->Nk; ++t) { s[t] = exp(s[t] - mx); den += s[t]; }
    double *o = A->out + ((size_t)i * A->Hq + hq) * d;
    for (int j = 0; j < d; ++j) o[j] = 0.0;
    for (int t = 0; t < A->Nk; ++t) {
        const float *vr = A->v + ((size_t)t * A->H + h) * d;
        const double p = s[t] / den;
        for (int j = 0; j < d; ++j) o[j] += p * (double)vr[j];
    }
    if (A->lse) A->lse[(size_t)hq * A->Nq + i] = mx + log(den);
    if (A->argmax) A->argmax[(size_t)hq * A->Nq + i] = arg;
    free(s);
}

int orc_attention(const float *q, int Nq, int Hq, const float *k,
                  const float *v, int Nk, int H, int d, double scale,
                  double *out, double *lse, int32_t *argmax, int nthreads) {
    if (Nq < 0 || Nk < 1 || H < 1 || Hq % H != 0 || d < 1) return -1;
    if (scale <= 0.0) scale = 1.0 / sqrt((double)d);
    attn_job A = {q, k, v, Nq, Hq, Nk, H, d, scale, out, lse, argmax};
    run_units(attn_unit, &A, Nq * Hq, nthreads);
    return 0;
}

/* Top-1 key only (for the shift rate over long caches). */
typedef struct {
    const float *q, *k;
    int Nq, Hq, Nk, H, d;
    int32_t *argmax;
} top1_job;

static void top1_unit(const void *ctx, int unit) {
    const top1_job *A = (const top1_job *)ctx;
    const int hq = unit / A->Nq, i = unit % A->Nq;
    const int h = hq / (A->Hq / A->H), d = A->d;
    const float *qr = A->q + ((size_t)i * A->Hq + hq) * d;
    double mx = -INFINITY;
    int arg = 0;
    for (int t = 0; t < A->Nk; ++t) {
        const float *kr = A->k + ((size_t)t * A->H + h) * d;
        double dot = 0.0;
        for (int j = 0; j < d; ++j) dot += (double)qr[j] * (double)kr[j];
        if (dot > mx) { mx = dot; arg = t; }
    }
    A->argmax[(size_t)hq * A->Nq + i] = arg;
}

int orc_top1(const float *q, int Nq, int Hq, const float *k, int Nk, int H,
             int d, int32_t *argmax, int nthreads) {
    if (Nq < 0 || Nk < 1 || H < 1 || Hq % H != 0) return -1;
    top1_job A = {q, k, Nq, Hq, Nk, H, d, argmax};
    run_units(top1_unit, &A, Nq * Hq, nthreads);
    return 0;
}

/* ------------------------------------------------------------------ */
/* QuantWM statistics and PSAC basis.                                  */
/* ------------------------------------------------------------------ */

/*
 * History-query statistics ([QWM] QSAC: per-channel query activity; PSAC:
 * second-moment matrix of the history queries).  Readings: the activity of
 * channel j is E[q_j^2]; a KV head's statistics pool the query heads that
 * read it (query head hq reads KV head hq / (Hq/H)).  M [H][d][d] is
 * accumulated in place in fp64 (M += sum q q^T); count[0] += n * Hq/H.
 */
int orc_query_stats(const float *q, int n, int Hq, int H, int d, double *M,
                    int64_t *count) {
    if (H < 1 || Hq % H != 0) return -1;
    const int grp = Hq / H;
    for (int hq = 0; hq < Hq; ++hq) {
        double *Mh = M + (size_t)(hq / grp) * d * d;
        for (int t = 0; t < n; ++t) {
            const float *qr = q + ((size_t)t * Hq + hq) * d;
            for (int a = 0; a < d; ++a)
                for (int b = 0; b < d; ++b)
                    Mh[(size_t)a * d + b] += (double)qr[a] * (double)qr[b];
        }
    }
    count[0] += (int64_t)n * grp;
    return 0;
}

/*
 * Cyclic Jacobi eigenvalue method for a symmetric d x d matrix (Golub & Van
 * Loan, "Matrix Computations", cyclic Jacobi with the stable rotation of
 * Rutishauser): sweep the pairs (p, q), p < q, in row order and annihilate
 * a_pq; stop when off(A) <= tol * ||A||_F or after max_sweeps.
 * On return evals are sorted descending and column k of vecs (d x d,
 * row-major) is the eigenvector of evals[k], sign fixed so that its
 * largest-magnitude component (lowest index on ties) is positive.
 * Returns the number of sweeps used.
 */
int orc_jacobi(const double *Min, int d, double tol, int max_sweeps,
               double *evals, double *vecs) {
    double *A = (double *)malloc(sizeof(double) * (size_t)d * d);
    double *V = (double *)calloc((size_t)d * d, sizeof(double));
    memcpy(A, Min, sizeof(double) * (size_t)d * d);
    for (int i = 0; i < d; ++i) V[(size_t)i * d + i] = 1.0;
    double fro = 0.0;
    for (size_t i = 0; i < (size_t)d * d; ++i) fro += A[i] * A[i];
    fro = sqrt(fro);
    int sweep = 0;
    for (; sweep < max_sweeps; ++sweep) {
        double off = 0.0;
        for (int p = 0; p < d; ++p)
            for (int q = 0; q < d; ++q)
                if (p != q) off += A[(size_t)p * d + q] * A[(size_t)p * d + q];
        if (sqrt(off) <= tol * fro) break;
        for (int p = 0; p < d - 1; ++p)
            for (int q = p + 1; q < d; ++q) {
                const double apq = A[(size_t)p * d + q];
                if (apq == 0.0) continue;
                const double app = A[(size_t)p * d + p], aqq = A[(size_t)q * d + q];
                const double theta = (aqq - app) / (2.0 * apq);
                const double t = (theta >= 0.0 ? 1.0 : -1.0) /
                                 (fabs(theta) + sqrt(1.0 + theta * theta));
                const double c = 1.0 / sqrt(1.0 + t * t), s = t * c;
                /* A <- J^T A J with J the rotation in the (p, q) plane. */
                for (int k = 0; k < d; ++k) {
                    const double akp = A[(size_t)k * d + p], akq = A[(size_t)k * d + q];
                    A[(size_t)k * d + p] = c * akp - s * akq;
                    A[(size_t)k * d + q] = s * akp + c * akq;
                }
                for (int k = 0; k < d; ++k) {
                    const double apk = A[(size_t)p * d + k], aqk = A[(size_t)q * d + k];
                    A[(size_t)p * d + k] = c * apk - s * aqk;
                    A[(size_t)q * d + k] = s * apk + c * aqk;
                }
                for (int k = 0; k < d; ++k) {
                    const double vkp = V[(size_t)k * d + p], vkq = V[(size_t)k * d + q];
                    V[(size_t)k * d + p] = c * vkp - s * vkq;
                    V[(size_t)k * d + q] = s * vkp + c * vkq;
                }
            }
    }
    /* Sort eigenpairs by eigenvalue, descending (selection sort, stable). */
    int *ord = (int *)malloc(sizeof(int) * (size_t)d);
    for (int i = 0; i < d; ++i) ord[i] = i;
    for (int i = 0; i < d; ++i) {
        int b = i;
        for (int k = i + 1; k < d; ++k)
            if (A[(size_t)ord[k] * d + ord[k]] > A[(size_t)ord[b] * d + ord[b]]) b = k;
        const int tmp = ord[i]; ord[i] = ord[b]; ord[b] = tmp;
    }
    for (int i = 0; i < d; ++i) {
        const int src = ord[i];
        evals[i] = A[(size_t)src * d + src];
        int big = 0;
        for (int k = 1; k < d; ++k)
            if (fabs(V[(size_t)k * d + src]) > fabs(V[(size_t)big * d + src])) big = k;
        const double sg = V[(size_t)big * d + src] < 0.0 ? -1.0 : 1.0;
        for (int k = 0; k < d; ++k) vecs[(size_t)k * d + i] = sg * V[(size_t)k * d + src];
    }
    free(ord); free(A); free(V);
    return sweep;
}

/*
 * PSAC basis ([QWM] PSAC: eigendecompose the history-query second moment,
 * keep the top-8 eigenvectors as the principal subspace; the page reports
 * the share of query energy they hold).  M [H][d][d] are sums of q q^T;
 * the basis is that of M / count (scaling does not move eigenvectors).
 * U [H][d][r] (column k = k-th eigenvector), eig [H][r] eigenvalues of
 * M / count, frac [H] = sum of the top-r eigenvalues / trace.
 */
int orc_psac_basis(const double *M, int64_t count, int H, int d, int r,
                   double *U, double *eig, double *frac) {
    if (r < 1 || r > d || count < 1) return -1;
    double *ev = (double *)malloc(sizeof(double) * (size_t)d);
    double *vec = (double *)malloc(sizeof(double) * (size_t)d * d);
    double *Mn = (double *)malloc(sizeof(double) * (size_t)d * d);
    for (int h = 0; h < H; ++h) {
        for (size_t i = 0; i < (size_t)d * d; ++i)
            Mn[i] = M[(size_t)h * d * d + i] / (double)count;
        orc_jacobi(Mn, d, 1e-12, 100, ev, vec);
        double tr = 0.0, top = 0.0;
        for (int i = 0; i < d; ++i) tr += Mn[(size_t)i * d + i];
        for (int k = 0; k < r; ++k) {
            eig[(size_t)h * r + k] = ev[k];
            top += ev[k];
            for (int j = 0; j < d; ++j)
                U[((size_t)h * d + j) * r + k] = vec[(size_t)j * d + k];
        }
        frac[h] = (tr > 0.0) ? top / tr : 0.0;
    }
    free(ev); free(vec); free(Mn);
    return 0;
}
