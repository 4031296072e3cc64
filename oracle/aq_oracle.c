/*
 * Reference oracle for the affine group-64 quantized matmul y = x . W^T.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is used by tests/, by the smoke check
 * and by the CPU-baseline leg of bench.py.  The product library never links,
 * loads or calls it, and it shares no code with the CUDA path.
 *
 * It is plain, slow and written to be checked by eye against the definition
 * of the format on the mlx-bun pages (@mlx-bun/inference 1.0.0,
 * kernels/quantization/*):
 *
 *  - affine-split-mma.ts, helper affine_unit: value v of a 64-value group is
 *    bits [v*B, v*B + B) of the group's LSB-first bit stream, and may straddle
 *    two 32-bit words;
 *  - affine3-mma.ts / affine4-mma.ts (helpers affine_q3 / affine_q4): a group
 *    is 2*B consecutive uint32 words, so a row of K values is K*B/32 words;
 *  - affine3-rows.ts / affine4-rows.ts header comments: eight 3-bit values in
 *    three little-endian bytes, eight 4-bit values per little-endian word;
 *  - every kernel: scales and biases are [N, K/64], and a weight is
 *    w = scale * q + bias (the mma kernels' fma(s, q, b)).
 *
 * All floating-point arithmetic is in double precision, summing over k in
 * ascending order.  Inputs arrive as doubles: the fp16 / bf16 values of x,
 * scales and biases widen to double exactly, so nothing is lost on the way in.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_GROUP 64

static int valid_shape(int64_t N, int64_t K, int bits) {
    if (N < 0 || K < 0) return 0;
    if (K % ORACLE_GROUP != 0) return 0;
    if (bits != 3 && bits != 4) return 0;
    return 1;
}

/*
 * Other code widths and group sizes (the "_g" functions below): B in
 * {2,3,4,5,6,8} and groups of 32, 64 or 128 values.  The bit stream is the
 * same LSB-first stream per row (code v at bits [v*B, v*B+B)), which needs
 * K*B to be a multiple of 32; scales and biases are [N][K/group].  The pages'
 * fused-decode kernel takes 4 and 8 bits with groups of 32, 64 and 128.
 */
static int valid_bits(int bits) {
    return bits == 2 || bits == 3 || bits == 4 || bits == 5 || bits == 6 || bits == 8;
}

static int valid_shape_g(int64_t N, int64_t K, int bits, int group) {
    if (N < 0 || K < 0 || !valid_bits(bits)) return 0;
    if (group != 32 && group != 64 && group != 128) return 0;
    return K % group == 0;
}

/* Words per row: K values of B bits each, 32 bits per word. */
int64_t oracle_words_per_row(int64_t K, int bits) { return K * bits / 32; }

/*
 * Pack: code v of a row becomes bits [v*B, v*B+B) of the row's bit stream;
 * stream bit i lives in word i/32 at bit i%32 (least significant first).
 * Only the low B bits of each code are used.
 */
static void pack_rows(const uint8_t *codes, int64_t N, int64_t K, int bits, uint32_t *words) {
    const int64_t wpr = oracle_words_per_row(K, bits);
    const uint32_t mask = (1u << bits) - 1u;
    memset(words, 0, (size_t)(N * wpr) * sizeof(uint32_t));
    for (int64_t n = 0; n < N; ++n) {
        uint32_t *row = words + n * wpr;
        for (int64_t v = 0; v < K; ++v) {
            const uint32_t q = codes[n * K + v] & mask;
            const int64_t bit = v * bits;
            const int64_t w = bit / 32;
            const int off = (int)(bit % 32);
            row[w] |= q << off;
            if (off + bits > 32) row[w + 1] |= q >> (32 - off);
        }
    }
}

int oracle_pack(const uint8_t *codes, int64_t N, int64_t K, int bits, uint32_t *words) {
    if (!valid_shape(N, K, bits)) return 1;
    pack_rows(codes, N, K, bits, words);
    return 0;
}

/* Any width of valid_bits, K a multiple of 32. */
int oracle_pack_g(const uint8_t *codes, int64_t N, int64_t K, int bits, uint32_t *words) {
    if (!valid_shape_g(N, K, bits, 32)) return 1;
    pack_rows(codes, N, K, bits, words);
    return 0;
}

/* Code v of row n, read back from the bit stream (the inverse of pack). */
static uint32_t oracle_code(const uint32_t *row, int64_t v, int bits) {
    const int64_t bit = v * bits;
    const int64_t w = bit / 32;
    const int off = (int)(bit % 32);
    uint32_t q = row[w] >> off;
    if (off + bits > 32) q |= row[w + 1] << (32 - off);
    return q & ((1u << bits) - 1u);
}

static void unpack_rows(const uint32_t *words, int64_t N, int64_t K, int bits, uint8_t *codes) {
    const int64_t wpr = oracle_words_per_row(K, bits);
    for (int64_t n = 0; n < N; ++n)
        for (int64_t v = 0; v < K; ++v)
            codes[n * K + v] = (uint8_t)oracle_code(words + n * wpr, v, bits);
}

int oracle_unpack(const uint32_t *words, int64_t N, int64_t K, int bits, uint8_t *codes) {
    if (!valid_shape(N, K, bits)) return 1;
    unpack_rows(words, N, K, bits, codes);
    return 0;
}

int oracle_unpack_g(const uint32_t *words, int64_t N, int64_t K, int bits, uint8_t *codes) {
    if (!valid_shape_g(N, K, bits, 32)) return 1;
    unpack_rows(words, N, K, bits, codes);
    return 0;
}

/* Dequantise: W[n][k] = scale[n][k/group] * q[n][k] + bias[n][k/group]. */
int oracle_dequant_g(const uint32_t *words, const double *scales, const double *biases,
                     int64_t N, int64_t K, int bits, int group, double *W) {
    if (!valid_shape_g(N, K, bits, group)) return 1;
    const int64_t wpr = oracle_words_per_row(K, bits);
    const int64_t G = K / group;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
            const int64_t g = k / group;
            const double q = (double)oracle_code(words + n * wpr, k, bits);
            W[n * K + k] = scales[n * G + g] * q + biases[n * G + g];
        }
    return 0;
}

int oracle_dequant(const uint32_t *words, const double *scales, const double *biases,
                   int64_t N, int64_t K, int bits, double *W) {
    if (!valid_shape(N, K, bits)) return 1;
    return oracle_dequant_g(words, scales, biases, N, K, bits, ORACLE_GROUP, W);
}

/*
 * One output element and its error scale:
 *   y[m][n]     = sum_k x[m][k] * (scale[n][g(k)] * q[n][k] + bias[n][g(k)])
 *   bound[m][n] = sum_k |x[m][k] * w[n][k]|
 */
static void oracle_element(const double *xrow, const uint32_t *wrow, const double *srow,
                           const double *brow, int64_t K, int bits, int group, double *y,
                           double *bound) {
    double acc = 0.0, mag = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        const int64_t g = k / group;
        const double w = srow[g] * (double)oracle_code(wrow, k, bits) + brow[g];
        const double p = xrow[k] * w;
        acc += p;
        mag += fabs(p);
    }
    *y = acc;
    if (bound) *bound = mag;
}

/* y[M][N] (and bound[M][N] if non-null) for all outputs, single-threaded. */
int oracle_matmul(const double *x, const uint32_t *words, const double *scales,
                  const double *biases, int64_t M, int64_t N, int64_t K, int bits,
                  double *y, double *bound) {
    if (!valid_shape(N, K, bits) || M < 0) return 1;
    const int64_t wpr = oracle_words_per_row(K, bits);
    const int64_t G = K / ORACLE_GROUP;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n)
            oracle_element(x + m * K, words + n * wpr, scales + n * G, biases + n * G, K, bits,
                           ORACLE_GROUP, &y[m * N + n], bound ? &bound[m * N + n] : NULL);
    return 0;
}

/*
 * The same elements for a chosen list of output columns: y[m][j] is output
 * column cols[j].  Used to check sampled outputs of full-size problems.
 */
int oracle_matmul_cols(const double *x, const uint32_t *words, const double *scales,
                       const double *biases, int64_t M, int64_t N, int64_t K, int bits,
                       const int64_t *cols, int64_t ncols, double *y, double *bound) {
    if (!valid_shape(N, K, bits) || M < 0) return 1;
    const int64_t wpr = oracle_words_per_row(K, bits);
    const int64_t G = K / ORACLE_GROUP;
    for (int64_t j = 0; j < ncols; ++j)
        if (cols[j] < 0 || cols[j] >= N) return 1;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t j = 0; j < ncols; ++j) {
            const int64_t n = cols[j];
            oracle_element(x + m * K, words + n * wpr, scales + n * G, biases + n * G, K, bits,
                           ORACLE_GROUP, &y[m * ncols + j], bound ? &bound[m * ncols + j] : NULL);
        }
    return 0;
}

/*
 * Gated MLP input of a decoder layer, h = silu(g) * u, where
 *   g[m][n] = sum_k x[m][k] * w_gate[n][k]   (oracle_element on the gate weights)
 *   u[m][n] = sum_k x[m][k] * w_up[n][k]     (oracle_element on the up weights)
 *   silu(g) = g * sigmoid(g) = g / (1 + exp(-g)).
 * The mlx-bun 0.4.0 -> 1.0.0 page (src/model/trellis-shared-m.ts, the gate/up
 * kernel's epilogue) forms sigmoid(gate) = 1 / (1 + exp(-gate)), multiplies
 * it by gate and the result by up.  The pages round gate, up, the sigmoid and
 * the product to the activation type at every step; the operator itself is
 * the exact value, computed here in double precision from the exact fp64
 * products.  Columns: cols[j] for j < ncols, or every column 0..N-1 in order
 * when cols is NULL (ncols must then be N).  Outputs are [M][ncols]; any of
 * g, u, silu, bound_g, bound_u may be NULL.
 */
int oracle_gate_up_cols(const double *x, const uint32_t *wg, const double *sg, const double *bg,
                        const uint32_t *wu, const double *su, const double *bu, int64_t M,
                        int64_t N, int64_t K, int bits, const int64_t *cols, int64_t ncols,
                        double *h, double *g, double *u, double *silu, double *bound_g,
                        double *bound_u) {
    if (!valid_shape(N, K, bits) || M < 0 || ncols < 0) return 1;
    if (cols == NULL && ncols != N) return 1;
    const int64_t wpr = oracle_words_per_row(K, bits);
    const int64_t G = K / ORACLE_GROUP;
    for (int64_t j = 0; j < ncols; ++j)
        if (cols != NULL && (cols[j] < 0 || cols[j] >= N)) return 1;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t j = 0; j < ncols; ++j) {
            const int64_t n = cols != NULL ? cols[j] : j;
            const int64_t o = m * ncols + j;
            double gv, uv, gb, ub;
            oracle_element(x + m * K, wg + n * wpr, sg + n * G, bg + n * G, K, bits,
                           ORACLE_GROUP, &gv, &gb);
            oracle_element(x + m * K, wu + n * wpr, su + n * G, bu + n * G, K, bits,
                           ORACLE_GROUP, &uv, &ub);
            const double sig = 1.0 / (1.0 + exp(-gv));
            const double sv = gv * sig;
            h[o] = sv * uv;
            if (g) g[o] = gv;
            if (u) u[o] = uv;
            if (silu) silu[o] = sv;
            if (bound_g) bound_g[o] = gb;
            if (bound_u) bound_u[o] = ub;
        }
    return 0;
}

/*
 * Row-parallel form of oracle_matmul: output columns are dealt out to
 * nthreads POSIX threads in contiguous blocks.  Every element is computed by
 * exactly the same oracle_element call, so the result is identical to the
 * single-threaded one.  Used for large parity checks and the CPU baseline.
 */
struct oracle_job {
    const double *x;
    const uint32_t *words;
    const double *scales, *biases;
    int64_t M, N, K;
    int bits, group;
    int64_t n_begin, n_end;
    double *y, *bound;
};

static void *oracle_worker(void *arg) {
    const struct oracle_job *j = (const struct oracle_job *)arg;
    const int64_t wpr = oracle_words_per_row(j->K, j->bits);
    const int64_t G = j->K / j->group;
    for (int64_t m = 0; m < j->M; ++m)
        for (int64_t n = j->n_begin; n < j->n_end; ++n)
            oracle_element(j->x + m * j->K, j->words + n * wpr, j->scales + n * G,
                           j->biases + n * G, j->K, j->bits, j->group, &j->y[m * j->N + n],
                           j->bound ? &j->bound[m * j->N + n] : NULL);
    return NULL;
}

/* y and bound for any width and group size, on nthreads threads. */
int oracle_matmul_g(const double *x, const uint32_t *words, const double *scales,
                    const double *biases, int64_t M, int64_t N, int64_t K, int bits, int group,
                    double *y, double *bound, int nthreads) {
    if (!valid_shape_g(N, K, bits, group) || M < 0) return 1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    pthread_t tid[256];
    int running[256];
    struct oracle_job jobs[256];
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = (struct oracle_job){x, words, scales, biases, M, N, K, bits, group,
                                      N * t / nthreads, N * (t + 1) / nthreads, y, bound};
        running[t] = pthread_create(&tid[t], NULL, oracle_worker, &jobs[t]) == 0;
        if (!running[t]) oracle_worker(&jobs[t]); /* no thread available: run it here */
    }
    for (int t = 0; t < nthreads; ++t)
        if (running[t]) pthread_join(tid[t], NULL);
    return 0;
}

int oracle_matmul_threads(const double *x, const uint32_t *words, const double *scales,
                          const double *biases, int64_t M, int64_t N, int64_t K, int bits,
                          double *y, double *bound, int nthreads) {
    if (!valid_shape(N, K, bits) || M < 0) return 1;
    return oracle_matmul_g(x, words, scales, biases, M, N, K, bits, ORACLE_GROUP, y, bound,
                           nthreads);
}

/* ------------------------------------------------------------------------
 * Quantiser: float weights -> (codes, fp16 scale, fp16 bias) per group.
 *
 * The pages fix the stored format and the dequantisation w = scale*q + bias,
 * but not how a quantiser picks scale, bias and codes.  This is the plain
 * reading, decided in single precision (the precision the GPU kernel decides
 * the codes in, so both sides take the same integer decisions):
 *
 *   lo = min of the group's 64 values, hi = max           (exact)
 *   scale = fp16( (hi - lo) / (2^B - 1) )                 (fp32 ops, RNE)
 *   bias  = fp16( lo )                                    (RNE)
 *   q = clamp( rint((w - bias) / scale), 0, 2^B - 1 )      (fp32 ops, rint
 *                                                          ties to even;
 *                                                          q = 0 if scale = 0)
 *
 * The fp16 conversions below are written from the IEEE 754 binary16
 * definition (11-bit significand, exponent bias 15, subnormal step 2^-24,
 * round to nearest with ties to even, overflow to infinity).
 * ------------------------------------------------------------------------ */

/* binary16 bits -> float (exact). */
float oracle_f16_to_f32(uint16_t h) {
    const int sign = (h >> 15) & 1;
    const int e = (h >> 10) & 0x1F;
    const int m = h & 0x3FF;
    double v;
    if (e == 0x1F)
        v = m ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
    else
        v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
    return (float)(sign ? -v : v);
}

/* float -> binary16 bits, round to nearest, ties to even. */
uint16_t oracle_f32_to_f16(float f) {
    const uint16_t sign = signbit(f) ? 0x8000u : 0u;
    const double a = fabs((double)f);
    if (isnan(f)) return (uint16_t)(sign | 0x7E00u);
    /* 65520 lies halfway between 65504 (largest finite, odd significand) and
       2^16, so it and everything above round to infinity */
    if (a >= 65520.0) return (uint16_t)(sign | 0x7C00u);
    if (a == 0.0) return sign;
    int e2;
    frexp(a, &e2);                    /* a = m * 2^e2, m in [0.5, 1) */
    int e = e2 - 1;                   /* floor(log2 a) */
    if (e < -14) e = -14;             /* subnormal range: fixed quantum 2^-24 */
    const double quantum = ldexp(1.0, e - 10);
    const double r = nearbyint(a / quantum); /* exact quotient; ties to even */
    const double v = r * quantum;     /* the rounded magnitude (may reach 2^(e+1)) */
    if (v < ldexp(1.0, -14)) return (uint16_t)(sign | (uint16_t)r); /* subnormal */
    int ev2;
    const double mv = frexp(v, &ev2); /* v = mv * 2^ev2 */
    const int ev = ev2 - 1;
    const uint16_t mant = (uint16_t)((mv * 2.0 - 1.0) * 1024.0);
    return (uint16_t)(sign | (uint16_t)((ev + 15) << 10) | mant);
}

int oracle_quantize_g(const float *w, int64_t N, int64_t K, int bits, int group, uint8_t *codes,
                      uint16_t *scale_bits, uint16_t *bias_bits) {
    if (!valid_shape_g(N, K, bits, group)) return 1;
    const int64_t G = K / group;
    const int qmax = (1 << bits) - 1;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t g = 0; g < G; ++g) {
            const float *wg = w + n * K + g * group;
            float lo = wg[0], hi = wg[0];
            for (int v = 1; v < group; ++v) {
                if (wg[v] < lo) lo = wg[v];
                if (wg[v] > hi) hi = wg[v];
            }
            const float range = hi - lo;
            const float scale32 = range / (float)qmax;
            const uint16_t sb = oracle_f32_to_f16(scale32);
            const uint16_t bb = oracle_f32_to_f16(lo);
            scale_bits[n * G + g] = sb;
            bias_bits[n * G + g] = bb;
            const float s = oracle_f16_to_f32(sb);
            const float b = oracle_f16_to_f32(bb);
            for (int v = 0; v < group; ++v) {
                int q = 0;
                if (s != 0.0f) {
                    const float t = (wg[v] - b) / s;
                    const float r = rintf(t);
                    q = r < 0.0f ? 0 : r > (float)qmax ? qmax : (int)r;
                }
                codes[n * K + g * group + v] = (uint8_t)q;
            }
        }
    return 0;
}

int oracle_quantize(const float *w, int64_t N, int64_t K, int bits, uint8_t *codes,
                    uint16_t *scale_bits, uint16_t *bias_bits) {
    if (!valid_shape(N, K, bits)) return 1;
    return oracle_quantize_g(w, N, K, bits, ORACLE_GROUP, codes, scale_bits, bias_bits);
}

/* ------------------------------------------------------------------------
 * Decode attention over a quantised KV cache (one query row per head):
 *
 *   s[h][n] = sum_d q[h][d] * Kd[kv][n][d],   kv = h / (H / KV)
 *   p[h][n] = exp(s[h][n] - max_n s[h][n]) / sum_n exp(...)
 *   o[h][d] = sum_n p[h][n] * Vd[kv][n][d]
 *
 * with Kd, Vd the caches dequantised as scale * q + bias per group of
 * `group` values along d (rows [KV][N], D values each, packed as the weight
 * format: K*B/32 words per row, LSB-first).  This is the operator of the
 * fused decode kernel of the mlx-bun 0.0.4 page
 * (src/model/fused-decode-kernel.ts: L = 1, quantised K and V,
 * grouped-query heads), taken as its plain definition in fp64; the
 * query is used as given (any 1/sqrt(D) is the caller's).  Also returned,
 * for the tolerance: smag[h][n] = sum_d |q*Kd| and vmag[h][d] =
 * sum_n p * |Vd|.
 * ------------------------------------------------------------------------ */
int oracle_attention(const double *q, const uint32_t *kw, const double *ks, const double *kb,
                     const uint32_t *vw, const double *vs, const double *vb, int64_t H,
                     int64_t KV, int64_t N, int64_t D, int bits, int group, double *o,
                     double *smag, double *vmag) {
    if (H < 1 || KV < 1 || H % KV != 0 || N < 1 || !valid_shape_g(KV * N, D, bits, group))
        return 1;
    const int64_t wpr = oracle_words_per_row(D, bits);
    const int64_t G = D / group;
    double *s = (double *)malloc((size_t)N * sizeof(double));
    if (!s) return 1;
    for (int64_t h = 0; h < H; ++h) {
        const int64_t kv = h / (H / KV);
        const double *qh = q + h * D;
        double mx = -INFINITY;
        for (int64_t n = 0; n < N; ++n) {
            const int64_t r = kv * N + n;
            double acc = 0.0, mag = 0.0;
            for (int64_t d = 0; d < D; ++d) {
                const double kd = ks[r * G + d / group] * (double)oracle_code(kw + r * wpr, d, bits) +
                                  kb[r * G + d / group];
                acc += qh[d] * kd;
                mag += fabs(qh[d] * kd);
            }
            s[n] = acc;
            if (smag) smag[h * N + n] = mag;
            if (acc > mx) mx = acc;
        }
        double den = 0.0;
        for (int64_t n = 0; n < N; ++n) {
            s[n] = exp(s[n] - mx);
            den += s[n];
        }
        for (int64_t d = 0; d < D; ++d) {
            double acc = 0.0, mag = 0.0;
            for (int64_t n = 0; n < N; ++n) {
                const int64_t r = kv * N + n;
                const double vd = vs[r * G + d / group] * (double)oracle_code(vw + r * wpr, d, bits) +
                                  vb[r * G + d / group];
                const double p = s[n] / den;
                acc += p * vd;
                mag += p * fabs(vd);
            }
            o[h * D + d] = acc;
            if (vmag) vmag[h * D + d] = mag;
        }
    }
    free(s);
    return 0;
}
