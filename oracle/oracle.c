/*
 * ORACLE for the int4-g128 weight-streaming GEMV.  TEST INFRASTRUCTURE ONLY:
 * only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may
 * load this library.  The product path (int4_weight_only_g128_gb300) never
 * calls it and shares no code with it.
 *
 * What it computes, written out as the plain definition in fp64:
 *
 *   Format (Token Rush README, intro bullet "4.25 bits per weight" and the
 *   "Quantization" section): group-wise asymmetric int4, 128 consecutive
 *   K-weights of a column share one bf16 scale and one bf16 minimum,
 *        w[k][n] = min[k/128][n] + q[k][n] * scale[k/128][n],  q in 0..15,
 *   which costs 4 + 32/128 = 4.25 bits per weight.
 *
 *   Product (Token Rush README, "bandwidth ceiling" paragraph: every decode
 *   step reads all weights once; the M-row verify of the progress table,
 *   steps 13-14 and 28):
 *        y[m][n] = sum_k x[m][k] * w[k][n],   m < M <= 8,
 *   with bf16 x and bf16 y.  The oracle keeps y in fp64 (no output rounding)
 *   and sums in ascending k.  It also returns a[m][n] = sum_k |x[m][k]*w[k][n]|,
 *   the scale of the acceptance bound |y_gpu - y| <= 4e-3*a + ulp_bf16(y).
 *
 * Readings the pages leave open:
 *   - canonical code order: code k = 8j+i sits in bits 4i..4i+3 of word j of
 *     column n, words stored [K/8][N] row-major;
 *   - a group is 128 consecutive k of one column, k in [128g, 128g+128);
 *   - "minimum" is an additive bf16 offset, not an integer zero point.
 *
 * Every bf16 -> double widening is exact, every dequantised weight is exact
 * in fp64 (<= 12 significant bits in the product, well inside 53), so the
 * only rounding in y is the fp64 summation.
 *
 * The tiled device layout (oracle_pack_tiled) is this library's own
 * restatement of the packed format that include/w4g128.h specifies in prose;
 * it is written from that specification and shares no code with the device
 * packer.
 *
 * oracle_add_rmsnorm (at the end) folds the product into the residual add and
 * RMS normalisation that follow it in the model (its own header there).
 *
 * The quantizer (oracle_quantize, below) chooses codes, scales and minimums
 * from bf16 weights: round-to-nearest on the 16-level grid of each group,
 * optionally with a range search that clips outliers (its own header below).
 *
 * Mutants for negative-control tests (compile with -DORACLE_MUTANT=n):
 *   1 = nibbles read in reversed order within a word,
 *   2 = group index off by one (k = 128g is assigned to group g-1),
 *   3 = the minimum term dropped,
 *   4 = quantizer rounds toward zero instead of to nearest,
 *   5 = quantizer spreads the range over 16 steps instead of 15,
 *   6 = quantizer keeps the candidate with the largest error,
 *   7, 8, 9 = mistakes in the residual add and RMS norm (listed there).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

/* ---- bf16 ------------------------------------------------------------- */

/* bf16 bit pattern -> exact double (bf16 is the top half of an fp32). */
static double bf16_val(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

double oracle_bf16_value(uint16_t h) { return bf16_val(h); }

/* Round a double to the nearest bf16 (ties to even), returning the bits.
 * bf16 keeps 8 significant bits; its normal range is 2^-126 .. (2-2^-7)*2^127
 * and its subnormals are multiples of 2^-133. */
uint16_t oracle_bf16_rn(double v) {
    if (isnan(v)) return 0x7FC0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);                    /* a = f * 2^e, f in [0.5, 1) */
    int ex = e - 1;                  /* floor(log2 a) */
    if (ex < -126) ex = -126;        /* subnormal quantum is 2^-133 */
    double quantum = ldexp(1.0, ex - 7);
    double r = nearbyint(a / quantum) * quantum;  /* a/quantum is exact; ties to even */
    if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80);
    float f = (float)r;              /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(sign | (u >> 16));
}

/* oracle_bf16_rn over an array (for comparing whole outputs bit for bit). */
void oracle_bf16_rn_array(const double* v, size_t n, uint16_t* out) {
    for (size_t i = 0; i < n; i++) out[i] = oracle_bf16_rn(v[i]);
}

/* One unit in the last place of bf16 at v: 2^(max(floor(log2|v|), -126) - 7);
 * 2^-133 at v = 0. */
double oracle_bf16_ulp(double v) {
    double a = fabs(v);
    if (a == 0.0) return ldexp(1.0, -133);
    int e;
    frexp(a, &e);
    int ex = e - 1;
    if (ex < -126) ex = -126;
    return ldexp(1.0, ex - 7);
}

/* ---- canonical codes ---------------------------------------------------- */

static int code_at(const uint32_t* codes, int N, int k, int n) {
    uint32_t word = codes[(size_t)(k / 8) * (size_t)N + (size_t)n];
    int i = k % 8;
#if ORACLE_MUTANT == 1
    i = 7 - i;
#endif
    return (int)((word >> (4 * i)) & 0xFu);
}

static int group_of(int k) {
#if ORACLE_MUTANT == 2
    return k == 0 ? 0 : (k - 1) / 128;
#else
    return k / 128;
#endif
}

/* q[K][N] (values 0..15) -> codes[K/8][N]. */
void oracle_pack_canonical(const uint8_t* q, int K, int N, uint32_t* codes) {
    for (int j = 0; j < K / 8; j++)
        for (int n = 0; n < N; n++) {
            uint32_t w = 0;
            for (int i = 0; i < 8; i++)
                w |= (uint32_t)(q[(size_t)(8 * j + i) * N + n] & 0xF) << (4 * i);
            codes[(size_t)j * N + n] = w;
        }
}

void oracle_unpack_canonical(const uint32_t* codes, int K, int N, uint8_t* q) {
    for (int k = 0; k < K; k++)
        for (int n = 0; n < N; n++)
            q[(size_t)k * N + n] = (uint8_t)code_at(codes, N, k, n);
}

/* ---- dequantise, then multiply ------------------------------------------ */

/* Dequantised weight, exact in fp64. */
static double weight(const uint32_t* codes, const uint16_t* scales, const uint16_t* mins,
                     int N, int k, int n) {
    int g = group_of(k);
    double s = bf16_val(scales[(size_t)g * N + n]);
    double mn = bf16_val(mins[(size_t)g * N + n]);
    double q = (double)code_at(codes, N, k, n);
#if ORACLE_MUTANT == 3
    mn = 0.0;
#endif
    return mn + q * s;
}

/* y[M][N] = x[M][K] . dequant(W)[K][N] and a[M][N] = sum_k |x w|, fp64,
 * ascending k, one column at a time (the dequantised column is formed in
 * full before it is multiplied).  nthreads <= 0 means "all available". */
void oracle_gemm(int M, int K, int N, const uint16_t* x, const uint32_t* codes,
                 const uint16_t* scales, const uint16_t* mins, double* y, double* a, int nthreads) {
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel num_threads(nthreads)
#endif
    {
        double* col = (double*)malloc(sizeof(double) * (size_t)K);
        double* xd = (double*)malloc(sizeof(double) * (size_t)K * (size_t)M);
        for (size_t i = 0; i < (size_t)K * (size_t)M; i++) xd[i] = bf16_val(x[i]);
#ifdef _OPENMP
#pragma omp for schedule(static)
#endif
        for (int n = 0; n < N; n++) {
            for (int k = 0; k < K; k++) col[k] = weight(codes, scales, mins, N, k, n);
            for (int m = 0; m < M; m++) {
                const double* xm = xd + (size_t)m * K;
                double acc = 0.0, abs_acc = 0.0;
                for (int k = 0; k < K; k++) {
                    double p = xm[k] * col[k];
                    acc += p;
                    abs_acc += fabs(p);
                }
                y[(size_t)m * N + n] = acc;
                if (a) a[(size_t)m * N + n] = abs_acc;
            }
        }
        free(col);
        free(xd);
    }
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---- the tiled device layout, restated from its specification ------------ */
/*
 * Specification (include/w4g128.h, "packed layout"): K % 128 == 0, N % 16 == 0,
 * G = K/128 groups, T = N/16 column tiles, quads of 4 tiles, quad q holding
 * nt(q) = min(4, T - 4q) tiles.  Block (t, g) is 1088 bytes at offset
 * q*G*4352 + g*nt(q)*1088 + i*1088 with q = t/4, i = t%4.  Bytes [0, 1024)
 * hold codes: half h (0, 1) at 512*h, lane l (0..31) at +16*l, little-endian
 * word j (0..3) at +4*j.  With r = l / 4 and c = l % 4, word j covers rows
 * k0 = 128g + 64h + 16j and holds in nibble p = 4*b + 2*a + e (bits 4p..4p+3)
 * the code of row k0 + 2c + 8a + b of column 16t + r + 8e.  Bytes
 * [1024, 1088) hold 8 entries of 8 bytes; entry r has the little-endian bf16
 * values scale, min of column 16t + r and scale, min of column 16t + r + 8,
 * all for group g.
 */

static size_t block_offset(int t, int g, int G, int T) {
    int q = t / 4, i = t % 4;
    int nt = T - 4 * q < 4 ? T - 4 * q : 4;
    return (size_t)q * (size_t)G * 4352u + (size_t)g * (size_t)nt * 1088u + (size_t)i * 1088u;
}

size_t oracle_packed_bytes(int K, int N) {
    return (size_t)(N / 16) * (size_t)(K / 128) * 1088u;
}

static void put_u16(uint8_t* p, uint16_t v) { p[0] = (uint8_t)(v & 0xFF); p[1] = (uint8_t)(v >> 8); }
static uint16_t get_u16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }

void oracle_pack_tiled(const uint32_t* codes, const uint16_t* scales, const uint16_t* mins,
                       int K, int N, uint8_t* out) {
    int G = K / 128, T = N / 16;
    for (int t = 0; t < T; t++)
        for (int g = 0; g < G; g++) {
            uint8_t* blk = out + block_offset(t, g, G, T);
            for (int h = 0; h < 2; h++)
                for (int l = 0; l < 32; l++) {
                    int r = l / 4, c = l % 4;
                    for (int j = 0; j < 4; j++) {
                        int k0 = 128 * g + 64 * h + 16 * j;
                        uint32_t word = 0;
                        for (int p = 0; p < 8; p++) {
                            int b = (p >> 2) & 1, a = (p >> 1) & 1, e = p & 1;
                            int k = k0 + 2 * c + 8 * a + b;
                            int n = 16 * t + r + 8 * e;
                            uint32_t q = (codes[(size_t)(k / 8) * N + n] >> (4 * (k % 8))) & 0xFu;
                            word |= q << (4 * p);
                        }
                        uint8_t* wp = blk + 512 * h + 16 * l + 4 * j;
                        wp[0] = (uint8_t)(word & 0xFF);
                        wp[1] = (uint8_t)((word >> 8) & 0xFF);
                        wp[2] = (uint8_t)((word >> 16) & 0xFF);
                        wp[3] = (uint8_t)(word >> 24);
                    }
                }
            for (int r = 0; r < 8; r++) {
                uint8_t* e = blk + 1024 + 8 * r;
                size_t lo = (size_t)g * N + 16 * t + r, hi = lo + 8;
                put_u16(e + 0, scales[lo]);
                put_u16(e + 2, mins[lo]);
                put_u16(e + 4, scales[hi]);
                put_u16(e + 6, mins[hi]);
            }
        }
}

void oracle_unpack_tiled(const uint8_t* packed, int K, int N, uint32_t* codes,
                         uint16_t* scales, uint16_t* mins) {
    int G = K / 128, T = N / 16;
    memset(codes, 0, sizeof(uint32_t) * (size_t)(K / 8) * N);
    for (int t = 0; t < T; t++)
        for (int g = 0; g < G; g++) {
            const uint8_t* blk = packed + block_offset(t, g, G, T);
            for (int h = 0; h < 2; h++)
                for (int l = 0; l < 32; l++) {
                    int r = l / 4, c = l % 4;
                    for (int j = 0; j < 4; j++) {
                        const uint8_t* wp = blk + 512 * h + 16 * l + 4 * j;
                        uint32_t word = (uint32_t)wp[0] | ((uint32_t)wp[1] << 8) |
                                        ((uint32_t)wp[2] << 16) | ((uint32_t)wp[3] << 24);
                        int k0 = 128 * g + 64 * h + 16 * j;
                        for (int p = 0; p < 8; p++) {
                            int b = (p >> 2) & 1, a = (p >> 1) & 1, e = p & 1;
                            int k = k0 + 2 * c + 8 * a + b;
                            int n = 16 * t + r + 8 * e;
                            uint32_t q = (word >> (4 * p)) & 0xFu;
                            codes[(size_t)(k / 8) * N + n] |= q << (4 * (k % 8));
                        }
                    }
                }
            for (int r = 0; r < 8; r++) {
                const uint8_t* e = blk + 1024 + 8 * r;
                size_t lo = (size_t)g * N + 16 * t + r, hi = lo + 8;
                scales[lo] = get_u16(e + 0);
                mins[lo] = get_u16(e + 2);
                scales[hi] = get_u16(e + 4);
                mins[hi] = get_u16(e + 6);
            }
        }
}

/* ---- quantizer ------------------------------------------------------------
 *
 * From bf16 weights w[K][N] (row-major) to the canonical format: codes
 * [K/8][N], scales and minimums [K/128][N].  Token Rush README, section
 * "Quantization": group-wise asymmetric int4, 128 weights per bf16 scale and
 * minimum; the round-to-nearest row of the quality table; and "an MSE range
 * search per group that clips a few outliers to buy precision for the rest".
 * The pages give no formulas.  Reading taken (the plainest one):
 *
 *   For one group (column n, rows 128g .. 128g+127), lo = min w, hi = max w.
 *   A candidate p in (0, 1] spans [a, b] = [p*lo, p*hi] with 15 equal steps:
 *       s = (b - a) / 15,  sb = bf16(s),  mb = bf16(a),
 *       q_k = clamp(round_half_even((w_k - mb) / sb), 0, 15)   (q = 0 if sb == 0),
 *       e = sum over k ascending of (w_k - (mb + q_k * sb))^2.
 *   Round-to-nearest is the single candidate p = 1.  The range search tries
 *   p = (100 - i) / 100 for i = 0 .. 20 and keeps the candidate with the
 *   smallest e (the first one, i.e. the widest range, on ties).
 *
 * Every step is one IEEE fp32 operation rounded to nearest (no fused
 * multiply-add): where the result is an integer decision (a code, the chosen
 * candidate) both this oracle and the device kernel must take it in the same
 * precision, and fp32 is the plainest precision for bf16 data.  bf16(.) is
 * round-to-nearest-even of an fp32 value.
 */
#define QUANT_CANDIDATES 21

static float f32_of_bf16(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

static float bf16_round_f32(float v) { return f32_of_bf16(oracle_bf16_rn((double)v)); }

static int code_of(float w, float mb, float sb) {
    if (sb == 0.0f) return 0;
    volatile float d = w - mb;
    volatile float t = d / sb;
#if ORACLE_MUTANT == 4
    float r = truncf(t);
#else
    float r = nearbyintf(t);       /* default rounding mode: ties to even */
#endif
    if (!(r > 0.0f)) return 0;     /* also maps -0 and NaN to 0 */
    if (r > 15.0f) return 15;
    return (int)r;
}

/* Quantise one group of 128 fp32 values with candidate p; returns the error
 * and writes the codes and the bf16 scale / minimum. */
static float quant_candidate(const float* w, float lo, float hi, float p, uint8_t* q,
                             float* sb_out, float* mb_out) {
    volatile float a = p * lo;
    volatile float b = p * hi;
    volatile float span = b - a;
#if ORACLE_MUTANT == 5
    volatile float s = span / 16.0f;
#else
    volatile float s = span / 15.0f;
#endif
    float sb = bf16_round_f32(s);
    float mb = bf16_round_f32(a);
    float e = 0.0f;
    for (int k = 0; k < 128; k++) {
        q[k] = (uint8_t)code_of(w[k], mb, sb);
        volatile float prod = (float)q[k] * sb;
        volatile float dq = mb + prod;
        volatile float r = w[k] - dq;
        volatile float r2 = r * r;
        e = e + r2;
    }
    *sb_out = sb;
    *mb_out = mb;
    return e;
}

/* errs (optional): per group and candidate, the error e, [G][N][21]. */
void oracle_quantize(const uint16_t* w, int K, int N, int search, uint32_t* codes,
                     uint16_t* scales, uint16_t* mins, float* errs) {
    int G = K / 128;
    memset(codes, 0, sizeof(uint32_t) * (size_t)(K / 8) * N);
    #pragma omp parallel for schedule(static)
    for (long gn = 0; gn < (long)G * N; gn++) {
        int g = (int)(gn / N), n = (int)(gn % N);
        float v[128];
        float lo = 0.0f, hi = 0.0f;
        for (int k = 0; k < 128; k++) {
            v[k] = f32_of_bf16(w[(size_t)(128 * g + k) * N + n]);
            if (k == 0 || v[k] < lo) lo = v[k];
            if (k == 0 || v[k] > hi) hi = v[k];
        }
        int ncand = search ? QUANT_CANDIDATES : 1;
        uint8_t q[128], best_q[128];
        float best_e = 0.0f, best_s = 0.0f, best_m = 0.0f;
        for (int i = 0; i < ncand; i++) {
            volatile float num = (float)(100 - i);
            float p = num / 100.0f;
            float sb, mb;
            float e = quant_candidate(v, lo, hi, p, q, &sb, &mb);
            if (errs) errs[(size_t)gn * QUANT_CANDIDATES + i] = e;
#if ORACLE_MUTANT == 6
            int better = (i == 0) || (e >= best_e);
#else
            int better = (i == 0) || (e < best_e);
#endif
            if (better) {
                best_e = e;
                best_s = sb;
                best_m = mb;
                memcpy(best_q, q, 128);
            }
        }
        for (int k = 0; k < 128; k++) {
            int kk = 128 * g + k;
            codes[(size_t)(kk / 8) * N + n] |= (uint32_t)best_q[k] << (4 * (kk % 8));
        }
        scales[(size_t)g * N + n] = oracle_bf16_rn((double)best_s);
        mins[(size_t)g * N + n] = oracle_bf16_rn((double)best_m);
    }
}

/* ---- the product folded into the residual add and RMS norm -------------
 *
 * Token Rush README, progress table steps 8-9: the split-K GEMV's partial
 * sums are added up inside the normalisation that follows the projection,
 * not in a pass of their own.  The pages name the norm and nothing more; the
 * reading taken here is the pre-norm transformer's residual update followed by
 * RMS normalisation (Zhang and Sennrich, "Root Mean Square Layer
 * Normalization", 2019), per output row m over the N columns:
 *
 *   h[m][n]   = residual[m][n] + y[m][n]            (the new residual stream)
 *   out[m][n] = gamma[n] * h[m][n] / sqrt( (1/N) sum_j h[m][j]^2 + eps )
 *
 * y is the product computed above (fp64, not rounded); residual and gamma are
 * bf16, eps a non-negative real.  Everything is fp64, summed in ascending j;
 * neither h nor out is rounded to bf16 here.
 *
 * Mutants: 7 = mean taken over N - 1 columns, 8 = eps dropped,
 *          9 = residual not added.
 */
void oracle_add_rmsnorm(int M, int N, const double* y, const uint16_t* residual, const uint16_t* gamma,
                        double eps, double* h, double* out) {
    for (int m = 0; m < M; m++) {
        const size_t row = (size_t)m * (size_t)N;
        double ss = 0.0;
        for (int n = 0; n < N; n++) {
            double r = bf16_val(residual[row + n]);
#if ORACLE_MUTANT == 9
            r = 0.0;
#endif
            const double v = r + y[row + n];
            h[row + n] = v;
            ss += v * v;
        }
        double cols = (double)N;
#if ORACLE_MUTANT == 7
        cols = (double)(N - 1);
#endif
        double e = eps;
#if ORACLE_MUTANT == 8
        e = 0.0;
#endif
        const double inv_rms = 1.0 / sqrt(ss / cols + e);
        for (int n = 0; n < N; n++) out[row + n] = bf16_val(gamma[n]) * (h[row + n] * inv_rms);
    }
}
