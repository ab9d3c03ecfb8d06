/*
 * qlin oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct CPU statement of what the quantized linear
 * layer computes.  Only the test-suite, the smoke check and the CPU-baseline
 * leg of the benchmark may load this library; the product path never does.
 * It shares no code, header or table with the CUDA library.
 *
 * Sources (web pages; section names as printed on each page):
 *  [LP]  "Low-precision LLM inference: FP8/INT8/INT4/FP4 kernels and
 *         calibration" (blog.ruahverce.com, post 68)
 *        S1  precision manifest: accumulate in a wider type, output BF16
 *        S2  Uniform Integer Quantization: q = clamp(round(x/s)+z, qmin, qmax),
 *            x_hat = s(q - z)
 *        S3  Symmetric (z = 0, s = max|x|/qmax) and Asymmetric (range from the
 *            observed min/max)
 *        S4  granularity: per-tensor, per-token/row, per-group (128 weights)
 *        S5  effective bits b + m/G
 *        S7  FP8 E4M3 = 1 sign, 4 exponent, 3 mantissa bits
 *        S8  current scaling: scale = amax / max_representable_fp8
 *        S22 accumulator precision
 *  [TP]  "Quantization throughput by batch size: why W4A16 is overtaken by
 *         W8A8" (hrletsgo.me) -- roofline arithmetic only (not in this file).
 *
 * Readings of points the pages leave open (each also listed in the design
 * notes): asymmetric s = (hi-lo)/15 with the range widened to include 0,
 * z = clamp(rint(-lo/s),0,15); round() is round-half-to-even; x/s is an IEEE
 * binary32 division by the stored FP16 scale; a group whose FP16 scale
 * rounds to 0 stores s = 1, z = 0; E4M3 is the OCP "fn" variant (max 448,
 * no infinities) with round-to-nearest-even and saturation; an all-zero FP8
 * row or tensor takes scale 1.
 *
 * Build: gcc -O2 -std=c11 -fopenmp -ffp-contract=off -fPIC -shared
 * (no -ffast-math: every rounding here is the IEEE one).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* Number formats, written from their definitions.                      */
/* ------------------------------------------------------------------ */

/* bfloat16 is the upper half of an IEEE binary32. */
static float bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* IEEE binary16 -> value. */
double orc_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int m = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);
    return sign ? -v : v;
}

/* binary32 -> IEEE binary16, round to nearest, ties to even; overflow to inf. */
uint16_t orc_f32_to_f16_rn(float f)
{
    uint16_t sign = signbit(f) ? 0x8000 : 0;
    double a = fabs((double)f);
    int e2;
    if (isnan(f))
        return sign | 0x7e00;
    if (isinf(f))
        return sign | 0x7c00;
    if (a == 0.0)
        return sign;
    frexp(a, &e2);          /* a = frac * 2^e2, frac in [0.5, 1) */
    int E = e2 - 1;         /* a = 1.xxx * 2^E */
    if (E < -14) {          /* subnormal range: quantum 2^-24 */
        double r = rint(ldexp(a, 24));
        return sign | (uint16_t)r;       /* r == 1024 is the smallest normal */
    }
    double r = rint(ldexp(a, 10 - E));  /* 11-bit significand in [1024, 2048] */
    if (r == 2048.0) {
        r = 1024.0;
        E += 1;
    }
    if (E > 15)
        return sign | 0x7c00;
    return sign | (uint16_t)((E + 15) << 10) | (uint16_t)(r - 1024.0);
}

/* OCP FP8 E4M3 ("fn"): bias 7, no infinities, S.1111.111 is NaN, max 448. */
double orc_e4m3_to_f64(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 15;
    int m = c & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp((double)(8 + m), e - 10);
    return sign ? -v : v;
}

/* binary32 -> E4M3, round to nearest even, then saturate to +-448. */
uint8_t orc_f32_to_e4m3_rn_sat(float x)
{
    uint8_t sign = signbit(x) ? 0x80 : 0;
    if (isnan(x))
        return sign | 0x7f;
    if (isinf(x))
        return sign | 0x7e;
    double a = fabs((double)x);
    if (a == 0.0)
        return sign;
    int e2;
    frexp(a, &e2);
    int E = e2 - 1;
    if (E < -6) {                          /* subnormal quantum 2^-9 */
        double r = rint(ldexp(a, 9));      /* 0..8; 8 is the smallest normal */
        return sign | (uint8_t)r;
    }
    double r = rint(ldexp(a, 3 - E));      /* 4-bit significand in [8, 16] */
    if (r == 16.0) {
        r = 8.0;
        E += 1;
    }
    if (E + 7 > 15)
        return sign | 0x7e;
    int code = ((E + 7) << 3) | (int)(r - 8.0);
    if (code > 0x7e)                       /* would be the NaN pattern: saturate */
        code = 0x7e;
    return sign | (uint8_t)code;
}

/* ------------------------------------------------------------------ */
/* INT4 weight quantisation, one group of G weights along K per scale.  */
/* [LP] S2 (formula), S3 (symmetric / asymmetric), S4 (per-group).      */
/* ------------------------------------------------------------------ */

/*
 * W    : [N][K] bfloat16 bits
 * q    : [N][K] stored code per weight, one per byte, 0..15
 * s    : [N][K/G] IEEE binary16 bits of the scale
 * z    : [N][K/G] stored zero-point nibble, 0..15
 * Asymmetric: q = clamp(rint(w/s) + z, 0, 15), x_hat = s (q - z).
 * Symmetric : signed code c = clamp(rint(w/s), -8, 7) stored as q = c + 8
 *             with stored zero 8, so that s (q - z) = s c (logical z = 0).
 * Returns the number of groups whose scale overflowed binary16.
 */
int orc_quantize_w4(const uint16_t *W, int64_t N, int64_t K, int G, int symmetric,
                    uint8_t *q, uint16_t *s, uint8_t *z)
{
    int64_t ng = K / G;
    int overflow = 0;
#pragma omp parallel for reduction(+ : overflow) schedule(static)
    for (int64_t n = 0; n < N; n++) {
        for (int64_t g = 0; g < ng; g++) {
            const uint16_t *w = W + n * K + g * G;
            float lo = 0.0f, hi = 0.0f, amax = 0.0f;   /* range widened to include 0 */
            for (int i = 0; i < G; i++) {
                float v = bf16_to_f32(w[i]);
                if (v < lo) lo = v;
                if (v > hi) hi = v;
                if (fabsf(v) > amax) amax = fabsf(v);
            }
            float s32 = symmetric ? amax / 7.0f : (hi - lo) / 15.0f;
            uint16_t s16 = orc_f32_to_f16_rn(s32);
            float sc = (float)orc_f16_to_f64(s16);
            int zp;
            if (sc == 0.0f) {            /* degenerate group */
                s16 = 0x3c00;            /* 1.0 */
                sc = 1.0f;
                zp = symmetric ? 8 : 0;
            } else if (symmetric) {
                zp = 8;
            } else {
                float zf = rintf(-lo / sc);
                if (zf < 0.0f) zf = 0.0f;
                if (zf > 15.0f) zf = 15.0f;
                zp = (int)zf;
            }
            if (isinf(sc))
                overflow += 1;
            s[n * ng + g] = s16;
            z[n * ng + g] = (uint8_t)zp;
            for (int i = 0; i < G; i++) {
                float v = bf16_to_f32(w[i]);
                float r = rintf(v / sc);
                int c;
                if (symmetric) {
                    if (r < -8.0f) r = -8.0f;
                    if (r > 7.0f) r = 7.0f;
                    c = (int)r + 8;
                } else {
                    r = r + (float)zp;
                    if (r < 0.0f) r = 0.0f;
                    if (r > 15.0f) r = 15.0f;
                    c = (int)r;
                }
                q[n * K + g * G + i] = (uint8_t)c;
            }
        }
    }
    return overflow;
}

/* x_hat = s (q - z) for every weight, as double (exact). [LP] S2. */
void orc_dequant_w4(const uint8_t *q, const uint16_t *s, const uint8_t *z,
                    int64_t N, int64_t K, int G, double *Wdeq)
{
    int64_t ng = K / G;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; n++)
        for (int64_t k = 0; k < K; k++) {
            double sc = orc_f16_to_f64(s[n * ng + k / G]);
            Wdeq[n * K + k] = sc * ((double)q[n * K + k] - (double)z[n * ng + k / G]);
        }
}

/*
 * Canonical packed layout (format version 1):
 *   codes [N][K/2]   byte n*K/2 + k/2, low nibble = even k
 *   zeros [N][K/2G]  byte n*(K/G)/2 + g/2, low nibble = even g
 *   scales are already [N][K/G] binary16.
 */
void orc_pack_canonical(const uint8_t *q, const uint8_t *z, int64_t N, int64_t K, int G,
                        uint8_t *codes, uint8_t *zeros)
{
    int64_t ng = K / G;
    memset(codes, 0, (size_t)(N * K / 2));
    memset(zeros, 0, (size_t)((N * ng + 1) / 2));
    for (int64_t n = 0; n < N; n++) {
        for (int64_t k = 0; k < K; k++) {
            uint8_t v = q[n * K + k] & 15;
            codes[n * (K / 2) + k / 2] |= (k % 2 == 0) ? v : (uint8_t)(v << 4);
        }
        for (int64_t g = 0; g < ng; g++) {
            uint8_t v = z[n * ng + g] & 15;
            int64_t idx = n * ng + g;
            zeros[idx / 2] |= (idx % 2 == 0) ? v : (uint8_t)(v << 4);
        }
    }
}

/*
 * Tile layout (format version 2), restated from its written description:
 * tiles of 128 rows (n) by 64 columns (k); G is 32, 64 or 128.
 *   codes : tile (nb = n/128, kb = k/64) is 4096 bytes at
 *           (nb * (K/64) + kb) * 4096; inside it, half h = (k%64)/32 and row
 *           r = n%128 own the 16 bytes at h*2048 + r*16, the 32 columns
 *           c = k%32 of that half.  Those 16 bytes are four little-endian
 *           32-bit words.  With c = 16a + 8b + 2t + e (a, b, e in {0,1},
 *           t in 0..3), column c sits in word t at nibble position
 *           p = 2a + b + 4e (bits 4p..4p+3).
 *   scales: binary16 at element (nb * (K/G) + g) * 128 + r, g = k / G.
 *   zeros : byte (nb * (K/G) + g) * 64 + r/2, low nibble for even r.
 */
void orc_pack_tile(const uint8_t *q, const uint16_t *s, const uint8_t *z,
                   int64_t N, int64_t K, int64_t G, uint8_t *codes, uint16_t *scales, uint8_t *zeros)
{
    int64_t ng = K / G;
    memset(codes, 0, (size_t)(N * K / 2));
    memset(zeros, 0, (size_t)(N * ng / 2));
    for (int64_t n = 0; n < N; n++) {
        int64_t nb = n / 128, r = n % 128;
        for (int64_t k = 0; k < K; k++) {
            int64_t kb = k / 64, h = (k % 64) / 32, c = k % 32;
            int64_t a = c / 16, b = (c % 16) / 8, t = (c % 8) / 2, e = c % 2;
            int64_t p = 2 * a + b + 4 * e;
            int64_t byte = (nb * (K / 64) + kb) * 4096 + h * 2048 + r * 16 + t * 4 + p / 2;
            uint8_t v = q[n * K + k] & 15;
            codes[byte] |= (p % 2 == 0) ? v : (uint8_t)(v << 4);
        }
        for (int64_t g = 0; g < ng; g++) {
            scales[(nb * ng + g) * 128 + r] = s[n * ng + g];
            uint8_t v = z[n * ng + g] & 15;
            zeros[(nb * ng + g) * 64 + r / 2] |= (r % 2 == 0) ? v : (uint8_t)(v << 4);
        }
    }
}

/* ------------------------------------------------------------------ */
/* FP8 E4M3 quantisation with current (amax) scaling.                   */
/* [LP] S4 per-token and per-tensor, S7 E4M3, S8 scale = amax / 448.    */
/* ------------------------------------------------------------------ */

static float amax_scale(float amax)
{
    return amax == 0.0f ? 1.0f : amax / 448.0f;
}

/* Per-row (per-token) scales: X [M][K] bf16 -> Xq [M][K] e4m3, sx [M]. */
void orc_quant_fp8_rows(const uint16_t *X, int64_t M, int64_t K, uint8_t *Xq, float *sx)
{
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; m++) {
        float amax = 0.0f;
        for (int64_t k = 0; k < K; k++) {
            float a = fabsf(bf16_to_f32(X[m * K + k]));
            if (a > amax) amax = a;
        }
        float sc = amax_scale(amax);
        sx[m] = sc;
        for (int64_t k = 0; k < K; k++)
            Xq[m * K + k] = orc_f32_to_e4m3_rn_sat(bf16_to_f32(X[m * K + k]) / sc);
    }
}

/* One scale for the whole tensor: W [N][K] bf16 -> Wq [N][K] e4m3, *sw. */
void orc_quant_fp8_tensor(const uint16_t *W, int64_t N, int64_t K, uint8_t *Wq, float *sw)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < N * K; i++) {
        float a = fabsf(bf16_to_f32(W[i]));
        if (a > amax) amax = a;
    }
    float sc = amax_scale(amax);
    *sw = sc;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < N * K; i++)
        Wq[i] = orc_f32_to_e4m3_rn_sat(bf16_to_f32(W[i]) / sc);
}

/* ------------------------------------------------------------------ */
/* FP8 block scaling ([LP] S8 "Block Scaling": every block has its own    */
/* scale, x ~ x_fp8 * scale_block, scale_block = amax_block / max_fp8).   */
/* Blocks: 1 x 128 for activations (token m, columns 128b .. 128b+127),   */
/* 128 x 128 for weights (rows 128i.., columns 128b..).  Scales FP32,     */
/* the same amax / 448 (1 for an all-zero block) and E4M3 RNE-saturating  */
/* cast of x / scale (binary32 division) as the per-token recipe.         */
/* Activation scales are stored block-major: sx[b][m], b = k / 128.       */
/* ------------------------------------------------------------------ */

void orc_quant_fp8_act_blocks(const uint16_t *X, int64_t M, int64_t K, uint8_t *Xq, float *sx)
{
    int64_t nb = K / 128;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t m = 0; m < M; m++)
        for (int64_t b = 0; b < nb; b++) {
            float amax = 0.0f;
            for (int64_t k = b * 128; k < b * 128 + 128; k++) {
                float a = fabsf(bf16_to_f32(X[m * K + k]));
                if (a > amax) amax = a;
            }
            float sc = amax_scale(amax);
            sx[b * M + m] = sc;
            for (int64_t k = b * 128; k < b * 128 + 128; k++)
                Xq[m * K + k] = orc_f32_to_e4m3_rn_sat(bf16_to_f32(X[m * K + k]) / sc);
        }
}

/* Weight blocks: W [N][K] -> Wq [N][K], sw[i][b] for rows 128i.., columns 128b... */
void orc_quant_fp8_weight_blocks(const uint16_t *W, int64_t N, int64_t K, uint8_t *Wq, float *sw)
{
    int64_t nr = N / 128, nb = K / 128;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t i = 0; i < nr; i++)
        for (int64_t b = 0; b < nb; b++) {
            float amax = 0.0f;
            for (int64_t n = i * 128; n < i * 128 + 128; n++)
                for (int64_t k = b * 128; k < b * 128 + 128; k++) {
                    float a = fabsf(bf16_to_f32(W[n * K + k]));
                    if (a > amax) amax = a;
                }
            float sc = amax_scale(amax);
            sw[i * nb + b] = sc;
            for (int64_t n = i * 128; n < i * 128 + 128; n++)
                for (int64_t k = b * 128; k < b * 128 + 128; k++)
                    Wq[n * K + k] = orc_f32_to_e4m3_rn_sat(bf16_to_f32(W[n * K + k]) / sc);
        }
}

/* Block-scaled W8A8: Y[m][n] = sum_b sx[b][m] * sw[n/128][b] *            */
/* sum_{k in block b} e4m3(Xq[m][k]) * e4m3(Wq[n][k]), in double, at       */
/* `cnt` (m, n) pairs.                                                     */
void orc_w8a8_blocks_at(const uint8_t *Xq, const float *sx, const uint8_t *Wq, const float *sw,
                        int64_t M, int64_t N, int64_t K,
                        const int64_t *ms, const int64_t *ns, int64_t cnt, double *out)
{
    int64_t nb = K / 128;
    (void)N;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < cnt; i++) {
        int64_t m = ms[i], n = ns[i];
        double acc = 0.0;
        for (int64_t b = 0; b < nb; b++) {
            double part = 0.0;
            for (int64_t k = b * 128; k < b * 128 + 128; k++)
                part += orc_e4m3_to_f64(Xq[m * K + k]) * orc_e4m3_to_f64(Wq[n * K + k]);
            acc += part * (double)sx[b * M + m] * (double)sw[(n / 128) * nb + b];
        }
        out[i] = acc;
    }
}

/* ------------------------------------------------------------------ */
/* The linear layer Y = A . B^T, accumulated in double, no rounding of Y. */
/* [LP] S1 / S22: wide accumulation; the double result is the exact      */
/* target that the device's FP32-accumulated, BF16-rounded Y is held to. */
/* ------------------------------------------------------------------ */

void orc_gemm_nt_f64(const double *A, const double *B, int64_t M, int64_t N, int64_t K, double *Y)
{
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t m = 0; m < M; m++)
        for (int64_t n = 0; n < N; n++) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; k++)
                acc += A[m * K + k] * B[n * K + k];
            Y[m * N + n] = acc;
        }
}

/* W4A16: Y[m][n] = sum_k X[m][k] * s[n][k/G] * (q[n][k] - z[n][k/G]).   */
/* Evaluated at `cnt` (m, n) pairs; every term in double.  [LP] S2, S11. */
void orc_w4a16_at(const uint16_t *X, const uint8_t *q, const uint16_t *s, const uint8_t *z,
                  int64_t M, int64_t N, int64_t K, int G,
                  const int64_t *ms, const int64_t *ns, int64_t cnt, double *out)
{
    int64_t ng = K / G;
    (void)M;
    (void)N;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < cnt; i++) {
        int64_t m = ms[i], n = ns[i];
        double acc = 0.0;
        for (int64_t k = 0; k < K; k++) {
            double sc = orc_f16_to_f64(s[n * ng + k / G]);
            double w = sc * ((double)q[n * K + k] - (double)z[n * ng + k / G]);
            acc += (double)bf16_to_f32(X[m * K + k]) * w;
        }
        out[i] = acc;
    }
}

/* W4A8 ([LP] S1: INT4 weights, FP8 activations, FP32 accumulation, BF16
 * output): the INT4 weights of the W4A16 quantiser (x_hat = s (q - z) per
 * group) times the per-token E4M3 activations (sx[m] e4m3(Xq[m][k])):
 * Y[m][n] = sum_k sx[m] e4m3(Xq[m][k]) * s[n][k/G] (q[n][k] - z[n][k/G]),
 * in double, for sampled (m, n). */
void orc_w4a8_at(const uint8_t *Xq, const float *sx, const uint8_t *q, const uint16_t *s, const uint8_t *z,
                 int64_t M, int64_t N, int64_t K, int G,
                 const int64_t *ms, const int64_t *ns, int64_t cnt, double *out)
{
    int64_t ng = K / G;
    (void)M;
    (void)N;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < cnt; i++) {
        int64_t m = ms[i], n = ns[i];
        double acc = 0.0;
        for (int64_t k = 0; k < K; k++) {
            double x = (double)sx[m] * orc_e4m3_to_f64(Xq[m * K + k]);
            double w = orc_f16_to_f64(s[n * ng + k / G]) * ((double)q[n * K + k] - (double)z[n * ng + k / G]);
            acc += x * w;
        }
        out[i] = acc;
    }
}

/* W8A8: Y[m][n] = sx[m] * sw * sum_k e4m3(Xq[m][k]) * e4m3(Wq[n][k]).   */
void orc_w8a8_at(const uint8_t *Xq, const float *sx, const uint8_t *Wq, float sw,
                 int64_t M, int64_t N, int64_t K,
                 const int64_t *ms, const int64_t *ns, int64_t cnt, double *out)
{
    (void)M;
    (void)N;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < cnt; i++) {
        int64_t m = ms[i], n = ns[i];
        double acc = 0.0;
        for (int64_t k = 0; k < K; k++)
            acc += orc_e4m3_to_f64(Xq[m * K + k]) * orc_e4m3_to_f64(Wq[n * K + k]);
        out[i] = acc * (double)sx[m] * (double)sw;
    }
}

/* Thread count of the parallel loops (the CPU baseline times the oracle on
 * one core as well as on all of them); n <= 0 leaves it unchanged. */
void orc_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------ */
/* MXFP8 (the OCP Microscaling Formats specification v1.0, which [LP]  */
/* S10 names for the MX block formats): blocks of 32 consecutive       */
/* elements along a row share one power-of-two scale X = 2^e, stored   */
/* as an E8M0 byte e + 127.  e = floor(log2(amax)) - 8, 8 being the     */
/* exponent of the largest E4M3 normal (448 = 1.75 * 2^8), clamped to   */
/* [-127, 127]; an all-zero block takes e = -127.  Each element becomes */
/* E4M3(v / X), round to nearest even, saturating at +-448.             */
/* ------------------------------------------------------------------ */

/* emax: exponent of the element type's largest normal (E4M3 8, E2M1 2) */
static int mx_exponent_of(float amax, int emax)
{
    if (amax == 0.0f) return -127;
    int ex;
    frexpf(amax, &ex);          /* amax = f * 2^ex, f in [0.5, 1): floor(log2 amax) = ex - 1 */
    int e = (ex - 1) - emax;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return e;
}

static int mx_exponent(float amax) { return mx_exponent_of(amax, 8); }

/* X [R][K] bf16 -> codes [R][K] e4m3 and scales [R][K/32] e8m0 */
void orc_quant_mxfp8_rows(const uint16_t *X, int64_t R, int64_t K, uint8_t *codes, uint8_t *scales)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; r++) {
        for (int64_t b = 0; b < K / 32; b++) {
            float amax = 0.0f;
            for (int64_t k = b * 32; k < b * 32 + 32; k++) {
                float a = fabsf(bf16_to_f32(X[r * K + k]));
                if (a > amax) amax = a;
            }
            int e = mx_exponent(amax);
            scales[r * (K / 32) + b] = (uint8_t)(e + 127);
            double xs = ldexp(1.0, e);
            for (int64_t k = b * 32; k < b * 32 + 32; k++)
                codes[r * K + k] = orc_f32_to_e4m3_rn_sat((float)((double)bf16_to_f32(X[r * K + k]) / xs));
        }
    }
}

/* Y[m][n] = sum over 32-blocks b of 2^(xs[m][b]-127) 2^(ws[n][b]-127)
 *           * sum_{k in b} e4m3(Xq[m][k]) e4m3(Wq[n][k]), in double, for sampled (m, n) */
void orc_w8a8_mx_at(const uint8_t *Xq, const uint8_t *xs, const uint8_t *Wq, const uint8_t *ws,
                    int64_t M, int64_t N, int64_t K, const int64_t *ms, const int64_t *ns, int64_t cnt, double *out)
{
    (void)M; (void)N;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < cnt; i++) {
        int64_t m = ms[i], n = ns[i];
        double acc = 0.0;
        for (int64_t b = 0; b < K / 32; b++) {
            double part = 0.0;
            for (int64_t k = b * 32; k < b * 32 + 32; k++)
                part += orc_e4m3_to_f64(Xq[m * K + k]) * orc_e4m3_to_f64(Wq[n * K + k]);
            acc += part * ldexp(1.0, (int)xs[m * (K / 32) + b] - 127) * ldexp(1.0, (int)ws[n * (K / 32) + b] - 127);
        }
        out[i] = acc;
    }
}

/* ------------------------------------------------------------------ */
/* FP4 E2M1 ([LP] S10: 1 sign, 2 exponent and 1 mantissa bit).  With    */
/* the exponent bias 1 the eight magnitudes are 0, 0.5 (the subnormal), */
/* 1, 1.5, 2, 3, 4 and 6; the format has no infinity and no NaN.        */
/* ------------------------------------------------------------------ */

double orc_e2m1_to_f64(uint8_t c)
{
    int sign = (c >> 3) & 1;
    int e = (c >> 1) & 3;
    int m = c & 1;
    double v = e == 0 ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return sign ? -v : v;
}

/* binary32 -> E2M1: the nearest of the eight magnitudes, a tie going to the
 * even code (mantissa bit 0); above 6 (infinity included) the result
 * saturates to 6.  The sign bit is kept, also when the result is 0. */
uint8_t orc_f32_to_e2m1_rn_sat(float x)
{
    uint8_t sign = signbit(x) ? 8 : 0;
    double a = fabs((double)x);
    if (a >= 6.0)                /* 6 and beyond (infinity too): the largest magnitude */
        return sign | 7;
    int best = 0;
    for (int c = 1; c < 8; c++) {
        double d = fabs(a - orc_e2m1_to_f64((uint8_t)c));
        double db = fabs(a - orc_e2m1_to_f64((uint8_t)best));
        if (d < db || (d == db && (c & 1) == 0))
            best = c;
    }
    return sign | (uint8_t)best;
}

/* ------------------------------------------------------------------ */
/* MXFP4 (the OCP MX specification's FP4 block format, named in [LP]    */
/* S10): the MXFP8 recipe above with E2M1 elements -- blocks of 32 along */
/* a row share 2^e (E8M0 byte e + 127), e = floor(log2 amax) - 2, 2      */
/* being the exponent of E2M1's largest normal (6 = 1.5 * 2^2), clamped  */
/* to [-127, 127], -127 for an all-zero block; each element becomes      */
/* E2M1(v / 2^e).  Codes are returned one per byte (0..15).             */
/* ------------------------------------------------------------------ */

void orc_quant_mxfp4_rows(const uint16_t *X, int64_t R, int64_t K, uint8_t *codes, uint8_t *scales)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; r++) {
        for (int64_t b = 0; b < K / 32; b++) {
            float amax = 0.0f;
            for (int64_t k = b * 32; k < b * 32 + 32; k++) {
                float a = fabsf(bf16_to_f32(X[r * K + k]));
                if (a > amax) amax = a;
            }
            int e = mx_exponent_of(amax, 2);
            scales[r * (K / 32) + b] = (uint8_t)(e + 127);
            double xs = ldexp(1.0, e);
            for (int64_t k = b * 32; k < b * 32 + 32; k++)
                codes[r * K + k] = orc_f32_to_e2m1_rn_sat((float)((double)bf16_to_f32(X[r * K + k]) / xs));
        }
    }
}

/* Y[m][n] = sum over 32-blocks b of 2^(xs[m][b]-127) 2^(ws[n][b]-127)
 *           * sum_{k in b} e2m1(Xq[m][k]) e2m1(Wq[n][k]), in double, for sampled (m, n);
 * codes one per byte */
void orc_w4a4_mx_at(const uint8_t *Xq, const uint8_t *xs, const uint8_t *Wq, const uint8_t *ws,
                    int64_t M, int64_t N, int64_t K, const int64_t *ms, const int64_t *ns, int64_t cnt, double *out)
{
    (void)M; (void)N;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < cnt; i++) {
        int64_t m = ms[i], n = ns[i];
        double acc = 0.0;
        for (int64_t b = 0; b < K / 32; b++) {
            double part = 0.0;
            for (int64_t k = b * 32; k < b * 32 + 32; k++)
                part += orc_e2m1_to_f64(Xq[m * K + k]) * orc_e2m1_to_f64(Wq[n * K + k]);
            acc += part * ldexp(1.0, (int)xs[m * (K / 32) + b] - 127) * ldexp(1.0, (int)ws[n * (K / 32) + b] - 127);
        }
        out[i] = acc;
    }
}

/* ------------------------------------------------------------------ */
/* NVFP4 ([LP] S10 names it as a vendor recipe on the same E2M1         */
/* elements with its own block size and scale hierarchy; the reading    */
/* here is that vendor's published two-level recipe): a per-tensor FP32 */
/* scale sg = amax(|X|) / (6 * 448) (1 when that is 0), blocks of 16    */
/* along a row with an E4M3 block scale sb = E4M3(amax_b / (6 sg))      */
/* (round to nearest even, saturating), elements E2M1(v / (sb sg)); a   */
/* block whose scale rounds to 0 stores code 0 for every element.       */
/* Every step is one binary32 operation, so both sides of a comparison  */
/* take the same rounding decisions.                                    */
/* ------------------------------------------------------------------ */

float orc_nvfp4_global_scale(const uint16_t *X, int64_t n)
{
    float amax = 0.0f;
    for (int64_t i = 0; i < n; i++) {
        float a = fabsf(bf16_to_f32(X[i]));
        if (a > amax) amax = a;
    }
    float sg = amax / 2688.0f;   /* 6 (E2M1's largest) * 448 (E4M3's largest) */
    return sg == 0.0f ? 1.0f : sg;
}

/* X [R][K] bf16 -> codes [R][K] (one E2M1 code per byte), scales [R][K/16] E4M3 */
void orc_quant_nvfp4_rows(const uint16_t *X, int64_t R, int64_t K, float sg, uint8_t *codes, uint8_t *scales)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < R; r++) {
        for (int64_t b = 0; b < K / 16; b++) {
            float amax = 0.0f;
            for (int64_t k = b * 16; k < b * 16 + 16; k++) {
                float a = fabsf(bf16_to_f32(X[r * K + k]));
                if (a > amax) amax = a;
            }
            float d6 = 6.0f * sg;
            float q = amax / d6;
            uint8_t sc = orc_f32_to_e4m3_rn_sat(q);
            scales[r * (K / 16) + b] = sc;
            float den = (float)orc_e4m3_to_f64(sc) * sg;
            for (int64_t k = b * 16; k < b * 16 + 16; k++)
                codes[r * K + k] = sc == 0 ? 0 : orc_f32_to_e2m1_rn_sat(bf16_to_f32(X[r * K + k]) / den);
        }
    }
}

/* Y[m][n] = sgx sgw * sum over 16-blocks b of e4m3(xs[m][b]) e4m3(ws[n][b])
 *           * sum_{k in b} e2m1(Xq[m][k]) e2m1(Wq[n][k]), in double, for sampled (m, n) */
void orc_w4a4_nv_at(const uint8_t *Xq, const uint8_t *xs, float sgx, const uint8_t *Wq, const uint8_t *ws, float sgw,
                    int64_t M, int64_t N, int64_t K, const int64_t *ms, const int64_t *ns, int64_t cnt, double *out)
{
    (void)M; (void)N;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < cnt; i++) {
        int64_t m = ms[i], n = ns[i];
        double acc = 0.0;
        for (int64_t b = 0; b < K / 16; b++) {
            double part = 0.0;
            for (int64_t k = b * 16; k < b * 16 + 16; k++)
                part += orc_e2m1_to_f64(Xq[m * K + k]) * orc_e2m1_to_f64(Wq[n * K + k]);
            acc += part * orc_e4m3_to_f64(xs[m * (K / 16) + b]) * orc_e4m3_to_f64(ws[n * (K / 16) + b]);
        }
        out[i] = acc * (double)sgx * (double)sgw;
    }
}
