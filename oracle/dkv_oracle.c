/*
 * CPU oracle for the zero-copy KV-cache attention path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this file's library.  It shares no code,
 * header, table or helper with the CUDA library and must never be linked
 * into it.
 *
 * What it computes is the plain definition on "Paper Notes: DirectKV"
 * (Fundamental Underlying Technologies, Kernel Fusion): K = X.Wk, V = X.Wv,
 * and attention softmax(Q.K^T / sqrt(d)).V; the KV Cache Manager paragraph
 * (System Architecture) says new K/V rows are written once into the pinned
 * host cache and reused.  The method is exact ("Does DirectKV degrade output
 * quality", aifetchly DirectKV page, FAQ), so the oracle is the definition
 * itself with no tiling, splitting or online rescaling:
 *
 *   dkv_oracle_round     round a real value to bf16/fp16, nearest, ties to even
 *   dkv_oracle_round_e4m3  the same to 8-bit E4M3, saturating (FP8 caches)
 *   dkv_oracle_project   projection: fp32 products (exact for 16-bit inputs)
 *                        accumulated in fp32 in sequential order j = 0..H-1,
 *                        then rounded to the storage dtype; also the fp64 sum
 *   dkv_oracle_attend    softmax attention in fp64 for one (sequence, KV head):
 *                        row i sees keys 0..pos[i] inclusive (causal; a decode
 *                        query sees the whole cache including its own new row)
 *
 * Built with -O2 -fno-fast-math so no floating-point sum is reassociated.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_BF16 = 0, ORC_FP16 = 1 };

/* ---- 16-bit float formats, decoded from their definition ---------------- */

/* Exact value of a bf16 / fp16 bit pattern. */
static double orc_decode(uint16_t h, int dt) {
    int sign = (h >> 15) & 1;
    int ebits = dt == ORC_BF16 ? 8 : 5;
    int mbits = dt == ORC_BF16 ? 7 : 10;
    int bias = (1 << (ebits - 1)) - 1;
    int e = (h >> mbits) & ((1 << ebits) - 1);
    int m = h & ((1 << mbits) - 1);
    double v;
    if (e == (1 << ebits) - 1) {
        v = m ? NAN : INFINITY;
    } else if (e == 0) {
        v = ldexp((double)m, 1 - bias - mbits);
    } else {
        v = ldexp((double)(m + (1 << mbits)), e - bias - mbits);
    }
    return sign ? -v : v;
}

/* Nearest representable value, ties to even, of a real number v, encoded as
 * bits.  Precision p = mbits + 1 significant bits; the smallest normal
 * exponent is 1 - bias.  The quantum at v is 2^(max(floor(log2|v|), emin) -
 * mbits); v / quantum is exact in double (a power-of-two scaling), nearbyint
 * rounds it to the nearest integer with ties to even, and a result past the
 * largest finite value becomes infinity. */
static uint16_t orc_encode(double v, int dt) {
    int ebits = dt == ORC_BF16 ? 8 : 5;
    int mbits = dt == ORC_BF16 ? 7 : 10;
    int bias = (1 << (ebits - 1)) - 1;
    int emin = 1 - bias;
    int emax = bias;
    uint16_t sign = signbit(v) ? 0x8000u : 0u;
    double a = fabs(v);
    if (isnan(v)) return (uint16_t)(((1u << ebits) - 1) << mbits | (1u << (mbits - 1)));
    if (a == 0.0) return sign;
    int E;
    (void)frexp(a, &E); /* a = f * 2^E, f in [0.5, 1) -> leading bit 2^(E-1) */
    int lead = E - 1;
    if (lead < emin) lead = emin;
    double quantum = ldexp(1.0, lead - mbits);
    double n = nearbyint(a / quantum); /* integer significand, ties to even */
    double r = n * quantum;
    double maxfin = ldexp((double)((1 << (mbits + 1)) - 1), emax - mbits);
    if (r > maxfin || isinf(a)) return sign | (uint16_t)(((1u << ebits) - 1) << mbits);
    if (r == 0.0) return sign; /* rounded down to zero */
    /* encode r exactly */
    (void)frexp(r, &E);
    lead = E - 1;
    if (lead < emin) { /* subnormal: exponent field 0, significand r / 2^(emin-mbits) */
        uint32_t m = (uint32_t)ldexp(r, mbits - emin);
        return sign | (uint16_t)m;
    }
    uint32_t sig = (uint32_t)ldexp(r, mbits - lead); /* in [2^mbits, 2^(mbits+1)) */
    uint32_t efield = (uint32_t)(lead + bias);
    return sign | (uint16_t)(efield << mbits) | (uint16_t)(sig - (1u << mbits));
}

/* ---- 8-bit E4M3 (OCP 8-bit floating point, E4M3 variant) --------------
 * 1 sign, 4 exponent (bias 7) and 3 mantissa bits; no infinities; exponent
 * and mantissa all ones is NaN, so the largest finite value is 1.75 * 2^8 =
 * 448; exponent 0 holds the subnormals m * 2^-9.  Used for the FP8 K/V cache
 * format (unscaled). */

static double orc_e4m3_decode(uint8_t b) {
    int sign = (b >> 7) & 1, e = (b >> 3) & 15, m = b & 7;
    double v;
    if (e == 15 && m == 7) v = NAN;
    else if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp((double)(m + 8), e - 10);
    return sign ? -v : v;
}

/* Nearest E4M3 value, ties to even, saturating at +-448 ("satfinite"): the
 * same quantum construction as orc_encode with 3 mantissa bits and the
 * smallest normal exponent -6; a result past 448 is clamped to 448. */
static uint8_t orc_e4m3_encode(double v) {
    const int mbits = 3, bias = 7, emin = -6;
    uint8_t sign = signbit(v) ? 0x80u : 0u;
    if (isnan(v)) return 0x7Fu;
    double a = fabs(v);
    if (a == 0.0) return sign;
    int E;
    (void)frexp(a, &E);
    int lead = E - 1;
    if (lead < emin) lead = emin;
    double r = nearbyint(a / ldexp(1.0, lead - mbits)) * ldexp(1.0, lead - mbits);
    if (r > 448.0 || isinf(a)) r = 448.0;
    if (r == 0.0) return sign;
    (void)frexp(r, &E);
    lead = E - 1;
    if (lead < emin) return sign | (uint8_t)ldexp(r, mbits - emin); /* subnormal */
    uint32_t sig = (uint32_t)ldexp(r, mbits - lead); /* in [8, 16) */
    return sign | (uint8_t)((uint32_t)(lead + bias) << mbits) | (uint8_t)(sig - 8u);
}

void dkv_oracle_decode_e4m3(const uint8_t* bits, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_decode(bits[i]);
}

void dkv_oracle_round_e4m3(const double* v, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_encode(v[i]);
}

void dkv_oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int dkv_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void dkv_oracle_decode(const uint16_t* bits, int64_t n, int dt, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_decode(bits[i], dt);
}

void dkv_oracle_round(const double* v, int64_t n, int dt, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_encode(v[i], dt);
}

/* Projection Y = X . W for X [rows, H] and W [H, ncols] (16-bit bits,
 * row-major).  Each output accumulates the exact fp32 products
 * x[r][j] * w[j][c] in fp32, j = 0, 1, ..., H-1 in that order, starting from
 * +0; the sum is rounded once to the storage dtype (out_bits, if non-null).
 * out_f32, if non-null, receives the fp32 sum itself (before that rounding,
 * for other storage formats); out_exact the same sum taken in fp64
 * (diagnostic). */
void dkv_oracle_project(const uint16_t* x, int rows, int H, const uint16_t* w, int ncols,
                        int dt, uint16_t* out_bits, double* out_exact, double* out_f32) {
    float* wf = (float*)malloc(sizeof(float) * (size_t)H * (size_t)ncols);
    for (int64_t i = 0; i < (int64_t)H * ncols; ++i) wf[i] = (float)orc_decode(w[i], dt);
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < rows; ++r) {
        float* acc = (float*)malloc(sizeof(float) * (size_t)ncols);
        double* accd = out_exact ? (double*)malloc(sizeof(double) * (size_t)ncols) : NULL;
        for (int c = 0; c < ncols; ++c) acc[c] = 0.0f;
        if (accd) for (int c = 0; c < ncols; ++c) accd[c] = 0.0;
        for (int j = 0; j < H; ++j) {
            float xv = (float)orc_decode(x[(size_t)r * H + j], dt);
            const float* wr = wf + (size_t)j * ncols;
            for (int c = 0; c < ncols; ++c) {
                float p = xv * wr[c];   /* exact: 8x8 or 11x11 significant bits */
                acc[c] = acc[c] + p;    /* one fp32 rounding per step */
            }
            if (accd)
                for (int c = 0; c < ncols; ++c) accd[c] += (double)xv * (double)wr[c];
        }
        for (int c = 0; c < ncols; ++c) {
            if (out_bits) out_bits[(size_t)r * ncols + c] = orc_encode((double)acc[c], dt);
            if (out_f32) out_f32[(size_t)r * ncols + c] = (double)acc[c];
        }
        if (accd) {
            memcpy(out_exact + (size_t)r * ncols, accd, sizeof(double) * (size_t)ncols);
            free(accd);
        }
        free(acc);
    }
    free(wf);
}

/* Attention for one (sequence, KV head) in fp64.
 *   K, V    [S][D] keys/values after the append (row-major, fp64)
 *   Q       [nq][D] query rows (any heads of the group, any positions)
 *   pos     [nq]    absolute position of each query; row i sees keys 0..pos[i]
 *   out     [nq][D] softmax(q.k_j / sqrt(D)) . v_j over the visible keys
 *   lse     [nq]    optional: m + ln(sum_j exp(s_j - m)), s_j = q.k_j / sqrt(D)
 *   weights [nq][S] optional: the softmax weights (0 for keys not visible)
 * Returns 0, or -1 if some pos[i] is outside [0, S). */
int dkv_oracle_attend(int D, int S, const double* K, const double* V, int nq,
                      const double* Q, const int32_t* pos, double* out, double* lse,
                      double* weights) {
    for (int i = 0; i < nq; ++i)
        if (pos[i] < 0 || pos[i] >= S) return -1;
    const double scale = 1.0 / sqrt((double)D);
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < nq; ++i) {
        const double* q = Q + (size_t)i * D;
        int n = pos[i] + 1;
        double* s = (double*)malloc(sizeof(double) * (size_t)n);
        double m = -INFINITY;
        for (int j = 0; j < n; ++j) {
            const double* k = K + (size_t)j * D;
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += q[d] * k[d];
            s[j] = dot * scale;
            if (s[j] > m) m = s[j];
        }
        double l = 0.0;
        for (int j = 0; j < n; ++j) {
            s[j] = exp(s[j] - m);
            l += s[j];
        }
        double* o = out + (size_t)i * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        for (int j = 0; j < n; ++j) {
            const double* v = V + (size_t)j * D;
            double p = s[j] / l;
            for (int d = 0; d < D; ++d) o[d] += p * v[d];
        }
        if (lse) lse[i] = m + log(l);
        if (weights) {
            double* wrow = weights + (size_t)i * S;
            for (int j = 0; j < S; ++j) wrow[j] = j < n ? s[j] / l : 0.0;
        }
        free(s);
    }
    return 0;
}
