/* Plain CPU oracle of the decode step (TEST INFRASTRUCTURE ONLY).
 *
 * Only tests, the smoke check and the CPU-baseline legs of the bench may
 * load this library.  It shares no code with the CUDA path.  Weights and
 * caches arrive as bf16 bit patterns (uint16); the reference arithmetic is
 * double (``*_f64``); ``*_f32`` is the same code in float, used only to time
 * the CPU baseline.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int L, H, Hq, Hkv, D, F, V, qk_norm;
    double eps, theta;
} orc_shape;

typedef struct {
    const uint16_t *embed, *lm_head, *norm_final;
    const uint16_t *const *wq, *const *wk, *const *wv, *const *wo, *const *wg, *const *wu, *const *wd;
    const uint16_t *const *norm_attn, *const *norm_mlp, *const *qnorm, *const *knorm;
    /* fp8 != 0: the seven projections are e4m3 codes w8[m][layer] [N][K]
     * with fp32 scales s8[m][layer] [ceil(N/128)][K/128], m = q, k, v, o,
     * gate, up, down (the bf16 pointers above are then unused) */
    int fp8;
    const uint8_t *const *w8[7];
    const float *const *s8[7];
} orc_weights;

/* Value of an e4m3 ("fn") byte: sign, 4 exponent bits with bias 7, 3
 * mantissa bits; exponent field 0 is subnormal (m / 8 * 2^-6); S.1111.111 is
 * NaN and there are no infinities (the OCP 8-bit floating point format). */
double e4m3_to_double(uint8_t c) {
    int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    double v = e == 0 ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

double bf16_to_double(uint16_t u) {
    uint32_t bits = (uint32_t)u << 16;
    float f;
    memcpy(&f, &bits, 4);
    return (double)f;
}

/* Round a double to the nearest bf16 (ties to even), saturating to inf.
 * bf16 keeps 8 significant bits and float's exponent range. */
uint16_t double_to_bf16(double v) {
    if (isnan(v)) return 0x7fc0;
    if (v == 0.0) return signbit(v) ? 0x8000 : 0x0000;
    int e;
    double m = frexp(fabs(v), &e);          /* |v| = m * 2^e, 0.5 <= m < 1 */
    (void)m;
    int q_exp = e - 8;                       /* ulp of an 8-bit significand */
    if (q_exp < -133) q_exp = -133;          /* subnormal spacing 2^-133 */
    double ulp = ldexp(1.0, q_exp);
    double r = nearbyint(fabs(v) / ulp) * ulp;   /* default mode: ties to even */
    if (r >= ldexp(1.0, 128)) r = INFINITY;
    float f = (float)r;                      /* exact: r has <= 8 significant bits */
    uint32_t bits;
    memcpy(&bits, &f, 4);
    uint16_t out = (uint16_t)(bits >> 16);
    return signbit(v) ? (uint16_t)(out | 0x8000) : out;
}

#define REAL double
#define FN(name) name##_f64
#include "forward_impl.h"
#undef REAL
#undef FN

#define REAL float
#define FN(name) name##_f32
#include "forward_impl.h"
#undef REAL
#undef FN

/* ---- exported entry points ---- */

int orc_decode_step_f64(const orc_shape *sh, const orc_weights *w, uint16_t *kc, uint16_t *vc, int B, int Smax,
                        const int *pos, const int *tok, int nthreads, double *logits, double *hidden) {
    return decode_step_f64(sh, w, kc, vc, B, Smax, pos, tok, nthreads, logits, hidden);
}

int orc_decode_step_f32(const orc_shape *sh, const orc_weights *w, uint16_t *kc, uint16_t *vc, int B, int Smax,
                        const int *pos, const int *tok, int nthreads, float *logits, float *hidden) {
    return decode_step_f32(sh, w, kc, vc, B, Smax, pos, tok, nthreads, logits, hidden);
}

void orc_rmsnorm(const double *x, int n, const uint16_t *w, double eps, double *y) { rmsnorm_f64(x, n, w, eps, y); }
void orc_matvec(const uint16_t *W, int N, int K, const double *x, double *y) { matvec_f64(W, N, K, x, y, 1); }
void orc_rope(double *v, int D, int pos, double theta) { rope_f64(v, D, pos, theta); }
void orc_attend(const double *q, const uint16_t *K, const uint16_t *V, int n, int D, double *o) {
    double *scr = malloc(sizeof(double) * (n > 0 ? n : 1));
    attend_f64(q, K, V, n, D, o, scr);
    free(scr);
}
void orc_to_bf16(const double *x, uint16_t *y, long n) { for (long i = 0; i < n; i++) y[i] = double_to_bf16(x[i]); }
void orc_matvec8(const uint8_t *W, const float *S, int N, int K, const double *x, double *y) {
    matvec8_f64(W, S, N, K, x, y, 1);
}
