/* Decoder forward body, included twice by forward.c: once with REAL=double
 * (the reference arithmetic) and once with REAL=float (a faster twin used
 * only to time the CPU baseline).  TEST INFRASTRUCTURE ONLY.
 *
 * One decode step of a dense Llama-style decoder, per sequence b, new token
 * at position pos[b] (0-based, equal to the number of cached tokens):
 *   h = E[token]
 *   per layer:  x = RMSNorm(h; w_attn)
 *               q, k, v = Wq x, Wk x, Wv x   (projections bf16, or e4m3 with
 *                                            128 x 128 block scales)
 *               [qk_norm] q_j = RMSNorm_D(q_j; w_q), k_g = RMSNorm_D(k_g; w_k)
 *               RoPE(q, k, pos)
 *               cache[pos] = bf16(k), bf16(v)
 *               o_j = softmax(q_j . K_g[0..pos] / sqrt(D)) . V_g[0..pos]
 *               h += Wo o
 *               x = RMSNorm(h; w_mlp);  h += Wd (silu(Wg x) * (Wu x))
 *   logits = W_lm RMSNorm(h; w_final)
 * Sources: "CMU 15-779 Lecture 7 notes" section 5.1 (the seven fused
 * instruction types name these steps); RoPE in rotate-half form with
 * theta_i = theta^(-2i/D); norm eps and theta from the model description.
 */

static void FN(rmsnorm)(const REAL *x, int n, const uint16_t *w, double eps, REAL *y) {
    REAL ss = 0;
    for (int i = 0; i < n; i++) ss += x[i] * x[i];
    REAL scale = (REAL)(1.0 / sqrt((double)ss / n + eps));
    for (int i = 0; i < n; i++) y[i] = x[i] * scale * (REAL)bf16_to_double(w[i]);
}

static void FN(matvec)(const uint16_t *W, int N, int K, const REAL *x, REAL *y, int nthreads) {
#pragma omp parallel for schedule(static) num_threads(nthreads)
    for (int n = 0; n < N; n++) {
        const uint16_t *row = W + (size_t)n * K;
        REAL acc = 0;
        for (int k = 0; k < K; k++) acc += (REAL)bf16_to_double(row[k]) * x[k];
        y[n] = acc;
    }
}

/* FP8 weights: w[n][k] = e4m3 code x the fp32 scale of its 128 x 128 block
 * (row block n / 128, column block k / 128) -- the block-scale convention of
 * the "MegaRTP megakernel article", section 4 -- then the same dot product. */
static void FN(matvec8)(const uint8_t *W, const float *S, int N, int K, const REAL *x, REAL *y, int nthreads) {
    const int KB = K / 128;
#pragma omp parallel for schedule(static) num_threads(nthreads)
    for (int n = 0; n < N; n++) {
        const uint8_t *row = W + (size_t)n * K;
        const float *srow = S + (size_t)(n / 128) * KB;
        REAL acc = 0;
        for (int k = 0; k < K; k++) acc += (REAL)(e4m3_to_double(row[k]) * (double)srow[k / 128]) * x[k];
        y[n] = acc;
    }
}

static void FN(rope)(REAL *v, int D, int pos, double theta) {
    int half = D / 2;
    for (int i = 0; i < half; i++) {
        double inv_freq = pow(theta, -2.0 * i / D);
        double ang = (double)pos * inv_freq;
        REAL c = (REAL)cos(ang), s = (REAL)sin(ang);
        REAL a = v[i], b = v[i + half];
        v[i] = a * c - b * s;
        v[i + half] = a * s + b * c;
    }
}

/* o = softmax(q . K[0..n) / sqrt(D)) . V[0..n); K, V rows are bf16 [n][D]. */
static void FN(attend)(const REAL *q, const uint16_t *K, const uint16_t *V, int n, int D, REAL *o, REAL *scratch) {
    REAL inv = (REAL)(1.0 / sqrt((double)D));
    REAL m = -INFINITY;
    for (int t = 0; t < n; t++) {
        REAL s = 0;
        for (int d = 0; d < D; d++) s += q[d] * (REAL)bf16_to_double(K[(size_t)t * D + d]);
        s *= inv;
        scratch[t] = s;
        if (s > m) m = s;
    }
    REAL l = 0;
    for (int t = 0; t < n; t++) { scratch[t] = (REAL)exp((double)(scratch[t] - m)); l += scratch[t]; }
    for (int d = 0; d < D; d++) o[d] = 0;
    for (int t = 0; t < n; t++) {
        REAL p = scratch[t] / l;
        for (int d = 0; d < D; d++) o[d] += p * (REAL)bf16_to_double(V[(size_t)t * D + d]);
    }
}

/* A projection of layer l: matrix m (0 q, 1 k, 2 v, 3 o, 4 gate, 5 up, 6 down) in bf16 or fp8. */
static void FN(project)(const orc_weights *w, int m, const uint16_t *const *bf, int l, int N, int K, const REAL *x,
                        REAL *y, int nthreads) {
    if (w->fp8) FN(matvec8)(w->w8[m][l], w->s8[m][l], N, K, x, y, nthreads);
    else FN(matvec)(bf[l], N, K, x, y, nthreads);
}

static int FN(decode_step)(const orc_shape *sh, const orc_weights *w, uint16_t *kcache, uint16_t *vcache,
                           int B, int Smax, const int *pos, const int *tokens, int nthreads,
                           REAL *logits, REAL *hidden) {
    const int H = sh->H, Hq = sh->Hq, Hkv = sh->Hkv, D = sh->D, F = sh->F, V = sh->V, L = sh->L;
    const int G = Hq / Hkv;
    REAL *h = malloc(sizeof(REAL) * H), *x = malloc(sizeof(REAL) * (H > F ? H : F));
    REAL *q = malloc(sizeof(REAL) * Hq * D), *k = malloc(sizeof(REAL) * Hkv * D), *v = malloc(sizeof(REAL) * Hkv * D);
    REAL *o = malloc(sizeof(REAL) * Hq * D), *t1 = malloc(sizeof(REAL) * (H > F ? H : F));
    REAL *gt = malloc(sizeof(REAL) * F), *ut = malloc(sizeof(REAL) * F);
    REAL *sc = malloc(sizeof(REAL) * (Smax + 1)), *tmp = malloc(sizeof(REAL) * D);
    if (!h || !x || !q || !k || !v || !o || !t1 || !gt || !ut || !sc || !tmp) return -1;
    for (int b = 0; b < B; b++) {
        int p = pos[b];
        if (p < 0 || p >= Smax || tokens[b] < 0 || tokens[b] >= V) return -2;
        for (int i = 0; i < H; i++) h[i] = (REAL)bf16_to_double(w->embed[(size_t)tokens[b] * H + i]);
        for (int l = 0; l < L; l++) {
            FN(rmsnorm)(h, H, w->norm_attn[l], sh->eps, x);
            FN(project)(w, 0, w->wq, l, Hq * D, H, x, q, nthreads);
            FN(project)(w, 1, w->wk, l, Hkv * D, H, x, k, nthreads);
            FN(project)(w, 2, w->wv, l, Hkv * D, H, x, v, nthreads);
            if (sh->qk_norm) {
                for (int j = 0; j < Hq; j++) { FN(rmsnorm)(q + j * D, D, w->qnorm[l], sh->eps, tmp); memcpy(q + j * D, tmp, sizeof(REAL) * D); }
                for (int g = 0; g < Hkv; g++) { FN(rmsnorm)(k + g * D, D, w->knorm[l], sh->eps, tmp); memcpy(k + g * D, tmp, sizeof(REAL) * D); }
            }
            for (int j = 0; j < Hq; j++) FN(rope)(q + j * D, D, p, sh->theta);
            for (int g = 0; g < Hkv; g++) FN(rope)(k + g * D, D, p, sh->theta);
            for (int g = 0; g < Hkv; g++) {
                size_t base = ((((size_t)l * B + b) * Hkv + g) * Smax + p) * D;
                for (int d = 0; d < D; d++) {
                    kcache[base + d] = double_to_bf16((double)k[g * D + d]);
                    vcache[base + d] = double_to_bf16((double)v[g * D + d]);
                }
            }
#pragma omp parallel for schedule(static) num_threads(nthreads)
            for (int j = 0; j < Hq; j++) {
                int g = j / G;
                size_t base = (((size_t)l * B + b) * Hkv + g) * Smax * (size_t)D;
                REAL *scr = malloc(sizeof(REAL) * (p + 1));
                FN(attend)(q + j * D, kcache + base, vcache + base, p + 1, D, o + j * D, scr);
                free(scr);
            }
            FN(project)(w, 3, w->wo, l, H, Hq * D, o, t1, nthreads);
            for (int i = 0; i < H; i++) h[i] += t1[i];
            FN(rmsnorm)(h, H, w->norm_mlp[l], sh->eps, x);
            FN(project)(w, 4, w->wg, l, F, H, x, gt, nthreads);
            FN(project)(w, 5, w->wu, l, F, H, x, ut, nthreads);
            for (int i = 0; i < F; i++) {
                REAL g = gt[i];
                gt[i] = g / (1 + (REAL)exp(-(double)g)) * ut[i];
            }
            FN(project)(w, 6, w->wd, l, H, F, gt, t1, nthreads);
            for (int i = 0; i < H; i++) h[i] += t1[i];
            if (hidden) memcpy(hidden + ((size_t)l * B + b) * H, h, sizeof(REAL) * H);
        }
        FN(rmsnorm)(h, H, w->norm_final, sh->eps, x);
        FN(matvec)(w->lm_head, V, H, x, logits + (size_t)b * V, nthreads);
    }
    free(h); free(x); free(q); free(k); free(v); free(o); free(t1); free(gt); free(ut); free(sc); free(tmp);
    return 0;
}
