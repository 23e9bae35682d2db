/*
 * k3mx_oracle.c - plain, slow CPU reference of the MXFP4 routed-expert layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only the tests, the smoke check and the bench's CPU
 * baseline do.  It shares no code with the CUDA kernels.
 *
 * Every step is the plain definition, written in the order the pages give it,
 * with double accumulation, no blocking and no reordering.  Build with
 * -ffp-contract=off so that every multiply and add rounds as written.  OpenMP
 * splits independent output rows across threads; each row is still summed by
 * one thread in one fixed order, so results do not depend on the thread count
 * (the determinism argument of "A floating-point contract, not a convention",
 * kimi-k3-in-c: 2.78 trillion parameters, one CPU, 8 GB of RAM).
 *
 * Sources (page title, section):
 *   [W]  Kimi K3 engine (c/kimi_k3.c), "Weights": e2m1 nibbles two per byte,
 *        low nibble = even column, bit 3 = sign, one ue8m0 scale per 32
 *        columns, w = v * 2^(scale - 127).
 *   [R1] kimi-k3-in-c: 2.78 trillion parameters, one CPU, 8 GB of RAM,
 *        "Reduction one: the experts already ship at half a byte": per
 *        32-group sub-dot, one scale per group, scale byte 255 (NaN) skipped,
 *        double accumulator, result rounded to float once per row.
 *   [A]  Kimi K3 engine (c/kimi_k3.c), "Architecture notes", Stable LatentMoE
 *        bullet: sigmoid router, top-16 on biased scores, weights are the raw
 *        scores renormalised, experts are GLUs of inter width 3072 in the
 *        3584 latent, activation SiTU-GLU 4 tanh(g/4) sigma(g) 25 tanh(u/25).
 *   [I3] kimi-k3-in-c README, "Three invariants", item 3: the routing bias
 *        steers selection only; the combining weights use the unbiased
 *        sigmoid scores.
 *   [C]  kimi-k3-in-c README, "2. The config reader that refuses to guess",
 *        K3Cfg: n_experts 896, topk 16, latent 3584, moe_inter 3072,
 *        routed_scale 1.0, moe_renorm 1, situ_b1 4.0, situ_b2 25.0.
 *   [P]  Kimi K3 engine (c/kimi_k3.c), "Chunked prefill": within a chunk every
 *        unique expert is loaded once for all the tokens that chose it.
 *   [RG] Kimi K3 engine (c/kimi_k3.c), "Architecture notes", Stable
 *        LatentMoE bullet: the sigmoid router is a [896, 7168] matrix applied
 *        to the 7168-wide hidden state; its outputs are the logits [A] takes.
 *        The trunk (router included) is bf16 (kimi-k3-in-c README, the
 *        resident set of budget.py: "norms, router gates, biases").
 *   [LM] Kimi K3 engine (c/kimi_k3.c), "Architecture notes", Stable
 *        LatentMoE bullet: the token is projected 7168 -> 3584, the experts
 *        run in that latent, the aggregate is RMSNorm-ed and projected back
 *        3584 -> 7168, and two fused full-width shared experts (inter 6144)
 *        are added; K3Cfg (kimi-k3-in-c README, "2. The config reader that
 *        refuses to guess"): n_shared 2 "full width, added UNWEIGHTED",
 *        latent_norm 1 "RMSNorm on the AGGREGATE", rms_eps 1e-5.
 *   [TP] Kimi K3 engine (c/kimi_k3.c), "Streaming design" (K3_TOPP) and the
 *        environment table: optionally keep the routed experts only up to a
 *        cumulative weight p, dropping the low-weight tail of the top-16 and
 *        renormalising the rest (0 = off).
 *
 * Readings where the pages are silent (each listed in the design notes):
 *   - sigma is evaluated in double with libm exp and rounded to fp32 once;
 *     the selection key is that fp32 score plus the fp32 bias, one fp32 add.
 *   - ties between equal keys go to the lower expert index; -0 counts as +0;
 *     a NaN key ranks below every number.
 *   - the 16 indices are returned in selection order (key descending).
 *   - renormalisation has no epsilon; routed_scale 1.0 is applied explicitly.
 *   - g = W1 x and u = W3 x (W1 is the gate).  g and u are the fp32 outputs
 *     of the GEMV; h is evaluated in double and rounded to fp32.
 *   - tokens are grouped by expert with a stable order (token, slot).
 *   - [TP]: the 16 are taken in order of decreasing raw score (ties: lower
 *     expert index); an expert is kept while the scores before it sum to
 *     less than p times the sum of all 16 (so the kept set is the shortest
 *     prefix reaching p); kept weights are raw scores over the kept sum;
 *     a dropped slot has index -1 and weight 0 and runs no expert.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* [W]: code = nibble; bit 3 is the sign, bits 2..0 index the magnitudes
 * {0, 0.5, 1, 1.5, 2, 3, 4, 6}. */
static const double ORC_E2M1[16] = {
    0.0,  0.5,  1.0,  1.5,  2.0,  3.0,  4.0,  6.0,
   -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0,
};

double orc_e2m1(int code) { return ORC_E2M1[code & 15]; }

/* [W]: ue8m0 byte s means 2^(s - 127); 255 is NaN and is never used. */
double orc_e8m0(int s)
{
    if (s == 255) return NAN;
    return ldexp(1.0, s - 127);
}

/* the nibble of column c of a packed row: low nibble = even column [W] */
static inline int nib(const uint8_t *row_packed, int c)
{
    return (row_packed[c >> 1] >> (4 * (c & 1))) & 15;
}

/*
 * y[r] = sum_g 2^(s_rg - 127) * sum_{i<32} v(r, 32g+i) * x[32g+i]   [R1]
 * packed: [rows][in/2] bytes, scales: [rows][in/32] bytes, row-major.
 * Groups whose scale byte is 255 contribute nothing.
 */
void orc_gemv(float *y, const float *x, const uint8_t *packed,
              const uint8_t *scales, int in, int rows)
{
    const int ngrp = in / 32;
    #pragma omp parallel for schedule(static)
    for (int r = 0; r < rows; r++) {
        const uint8_t *pr = packed + (size_t)r * (in / 2);
        const uint8_t *sr = scales + (size_t)r * ngrp;
        double acc = 0.0;
        for (int g = 0; g < ngrp; g++) {
            const int sb = sr[g];
            if (sb == 255) continue;                 /* NaN scale: nothing */
            double sub = 0.0;
            for (int i = 0; i < 32; i++) {
                const int c = 32 * g + i;
                sub += ORC_E2M1[nib(pr, c)] * (double)x[c];
            }
            acc += sub * orc_e8m0(sb);
        }
        y[r] = (float)acc;
    }
}

/*
 * Tolerance helper, not part of the method: b[r] = sum_c |w_rc| |x_c| over
 * the groups whose scale is not 255, in double.
 */
void orc_gemv_absdot(double *b, const double *xabs, const uint8_t *packed,
                     const uint8_t *scales, int in, int rows)
{
    const int ngrp = in / 32;
    #pragma omp parallel for schedule(static)
    for (int r = 0; r < rows; r++) {
        const uint8_t *pr = packed + (size_t)r * (in / 2);
        const uint8_t *sr = scales + (size_t)r * ngrp;
        double acc = 0.0;
        for (int g = 0; g < ngrp; g++) {
            const int sb = sr[g];
            if (sb == 255) continue;
            double sub = 0.0;
            for (int i = 0; i < 32; i++) {
                const int c = 32 * g + i;
                sub += fabs(ORC_E2M1[nib(pr, c)]) * xabs[c];
            }
            acc += sub * orc_e8m0(sb);
        }
        b[r] = acc;
    }
}

/* sigma(z) = 1 / (1 + exp(-z)), in double */
double orc_sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

/* SiTU-GLU [A], betas 4.0 and 25.0 [C]: 4 tanh(g/4) sigma(g) * 25 tanh(u/25) */
double orc_situ(double g, double u)
{
    const double b1 = 4.0, b2 = 25.0;
    return (b1 * tanh(g / b1) * orc_sigmoid(g)) * (b2 * tanh(u / b2));
}

/*
 * One routed expert [A]: g = W1 x, u = W3 x (each [F x D], fp32 results),
 * h_j = SiTU(g_j, u_j) rounded to fp32, y = W2 h (W2 is [D x F]).
 * g, u, h may be NULL; otherwise they receive the intermediate vectors.
 * The scratch for g, u and h when NULL is the caller's buffer `tmp` of 3F
 * floats.
 */
void orc_expert(float *y, float *g, float *u, float *h, float *tmp,
                const float *x,
                const uint8_t *w1p, const uint8_t *w1s,
                const uint8_t *w3p, const uint8_t *w3s,
                const uint8_t *w2p, const uint8_t *w2s, int D, int F)
{
    float *gg = g ? g : tmp, *uu = u ? u : tmp + F, *hh = h ? h : tmp + 2 * F;
    orc_gemv(gg, x, w1p, w1s, D, F);
    orc_gemv(uu, x, w3p, w3s, D, F);
    for (int j = 0; j < F; j++) hh[j] = (float)orc_situ((double)gg[j], (double)uu[j]);
    orc_gemv(y, hh, w2p, w2s, F, D);
}

/*
 * Tolerance helper, not part of the method.  bound[i] =
 *   sum_j |w2_ij| (|h_j| + 30 E_j),  E_j = sum_c (|w1_jc| + |w3_jc|) |x_c|.
 * 30 bounds how far an error in g or u moves h:  |dh/dg| <= 25 max|A'(g)|
 * with A(g) = 4 tanh(g/4) sigma(g) (about 0.93, so about 23.3) and
 * |dh/du| <= 4.  `work` holds 2D + 3F doubles.
 */
void orc_expert_bound(double *bound, double *work, const float *x, const float *h,
                      const uint8_t *w1p, const uint8_t *w1s,
                      const uint8_t *w3p, const uint8_t *w3s,
                      const uint8_t *w2p, const uint8_t *w2s, int D, int F)
{
    double *xa = work, *e1 = work + D, *e3 = e1 + F, *hb = e3 + F;
    for (int c = 0; c < D; c++) xa[c] = fabs((double)x[c]);
    orc_gemv_absdot(e1, xa, w1p, w1s, D, F);
    orc_gemv_absdot(e3, xa, w3p, w3s, D, F);
    for (int j = 0; j < F; j++) hb[j] = fabs((double)h[j]) + 30.0 * (e1[j] + e3[j]);
    orc_gemv_absdot(bound, hb, w2p, w2s, F, D);
}

/* order used by the selection: -0 -> +0, NaN -> -inf [reading] */
static inline float canon_key(float k)
{
    if (k != k) return -INFINITY;
    if (k == 0.0f) return 0.0f;
    return k;
}

/*
 * Router [A][I3][C], per token t:
 *   s_e   = (float) sigma(logit_e)           (double, rounded once)
 *   key_e = s_e + bias_e                     (one fp32 add)
 *   idx   = the K experts of largest key, by repeated argmax:
 *           the largest key wins, equal keys go to the lower e
 *   w_k   = (float)( s_{idx_k} / sum_j s_{idx_j} ) * routed_scale
 * The sum over the selected raw scores is taken in double in slot order.
 * `s_out` (T x E, may be NULL) receives the fp32 scores.
 */
void orc_route(int32_t *idx, float *w, float *s_out, const float *logits,
               const float *bias, int T, int E, int K, float routed_scale)
{
    #pragma omp parallel for schedule(static)
    for (int t = 0; t < T; t++) {
        float s[1024], key[1024];
        unsigned char taken[1024];
        const float *lt = logits + (size_t)t * E;
        for (int e = 0; e < E; e++) {
            s[e] = (float)orc_sigmoid((double)lt[e]);
            key[e] = canon_key(s[e] + bias[e]);
            taken[e] = 0;
        }
        if (s_out) memcpy(s_out + (size_t)t * E, s, sizeof(float) * (size_t)E);
        for (int k = 0; k < K; k++) {
            int best = -1;
            for (int e = 0; e < E; e++) {
                if (taken[e]) continue;
                if (best < 0 || key[e] > key[best]) best = e;   /* strict: ties keep lower e */
            }
            taken[best] = 1;
            idx[(size_t)t * K + k] = best;
        }
        double sum = 0.0;
        for (int k = 0; k < K; k++) sum += (double)s[idx[(size_t)t * K + k]];
        for (int k = 0; k < K; k++)
            w[(size_t)t * K + k] =
                (float)((double)s[idx[(size_t)t * K + k]] / sum) * routed_scale;
    }
}

/* a bf16 bit pattern as a double: the upper half of an fp32 */
double orc_bf16(uint16_t b)
{
    const uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Router logits [RG]:  logits[t][e] = (float) sum_c W[e][c] * h[t][c]
 * W: [E][C] bf16 row-major; h: [T][C] fp32 (h_bf16 = 0) or bf16 (h_bf16 = 1).
 * Every product is exact in double (8 + 24 significant bits); the sum runs
 * over c in ascending order in double and is rounded to fp32 once.
 */
void orc_router_logits(float *logits, const uint16_t *W, const void *h, int h_bf16, int T, int E, int C)
{
    #pragma omp parallel for collapse(2) schedule(static)
    for (int t = 0; t < T; t++) {
        for (int e = 0; e < E; e++) {
            const uint16_t *we = W + (size_t)e * C;
            double acc = 0.0;
            for (int c = 0; c < C; c++) {
                const double hv = h_bf16 ? orc_bf16(((const uint16_t *)h)[(size_t)t * C + c])
                                         : (double)((const float *)h)[(size_t)t * C + c];
                acc += orc_bf16(we[c]) * hv;
            }
            logits[(size_t)t * E + e] = (float)acc;
        }
    }
}

/* The tolerance scale of a logit: sum_c |W[e][c] h[t][c]| in double. */
void orc_router_absdot(double *b, const uint16_t *W, const void *h, int h_bf16, int T, int E, int C)
{
    #pragma omp parallel for collapse(2) schedule(static)
    for (int t = 0; t < T; t++) {
        for (int e = 0; e < E; e++) {
            const uint16_t *we = W + (size_t)e * C;
            double acc = 0.0;
            for (int c = 0; c < C; c++) {
                const double hv = h_bf16 ? orc_bf16(((const uint16_t *)h)[(size_t)t * C + c])
                                         : (double)((const float *)h)[(size_t)t * C + c];
                acc += fabs(orc_bf16(we[c]) * hv);
            }
            b[(size_t)t * E + e] = acc;
        }
    }
}

/*
 * RMSNorm [LM]: y[t][i] = x[t][i] / sqrt(mean_i x[t][i]^2 + eps) * g[i],
 * g bf16; in double, rounded to fp32 once.
 */
void orc_rmsnorm(float *y, const float *x, const uint16_t *g, int T, int D, double eps)
{
    for (int t = 0; t < T; t++) {
        const float *xt = x + (size_t)t * D;
        double ss = 0.0;
        for (int i = 0; i < D; i++) ss += (double)xt[i] * (double)xt[i];
        const double r = 1.0 / sqrt(ss / (double)D + eps);
        for (int i = 0; i < D; i++) y[(size_t)t * D + i] = (float)((double)xt[i] * r * orc_bf16(g[i]));
    }
}

/* SiTU-GLU elementwise [A][LM]: a[i] = (float) SiTU(g[i], u[i]) */
void orc_situ_vec(float *a, const float *g, const float *u, long long n)
{
    #pragma omp parallel for schedule(static)
    for (long long i = 0; i < n; i++) a[i] = (float)orc_situ((double)g[i], (double)u[i]);
}

/*
 * Token-to-expert grouping [P]:
 *   counts[e]   = number of (t, k) with idx[t][k] = e
 *   offsets[0]  = 0, offsets[e+1] = offsets[e] + counts[e]
 *   perm        = the pairs p = t*K + k listed expert by expert, and inside an
 *                 expert in increasing p (stable).
 * Returns 0, or -1 if an index lies outside 0..E-1.
 */
/* [TP] on the result of orc_route (idx, w and the scores s [T][E]): drops
 * the low-weight tail of each token's K experts.  p <= 0 keeps all K.  The
 * sums are of at most K floats in [2^-24, 1] (multiples of 2^-47 below 2^5),
 * so every one is exact in double. */
void orc_topp(int32_t *idx, float *w, const float *s, int T, int E, int K, float routed_scale, double p)
{
    if (p <= 0.0) return;
    for (int t = 0; t < T; t++) {
        int32_t *it = idx + (size_t)t * K;
        float *wt = w + (size_t)t * K;
        const float *st = s + (size_t)t * E;
        double total = 0.0;
        for (int k = 0; k < K; k++) total += (double)st[it[k]];
        const double limit = p * total;
        unsigned char keep[64];
        double kept = 0.0;
        for (int k = 0; k < K; k++) {
            /* the scores ranked before slot k: larger, or equal with a lower index */
            double before = 0.0;
            for (int j = 0; j < K; j++) {
                const float sj = st[it[j]], sk = st[it[k]];
                if (sj > sk || (sj == sk && it[j] < it[k])) before += (double)sj;
            }
            keep[k] = before < limit;
            if (keep[k]) kept += (double)st[it[k]];
        }
        for (int k = 0; k < K; k++) {
            if (keep[k]) {
                wt[k] = (float)((double)st[it[k]] / kept) * routed_scale;
            } else {
                it[k] = -1;
                wt[k] = 0.0f;
            }
        }
    }
}

/* Grouping ([P]): index -1 marks a slot dropped by [TP]; it is not grouped. */
int orc_group(int32_t *counts, int32_t *offsets, int32_t *perm,
              const int32_t *idx, int T, int E, int K)
{
    const long long n = (long long)T * K;
    for (int e = 0; e < E; e++) counts[e] = 0;
    for (long long p = 0; p < n; p++) {
        if (idx[p] == -1) continue;
        if (idx[p] < 0 || idx[p] >= E) return -1;
        counts[idx[p]]++;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; e++) offsets[e + 1] = offsets[e] + counts[e];
    /* fill each expert's list by walking the pairs in order */
    for (int e = 0; e < E; e++) counts[e] = 0;
    for (long long p = 0; p < n; p++) {
        const int e = idx[p];
        if (e < 0) continue;
        perm[offsets[e] + counts[e]] = (int32_t)p;
        counts[e]++;
    }
    return 0;
}

/*
 * The routed weighted sum [A]:  y_t = (float) sum_k w_tk * expert_{idx_tk}(x_t)
 * with each expert output the fp32 result of orc_expert, widened to double,
 * and the K terms added in slot order.  `ptrs` holds 6 pointers per expert
 * (w1p, w1s, w3p, w3s, w2p, w2s) indexed by expert id; only the selected
 * experts are read, so unselected entries may be NULL.  `tmp` holds
 * 3F + D floats.  Tokens run one after another; rows inside each GEMV run in
 * parallel.
 */
void orc_moe(float *y, const float *x, int T, const uint8_t *const *ptrs,
             const int32_t *idx, const float *w, int D, int F, int K, float *tmp)
{
    float *ye = tmp + 3 * F;
    double acc[8192];
    for (int t = 0; t < T; t++) {
        for (int i = 0; i < D; i++) acc[i] = 0.0;
        for (int k = 0; k < K; k++) {
            const int e = idx[(size_t)t * K + k];
            if (e < 0) continue;                  /* dropped by [TP] */
            const uint8_t *const *p = ptrs + (size_t)6 * e;
            orc_expert(ye, NULL, NULL, NULL, tmp, x + (size_t)t * D,
                       p[0], p[1], p[2], p[3], p[4], p[5], D, F);
            const double wk = (double)w[(size_t)t * K + k];
            for (int i = 0; i < D; i++) acc[i] += wk * (double)ye[i];
        }
        for (int i = 0; i < D; i++) y[(size_t)t * D + i] = (float)acc[i];
    }
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
