/*
 * moe_oracle.c -- plain, slow CPU oracle for one GLM-5.2 routed-MoE layer.
 *
 * TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the
 * benchmark's CPU-baseline leg, never by the product path.  It shares no code
 * with the CUDA library.  Build: C11, -O2 -ffp-contract=off, no fast-math, so
 * every float operation below is one IEEE fp32 operation in source order.
 *
 * Each function states the passage it restates; the page names are spelled
 * out in moe_oracle.h ([A] = reader.mx article, [B] = besthub.dev summary).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *  - sigmoid has the same form as siluf: 1/(1+expf(-x));
 *  - the router weight is [E, D] out-major and the logits are accumulated in
 *    fp32 in ascending d order (the matmul body is not shown);
 *  - scales are applied as ((float)acc * s_act) * s_row;
 *  - the shared expert is a full-size int4 SwiGLU expert with weight 1.0,
 *    added after the routed experts;
 *  - the intermediate h of every expert is requantised per row to int8 with
 *    the same quantiser as the layer input (integer path at every batch size).
 *
 * No parity pin is missing: every function here is checked by the non-GPU
 * tests against worked examples, closed forms, brute force or numpy.
 */
#include "moe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

int orc_version(void) { return 1; }

void orc_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int orc_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------------------
 * int4 weights.  [A] §06 (C packer and Python converter), [B] §06.
 * Row scale s = amax/7, floored at 1e-8; each value becomes the nearest
 * integer of w/s (a true division, ties to even as lrintf / np.rint), clamped
 * to [-8, 7], stored offset by +8 as a nibble; element 2j is the low nibble of
 * byte j, element 2j+1 the high nibble; an odd row pads the last high nibble
 * with the code for 0 (i.e. 8).
 * ------------------------------------------------------------------------- */
static int quant_nibble(float v, float s) {
    int q = (int)lrintf(v / s);
    if (q < -8) q = -8;
    if (q > 7) q = 7;
    return q + 8;
}

void orc_pack_int4(const float *w, uint8_t *q4, float *scale, int64_t O, int64_t I) {
    const int64_t nbytes = (I + 1) / 2;
#pragma omp parallel for schedule(static)
    for (int64_t o = 0; o < O; o++) {
        const float *row = w + o * I;
        float amax = 0.f;
        for (int64_t i = 0; i < I; i++) {
            float a = fabsf(row[i]);
            if (a > amax) amax = a;
        }
        float s = amax / 7.f;
        if (s < 1e-8f) s = 1e-8f;
        scale[o] = s;
        uint8_t *dst = q4 + o * nbytes;
        for (int64_t j = 0; j < nbytes; j++) {
            int lo = quant_nibble(row[2 * j], s);
            int hi = (2 * j + 1 < I) ? quant_nibble(row[2 * j + 1], s) : 8;
            dst[j] = (uint8_t)(lo | (hi << 4));
        }
    }
}

/* ---------------------------------------------------------------------------
 * FP8 checkpoint decoding.  [A] §06 "FP8 block scale 解码" and the model
 * config (quant_method fp8, fmt e4m3, weight_block_size [128, 128]); [B] §06.
 * The checkpoint stores each weight as one FP8 E4M3 byte and one fp32
 * scale_inv per 128 x 128 block; the converter widens the bytes to fp32 and
 * multiplies element (o, i) by scale_inv[o / 128][i / 128] (an fp32 product),
 * then packs the result to int4 with the row packer below.
 *
 * E4M3 ("fn" variant, the only one with 448 as its largest value): bit 7 is
 * the sign, bits 6..3 the exponent e (bias 7), bits 2..0 the mantissa m.
 * e > 0: (1 + m/8) * 2^(e-7); e == 0: (m/8) * 2^-6 (subnormal); the codes
 * S.1111.111 are NaN and there is no infinity.  Written from that definition.
 * ------------------------------------------------------------------------- */
float orc_fp8_e4m3_decode(uint8_t b) {
    const int neg = b >> 7, e = (b >> 3) & 15, m = b & 7;
    if (e == 15 && m == 7) return NAN;
    /* both cases are an integer times a power of two: exact in fp32 */
    const float v = e == 0 ? ldexpf((float)m, -9) : ldexpf((float)(8 + m), e - 10);
    return neg ? -v : v;
}

void orc_fp8_block_dequant(const uint8_t *w8, const float *scale_inv, float *w, int64_t O, int64_t I) {
    const int64_t nbi = (I + 127) / 128;  /* scale blocks per row of blocks */
#pragma omp parallel for schedule(static)
    for (int64_t o = 0; o < O; o++)
        for (int64_t i = 0; i < I; i++)
            w[o * I + i] = orc_fp8_e4m3_decode(w8[o * I + i]) * scale_inv[(o / 128) * nbi + i / 128];
}

/* The converter's whole step for one FP8 matrix: block dequantisation, then
 * the int4 row packer ([A] §06: dequant, then quant_int4 / pack_int4). */
void orc_fp8_block_to_int4(const uint8_t *w8, const float *scale_inv, uint8_t *q4, float *scale, int64_t O,
                           int64_t I) {
    float *w = (float *)malloc(sizeof(float) * (size_t)(O * I) + 4);
    orc_fp8_block_dequant(w8, scale_inv, w, O, I);
    orc_pack_int4(w, q4, scale, O, I);
    free(w);
}

/* Inverse of the nibble layout: value = nibble - 8.  [A] §06 worked example. */
static inline int nibble_value(const uint8_t *row, int64_t i) {
    uint8_t b = row[i >> 1];
    int n = (i & 1) ? (b >> 4) : (b & 15);
    return n - 8;
}

void orc_unpack_int4(const uint8_t *q4, int8_t *v, int64_t O, int64_t I) {
    const int64_t nbytes = (I + 1) / 2;
    for (int64_t o = 0; o < O; o++)
        for (int64_t i = 0; i < I; i++) v[o * I + i] = (int8_t)nibble_value(q4 + o * nbytes, i);
}

/* ---------------------------------------------------------------------------
 * Per-row int8 activation quantiser.  [A] §12 qrow_i8, [B] §12.
 * s = amax/127 floored at 1e-12, inv = 1/s, q = nearest integer of x*inv
 * (multiplication by the reciprocal, ties to even).  |x*inv| < 127.5 so no
 * clamp is needed; none is applied.  Returns s.
 * ------------------------------------------------------------------------- */
float orc_qrow_i8(const float *x, int8_t *q, int64_t n) {
    float amax = 0.f;
    for (int64_t i = 0; i < n; i++) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    float s = amax / 127.f;
    if (s < 1e-12f) s = 1e-12f;
    const float inv = 1.f / s;
    for (int64_t i = 0; i < n; i++) q[i] = (int8_t)lrintf(x[i] * inv);
    return s;
}

void orc_quant_act(const float *x, int8_t *xq, float *sx, int64_t T, int64_t D) {
    for (int64_t t = 0; t < T; t++) sx[t] = orc_qrow_i8(x + t * D, xq + t * D, D);
}

/* Integer dot of one packed int4 row with int8 activations: the plain
 * definition sum_i w[i]*x[i] in int32 ([A] §12, the scalar tail of dot_i8i8,
 * applied to unpacked int4 values). */
int32_t orc_dot_i4_i8(const uint8_t *q4row, const int8_t *x, int64_t n) {
    int32_t acc = 0;
    for (int64_t i = 0; i < n; i++) acc += (int32_t)nibble_value(q4row, i) * (int32_t)x[i];
    return acc;
}

/* ---------------------------------------------------------------------------
 * int8 weights.  [A] §05 quantize_rows (the OLMoE prototype's per-row int8
 * weights, also the engine's fmt 1): qmax = 2^(bits-1) - 1, s = amax/qmax
 * floored at 1e-8, value = nearest integer of w/s (a true division, ties to
 * even as lrintf), clamped to [-qmax-1, qmax], one value per int8.  [A] §12
 * dot_i8i8: the int8 x int8 dot, exact in int32 (its scalar tail is the
 * plain definition).
 * ------------------------------------------------------------------------- */
void orc_quantize_rows(const float *w, int8_t *q, float *scale, int64_t O, int64_t I, int bits) {
    const int qmax = (1 << (bits - 1)) - 1;
#pragma omp parallel for schedule(static)
    for (int64_t o = 0; o < O; o++) {
        const float *row = w + o * I;
        float amax = 0.f;
        for (int64_t i = 0; i < I; i++) {
            float a = fabsf(row[i]);
            if (a > amax) amax = a;
        }
        float s = amax / (float)qmax;
        if (s < 1e-8f) s = 1e-8f;
        scale[o] = s;
        for (int64_t i = 0; i < I; i++) {
            int v = (int)lrintf(row[i] / s);
            if (v > qmax) v = qmax;
            if (v < -qmax - 1) v = -qmax - 1;
            q[o * I + i] = (int8_t)v;
        }
    }
}

int32_t orc_dot_i8_i8(const int8_t *w, const int8_t *x, int64_t n) {
    int32_t acc = 0;
    for (int64_t i = 0; i < n; i++) acc += (int32_t)w[i] * (int32_t)x[i];
    return acc;
}

/* ---------------------------------------------------------------------------
 * Router.  [A] §11 ("sigmoid(logit)+bias picks top-K, weight is plain
 * sigmoid"), [B] §11, model config (scoring_func sigmoid, 256 experts, top-8,
 * routed_scaling_factor 2.5).
 * For each token: logit[e] = x . Wr[e]; p = sigmoid(logit); c = p + bias.
 * K rounds: pick the not-yet-taken expert with the largest c, scanning e in
 * ascending order with a strict '>' starting from -1e30 (the lowest index wins
 * an exact tie).  weight = p[pick] * routed_scale (no renormalisation).
 * ------------------------------------------------------------------------- */
static float sigmoid_f(float v) { return 1.f / (1.f + expf(-v)); }

void orc_router(const float *x, const float *Wr, const float *bias, int T, int D, int E,
                int K, float routed_scale, int32_t *idx, float *w, float *p_out) {
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; t++) {
        const float *xt = x + (int64_t)t * D;
        float *p = (float *)malloc(sizeof(float) * (size_t)E);
        float *c = (float *)malloc(sizeof(float) * (size_t)E);
        unsigned char *taken = (unsigned char *)calloc((size_t)E, 1);
        for (int e = 0; e < E; e++) {
            const float *we = Wr + (int64_t)e * D;
            float logit = 0.f;
            for (int d = 0; d < D; d++) logit += xt[d] * we[d];
            p[e] = sigmoid_f(logit);
            c[e] = p[e] + bias[e];
        }
        for (int k = 0; k < K; k++) {
            int best = -1;
            float bv = -1e30f;
            for (int e = 0; e < E; e++)
                if (!taken[e] && c[e] > bv) {
                    bv = c[e];
                    best = e;
                }
            idx[(int64_t)t * K + k] = best;
            if (best >= 0) taken[best] = 1;
            w[(int64_t)t * K + k] = (best >= 0 ? p[best] : 0.f) * routed_scale;
        }
        if (p_out) memcpy(p_out + (int64_t)t * E, p, sizeof(float) * (size_t)E);
        free(p);
        free(c);
        free(taken);
    }
}

/* Double twin of the router scores: gap[t] = c_(K) - c_(K+1), the margin
 * between the K-th and (K+1)-th largest selection score computed entirely in
 * double.  +inf when K >= E.  Used only to decide whether a token's selection
 * is numerically unambiguous. */
void orc_router_gap_f64(const float *x, const float *Wr, const float *bias, int T, int D,
                        int E, int K, double *gap) {
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; t++) {
        const float *xt = x + (int64_t)t * D;
        double *c = (double *)malloc(sizeof(double) * (size_t)E);
        for (int e = 0; e < E; e++) {
            const float *we = Wr + (int64_t)e * D;
            double logit = 0.0;
            for (int d = 0; d < D; d++) logit += (double)xt[d] * (double)we[d];
            c[e] = 1.0 / (1.0 + exp(-logit)) + (double)bias[e];
        }
        if (K >= E) {
            gap[t] = INFINITY;
        } else {
            /* the K-th largest and the (K+1)-th largest by repeated extraction */
            unsigned char *used = (unsigned char *)calloc((size_t)E, 1);
            double kth = 0.0, next = 0.0;
            for (int k = 0; k <= K; k++) {
                int best = -1;
                for (int e = 0; e < E; e++)
                    if (!used[e] && (best < 0 || c[e] > c[best])) best = e;
                used[best] = 1;
                if (k == K - 1) kth = c[best];
                if (k == K) next = c[best];
            }
            gap[t] = kth - next;
            free(used);
        }
        free(c);
    }
}

/* Adaptive expert top-p.  [C] 使用方法 item 4 (--topp: adaptive expert top-p,
 * fewer expert reads) and [A] §11 (the union runs over the first keff[s]
 * selections of token s; how keff is chosen is not shown).  Reading: keff is
 * the length of the shortest prefix of the token's selections, in selection
 * order, whose routing weights sum to at least top_p times the sum of all K
 * weights (sums in fp32, left to right; the bound one fp32 product), and at
 * least 1.  top_p <= 0 or >= 1 keeps all K.  The kept selections keep their
 * weights (no renormalisation), as [A]'s weighted add uses w unchanged. */
int orc_topp_keff(const float *w, int K, float top_p) {
    if (!(top_p > 0.f && top_p < 1.f)) return K;
    float total = 0.f;
    for (int k = 0; k < K; k++) total += w[k];
    const float bound = top_p * total;
    float run = 0.f;
    for (int k = 0; k < K; k++) {
        run += w[k];
        if (run >= bound) return k + 1;
    }
    return K;
}

/* Union of the routed experts over a batch in first-appearance order over
 * (token, slot).  [A] §11 (each expert's weights are read once per batch),
 * [B] §11.  Returns the number of distinct experts. */
int orc_union(const int32_t *idx, int T, int K, int E, int32_t *uniq) {
    unsigned char *seen = (unsigned char *)calloc((size_t)E, 1);
    int nu = 0;
    for (int t = 0; t < T; t++)
        for (int k = 0; k < K; k++) {
            int e = idx[(int64_t)t * K + k];
            if (e >= 0 && e < E && !seen[e]) {
                seen[e] = 1;
                uniq[nu++] = e;
            }
        }
    free(seen);
    return nu;
}

/* RMSNorm.  [A] §04: mean of squares accumulated in double, r = 1/sqrtf of
 * (float)(ms/D) + eps, out = x * r * w evaluated left to right in fp32. */
void orc_rmsnorm(const float *x, const float *w, float *out, int D, float eps) {
    double ms = 0.0;
    for (int i = 0; i < D; i++) ms += (double)x[i] * (double)x[i];
    const float r = 1.f / sqrtf((float)(ms / D) + eps);
    for (int i = 0; i < D; i++) out[i] = x[i] * r * w[i];
}

/* ---------------------------------------------------------------------------
 * One SwiGLU expert on one activation row, integer path.
 * [A] §11 (gate/up, siluf(g)*u, down), §04 siluf, §12 (int8 activations x
 * int4 weights, or int8 weights for fmt 1, integer dot, then scales).
 *   ag[o] = dot(gate row o, xq), au[o] likewise            (int32, exact)
 *   g = (ag*sx)*sg[o], u = (au*sx)*su[o], h[o] = g/(1+expf(-g)) * u
 *   (hq, sh) = per-row int8 quantisation of h
 *   ad[o] = dot(down row o, hq); y[o] = (ad*sh)*sd[o]
 * ------------------------------------------------------------------------- */
/* Dot of output row o of a weight matrix with n columns (int4 packed or
 * int8 rows) against int8 activations. */
static int32_t row_dot(const uint8_t *mat, int bits, int64_t o, const int8_t *x, int64_t n) {
    if (bits == 8) return orc_dot_i8_i8((const int8_t *)mat + o * n, x, n);
    return orc_dot_i4_i8(mat + o * ((n + 1) / 2), x, n);
}

static void expert_row(const OrcExpert *ex, int bits, int D, int I, const int8_t *xq, float sx,
                       float *h, int8_t *hq, float *y, int32_t *gacc, int32_t *uacc,
                       float *sh_out, int32_t *dacc) {
#pragma omp parallel for schedule(static)
    for (int o = 0; o < I; o++) {
        int32_t ag = row_dot(ex->gq, bits, o, xq, D);
        int32_t au = row_dot(ex->uq, bits, o, xq, D);
        if (gacc) gacc[o] = ag;
        if (uacc) uacc[o] = au;
        float g = ((float)ag * sx) * ex->gs[o];
        float u = ((float)au * sx) * ex->us[o];
        float silu = g / (1.f + expf(-g));
        h[o] = silu * u;
    }
    const float sh = orc_qrow_i8(h, hq, I);
    if (sh_out) *sh_out = sh;
#pragma omp parallel for schedule(static)
    for (int o = 0; o < D; o++) {
        int32_t ad = row_dot(ex->dq, bits, o, hq, I);
        if (dacc) dacc[o] = ad;
        y[o] = ((float)ad * sh) * ex->ds[o];
    }
}

/* ---------------------------------------------------------------------------
 * The layer.  [A] §11 and §12, [B] §11:
 *   xq, sx = per-token int8 quantisation of x;
 *   router on the fp32 x (not on xq);
 *   adaptive top-p: each token keeps its first keff selections (orc_topp_keff);
 *   union of the kept experts; for each union expert, in union order,
 *   every (token, slot) routed to it runs the expert and adds w * y into
 *   out[token] (fp32, one rounding for the product, one for the sum);
 *   then the shared expert adds its y with weight 1.
 * Returns 0, or -1 when a needed expert entry is NULL / K is out of range.
 * ------------------------------------------------------------------------- */
int orc_layer_forward(const OrcLayer *L, const float *x, int T, float *out, OrcDebug *dbg) {
    const int D = L->D, I = L->I, E = L->E, K = L->K, S = L->K + L->n_shared;
    if (K < 1 || K > E || L->n_shared < 0 || L->n_shared > 1) return -1;
    if (L->weight_bits != 0 && L->weight_bits != 4 && L->weight_bits != 8) return -1;
    int8_t *xq = (int8_t *)malloc((size_t)T * D + 1);
    float *sx = (float *)malloc(sizeof(float) * ((size_t)T + 1));
    int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * ((size_t)T * K + 1));
    float *w = (float *)malloc(sizeof(float) * ((size_t)T * K + 1));
    int32_t *uniq = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    float *h = (float *)malloc(sizeof(float) * (size_t)I);
    int8_t *hq = (int8_t *)malloc((size_t)I);
    float *y = (float *)malloc(sizeof(float) * (size_t)D);
    int rc = 0;

    orc_quant_act(x, xq, sx, T, D);
    orc_router(x, L->Wr, L->bias, T, D, E, K, L->routed_scale, idx, w, NULL);
    /* adaptive top-p: selections past keff are dropped (id -1, weight 0) */
    for (int t = 0; t < T; t++) {
        const int keff = orc_topp_keff(w + (int64_t)t * K, K, L->top_p);
        for (int k = keff; k < K; k++) {
            idx[(int64_t)t * K + k] = -1;
            w[(int64_t)t * K + k] = 0.f;
        }
    }
    const int nu = orc_union(idx, T, K, E, uniq);
    memset(out, 0, sizeof(float) * (size_t)T * D);

    /* routed experts in union order, then the shared expert */
    for (int u = 0; u < nu + L->n_shared && rc == 0; u++) {
        const int shared = (u >= nu);
        const int e = shared ? E : uniq[u];
        const OrcExpert *ex = &L->experts[e];
        if (!ex->gq || !ex->uq || !ex->dq || !ex->gs || !ex->us || !ex->ds) {
            rc = -1;
            break;
        }
        for (int t = 0; t < T; t++) {
            for (int k = 0; k < (shared ? 1 : K); k++) {
                if (!shared && idx[(int64_t)t * K + k] != e) continue;
                const int slot = shared ? K : k;
                const float wt = shared ? 1.f : w[(int64_t)t * K + k];
                const int64_t ts = (int64_t)t * S + slot;
                expert_row(ex, L->weight_bits == 8 ? 8 : 4, D, I, xq + (int64_t)t * D, sx[t], h, hq, y,
                           dbg && dbg->gate_acc ? dbg->gate_acc + ts * I : NULL,
                           dbg && dbg->up_acc ? dbg->up_acc + ts * I : NULL,
                           dbg && dbg->sh ? dbg->sh + ts : NULL,
                           dbg && dbg->down_acc ? dbg->down_acc + ts * D : NULL);
                if (dbg && dbg->hq) memcpy(dbg->hq + ts * I, hq, (size_t)I);
                if (dbg && dbg->y) memcpy(dbg->y + ts * D, y, sizeof(float) * (size_t)D);
                float *ot = out + (int64_t)t * D;
                for (int d = 0; d < D; d++) ot[d] += wt * y[d];
            }
        }
    }

    if (dbg) {
        if (dbg->idx) memcpy(dbg->idx, idx, sizeof(int32_t) * (size_t)T * K);
        if (dbg->w) memcpy(dbg->w, w, sizeof(float) * (size_t)T * K);
        if (dbg->xq) memcpy(dbg->xq, xq, (size_t)T * D);
        if (dbg->sx) memcpy(dbg->sx, sx, sizeof(float) * (size_t)T);
        if (dbg->uniq) memcpy(dbg->uniq, uniq, sizeof(int32_t) * (size_t)nu);
        if (dbg->n_uniq) *dbg->n_uniq = nu;
    }
    free(xq); free(sx); free(idx); free(w); free(uniq); free(h); free(hq); free(y);
    return rc;
}

/* Residual block of the layer stack: x <- x + MoE(RMSNorm(x)).  [A] §04
 * (layer order: post-attention norm, MoE, residual add). */
int orc_block_forward(const OrcLayer *L, float *x, const float *norm_w, float eps, int T) {
    const int D = L->D;
    float *n = (float *)malloc(sizeof(float) * (size_t)T * D + 4);
    float *o = (float *)malloc(sizeof(float) * (size_t)T * D + 4);
    for (int t = 0; t < T; t++) orc_rmsnorm(x + (int64_t)t * D, norm_w, n + (int64_t)t * D, D, eps);
    int rc = orc_layer_forward(L, n, T, o, NULL);
    if (rc == 0)
        for (int64_t j = 0; j < (int64_t)T * D; j++) x[j] += o[j];
    free(n);
    free(o);
    return rc;
}
