/*
 * CPU oracle for the top-k MoE layer: gate, capacity/locations, encode, expert
 * FFN, decode, and the backward of encode/decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the package's smoke check and the
 * bench's CPU-baseline leg may load this library.  It shares no code, header,
 * table or constant with the CUDA library, and the CUDA library never calls it.
 *
 * Plain loops, no blocking or fusion.  Arithmetic is in double unless a
 * function states the precision the method fixes:
 *   - gate logits are fp32 (the decision top-k takes is made in fp32; see
 *     orc_gate_logits for the exact summation order);
 *   - combine (decode) and its K0 twin (encode backward) accumulate in fp32,
 *     as the DeepSpeed index-dispatch change requires (PR #8195, change 3:
 *     "combine accumulates in fp32").
 * Values that are bf16 in the layer are passed in as fp32 (exact widening);
 * functions with a `bf16` flag round their outputs to bf16 (round to nearest,
 * ties to even) and return them stored in fp32.
 *
 * Sources (the pages this oracle restates):
 *   [Tutel]   "Tutel" project profile, FAQ on gate_type k and capacity_factor,
 *             and the key-configuration table (MOELayer gate_type / experts).
 *   [Blog]    "MoE training systems: DeepSpeed-MoE vs Tutel", section 1.4
 *             (kernel optimisation: dense mapping table, fused top-k + cumsum)
 *             and section 3.5 (fast encode/decode; dynamic capacity factor).
 *   [PR8195]  DeepSpeed PR #8195 (follow-up to #8174), changes 1 and 3.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_ACT_RELU 0
#define ORC_ACT_GELU 1
#define ORC_ACT_SWIGLU 2

/* ---------------------------------------------------------------- helpers */

/* Round a double to the nearest bf16 value (ties to even), returned as float.
 * bf16 keeps 8 significant bits; its smallest subnormal step is 2^-133. */
static float round_bf16(double v)
{
    if (v == 0.0 || !isfinite(v)) return (float)v;
    int ex;
    frexp(v, &ex);               /* |v| in [2^(ex-1), 2^ex) */
    int lsb = ex - 8;            /* weight of the last kept bit */
    if (lsb < -133) lsb = -133;
    double r = nearbyint(ldexp(v, -lsb));   /* default mode: ties to even */
    double res = ldexp(r, lsb);
    if (fabs(res) > 3.3895313892515355e38) return (float)copysign(INFINITY, v);
    return (float)res;           /* exact: res has at most 8 significant bits */
}

static float round_to(double v, int bf16) { return bf16 ? round_bf16(v) : (float)v; }

float orc_round_bf16(double v) { return round_bf16(v); }

void orc_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int orc_get_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------- gate */

/* Gate logits l[t,j] = x[t,:] . wg[:,j] + bias[j]   ([Tutel] gate_type 'top').
 *
 * Precision and order (the reading adopted here, so that top-k is
 * reproducible bit for bit): fp32 with one rounding per fused multiply-add,
 * then one fp32 add of bias[j] (skipped when bias is NULL).  The summation
 * order depends on `chunk`:
 *   chunk = V > 0 (V = 8 for bf16 x, 4 for fp32 x; used for e <= 32): the
 *     features are cut into chunks of V consecutive elements; chunk c belongs
 *     to lane (c mod 32).  Each of the 32 lanes keeps one accumulator from +0
 *     and applies acc = fmaf(x[t,i], wg[i,j], acc) to its features in
 *     ascending i.  The lanes are then combined by a butterfly: for
 *     o = 16, 8, 4, 2, 1 every lane l takes acc[l] + acc[l xor o] (one fp32
 *     add; both partners get the same value), and the logit is lane 0's.
 *   chunk = 0 (used for e > 32): one accumulator from +0, updated with fmaf
 *     for i = 0, 1, ..., m-1 in ascending order.
 * x is [s, m] row-major, wg is [m, e] row-major, logits is [s, e]. */
void orc_gate_logits(const float *x, const float *wg, const float *bias,
                     int64_t s, int m, int e, int chunk, float *logits)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < s; t++) {
        float *out = logits + t * e;
        if (chunk <= 0) {
            /* out[j] is logit (t, j)'s single accumulator; the loops visit i
             * in ascending order for every j (walking wg row by row). */
            for (int j = 0; j < e; j++) out[j] = 0.0f;
            for (int i = 0; i < m; i++) {
                const float xi = x[t * m + i];
                const float *wr = wg + (int64_t)i * e;
                for (int j = 0; j < e; j++) out[j] = fmaf(xi, wr[j], out[j]);
            }
        } else {
            float *lane = (float *)malloc(sizeof(float) * 32 * (size_t)e);
            float nxt[32];
            for (int q = 0; q < 32 * e; q++) lane[q] = 0.0f;
            /* lane[l * e + j]: lane l's accumulator for expert j; features
             * are visited in ascending order, so each lane's own features
             * are too. */
            for (int i = 0; i < m; i++) {
                const int l = (i / chunk) % 32;
                const float xi = x[t * m + i];
                const float *wr = wg + (int64_t)i * e;
                for (int j = 0; j < e; j++) lane[l * e + j] = fmaf(xi, wr[j], lane[l * e + j]);
            }
            for (int j = 0; j < e; j++) {
                float v[32];
                for (int l = 0; l < 32; l++) v[l] = lane[l * e + j];
                for (int o = 16; o >= 1; o >>= 1) {
                    for (int l = 0; l < 32; l++) nxt[l] = v[l] + v[l ^ o];
                    for (int l = 0; l < 32; l++) v[l] = nxt[l];
                }
                out[j] = v[0];
            }
            free(lane);
        }
        if (bias)
            for (int j = 0; j < e; j++) out[j] = out[j] + bias[j];
    }
}

typedef struct { float v; int j; } orc_vj;

/* Larger logit first; equal logits: lower expert index first. */
static int cmp_logit_desc(const void *a, const void *b)
{
    const orc_vj *p = (const orc_vj *)a, *q = (const orc_vj *)b;
    if (p->v > q->v) return -1;
    if (p->v < q->v) return 1;
    return (p->j > q->j) - (p->j < q->j);
}

/* Top-k routing: route r of token t is the expert in position r when all e
 * experts are ordered by (logit descending, index ascending).  Selecting on
 * logits equals selecting on softmax probabilities (softmax is monotone).
 * idx is route-major [k, s]: idx[r*s + t]. */
void orc_topk(const float *logits, int64_t s, int e, int k, int32_t *idx)
{
    orc_vj *a = (orc_vj *)malloc(sizeof(orc_vj) * (size_t)e);
    for (int64_t t = 0; t < s; t++) {
        for (int j = 0; j < e; j++) { a[j].v = logits[t * e + j]; a[j].j = j; }
        qsort(a, (size_t)e, sizeof(orc_vj), cmp_logit_desc);
        for (int r = 0; r < k; r++) idx[(int64_t)r * s + t] = a[r].j;
    }
    free(a);
}

/* Gate values (double, rounded once to fp32): p = softmax over all e logits;
 * route r's gate is p[idx[r,t]], divided by the sum of the k selected p's when
 * `normalize` is set.  Normalisation happens before any capacity drop and is
 * not redone after drops. */
void orc_gates(const float *logits, const int32_t *idx, int64_t s, int e, int k,
               int normalize, float *gates)
{
    for (int64_t t = 0; t < s; t++) {
        const float *l = logits + t * e;
        double mx = l[0];
        for (int j = 1; j < e; j++) if (l[j] > mx) mx = l[j];
        double z = 0.0;
        for (int j = 0; j < e; j++) z += exp((double)l[j] - mx);
        double sel = 0.0;
        for (int r = 0; r < k; r++) sel += exp((double)l[idx[(int64_t)r * s + t]] - mx) / z;
        for (int r = 0; r < k; r++) {
            double p = exp((double)l[idx[(int64_t)r * s + t]] - mx) / z;
            gates[(int64_t)r * s + t] = (float)(normalize ? p / sel : p);
        }
    }
}

/* Backward of the gate values ([Tutel] gate_type 'top': gates are softmax
 * probabilities of the k selected experts, renormalised over them when
 * `normalize`).  Top-k selection is piecewise constant, so gradients flow only
 * through the softmax.  In double, from the forward's fp32 logits:
 *   p = softmax(l) over all e experts, A = sum_r dg_r g_r with g_r the gate
 *   value of route r (recomputed in double);
 *   normalize:  g_r = p_{i_r} / sum_q p_{i_q};  dl_{i_r} = g_r (dg_r - A), other
 *               experts 0  (the renormalised gates are a softmax over the
 *               selected logits alone);
 *   otherwise:  g_r = p_{i_r};  dl_j = -p_j A + sum_{r: i_r = j} dg_r g_r.
 * Then through l = x Wg + b:  d_wg[i,j] = sum_t x[t,i] dl[t,j],
 * d_bias[j] = sum_t dl[t,j],  d_x[t,i] = sum_j dl[t,j] wg[i,j].
 * Shapes: x [s, m], wg [m, e], logits [s, e], idx / d_gates [k, s];
 * outputs d_logits [s, e], d_wg [m, e], d_bias [e], d_x [s, m] (double). */
void orc_gate_bwd(const float *x, const float *wg, const float *logits, const int32_t *idx,
                  const float *d_gates, int64_t s, int m, int e, int k, int normalize,
                  double *d_logits, double *d_wg, double *d_bias, double *d_x)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < s; t++) {
        const float *l = logits + t * e;
        double *dl = d_logits + t * e;
        double mx = l[0];
        for (int j = 1; j < e; j++) if (l[j] > mx) mx = l[j];
        double z = 0.0;
        for (int j = 0; j < e; j++) z += exp((double)l[j] - mx);
        double sel = 0.0;
        for (int r = 0; r < k; r++) sel += exp((double)l[idx[(int64_t)r * s + t]] - mx) / z;
        double a = 0.0;
        for (int r = 0; r < k; r++) {
            const int j = idx[(int64_t)r * s + t];
            const double p = exp((double)l[j] - mx) / z;
            const double g = normalize ? p / sel : p;
            a += (double)d_gates[(int64_t)r * s + t] * g;
        }
        for (int j = 0; j < e; j++) dl[j] = normalize ? 0.0 : -(exp((double)l[j] - mx) / z) * a;
        for (int r = 0; r < k; r++) {
            const int j = idx[(int64_t)r * s + t];
            const double p = exp((double)l[j] - mx) / z;
            const double g = normalize ? p / sel : p;
            const double dg = d_gates[(int64_t)r * s + t];
            dl[j] += normalize ? g * (dg - a) : dg * g;
        }
        for (int i = 0; i < m; i++) {
            double acc = 0.0;
            for (int j = 0; j < e; j++) acc += dl[j] * (double)wg[(int64_t)i * e + j];
            d_x[t * m + i] = acc;
        }
    }
    for (int j = 0; j < e; j++) {
        double acc = 0.0;
        for (int64_t t = 0; t < s; t++) acc += d_logits[t * e + j];
        d_bias[j] = acc;
    }
#pragma omp parallel for schedule(static)
    for (int i = 0; i < m; i++)
        for (int j = 0; j < e; j++) {
            double acc = 0.0;
            for (int64_t t = 0; t < s; t++) acc += (double)x[t * m + i] * d_logits[t * e + j];
            d_wg[(int64_t)i * e + j] = acc;
        }
}

/* --------------------------------------------------------------- capacity */

/* Slot assignment as a sequential queue ([Blog] 1.4: the cumsum over the
 * token-to-expert table; route-priority order): for r = 0..k-1, for
 * t = 0..s-1, loc[r,t] = fill[idx[r,t]]++.  needed[e] = routes sent to e
 * before any drop.  Locations are returned un-clipped. */
void orc_locations(const int32_t *idx, int64_t s, int e, int k, int32_t *loc, int64_t *needed)
{
    for (int j = 0; j < e; j++) needed[j] = 0;
    for (int r = 0; r < k; r++)
        for (int64_t t = 0; t < s; t++) {
            int32_t x = idx[(int64_t)r * s + t];
            loc[(int64_t)r * s + t] = (int32_t)needed[x]++;
        }
}

/* ceil(x / e) for a non-negative double x that is exact (f*k*s with f a float
 * and k*s < 2^29 is exact in double). */
static int64_t ceil_div_exact(double x, int e)
{
    int64_t c = (int64_t)ceil(x / (double)e);
    while (c > 0 && (double)(c - 1) * (double)e >= x) c--;
    while ((double)c * (double)e < x) c++;
    return c;
}

/* Capacity c from capacity_factor f ([Tutel] FAQ; [Blog] 3.5 "dynamic capacity
 * factor"):
 *   f > 0: fixed factor, c = ceil(f*k*s/e);
 *   f = 0: just enough that nothing is dropped, c = max_e needed[e];
 *   f < 0: -f is an upper bound, c = min(ceil(-f*k*s/e), max_e needed[e]). */
int64_t orc_capacity(double f, int64_t s, int e, int k, const int64_t *needed)
{
    int64_t mx = 0;
    for (int j = 0; j < e; j++) if (needed[j] > mx) mx = needed[j];
    if (f > 0) return ceil_div_exact(f * (double)k * (double)s, e);
    if (f == 0) return mx;
    int64_t bound = ceil_div_exact(-f * (double)k * (double)s, e);
    return bound < mx ? bound : mx;
}

/* --------------------------------------------------- encode / decode (sparse) */

/* Fast encode ([Blog] 3.5, kernel K1 forward): for each kept route (r,t)
 * (loc < c), buf[idx, loc, :] = x[t, :].  Unweighted copy.  buf is the
 * physical [e, cmax, m] buffer; rows not written are left untouched. */
void orc_encode(const float *x, const int32_t *idx, const int32_t *loc, int64_t c,
                int64_t s, int m, int e, int k, int64_t cmax, float *buf)
{
    (void)e;
    for (int r = 0; r < k; r++)
        for (int64_t t = 0; t < s; t++) {
            int64_t o = (int64_t)r * s + t;
            if (loc[o] >= c) continue;
            memcpy(buf + ((int64_t)idx[o] * cmax + loc[o]) * m, x + t * m, sizeof(float) * (size_t)m);
        }
}

/* Fast decode ([Blog] 3.5, K0 forward; [PR8195] change 3): y[t,:] =
 * sum over kept routes r of gates[r,t] * out[idx, loc, :], accumulated in fp32
 * in ascending r with acc = fmaf(g, v, acc) from +0, rounded once to the
 * output dtype.  A token whose routes were all dropped gets 0. */
void orc_decode(const float *out, const int32_t *idx, const int32_t *loc, const float *gates,
                int64_t c, int64_t s, int m, int e, int k, int64_t cmax, int bf16, float *y)
{
    (void)e;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < s; t++) {
        for (int i = 0; i < m; i++) {
            float acc = 0.0f;
            for (int r = 0; r < k; r++) {
                int64_t o = (int64_t)r * s + t;
                if (loc[o] >= c) continue;
                acc = fmaf(gates[o], out[((int64_t)idx[o] * cmax + loc[o]) * m + i], acc);
            }
            y[t * m + i] = round_to(acc, bf16);
        }
    }
}

/* Backward of decode ([Blog] 3.5: K1 is combine's backward, K2 the cross
 * term).  For kept (r,t): d_out[idx, loc, :] = gates[r,t] * dy[t,:] (exact
 * product rounded once to the dtype) and d_gates[r,t] = sum_i dy[t,i] *
 * out[idx, loc, i] (double, rounded to fp32).  Dropped routes: d_gates = 0. */
void orc_decode_bwd(const float *dy, const float *out, const int32_t *idx, const int32_t *loc,
                    const float *gates, int64_t c, int64_t s, int m, int e, int k, int64_t cmax,
                    int bf16, float *d_out, float *d_gates)
{
    (void)e;
    for (int r = 0; r < k; r++)
        for (int64_t t = 0; t < s; t++) {
            int64_t o = (int64_t)r * s + t;
            if (loc[o] >= c) { d_gates[o] = 0.0f; continue; }
            int64_t row = ((int64_t)idx[o] * cmax + loc[o]) * m;
            double dot = 0.0;
            for (int i = 0; i < m; i++) {
                d_out[row + i] = round_to((double)gates[o] * (double)dy[t * m + i], bf16);
                dot += (double)dy[t * m + i] * (double)out[row + i];
            }
            d_gates[o] = (float)dot;
        }
}

/* Backward of encode ([Blog] 3.5: K0 with unit weights): dx[t,:] = sum over
 * kept routes of d_buf[idx, loc, :], fp32 accumulation in ascending r from +0,
 * rounded once to the dtype. */
void orc_encode_bwd(const float *d_buf, const int32_t *idx, const int32_t *loc, int64_t c,
                    int64_t s, int m, int e, int k, int64_t cmax, int bf16, float *dx)
{
    (void)e;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < s; t++) {
        for (int i = 0; i < m; i++) {
            float acc = 0.0f;
            for (int r = 0; r < k; r++) {
                int64_t o = (int64_t)r * s + t;
                if (loc[o] >= c) continue;
                acc = acc + d_buf[((int64_t)idx[o] * cmax + loc[o]) * m + i];
            }
            dx[t * m + i] = round_to(acc, bf16);
        }
    }
}

/* ------------------------------------------------------------- expert FFN */

/* One expert MLP row ([Tutel] experts {'type': 'ffn', hidden_size_per_expert,
 * has_fc1_bias, has_fc2_bias}).  For the requested (expert, row) pairs:
 *   ReLU/GELU: hid = act(x . w1[e]^T + b1[e]),  out = hid . w2[e]^T + b2[e]
 *   SwiGLU:    hid = silu(x . w1[e]^T) * (x . w3[e]^T), out = hid . w2[e]^T
 * Layouts: buf [e, cmax, m]; w1, w3 [e, h, m]; w2 [e, m, h]; b1 [e, h];
 * b2 [e, m].  Sums in double; the hidden activation is rounded to the layer
 * dtype (bf16 or fp32) before fc2, and each output once more.  GELU is the
 * exact erf form; biases may be NULL. */
void orc_ffn_rows(const float *buf, const float *w1, const float *b1, const float *w3,
                  const float *w2, const float *b2, int act, int e, int64_t cmax, int m, int h,
                  int bf16, const int32_t *row_e, const int64_t *row_j, int64_t nrows,
                  float *out_rows)
{
    (void)e;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t q = 0; q < nrows; q++) {
        int64_t ex = row_e[q];
        const float *xr = buf + (ex * cmax + row_j[q]) * m;
        float *hid = (float *)malloc(sizeof(float) * (size_t)h);
        for (int u = 0; u < h; u++) {
            const float *w1r = w1 + (ex * h + u) * (int64_t)m;
            double a = 0.0;
            for (int i = 0; i < m; i++) a += (double)xr[i] * (double)w1r[i];
            double v;
            if (act == ORC_ACT_SWIGLU) {
                const float *w3r = w3 + (ex * h + u) * (int64_t)m;
                double b = 0.0;
                for (int i = 0; i < m; i++) b += (double)xr[i] * (double)w3r[i];
                v = a / (1.0 + exp(-a)) * b;
            } else {
                if (b1) a += (double)b1[ex * h + u];
                v = act == ORC_ACT_RELU ? (a > 0.0 ? a : 0.0)
                                        : 0.5 * a * (1.0 + erf(a / sqrt(2.0)));
            }
            hid[u] = round_to(v, bf16);
        }
        for (int i = 0; i < m; i++) {
            const float *w2r = w2 + (ex * m + i) * (int64_t)h;
            double o = 0.0;
            for (int u = 0; u < h; u++) o += (double)hid[u] * (double)w2r[u];
            if (b2 && act != ORC_ACT_SWIGLU) o += (double)b2[ex * m + i];
            out_rows[q * m + i] = round_to(o, bf16);
        }
        free(hid);
    }
}

/* ---------------------------------------------------- expert FFN backward */

/* Backward of orc_ffn_rows over every kept row (row j < kept[e] of expert e),
 * for L = sum over kept rows of <d_out, out>.  The forward's roundings are
 * taken as the identity (their derivative almost everywhere); the hidden
 * activation fc2 consumed is the rounded one, recomputed exactly as the
 * forward does.  All sums in double; d_buf is rounded once to the layer
 * dtype, the weight and bias gradients once to fp32.
 *   ReLU/GELU: pre = x w1^T + b1, hid = act(pre);
 *              d_hid = d_out w2, d_pre = d_hid * act'(pre)
 *              (ReLU' = 1 where pre > 0, else 0; GELU' = Phi(z) + z phi(z));
 *   SwiGLU:    a = x w1^T, b = x w3^T, hid = silu(a) b;
 *              d_a = d_hid * b * sigma(a) (1 + a (1 - sigma(a))), d_b = d_hid * silu(a);
 *   d_w2[e] = sum_rows d_out^T hid,  d_b2[e] = sum_rows d_out,
 *   d_w1[e] = sum_rows d_pre^T x (d_a for SwiGLU),  d_b1[e] = sum_rows d_pre,
 *   d_w3[e] = sum_rows d_b^T x,  d_buf = d_pre w1 (+ d_b w3).
 * Rows of d_buf at or past kept[e] are 0.  SwiGLU has no biases: d_b1, d_b2
 * are then not written.  Any output may be NULL.  Layouts as orc_ffn_rows;
 * d_out and d_buf [e, cmax, m]. */
void orc_ffn_bwd(const float *buf, const float *w1, const float *b1, const float *w3,
                 const float *w2, int act, int e, int64_t cmax, int m, int h, int bf16,
                 const int64_t *kept, const float *d_out, float *d_buf, float *d_w1,
                 float *d_b1, float *d_w3, float *d_w2, float *d_b2)
{
    const int swiglu = act == ORC_ACT_SWIGLU;
#pragma omp parallel for schedule(dynamic, 1)
    for (int ex = 0; ex < e; ex++) {
        const int64_t rows = kept[ex];
        double *gw1 = (double *)calloc((size_t)h * m, sizeof(double));
        double *gw3 = (double *)calloc((size_t)h * m, sizeof(double));
        double *gw2 = (double *)calloc((size_t)m * h, sizeof(double));
        double *gb1 = (double *)calloc((size_t)h, sizeof(double));
        double *gb2 = (double *)calloc((size_t)m, sizeof(double));
        double *hid = (double *)malloc(sizeof(double) * (size_t)h);
        double *dp = (double *)malloc(sizeof(double) * (size_t)h);    /* d_pre or d_a */
        double *dq = (double *)malloc(sizeof(double) * (size_t)h);    /* d_b (SwiGLU) */
        double *dh = (double *)malloc(sizeof(double) * (size_t)h);    /* d_hid */
        double *dx = (double *)malloc(sizeof(double) * (size_t)m);    /* d_buf row */
        for (int64_t j = 0; j < cmax; j++) {
            const float *xr = buf + ((int64_t)ex * cmax + j) * m;
            const float *gr = d_out + ((int64_t)ex * cmax + j) * m;
            float *dbr = d_buf ? d_buf + ((int64_t)ex * cmax + j) * m : NULL;
            if (j >= rows) {
                if (dbr)
                    for (int i = 0; i < m; i++) dbr[i] = 0.0f;
                continue;
            }
            /* forward of this row: the derivative factors and the rounded hidden */
            for (int u = 0; u < h; u++) {
                const float *w1r = w1 + ((int64_t)ex * h + u) * m;
                double a = 0.0;
                for (int i = 0; i < m; i++) a += (double)xr[i] * (double)w1r[i];
                if (swiglu) {
                    const float *w3r = w3 + ((int64_t)ex * h + u) * m;
                    double b = 0.0;
                    for (int i = 0; i < m; i++) b += (double)xr[i] * (double)w3r[i];
                    const double sg = 1.0 / (1.0 + exp(-a));
                    hid[u] = round_to(a * sg * b, bf16);
                    dp[u] = b * sg * (1.0 + a * (1.0 - sg));   /* d hid / d a */
                    dq[u] = a * sg;                            /* d hid / d b */
                } else {
                    if (b1) a += (double)b1[(int64_t)ex * h + u];
                    if (act == ORC_ACT_RELU) {
                        hid[u] = round_to(a > 0.0 ? a : 0.0, bf16);
                        dp[u] = a > 0.0 ? 1.0 : 0.0;
                    } else {
                        const double cdf = 0.5 * (1.0 + erf(a / sqrt(2.0)));
                        /* standard normal density; 1/sqrt(2 pi) written out */
                        const double pdf = exp(-0.5 * a * a) * 0.39894228040143267794;
                        hid[u] = round_to(a * cdf, bf16);
                        dp[u] = cdf + a * pdf;
                    }
                    dq[u] = 0.0;
                }
            }
            /* fc2: d_hid[u] = sum over i ascending of d_out[i] w2[i, u] (the
             * rows of w2 are walked in order; each sum still adds its terms in
             * ascending i), then d_w2, d_b2 */
            for (int u = 0; u < h; u++) dh[u] = 0.0;
            for (int i = 0; i < m; i++) {
                const float *w2r = w2 + ((int64_t)ex * m + i) * h;
                for (int u = 0; u < h; u++) dh[u] += (double)gr[i] * (double)w2r[u];
            }
            for (int u = 0; u < h; u++) {
                dp[u] *= dh[u];
                dq[u] *= dh[u];
            }
            for (int i = 0; i < m; i++) {
                gb2[i] += (double)gr[i];
                for (int u = 0; u < h; u++) gw2[(int64_t)i * h + u] += (double)gr[i] * hid[u];
            }
            /* fc1: d_w1 (d_w3), d_b1, d_buf */
            for (int u = 0; u < h; u++) {
                gb1[u] += dp[u];
                for (int i = 0; i < m; i++) {
                    gw1[(int64_t)u * m + i] += dp[u] * (double)xr[i];
                    if (swiglu) gw3[(int64_t)u * m + i] += dq[u] * (double)xr[i];
                }
            }
            if (dbr) {
                /* d_buf[i] = sum over u ascending of d_pre[u] w1[u, i] (+ d_b[u]
                 * w3[u, i] after each w1 term), rows of w1 / w3 walked in order */
                for (int i = 0; i < m; i++) dx[i] = 0.0;
                for (int u = 0; u < h; u++) {
                    const float *w1r = w1 + ((int64_t)ex * h + u) * m;
                    const float *w3r = swiglu ? w3 + ((int64_t)ex * h + u) * m : NULL;
                    for (int i = 0; i < m; i++) {
                        dx[i] += dp[u] * (double)w1r[i];
                        if (swiglu) dx[i] += dq[u] * (double)w3r[i];
                    }
                }
                for (int i = 0; i < m; i++) dbr[i] = round_to(dx[i], bf16);
            }
        }
        for (int64_t q = 0; q < (int64_t)h * m; q++) {
            if (d_w1) d_w1[(int64_t)ex * h * m + q] = (float)gw1[q];
            if (d_w3 && swiglu) d_w3[(int64_t)ex * h * m + q] = (float)gw3[q];
            if (d_w2) d_w2[(int64_t)ex * m * h + q] = (float)gw2[q];
        }
        for (int u = 0; u < h; u++)
            if (d_b1 && !swiglu) d_b1[(int64_t)ex * h + u] = (float)gb1[u];
        for (int i = 0; i < m; i++)
            if (d_b2 && !swiglu) d_b2[(int64_t)ex * m + i] = (float)gb2[i];
        free(gw1); free(gw3); free(gw2); free(gb1); free(gb2); free(hid); free(dp); free(dq);
        free(dh); free(dx);
    }
}

/* ------------------------------------------------- FP8 (e4m3) experts */

/* Low-precision experts ([Tutel] profile, "notes" and "highlights": the
 * inference formats FP8 / blockwise FP8).  The pages name the formats but no
 * block size; this restatement scales every row of an operand by one fp32
 * factor (one per token row of the activations, one per output channel of the
 * weights), so that the factors apply once, after the contraction.
 *
 * e4m3 (the OCP FP8 E4M3 format): sign, 4 exponent bits with bias 7, 3
 * mantissa bits; exponent field 0 holds the subnormals m * 2^-9; no
 * infinities; exponent field 15 with mantissa 7 is NaN, so the largest finite
 * magnitude is 1.75 * 2^8 = 448.  Encoding rounds to nearest, ties to even,
 * and saturates finite values beyond 448 to +-448. */
float orc_fp8_decode(uint8_t c)
{
    int s = c >> 7, ef = (c >> 3) & 15, mf = c & 7;
    double v;
    if (ef == 15 && mf == 7) return NAN;
    if (ef == 0) v = ldexp((double)mf, -9);
    else v = ldexp(1.0 + mf / 8.0, ef - 7);
    return (float)(s ? -v : v);
}

uint8_t orc_fp8_encode(float x)
{
    if (isnan(x)) return 0x7F;
    uint8_t sgn = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0) return sgn | 0x7E;
    if (a < ldexp(1.0, -6)) {                       /* subnormal range: quantum 2^-9 */
        double r = nearbyint(ldexp(a, 9));          /* ties to even */
        return sgn | (uint8_t)r;                    /* r = 8 is the smallest normal */
    }
    int ex;
    frexp(a, &ex);                                  /* a in [2^(ex-1), 2^ex) */
    int E = ex - 1;                                 /* unbiased exponent, >= -6 */
    double r = nearbyint(ldexp(a, 3 - E));          /* in [8, 16], ties to even */
    if (r == 16.0) { E += 1; r = 8.0; }
    if (E > 8 || (E == 8 && r > 14.0)) return sgn | 0x7E;   /* past 448: saturate */
    return sgn | (uint8_t)(((E + 7) << 3) | ((int)r - 8));
}

/* Row quantisation: for each of `rows` rows of `cols` values, amax = max |x|,
 * scale = amax / 448 (fp32 division; 1 for an all-zero row), and every value
 * x / scale (fp32 division) encoded as e4m3. */
void orc_quantize_rows_fp8(const float *x, int64_t rows, int cols, uint8_t *q, float *scale)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++) {
        const float *xr = x + r * cols;
        float amax = 0.0f;
        for (int i = 0; i < cols; i++) {
            float v = fabsf(xr[i]);
            if (v > amax) amax = v;
        }
        float s = amax > 0.0f ? amax / 448.0f : 1.0f;
        scale[r] = s;
        for (int i = 0; i < cols; i++) q[r * cols + i] = orc_fp8_encode(xr[i] / s);
    }
}

/* One e4m3 product layer: out[r, n] = act(sa[r] * sw[n] * sum_k a[r, k] w[n, k]
 * + bias[n]) with a and w the decoded e4m3 codes, the sum in double, rounded
 * once to bf16.  act: -1 none, ORC_ACT_RELU, ORC_ACT_GELU (exact erf).  a
 * [rows, K], w [N, K], bias [N] or NULL, out [rows, N]. */
void orc_fc_fp8(const uint8_t *qa, const float *sa, const uint8_t *qw, const float *sw,
                const float *bias, int act, int64_t rows, int K, int N, float *out)
{
    float dec[256];
    for (int c = 0; c < 256; c++) dec[c] = orc_fp8_decode((uint8_t)c);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++) {
        for (int n = 0; n < N; n++) {
            double acc = 0.0;
            for (int k = 0; k < K; k++)
                acc += (double)dec[qa[r * K + k]] * (double)dec[qw[(int64_t)n * K + k]];
            double v = (double)sa[r] * (double)sw[n] * acc;
            if (bias) v += (double)bias[n];
            if (act == ORC_ACT_RELU) v = v > 0.0 ? v : 0.0;
            else if (act == ORC_ACT_GELU) v = 0.5 * v * (1.0 + erf(v / sqrt(2.0)));
            out[r * N + n] = round_bf16(v);
        }
    }
}
