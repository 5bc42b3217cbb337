/*
 * ORACLE -- test infrastructure, not part of the product.
 *
 * A plain, slow, single-threaded CPU statement of what the routed-expert
 * (MoE) layer computes: router logits, top-K gates, fixed-capacity slot
 * assignment, rowwise dispatch, bias-free SwiGLU experts, gate-weighted
 * combine, the backward of combine, experts, dispatch and router, and the
 * MXFP8 variant of dispatch, experts and combine.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may
 * load this library.  It shares no source with the CUDA path.
 *
 * Sources (page title, then section / figure / table):
 *   [EP]   OLMo-core MoE report, "Section 05: Expert Parallelism"
 *          -- 5.2 (local MoE: route, permute, grouped MLPs, combine), Figure 14
 *             (Linear 1 -> SwiGLU -> Linear 2 lanes), Figure 15 (router output,
 *             zero for a dropped route, weighted merge), 5.4 and Figure 16
 *             (route map: row = expert offset + earlier accepted routes,
 *             capacity decided before movement, negative = dropped),
 *             5.6 and Table 8 (PUT/GET adjoint movements), 5.7 (dense prefix,
 *             unwritten tail never consumed).
 *   [SYNC] OLMo-core MoE report, "Section 08: Synchronization-Free Training"
 *          -- 8.5 and Table 14 (counts and int32 cumulative offsets stay on the
 *             device; grouped GEMM stops at the valid rows; tail-aware SwiGLU).
 *   [DDP]  OLMo-core MoE report, "Section 04: Distributed Data Parallel"
 *          -- 4.1 (bias-free SwiGLU expert: 3*N*d*h parameters).
 *   [NRN]  AWS Neuron "Expert Parallelism (EP)" -- "Router Weights" (affinities
 *          for all experts from a replicated router weight).
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - logits: fp32, one fused multiply-add chain from 0 over j ascending (the
 *     plain left-to-right dot product), then + bias as a separate addition;
 *   - top-K: logit descending, lower expert index first on ties, NaN as -inf;
 *   - gates: softmax over the K selected logits (equal, in exact arithmetic, to
 *     a full softmax renormalised over the K selected); computed in fp64;
 *   - capacity: routes claim slots in token order; slot >= cap is dropped;
 *     experts packed back to back from row 0 at cumulative offsets;
 *   - expert FFN: separate W_gate, W_up [N,h,d] and W_down [N,d,h];
 *     silu(z) = z / (1 + exp(-z)); reductions in fp64; bf16 rounding (nearest
 *     even) only where a payload is stored (H, Y, saved G/U, dG/dU, dX);
 *   - combine / dispatch backward: fp32 accumulation over k ascending from 0;
 *     dropped routes add nothing and the kept gates are not renormalised;
 *   - MXFP8 variant ([EP] 5.4, 5.7, 5.8 name E4M3 data with E8M0 scales but
 *     not the format's rules): the OCP Microscaling (MX) v1.0 definition,
 *     blocks of 32 along each product's reduction dimension, shared exponent
 *     floor(log2 max|v|) - 8, elements rounded to nearest even and saturated
 *     at 448; G, U, H and Y in fp64 between the quantization points.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- bf16 --- */

static float bf16_to_f32(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* fp32 -> bf16, round to nearest, ties to even; NaN stays a quiet NaN. */
static uint16_t bf16_from_f32(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu))
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;
    return (uint16_t)((u + 0x7FFFu + lsb) >> 16);
}

/* fp64 -> bf16 with a single rounding (nearest, ties to even). */
static uint16_t bf16_from_f64(double v) {
    if (isnan(v)) return 0x7FC0u;
    if (v == 0.0 || isinf(v)) return bf16_from_f32((float)v);
    int e;
    frexp(v, &e);                 /* |v| = m * 2^e, 0.5 <= m < 1 */
    int q = e - 8;                /* quantum of an 8-significant-bit value */
    if (q < -133) q = -133;       /* bf16 subnormal spacing */
    double r = ldexp(nearbyint(ldexp(v, -q)), q);
    if (fabs(r) >= 0x1p128)       /* rounded past the largest finite bf16 */
        return (uint16_t)(r > 0 ? 0x7F80u : 0xFF80u);
    float f = (float)r;           /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

void oracle_bf16_from_f64(int64_t n, const double *v, uint16_t *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = bf16_from_f64(v[i]);
}

void oracle_bf16_from_f32(int64_t n, const float *v, uint16_t *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = bf16_from_f32(v[i]);
}

/* ------------------------------------------------------- R0: router logits ---
 * [NRN] "Router Weights": every token gets an affinity for every expert from
 * the replicated router weight, logit[t][e] = <x_t, W_r[e]> (+ bias[e]).
 * The pages fix no summation order.  Reading: the dot product as written,
 * summed left to right in fp32 -- one fused multiply-add chain that starts
 * at 0 and takes j = 0, 1, ..., d-1 in turn (x widened exactly from bf16) --
 * then + bias[e] as one fp32 addition.
 */
void oracle_router_logits(int T, int d, int N, const uint16_t *x, const float *w_r,
                          const float *bias, float *logits) {
    for (int t = 0; t < T; ++t)
        for (int e = 0; e < N; ++e) {
            float acc = 0.0f;
            for (int j = 0; j < d; ++j)
                acc = fmaf(bf16_to_f32(x[(int64_t)t * d + j]), w_r[(int64_t)e * d + j], acc);
            if (bias) acc = acc + bias[e];
            logits[(int64_t)t * N + e] = acc;
        }
}

/* ---------------------------------------------------- R1: top-K and gates ---
 * [EP] Figure 15, stage "Route": each token gets K expert indices and K router
 * weights; the weights of a token sum to one and are listed largest first.
 */
static float canon(float v) { return isnan(v) ? -INFINITY : v; }

static int beats(float a, int ia, float b, int ib) {
    return a > b || (a == b && ia < ib);
}

void oracle_topk_gates(int T, int N, int K, const float *logits, int32_t *idx, float *gate) {
    int *taken = (int *)calloc((size_t)N, sizeof(int));
    double *ex = (double *)malloc((size_t)K * sizeof(double));
    for (int t = 0; t < T; ++t) {
        const float *l = logits + (int64_t)t * N;
        memset(taken, 0, (size_t)N * sizeof(int));
        for (int k = 0; k < K; ++k) {
            int best = -1;
            for (int e = 0; e < N; ++e) {
                if (taken[e]) continue;
                if (best < 0 || beats(canon(l[e]), e, canon(l[best]), best)) best = e;
            }
            taken[best] = 1;
            idx[(int64_t)t * K + k] = best;
        }
        /* softmax over the K selected logits, shifted by the largest one; a
         * logit equal to the largest contributes exp(0) = 1 (this also fixes
         * the all -inf and +inf cases). */
        double m = (double)canon(l[idx[(int64_t)t * K]]);
        double s = 0.0;
        for (int k = 0; k < K; ++k) {
            double v = (double)canon(l[idx[(int64_t)t * K + k]]);
            ex[k] = (v == m) ? 1.0 : exp(v - m);
            s += ex[k];
        }
        for (int k = 0; k < K; ++k) gate[(int64_t)t * K + k] = (float)(ex[k] / s);
    }
    free(ex);
    free(taken);
}

/* ---------------------------------------------- R2/R3: slots and route map ---
 * [EP] 5.4, Figure 16: row = offset of the expert + number of earlier accepted
 * routes for that expert; the capacity decision is taken before any data
 * moves; a dropped route gets -1.  [EP] 5.7: experts packed back to back from
 * row 0.  [SYNC] Table 14: counts and int32 cumulative offsets.
 */
void oracle_route_slots(int T, int N, int K, int cap, const int32_t *idx, int32_t *route_row,
                        int32_t *count, int32_t *offset, int32_t *demand) {
    int32_t *seen = (int32_t *)calloc((size_t)N, sizeof(int32_t));
    for (int t = 0; t < T; ++t)
        for (int k = 0; k < K; ++k) {
            int e = idx[(int64_t)t * K + k];
            int s = seen[e]++;
            route_row[(int64_t)t * K + k] = (s < cap) ? s : -1;
        }
    for (int e = 0; e < N; ++e) {
        demand[e] = seen[e];
        count[e] = seen[e] < cap ? seen[e] : cap;
    }
    offset[0] = 0;
    for (int e = 0; e < N; ++e) offset[e + 1] = offset[e] + count[e];
    for (int t = 0; t < T; ++t)
        for (int k = 0; k < K; ++k) {
            int64_t i = (int64_t)t * K + k;
            if (route_row[i] >= 0) route_row[i] += offset[idx[i]];
        }
    free(seen);
}

/* --------------------------------------------------------------- D: dispatch ---
 * [EP] Table 8 "Dispatch forward PUT": x_t is copied to the capacity row of
 * each accepted route; negative rows are skipped (5.6).
 */
void oracle_dispatch(int T, int d, int K, const uint16_t *x, const int32_t *route_row,
                     uint16_t *x_disp) {
    for (int t = 0; t < T; ++t)
        for (int k = 0; k < K; ++k) {
            int32_t r = route_row[(int64_t)t * K + k];
            if (r < 0) continue;
            memcpy(x_disp + (int64_t)r * d, x + (int64_t)t * d, (size_t)d * sizeof(uint16_t));
        }
}

/* ----------------------------------------------- F: SwiGLU expert, fp64 core ---
 * [EP] Figure 14: Linear 1 -> SwiGLU -> Linear 2; [DDP] 4.1: bias-free, three
 * d x h matrices per expert.  For rows x (nrows x d):
 *   g = x W_gate^T, u = x W_up^T        (nrows x h)
 *   a = silu(g) * u, silu(z) = z / (1 + exp(-z))
 *   y = a W_down^T                       (nrows x d)
 * If round_a, a is rounded to bf16 before the second product (the stored H).
 */
static double silu(double z) { return z / (1.0 + exp(-z)); }

void oracle_ffn_fwd_f64(int nrows, int d, int h, const double *x, const double *wg,
                        const double *wu, const double *wd, int round_a, double *g, double *u,
                        double *a, double *y) {
    for (int r = 0; r < nrows; ++r) {
        const double *xr = x + (int64_t)r * d;
        for (int i = 0; i < h; ++i) {
            double sg = 0.0, su = 0.0;
            const double *wgi = wg + (int64_t)i * d, *wui = wu + (int64_t)i * d;
            for (int j = 0; j < d; ++j) {
                sg += xr[j] * wgi[j];
                su += xr[j] * wui[j];
            }
            double av = silu(sg) * su;
            if (round_a) av = (double)bf16_to_f32(bf16_from_f64(av));
            g[(int64_t)r * h + i] = sg;
            u[(int64_t)r * h + i] = su;
            a[(int64_t)r * h + i] = av;
        }
        for (int o = 0; o < d; ++o) {
            double s = 0.0;
            const double *wdo = wd + (int64_t)o * h;
            for (int i = 0; i < h; ++i) s += a[(int64_t)r * h + i] * wdo[i];
            y[(int64_t)r * d + o] = s;
        }
    }
}

/* Backward of the SwiGLU expert for rows x, given g, u (pre-activation), the
 * stored activation a, and dy (nrows x d).  Accumulates (+=) into dwg, dwu
 * (h x d) and dwd (d x h); writes dx (nrows x d).  If round_dgu, dg and du are
 * rounded to bf16 before they enter the two products that consume them (they
 * are then stored operands, i.e. bf16 payloads).
 *   da = dy W_down ;  dW_down += dy^T a
 *   du = da * silu(g) ;  dg = da * u * silu'(g),
 *   silu'(z) = s(z) (1 + z (1 - s(z))), s = logistic
 *   dx = dg W_gate + du W_up ;  dW_gate += dg^T x ;  dW_up += du^T x
 */
void oracle_ffn_bwd_f64(int nrows, int d, int h, const double *x, const double *g,
                        const double *u, const double *a, const double *dy, const double *wg,
                        const double *wu, const double *wd, int round_dgu, double *dx,
                        double *dwg, double *dwu, double *dwd) {
    double *dgv = (double *)malloc((size_t)h * sizeof(double));
    double *duv = (double *)malloc((size_t)h * sizeof(double));
    for (int r = 0; r < nrows; ++r) {
        const double *xr = x + (int64_t)r * d, *dyr = dy + (int64_t)r * d;
        for (int i = 0; i < h; ++i) {
            double da = 0.0;
            for (int o = 0; o < d; ++o) da += dyr[o] * wd[(int64_t)o * h + i];
            double z = g[(int64_t)r * h + i];
            double sg = 1.0 / (1.0 + exp(-z));
            duv[i] = da * z * sg;
            dgv[i] = da * u[(int64_t)r * h + i] * sg * (1.0 + z * (1.0 - sg));
            if (round_dgu) {
                duv[i] = (double)bf16_to_f32(bf16_from_f64(duv[i]));
                dgv[i] = (double)bf16_to_f32(bf16_from_f64(dgv[i]));
            }
        }
        for (int o = 0; o < d; ++o)
            for (int i = 0; i < h; ++i) dwd[(int64_t)o * h + i] += dyr[o] * a[(int64_t)r * h + i];
        for (int j = 0; j < d; ++j) {
            double s = 0.0;
            for (int i = 0; i < h; ++i)
                s += dgv[i] * wg[(int64_t)i * d + j] + duv[i] * wu[(int64_t)i * d + j];
            dx[(int64_t)r * d + j] = s;
        }
        for (int i = 0; i < h; ++i)
            for (int j = 0; j < d; ++j) {
                dwg[(int64_t)i * d + j] += dgv[i] * xr[j];
                dwu[(int64_t)i * d + j] += duv[i] * xr[j];
            }
    }
    free(dgv);
    free(duv);
}

/* ------------------------------------------- F: grouped expert FFN, bf16 I/O ---
 * [EP] 5.6/5.7 and [SYNC] 8.5: each expert runs over its valid row interval
 * [offset[e], offset[e] + count[e]) only; tail rows are never read or written.
 */
static double *widen_bf16(const uint16_t *src, int64_t n) {
    double *o = (double *)malloc((size_t)n * sizeof(double));
    for (int64_t i = 0; i < n; ++i) o[i] = (double)bf16_to_f32(src[i]);
    return o;
}

/* rows[i] (global row index) belongs to experts[i]; outputs are compact
 * (position i).  g_out/u_out may be NULL. */
void oracle_expert_ffn_rows(int d, int h, int nrows, const int32_t *rows, const int32_t *experts,
                            const uint16_t *x_disp, const uint16_t *wg, const uint16_t *wu,
                            const uint16_t *wd, uint16_t *h_out, uint16_t *g_out,
                            uint16_t *u_out, uint16_t *y_out) {
    double *g = (double *)malloc((size_t)h * sizeof(double));
    double *u = (double *)malloc((size_t)h * sizeof(double));
    double *a = (double *)malloc((size_t)h * sizeof(double));
    double *y = (double *)malloc((size_t)d * sizeof(double));
    int cur = -1;
    double *wge = NULL, *wue = NULL, *wde = NULL;
    for (int i = 0; i < nrows; ++i) {
        int e = experts[i];
        if (e != cur) {
            free(wge); free(wue); free(wde);
            wge = widen_bf16(wg + (int64_t)e * h * d, (int64_t)h * d);
            wue = widen_bf16(wu + (int64_t)e * h * d, (int64_t)h * d);
            wde = widen_bf16(wd + (int64_t)e * d * h, (int64_t)d * h);
            cur = e;
        }
        double *xr = widen_bf16(x_disp + (int64_t)rows[i] * d, d);
        oracle_ffn_fwd_f64(1, d, h, xr, wge, wue, wde, 1, g, u, a, y);
        free(xr);
        for (int c = 0; c < h; ++c) {
            h_out[(int64_t)i * h + c] = bf16_from_f64(a[c]);
            if (g_out) g_out[(int64_t)i * h + c] = bf16_from_f64(g[c]);
            if (u_out) u_out[(int64_t)i * h + c] = bf16_from_f64(u[c]);
        }
        for (int o = 0; o < d; ++o) y_out[(int64_t)i * d + o] = bf16_from_f64(y[o]);
    }
    free(wge); free(wue); free(wde);
    free(g); free(u); free(a); free(y);
}

/* Whole layer: writes the valid rows of h_act [R,h], g_save/u_save (may be
 * NULL) and y_disp [R,d]; rows past offset[N] are left untouched. */
void oracle_expert_ffn(int N, int d, int h, const int32_t *count, const int32_t *offset,
                       const uint16_t *x_disp, const uint16_t *wg, const uint16_t *wu,
                       const uint16_t *wd, uint16_t *h_act, uint16_t *g_save, uint16_t *u_save,
                       uint16_t *y_disp) {
    for (int e = 0; e < N; ++e) {
        int n = count[e];
        if (n <= 0) continue;
        int32_t *rows = (int32_t *)malloc((size_t)n * sizeof(int32_t));
        int32_t *ex = (int32_t *)malloc((size_t)n * sizeof(int32_t));
        for (int i = 0; i < n; ++i) { rows[i] = offset[e] + i; ex[i] = e; }
        int64_t r0 = offset[e];
        oracle_expert_ffn_rows(d, h, n, rows, ex, x_disp, wg, wu, wd, h_act + r0 * h,
                               g_save ? g_save + r0 * h : NULL, u_save ? u_save + r0 * h : NULL,
                               y_disp + r0 * d);
        free(rows);
        free(ex);
    }
}

/* ---------------------------------------------------------------- C: combine ---
 * [EP] Table 8 "Combine forward GET", 5.6, Figure 15: y_t is the router-weighted
 * sum of the selected expert rows; a dropped route contributes zero.  fp32
 * accumulation from 0 over k ascending; bf16 result.
 */
void oracle_combine(int T, int d, int K, const uint16_t *y_disp, const int32_t *route_row,
                    const float *gate, uint16_t *y) {
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < d; ++j) {
            float acc = 0.0f;
            for (int k = 0; k < K; ++k) {
                int32_t r = route_row[(int64_t)t * K + k];
                if (r < 0) continue;
                acc = fmaf(gate[(int64_t)t * K + k], bf16_to_f32(y_disp[(int64_t)r * d + j]), acc);
            }
            y[(int64_t)t * d + j] = bf16_from_f32(acc);
        }
}

/* ----------------------------------------------------- B1: combine backward ---
 * [EP] Table 8 "Combine backward PUT": the router-weighted output gradient is
 * pushed to each accepted route's row (fp32 product, bf16 payload).  5.6: the
 * router-weight gradient is <dy_t, gathered expert output> (fp64 sum, fp32
 * result; zero for a dropped route).
 */
void oracle_combine_bwd(int T, int d, int K, const uint16_t *dy, const uint16_t *y_disp,
                        const int32_t *route_row, const float *gate, uint16_t *dy_disp,
                        float *dgate) {
    for (int t = 0; t < T; ++t)
        for (int k = 0; k < K; ++k) {
            int64_t i = (int64_t)t * K + k;
            int32_t r = route_row[i];
            if (r < 0) { dgate[i] = 0.0f; continue; }
            double s = 0.0;
            for (int j = 0; j < d; ++j) {
                float v = bf16_to_f32(dy[(int64_t)t * d + j]);
                dy_disp[(int64_t)r * d + j] = bf16_from_f32(gate[i] * v);
                s += (double)v * (double)bf16_to_f32(y_disp[(int64_t)r * d + j]);
            }
            dgate[i] = (float)s;
        }
}

/* ---------------------------------------------------- B3: dispatch backward ---
 * [EP] Table 8 "Dispatch backward GET": the route gradients of a token are
 * pulled and summed into the gradient of its row (fp32, k ascending from 0).
 */
void oracle_dispatch_bwd(int T, int d, int K, const uint16_t *dx_disp, const int32_t *route_row,
                         float *dx) {
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < d; ++j) {
            float acc = 0.0f;
            for (int k = 0; k < K; ++k) {
                int32_t r = route_row[(int64_t)t * K + k];
                if (r < 0) continue;
                acc = acc + bf16_to_f32(dx_disp[(int64_t)r * d + j]);
            }
            dx[(int64_t)t * d + j] = acc;
        }
}

/* ------------------------------------------- B2: grouped expert backward ---
 * [EP] 5.7: expert backward and Wgrad run over the valid rows only.  Uses the
 * stored bf16 G, U and H of the forward; dG and dU are bf16 payloads between
 * the two backward products.  dx_disp is a bf16 payload; the weight
 * gradients are fp32 [N,h,d], [N,h,d], [N,d,h] (fully written; experts with no
 * rows get zero).
 */
void oracle_expert_ffn_bwd(int N, int d, int h, const int32_t *count, const int32_t *offset,
                           const uint16_t *x_disp, const uint16_t *g_save, const uint16_t *u_save,
                           const uint16_t *h_act, const uint16_t *dy_disp, const uint16_t *wg,
                           const uint16_t *wu, const uint16_t *wd, uint16_t *dx_disp,
                           float *dwg, float *dwu, float *dwd) {
    int64_t hd = (int64_t)h * d;
    double *dwg64 = (double *)malloc((size_t)hd * sizeof(double));
    double *dwu64 = (double *)malloc((size_t)hd * sizeof(double));
    double *dwd64 = (double *)malloc((size_t)hd * sizeof(double));
    for (int e = 0; e < N; ++e) {
        memset(dwg64, 0, (size_t)hd * sizeof(double));
        memset(dwu64, 0, (size_t)hd * sizeof(double));
        memset(dwd64, 0, (size_t)hd * sizeof(double));
        int n = count[e];
        if (n > 0) {
            int64_t r0 = offset[e];
            double *x = widen_bf16(x_disp + r0 * d, (int64_t)n * d);
            double *g = widen_bf16(g_save + r0 * h, (int64_t)n * h);
            double *u = widen_bf16(u_save + r0 * h, (int64_t)n * h);
            double *a = widen_bf16(h_act + r0 * h, (int64_t)n * h);
            double *dy = widen_bf16(dy_disp + r0 * d, (int64_t)n * d);
            double *wge = widen_bf16(wg + (int64_t)e * hd, hd);
            double *wue = widen_bf16(wu + (int64_t)e * hd, hd);
            double *wde = widen_bf16(wd + (int64_t)e * hd, hd);
            double *dx = (double *)malloc((size_t)n * d * sizeof(double));
            oracle_ffn_bwd_f64(n, d, h, x, g, u, a, dy, wge, wue, wde, 1, dx, dwg64, dwu64, dwd64);
            for (int64_t i = 0; i < (int64_t)n * d; ++i) dx_disp[r0 * d + i] = bf16_from_f64(dx[i]);
            free(x); free(g); free(u); free(a); free(dy); free(wge); free(wue); free(wde); free(dx);
        }
        for (int64_t i = 0; i < hd; ++i) {
            dwg[(int64_t)e * hd + i] = (float)dwg64[i];
            dwu[(int64_t)e * hd + i] = (float)dwu64[i];
            dwd[(int64_t)e * hd + i] = (float)dwd64[i];
        }
    }
    free(dwg64); free(dwu64); free(dwd64);
}

/* ---------------------------------------------------- router backward ---
 * Gradient of the router for one step whose top-K selection is fixed
 * ([EP] 5.6: the router-weight gradient comes from the gathered expert outputs
 * through dgate; Figure 15: the gates are a softmax over the K chosen logits).
 * With g the gates and dg = dL/dg (dgate, 0 for a dropped route):
 *   dlogit_k = g_k * (dg_k - sum_k' g_k' dg_k')      (chosen experts; others 0)
 *   dx[t]    = sum_k dlogit_k W_r[idx_k]              (added to dx)
 *   dW_r[e]  = sum over routes (t, k) with idx = e of dlogit_k x_t
 *   dbias[e] = sum over the same routes of dlogit_k    (dbias may be NULL)
 * fp64 sums, fp32 results.
 */
void oracle_router_bwd(int T, int d, int N, int K, const uint16_t *x, const float *w_r,
                       const int32_t *idx, const float *gate, const float *dgate, float *dlogit,
                       float *dx, float *dw, float *dbias) {
    double *acc = (double *)calloc((size_t)N * d, sizeof(double));
    double *accb = (double *)calloc((size_t)N, sizeof(double));
    double *dl = (double *)malloc((size_t)K * sizeof(double));
    double *row = (double *)malloc((size_t)d * sizeof(double));
    for (int t = 0; t < T; ++t) {
        double dot = 0.0;
        for (int k = 0; k < K; ++k)
            dot += (double)gate[(int64_t)t * K + k] * (double)dgate[(int64_t)t * K + k];
        for (int k = 0; k < K; ++k) {
            dl[k] = (double)gate[(int64_t)t * K + k] * ((double)dgate[(int64_t)t * K + k] - dot);
            dlogit[(int64_t)t * K + k] = (float)dl[k];
        }
        for (int j = 0; j < d; ++j) {
            double sx = 0.0;
            for (int k = 0; k < K; ++k)
                sx += dl[k] * (double)w_r[(int64_t)idx[(int64_t)t * K + k] * d + j];
            row[j] = sx;
        }
        for (int j = 0; j < d; ++j)
            dx[(int64_t)t * d + j] = (float)((double)dx[(int64_t)t * d + j] + row[j]);
        for (int k = 0; k < K; ++k) {
            int e = idx[(int64_t)t * K + k];
            accb[e] += dl[k];
            for (int j = 0; j < d; ++j)
                acc[(int64_t)e * d + j] += dl[k] * (double)bf16_to_f32(x[(int64_t)t * d + j]);
        }
    }
    for (int64_t i = 0; i < (int64_t)N * d; ++i) dw[i] = (float)acc[i];
    if (dbias)
        for (int e = 0; e < N; ++e) dbias[e] = (float)accb[e];
    free(acc);
    free(accb);
    free(dl);
    free(row);
}

/* ================================================================ MXFP8 ===
 * [EP] 5.4 (rows are quantized as they are dispatched; the grouped GEMM reads
 * the quantized data and its scales as they arrived; the experts' outputs go
 * back quantized and are dequantized by the local reduction), 5.7 (a quantized
 * route carries a data row and a scale row at the same destination row and
 * with the same validity as the bf16 row), 5.8 (data in E4M3, scales in E8M0,
 * both expert GEMMs in MXFP8).
 * The pages name the format but not its rules.  Reading: MXFP8 as the OCP
 * Microscaling (MX) v1.0 specification defines it -- blocks of 32 consecutive
 * elements along a row share one power-of-two scale X = 2^E, stored as the
 * E8M0 byte E + 127, with E = floor(log2(max |v|)) - 8 (8 is the exponent of
 * the largest E4M3 normal, 448 = 1.75 * 2^8) clamped to [-127, 127]; each
 * element is stored as v / X rounded to the nearest E4M3 value, ties to the
 * even code, magnitudes past 448 saturating to 448.  An all-zero block gets
 * E = -127 (byte 0).  Inputs are finite.
 */

/* E4M3 code -> value: sign bit 7, exponent bits 6-3 (bias 7), mantissa bits
 * 2-0; exponent field 0 holds the subnormals m * 2^-9; S.1111.111 is NaN and
 * there are no infinities. */
static double e4m3_value(uint8_t c) {
    int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    double v = e == 0 ? ldexp((double)m, -9) : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* value -> the nearest finite E4M3 code by exhaustive search over the 127
 * non-negative finite codes (ties: the code whose mantissa LSB is 0); the sign
 * is copied, so values that round to zero keep it. */
static uint8_t e4m3_nearest(double v) {
    static double table[127];
    static int ready = 0;
    if (!ready) {
        for (int c = 0; c < 127; ++c) table[c] = e4m3_value((uint8_t)c);
        ready = 1;
    }
    double a = fabs(v), best_d = INFINITY;
    int best = 0;
    for (int c = 0; c < 127; ++c) {
        double dist = fabs(table[c] - a);
        if (dist < best_d || (dist == best_d && (c & 1) == 0)) {
            best_d = dist;
            best = c;
        }
    }
    return (uint8_t)(best | (signbit(v) ? 0x80 : 0));
}

/* Shared exponent E of one block (see the reading above). */
static int mx_block_exponent(const double *v, int n) {
    double amax = 0.0;
    for (int i = 0; i < n; ++i) amax = fmax(amax, fabs(v[i]));
    if (amax == 0.0) return -127;
    int e;
    frexp(amax, &e); /* amax = m * 2^e, 0.5 <= m < 1, so floor(log2 amax) = e - 1 */
    int E = (e - 1) - 8;
    return E < -127 ? -127 : (E > 127 ? 127 : E);
}

#define MX_BLOCK 32

/* rows x k values (k a multiple of 32) -> codes q [rows, k] and E8M0 scale
 * bytes [rows, k / 32], row-major. */
void oracle_mx_quantize_f64(int64_t rows, int k, const double *v, uint8_t *q, uint8_t *scale) {
    const int nb = k / MX_BLOCK;
    for (int64_t r = 0; r < rows; ++r)
        for (int b = 0; b < nb; ++b) {
            const double *blk = v + r * k + (int64_t)b * MX_BLOCK;
            int E = mx_block_exponent(blk, MX_BLOCK);
            scale[r * nb + b] = (uint8_t)(E + 127);
            for (int i = 0; i < MX_BLOCK; ++i)
                q[r * k + (int64_t)b * MX_BLOCK + i] = e4m3_nearest(ldexp(blk[i], -E));
        }
}

void oracle_mx_quantize_bf16(int64_t rows, int k, const uint16_t *x, uint8_t *q, uint8_t *scale) {
    double *v = (double *)malloc((size_t)k * sizeof(double));
    for (int64_t r = 0; r < rows; ++r) {
        for (int i = 0; i < k; ++i) v[i] = (double)bf16_to_f32(x[r * k + i]);
        oracle_mx_quantize_f64(1, k, v, q + r * k, scale + r * (k / MX_BLOCK));
    }
    free(v);
}

/* codes and scale bytes -> values: e4m3(q) * 2^(scale - 127); a scale byte of
 * 255 (NaN) gives NaN. */
void oracle_mx_dequantize(int64_t rows, int k, const uint8_t *q, const uint8_t *scale,
                          double *out) {
    const int nb = k / MX_BLOCK;
    for (int64_t r = 0; r < rows; ++r)
        for (int i = 0; i < k; ++i) {
            uint8_t s = scale[r * nb + i / MX_BLOCK];
            out[r * k + i] = s == 255 ? NAN : ldexp(e4m3_value(q[r * k + i]), (int)s - 127);
        }
}

/* Grouped SwiGLU experts in MXFP8 over each expert's valid rows ([EP] 5.4,
 * 5.8; [SYNC] 8.5).  Inputs: dispatched rows xq [R, d] with scales xs [R, d/32];
 * weights wgq, wuq [N, h, d] with scales [N, h, d/32] and wdq [N, d, h] with
 * scales [N, d, h/32] (blocks run along each product's reduction dimension).
 * Per valid row, in fp64 on the dequantized values:
 *   g = x Wg^T, u = x Wu^T, a = silu(g) * u, (hq, hs) = MX(a) along h,
 *   y = deq(hq, hs) Wd^T, (yq, ys) = MX(y) along d.
 * Rows outside every expert's interval are left untouched. */
void oracle_expert_ffn_mx(int N, int d, int h, const int32_t *count, const int32_t *offset,
                          const uint8_t *xq, const uint8_t *xs, const uint8_t *wgq,
                          const uint8_t *wgs, const uint8_t *wuq, const uint8_t *wus,
                          const uint8_t *wdq, const uint8_t *wds, uint8_t *hq, uint8_t *hs,
                          uint8_t *yq, uint8_t *ys) {
    const int64_t hd = (int64_t)h * d;
    double *wg = (double *)malloc((size_t)hd * sizeof(double));
    double *wu = (double *)malloc((size_t)hd * sizeof(double));
    double *wd = (double *)malloc((size_t)hd * sizeof(double));
    double *x = (double *)malloc((size_t)d * sizeof(double));
    double *a = (double *)malloc((size_t)h * sizeof(double));
    double *ad = (double *)malloc((size_t)h * sizeof(double));
    double *y = (double *)malloc((size_t)d * sizeof(double));
    for (int e = 0; e < N; ++e) {
        if (count[e] <= 0) continue;
        oracle_mx_dequantize(h, d, wgq + e * hd, wgs + e * hd / MX_BLOCK, wg);
        oracle_mx_dequantize(h, d, wuq + e * hd, wus + e * hd / MX_BLOCK, wu);
        oracle_mx_dequantize(d, h, wdq + e * hd, wds + e * hd / MX_BLOCK, wd);
        for (int i = 0; i < count[e]; ++i) {
            const int64_t r = (int64_t)offset[e] + i;
            oracle_mx_dequantize(1, d, xq + r * d, xs + r * (d / MX_BLOCK), x);
            for (int c = 0; c < h; ++c) {
                double g = 0.0, u = 0.0;
                for (int j = 0; j < d; ++j) {
                    g += x[j] * wg[(int64_t)c * d + j];
                    u += x[j] * wu[(int64_t)c * d + j];
                }
                a[c] = silu(g) * u;
            }
            oracle_mx_quantize_f64(1, h, a, hq + r * h, hs + r * (h / MX_BLOCK));
            oracle_mx_dequantize(1, h, hq + r * h, hs + r * (h / MX_BLOCK), ad);
            for (int o = 0; o < d; ++o) {
                double s = 0.0;
                for (int c = 0; c < h; ++c) s += ad[c] * wd[(int64_t)o * h + c];
                y[o] = s;
            }
            oracle_mx_quantize_f64(1, d, y, yq + r * d, ys + r * (d / MX_BLOCK));
        }
    }
    free(wg); free(wu); free(wd); free(x); free(a); free(ad); free(y);
}

/* Combine of quantized expert outputs ([EP] 5.4: the reduction dequantizes):
 * y[t] = bf16( sum over k ascending (route_row >= 0) of gate[t, k] *
 * deq(yq, ys)[route_row[t, k]] ), fp32 fused multiply-add chain from 0; the
 * dequantized values are exact in fp32. */
void oracle_combine_mx(int T, int d, int K, const uint8_t *yq, const uint8_t *ys,
                       const int32_t *route_row, const float *gate, uint16_t *y) {
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < d; ++j) {
            float acc = 0.0f;
            for (int k = 0; k < K; ++k) {
                int32_t r = route_row[(int64_t)t * K + k];
                if (r < 0) continue;
                uint8_t s = ys[(int64_t)r * (d / MX_BLOCK) + j / MX_BLOCK];
                float v = (float)ldexp(e4m3_value(yq[(int64_t)r * d + j]), (int)s - 127);
                acc = fmaf(gate[(int64_t)t * K + k], v, acc);
            }
            y[(int64_t)t * d + j] = bf16_from_f32(acc);
        }
}
