/*
 * moe.h -- C ABI of the routed-expert (MoE) layer hot path on one GPU.
 *
 * Path: route (router logits, top-K gates, fixed-capacity slots) -> rowwise
 * dispatch into packed per-expert buffers -> grouped bias-free SwiGLU expert
 * GEMMs over the valid rows -> gate-weighted combine back to token order; plus
 * the backward of combine, experts and dispatch.
 *
 * Sources (page title, then section / figure / table):
 *   OLMo-core MoE report, "Section 05: Expert Parallelism": 5.2 and Figure 14
 *   (route, expert-contiguous layout, Linear 1 -> SwiGLU -> Linear 2, combine),
 *   Figures 15 and 16 (router output, route map, dropped route), 5.4, 5.6 and
 *   Table 8 (dispatch PUT, combine GET and their adjoint backward), 5.7 (dense
 *   prefix per buffer, unwritten tail never consumed).
 *   OLMo-core MoE report, "Section 08: Synchronization-Free Training": 8.5 and
 *   Table 14 (route maps, counts and int32 cumulative offsets stay on the
 *   device; capacity-shaped buffers; grouped GEMM with device offsets).
 *   OLMo-core MoE report, "Section 04: Distributed Data Parallel": 4.1
 *   (bias-free SwiGLU expert).
 *   AWS Neuron "Expert Parallelism (EP)": "Router Weights" (affinities for all
 *   experts from one router weight).
 *
 * Conventions shared by every call
 *   - All pointers are DEVICE pointers unless stated otherwise, owned by the
 *     caller; the library never allocates or frees device memory.
 *   - Every call is asynchronous on `stream` and never synchronises the host
 *     or reads device data back; route-dependent values (counts, offsets,
 *     rows) are produced and consumed on the device only.
 *   - bf16 tensors are 16-bit bfloat16 bit patterns (moe_bf16); every pointer
 *     must be 16-byte aligned and d, h must be multiples of 8.
 *   - Row-major layouts.  T tokens, d model width, N experts, K routes per
 *     token, h expert hidden width, cap rows per expert, R = min(N * cap, T * K)
 *     rows in every capacity buffer (moe_buffer_rows; the packed rows never
 *     exceed either bound, so a dropless caller with cap = T needs T * K rows,
 *     not N * T).  Larger buffers are accepted; the extra rows are tail.
 *   - Capacity buffers hold the experts' rows packed back to back from row 0:
 *     expert e owns rows [expert_offset[e], expert_offset[e] + expert_count[e]).
 *     Rows from expert_offset[N] to R - 1 (the tail) are neither read nor
 *     written by any call and may hold anything, including NaN.
 *   - Host-side argument errors are returned before anything is enqueued.
 *     Errors seen on the device (a wait that timed out; in the *_checked
 *     calls, a route row outside the buffers) are recorded in the
 *     workspace's status word; moe_read_device_error() reads it.
 *   - Results are deterministic: no floating-point atomics anywhere.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *cudaStream_t;
typedef uint16_t moe_bf16;

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* bad shape, null pointer, K > N, ... */
    MOE_ERR_ALIGNMENT = 2,    /* pointer not 16-byte aligned or d, h not multiples of 8 */
    MOE_ERR_WORKSPACE = 3,    /* workspace missing or smaller than the *_workspace_bytes query */
    MOE_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed */
    MOE_ERR_UNSUPPORTED = 5,  /* shape outside what the kernels handle (see each call) */
    MOE_ERR_DEVICE_TIMEOUT = 6, /* device status word: a bounded wait inside a kernel expired */
    MOE_ERR_DEVICE_ROUTE_RANGE = 7 /* device status word: a *_checked call met a route row
                                      >= R and skipped that route */
} moe_status;

/* Layer shape.  cap is chosen by the caller before its loop, e.g.
 * cap = ceil(cf * T * K / N) for a capacity factor cf. */
typedef struct {
    int32_t T, d, N, K, h, cap;
} moe_shape;

/* Limits: 1 <= K <= 16, K <= N <= 1024, 0 <= cap, T >= 0, T * K < 2^31,
 * 8 <= d, h with d, h multiples of 8. */

/* Rows R of every capacity buffer (x_disp, h_act, g_save, u_save, y_disp,
 * dy_disp, dx_disp) for this shape: min(N * cap, T * K); -1 if the shape is
 * invalid.  The packed layout (Section 05, 5.7: experts back to back in a
 * dense prefix; Section 08, 8.5 and Table 14: int32 cumulative offsets on the
 * device) never places a row at or past it. */
int64_t moe_buffer_rows(const moe_shape *s);

/* Human-readable name of a status code (static string). */
const char *moe_status_string(moe_status s);

/* Bytes of workspace moe_route needs for this shape (0 if the shape is invalid). */
size_t moe_route_workspace_bytes(const moe_shape *s);

/* Byte offset, inside the moe_route workspace, of the router logits [T, N]
 * fp32 (row-major, bias included) that moe_route leaves there; a multiple of
 * 256.  0 if the shape is invalid (the logits never start at 0: word 0 is the
 * status word). */
size_t moe_route_logits_offset(const moe_shape *s);

/*
 * moe_route -- steps R0-R3: router logits, top-K, gates, slots, route map.
 * Report: Neuron "Router Weights" (logits over all N experts); Section 05
 * Figure 15 (K indices and K weights per token, larger weight first, summing
 * to one); 5.4 and Figure 16 (row = offset of the expert + number of earlier
 * accepted routes to it; capacity decided before any row moves; negative =
 * dropped); Section 08 Table 14 (counts and cumulative offsets on the device).
 *
 *   x            [T, d] bf16 token rows.
 *   w_router     [N, d] fp32 router weight.
 *   bias         [N] fp32 per-expert logit offset, or NULL.
 *   topk_idx     out [T, K] int32: experts by logit descending, ties to the
 *                lower index; NaN logits rank as -inf.
 *   topk_gate    out [T, K] fp32: softmax over the K chosen logits.
 *   route_row    out [T, K] int32: capacity-buffer row of each route, -1 if
 *                the route was dropped.  Routes claim slots in token order.
 *   expert_count out [N] int32: accepted routes per expert (<= cap).
 *   expert_offset out [N + 1] int32: exclusive prefix sum of expert_count;
 *                expert_offset[N] = accepted routes A.
 *   expert_demand out [N] int32: routes that chose each expert (before the
 *                capacity decision); dropped = sum(demand - count).
 *   ws, ws_bytes device workspace of at least moe_route_workspace_bytes(s)
 *                bytes, 256-byte aligned; word 0 is the device status word.
 * Logits are fp32: one fused multiply-add chain per (token, expert) from 0
 * over j = 0 .. d-1 in order (the dot product summed left to right), then
 * + bias[e] as one fp32 addition.  The pages fix no order; this one is the
 * plain reading, and it makes the logits, and with them every top-K
 * decision, reproducible bit for bit.  The call leaves the logits [T, N] fp32
 * in the workspace at byte moe_route_logits_offset(s), where they stay until
 * the workspace is used again.
 */
moe_status moe_route(const moe_shape *s, const moe_bf16 *x, const float *w_router,
                     const float *bias, int32_t *topk_idx, float *topk_gate, int32_t *route_row,
                     int32_t *expert_count, int32_t *expert_offset, int32_t *expert_demand,
                     void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * moe_route_noalloc -- moe_route without a workspace argument, for callers
 * that cannot allocate device memory: for example a plugin that a host
 * framework hands only its input and output buffers (the framework owns the
 * allocator), or a latency-critical loop in which cudaMalloc is not allowed
 * because it can synchronise the device.  The report has no counterpart of
 * this entry point.
 *
 * Same arguments, outputs and results as moe_route.  The scratch that
 * moe_route keeps in `ws` lives instead in a fixed device array of
 * MOE_ROUTE_NOALLOC_SCRATCH_BYTES (64 MiB) inside this library; every GPU that
 * loads the library holds that array until the process exits.  The call
 * allocates nothing.  Shapes whose scratch (moe_route_workspace_bytes: the
 * 256-byte status word, the per-block counts, 4 * ceil(T / 256) * N bytes,
 * the logits, 4 * T * N bytes, and the router weight regrouped by experts,
 * 4 * d * N bytes rounded up to whole groups of 32 or 64 experts) would
 * exceed the array -- roughly T * N + d * N > 16.7 million -- are rejected
 * with MOE_ERR_UNSUPPORTED before anything is enqueued.
 *
 * The first call on a device looks up the array's device address there
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before any stream capture.  All calls on one device share the array, which
 * keeps the previous call's contents; nothing in it needs clearing.  Calls
 * that overlap on the GPU (e.g. on two streams at once) race on the array.
 * Routing records no device-side error (its kernels have no waits and no
 * data-dependent addresses outside the checked shape), in moe_route or here,
 * so there is no status to read back.
 */
#define MOE_ROUTE_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
moe_status moe_route_noalloc(const moe_shape *s, const moe_bf16 *x, const float *w_router,
                             const float *bias, int32_t *topk_idx, float *topk_gate,
                             int32_t *route_row, int32_t *expert_count, int32_t *expert_offset,
                             int32_t *expert_demand, cudaStream_t stream);

/*
 * moe_dispatch -- step D.  Section 05 Table 8 "Dispatch forward PUT" and 5.6:
 * x_disp[route_row[t, k]] = x[t] for every route with route_row >= 0; each
 * token row is read once and written to each of its accepted rows (Figure 19,
 * source-initiated fan-out).  Rows not named by route_row are untouched.
 *   x [T, d] bf16;  route_row [T, K];  x_disp out [R, d] bf16 (may be NULL when
 *   cap = 0: every route is then dropped and nothing is written).
 */
moe_status moe_dispatch(const moe_shape *s, const moe_bf16 *x, const int32_t *route_row,
                        moe_bf16 *x_disp, cudaStream_t stream);

/* Bytes of workspace moe_expert_ffn / moe_expert_ffn_backward need. */
size_t moe_expert_ffn_workspace_bytes(const moe_shape *s);

/*
 * moe_expert_ffn -- steps F1, F2: grouped bias-free SwiGLU experts.
 * Section 05 Figure 14 (Linear 1 -> SwiGLU -> Linear 2), 5.7 and Section 08
 * 8.5 (per-expert row intervals from device offsets; the activation is applied
 * to the valid prefix only; tails are skipped).  For each expert e and each
 * row r of its interval:
 *   G = x_disp[r] W_gate[e]^T,  U = x_disp[r] W_up[e]^T   (fp32 accumulation)
 *   h_act[r] = bf16(silu(G) * U),   silu(z) = z / (1 + exp(-z))
 *   y_disp[r] = bf16(h_act[r] W_down[e]^T)                (fp32 accumulation)
 *   x_disp [R, d] bf16; expert_count [N]; expert_offset [N + 1] (from moe_route);
 *   w_gate, w_up [N, h, d] bf16; w_down [N, d, h] bf16;
 *   h_act out [R, h] bf16; g_save, u_save out [R, h] bf16 (bf16(G), bf16(U),
 *   kept for the backward) or both NULL; y_disp out [R, d] bf16;
 *   ws, ws_bytes: workspace of moe_expert_ffn_workspace_bytes(s) bytes.
 * Runs on tcgen05 tensor cores; d and h must be multiples of 64
 * (MOE_ERR_UNSUPPORTED otherwise).
 */
moe_status moe_expert_ffn(const moe_shape *s, const moe_bf16 *x_disp, const int32_t *expert_count,
                          const int32_t *expert_offset, const moe_bf16 *w_gate,
                          const moe_bf16 *w_up, const moe_bf16 *w_down, moe_bf16 *h_act,
                          moe_bf16 *g_save, moe_bf16 *u_save, moe_bf16 *y_disp, void *ws,
                          size_t ws_bytes, cudaStream_t stream);

/* Bytes of workspace moe_expert_ffn_gather needs: the device status word plus
 * one int32 per capacity-buffer row (0 if the shape is invalid). */
size_t moe_expert_ffn_gather_workspace_bytes(const moe_shape *s);

/*
 * moe_expert_ffn_gather -- steps D and F1-F2 fused: the same results as
 * moe_dispatch followed by moe_expert_ffn (h_act, g_save, u_save and y_disp
 * bit for bit), without writing or reading x_disp.  Section 05 Table 8
 * "Dispatch forward PUT" and 5.6 (each accepted route's row is the token's
 * row); Section 08, 8.5 (grouped GEMM over device offsets).  GEMM1 fetches
 * each packed row straight from x: a small kernel inverts the route map
 * (row -> token, into ws) and the GEMM's producer loads four token rows at a
 * time by TMA gather.  For a forward without backward: the expert backward
 * reads x_disp, which this call does not produce.
 *   x [T, d] bf16; route_row [T, K] as moe_route wrote it; the rest as in
 *   moe_expert_ffn; ws of moe_expert_ffn_gather_workspace_bytes bytes,
 *   256-byte aligned.
 * Errors: as moe_expert_ffn.
 */
moe_status moe_expert_ffn_gather(const moe_shape *s, const moe_bf16 *x, const int32_t *route_row,
                                 const int32_t *expert_count, const int32_t *expert_offset,
                                 const moe_bf16 *w_gate, const moe_bf16 *w_up,
                                 const moe_bf16 *w_down, moe_bf16 *h_act, moe_bf16 *g_save,
                                 moe_bf16 *u_save, moe_bf16 *y_disp, void *ws, size_t ws_bytes,
                                 cudaStream_t stream);

/* Bytes of workspace moe_expert_ffn_backward needs: the device status word,
 * the two [R, h] bf16 intermediates dG and dU, and 1 MiB of tensor-map copies
 * (the weight-gradient kernels bound each tile's last k-block to its expert's
 * rows through per-CTA copies of their maps). */
size_t moe_expert_ffn_backward_workspace_bytes(const moe_shape *s);

/*
 * moe_expert_ffn_backward -- step B2: data and weight gradients of the
 * grouped SwiGLU experts.  Section 05, 5.7 (expert backward and the weight-
 * gradient GEMM run over each expert's valid rows, given the real offsets,
 * and skip the unwritten tail); Figure 14 (Linear 1 -> SwiGLU -> Linear 2).
 * For each expert e over its rows, with X = x_disp, G = g_save, U = u_save,
 * H = h_act and dY = dy_disp (the combine backward's output):
 *   dH = dY W_down[e];  dU = dH * silu(G);  dG = dH * U * silu'(G)
 *   dx_disp = bf16(dG W_gate[e] + dU W_up[e])
 *   dw_down[e] = dY^T H;  dw_gate[e] = dG^T X;  dw_up[e] = dU^T X   (fp32)
 * with fp32 accumulation on tcgen05 tensor cores; dG and dU are rounded to
 * bf16 (they are operands of the next products) and kept in the workspace.
 *   x_disp, dy_disp [R, d] bf16; g_save, u_save, h_act [R, h] bf16 (from
 *   moe_expert_ffn with saving on); counts and offsets from moe_route;
 *   weights as in moe_expert_ffn; dx_disp out [R, d] bf16 (valid rows only);
 *   dw_gate, dw_up out [N, h, d] fp32; dw_down out [N, d, h] fp32 (every
 *   element written: experts without rows get zeros);
 *   ws, ws_bytes: moe_expert_ffn_backward_workspace_bytes(s) bytes, 256-byte
 *   aligned.  d and h must be multiples of 64 (MOE_ERR_UNSUPPORTED otherwise).
 */
moe_status moe_expert_ffn_backward(const moe_shape *s, const moe_bf16 *x_disp,
                                   const int32_t *expert_count, const int32_t *expert_offset,
                                   const moe_bf16 *w_gate, const moe_bf16 *w_up,
                                   const moe_bf16 *w_down, const moe_bf16 *g_save,
                                   const moe_bf16 *u_save, const moe_bf16 *h_act,
                                   const moe_bf16 *dy_disp, moe_bf16 *dx_disp, float *dw_gate,
                                   float *dw_up, float *dw_down, void *ws, size_t ws_bytes,
                                   cudaStream_t stream);

/*
 * moe_combine -- step C.  Section 05 Table 8 "Combine forward GET", 5.6 and
 * Figure 15: y[t] = bf16( sum over k ascending of topk_gate[t, k] *
 * y_disp[route_row[t, k]] ), fp32 fused multiply-add accumulation from 0;
 * dropped routes contribute zero and the kept gates are not renormalised.
 *   y_disp [R, d] bf16; route_row, topk_gate [T, K]; y out [T, d] bf16.
 */
moe_status moe_combine(const moe_shape *s, const moe_bf16 *y_disp, const int32_t *route_row,
                       const float *topk_gate, moe_bf16 *y, cudaStream_t stream);

/*
 * moe_combine_backward -- step B1.  Section 05 Table 8 "Combine backward PUT"
 * and 5.6 (router-weight gradient from the gathered expert outputs):
 *   dy_disp[route_row[t, k]] = bf16(topk_gate[t, k] * dy[t])   (fp32 product)
 *   dgate[t, k] = <dy[t], y_disp[route_row[t, k]]>   (fp32; 0 if dropped)
 *   dy [T, d] bf16; y_disp [R, d] bf16; dy_disp out [R, d] bf16;
 *   dgate out [T, K] fp32.
 */
moe_status moe_combine_backward(const moe_shape *s, const moe_bf16 *dy, const moe_bf16 *y_disp,
                                const int32_t *route_row, const float *topk_gate,
                                moe_bf16 *dy_disp, float *dgate, cudaStream_t stream);

/*
 * moe_dispatch_backward -- step B3.  Section 05 Table 8 "Dispatch backward
 * GET": dx[t] = sum over k ascending (route_row >= 0) of dx_disp[route_row[t, k]],
 * fp32 accumulation from 0.
 *   dx_disp [R, d] bf16; route_row [T, K]; dx out [T, d] fp32.
 */
moe_status moe_dispatch_backward(const moe_shape *s, const moe_bf16 *dx_disp,
                                 const int32_t *route_row, float *dx, cudaStream_t stream);

/*
 * Checked variants of the four row movements, for debugging a route map that
 * did not come from moe_route (Section 05, 5.4: a negative row marks a
 * dropped route; every other row must name a row of the capacity buffers).
 * Same arguments and results as moe_dispatch, moe_combine,
 * moe_combine_backward and moe_dispatch_backward, plus status_ws: a device
 * workspace of at least 256 bytes, 256-byte aligned, whose word 0 is the
 * status word (zero it before the first call; moe_read_device_error reads
 * and clears it).  The kernels compare every route row with
 * R = moe_buffer_rows(s) before using it: a row >= R records
 * MOE_ERR_DEVICE_ROUTE_RANGE in the status word and the route is skipped as
 * if it were dropped (nothing is read or written through it), so the outputs
 * equal those of the same route map with that entry set to -1.  The check
 * costs one comparison per route; the release calls above run kernels with
 * the check compiled out.  Host-side errors: as the release calls, plus
 * MOE_ERR_WORKSPACE for a missing or misaligned status_ws.
 */
moe_status moe_dispatch_checked(const moe_shape *s, const moe_bf16 *x, const int32_t *route_row,
                                moe_bf16 *x_disp, void *status_ws, cudaStream_t stream);
moe_status moe_combine_checked(const moe_shape *s, const moe_bf16 *y_disp,
                               const int32_t *route_row, const float *topk_gate, moe_bf16 *y,
                               void *status_ws, cudaStream_t stream);
moe_status moe_combine_backward_checked(const moe_shape *s, const moe_bf16 *dy,
                                        const moe_bf16 *y_disp, const int32_t *route_row,
                                        const float *topk_gate, moe_bf16 *dy_disp, float *dgate,
                                        void *status_ws, cudaStream_t stream);
moe_status moe_dispatch_backward_checked(const moe_shape *s, const moe_bf16 *dx_disp,
                                         const int32_t *route_row, float *dx, void *status_ws,
                                         cudaStream_t stream);

/* Bytes of workspace moe_router_backward and moe_router_weight_backward need
 * (per-chunk partial sums of dW_r and dbias: at most 32 * N * (d + 1) floats;
 * 0 if the shape is invalid). */
size_t moe_router_backward_workspace_bytes(const moe_shape *s);

/*
 * moe_router_backward -- the router's share of the backward, with the top-K
 * selection of the forward held fixed.  Section 05, 5.6 (the router-weight
 * gradient starts from dgate, the gathered expert outputs against the token-
 * output gradient) and Figure 15 (the K gates of a token are a softmax over
 * its K chosen logits); AWS Neuron "Router Weights" (one fp32 [N, d] router
 * weight scores every expert).  For token t with gates g and dgate dg:
 *   dlogit[t, k] = g[t, k] * (dg[t, k] - dot),  dot = sum_k' g[t, k'] * dg[t, k']
 *   dx[t, :]    += sum_k dlogit[t, k] * w_router[topk_idx[t, k], :]
 *   dw_router[e, :] = sum over routes with topk_idx = e of dlogit * x[t, :]
 *   dbias[e]        = sum over the same routes of dlogit
 * A dropped route keeps its gate in the softmax, so its dlogit is not zero
 * even though its dgate is.  Experts that are not selected get no gradient.
 *   x [T, d] bf16 (the forward's input); w_router [N, d] fp32;
 *   topk_idx, topk_gate [T, K] as moe_route wrote them (entries outside
 *   [0, N) are skipped); dgate [T, K] fp32 as moe_combine_backward wrote it;
 *   dlogit out [T, K] fp32; dx in/out [T, d] fp32 (the router term is ADDED:
 *   call after moe_dispatch_backward to get the layer's whole input
 *   gradient); dw_router out [N, d] fp32 (overwritten); dbias out [N] fp32 or
 *   NULL.  fp32 arithmetic: dot is a fused multiply-add chain over k
 *   ascending; the dx term is summed over k ascending and then added; dW_r is
 *   summed per expert in token order within fixed 128-token chunks, the
 *   chunk sums added in a fixed order (deterministic, bit-identical run to run).
 * Errors: MOE_ERR_INVALID_ARG for null required pointers; MOE_ERR_ALIGNMENT;
 * MOE_ERR_WORKSPACE if ws is short or not 256-byte aligned;
 * MOE_ERR_UNSUPPORTED if N and K need more than 227 KB of shared memory.
 * Same result as moe_dispatch_router_backward (in place of
 * moe_dispatch_backward) followed by moe_router_weight_backward, which is the
 * faster pair: it walks each token's rows once for both dx terms.
 */
moe_status moe_router_backward(const moe_shape *s, const moe_bf16 *x, const float *w_router,
                               const int32_t *topk_idx, const float *topk_gate,
                               const float *dgate, float *dlogit, float *dx, float *dw_router,
                               float *dbias, void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * moe_dispatch_router_backward -- steps B3 and the router's input gradient in
 * one pass over each token (Section 05 Table 8 "Dispatch backward GET", 5.6,
 * Figure 15):
 *   dlogit[t, k] as in moe_router_backward (written);
 *   dx[t] = (sum over k ascending, route_row >= 0, of dx_disp[route_row[t, k]])
 *           + (sum over k ascending of dlogit[t, k] * w_router[topk_idx[t, k]])
 * each sum fp32 from 0, then the two added: bit-identical to
 * moe_dispatch_backward followed by the dx part of moe_router_backward.
 *   dx_disp [R, d] bf16; route_row, topk_idx, topk_gate, dgate [T, K];
 *   w_router [N, d] fp32; dlogit out [T, K] fp32; dx out [T, d] fp32.
 * Errors: as moe_dispatch_backward, plus MOE_ERR_INVALID_ARG for a null
 * router pointer.
 */
moe_status moe_dispatch_router_backward(const moe_shape *s, const moe_bf16 *dx_disp,
                                        const int32_t *route_row, const float *w_router,
                                        const int32_t *topk_idx, const float *topk_gate,
                                        const float *dgate, float *dlogit, float *dx,
                                        cudaStream_t stream);

/*
 * moe_router_weight_backward -- dw_router and dbias (NULL allowed) from the
 * dlogit that moe_dispatch_router_backward wrote, as in moe_router_backward.
 *   x [T, d] bf16; topk_idx [T, K]; dlogit [T, K] fp32; dw_router out [N, d]
 *   fp32; ws of moe_router_backward_workspace_bytes bytes, 256-byte aligned.
 */
moe_status moe_router_weight_backward(const moe_shape *s, const moe_bf16 *x,
                                      const int32_t *topk_idx, const float *dlogit,
                                      float *dw_router, float *dbias, void *ws, size_t ws_bytes,
                                      cudaStream_t stream);

/*
 * moe_read_device_error -- copies the device status word of a workspace to
 * *code_out (a moe_status value; MOE_OK if no kernel recorded an error) and
 * clears it.  ws is a device pointer; code_out a HOST pointer.  This call
 * synchronises `stream`: meant for tests and diagnostics, not the hot path.
 */
moe_status moe_read_device_error(void *ws, int32_t *code_out, cudaStream_t stream);

/*
 * moe_selftest_wait_timeout -- diagnostic for the device-side failure path.
 * Launches one small kernel that waits, with the same bounded mbarrier wait
 * every kernel of this library uses, on a barrier that nothing completes.
 * After limit_ns (1 ns .. 100 ms) the wait gives up and records
 * MOE_ERR_DEVICE_TIMEOUT in the workspace's status word, exactly as a stuck
 * GEMM pipeline would, and the kernel returns; the CUDA context stays usable.
 * ws: any 256-byte aligned workspace of this library.  No counterpart in the
 * report (it describes no failure handling for this path).
 */
moe_status moe_selftest_wait_timeout(void *ws, uint64_t limit_ns, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
