/*
 * moe_mxfp8.h -- C ABI of the MXFP8 variant of the routed-expert layer:
 * dispatch that quantizes the token rows as it places them, grouped SwiGLU
 * experts whose two GEMMs read E4M3 data with E8M0 block scales on the
 * tensor cores, and a combine that dequantizes the experts' quantized outputs
 * in its weighted sum.  Routing (moe_route) is shared with the bf16 path.
 *
 * Sources (page title, then section):
 *   OLMo-core MoE report, "Section 05: Expert Parallelism": 5.4 (rows are
 *   quantized during dispatch; expert grouped GEMM consumes the received
 *   quantized data and scales directly; outputs return quantized before the
 *   local reduction, with no bf16 copy in between), 5.7 (a quantized route
 *   carries a data row and a scale row that follow the same destination rows
 *   and validity as the bf16 row), 5.8 (E4M3 data with E8M0 scales; both
 *   expert GEMMs in MXFP8).
 *
 * Format (the pages name it; the rules are the OCP Microscaling (MX) v1.0
 * definition of MXFP8): blocks of 32 consecutive elements along a row share
 * one scale 2^E, stored as the byte E + 127, E = floor(log2 max|v|) - 8
 * clamped to [-127, 127] (an all-zero block gets byte 0); each element is
 * v / 2^E rounded to the nearest E4M3 value, ties to even, magnitudes past 448
 * saturated to 448.  Inputs must be finite.
 *
 * Scale layouts.  A row-major scale row [rows, k / 32] ("scale rows") is used
 * where rows are read one by one (the experts' outputs y_scale).  Operands of
 * the tensor cores keep their scales in scale chunks instead: one 512-byte
 * chunk per 128 rows x 128 columns, the scale of row r (0-127) and block b
 * (0-3) at byte (r % 32) * 16 + (r / 32) * 4 + b, chunk (block128, g) at byte
 * (block128 * k / 128 + g) * 512.  Weights number their row blocks
 * e * rows / 128 + row / 128 and store every chunk four times in a row:
 * copy c (0-3) of chunk (block128, g) at byte
 * ((block128 * k / 128 + g) * 4 + c) * 512 -- the GEMM moves the copies into
 * tensor memory, one per lane quadrant, with a single copy instruction.
 * Packed capacity-buffer rows number them per
 * expert: block128 = pad_block[e] + (row - expert_offset[e]) / 128 with
 * pad_block[e] = sum over e' < e of ceil(expert_count[e'] / 128), so every
 * expert starts a fresh chunk and a GEMM tile never straddles two experts'
 * chunks.  Chunk bytes of rows that hold no route are never written or read
 * for a result.
 *
 * Conventions as in moe.h (device pointers, asynchronous on `stream`, no
 * host synchronisation, 16-byte aligned pointers, argument errors returned
 * before anything is enqueued).  MXFP8 calls need d and h to be multiples of
 * 128 (MOE_ERR_UNSUPPORTED otherwise).
 */
#ifndef MOE_GB300_MXFP8_H
#define MOE_GB300_MXFP8_H

#include "moe.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Bytes of the scale-chunk array of a packed capacity buffer with k columns
 * (k = d for the dispatched rows, k = h for the SwiGLU outputs):
 * (ceil(R / 128) + N) * (k / 128) * 512; 0 if the shape is invalid or k is not
 * a positive multiple of 128. */
size_t moe_mx_act_scale_bytes(const moe_shape *s, int32_t k);

/*
 * moe_mx_quantize_weights -- quantizes E stacked [rows, k] bf16 matrices
 * along k (the reduction dimension of the product that reads them):
 *   w [E, rows, k] bf16 -> q [E, rows, k] E4M3 codes and
 *   sf: E * rows * k / 8 bytes of scale chunks, each chunk four times over
 *   (block128 = e * rows / 128 + row / 128).  For the experts: w_gate, w_up
 *   [N, h, d] (rows = h, k = d) and w_down [N, d, h] (rows = d, k = h).
 * rows and k must be multiples of 128 (MOE_ERR_UNSUPPORTED otherwise).
 */
moe_status moe_mx_quantize_weights(int32_t E, int32_t rows, int32_t k, const moe_bf16 *w,
                                   uint8_t *q, uint8_t *sf, cudaStream_t stream);

/*
 * moe_dispatch_mxfp8 -- step D in MXFP8 (Section 05, 5.4 and 5.7): each token
 * row x[t] is quantized once along d and its codes and scales are written to
 * every accepted route row r = route_row[t, k] >= 0 of expert
 * e = topk_idx[t, k]:
 *   x_q [R, d] E4M3 codes, row r;
 *   x_sf scale chunks (moe_mx_act_scale_bytes(s, d) bytes), row r's bytes.
 * Rows not named by route_row are untouched.  expert_count and
 * expert_offset [N + 1] are moe_route's.  Nothing is written when cap = 0.
 */
moe_status moe_dispatch_mxfp8(const moe_shape *s, const moe_bf16 *x, const int32_t *route_row,
                              const int32_t *topk_idx, const int32_t *expert_count,
                              const int32_t *expert_offset, uint8_t *x_q, uint8_t *x_sf,
                              cudaStream_t stream);

/*
 * moe_expert_ffn_mxfp8 -- steps F1, F2 in MXFP8 (Section 05, 5.4 and 5.8;
 * Section 08, 8.5: device offsets, valid rows only).  For each expert e and
 * each of its rows r:
 *   G = X W_gate[e]^T, U = X W_up[e]^T   (X, W dequantized exactly inside the
 *                                          block-scaled MMA; fp32 accumulation)
 *   (h_q[r], h_sf) = MXFP8(silu(G) * U) along h     (fp32 SwiGLU)
 *   Y = H W_down[e]^T                                (fp32 accumulation)
 *   (y_q[r], y_scale[r]) = MXFP8(Y) along d
 *   x_q [R, d], x_sf as moe_dispatch_mxfp8 wrote them;
 *   w_*_q and w_*_sf as moe_mx_quantize_weights wrote them;
 *   h_q out [R, h] and h_sf out (moe_mx_act_scale_bytes(s, h) bytes of
 *   chunks): the SwiGLU output, F2's A operand;
 *   y_q out [R, d] codes and y_scale out [R, d / 32] row-major scale rows;
 *   ws of moe_expert_ffn_workspace_bytes(s) bytes (device status word).
 * Errors: as moe_expert_ffn; MOE_ERR_UNSUPPORTED unless d and h are
 * multiples of 128.
 */
moe_status moe_expert_ffn_mxfp8(const moe_shape *s, const uint8_t *x_q, const uint8_t *x_sf,
                                const int32_t *expert_count, const int32_t *expert_offset,
                                const uint8_t *w_gate_q, const uint8_t *w_gate_sf,
                                const uint8_t *w_up_q, const uint8_t *w_up_sf,
                                const uint8_t *w_down_q, const uint8_t *w_down_sf, uint8_t *h_q,
                                uint8_t *h_sf, uint8_t *y_q, uint8_t *y_scale, void *ws,
                                size_t ws_bytes, cudaStream_t stream);

/*
 * moe_combine_mxfp8 -- step C over quantized expert outputs (Section 05,
 * 5.4: the local reduction dequantizes): y[t] = bf16( sum over k ascending
 * (route_row >= 0) of topk_gate[t, k] * deq(y_q, y_scale)[route_row[t, k]] ),
 * an fp32 fused multiply-add chain from 0 over exactly dequantized values.
 *   y_q [R, d]; y_scale [R, d / 32]; route_row, topk_gate [T, K]; y out [T, d].
 */
moe_status moe_combine_mxfp8(const moe_shape *s, const uint8_t *y_q, const uint8_t *y_scale,
                             const int32_t *route_row, const float *topk_gate, moe_bf16 *y,
                             cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_MXFP8_H */
