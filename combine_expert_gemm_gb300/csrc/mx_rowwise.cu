// MXFP8 row kernels: weight quantization, the quantizing dispatch (step D)
// and the dequantizing combine (step C).
//
// OLMo-core MoE report, "Section 05: Expert Parallelism": 5.4 (rows are
// quantized as they are dispatched; the outputs come back quantized and the
// local reduction dequantizes them), 5.7 (a quantized route's data row and
// scale row follow the bf16 row's destination and validity), 5.8 (E4M3 data,
// E8M0 scales), Table 8 ("Dispatch forward PUT", "Combine forward GET").
// Format: OCP Microscaling (MX) v1.0 MXFP8, blocks of 32 along each row.
//
// All three are HBM-bound row movers, one warp per row (a token, or a weight
// row) and persistent grids of a few CTAs per SM.  In the weight quantizer a
// lane holds 4 consecutive elements of a 128-column group (a block of 32 is 8
// lanes); in the dispatch and the combine a lane holds 16 (a block is two
// lanes, so its maximum is one xor-shuffle away, and every access is 16
// bytes).  The four scale bytes of a 128-column group meet in the group's
// first lane and leave as one 32-bit store into the scale chunk.
#include <algorithm>

#include "../../include/moe_mxfp8.h"
#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int kMxThreads = 256;
constexpr int kMxWarps = kMxThreads / 32;

inline unsigned mx_grid(int64_t items) {
    const int64_t per_cta = kMxWarps;
    const int64_t want = (items + per_cta - 1) / per_cta;
    return (unsigned)std::max<int64_t>(1, std::min<int64_t>(want, (int64_t)num_sms() * 8));
}

// The quantization of one lane's 4 elements within its 8-lane block: codes
// (a0 in the low byte) and, in every lane, the block's E8M0 byte.
__device__ __forceinline__ uint32_t mx_quant_lane(float a0, float a1, float a2, float a3,
                                                  uint32_t &scale_byte) {
    float m = fmaxf(fmaxf(fabsf(a0), fabsf(a1)), fmaxf(fabsf(a2), fabsf(a3)));
    m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
    m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 4));
    const int E = mx_exponent(m);
    const float inv = mx_inv_scale(E);
    scale_byte = (uint32_t)(E + 127);
    return e4m3x4(a0 * inv, a1 * inv, a2 * inv, a3 * inv);
}

// The four blocks' scale bytes of a 128-column group, block 0 in the low byte
// (valid in lane 0).
__device__ __forceinline__ uint32_t mx_group_scales(uint32_t scale_byte) {
    const uint32_t s1 = __shfl_sync(0xFFFFFFFFu, scale_byte, 8);
    const uint32_t s2 = __shfl_sync(0xFFFFFFFFu, scale_byte, 16);
    const uint32_t s3 = __shfl_sync(0xFFFFFFFFu, scale_byte, 24);
    return scale_byte | (s1 << 8) | (s2 << 16) | (s3 << 24);
}

__device__ __forceinline__ void bf16x4(uint2 w, float &a0, float &a1, float &a2, float &a3) {
    a0 = bf16_lo(w.x);
    a1 = bf16_hi(w.x);
    a2 = bf16_lo(w.y);
    a3 = bf16_hi(w.y);
}

// Weights: item = (matrix row, 128-column group); the group's scale word goes
// into each of the four copies of its chunk.
__global__ void __launch_bounds__(kMxThreads)
mx_quantize_weight_rows(int64_t rows, int k, const uint2 *__restrict__ w, uint32_t *__restrict__ q,
                        uint8_t *__restrict__ sf) {
    pdl_enter();
    const int lane = threadIdx.x & 31;
    const int groups = k / 128;
    const int64_t items = rows * groups;
    for (int64_t it = (int64_t)blockIdx.x * kMxWarps + (threadIdx.x >> 5); it < items;
         it += (int64_t)gridDim.x * kMxWarps) {
        const int64_t row = it / groups;
        const int g = (int)(it % groups);
        const int64_t e4 = (row * k + (int64_t)g * 128) / 4 + lane;  // in 4-element units
        float a0, a1, a2, a3;
        bf16x4(__ldcs(w + e4), a0, a1, a2, a3);
        uint32_t sb;
        q[e4] = mx_quant_lane(a0, a1, a2, a3, sb);
        const uint32_t word = __shfl_sync(0xFFFFFFFFu, mx_group_scales(sb), 0);
        if (lane < kMxWeightCopies)  // the same word into each of the chunk's copies
            *reinterpret_cast<uint32_t *>(
                sf + mx_wchunk_byte(row / 128, k, (int)(row % 128), 4 * g, lane)) = word;
    }
}

// pad_block[e] = sum over e' < e of ceil(count[e'] / 128), by warp 0.
__device__ __forceinline__ void pad_block_prefix(int N, const int32_t *__restrict__ count,
                                                 int32_t *pad_block, int lane) {
    int carry = 0;
    for (int base = 0; base < N; base += 32) {
        const int e = base + lane;
        const int v = e < N ? (count[e] + 127) / 128 : 0;
        int incl = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int u = __shfl_up_sync(0xFFFFFFFFu, incl, off);
            if (lane >= off) incl += u;
        }
        if (e < N) pad_block[e] = carry + incl - v;
        carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
}

// 16 fp32 values of one lane (half of a 32-block; the other half is in the
// neighbouring lane, lane ^ 1) -> 16 E4M3 codes and the block's E8M0 byte.
__device__ __forceinline__ uint4 mx_quant_lane16(const float (&a)[16], uint32_t &scale_byte) {
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(a[i]));
    m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
    const int E = mx_exponent(m);
    const float inv = mx_inv_scale(E);
    scale_byte = (uint32_t)(E + 127);
    return make_uint4(e4m3x4(a[0] * inv, a[1] * inv, a[2] * inv, a[3] * inv),
                      e4m3x4(a[4] * inv, a[5] * inv, a[6] * inv, a[7] * inv),
                      e4m3x4(a[8] * inv, a[9] * inv, a[10] * inv, a[11] * inv),
                      e4m3x4(a[12] * inv, a[13] * inv, a[14] * inv, a[15] * inv));
}

__device__ __forceinline__ void bf16x8(uint4 w, float *a) {
    a[0] = bf16_lo(w.x); a[1] = bf16_hi(w.x); a[2] = bf16_lo(w.y); a[3] = bf16_hi(w.y);
    a[4] = bf16_lo(w.z); a[5] = bf16_hi(w.z); a[6] = bf16_lo(w.w); a[7] = bf16_hi(w.w);
}

// Dispatch: one warp per token, a lane owns 16 consecutive columns of a
// 512-column step (a block of 32 is two lanes, a 128-column group eight).
// Each step is quantized once; its codes (16 bytes per lane) and the four
// scale words (lanes 0, 8, 16, 24) go to every accepted route row.
constexpr int kDispStep = 512;

__global__ void __launch_bounds__(kMxThreads)
dispatch_mx_rows(int T, int d, int K, int N, const uint4 *__restrict__ x,
                 const int32_t *__restrict__ route_row, const int32_t *__restrict__ topk_idx,
                 const int32_t *__restrict__ count, const int32_t *__restrict__ offset,
                 uint4 *__restrict__ xq, uint8_t *__restrict__ xsf) {
    pdl_enter();
    extern __shared__ int32_t pad_block[];
    const int lane = threadIdx.x & 31;
    if ((threadIdx.x >> 5) == 0) pad_block_prefix(N, count, pad_block, lane);
    __syncthreads();
    const int steps = (d + kDispStep - 1) / kDispStep;
    const int64_t x8 = d / 8;    // uint4 (8 bf16) per token row
    const int64_t q16 = d / 16;  // uint4 (16 codes) per packed row
    for (int t = blockIdx.x * kMxWarps + (threadIdx.x >> 5); t < T; t += gridDim.x * kMxWarps) {
        int32_t my_row = -1, my_blk = 0, my_rin = 0;
        if (lane < K) {
            my_row = route_row[(int64_t)t * K + lane];
            if (my_row >= 0) {
                const int e = topk_idx[(int64_t)t * K + lane];
                const int slot = my_row - offset[e];
                my_blk = pad_block[e] + slot / 128;
                my_rin = slot % 128;
            }
        }
        const uint4 *src = x + (int64_t)t * x8;
        for (int st0 = 0; st0 < steps; st0 += 2) {
            uint4 v[2][2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int col = (st0 + u) * kDispStep + lane * 16;
                if (col < d) {
                    v[u][0] = __ldcs(src + col / 8);
                    v[u][1] = __ldcs(src + col / 8 + 1);
                }
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int st = st0 + u;
                if (st >= steps) break;  // warp-uniform
                const int col = st * kDispStep + lane * 16;
                const bool on = col < d;  // whole 8-lane groups (d is a multiple of 128)
                float a[16];
                if (on) {
                    bf16x8(v[u][0], a);
                    bf16x8(v[u][1], a + 8);
                } else {
#pragma unroll
                    for (int i = 0; i < 16; ++i) a[i] = 0.0f;
                }
                uint32_t sb;
                const uint4 codes = mx_quant_lane16(a, sb);
                // the group's four block scales meet in the group's first lane
                const uint32_t s1 = __shfl_down_sync(0xFFFFFFFFu, sb, 2);
                const uint32_t s2 = __shfl_down_sync(0xFFFFFFFFu, sb, 4);
                const uint32_t s3 = __shfl_down_sync(0xFFFFFFFFu, sb, 6);
                const uint32_t word = sb | (s1 << 8) | (s2 << 16) | (s3 << 24);
                const bool group_lead = on && (lane & 7) == 0;
                const int kb = col / 32;  // first block of the lane's group when group_lead
                for (int k = 0; k < K; ++k) {
                    const int32_t r = __shfl_sync(0xFFFFFFFFu, my_row, k);
                    if (r < 0) continue;
                    const int32_t blk = __shfl_sync(0xFFFFFFFFu, my_blk, k);
                    const int32_t rin = __shfl_sync(0xFFFFFFFFu, my_rin, k);
                    if (on) xq[(int64_t)r * q16 + col / 16] = codes;
                    if (group_lead)
                        *reinterpret_cast<uint32_t *>(xsf + mx_chunk_byte(blk, d, rin, kb)) = word;
                }
            }
        }
    }
}

// Combine: one warp per token, a lane owns 16 consecutive columns of a
// 512-column step; y[t] = bf16(sum_k gate_k * deq(row_k)) with an fp32 FMA
// chain over k ascending (each dequantized value e4m3 * 2^(s - 127) is exact).
// For K <= 4 the token's accepted routes are first compacted to lanes
// 0..nv-1 (k ascending) and each pass covers two steps per lane, so 8 code
// loads per lane are in flight with 4 accepted routes (the K > 4 kernel
// below keeps one step of all K routes in flight instead: two steps of 8
// rows would need more registers than the occupancy allows).
__device__ __forceinline__ void mx_fma16(float (&acc)[16], float g, uint4 code, uint32_t sc) {
    const float s = e8m0_value(sc);
    const uint32_t w[4] = {code.x, code.y, code.z, code.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 lo = e4m3x2_to_f32((uint16_t)(w[j] & 0xFFFFu));
        const float2 hi = e4m3x2_to_f32((uint16_t)(w[j] >> 16));
        acc[4 * j] = fmaf(g, lo.x * s, acc[4 * j]);
        acc[4 * j + 1] = fmaf(g, lo.y * s, acc[4 * j + 1]);
        acc[4 * j + 2] = fmaf(g, hi.x * s, acc[4 * j + 2]);
        acc[4 * j + 3] = fmaf(g, hi.y * s, acc[4 * j + 3]);
    }
}

__device__ __forceinline__ void store_bf16x16(uint4 *dst, const float (&acc)[16]) {
    dst[0] = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                        pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
    dst[1] = make_uint4(pack_bf16x2(acc[8], acc[9]), pack_bf16x2(acc[10], acc[11]),
                        pack_bf16x2(acc[12], acc[13]), pack_bf16x2(acc[14], acc[15]));
}

template <int MAXK>
__global__ void __launch_bounds__(kMxThreads)
combine_mx_rows(int T, int d, int K, const uint4 *__restrict__ yq, const uint8_t *__restrict__ ys,
                const int32_t *__restrict__ route_row, const float *__restrict__ gate,
                uint4 *__restrict__ y) {
    pdl_enter();
    const int lane = threadIdx.x & 31;
    const int64_t q16 = d / 16;
    const int64_t y8 = d / 8;
    const int sc_row = d / 32;
    for (int t = blockIdx.x * kMxWarps + (threadIdx.x >> 5); t < T; t += gridDim.x * kMxWarps) {
        const int32_t my_row = lane < K ? route_row[(int64_t)t * K + lane] : -1;
        const float my_g = lane < K ? gate[(int64_t)t * K + lane] : 0.0f;
        // lane j < nv gets the j-th accepted route (k ascending)
        int32_t rc = -1;
        float gc = 0.0f;
        int nv = 0;  // warp-uniform
#pragma unroll
        for (int k = 0; k < MAXK; ++k) {
            const int32_t r = __shfl_sync(0xFFFFFFFFu, my_row, k);
            const float g = __shfl_sync(0xFFFFFFFFu, my_g, k);
            if (k < K && r >= 0) {
                if (lane == nv) {
                    rc = r;
                    gc = g;
                }
                ++nv;
            }
        }
        for (int c0 = 0; c0 < d; c0 += 2 * kDispStep) {  // warp-uniform
            const int ca = c0 + lane * 16, cb = ca + kDispStep;
            float acc[2][16];
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int i = 0; i < 16; ++i) acc[h][i] = 0.0f;
#pragma unroll
            for (int g0 = 0; g0 < MAXK; g0 += 4) {
                if (g0 >= nv) break;
                float gg[4];
                uint4 code[4][2];
                uint32_t sc[4][2];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int32_t r = __shfl_sync(0xFFFFFFFFu, rc, g0 + u);
                    gg[u] = __shfl_sync(0xFFFFFFFFu, gc, g0 + u);
                    if (g0 + u < nv) {
                        if (ca < d) {
                            code[u][0] = __ldcs(yq + (int64_t)r * q16 + ca / 16);
                            sc[u][0] = ys[(int64_t)r * sc_row + ca / 32];
                        }
                        if (cb < d) {
                            code[u][1] = __ldcs(yq + (int64_t)r * q16 + cb / 16);
                            sc[u][1] = ys[(int64_t)r * sc_row + cb / 32];
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if (g0 + u >= nv) continue;
                    if (ca < d) mx_fma16(acc[0], gg[u], code[u][0], sc[u][0]);
                    if (cb < d) mx_fma16(acc[1], gg[u], code[u][1], sc[u][1]);
                }
            }
            if (ca < d) store_bf16x16(y + (int64_t)t * y8 + ca / 8, acc[0]);
            if (cb < d) store_bf16x16(y + (int64_t)t * y8 + cb / 8, acc[1]);
        }
    }
}

// Combine for K > 4: one 512-column step per pass, all K route rows of the
// step in flight (the same fp32 FMA chain over k ascending).
template <int MAXK>
__global__ void __launch_bounds__(kMxThreads)
combine_mx_rows_wide_k(int T, int d, int K, const uint4 *__restrict__ yq, const uint8_t *__restrict__ ys,
                const int32_t *__restrict__ route_row, const float *__restrict__ gate,
                uint4 *__restrict__ y) {
    pdl_enter();
    const int lane = threadIdx.x & 31;
    const int64_t q16 = d / 16;
    const int64_t y8 = d / 8;
    const int sc_row = d / 32;
    for (int t = blockIdx.x * kMxWarps + (threadIdx.x >> 5); t < T; t += gridDim.x * kMxWarps) {
        const int32_t my_row = lane < K ? route_row[(int64_t)t * K + lane] : -1;
        const float my_g = lane < K ? gate[(int64_t)t * K + lane] : 0.0f;
        int32_t rows[MAXK];
        float gs[MAXK];
#pragma unroll
        for (int k = 0; k < MAXK; ++k) {
            rows[k] = __shfl_sync(0xFFFFFFFFu, my_row, k);
            gs[k] = __shfl_sync(0xFFFFFFFFu, my_g, k);
        }
        for (int col = lane * 16; col < d; col += kDispStep) {
            uint4 code[MAXK];
            uint32_t sc[MAXK];
#pragma unroll
            for (int k = 0; k < MAXK; ++k) {
                if (k < K && rows[k] >= 0) {
                    code[k] = __ldcs(yq + (int64_t)rows[k] * q16 + col / 16);
                    sc[k] = ys[(int64_t)rows[k] * sc_row + col / 32];
                }
            }
            float acc[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
#pragma unroll
            for (int k = 0; k < MAXK; ++k) {
                if (k < K && rows[k] >= 0) {
                    const float s = e8m0_value(sc[k]);
                    const uint32_t w[4] = {code[k].x, code[k].y, code[k].z, code[k].w};
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const float2 lo = e4m3x2_to_f32((uint16_t)(w[j] & 0xFFFFu));
                        const float2 hi = e4m3x2_to_f32((uint16_t)(w[j] >> 16));
                        acc[4 * j] = fmaf(gs[k], lo.x * s, acc[4 * j]);
                        acc[4 * j + 1] = fmaf(gs[k], lo.y * s, acc[4 * j + 1]);
                        acc[4 * j + 2] = fmaf(gs[k], hi.x * s, acc[4 * j + 2]);
                        acc[4 * j + 3] = fmaf(gs[k], hi.y * s, acc[4 * j + 3]);
                    }
                }
            }
            uint4 *dst = y + (int64_t)t * y8 + col / 8;
            dst[0] = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]),
                                pack_bf16x2(acc[4], acc[5]), pack_bf16x2(acc[6], acc[7]));
            dst[1] = make_uint4(pack_bf16x2(acc[8], acc[9]), pack_bf16x2(acc[10], acc[11]),
                                pack_bf16x2(acc[12], acc[13]), pack_bf16x2(acc[14], acc[15]));
        }
    }
}

}  // namespace
}  // namespace moe

using namespace moe;

MOE_API size_t moe_mx_act_scale_bytes(const moe_shape *s, int32_t k) {
    if (check_shape(s) != MOE_OK || k <= 0 || k % 128 != 0) return 0;
    return mx_act_scale_bytes(buffer_rows(s), s->N, k);
}

MOE_API moe_status moe_mx_quantize_weights(int32_t E, int32_t rows, int32_t k, const moe_bf16 *w,
                                           uint8_t *q, uint8_t *sf, cudaStream_t stream) {
    if (E < 0 || rows < 0 || k < 0) return MOE_ERR_INVALID_ARG;
    if (rows % 128 != 0 || k % 128 != 0) return MOE_ERR_UNSUPPORTED;
    const int64_t n = (int64_t)E * rows;
    if (n == 0 || k == 0) return MOE_OK;
    if (!w || !q || !sf) return MOE_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(q) || !aligned16(sf)) return MOE_ERR_ALIGNMENT;
    launch_pdl(mx_quantize_weight_rows, mx_grid(n * (k / 128)), kMxThreads, 0, stream, n, k,
               reinterpret_cast<const uint2 *>(w), reinterpret_cast<uint32_t *>(q), sf);
    return launch_status();
}

MOE_API moe_status moe_dispatch_mxfp8(const moe_shape *s, const moe_bf16 *x,
                                      const int32_t *route_row, const int32_t *topk_idx,
                                      const int32_t *expert_count, const int32_t *expert_offset,
                                      uint8_t *x_q, uint8_t *x_sf, cudaStream_t stream) {
    moe_status r = check_shape(s);
    if (r != MOE_OK) return r;
    if (s->d % 128 != 0) return MOE_ERR_UNSUPPORTED;
    if (s->T == 0 || s->cap == 0) return MOE_OK;
    if (!x || !route_row || !topk_idx || !expert_count || !expert_offset || !x_q || !x_sf)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(route_row) || !aligned16(topk_idx) || !aligned16(x_q) ||
        !aligned16(x_sf))
        return MOE_ERR_ALIGNMENT;
    launch_pdl(dispatch_mx_rows, mx_grid(s->T), kMxThreads, sizeof(int32_t) * s->N, stream, s->T,
               s->d, s->K, s->N, reinterpret_cast<const uint4 *>(x), route_row, topk_idx,
               expert_count, expert_offset, reinterpret_cast<uint4 *>(x_q), x_sf);
    return launch_status();
}

MOE_API moe_status moe_combine_mxfp8(const moe_shape *s, const uint8_t *y_q, const uint8_t *y_scale,
                                     const int32_t *route_row, const float *topk_gate, moe_bf16 *y,
                                     cudaStream_t stream) {
    moe_status r = check_shape(s);
    if (r != MOE_OK) return r;
    if (s->d % 128 != 0) return MOE_ERR_UNSUPPORTED;
    if (s->T == 0) return MOE_OK;
    if (!route_row || !topk_gate || !y || (s->cap > 0 && (!y_q || !y_scale)))
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(y_q) || !aligned16(y_scale) || !aligned16(route_row) || !aligned16(topk_gate) ||
        !aligned16(y))
        return MOE_ERR_ALIGNMENT;
    auto *kern = s->K <= 4   ? combine_mx_rows<4>
                 : s->K <= 8 ? combine_mx_rows_wide_k<8>
                             : combine_mx_rows_wide_k<16>;
    launch_pdl(kern, mx_grid(s->T), kMxThreads, 0, stream, s->T, s->d, s->K,
               reinterpret_cast<const uint4 *>(y_q), y_scale, route_row, topk_gate,
               reinterpret_cast<uint4 *>(y));
    return launch_status();
}
