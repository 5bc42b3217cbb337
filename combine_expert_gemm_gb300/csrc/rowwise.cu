// Rowwise movement between token order and the packed capacity buffers.
//
// OLMo-core MoE report, "Section 05: Expert Parallelism", 5.6 and Table 8:
// dispatch forward is a PUT of x_t to each accepted route's row, combine
// forward a GET of the K expert rows with the router-weighted reduction done at
// the token, and the backward pair applies the transposed movements with the
// same route map; negative rows are skipped and contribute zero.  Figure 19:
// the token row is read once and fanned out by its source.
//
// One warp per token; every access is a 16-byte vector (8 bf16); the K route
// rows and gates of the token are read once by lanes 0..K-1 and broadcast with
// shuffles.  All four kernels are HBM-bound.  The dispatch backward can also
// add the router's share of dx (and write dlogit) in the same pass over the
// token's rows.
//
// Checked variants (CHECK = true; the *_checked entry points): every route
// row a kernel takes is first compared with the R rows of the capacity
// buffers.  A row at or past R is recorded as MOE_ERR_DEVICE_ROUTE_RANGE in the caller's status word
// and the route is skipped as if it were dropped, so no address outside the
// buffers is formed.  The release instantiations compile the check out.
#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kSeg = 8;  // 16-byte chunks per lane per pass (2048 bf16 per warp pass)

__device__ __forceinline__ void unpack8(const uint4 &v, float (&f)[8]) {
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x);
    f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z);
    f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8]) {
    return make_uint4(pack_bf16x2(f[0], f[1]), pack_bf16x2(f[2], f[3]), pack_bf16x2(f[4], f[5]),
                      pack_bf16x2(f[6], f[7]));
}

// A route row for a checked kernel: rows at or past R are recorded in the
// status word and read as -1 (dropped).
template <bool CHECK>
__device__ __forceinline__ int32_t checked_row(int32_t r, int64_t R, int32_t *status) {
    if (CHECK && r >= R) {
        atomicCAS(status, 0, (int32_t)MOE_ERR_DEVICE_ROUTE_RANGE);
        return -1;
    }
    return r;
}

template <bool CHECK>
__global__ void __launch_bounds__(kThreads)
dispatch_rows(int T, int nchunk, int K, const uint4 *__restrict__ x,
              const int32_t *__restrict__ route_row, uint4 *__restrict__ x_disp, int64_t R,
              int32_t *status) {
    pdl_enter();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (t >= T) return;
    const int32_t my_row =
        lane < K ? checked_row<CHECK>(route_row[(int64_t)t * K + lane], R, status) : -1;
    const uint4 *src = x + (int64_t)t * nchunk;
    for (int c0 = 0; c0 < nchunk; c0 += 32 * kSeg) {
        uint4 v[kSeg];
#pragma unroll
        for (int u = 0; u < kSeg; ++u) {
            const int c = c0 + u * 32 + lane;
            if (c < nchunk) v[u] = __ldcs(src + c);
        }
        for (int k = 0; k < K; ++k) {
            const int32_t r = __shfl_sync(0xFFFFFFFFu, my_row, k);
            if (r < 0) continue;
            uint4 *dst = x_disp + (int64_t)r * nchunk;
#pragma unroll
            for (int u = 0; u < kSeg; ++u) {
                const int c = c0 + u * 32 + lane;
                if (c < nchunk) dst[c] = v[u];
            }
        }
    }
}

// MAXK (8 or 16) bounds the route count K.  The token's accepted routes are
// first compacted to lanes 0..nv-1 (k ascending); each pass then covers two
// 16-byte chunks per lane and takes the accepted rows four at a time, so a
// token with few accepted routes (a drop-heavy layer) still keeps 8 loads per
// lane in flight.  The fp32 fma chain of every element runs over the
// accepted routes in k order, as before the compaction.
template <int MAXK, bool CHECK>
__global__ void __launch_bounds__(kThreads, MAXK <= 8 ? 4 : 2)
combine_rows(int T, int nchunk, int K, const uint4 *__restrict__ y_disp,
             const int32_t *__restrict__ route_row, const float *__restrict__ gate,
             uint4 *__restrict__ y, int64_t R, int32_t *status) {
    pdl_enter();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (t >= T) return;
    const int32_t my_row =
        lane < K ? checked_row<CHECK>(route_row[(int64_t)t * K + lane], R, status) : -1;
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
    // the chunk loop is warp-uniform (the shuffles need every lane)
    for (int c0 = 0; c0 < nchunk; c0 += 64) {
        const int ca = c0 + lane, cb = ca + 32;
        float acc[2][8];
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[h][i] = 0.0f;
#pragma unroll
        for (int g0 = 0; g0 < MAXK; g0 += 4) {
            if (g0 >= nv) break;
            int32_t r[4];
            float gg[4];
            uint4 v[4][2];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                r[u] = __shfl_sync(0xFFFFFFFFu, rc, g0 + u);
                gg[u] = __shfl_sync(0xFFFFFFFFu, gc, g0 + u);
                if (g0 + u < nv) {
                    const uint4 *src = y_disp + (int64_t)r[u] * nchunk;
                    if (ca < nchunk) v[u][0] = __ldcs(src + ca);
                    if (cb < nchunk) v[u][1] = __ldcs(src + cb);
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                if (g0 + u >= nv) continue;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    float f[8];
                    unpack8(v[u][h], f);
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[h][i] = __fmaf_rn(gg[u], f[i], acc[h][i]);
                }
            }
        }
        if (ca < nchunk) y[(int64_t)t * nchunk + ca] = pack8(acc[0]);
        if (cb < nchunk) y[(int64_t)t * nchunk + cb] = pack8(acc[1]);
    }
}

// Chunk-outer: for each 16-byte chunk of the token row, all K route rows are
// read at once; the K partial dot products for dgate stay in registers and
// are reduced across the warp at the end.
template <int MAXK, bool CHECK>
__global__ void __launch_bounds__(kThreads, MAXK <= 8 ? 3 : 2)
combine_bwd_rows(int T, int nchunk, int K, const uint4 *__restrict__ dy,
                 const uint4 *__restrict__ y_disp, const int32_t *__restrict__ route_row,
                 const float *__restrict__ gate, uint4 *__restrict__ dy_disp,
                 float *__restrict__ dgate, int64_t R, int32_t *status) {
    pdl_enter();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (t >= T) return;
    const int32_t my_row =
        lane < K ? checked_row<CHECK>(route_row[(int64_t)t * K + lane], R, status) : -1;
    const float my_g = lane < K ? gate[(int64_t)t * K + lane] : 0.0f;
    int32_t rows[MAXK];
    float gs[MAXK], part[MAXK];
#pragma unroll
    for (int k = 0; k < MAXK; ++k) {
        rows[k] = __shfl_sync(0xFFFFFFFFu, my_row, k);
        gs[k] = __shfl_sync(0xFFFFFFFFu, my_g, k);
        part[k] = 0.0f;
    }
    const uint4 *src = dy + (int64_t)t * nchunk;
    for (int c = lane; c < nchunk; c += 32) {
        float f[8];
        unpack8(src[c], f);
        uint4 v[MAXK];
#pragma unroll
        for (int k = 0; k < MAXK; ++k)
            if (k < K && rows[k] >= 0) v[k] = __ldcs(y_disp + (int64_t)rows[k] * nchunk + c);
#pragma unroll
        for (int k = 0; k < MAXK; ++k) {
            if (k >= K || rows[k] < 0) continue;
            float o[8], pr[8];
            unpack8(v[k], o);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                pr[i] = __fmul_rn(gs[k], f[i]);
                part[k] = __fmaf_rn(f[i], o[i], part[k]);
            }
            dy_disp[(int64_t)rows[k] * nchunk + c] = pack8(pr);
        }
    }
#pragma unroll
    for (int k = 0; k < MAXK; ++k) {
        if (k >= K) break;
        float v = part[k];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
        if (lane == 0) dgate[(int64_t)t * K + k] = rows[k] >= 0 ? v : 0.0f;
    }
}

// Dispatch backward, optionally with the router's share of the input
// gradient in the same pass over the token's row:
//   DBWD_PLAIN       dx[t]  = sum_k dx_disp[row_k]
//   DBWD_ROUTER      dx[t]  = sum_k dx_disp[row_k] + sum_k dlogit_k W_r[e_k]
//   DBWD_ROUTER_ADD  dx[t] += sum_k dlogit_k W_r[e_k]
// The router modes also compute and write dlogit (gate softmax Jacobian over
// the K chosen experts, "Section 05" Figure 15 and 5.6):
//   dot = fmaf chain over k ascending of g_k dgate_k;  dlogit_k = g_k (dgate_k - dot).
// W_r rows are fp32 and read through L1/L2 (the [N, d] weight is shared by
// every token).  Each sum runs over k ascending from 0 (deterministic); the
// router term is summed apart and added last, so DBWD_ROUTER gives the same
// bits as DBWD_PLAIN followed by DBWD_ROUTER_ADD.
enum { DBWD_PLAIN = 0, DBWD_ROUTER = 1, DBWD_ROUTER_ADD = 2 };

template <int MAXK, int MODE, bool CHECK = false>
__global__ void __launch_bounds__(kThreads, MODE == DBWD_PLAIN ? (MAXK <= 8 ? 4 : 2) : (MAXK <= 8 ? 2 : 1))
dispatch_bwd_rows(int T, int nchunk, int K, int N, const uint4 *__restrict__ dx_disp,
                  const int32_t *__restrict__ route_row, float4 *__restrict__ dx,
                  const float4 *__restrict__ w_r, const int32_t *__restrict__ topk_idx,
                  const float *__restrict__ gate, const float *__restrict__ dgate,
                  float *__restrict__ dlogit, int64_t R = 0, int32_t *status = nullptr) {
    pdl_enter();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (t >= T) return;
    // lane k < K holds route k's row, expert and dlogit; the chunk loop
    // broadcasts them with shuffles (fewer live registers than arrays)
    int32_t my_row = -1;
    if (MODE != DBWD_ROUTER_ADD && lane < K)
        my_row = checked_row<CHECK>(route_row[(int64_t)t * K + lane], R, status);
    float my_dl = 0.f;
    int32_t my_e = -1;
    if (MODE != DBWD_PLAIN) {
        float g = 0.f, dg = 0.f;
        if (lane < K) {
            g = gate[(int64_t)t * K + lane];
            dg = dgate[(int64_t)t * K + lane];
            my_e = topk_idx[(int64_t)t * K + lane];
            if (my_e < 0 || my_e >= N) my_e = -1;
        }
        float dot = 0.f;
#pragma unroll
        for (int k = 0; k < MAXK; ++k) {
            const float gk = __shfl_sync(0xFFFFFFFFu, g, k);
            const float dk = __shfl_sync(0xFFFFFFFFu, dg, k);
            if (k < K) dot = fmaf(gk, dk, dot);
        }
        my_dl = g * (dg - dot);
        if (lane < K) dlogit[(int64_t)t * K + lane] = my_dl;
    }
    int32_t rows_h[MAXK];
    if (MODE == DBWD_PLAIN) {
#pragma unroll
        for (int k = 0; k < MAXK; ++k) rows_h[k] = __shfl_sync(0xFFFFFFFFu, my_row, k);
    }
    // warp-uniform chunk loop: the shuffles below need every lane present
    for (int c0 = 0; c0 < nchunk; c0 += 32) {
        const int c = c0 + lane;
        const bool on = c < nchunk;
        float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (MODE == DBWD_ROUTER_ADD) {
            if (on) {
                const float4 *p = dx + ((int64_t)t * nchunk + c) * 2;
                const float4 a = p[0], b = p[1];
                acc[0] = a.x; acc[1] = a.y; acc[2] = a.z; acc[3] = a.w;
                acc[4] = b.x; acc[5] = b.y; acc[6] = b.z; acc[7] = b.w;
            }
        } else {
            uint4 v[MAXK];
            int32_t rows[MAXK];
#pragma unroll
            for (int k = 0; k < MAXK; ++k) {
                rows[k] = MODE == DBWD_PLAIN ? rows_h[k] : __shfl_sync(0xFFFFFFFFu, my_row, k);
                if (on && k < K && rows[k] >= 0)
                    v[k] = __ldcs(dx_disp + (int64_t)rows[k] * nchunk + c);
            }
#pragma unroll
            for (int k = 0; k < MAXK; ++k) {
                if (k >= K || rows[k] < 0) continue;
                float f[8];
                unpack8(v[k], f);
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = __fadd_rn(acc[i], f[i]);
            }
        }
        if (MODE != DBWD_PLAIN) {
            float r[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
            for (int k0 = 0; k0 < MAXK; k0 += 4) {
                float4 wa[4], wb[4];
                float dl[4];
                int32_t e[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    e[u] = __shfl_sync(0xFFFFFFFFu, my_e, k0 + u);
                    dl[u] = __shfl_sync(0xFFFFFFFFu, my_dl, k0 + u);
                    if (on && k0 + u < K && e[u] >= 0) {
                        const float4 *wp = w_r + ((int64_t)e[u] * nchunk + c) * 2;
                        wa[u] = __ldg(wp);
                        wb[u] = __ldg(wp + 1);
                    }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    if (k0 + u >= K || e[u] < 0) continue;
                    r[0] = fmaf(dl[u], wa[u].x, r[0]); r[1] = fmaf(dl[u], wa[u].y, r[1]);
                    r[2] = fmaf(dl[u], wa[u].z, r[2]); r[3] = fmaf(dl[u], wa[u].w, r[3]);
                    r[4] = fmaf(dl[u], wb[u].x, r[4]); r[5] = fmaf(dl[u], wb[u].y, r[5]);
                    r[6] = fmaf(dl[u], wb[u].z, r[6]); r[7] = fmaf(dl[u], wb[u].w, r[7]);
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = __fadd_rn(acc[i], r[i]);
        }
        if (on) {
            float4 *o = dx + ((int64_t)t * nchunk + c) * 2;
            __stcs(o, make_float4(acc[0], acc[1], acc[2], acc[3]));
            __stcs(o + 1, make_float4(acc[4], acc[5], acc[6], acc[7]));
        }
    }
}

inline int grid_for(int T) { return (T + kWarps - 1) / kWarps; }

// Launchers shared by the release and the checked entry points; arguments are
// checked by the callers.  status is the checked calls' status word (unused
// when CHECK is false).
template <bool CHECK>
moe_status launch_dispatch(const moe_shape *s, const moe_bf16 *x, const int32_t *route_row,
                           moe_bf16 *x_disp, int32_t *status, cudaStream_t stream) {
    launch_pdl(dispatch_rows<CHECK>, grid_for(s->T), kThreads, 0, stream, s->T, s->d / 8, s->K,
               reinterpret_cast<const uint4 *>(x), route_row, reinterpret_cast<uint4 *>(x_disp),
               buffer_rows(s), status);
    return launch_status();
}

template <bool CHECK>
moe_status launch_combine(const moe_shape *s, const moe_bf16 *y_disp, const int32_t *route_row,
                          const float *topk_gate, moe_bf16 *y, int32_t *status,
                          cudaStream_t stream) {
    auto *kern = s->K <= 8 ? combine_rows<8, CHECK> : combine_rows<16, CHECK>;
    launch_pdl(kern, grid_for(s->T), kThreads, 0, stream, s->T, s->d / 8, s->K,
               reinterpret_cast<const uint4 *>(y_disp), route_row, topk_gate,
               reinterpret_cast<uint4 *>(y), buffer_rows(s), status);
    return launch_status();
}

template <bool CHECK>
moe_status launch_combine_bwd(const moe_shape *s, const moe_bf16 *dy, const moe_bf16 *y_disp,
                              const int32_t *route_row, const float *topk_gate, moe_bf16 *dy_disp,
                              float *dgate, int32_t *status, cudaStream_t stream) {
    auto *kern = s->K <= 8 ? combine_bwd_rows<8, CHECK> : combine_bwd_rows<16, CHECK>;
    launch_pdl(kern, grid_for(s->T), kThreads, 0, stream, s->T, s->d / 8, s->K,
               reinterpret_cast<const uint4 *>(dy), reinterpret_cast<const uint4 *>(y_disp),
               route_row, topk_gate, reinterpret_cast<uint4 *>(dy_disp), dgate, buffer_rows(s),
               status);
    return launch_status();
}

template <bool CHECK>
moe_status launch_dispatch_bwd(const moe_shape *s, const moe_bf16 *dx_disp,
                               const int32_t *route_row, float *dx, int32_t *status,
                               cudaStream_t stream) {
    auto *kern = s->K <= 8 ? dispatch_bwd_rows<8, DBWD_PLAIN, CHECK>
                           : dispatch_bwd_rows<16, DBWD_PLAIN, CHECK>;
    launch_pdl(kern, grid_for(s->T), kThreads, 0, stream, s->T, s->d / 8, s->K, s->N,
               reinterpret_cast<const uint4 *>(dx_disp), route_row, reinterpret_cast<float4 *>(dx),
               nullptr, nullptr, nullptr, nullptr, nullptr, buffer_rows(s), status);
    return launch_status();
}

// The status word of a checked call: word 0 of a 256-byte-aligned workspace.
inline int32_t *status_word(void *status_ws) { return static_cast<int32_t *>(status_ws); }
inline bool status_ws_ok(const void *p) {
    return p && (reinterpret_cast<uintptr_t>(p) & 255u) == 0;
}

// ---- argument checks shared by the release and checked entry points -------

inline moe_status check_dispatch(const moe_shape *s, const moe_bf16 *x, const int32_t *route_row,
                                 const moe_bf16 *x_disp) {
    if (!x || !route_row || !x_disp) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(route_row) || !aligned16(x_disp)) return MOE_ERR_ALIGNMENT;
    return MOE_OK;
}

inline moe_status check_combine(const moe_shape *s, const moe_bf16 *y_disp,
                                const int32_t *route_row, const float *topk_gate,
                                const moe_bf16 *y) {
    if (!route_row || !topk_gate || !y || (s->cap > 0 && !y_disp)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(y_disp) || !aligned16(route_row) || !aligned16(topk_gate) || !aligned16(y))
        return MOE_ERR_ALIGNMENT;
    return MOE_OK;
}

inline moe_status check_combine_bwd(const moe_shape *s, const moe_bf16 *dy,
                                    const moe_bf16 *y_disp, const int32_t *route_row,
                                    const float *topk_gate, const moe_bf16 *dy_disp,
                                    const float *dgate) {
    if (!dy || !route_row || !topk_gate || !dgate || (s->cap > 0 && (!y_disp || !dy_disp)))
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(dy) || !aligned16(y_disp) || !aligned16(route_row) || !aligned16(topk_gate) ||
        !aligned16(dy_disp) || !aligned16(dgate))
        return MOE_ERR_ALIGNMENT;
    return MOE_OK;
}

inline moe_status check_dispatch_bwd(const moe_shape *s, const moe_bf16 *dx_disp,
                                     const int32_t *route_row, const float *dx) {
    if (!route_row || !dx || (s->cap > 0 && !dx_disp)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(dx_disp) || !aligned16(route_row) || !aligned16(dx)) return MOE_ERR_ALIGNMENT;
    return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

MOE_API moe_status moe_dispatch(const moe_shape *s, const moe_bf16 *x, const int32_t *route_row,
                                moe_bf16 *x_disp, cudaStream_t stream) {
    moe_status r = check_shape(s);
    if (r != MOE_OK) return r;
    if (s->T == 0 || s->cap == 0) return MOE_OK;  // no row can be written
    if ((r = check_dispatch(s, x, route_row, x_disp)) != MOE_OK) return r;
    return launch_dispatch<false>(s, x, route_row, x_disp, nullptr, stream);
}

MOE_API moe_status moe_combine(const moe_shape *s, const moe_bf16 *y_disp,
                               const int32_t *route_row, const float *topk_gate, moe_bf16 *y,
                               cudaStream_t stream) {
    moe_status r = check_shape(s);
    if (r != MOE_OK) return r;
    if (s->T == 0) return MOE_OK;
    if ((r = check_combine(s, y_disp, route_row, topk_gate, y)) != MOE_OK) return r;
    return launch_combine<false>(s, y_disp, route_row, topk_gate, y, nullptr, stream);
}

MOE_API moe_status moe_combine_backward(const moe_shape *s, const moe_bf16 *dy,
                                        const moe_bf16 *y_disp, const int32_t *route_row,
                                        const float *topk_gate, moe_bf16 *dy_disp, float *dgate,
                                        cudaStream_t stream) {
    moe_status r = check_shape(s);
    if (r != MOE_OK) return r;
    if (s->T == 0) return MOE_OK;
    if ((r = check_combine_bwd(s, dy, y_disp, route_row, topk_gate, dy_disp, dgate)) != MOE_OK)
        return r;
    return launch_combine_bwd<false>(s, dy, y_disp, route_row, topk_gate, dy_disp, dgate, nullptr,
                                     stream);
}

MOE_API moe_status moe_dispatch_backward(const moe_shape *s, const moe_bf16 *dx_disp,
                                         const int32_t *route_row, float *dx,
                                         cudaStream_t stream) {
    moe_status r = check_shape(s);
    if (r != MOE_OK) return r;
    if (s->T == 0) return MOE_OK;
    if ((r = check_dispatch_bwd(s, dx_disp, route_row, dx)) != MOE_OK) return r;
    return launch_dispatch_bwd<false>(s, dx_disp, route_row, dx, nullptr, stream);
}

// ---- checked variants: route rows validated on the device ------------------

MOE_API moe_status moe_dispatch_checked(const moe_shape *s, const moe_bf16 *x,
                                        const int32_t *route_row, moe_bf16 *x_disp,
                                        void *status_ws, cudaStream_t stream) {
    moe_status r = check_shape(s);
    if (r != MOE_OK) return r;
    if (!status_ws_ok(status_ws)) return MOE_ERR_WORKSPACE;
    if (s->T == 0 || s->cap == 0) return MOE_OK;
    if ((r = check_dispatch(s, x, route_row, x_disp)) != MOE_OK) return r;
    return launch_dispatch<true>(s, x, route_row, x_disp, status_word(status_ws), stream);
}

MOE_API moe_status moe_combine_checked(const moe_shape *s, const moe_bf16 *y_disp,
                                       const int32_t *route_row, const float *topk_gate,
                                       moe_bf16 *y, void *status_ws, cudaStream_t stream) {
    moe_status r = check_shape(s);
    if (r != MOE_OK) return r;
    if (!status_ws_ok(status_ws)) return MOE_ERR_WORKSPACE;
    if (s->T == 0) return MOE_OK;
    if ((r = check_combine(s, y_disp, route_row, topk_gate, y)) != MOE_OK) return r;
    return launch_combine<true>(s, y_disp, route_row, topk_gate, y, status_word(status_ws), stream);
}

MOE_API moe_status moe_combine_backward_checked(const moe_shape *s, const moe_bf16 *dy,
                                                const moe_bf16 *y_disp, const int32_t *route_row,
                                                const float *topk_gate, moe_bf16 *dy_disp,
                                                float *dgate, void *status_ws,
                                                cudaStream_t stream) {
    moe_status r = check_shape(s);
    if (r != MOE_OK) return r;
    if (!status_ws_ok(status_ws)) return MOE_ERR_WORKSPACE;
    if (s->T == 0) return MOE_OK;
    if ((r = check_combine_bwd(s, dy, y_disp, route_row, topk_gate, dy_disp, dgate)) != MOE_OK)
        return r;
    return launch_combine_bwd<true>(s, dy, y_disp, route_row, topk_gate, dy_disp, dgate,
                                    status_word(status_ws), stream);
}

MOE_API moe_status moe_dispatch_backward_checked(const moe_shape *s, const moe_bf16 *dx_disp,
                                                 const int32_t *route_row, float *dx,
                                                 void *status_ws, cudaStream_t stream) {
    moe_status r = check_shape(s);
    if (r != MOE_OK) return r;
    if (!status_ws_ok(status_ws)) return MOE_ERR_WORKSPACE;
    if (s->T == 0) return MOE_OK;
    if ((r = check_dispatch_bwd(s, dx_disp, route_row, dx)) != MOE_OK) return r;
    return launch_dispatch_bwd<true>(s, dx_disp, route_row, dx, status_word(status_ws), stream);
}

namespace moe {
// Router term of dx (and dlogit), alone (add = true: dx += ...) or fused into
// the dispatch backward (dx = dispatch sum + ...).  Arguments checked by the
// callers.
moe_status launch_router_dx(const moe_shape *s, const moe_bf16 *dx_disp, const int32_t *route_row,
                            const float *w_router, const int32_t *topk_idx,
                            const float *topk_gate, const float *dgate, float *dlogit, float *dx,
                            bool add, cudaStream_t stream) {
    using Fn = void (*)(int, int, int, int, const uint4 *, const int32_t *, float4 *,
                        const float4 *, const int32_t *, const float *, const float *, float *,
                        int64_t, int32_t *);
    Fn kern;
    if (add)
        kern = s->K <= 8 ? dispatch_bwd_rows<8, DBWD_ROUTER_ADD>
                         : dispatch_bwd_rows<16, DBWD_ROUTER_ADD>;
    else
        kern = s->K <= 8 ? dispatch_bwd_rows<8, DBWD_ROUTER> : dispatch_bwd_rows<16, DBWD_ROUTER>;
    launch_pdl(kern, grid_for(s->T), kThreads, 0, stream, s->T, s->d / 8, s->K, s->N,
               reinterpret_cast<const uint4 *>(dx_disp), route_row, reinterpret_cast<float4 *>(dx),
               reinterpret_cast<const float4 *>(w_router), topk_idx, topk_gate, dgate, dlogit,
               buffer_rows(s), static_cast<int32_t *>(nullptr));
    return launch_status();
}
}  // namespace moe

MOE_API moe_status moe_dispatch_router_backward(const moe_shape *s, const moe_bf16 *dx_disp,
                                                const int32_t *route_row, const float *w_router,
                                                const int32_t *topk_idx, const float *topk_gate,
                                                const float *dgate, float *dlogit, float *dx,
                                                cudaStream_t stream) {
    moe_status r = check_shape(s);
    if (r != MOE_OK) return r;
    if (s->T == 0) return MOE_OK;
    if (!route_row || !dx || (s->cap > 0 && !dx_disp) || !w_router || !topk_idx || !topk_gate ||
        !dgate || !dlogit)
        return MOE_ERR_INVALID_ARG;
    const void *ptrs[] = {dx_disp, route_row, dx, w_router, topk_idx, topk_gate, dgate, dlogit};
    for (const void *q : ptrs)
        if (!aligned16(q)) return MOE_ERR_ALIGNMENT;
    return launch_router_dx(s, dx_disp, route_row, w_router, topk_idx, topk_gate, dgate, dlogit,
                            dx, false, stream);
}
