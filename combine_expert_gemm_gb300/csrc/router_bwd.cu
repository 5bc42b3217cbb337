// Router backward: from the gate gradient to the router's input and weights.
//
// OLMo-core MoE report, "Section 05: Expert Parallelism", 5.6: the router-
// weight gradient starts from the gathered expert outputs and the token-output
// gradient of the accepted routes (dgate, written by the combine backward);
// Figure 15: the K gates of a token are a softmax over its K chosen logits.
// With the selection held fixed, for token t and its routes k:
//   dlogit[t,k] = g[t,k] * (dgate[t,k] - sum_k' g[t,k'] * dgate[t,k'])
//   dx[t,:]    += sum_k dlogit[t,k] * W_r[idx[t,k], :]
//   dW_r[e,:]   = sum over routes (t,k) with idx[t,k] = e of dlogit[t,k] * x[t,:]
//   dbias[e]    = sum over the same routes of dlogit[t,k]
// AWS Neuron "Expert Parallelism (EP)", "Router Weights": one replicated fp32
// router weight scores all N experts, so its gradient has the same [N, d].
//
// dlogit and the dx term are a per-token pass (rowwise.cu: alone, or fused
// into the dispatch backward, which walks the same token rows).  This file
// holds the weight gradient, fp32 on CUDA cores (the contraction is sparse:
// K of N experts per token) and deterministic (fixed summation orders, no
// floating-point atomics):
//   router_dw_tile one CTA per (token chunk, 256-column slab).  Each 128-token
//                  sub-chunk's x slab is staged in shared memory by cp.async
//                  while its routes are sorted by expert (stable counting
//                  sort: per-warp token bitmasks, popc ranks); each warp then
//                  sums whole experts in registers in token order (8 columns
//                  per lane, paired fp32 FMAs).  A chunk's partial dW_r /
//                  dbias goes to the workspace (straight to the output when
//                  there is one chunk).
//   router_dw_sum  sums the chunk partials in a fixed order.
#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int RB_TC = 128;       // tokens per sub-chunk (threads 0..127 own one each)
constexpr int RB_THREADS = 256;  // 8 warps
constexpr int RB_WARPS = RB_THREADS / 32;
constexpr int RB_TWARPS = RB_TC / 32;  // warps that own tokens
constexpr int RB_SLAB = 256;     // columns per CTA: 32 lanes x 8
constexpr int RB_CMAX = 32;      // CTAs along tokens; each strides over sub-chunks

struct RbSmem {
    // carved from dynamic shared memory; sizes depend on N and K
    uint16_t *xs;      // [RB_TC][RB_SLAB] bf16 slab of the sub-chunk's tokens
    uint32_t *mask;    // [RB_TWARPS][N] tokens of warp w (bits) routed to e
    int32_t *pre;      // [RB_TWARPS][N] routes to e in the token warps before w
    int32_t *cnt;      // [N] routes to e in the sub-chunk
    int32_t *start;    // [N + 32] exclusive scan of cnt (+ scan scratch)
    float *sdl;        // [RB_TC * K] dlogit of each sorted route
    float *tdl;        // [RB_TC * K] dlogit of route (t, k), token order
    uint16_t *list;    // [RB_TC * K] token (local) of each sorted route
    int16_t *sidx;     // [RB_TC * K] expert of route (t, k), token order (-1: skipped)
};

inline size_t rb_smem_bytes(int N, int K) {
    size_t b = (size_t)RB_TC * RB_SLAB * 2;
    b += (size_t)RB_TWARPS * N * 4 * 2;
    b += (size_t)N * 4 + (size_t)(N + 32) * 4;
    b += (size_t)RB_TC * K * (4 + 4 + 2 + 2);
    return (b + 15) & ~(size_t)15;
}

__device__ __forceinline__ RbSmem rb_carve(uint8_t *base, int N, int K) {
    RbSmem s;
    uint8_t *p = base;
    s.xs = reinterpret_cast<uint16_t *>(p); p += (size_t)RB_TC * RB_SLAB * 2;
    s.mask = reinterpret_cast<uint32_t *>(p); p += (size_t)RB_TWARPS * N * 4;
    s.pre = reinterpret_cast<int32_t *>(p); p += (size_t)RB_TWARPS * N * 4;
    s.cnt = reinterpret_cast<int32_t *>(p); p += (size_t)N * 4;
    s.start = reinterpret_cast<int32_t *>(p); p += (size_t)(N + 32) * 4;
    s.sdl = reinterpret_cast<float *>(p); p += (size_t)RB_TC * K * 4;
    s.tdl = reinterpret_cast<float *>(p); p += (size_t)RB_TC * K * 4;
    s.list = reinterpret_cast<uint16_t *>(p); p += (size_t)RB_TC * K * 2;
    s.sidx = reinterpret_cast<int16_t *>(p);
    return s;
}

// Exclusive scan of cnt[0..N) into start[0..N) by the whole block (N <= 1024:
// each thread owns up to 4 consecutive entries).  Uses start[N..N+32) as the
// per-warp scratch.  Ends with a __syncthreads().
__device__ __forceinline__ void rb_scan(const int32_t *cnt, int32_t *start, int N) {
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    int v[4], sum = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int e = tid * 4 + i;
        v[i] = e < N ? cnt[e] : 0;
        sum += v[i];
    }
    int inc = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xFFFFFFFFu, inc, o);
        if (lane >= o) inc += u;
    }
    int32_t *wsum = start + N;
    if (lane == 31) wsum[w] = inc;
    __syncthreads();
    int base = 0;
    for (int i = 0; i < w; ++i) base += wsum[i];
    int run = base + inc - sum;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int e = tid * 4 + i;
        if (e < N) start[e] = run;
        run += v[i];
    }
    __syncthreads();
}

// a += dl * (8 bf16 of xv), as four paired fp32 FMAs
__device__ __forceinline__ void fma8(float2 (&a)[4], float dl, const uint4 &xv) {
    const float2 d2 = make_float2(dl, dl);
    a[0] = __ffma2_rn(d2, make_float2(bf16_lo(xv.x), bf16_hi(xv.x)), a[0]);
    a[1] = __ffma2_rn(d2, make_float2(bf16_lo(xv.y), bf16_hi(xv.y)), a[1]);
    a[2] = __ffma2_rn(d2, make_float2(bf16_lo(xv.z), bf16_hi(xv.z)), a[2]);
    a[3] = __ffma2_rn(d2, make_float2(bf16_lo(xv.w), bf16_hi(xv.w)), a[3]);
}

__global__ void __launch_bounds__(RB_THREADS, 2)
router_dw_tile(int T, int d, int N, int K, int nchunk, const uint16_t *__restrict__ x,
               const int32_t *__restrict__ topk_idx, const float *__restrict__ dlogit,
               float *__restrict__ pdw, float *__restrict__ pdb) {
    pdl_enter();
    extern __shared__ __align__(16) uint8_t rb_smem[];
    const RbSmem s = rb_carve(rb_smem, N, K);
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int c = blockIdx.x;                 // chunk: sub-chunks c, c + nchunk, ...
    const int col0 = blockIdx.y * RB_SLAB;
    const int ncols = min(RB_SLAB, d - col0);  // multiple of 8
    const bool lane_on = lane * 8 < ncols;    // a lane's 8 columns are all in or all out
    float *my_dw = pdw + (size_t)c * N * d;   // this chunk's partial [N, d]
    float *my_db = pdb ? pdb + (size_t)c * N : nullptr;
    const int nsub = (T + RB_TC - 1) / RB_TC;

    for (int sub = c, it = 0; sub < nsub; sub += nchunk, ++it) {
        const int t0 = sub * RB_TC;
        const int tn = min(RB_TC, T - t0);

        // 1. stage x[t0 .. t0+tn, col0 .. col0+ncols) with 16-byte cp.async
        //    pieces; they land while the routes are sorted (steps 2-4)
        {
            const int per_row = ncols / 8;
            const int total = tn * per_row;
            for (int i = tid; i < total; i += RB_THREADS) {
                const int r = i / per_row, q = i - r * per_row;
                cp_async16(s.xs + r * RB_SLAB + q * 8, x + (int64_t)(t0 + r) * d + col0 + q * 8);
            }
            cp_async_commit();
        }
        for (int i = tid; i < RB_TWARPS * N; i += RB_THREADS) s.mask[i] = 0u;
        __syncthreads();

        // 2. routes of the sub-chunk: thread = token; per-warp token masks per expert
        if (tid < tn) {
            const int64_t base = (int64_t)(t0 + tid) * K;
            int ev[kMaxK];
            float dv[kMaxK];
#pragma unroll
            for (int k = 0; k < kMaxK; ++k)
                if (k < K) {
                    ev[k] = topk_idx[base + k];
                    dv[k] = dlogit[base + k];
                }
#pragma unroll
            for (int k = 0; k < kMaxK; ++k)
                if (k < K) {
                    const int e = ev[k];
                    const bool ok = e >= 0 && e < N;
                    s.sidx[tid * K + k] = ok ? (int16_t)e : (int16_t)-1;
                    s.tdl[tid * K + k] = dv[k];
                    if (ok) atomicOr(&s.mask[w * N + e], 1u << lane);
                }
        }
        __syncthreads();

        // 3. per expert: routes in each token warp and in the sub-chunk
        for (int e = tid; e < N; e += RB_THREADS) {
            int run = 0;
#pragma unroll
            for (int ww = 0; ww < RB_TWARPS; ++ww) {
                s.pre[ww * N + e] = run;
                run += __popc(s.mask[ww * N + e]);
            }
            s.cnt[e] = run;
        }
        __syncthreads();
        rb_scan(s.cnt, s.start, N);

        // 4. stable placement: routes of expert e in token order
        if (tid < tn) {
            const uint32_t lt = (1u << lane) - 1u;
            for (int k = 0; k < K; ++k) {
                const int e = s.sidx[tid * K + k];
                if (e < 0) continue;
                const int pos = s.start[e] + s.pre[w * N + e] + __popc(s.mask[w * N + e] & lt);
                s.list[pos] = (uint16_t)tid;
                s.sdl[pos] = s.tdl[tid * K + k];
            }
        }
        cp_async_wait<0>();
        __syncthreads();

        // 5. dW_r and dbias partials: warp w owns experts w, w + 8, ...
        for (int e = w; e < N; e += RB_WARPS) {
            const int j0 = s.start[e], j1 = j0 + s.cnt[e];
            if (it > 0 && j0 == j1) continue;
            float2 a[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
            float bsum = 0.f;
            int j = j0;
            for (; j + 4 <= j1; j += 4) {
                uint4 xv[4];
                float dl[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    dl[u] = s.sdl[j + u];
                    xv[u] = *reinterpret_cast<const uint4 *>(s.xs + s.list[j + u] * RB_SLAB + lane * 8);
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    fma8(a, dl[u], xv[u]);
                    bsum += dl[u];
                }
            }
            for (; j < j1; ++j) {
                const float dl = s.sdl[j];
                const uint4 xv = *reinterpret_cast<const uint4 *>(s.xs + s.list[j] * RB_SLAB + lane * 8);
                fma8(a, dl, xv);
                bsum += dl;
            }
            if (lane_on) {
                float4 *dst = reinterpret_cast<float4 *>(my_dw + (size_t)e * d + col0 + lane * 8);
                float4 lo = make_float4(a[0].x, a[0].y, a[1].x, a[1].y);
                float4 hi = make_float4(a[2].x, a[2].y, a[3].x, a[3].y);
                if (it > 0) {
                    const float4 p = dst[0], q = dst[1];
                    lo.x += p.x; lo.y += p.y; lo.z += p.z; lo.w += p.w;
                    hi.x += q.x; hi.y += q.y; hi.z += q.z; hi.w += q.w;
                }
                dst[0] = lo;
                dst[1] = hi;
            }
            if (my_db && blockIdx.y == 0 && lane == 0) my_db[e] = (it > 0 ? my_db[e] : 0.f) + bsum;
        }
        __syncthreads();
    }
}

// dw[e, j] = sum over chunks of pdw[c][e, j]; dbias likewise.  A block covers
// 32 float4 positions; its 8 warps each sum a fixed run of chunks (c = g,
// g + 8, ...) and warp 0 adds the 8 runs in order: a fixed order, with 8
// times the loads in flight of a thread-per-position loop.
constexpr int RS_GROUPS = 8;

__global__ void __launch_bounds__(32 * RS_GROUPS)
router_dw_sum(int64_t n4, int N, int nchunk, const float4 *__restrict__ pdw,
              const float *__restrict__ pdb, float4 *__restrict__ dw, float *__restrict__ dbias) {
    pdl_enter();
    __shared__ float4 part[RS_GROUPS][32];
    __shared__ float bpart[RS_GROUPS][32];
    const int lane = threadIdx.x & 31, g = threadIdx.x >> 5;
    const int64_t i = (int64_t)blockIdx.x * 32 + lane;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    float b = 0.f;
    if (i < n4) {
        int c = g;
        for (; c + 3 * RS_GROUPS < nchunk; c += 4 * RS_GROUPS) {
            float4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u] = __ldcs(pdw + (int64_t)(c + u * RS_GROUPS) * n4 + i);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                a.x += v[u].x; a.y += v[u].y; a.z += v[u].z; a.w += v[u].w;
            }
        }
        for (; c < nchunk; c += RS_GROUPS) {
            const float4 v = __ldcs(pdw + (int64_t)c * n4 + i);
            a.x += v.x; a.y += v.y; a.z += v.z; a.w += v.w;
        }
    }
    const bool bias_here = dbias && i < N;
    if (bias_here)
        for (int c = g; c < nchunk; c += RS_GROUPS) b += pdb[(int64_t)c * N + i];
    part[g][lane] = a;
    bpart[g][lane] = b;
    __syncthreads();
    if (g == 0) {
        float4 s4 = part[0][lane];
        float sb = bpart[0][lane];
#pragma unroll
        for (int q = 1; q < RS_GROUPS; ++q) {
            const float4 v = part[q][lane];
            s4.x += v.x; s4.y += v.y; s4.z += v.z; s4.w += v.w;
            sb += bpart[q][lane];
        }
        if (i < n4) dw[i] = s4;
        if (bias_here) dbias[i] = sb;
    }
}

inline int rb_chunks(int T) {
    const int nsub = (T + RB_TC - 1) / RB_TC;
    return nsub < RB_CMAX ? nsub : RB_CMAX;
}

moe_status launch_router_dw(const moe_shape *s, const moe_bf16 *x, const int32_t *topk_idx,
                            const float *dlogit, float *dw_router, float *dbias, void *ws,
                            cudaStream_t stream) {
    static PerDeviceOnce smem_attr;
    if (!device_once(smem_attr, [] { return set_smem_limit(router_dw_tile, 227 * 1024); }))
        return MOE_ERR_CUDA;
    const int C = rb_chunks(s->T);
    float *pdw = dw_router, *pdb = dbias;
    if (C > 1) {
        pdw = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + 256);
        pdb = dbias ? pdw + (size_t)C * s->N * s->d : nullptr;
    }
    const dim3 grid(C, (s->d + RB_SLAB - 1) / RB_SLAB);
    launch_pdl(router_dw_tile, grid, RB_THREADS, rb_smem_bytes(s->N, s->K), stream, s->T, s->d,
               s->N, s->K, C, x, topk_idx, dlogit, pdw, pdb);
    moe_status r = launch_status();
    if (r != MOE_OK || C == 1) return r;
    const int64_t n4 = (int64_t)s->N * s->d / 4;
    const int64_t blocks = (std::max<int64_t>(n4, s->N) + 31) / 32;
    launch_pdl(router_dw_sum, (unsigned)blocks, 32 * RS_GROUPS, 0, stream, n4, s->N, C,
               reinterpret_cast<const float4 *>(pdw), pdb, reinterpret_cast<float4 *>(dw_router),
               dbias);
    return launch_status();
}

// Checks shared by both entry points; T == 0 zero-fills the outputs.
moe_status router_dw_checks(const moe_shape *s, const void *x, const void *topk_idx,
                            const void *dlogit, float *dw_router, float *dbias, void *ws,
                            size_t ws_bytes);

}  // namespace
}  // namespace moe

using namespace moe;

MOE_API size_t moe_router_backward_workspace_bytes(const moe_shape *s) {
    if (check_shape(s) != MOE_OK) return 0;
    const int C = rb_chunks(s->T);
    if (C <= 1) return 256;
    return 256 + (size_t)C * s->N * s->d * 4 + (size_t)C * s->N * 4;
}

namespace moe {
namespace {
moe_status router_dw_checks(const moe_shape *s, const void *x, const void *topk_idx,
                            const void *dlogit, float *dw_router, float *dbias, void *ws,
                            size_t ws_bytes) {
    if (!dw_router || !ws) return MOE_ERR_INVALID_ARG;
    if (s->T > 0 && (!x || !topk_idx || !dlogit)) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < moe_router_backward_workspace_bytes(s) ||
        (reinterpret_cast<uintptr_t>(ws) & 255u))
        return MOE_ERR_WORKSPACE;
    const void *ptrs[] = {x, topk_idx, dlogit, dw_router, dbias};
    for (const void *q : ptrs)
        if (q && !aligned16(q)) return MOE_ERR_ALIGNMENT;
    if (rb_smem_bytes(s->N, s->K) > 227 * 1024) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

moe_status router_dw_zero(const moe_shape *s, float *dw_router, float *dbias, cudaStream_t stream) {
    if (cudaMemsetAsync(dw_router, 0, (size_t)s->N * s->d * 4, stream) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (dbias && cudaMemsetAsync(dbias, 0, (size_t)s->N * 4, stream) != cudaSuccess)
        return MOE_ERR_CUDA;
    return MOE_OK;
}
}  // namespace
}  // namespace moe

MOE_API moe_status moe_router_weight_backward(const moe_shape *s, const moe_bf16 *x,
                                              const int32_t *topk_idx, const float *dlogit,
                                              float *dw_router, float *dbias, void *ws,
                                              size_t ws_bytes, cudaStream_t stream) {
    moe_status r = check_shape(s);
    if (r != MOE_OK) return r;
    if ((r = router_dw_checks(s, x, topk_idx, dlogit, dw_router, dbias, ws, ws_bytes)) != MOE_OK)
        return r;
    if (s->T == 0) return router_dw_zero(s, dw_router, dbias, stream);
    return launch_router_dw(s, x, topk_idx, dlogit, dw_router, dbias, ws, stream);
}

MOE_API moe_status moe_router_backward(const moe_shape *s, const moe_bf16 *x,
                                       const float *w_router, const int32_t *topk_idx,
                                       const float *topk_gate, const float *dgate, float *dlogit,
                                       float *dx, float *dw_router, float *dbias, void *ws,
                                       size_t ws_bytes, cudaStream_t stream) {
    moe_status r = check_shape(s);
    if (r != MOE_OK) return r;
    if (!w_router) return MOE_ERR_INVALID_ARG;
    if (s->T > 0 && (!topk_gate || !dgate || !dx)) return MOE_ERR_INVALID_ARG;
    if ((r = router_dw_checks(s, x, topk_idx, dlogit, dw_router, dbias, ws, ws_bytes)) != MOE_OK)
        return r;
    const void *ptrs[] = {w_router, topk_gate, dgate, dx};
    for (const void *q : ptrs)
        if (q && !aligned16(q)) return MOE_ERR_ALIGNMENT;
    if (s->T == 0) return router_dw_zero(s, dw_router, dbias, stream);
    if ((r = launch_router_dx(s, nullptr, nullptr, w_router, topk_idx, topk_gate, dgate, dlogit, dx,
                              true, stream)) != MOE_OK)
        return r;
    return launch_router_dw(s, x, topk_idx, dlogit, dw_router, dbias, ws, stream);
}
