// Routing: router logits, top-K and gates, fixed-capacity slots, route map.
//
// OLMo-core MoE report, "Section 05: Expert Parallelism", Figure 15 (K indices
// and K weights per token, larger first, summing to one), 5.4 and Figure 16
// (row = offset of the expert + number of earlier accepted routes to it; the
// capacity decision precedes any data movement; -1 marks a dropped route);
// "Section 08: Synchronization-Free Training", Table 14 (route map, counts and
// int32 cumulative offsets produced and kept on the device).  AWS Neuron
// "Expert Parallelism (EP)", "Router Weights" (logits for every expert).
//
// Four launches, none of which waits on another CTA:
//   1. route_logits_topk: per tile of tokens, fp32 logits for all experts in
//      shared memory (per 512-wide block of j one fused multiply-add chain
//      over j ascending, the block sums added in block order, so the values
//      are reproducible bit for bit), then one thread per token selects the
//      top K and computes the gates.
//   2. route_block_rank: per block of 256 tokens, a per-warp bitmask of the
//      tokens choosing each expert gives every route its rank among earlier
//      routes to the same expert inside the block, and the block's count per
//      expert.  Bitmask OR is order-free, so the ranks are deterministic.
//   3. route_scan: one CTA scans the per-block counts for every expert
//      (giving each block its base slot), clamps demand to capacity and scans
//      the counts into the cumulative offsets.
//   4. route_assign: slot = block base + rank; row = offset + slot, or -1 past
//      capacity.
#include <mutex>

#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int kRankBlock = 256;  // tokens per block of the slot ranking

__device__ __forceinline__ float canon(float v) { return isnan(v) ? -INFINITY : v; }

__device__ __forceinline__ bool beats(float a, int ia, float b, int ib) {
    return a > b || (a == b && ia < ib);
}

// Logit tile: WT x WE warps; a warp covers 16 tokens x 32 experts, each lane
// 4 tokens x 4 experts (16 independent fma chains, advanced in pairs by packed
// fp32x2 fma): lane = tx + 8 ty (tx in 0..7, ty in 0..3) owns tokens ty + 4a
// and experts tx + 8b of its warp's block.  A CTA covers TB = 16 WT tokens and
// EC = 32 WE experts per pass (passes loop over the experts).  The dot product
// over j is cut into 512-wide blocks: each chain restarts from 0 at a block
// boundary and the block sums are added in block order (the order the logits
// are defined by).  x (bf16) and W_r (fp32) stream through a 4-stage cp.async
// ring of 32-wide j-chunks in their natural row-major layouts; per 4 j a lane
// reads 8 bytes of each of its x rows and 16 bytes of each of its W rows (rows
// padded so that the 8 distinct rows of a warp load hit distinct banks).
constexpr int kLogitStages = 4;
constexpr int kLogitJC = 32;
constexpr int kLogitBlock = 512;  // j per block sum (a multiple of kLogitJC)

template <int WT, int WE>
struct LogitTile {
    static constexpr int THREADS = 32 * WT * WE;
    static constexpr int TB = 16 * WT;
    static constexpr int EC = 32 * WE;
    static constexpr int XR = kLogitJC + 8;  // bf16 per padded x row
    static constexpr int WR = kLogitJC + 4;  // fp32 per padded W row
    static constexpr int STAGE = TB * XR * 2 + EC * WR * 4;  // bytes
    static constexpr size_t smem_bytes(int N) {
        return (size_t)kLogitStages * STAGE + sizeof(float) * (size_t)TB * (N + 1);
    }
};

template <int WT, int WE>
__global__ void __launch_bounds__(LogitTile<WT, WE>::THREADS)
route_logits_topk(int T, int d, int N, int K, const uint16_t *__restrict__ x,
                  const float *__restrict__ w_r, const float *__restrict__ bias,
                  int32_t *__restrict__ topk_idx, float *__restrict__ topk_gate) {
    using L = LogitTile<WT, WE>;
    constexpr int TB = L::TB, EC = L::EC, XR = L::XR, WR = L::WR, JC = kLogitJC;
    constexpr int THREADS = L::THREADS;
    constexpr int CPB = kLogitBlock / JC;  // chunks per block
    extern __shared__ __align__(16) uint8_t smem_l[];
    const int LDS = N + 1;  // padded logit row: one thread per token reads its row
    float *lg = reinterpret_cast<float *>(smem_l + (size_t)kLogitStages * L::STAGE);  // [TB][LDS]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int tx = lane & 7, ty = lane >> 3;
    const int tok0 = (warp % WT) * 16 + ty;   // + 4a
    const int exp0 = (warp / WT) * 32 + tx;   // + 8b
    const int t0 = blockIdx.x * TB;
    const int nchunks = (d + JC - 1) / JC;

    for (int ec0 = 0; ec0 < N; ec0 += EC) {
        auto issue = [&](int c) {
            if (c < nchunks) {
                uint8_t *st = smem_l + (size_t)(c % kLogitStages) * L::STAGE;
                uint16_t *xs = reinterpret_cast<uint16_t *>(st);
                float *ws = reinterpret_cast<float *>(st + TB * XR * 2);
                const int j0 = c * JC, jn = min(JC, d - j0);
                for (int i = tid; i < TB * (JC / 8); i += THREADS) {
                    const int r = i / (JC / 8), q = (i % (JC / 8)) * 8;
                    if (t0 + r < T && q < jn)
                        cp_async16(xs + r * XR + q, x + (int64_t)(t0 + r) * d + j0 + q);
                }
                for (int i = tid; i < EC * (JC / 4); i += THREADS) {
                    const int r = i / (JC / 4), q = (i % (JC / 4)) * 4;
                    if (ec0 + r < N && q < jn)
                        cp_async16(ws + r * WR + q, w_r + (int64_t)(ec0 + r) * d + j0 + q);
                }
            }
            cp_async_commit();
        };

        // acc[ap][b] = the current block's chains (token 2ap, expert b) and
        // (token 2ap + 1, expert b), advanced together by one paired fma;
        // tot holds the sum of the finished blocks
        float2 acc[2][4], tot[2][4];
#pragma unroll
        for (int a = 0; a < 2; ++a)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                acc[a][q] = make_float2(0.0f, 0.0f);
                tot[a][q] = make_float2(0.0f, 0.0f);
            }
        auto fold = [&](bool first) {
#pragma unroll
            for (int a = 0; a < 2; ++a)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    tot[a][q] = first ? acc[a][q]
                                      : make_float2(__fadd_rn(tot[a][q].x, acc[a][q].x),
                                                    __fadd_rn(tot[a][q].y, acc[a][q].y));
                    acc[a][q] = make_float2(0.0f, 0.0f);
                }
        };

        __syncthreads();  // the previous pass is done with every stage
#pragma unroll
        for (int c = 0; c < kLogitStages - 1; ++c) issue(c);
        for (int c = 0; c < nchunks; ++c) {
            if (c > 0 && c % CPB == 0) fold(c == CPB);  // a block boundary
            cp_async_wait<kLogitStages - 2>();
            __syncthreads();
            issue(c + kLogitStages - 1);
            const uint8_t *st = smem_l + (size_t)(c % kLogitStages) * L::STAGE;
            const uint16_t *xs = reinterpret_cast<const uint16_t *>(st) + tok0 * XR;
            const float *ws = reinterpret_cast<const float *>(st + TB * XR * 2) + exp0 * WR;
            const int jn = min(JC, d - c * JC);  // a multiple of 8
#pragma unroll 4
            for (int j = 0; j < jn; j += 4) {
                // xp[ap][q] = (x of token 2ap, x of token 2ap + 1) at j + q
                float2 xp[2][4];
#pragma unroll
                for (int ap = 0; ap < 2; ++ap) {
                    const uint2 v0 = *reinterpret_cast<const uint2 *>(xs + 8 * ap * XR + j);
                    const uint2 v1 = *reinterpret_cast<const uint2 *>(xs + (8 * ap + 4) * XR + j);
                    xp[ap][0] = make_float2(bf16_lo(v0.x), bf16_lo(v1.x));
                    xp[ap][1] = make_float2(bf16_hi(v0.x), bf16_hi(v1.x));
                    xp[ap][2] = make_float2(bf16_lo(v0.y), bf16_lo(v1.y));
                    xp[ap][3] = make_float2(bf16_hi(v0.y), bf16_hi(v1.y));
                }
                float4 wf[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    wf[q] = *reinterpret_cast<const float4 *>(ws + 8 * q * WR + j);
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int eb = 0; eb < 4; ++eb) {
                        const float w = q == 0 ? wf[eb].x : q == 1 ? wf[eb].y : q == 2 ? wf[eb].z : wf[eb].w;
                        const float2 w2 = make_float2(w, w);
#pragma unroll
                        for (int ap = 0; ap < 2; ++ap) acc[ap][eb] = __ffma2_rn(xp[ap][q], w2, acc[ap][eb]);
                    }
            }
        }
        cp_async_wait<0>();
        fold(nchunks <= CPB);
#pragma unroll
        for (int eb = 0; eb < 4; ++eb) {
            const int e = ec0 + exp0 + 8 * eb;
            if (e < N) {
                const float bb = bias ? bias[e] : 0.0f;
#pragma unroll
                for (int ap = 0; ap < 2; ++ap) {
                    const float l0 = tot[ap][eb].x, l1 = tot[ap][eb].y;  // tokens 2ap, 2ap + 1
                    lg[(tok0 + 8 * ap) * LDS + e] = bias ? __fadd_rn(l0, bb) : l0;
                    lg[(tok0 + 8 * ap + 4) * LDS + e] = bias ? __fadd_rn(l1, bb) : l1;
                }
            }
        }
    }
    __syncthreads();

    // top-K and gates, one thread per token: the logits stream past a
    // sorted list of the best K so far (logit descending, lower expert first
    // on ties, NaN as -inf); a logit that beats the K-th is swapped down into
    // place.  The list sits at the end of a kMaxK-entry register array whose
    // first kMaxK - K entries hold sentinels that nothing beats, so the K-th
    // is always the last entry and every index is a constant.
    for (int tt = tid; tt < TB; tt += THREADS) {
        const int t = t0 + tt;
        if (t >= T) break;
        const float *l = lg + tt * LDS;
        const int first = kMaxK - K;
        float tv[kMaxK];
        int ti[kMaxK];
#pragma unroll
        for (int q = 0; q < kMaxK; ++q) {
            const bool real = q >= first;
            tv[q] = real ? -INFINITY : INFINITY;
            ti[q] = real ? 0x7FFFFFFF : -1;
        }
        for (int e = 0; e < N; ++e) {
            float v = canon(l[e]);
            if (!beats(v, e, tv[kMaxK - 1], ti[kMaxK - 1])) continue;
            int ie = e;
#pragma unroll
            for (int q = 0; q < kMaxK; ++q) {
                const bool sw = beats(v, ie, tv[q], ti[q]);
                const float sv = tv[q];
                const int si = ti[q];
                tv[q] = sw ? v : sv;
                ti[q] = sw ? ie : si;
                v = sw ? sv : v;
                ie = sw ? si : ie;
            }
        }
        float top = 0.0f;
#pragma unroll
        for (int q = 0; q < kMaxK; ++q)
            if (q == first) top = tv[q];
        float sum = 0.0f;
#pragma unroll
        for (int q = 0; q < kMaxK; ++q)
            if (q >= first) sum += (tv[q] == top) ? 1.0f : expf(tv[q] - top);
#pragma unroll
        for (int q = 0; q < kMaxK; ++q) {
            if (q >= first) {
                const float ex = (tv[q] == top) ? 1.0f : expf(tv[q] - top);
                topk_idx[(int64_t)t * K + (q - first)] = ti[q];
                topk_gate[(int64_t)t * K + (q - first)] = ex / sum;
            }
        }
    }
}

// Per block of 256 tokens: rank of each route among earlier routes of the
// block to the same expert (written to route_row for now) and the block's
// count per expert.
__global__ void __launch_bounds__(kRankBlock)
route_block_rank(int T, int N, int K, const int32_t *__restrict__ topk_idx,
                 int32_t *__restrict__ route_row, int32_t *__restrict__ block_count) {
    extern __shared__ uint32_t sm[];
    uint32_t *mask = sm;                       // [8][N]: bit lane of warp w chose e
    uint32_t *wpre = sm + (kRankBlock / 32) * N;  // [8][N]: routes to e in earlier warps
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < (kRankBlock / 32) * N; i += kRankBlock) mask[i] = 0;
    __syncthreads();
    const int t = blockIdx.x * kRankBlock + tid;
    int e_of[kMaxK];
    if (t < T) {
        for (int k = 0; k < K; ++k) {
            e_of[k] = topk_idx[(int64_t)t * K + k];
            atomicOr(&mask[warp * N + e_of[k]], 1u << lane);
        }
    }
    __syncthreads();
    for (int e = tid; e < N; e += kRankBlock) {
        uint32_t run = 0;
        for (int w = 0; w < kRankBlock / 32; ++w) {
            wpre[w * N + e] = run;
            run += __popc(mask[w * N + e]);
        }
        block_count[(int64_t)blockIdx.x * N + e] = (int32_t)run;
    }
    __syncthreads();
    if (t < T) {
        const uint32_t lt = (1u << lane) - 1u;
        for (int k = 0; k < K; ++k) {
            const int e = e_of[k];
            route_row[(int64_t)t * K + k] =
                (int32_t)(wpre[warp * N + e] + __popc(mask[warp * N + e] & lt));
        }
    }
}

// One CTA of 1024 threads: thread e turns the per-block counts of expert e
// into per-block base slots, then all threads scan the clamped counts.
__global__ void __launch_bounds__(1024)
route_scan(int nblk, int N, int cap, int32_t *__restrict__ block_count,
           int32_t *__restrict__ expert_count, int32_t *__restrict__ expert_offset,
           int32_t *__restrict__ expert_demand) {
    __shared__ int32_t warp_sum[32];
    const int e = threadIdx.x, lane = e & 31, warp = e >> 5;
    int32_t cnt = 0;
    if (e < N) {
        int32_t run = 0;
        int b = 0;
        for (; b + 8 <= nblk; b += 8) {
            int32_t c[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) c[q] = block_count[(int64_t)(b + q) * N + e];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                block_count[(int64_t)(b + q) * N + e] = run;
                run += c[q];
            }
        }
        for (; b < nblk; ++b) {
            const int32_t c = block_count[(int64_t)b * N + e];
            block_count[(int64_t)b * N + e] = run;
            run += c;
        }
        expert_demand[e] = run;
        cnt = min(run, cap);
        expert_count[e] = cnt;
    }
    // exclusive scan of cnt over e
    int32_t incl = cnt;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += v;
    }
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int32_t v = warp_sum[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t u = __shfl_up_sync(0xFFFFFFFFu, v, off);
            if (lane >= off) v += u;
        }
        warp_sum[lane] = v;  // inclusive over warps
    }
    __syncthreads();
    const int32_t base = warp > 0 ? warp_sum[warp - 1] : 0;
    if (e < N) expert_offset[e] = base + incl - cnt;
    if (e == N - 1) expert_offset[N] = base + incl;
}

__global__ void route_assign(int T, int N, int K, int cap, const int32_t *__restrict__ topk_idx,
                             const int32_t *__restrict__ block_base,
                             const int32_t *__restrict__ expert_offset,
                             int32_t *__restrict__ route_row) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)T * K) return;
    const int t = (int)(i / K);
    const int e = topk_idx[i];
    const int32_t slot = block_base[(int64_t)(t / kRankBlock) * N + e] + route_row[i];
    route_row[i] = slot < cap ? expert_offset[e] + slot : -1;
}

template <int WT, int WE>
moe_status launch_logits(const moe_shape *s, const uint16_t *x, const float *w, const float *b,
                         int32_t *idx, float *gate, cudaStream_t st) {
    using L = LogitTile<WT, WE>;
    const size_t smem = L::smem_bytes(s->N);
    static size_t configured = 0;
    if (smem > 48 * 1024 && smem > configured) {
        if (cudaFuncSetAttribute(route_logits_topk<WT, WE>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess)
            return MOE_ERR_CUDA;
        configured = smem;
    }
    const int grid = (s->T + L::TB - 1) / L::TB;
    route_logits_topk<WT, WE><<<grid, L::THREADS, smem, st>>>(s->T, s->d, s->N, s->K, x, w, b, idx,
                                                              gate);
    return launch_status();
}

}  // namespace

size_t route_ws_bytes(const moe_shape *s) {
    const size_t nblk = (size_t)(s->T + kRankBlock - 1) / kRankBlock;
    const size_t bc = (nblk * (size_t)s->N * sizeof(int32_t) + 255) & ~(size_t)255;
    return 256 + bc;
}

// Enqueues the four routing kernels; `status` is the device status word and
// `block_count` a [ceil(T/256), N] int32 scratch array.
moe_status route_enqueue(const moe_shape *s, const moe_bf16 *x, const float *w_router,
                         const float *bias, int32_t *topk_idx, float *topk_gate,
                         int32_t *route_row, int32_t *expert_count, int32_t *expert_offset,
                         int32_t *expert_demand, int32_t *block_count, cudaStream_t st) {
    const int nblk = (s->T + kRankBlock - 1) / kRankBlock;
    moe_status r = MOE_OK;
    if (s->T > 0) {
        const int n = s->N;
        if (n <= 32) r = launch_logits<2, 1>(s, x, w_router, bias, topk_idx, topk_gate, st);
        else if (n <= 64) r = launch_logits<2, 2>(s, x, w_router, bias, topk_idx, topk_gate, st);
        else r = launch_logits<2, 4>(s, x, w_router, bias, topk_idx, topk_gate, st);
        if (r != MOE_OK) return r;
        const size_t smem = sizeof(uint32_t) * 2 * (kRankBlock / 32) * (size_t)s->N;
        static bool configured = false;
        if (smem > 48 * 1024 && !configured) {
            if (cudaFuncSetAttribute(route_block_rank, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     2 * (kRankBlock / 32) * kMaxN * (int)sizeof(uint32_t)) !=
                cudaSuccess)
                return MOE_ERR_CUDA;
            configured = true;
        }
        route_block_rank<<<nblk, kRankBlock, smem, st>>>(s->T, s->N, s->K, topk_idx, route_row,
                                                          block_count);
        if ((r = launch_status()) != MOE_OK) return r;
    }
    route_scan<<<1, 1024, 0, st>>>(nblk, s->N, s->cap, block_count, expert_count, expert_offset,
                                   expert_demand);
    if ((r = launch_status()) != MOE_OK) return r;
    if (s->T > 0) {
        const int64_t routes = (int64_t)s->T * s->K;
        const int grid = (int)((routes + 255) / 256);
        route_assign<<<grid, 256, 0, st>>>(s->T, s->N, s->K, s->cap, topk_idx, block_count,
                                           expert_offset, route_row);
        r = launch_status();
    }
    return r;
}

}  // namespace moe

using namespace moe;

MOE_API size_t moe_route_workspace_bytes(const moe_shape *s) {
    if (check_shape(s) != MOE_OK) return 0;
    return route_ws_bytes(s);
}

MOE_API moe_status moe_route(const moe_shape *s, const moe_bf16 *x, const float *w_router,
                             const float *bias, int32_t *topk_idx, float *topk_gate,
                             int32_t *route_row, int32_t *expert_count, int32_t *expert_offset,
                             int32_t *expert_demand, void *ws, size_t ws_bytes,
                             cudaStream_t stream) {
    moe_status r = check_shape(s);
    if (r != MOE_OK) return r;
    if (!expert_count || !expert_offset || !expert_demand || !ws) return MOE_ERR_INVALID_ARG;
    if (s->T > 0 && (!x || !w_router || !topk_idx || !topk_gate || !route_row))
        return MOE_ERR_INVALID_ARG;
    if (ws_bytes < route_ws_bytes(s) || (reinterpret_cast<uintptr_t>(ws) & 255u))
        return MOE_ERR_WORKSPACE;
    if (!aligned16(x) || !aligned16(w_router) || !aligned16(topk_idx) || !aligned16(topk_gate) ||
        !aligned16(route_row) || !aligned16(expert_count) || !aligned16(expert_offset) ||
        !aligned16(expert_demand) || (bias && !aligned16(bias)))
        return MOE_ERR_ALIGNMENT;
    int32_t *block_count = reinterpret_cast<int32_t *>(static_cast<char *>(ws) + 256);
    return route_enqueue(s, x, w_router, bias, topk_idx, topk_gate, route_row, expert_count,
                         expert_offset, expert_demand, block_count, stream);
}

// ------------------------------------------------------------------------
// moe_route_noalloc: moe_route for callers that cannot allocate device memory.
//
// Its scratch (the device status word and the per-block count array) lives in
// the fixed array below instead of a caller-provided workspace.  Every GPU
// that loads this library holds the array until the process exits.  In host
// code `route_noalloc_scratch` names a host-side stand-in, not a device
// address, so the address each kernel gets is looked up once per device with
// cudaGetSymbolAddress (with that device current) on the first call there.
// All calls on a device share the array and it keeps the last call's
// contents; nothing in it needs clearing, because every entry a call reads
// is written earlier in the same call.  Calls that overlap on the GPU (for
// example on two streams) race on the array.
namespace moe {
namespace {

constexpr size_t kNoAllocScratchBytes = MOE_ROUTE_NOALLOC_SCRATCH_BYTES;
constexpr int kNoAllocMaxDevices = 64;

static __device__ __align__(256) uint8_t route_noalloc_scratch[kNoAllocScratchBytes];

std::mutex noalloc_mu;
void *noalloc_base[kNoAllocMaxDevices] = {};

// Device address of the scratch array on the current device (looked up once).
moe_status noalloc_scratch(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
    if (dev < 0 || dev >= kNoAllocMaxDevices) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(noalloc_mu);
    if (!noalloc_base[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, route_noalloc_scratch) != cudaSuccess || !p)
            return MOE_ERR_CUDA;
        noalloc_base[dev] = p;
    }
    *out = noalloc_base[dev];
    return MOE_OK;
}

}  // namespace
}  // namespace moe

MOE_API moe_status moe_route_noalloc(const moe_shape *s, const moe_bf16 *x, const float *w_router,
                                     const float *bias, int32_t *topk_idx, float *topk_gate,
                                     int32_t *route_row, int32_t *expert_count,
                                     int32_t *expert_offset, int32_t *expert_demand,
                                     cudaStream_t stream) {
    moe_status r = check_shape(s);
    if (r != MOE_OK) return r;
    if (!expert_count || !expert_offset || !expert_demand) return MOE_ERR_INVALID_ARG;
    if (s->T > 0 && (!x || !w_router || !topk_idx || !topk_gate || !route_row))
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w_router) || !aligned16(topk_idx) || !aligned16(topk_gate) ||
        !aligned16(route_row) || !aligned16(expert_count) || !aligned16(expert_offset) ||
        !aligned16(expert_demand) || (bias && !aligned16(bias)))
        return MOE_ERR_ALIGNMENT;
    if (route_ws_bytes(s) > kNoAllocScratchBytes) return MOE_ERR_UNSUPPORTED;
    void *base = nullptr;
    if ((r = noalloc_scratch(&base)) != MOE_OK) return r;
    int32_t *block_count = reinterpret_cast<int32_t *>(static_cast<char *>(base) + 256);
    return route_enqueue(s, x, w_router, bias, topk_idx, topk_gate, route_row, expert_count,
                         expert_offset, expert_demand, block_count, stream);
}
