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
// Five launches; no CTA spins on another, and each kernel waits only for the
// grid before it (programmatic dependent launch):
//   1. route_logit_blocks: fp32 block sums of the logits (per 512-wide block
//      of j one fused multiply-add chain over j ascending), one CTA per
//      (token tile, block, group of 64 experts);
//   1b. route_topk: the block sums added in block order (+ bias), so the
//      logits are reproducible bit for bit; then four lanes per token select
//      the top K and compute the gates.
//   2. route_block_rank: per block of 256 tokens, a per-warp bitmask of the
//      tokens choosing each expert gives every route its rank among earlier
//      routes to the same expert inside the block, and the block's count per
//      expert.  Bitmask OR is order-free, so the ranks are deterministic.
//   3. route_scan: one CTA scans the per-block counts for every expert
//      (giving each block its base slot; up to 32 threads per expert, each
//      over a contiguous chunk of blocks), clamps demand to capacity and scans
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

// Router logits in two launches.
//
// route_logit_blocks: the dot product over j is cut into 512-wide blocks (one
// fp32 chain per block; the block sums are added in block order, the order
// the logits are defined by).  CTA (token tile, block b, pass z) computes
// the block sums of 128 tokens x the z-th group of EC experts and writes them
// to part[b][t][e]; the passes sit in the grid rather than in a loop, so that
// a layer with many experts gets many short CTAs instead of a second, nearly
// empty wave of long ones.  4 warps, each 32 tokens x EC experts; lane =
// tx + 8 ty (tx in 0..7, ty in 0..3) owns tokens ty + 4i (i = 0..7) and
// experts tx + 8b (b < EPL): 8 EPL chains, advanced two tokens at a time by
// the packed fp32x2 fma; the j loop over a chunk is unrolled four ways.
// EPL = 8 (64 experts per pass) when N > 32, else 4: each widened pair of x
// values then feeds 8 paired fmas instead of 4, which halves the conversion
// and register-move instructions per fma (they, not memory, bound the loop).
// x (bf16) and W_r (fp32) stream through a 3-stage cp.async ring of 32-wide
// j-chunks in their natural layouts (rows padded so that a warp load's
// distinct rows hit distinct banks).  Splitting j into blocks gives 4 times
// the warps of a single chain per logit.
//
constexpr int kLogitJC = 32;
constexpr int kLogitBlock = 512;  // j per block sum (a multiple of kLogitJC)
constexpr int kLogitStages = 3;
constexpr int kLogitThreads = 128;
constexpr int kLogitXR = kLogitJC + 8;  // bf16 per padded x row
constexpr int kLogitWR = kLogitJC + 4;  // fp32 per padded W row

// WE warps along the experts, 4 / WE along the tokens; EPL experts per lane:
// 128 tokens x 64 experts per pass (EPL = 8), or 128 x 32 (EPL = 4) for
// N <= 32
template <int WE, int EPL = 4>
struct LogitTile {
    static constexpr int WT = 4 / WE;
    static constexpr int TB = 32 * WT;
    static constexpr int EC = 8 * EPL * WE;
    static constexpr int STAGE = TB * kLogitXR * 2 + EC * kLogitWR * 4;
    static constexpr size_t SMEM = (size_t)kLogitStages * STAGE;
};

inline int logit_blocks(int d) { return (d + kLogitBlock - 1) / kLogitBlock; }

template <int WE, int EPL>
__global__ void __launch_bounds__(kLogitThreads)
route_logit_blocks(int T, int d, int N, const uint16_t *__restrict__ x,
                   const float *__restrict__ w_r, float *__restrict__ part) {
    pdl_enter();
    using L = LogitTile<WE, EPL>;
    constexpr int JC = kLogitJC, XR = kLogitXR, WR = kLogitWR, TB = L::TB, EC = L::EC;
    constexpr int kLogitStage = L::STAGE;
    extern __shared__ __align__(16) uint8_t smem_l[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int tx = lane & 7, ty = lane >> 3;
    const int tok0 = (warp % L::WT) * 32 + ty;   // + 4i
    const int exp0 = (warp / L::WT) * (8 * EPL) + tx;   // + 8b
    const int t0 = blockIdx.x * TB;
    const int b = blockIdx.y;
    const int jb0 = b * kLogitBlock, jlen = min(kLogitBlock, d - jb0);  // a multiple of 8
    const int nchunks = (jlen + JC - 1) / JC;
    float *pb = part + (size_t)b * T * N;

    for (int ec0 = blockIdx.z * EC; ec0 < N; ec0 += EC * (int)gridDim.z) {
        auto issue = [&](int c) {
            if (c < nchunks) {
                uint8_t *st = smem_l + (size_t)(c % kLogitStages) * kLogitStage;
                uint16_t *xs = reinterpret_cast<uint16_t *>(st);
                float *ws = reinterpret_cast<float *>(st + TB * XR * 2);
                const int j0 = jb0 + c * JC, jn = min(JC, jlen - c * JC);
                for (int i = tid; i < TB * (JC / 8); i += kLogitThreads) {
                    const int r = i / (JC / 8), q = (i % (JC / 8)) * 8;
                    if (t0 + r < T && q < jn)
                        cp_async16(xs + r * XR + q, x + (int64_t)(t0 + r) * d + j0 + q);
                }
                for (int i = tid; i < EC * (JC / 4); i += kLogitThreads) {
                    const int r = i / (JC / 4), q = (i % (JC / 4)) * 4;
                    if (ec0 + r < N && q < jn)
                        cp_async16(ws + r * WR + q, w_r + (int64_t)(ec0 + r) * d + j0 + q);
                }
            }
            cp_async_commit();
        };

        // acc[p][e]: chains (token tok0 + 8p, expert e) and (token tok0 + 8p + 4,
        // expert e) of this lane, e = exp0 + 8 * (0..3)
        float2 acc[4][EPL];
#pragma unroll
        for (int p = 0; p < 4; ++p)
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[p][e] = make_float2(0.0f, 0.0f);

        __syncthreads();  // the previous pass is done with every stage
#pragma unroll
        for (int c = 0; c < kLogitStages - 1; ++c) issue(c);
        for (int c = 0; c < nchunks; ++c) {
            cp_async_wait<kLogitStages - 2>();
            __syncthreads();
            issue(c + kLogitStages - 1);
            const uint8_t *st = smem_l + (size_t)(c % kLogitStages) * kLogitStage;
            const uint16_t *xs = reinterpret_cast<const uint16_t *>(st) + tok0 * XR;
            const float *ws = reinterpret_cast<const float *>(st + TB * XR * 2) + exp0 * WR;
            const int jn = min(JC, jlen - c * JC);  // a multiple of 8
#pragma unroll 4
            for (int j = 0; j < jn; j += 4) {
                uint2 xv[8];  // tokens tok0 + 4i, 4 bf16 at j .. j + 3
#pragma unroll
                for (int i = 0; i < 8; ++i) xv[i] = *reinterpret_cast<const uint2 *>(xs + 4 * i * XR + j);
                float4 wv[EPL];
#pragma unroll
                for (int e = 0; e < EPL; ++e) wv[e] = *reinterpret_cast<const float4 *>(ws + 8 * e * WR + j);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
#pragma unroll
                    for (int p = 0; p < 4; ++p) {
                        const uint32_t a = (q < 2) ? xv[2 * p].x : xv[2 * p].y;
                        const uint32_t bb = (q < 2) ? xv[2 * p + 1].x : xv[2 * p + 1].y;
                        const float2 xp = (q & 1) ? make_float2(bf16_hi(a), bf16_hi(bb))
                                                  : make_float2(bf16_lo(a), bf16_lo(bb));
#pragma unroll
                        for (int e = 0; e < EPL; ++e) {
                            const float w = q == 0 ? wv[e].x : q == 1 ? wv[e].y : q == 2 ? wv[e].z : wv[e].w;
                            acc[p][e] = __ffma2_rn(xp, make_float2(w, w), acc[p][e]);
                        }
                    }
                }
            }
        }
        cp_async_wait<0>();
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const int ta = t0 + tok0 + 8 * p, tb = ta + 4;
#pragma unroll
            for (int e = 0; e < EPL; ++e) {
                const int ex = ec0 + exp0 + 8 * e;
                if (ex >= N) continue;
                if (ta < T) pb[(int64_t)ta * N + ex] = acc[p][e].x;
                if (tb < T) pb[(int64_t)tb * N + ex] = acc[p][e].y;
            }
        }
    }
}

constexpr int kTopkTB = 8;      // tokens per CTA (one warp)
constexpr int kTopkPlanes = 4;  // block-sum planes loaded before any is added
constexpr int kTopkGroups = 4;  // float4 groups per lane loaded before any is added

// Shared-memory row stride of the logits: at least N + 1 and 4 mod 32, so the
// 32 lanes of a selecting warp (8 tokens x 4 lanes, lane s reading expert
// s + 4i) fall on 32 distinct banks.
__host__ __device__ constexpr int topk_row_stride(int N) {
    return N + 1 + (4 - (N + 1) % 32 + 32) % 32;
}

// Sorts M (value, index) pairs best first (logit descending, lower expert
// first on ties) with a bitonic network: the compare-exchanges of a stage are
// independent, and every index is a constant.
template <int M>
__device__ __forceinline__ void topk_sort(float (&v)[M], int (&ix)[M]) {
#pragma unroll
    for (int k = 2; k <= M; k <<= 1) {
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
#pragma unroll
            for (int i = 0; i < M; ++i) {
                const int l = i ^ j;
                if (l <= i) continue;
                const bool sw = (i & k) == 0 ? beats(v[l], ix[l], v[i], ix[i])
                                             : beats(v[i], ix[i], v[l], ix[l]);
                const float a = v[i], b = v[l];
                const int ia = ix[i], ib = ix[l];
                v[i] = sw ? b : a;
                ix[i] = sw ? ib : ia;
                v[l] = sw ? a : b;
                ix[l] = sw ? ia : ib;
            }
        }
    }
}

// Replaces the sorted list (tv, ti) by the best M of its union with the
// sorted list (pv, pi): the better of entry q and entry M - 1 - q of the other
// list holds the best M of the union as a bitonic sequence, which the bitonic
// merge network then sorts.
template <int M>
__device__ __forceinline__ void topk_merge_list(float (&tv)[M], int (&ti)[M], const float (&pv)[M],
                                                const int (&pi)[M]) {
#pragma unroll
    for (int q = 0; q < M; ++q) {
        const bool take = beats(pv[M - 1 - q], pi[M - 1 - q], tv[q], ti[q]);
        tv[q] = take ? pv[M - 1 - q] : tv[q];
        ti[q] = take ? pi[M - 1 - q] : ti[q];
    }
#pragma unroll
    for (int s = M / 2; s > 0; s >>= 1) {
#pragma unroll
        for (int q = 0; q < M; ++q) {
            if (q & s) continue;
            const bool sw = beats(tv[q + s], ti[q + s], tv[q], ti[q]);
            const float a = tv[q], b = tv[q + s];
            const int ia = ti[q], ib = ti[q + s];
            tv[q] = sw ? b : a;
            ti[q] = sw ? ib : ia;
            tv[q + s] = sw ? a : b;
            ti[q + s] = sw ? ia : ib;
        }
    }
}

// The same with the list of lane ^ mask (both lanes end with the same list).
template <int M>
__device__ __forceinline__ void topk_merge(float (&tv)[M], int (&ti)[M], int mask) {
    float pv[M];
    int pi[M];
#pragma unroll
    for (int q = 0; q < M; ++q) {
        pv[q] = __shfl_xor_sync(0xFFFFFFFFu, tv[q], mask);
        pi[q] = __shfl_xor_sync(0xFFFFFFFFu, ti[q], mask);
    }
    topk_merge_list(tv, ti, pv, pi);
}

// route_topk: one CTA of one warp per 8 tokens (many small CTAs spread evenly
// over the SMs).  The block sums of the tile are contiguous in each block's
// [T][N] plane; every lane loads kTopkGroups float4 groups from kTopkPlanes
// planes before adding any of them (one memory round trip for d <= 2048),
// then adds them in block order (+ bias) into shared memory.  Selection: 4 lanes per token, lane
// s keeping the best MAXK of experts s, s + 4, s + 8, ... (logit descending,
// lower expert first on ties, NaN as -inf; unfilled entries are -inf with an
// index past every expert, so any expert beats them).  The lane takes its
// experts MAXK at a time, sorts them with a bitonic network and merges them
// into its list, so no step waits on a data-dependent branch; two merges over
// lane shuffles then give all four lanes the best MAXK of the token, whose
// first K are the top K.  The order is strict and total, so the result does not depend on
// how the experts were split.  Gates: softmax over the K, shifted by the
// largest, summed over k ascending.
template <int MAXK>
__global__ void __launch_bounds__(32)
route_topk(int T, int N, int K, int nb, const float *__restrict__ part,
           const float *__restrict__ bias, int32_t *__restrict__ topk_idx,
           float *__restrict__ topk_gate) {
    pdl_enter();
    extern __shared__ __align__(16) uint8_t smem_t[];
    const int LDS = topk_row_stride(N);
    float *lg = reinterpret_cast<float *>(smem_t);  // [kTopkTB][LDS]
    const int tid = threadIdx.x;
    const int t0 = blockIdx.x * kTopkTB;
    const int tn = min(kTopkTB, T - t0);
    const int64_t tile = (int64_t)t0 * N, n = (int64_t)tn * N;
    const int64_t plane = (int64_t)T * N;
    if ((N & 3) == 0) {
        // kTopkGroups groups x kTopkPlanes planes in flight per lane
        for (int64_t g0 = tid; g0 < n / 4; g0 += kTopkGroups * blockDim.x) {
            float4 v[kTopkGroups][kTopkPlanes];
#pragma unroll
            for (int u = 0; u < kTopkGroups; ++u) {
                const int64_t g = g0 + u * blockDim.x;
#pragma unroll
                for (int c = 0; c < kTopkPlanes; ++c)
                    if (g < n / 4 && c < nb)
                        v[u][c] = __ldcs(reinterpret_cast<const float4 *>(part + c * plane + tile) + g);
            }
#pragma unroll
            for (int u = 0; u < kTopkGroups; ++u) {
                const int64_t g = g0 + u * blockDim.x;
                if (g >= n / 4) continue;
                float4 a = v[u][0];
#pragma unroll
                for (int c = 1; c < kTopkPlanes; ++c) {
                    if (c >= nb) break;
                    a.x = __fadd_rn(a.x, v[u][c].x);
                    a.y = __fadd_rn(a.y, v[u][c].y);
                    a.z = __fadd_rn(a.z, v[u][c].z);
                    a.w = __fadd_rn(a.w, v[u][c].w);
                }
                for (int c = kTopkPlanes; c < nb; ++c) {  // d > 2048
                    const float4 w = __ldcs(reinterpret_cast<const float4 *>(part + c * plane + tile) + g);
                    a.x = __fadd_rn(a.x, w.x);
                    a.y = __fadd_rn(a.y, w.y);
                    a.z = __fadd_rn(a.z, w.z);
                    a.w = __fadd_rn(a.w, w.w);
                }
                const float vv[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const int i = (int)(4 * g + h), tt = i / N, e = i - tt * N;
                    lg[tt * LDS + e] = bias ? __fadd_rn(vv[h], bias[e]) : vv[h];
                }
            }
        }
    } else {
        for (int i = tid; i < n; i += blockDim.x) {
            const int tt = i / N, e = i - tt * N;
            float v = part[tile + i];
            for (int b = 1; b < nb; ++b) v = __fadd_rn(v, part[b * plane + tile + i]);
            if (bias) v = __fadd_rn(v, bias[e]);
            lg[tt * LDS + e] = v;
        }
    }
    __syncthreads();

    const int lane = tid & 31, sub = lane & 3;
    const int tt = lane >> 2;
    const int nloc = tt < tn ? N : 0;  // lanes past the tile only join the shuffles
    const float *l = lg + tt * LDS;
    float tv[MAXK];
    int ti[MAXK];
#pragma unroll
    for (int q = 0; q < MAXK; ++q) {
        tv[q] = -INFINITY;
        ti[q] = 0x7FFFFFFF;
    }
    // this lane's experts sub + 4i, i < nper, in blocks of MAXK
    const int nper = nloc > sub ? (nloc - sub + 3) / 4 : 0;
    for (int i0 = 0; i0 < nper; i0 += MAXK) {
        float bv[MAXK];
        int bi[MAXK];
#pragma unroll
        for (int u = 0; u < MAXK; ++u) {
            const bool ok = i0 + u < nper;
            const int e = sub + 4 * (i0 + u);
            const float raw = l[ok ? e : 0];
            bv[u] = ok ? canon(raw) : -INFINITY;
            bi[u] = ok ? e : 0x7FFFFFFF;
        }
        topk_sort(bv, bi);
        if (i0 == 0) {
#pragma unroll
            for (int q = 0; q < MAXK; ++q) {
                tv[q] = bv[q];
                ti[q] = bi[q];
            }
        } else {
            topk_merge_list(tv, ti, bv, bi);
        }
    }
    topk_merge(tv, ti, 1);
    topk_merge(tv, ti, 2);
    if (nloc == 0) return;
    const int t = t0 + tt;
    const float top = tv[0];
    float sum = 0.0f;
#pragma unroll
    for (int q = 0; q < MAXK; ++q)
        if (q < K) sum += (tv[q] == top) ? 1.0f : expf(tv[q] - top);
#pragma unroll
    for (int q = 0; q < MAXK; ++q) {
        if (q < K && (q & 3) == sub) {
            const float ex = (tv[q] == top) ? 1.0f : expf(tv[q] - top);
            topk_idx[(int64_t)t * K + q] = ti[q];
            topk_gate[(int64_t)t * K + q] = ex / sum;
        }
    }
}

// Per block of 256 tokens: rank of each route among earlier routes of the
// block to the same expert (written to route_row for now) and the block's
// count per expert.
__global__ void __launch_bounds__(kRankBlock)
route_block_rank(int T, int N, int K, const int32_t *__restrict__ topk_idx,
                 int32_t *__restrict__ route_row, int32_t *__restrict__ block_count) {
    pdl_enter();
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

// Sums the counts of blocks [b0, b1) of expert e.
__device__ __forceinline__ int32_t block_count_sum(const int32_t *__restrict__ block_count,
                                                   int N, int e, int b0, int b1) {
    int32_t s = 0;
    int b = b0;
    for (; b + 8 <= b1; b += 8) {
        int32_t c[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) c[q] = block_count[(int64_t)(b + q) * N + e];
#pragma unroll
        for (int q = 0; q < 8; ++q) s += c[q];
    }
    for (; b < b1; ++b) s += block_count[(int64_t)b * N + e];
    return s;
}

// Threads per expert in route_scan: at most 32, at most 1024 / N, and at
// least 4 blocks for each.
__host__ __device__ inline int scan_lanes_per_expert(int nblk, int N) {
    return max(1, min(min(32, kMaxN / N), nblk / 4));
}

// One CTA of 1024 threads.  Thread p * N + e (p < P, P threads per expert)
// owns the contiguous chunk p of the per-block counts of expert e: it sums
// its chunk, adds the sums of the chunks before it (in chunk order), and
// rewrites its chunk's counts as base slots.  Every count is read in two
// rounds of loads whatever the number of blocks, instead of one round per 8
// blocks.  Then threads 0..N-1 scan the clamped counts over the experts.
__global__ void __launch_bounds__(1024)
route_scan(int nblk, int N, int cap, int32_t *__restrict__ block_count,
           int32_t *__restrict__ expert_count, int32_t *__restrict__ expert_offset,
           int32_t *__restrict__ expert_demand) {
    pdl_enter();
    __shared__ int32_t warp_sum[32];
    __shared__ int32_t chunk_sum[kMaxN];  // [P][N]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int P = scan_lanes_per_expert(nblk, N);
    const int chunk = (nblk + P - 1) / P;
    const int p = tid / N, e = tid % N;
    const int b0 = min(p * chunk, nblk), b1 = min(b0 + chunk, nblk);
    if (p < P) chunk_sum[tid] = block_count_sum(block_count, N, e, b0, b1);
    __syncthreads();
    if (p < P) {
        int32_t run = 0;
        for (int q = 0; q < p; ++q) run += chunk_sum[q * N + e];
        int b = b0;
        for (; b + 8 <= b1; b += 8) {
            int32_t c[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) c[q] = block_count[(int64_t)(b + q) * N + e];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                block_count[(int64_t)(b + q) * N + e] = run;
                run += c[q];
            }
        }
        for (; b < b1; ++b) {
            const int32_t c = block_count[(int64_t)b * N + e];
            block_count[(int64_t)b * N + e] = run;
            run += c;
        }
    }
    int32_t cnt = 0;
    if (tid < N) {
        int32_t demand = 0;
        for (int q = 0; q < P; ++q) demand += chunk_sum[q * N + tid];
        expert_demand[tid] = demand;
        cnt = min(demand, cap);
        expert_count[tid] = cnt;
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
    if (tid < N) expert_offset[tid] = base + incl - cnt;
    if (tid == N - 1) expert_offset[N] = base + incl;
}

__global__ void route_assign(int T, int N, int K, int cap, const int32_t *__restrict__ topk_idx,
                             const int32_t *__restrict__ block_base,
                             const int32_t *__restrict__ expert_offset,
                             int32_t *__restrict__ route_row) {
    pdl_enter();
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (int64_t)T * K) return;
    const int t = (int)(i / K);
    const int e = topk_idx[i];
    const int32_t slot = block_base[(int64_t)(t / kRankBlock) * N + e] + route_row[i];
    route_row[i] = slot < cap ? expert_offset[e] + slot : -1;
}

moe_status launch_logits(const moe_shape *s, const uint16_t *x, const float *w, const float *b,
                         int32_t *idx, float *gate, float *part, cudaStream_t st) {
    static PerDeviceOnce smem_attr;
    if (!device_once(smem_attr, [] {
            const size_t topk_smem = sizeof(float) * kTopkTB * topk_row_stride(kMaxN);
            return set_smem_limit(route_logit_blocks<1, 4>, LogitTile<1, 4>::SMEM) &&
                   set_smem_limit(route_logit_blocks<1, 8>, LogitTile<1, 8>::SMEM) &&
                   set_smem_limit(route_topk<8>, topk_smem) &&
                   set_smem_limit(route_topk<kMaxK>, topk_smem);
        }))
        return MOE_ERR_CUDA;
    const int nb = logit_blocks(s->d);
    if (s->N <= 32) {
        const dim3 grid((s->T + LogitTile<1, 4>::TB - 1) / LogitTile<1, 4>::TB, nb,
                        (s->N + LogitTile<1, 4>::EC - 1) / LogitTile<1, 4>::EC);
        launch_pdl(route_logit_blocks<1, 4>, grid, kLogitThreads, LogitTile<1, 4>::SMEM, st, s->T,
                   s->d, s->N, x, w, part);
    } else {
        const dim3 grid((s->T + LogitTile<1, 8>::TB - 1) / LogitTile<1, 8>::TB, nb,
                        (s->N + LogitTile<1, 8>::EC - 1) / LogitTile<1, 8>::EC);
        launch_pdl(route_logit_blocks<1, 8>, grid, kLogitThreads, LogitTile<1, 8>::SMEM, st, s->T,
                   s->d, s->N, x, w, part);
    }
    moe_status r = launch_status();
    if (r != MOE_OK) return r;
    const size_t tsmem = sizeof(float) * kTopkTB * topk_row_stride(s->N);
    auto *topk = s->K <= 8 ? route_topk<8> : route_topk<kMaxK>;
    launch_pdl(topk, (s->T + kTopkTB - 1) / kTopkTB, 32, tsmem, st, s->T, s->N, s->K, nb, part, b,
               idx, gate);
    return launch_status();
}

}  // namespace

inline size_t route_block_count_bytes(const moe_shape *s) {
    const size_t nblk = (size_t)(s->T + kRankBlock - 1) / kRankBlock;
    return (nblk * (size_t)s->N * sizeof(int32_t) + 255) & ~(size_t)255;
}

// status word (256 B), the per-block count array, then the logit block sums
// [ceil(d / 512)][T][N] fp32
size_t route_ws_bytes(const moe_shape *s) {
    const size_t part = (size_t)logit_blocks(s->d) * s->T * s->N * sizeof(float);
    return 256 + route_block_count_bytes(s) + ((part + 255) & ~(size_t)255);
}

// Enqueues the routing kernels; `scratch` is the workspace past its status
// word (route_ws_bytes(s) - 256 bytes).
moe_status route_enqueue(const moe_shape *s, const moe_bf16 *x, const float *w_router,
                         const float *bias, int32_t *topk_idx, float *topk_gate,
                         int32_t *route_row, int32_t *expert_count, int32_t *expert_offset,
                         int32_t *expert_demand, void *scratch, cudaStream_t st) {
    const int nblk = (s->T + kRankBlock - 1) / kRankBlock;
    int32_t *block_count = static_cast<int32_t *>(scratch);
    float *part = reinterpret_cast<float *>(static_cast<char *>(scratch) + route_block_count_bytes(s));
    moe_status r = MOE_OK;
    if (s->T > 0) {
        r = launch_logits(s, x, w_router, bias, topk_idx, topk_gate, part, st);
        if (r != MOE_OK) return r;
        const size_t smem = sizeof(uint32_t) * 2 * (kRankBlock / 32) * (size_t)s->N;
        static PerDeviceOnce smem_attr;
        if (smem > 48 * 1024 && !device_once(smem_attr, [] {
                return set_smem_limit(route_block_rank,
                                      2 * (kRankBlock / 32) * kMaxN * sizeof(uint32_t));
            }))
            return MOE_ERR_CUDA;
        launch_pdl(route_block_rank, nblk, kRankBlock, smem, st, s->T, s->N, s->K, topk_idx,
                   route_row, block_count);
        if ((r = launch_status()) != MOE_OK) return r;
    }
    launch_pdl(route_scan, 1, 1024, 0, st, nblk, s->N, s->cap, block_count, expert_count,
               expert_offset, expert_demand);
    if ((r = launch_status()) != MOE_OK) return r;
    if (s->T > 0) {
        const int64_t routes = (int64_t)s->T * s->K;
        const int grid = (int)((routes + 255) / 256);
        launch_pdl(route_assign, grid, 256, 0, st, s->T, s->N, s->K, s->cap, topk_idx, block_count,
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
    return route_enqueue(s, x, w_router, bias, topk_idx, topk_gate, route_row, expert_count,
                         expert_offset, expert_demand, static_cast<char *>(ws) + 256, stream);
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
    return route_enqueue(s, x, w_router, bias, topk_idx, topk_gate, route_row, expert_count,
                         expert_offset, expert_demand, static_cast<char *>(base) + 256, stream);
}
