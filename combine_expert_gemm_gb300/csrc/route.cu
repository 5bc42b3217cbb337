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
// Six launches; no CTA spins on another, and each kernel waits only for the
// grid before it (programmatic dependent launch, except for route_logits):
//   1. route_wt_pack: W_r rewritten as groups of experts, transposed, so one
//      j of a group is contiguous;
//   1a. route_logits: one fp32 fused multiply-add chain per (token, expert)
//      over j ascending, + bias, written to the workspace (the logits the
//      oracle defines, bit for bit);
//   1b. route_topk: four lanes per token select the top K from the logits
//      and compute the gates.
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

// Router logits: one fp32 fused multiply-add chain per (token, expert) over
// j = 0 .. d-1 in order, then + bias[e] -- the dot product summed left to
// right.  Two launches:
//
// route_wt_pack: W_r [N][d] is rewritten as expert groups of EG experts,
// each [d][EG] (transposed, experts past N zero), so that the EG weights of
// one j are 4*EG contiguous bytes and a chunk of j rows of a group is one
// contiguous block.
//
// route_logits: CTA (token tile, expert group) runs TT tokens x EG experts
// over all of d.  x (bf16, natural layout) and the group's W chunk stream
// through a cp.async ring of JC-wide j-chunks.  Lane (lt, le) of a warp owns
// tokens lt + LT*i (i < TPT) and experts 4*le + 4*LE*q + {0..3} (q < EPT/4):
// TPT*EPT chains, advanced two tokens at a time by the packed fp32x2 fma
// (tokens 2p and 2p+1 of the lane share one expert weight).  What bounds the
// loop is the shared-memory data path (every 16-byte load delivers 512 bytes
// to a warp's registers, broadcast or not), so x stays bf16 there -- each
// 16-byte load brings 8 j of one token, widened in registers -- and each
// value loaded feeds TPT or EPT fmas.  The chains of one logit never leave
// their thread and take j in order, so every chain is the oracle's chain.
constexpr int kLogitJC = 32;      // j per chunk
constexpr int kLogitStages = 3;   // cp.async ring depth

template <int TPT_, int EPT_, int LE_, int NW_>
struct LogitCfg {
    static constexpr int TPT = TPT_, EPT = EPT_, LE = LE_, NW = NW_;
    static constexpr int LT = 32 / LE;
    static constexpr int EG = LE * EPT;               // experts per CTA
    static constexpr int TW = LT * TPT;               // tokens per warp
    static constexpr int TT = TW * NW;                // tokens per CTA
    static constexpr int NT = 32 * NW;
    static constexpr int XR = kLogitJC * 2 + 16;      // bytes per staged x row (padded)
    static constexpr int XS = TT * XR;
    static constexpr int WS = kLogitJC * EG * 4;
    static constexpr int STAGE = XS + WS;
    static constexpr size_t SMEM = (size_t)kLogitStages * STAGE;
    static_assert(EPT % 4 == 0 && TPT % 2 == 0 && 32 % LE == 0, "lane tile");
    static_assert(LT <= 8, "x rows of a warp load must fall on distinct bank groups");
};

// Tiles.  With 8 x 8 chains per lane each value a lane loads feeds 8 fmas
// (about 0.75 bytes of shared-memory traffic per fma, inside the data path's
// budget at the fma peak), but a layer with few logits then has too few warps
// to hide latency: below 2^20 logits the 4 x 4 tile (16 chains per lane, 4
// times the warps) is faster although each value feeds only 4 fmas.
using LogitWide = LogitCfg<8, 8, 8, 2>;    // 64 tokens x 64 experts per CTA, N > 32
using LogitNarrow = LogitCfg<8, 8, 4, 2>;  // 128 tokens x 32 experts per CTA, N <= 32
using LogitSmall = LogitCfg<4, 4, 8, 4>;   // 64 tokens x 32 experts per CTA
constexpr int64_t kLogitBigTile = (int64_t)1 << 20;  // T * N from which the 8 x 8 tiles run

template <int EG>
__global__ void __launch_bounds__(256)
route_wt_pack(int d, int N, const float *__restrict__ w_r, float *__restrict__ wt) {
    pdl_enter();
    __shared__ float tile[32][EG + 1];
    const int g = blockIdx.y, j0 = blockIdx.x * 32;
    for (int i = threadIdx.x; i < EG * 32; i += 256) {
        const int e = i / 32, j = i % 32, ex = g * EG + e;
        tile[j][e] = (ex < N && j0 + j < d) ? w_r[(int64_t)ex * d + j0 + j] : 0.0f;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < EG * 32; i += 256) {
        const int j = i / EG, e = i % EG;
        if (j0 + j < d) wt[((int64_t)g * d + j0 + j) * EG + e] = tile[j][e];
    }
}

template <class C>
__global__ void __launch_bounds__(C::NT)
route_logits(int T, int d, int N, const uint16_t *__restrict__ x, const float *__restrict__ wt,
             const float *__restrict__ bias, float *__restrict__ logits) {
    pdl_enter();
    constexpr int JC = kLogitJC, EG = C::EG, TT = C::TT, NT = C::NT, XR = C::XR;
    constexpr int TPT = C::TPT, EPT = C::EPT;
    extern __shared__ __align__(16) uint8_t smem_l[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int le = lane % C::LE, lt = lane / C::LE;
    const int t0 = blockIdx.x * TT, g = blockIdx.y;
    const float *wg = wt + (int64_t)g * d * EG;
    const int nchunks = (d + JC - 1) / JC;

    auto issue = [&](int c) {
        if (c < nchunks) {
            uint8_t *st = smem_l + (c % kLogitStages) * C::STAGE;
            const int j0 = c * JC, jn = min(JC, d - j0);  // a multiple of 8
            for (int i = tid; i < TT * (JC / 8); i += NT) {
                const int r = i / (JC / 8), q = (i % (JC / 8)) * 8;
                if (t0 + r < T && q < jn)
                    cp_async16(st + r * XR + q * 2, x + (int64_t)(t0 + r) * d + j0 + q);
            }
            float *ws = reinterpret_cast<float *>(st + C::XS);
            const float *src = wg + (int64_t)j0 * EG;
            for (int i = tid; i < jn * EG / 4; i += NT) cp_async16(ws + 4 * i, src + 4 * i);
        }
        cp_async_commit();
    };

    // acc[p][e]: (token lt + LT*2p, token lt + LT*(2p+1)) x expert e of the lane
    float2 acc[TPT / 2][EPT];
#pragma unroll
    for (int p = 0; p < TPT / 2; ++p)
#pragma unroll
        for (int e = 0; e < EPT; ++e) acc[p][e] = make_float2(0.0f, 0.0f);

#pragma unroll
    for (int c = 0; c < kLogitStages - 1; ++c) issue(c);
    for (int c = 0; c < nchunks; ++c) {
        cp_async_wait<kLogitStages - 2>();
        __syncthreads();  // chunk c has landed; every thread is done with chunk c - 1
        issue(c + kLogitStages - 1);
        const uint8_t *st = smem_l + (c % kLogitStages) * C::STAGE;
        const uint8_t *xs = st + (warp * C::TW + lt) * XR;
        const float *ws = reinterpret_cast<const float *>(st + C::XS) + 4 * le;
        const int jn = min(JC, d - c * JC);
        for (int j = 0; j < jn; j += 8) {
            uint4 xv[TPT];  // tokens lt + LT*i, bf16 at j .. j + 7
#pragma unroll
            for (int i = 0; i < TPT; ++i)
                xv[i] = *reinterpret_cast<const uint4 *>(xs + i * C::LT * XR + j * 2);
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                float4 wv[EPT / 4];
#pragma unroll
                for (int q = 0; q < EPT / 4; ++q)
                    wv[q] = *reinterpret_cast<const float4 *>(ws + (j + jj) * EG + 4 * C::LE * q);
#pragma unroll
                for (int p = 0; p < TPT / 2; ++p) {
                    const uint4 &a = xv[2 * p], &b = xv[2 * p + 1];
                    const uint32_t wa = jj < 2 ? a.x : jj < 4 ? a.y : jj < 6 ? a.z : a.w;
                    const uint32_t wb = jj < 2 ? b.x : jj < 4 ? b.y : jj < 6 ? b.z : b.w;
                    const float2 xp = (jj & 1) ? make_float2(bf16_hi(wa), bf16_hi(wb))
                                               : make_float2(bf16_lo(wa), bf16_lo(wb));
#pragma unroll
                    for (int q = 0; q < EPT / 4; ++q) {
                        const float w4[4] = {wv[q].x, wv[q].y, wv[q].z, wv[q].w};
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            acc[p][4 * q + u] =
                                __ffma2_rn(xp, make_float2(w4[u], w4[u]), acc[p][4 * q + u]);
                    }
                }
            }
        }
    }
    cp_async_wait<0>();
#pragma unroll
    for (int p = 0; p < TPT / 2; ++p) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int t = t0 + warp * C::TW + lt + C::LT * (2 * p + h);
            if (t >= T) continue;
            float *out = logits + (int64_t)t * N;
#pragma unroll
            for (int q = 0; q < EPT / 4; ++q)
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int e = g * EG + 4 * le + 4 * C::LE * q + u;
                    const float v = h ? acc[p][4 * q + u].y : acc[p][4 * q + u].x;
                    if (e < N) out[e] = bias ? __fadd_rn(v, bias[e]) : v;
                }
        }
    }
}

constexpr int kTopkTB = 8;      // tokens per CTA (one warp)
constexpr int kTopkGroups = 8;  // float4 groups per lane loaded before any is stored

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
// over the SMs).  The tile's logits are contiguous; every lane loads
// kTopkGroups float4 groups before storing any to shared memory (one memory
// round trip for N <= 128).  Selection: 4 lanes per token, lane s keeping
// the best MAXK of experts s, s + 4, s + 8, ... (logit descending, lower
// expert first on ties, NaN as -inf; unfilled entries are -inf with an index
// past every expert, so any expert beats them).  The lane takes its experts
// MAXK at a time, sorts them with a bitonic network and merges them into its
// list, so no step waits on a data-dependent branch; two merges over lane
// shuffles then give all four lanes the best MAXK of the token, whose first K
// are the top K.  The order is strict and total, so the result does not
// depend on how the experts were split.  Gates: softmax over the K, shifted
// by the largest, summed over k ascending.
template <int MAXK>
__global__ void __launch_bounds__(32)
route_topk(int T, int N, int K, const float *__restrict__ logits, int32_t *__restrict__ topk_idx,
           float *__restrict__ topk_gate) {
    pdl_enter();
    extern __shared__ __align__(16) uint8_t smem_t[];
    const int LDS = topk_row_stride(N);
    float *lg = reinterpret_cast<float *>(smem_t);  // [kTopkTB][LDS]
    const int tid = threadIdx.x;
    const int t0 = blockIdx.x * kTopkTB;
    const int tn = min(kTopkTB, T - t0);
    const int64_t tile = (int64_t)t0 * N, n = (int64_t)tn * N;
    if ((N & 3) == 0) {
        for (int64_t g0 = tid; g0 < n / 4; g0 += kTopkGroups * blockDim.x) {
            float4 v[kTopkGroups];
#pragma unroll
            for (int u = 0; u < kTopkGroups; ++u) {
                const int64_t g = g0 + u * blockDim.x;
                if (g < n / 4) v[u] = __ldcs(reinterpret_cast<const float4 *>(logits + tile) + g);
            }
#pragma unroll
            for (int u = 0; u < kTopkGroups; ++u) {
                const int64_t g = g0 + u * blockDim.x;
                if (g >= n / 4) continue;
                const float vv[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const int i = (int)(4 * g + h), tt = i / N, e = i - tt * N;
                    lg[tt * LDS + e] = vv[h];
                }
            }
        }
    } else {
        for (int i = tid; i < n; i += blockDim.x) {
            const int tt = i / N, e = i - tt * N;
            lg[tt * LDS + e] = logits[tile + i];
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

// Experts per group of the packed router weight (the tile's EG).
inline int logit_group(const moe_shape *s) {
    if ((int64_t)s->T * s->N < kLogitBigTile) return LogitSmall::EG;
    return s->N > 32 ? LogitWide::EG : LogitNarrow::EG;
}

// route_logits is one wave of CTAs, placed all at once when the grid starts.
// It is launched in plain stream order, not early beside the grid before it
// (programmatic dependent launch): CTAs placed while the SMs still hold
// another grid's CTAs pile onto the free SMs, and the kernel then runs at the
// pace of its most crowded SM (measured 2 to 3 times slower).
template <class C>
moe_status launch_logits_cfg(const moe_shape *s, const uint16_t *x, const float *w,
                             const float *b, float *logits, float *wt, cudaStream_t st) {
    const int G = (s->N + C::EG - 1) / C::EG;
    launch_pdl(route_wt_pack<C::EG>, dim3((s->d + 31) / 32, G), 256, 0, st, s->d, s->N, w, wt);
    moe_status r = launch_status();
    if (r != MOE_OK) return r;
    route_logits<C><<<dim3((s->T + C::TT - 1) / C::TT, G), C::NT, C::SMEM, st>>>(s->T, s->d, s->N,
                                                                             x, wt, b, logits);
    return launch_status();
}

moe_status launch_logits(const moe_shape *s, const uint16_t *x, const float *w, const float *b,
                         int32_t *idx, float *gate, float *logits, float *wt, cudaStream_t st) {
    static PerDeviceOnce smem_attr;
    if (!device_once(smem_attr, [] {
            const size_t topk_smem = sizeof(float) * kTopkTB * topk_row_stride(kMaxN);
            return set_smem_limit(route_logits<LogitWide>, LogitWide::SMEM) &&
                   set_smem_limit(route_logits<LogitNarrow>, LogitNarrow::SMEM) &&
                   set_smem_limit(route_logits<LogitSmall>, LogitSmall::SMEM) &&
                   set_smem_limit(route_topk<8>, topk_smem) &&
                   set_smem_limit(route_topk<kMaxK>, topk_smem);
        }))
        return MOE_ERR_CUDA;
    moe_status r;
    if ((int64_t)s->T * s->N < kLogitBigTile)
        r = launch_logits_cfg<LogitSmall>(s, x, w, b, logits, wt, st);
    else if (s->N > 32)
        r = launch_logits_cfg<LogitWide>(s, x, w, b, logits, wt, st);
    else
        r = launch_logits_cfg<LogitNarrow>(s, x, w, b, logits, wt, st);
    if (r != MOE_OK) return r;
    const size_t tsmem = sizeof(float) * kTopkTB * topk_row_stride(s->N);
    auto *topk = s->K <= 8 ? route_topk<8> : route_topk<kMaxK>;
    launch_pdl(topk, (s->T + kTopkTB - 1) / kTopkTB, 32, tsmem, st, s->T, s->N, s->K, logits, idx,
               gate);
    return launch_status();
}

}  // namespace

inline size_t route_block_count_bytes(const moe_shape *s) {
    const size_t nblk = (size_t)(s->T + kRankBlock - 1) / kRankBlock;
    return (nblk * (size_t)s->N * sizeof(int32_t) + 255) & ~(size_t)255;
}

inline size_t round256(size_t n) { return (n + 255) & ~(size_t)255; }

inline size_t route_logits_bytes(const moe_shape *s) {
    return round256((size_t)s->T * s->N * sizeof(float));
}

// status word (256 B), the per-block count array, the logits [T][N] fp32,
// then W_r packed by expert groups [ceil(N / EG)][d][EG] fp32
size_t route_ws_bytes(const moe_shape *s) {
    const int eg = logit_group(s);
    const size_t wt = (size_t)((s->N + eg - 1) / eg) * s->d * eg * sizeof(float);
    return 256 + route_block_count_bytes(s) + route_logits_bytes(s) + round256(wt);
}

// Enqueues the routing kernels; `scratch` is the workspace past its status
// word (route_ws_bytes(s) - 256 bytes).
moe_status route_enqueue(const moe_shape *s, const moe_bf16 *x, const float *w_router,
                         const float *bias, int32_t *topk_idx, float *topk_gate,
                         int32_t *route_row, int32_t *expert_count, int32_t *expert_offset,
                         int32_t *expert_demand, void *scratch, cudaStream_t st) {
    const int nblk = (s->T + kRankBlock - 1) / kRankBlock;
    int32_t *block_count = static_cast<int32_t *>(scratch);
    char *after_counts = static_cast<char *>(scratch) + route_block_count_bytes(s);
    float *logits = reinterpret_cast<float *>(after_counts);
    float *wt = reinterpret_cast<float *>(after_counts + route_logits_bytes(s));
    moe_status r = MOE_OK;
    if (s->T > 0) {
        r = launch_logits(s, x, w_router, bias, topk_idx, topk_gate, logits, wt, st);
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

MOE_API size_t moe_route_logits_offset(const moe_shape *s) {
    if (check_shape(s) != MOE_OK) return 0;
    return 256 + route_block_count_bytes(s);
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
// Its scratch -- the 256-byte status word (unused by routing), the per-block
// counts, the fp32 logits [T][N] and the router weight regrouped by experts,
// laid out as in moe_route's workspace -- lives in the fixed array below
// instead of a caller-provided workspace.  Every GPU
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
