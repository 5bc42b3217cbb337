// Grouped expert GEMMs over the packed capacity buffers (steps F1, F2).
//
// OLMo-core MoE report, "Section 05: Expert Parallelism", Figure 14 (Linear 1
// -> SwiGLU -> Linear 2) and 5.7 (experts packed back to back; expert forward
// receives the real per-expert row offsets and skips the unwritten tail);
// "Section 08: Synchronization-Free Training", 8.5 and Table 14 (grouped GEMM
// driven by a device int32 cumulative-offset tensor; a tail-aware SwiGLU that
// touches only the valid prefix); "Section 04: Distributed Data Parallel", 4.1
// (bias-free SwiGLU expert).
//
// One persistent kernel per GEMM, one CTA per SM, 10 warps:
//   warp 0     TMA producer: 128x64 A tiles and 256x64 B tiles into a
//              4-stage shared-memory ring (128-byte swizzle);
//   warp 1     tcgen05.mma issuer (one thread; M=128, N=256, K=16 steps) into a
//              double-buffered fp32 accumulator in tensor memory (2 x 256 of
//              the SM's 512 columns), and owner of the TMEM allocation;
//   warps 2-9  epilogue (two warps per TMEM lane quadrant, each taking half
//              of the columns): tcgen05.ld of the accumulator, then either SwiGLU
//              (F1: columns 0-127 are the gate rows, 128-255 the up rows of the
//              same 128 hidden units) or a plain bf16 store (F2).
// Work list: every CTA derives, from expert_count in device memory, the tiles
// of every expert (ceil(count/128) row tiles x output-column tiles) and walks
// them round-robin.  Rows past an expert's count (the next expert's rows or
// the tail) enter the MMA but are never stored; column tiles past the output
// width are never stored either.  No host round trip, no per-expert launch.
#include <algorithm>

#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int MMA_N = 256;
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = MMA_N * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int ACC_COLS = 256;
constexpr int TMEM_COLS = 512;
constexpr int kEpiThreads = 256;  // 8 epilogue warps
constexpr int kThreads = 64 + kEpiThreads;

enum { EPI_SWIGLU = 0, EPI_STORE = 1 };

struct alignas(8) Bars {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint32_t tmem_base;
    int abort;
};

constexpr size_t smem_bytes(int N) {
    return 1024 + (size_t)STAGES * STAGE_BYTES + sizeof(Bars) + sizeof(int32_t) * (N + 1) + 16;
}

struct TileMap {
    int e, m, n;
};

// Expert owning tile g: the last e with tile_start[e] <= g.
__device__ __forceinline__ TileMap map_tile(int g, int N, const int32_t *tile_start,
                                            const int32_t *count) {
    int lo = 0, hi = N - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tile_start[mid] <= g) lo = mid;
        else hi = mid - 1;
    }
    const int mt = (count[lo] + BM - 1) / BM;
    const int local = g - tile_start[lo];
    return TileMap{lo, local % mt, local / mt};
}

template <int EPI>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b0,
             const __grid_constant__ CUtensorMap tm_b1, int N, int Kdim, int Nout,
             const int32_t *__restrict__ count, const int32_t *__restrict__ offset,
             uint16_t *__restrict__ out, uint16_t *__restrict__ g_save,
             uint16_t *__restrict__ u_save, int *status) {
    constexpr int BN_OUT = EPI == EPI_SWIGLU ? MMA_N / 2 : MMA_N;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    Bars *bars = reinterpret_cast<Bars *>(smem + (size_t)STAGES * STAGE_BYTES);
    int32_t *tile_start = reinterpret_cast<int32_t *>(bars + 1);
    volatile int *abort = &bars->abort;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntn = (Nout + BN_OUT - 1) / BN_OUT;
    const int nk = (Kdim + BK - 1) / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&bars->full[s]), 1);
            mbar_init(smem_u32(&bars->empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&bars->tfull[b]), 1);
            mbar_init(smem_u32(&bars->tempty[b]), kEpiThreads);
        }
        bars->abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        // tile_start[e] = tiles of experts < e (warp-wide scan, 32 experts per step)
        int carry = 0;
        for (int base = 0; base < N; base += 32) {
            const int e = base + lane;
            const int v = e < N ? ((count[e] + BM - 1) / BM) * ntn : 0;
            int incl = v;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int u = __shfl_up_sync(0xFFFFFFFFu, incl, off);
                if (lane >= off) incl += u;
            }
            if (e < N) tile_start[e] = carry + incl - v;
            carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
        if (lane == 0) tile_start[N] = carry;
    }
    if (warp == 1) tmem_alloc(smem_u32(&bars->tmem_base), TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = bars->tmem_base;
    const int total = tile_start[N];

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&tm_a);
            tma_prefetch_desc(&tm_b0);
            if (EPI == EPI_SWIGLU) tma_prefetch_desc(&tm_b1);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int g = blockIdx.x; g < total && ok; g += gridDim.x) {
                const TileMap t = map_tile(g, N, tile_start, count);
                const int a_row = offset[t.e] + t.m * BM;
                const int b_row = t.e * Nout + t.n * BN_OUT;
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait(smem_u32(&bars->empty[stage]), phase ^ 1, status, abort)) {
                        ok = false;
                        break;
                    }
                    const uint32_t full = smem_u32(&bars->full[stage]);
                    const uint32_t sa = smem_u32(smem + (size_t)stage * STAGE_BYTES);
                    const uint32_t sb = sa + A_BYTES;
                    mbar_arrive_expect_tx(full, STAGE_BYTES);
                    tma_load_2d(sa, &tm_a, full, kb * BK, a_row);
                    if (EPI == EPI_SWIGLU) {
                        tma_load_2d(sb, &tm_b0, full, kb * BK, b_row);
                        tma_load_2d(sb + B_BYTES / 2, &tm_b1, full, kb * BK, b_row);
                    } else {
                        tma_load_2d(sb, &tm_b0, full, kb * BK, b_row);
                    }
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok) {
                // let copies already issued land before the CTA leaves
                for (int s = 0; s < STAGES; ++s) {
                    volatile int no_abort = 0;
                    mbar_wait(smem_u32(&bars->full[s]), phase ^ (s >= stage ? 1 : 0), status,
                              &no_abort);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(BM, MMA_N);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int g = blockIdx.x; g < total && ok; g += gridDim.x) {
                if (!mbar_wait(smem_u32(&bars->tempty[acc]), acc_phase ^ 1, status, abort)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * ACC_COLS);
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait(smem_u32(&bars->full[stage]), phase, status, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + (size_t)stage * STAGE_BYTES);
                    const uint32_t sb = sa + A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        tc_mma_bf16(d_tmem, sw128_kmajor_desc(sa + kk * 32),
                                    sw128_kmajor_desc(sb + kk * 32), idesc,
                                    (kb | kk) != 0 ? 1u : 0u);
                    }
                    tc_commit(smem_u32(&bars->empty[stage]));
                    if (++stage == STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                tc_commit(smem_u32(&bars->tfull[acc]));
                if (++acc == 2) { acc = 0; acc_phase ^= 1; }
            }
        }
    } else {
        // epilogue: warp w reads TMEM lanes 32 * (w % 4) .. + 31 = tile rows
        const int quad = warp & 3;
        const int half = (warp - 2) >> 2;  // which half of the columns
        const int row_in_tile = quad * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int g = blockIdx.x; g < total; g += gridDim.x) {
            const TileMap t = map_tile(g, N, tile_start, count);
            const int rows_valid = count[t.e] - t.m * BM;
            const bool row_ok = row_in_tile < rows_valid;
            const int64_t row = (int64_t)offset[t.e] + t.m * BM + row_in_tile;
            if (!mbar_wait(smem_u32(&bars->tfull[acc]), acc_phase, status, abort)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + ((uint32_t)(quad * 32) << 16) + acc * ACC_COLS;
            if (EPI == EPI_SWIGLU) {
                for (int c = half * (BN_OUT / 2); c < (half + 1) * (BN_OUT / 2); c += 16) {
                    uint32_t gr[16], ur[16];
                    tmem_ld16(tbase + c, gr);
                    tmem_ld16(tbase + BN_OUT + c, ur);
                    tmem_ld_wait();
                    reg_fence(gr);
                    reg_fence(ur);
                    const int col = t.n * BN_OUT + c;
                    if (row_ok && col < Nout) {
                        uint32_t hp[8], gp[8], up[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            const float g0 = __uint_as_float(gr[2 * i]);
                            const float g1 = __uint_as_float(gr[2 * i + 1]);
                            const float u0 = __uint_as_float(ur[2 * i]);
                            const float u1 = __uint_as_float(ur[2 * i + 1]);
                            const float h0 = __fdividef(g0, 1.0f + __expf(-g0)) * u0;
                            const float h1 = __fdividef(g1, 1.0f + __expf(-g1)) * u1;
                            hp[i] = pack_bf16x2(h0, h1);
                            gp[i] = pack_bf16x2(g0, g1);
                            up[i] = pack_bf16x2(u0, u1);
                        }
                        uint4 *dst = reinterpret_cast<uint4 *>(out + row * Nout + col);
                        dst[0] = make_uint4(hp[0], hp[1], hp[2], hp[3]);
                        dst[1] = make_uint4(hp[4], hp[5], hp[6], hp[7]);
                        if (g_save) {
                            uint4 *gd = reinterpret_cast<uint4 *>(g_save + row * Nout + col);
                            gd[0] = make_uint4(gp[0], gp[1], gp[2], gp[3]);
                            gd[1] = make_uint4(gp[4], gp[5], gp[6], gp[7]);
                            uint4 *ud = reinterpret_cast<uint4 *>(u_save + row * Nout + col);
                            ud[0] = make_uint4(up[0], up[1], up[2], up[3]);
                            ud[1] = make_uint4(up[4], up[5], up[6], up[7]);
                        }
                    }
                }
            } else {
                for (int c = half * (BN_OUT / 2); c < (half + 1) * (BN_OUT / 2); c += 32) {
                    uint32_t r0[16], r1[16];
                    tmem_ld16(tbase + c, r0);
                    tmem_ld16(tbase + c + 16, r1);
                    tmem_ld_wait();
                    reg_fence(r0);
                    reg_fence(r1);
                    const int col = t.n * BN_OUT + c;
                    if (row_ok && col < Nout) {
                        uint32_t p[16];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            p[i] = pack_bf16x2(__uint_as_float(r0[2 * i]),
                                               __uint_as_float(r0[2 * i + 1]));
                            p[8 + i] = pack_bf16x2(__uint_as_float(r1[2 * i]),
                                                   __uint_as_float(r1[2 * i + 1]));
                        }
                        uint4 *dst = reinterpret_cast<uint4 *>(out + row * Nout + col);
                        dst[0] = make_uint4(p[0], p[1], p[2], p[3]);
                        dst[1] = make_uint4(p[4], p[5], p[6], p[7]);
                        if (col + 16 < Nout) {
                            dst[2] = make_uint4(p[8], p[9], p[10], p[11]);
                            dst[3] = make_uint4(p[12], p[13], p[14], p[15]);
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&bars->tempty[acc]));
            if (++acc == 2) { acc = 0; acc_phase ^= 1; }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ---------------------------------------------------------------- host side --

template <int EPI>
moe_status launch_gemm(const CUtensorMap &a, const CUtensorMap &b0, const CUtensorMap &b1, int N,
                       int Kdim, int Nout, int max_row_tiles, const int32_t *count,
                       const int32_t *offset, uint16_t *out, uint16_t *gs, uint16_t *us,
                       int *status, cudaStream_t st) {
    const size_t smem = smem_bytes(N);
    static size_t configured = 0;
    if (smem > configured) {
        if (cudaFuncSetAttribute(grouped_gemm<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem_bytes(kMaxN)) != cudaSuccess)
            return MOE_ERR_CUDA;
        configured = smem_bytes(kMaxN);
    }
    constexpr int BN_OUT = EPI == EPI_SWIGLU ? MMA_N / 2 : MMA_N;
    const int64_t max_tiles = (int64_t)max_row_tiles * ((Nout + BN_OUT - 1) / BN_OUT);
    const int grid = (int)std::min<int64_t>(num_sms(), std::max<int64_t>(max_tiles, 1));
    grouped_gemm<EPI><<<grid, kThreads, smem, st>>>(a, b0, b1, N, Kdim, Nout, count, offset, out,
                                                    gs, us, status);
    return launch_status();
}

}  // namespace
}  // namespace moe

using namespace moe;

MOE_API size_t moe_expert_ffn_workspace_bytes(const moe_shape *s) {
    if (check_shape(s) != MOE_OK) return 0;
    return 256;
}

MOE_API moe_status moe_expert_ffn(const moe_shape *s, const moe_bf16 *x_disp,
                                  const int32_t *expert_count, const int32_t *expert_offset,
                                  const moe_bf16 *w_gate, const moe_bf16 *w_up,
                                  const moe_bf16 *w_down, moe_bf16 *h_act, moe_bf16 *g_save,
                                  moe_bf16 *u_save, moe_bf16 *y_disp, void *ws, size_t ws_bytes,
                                  cudaStream_t stream) {
    moe_status r = check_shape(s);
    if (r != MOE_OK) return r;
    if (s->d % BK != 0 || s->h % BK != 0) return MOE_ERR_UNSUPPORTED;
    if (!expert_count || !expert_offset || !ws) return MOE_ERR_INVALID_ARG;
    if ((g_save == nullptr) != (u_save == nullptr)) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < 256 || (reinterpret_cast<uintptr_t>(ws) & 255u)) return MOE_ERR_WORKSPACE;
    const int64_t R = (int64_t)s->N * s->cap;
    if (R == 0 || s->T == 0) return MOE_OK;
    if (!x_disp || !w_gate || !w_up || !w_down || !h_act || !y_disp) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x_disp) || !aligned16(w_gate) || !aligned16(w_up) || !aligned16(w_down) ||
        !aligned16(h_act) || !aligned16(y_disp) || (g_save && !aligned16(g_save)) ||
        (u_save && !aligned16(u_save)) || !aligned16(expert_count) || !aligned16(expert_offset))
        return MOE_ERR_ALIGNMENT;
    CUtensorMap ma, mg, mu, mh, md;
    if (!make_map(&ma, x_disp, s->d, R, BM) || !make_map(&mg, w_gate, s->d, (uint64_t)s->N * s->h, 128) ||
        !make_map(&mu, w_up, s->d, (uint64_t)s->N * s->h, 128) ||
        !make_map(&mh, h_act, s->h, R, BM) ||
        !make_map(&md, w_down, s->h, (uint64_t)s->N * s->d, MMA_N))
        return MOE_ERR_CUDA;
    int *status = static_cast<int *>(ws);
    const int64_t rows = std::min<int64_t>(R, (int64_t)s->T * s->K);
    const int max_row_tiles = (int)((rows + BM - 1) / BM + s->N);
    r = launch_gemm<EPI_SWIGLU>(ma, mg, mu, s->N, s->d, s->h, max_row_tiles, expert_count,
                                expert_offset, h_act, g_save, u_save, status, stream);
    if (r != MOE_OK) return r;
    return launch_gemm<EPI_STORE>(mh, md, md, s->N, s->h, s->d, max_row_tiles, expert_count,
                                  expert_offset, y_disp, nullptr, nullptr, status, stream);
}
