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
// One persistent kernel per GEMM; CTAs run in clusters of two, one CTA per SM,
// 10 warps each:
//   warp 0     TMA producer (both CTAs): this CTA's 128 rows of A and half of B
//              per 64-wide k-block, 32 KB, into a 6-stage ring (128-byte swizzle);
//   warp 1     in the pair's leader, one thread issues tcgen05.mma.cta_group::2
//              (M = 256 across the pair, N = 256, K = 16) into a double-buffered
//              fp32 accumulator in tensor memory (2 x 256 of 512 columns), and
//              the warp owns the pair-wide TMEM allocation;
//   warps 2-9  epilogue (two warps per TMEM lane quadrant, each half of the
//              columns): tcgen05.ld of this CTA's 128 accumulator rows, then
//              SwiGLU (F1: columns 0-127 are the gate rows, loaded by the leader,
//              128-255 the up rows, loaded by the peer) or a bf16 copy (F2);
//              a warp whose 32 rows are all valid writes each 32 x 32 output
//              block to its 2 KB of shared memory (64-byte swizzle) and stores
//              it with one TMA instruction; other warps store their valid rows.
// With GATHER (moe_expert_ffn_gather) two more warps per CTA gather the A rows
// straight from x by route (16-byte cp.async into the swizzled stage), so no
// dispatched copy is made; // from x by route (tile::gather4 loads), so no dispatched copy is made.
// Work list: every CTA derives, from expert_count in device memory, the tiles
// of every expert (ceil(count/256) row tiles x output-column tiles) and walks
// them round-robin.  Rows past an expert's count (the next expert's rows or
// the tail) enter the MMA but are never stored; column tiles past the output
// width are never stored either.  No host round trip, no per-expert launch.
// Swap tiles: an expert's last row tile with at most 128 valid rows (all of a
// small expert's rows, or a large expert's remainder) runs with the operands
// exchanged -- A = 256 weight rows, B = the tile's token rows rounded up to 32
// -- so the MMA computes those few columns instead of 256 rows; the
// accumulator then holds the outputs transposed (lane = output column, TMEM
// column = token) and they are stored token by token.
#include <algorithm>

#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int MMA_N = 256;
constexpr int A_BYTES = BM * BK * 2;
constexpr int ACC_COLS = 256;
constexpr int TMEM_COLS = 512;
constexpr int kEpiThreads = 256;  // 8 epilogue warps
constexpr int kThreads = 64 + kEpiThreads;
constexpr int kGatherWarps = 2;  // GATHER: warps 10-11 fetch the A rows
constexpr int kGatherThreads = 32 * kGatherWarps;
template <bool GATHER>
constexpr int pair_threads() { return kThreads + (GATHER ? kGatherThreads : 0); }

enum { EPI_SWIGLU = 0, EPI_STORE = 1 };

struct TileMap {
    int e, m, n;
};

// Epilogue of one accumulator tile for one warp: its 32 TMEM lanes (rows) and
// one half of the columns.  F1: columns [0, 128) hold G and [128, 256) hold U of
// the same hidden units; H = silu(G) * U.  F2: a plain bf16 store.
template <int EPI>
__device__ __forceinline__ void epilogue_tile(uint32_t tbase, int half, bool row_ok, int64_t row,
                                              int n, int Nout, uint16_t *__restrict__ out,
                                              uint16_t *__restrict__ g_save,
                                              uint16_t *__restrict__ u_save) {
    constexpr int BN_OUT = EPI == EPI_SWIGLU ? MMA_N / 2 : MMA_N;
    if (EPI == EPI_SWIGLU) {
        for (int c = half * (BN_OUT / 2); c < (half + 1) * (BN_OUT / 2); c += 16) {
            uint32_t gr[16], ur[16];
            tmem_ld16(tbase + c, gr);
            tmem_ld16(tbase + BN_OUT + c, ur);
            tmem_ld_wait();
            reg_fence(gr);
            reg_fence(ur);
            const int col = n * BN_OUT + c;
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
            const int col = n * BN_OUT + c;
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
}

// The same epilogue for a warp whose 32 rows are all valid: each 32-column
// chunk is packed to bf16 and stored through the warp's 2 KB shared-memory
// block by TMA (one instruction per chunk and output), instead of 32 row
// segments per store instruction.
template <int EPI>
__device__ __forceinline__ void epilogue_tile_tma(uint32_t tbase, int half, int row0, int n,
                                                  int Nout, uint8_t *blk, const CUtensorMap *mo,
                                                  const CUtensorMap *mg, const CUtensorMap *mu,
                                                  bool save, int lane) {
    constexpr int BN_OUT = EPI == EPI_SWIGLU ? MMA_N / 2 : MMA_N;
    for (int c = half * (BN_OUT / 2); c < (half + 1) * (BN_OUT / 2); c += 32) {
        const int col = n * BN_OUT + c;
        if (EPI == EPI_SWIGLU) {
            uint32_t g0[16], g1[16], u0[16], u1[16];
            tmem_ld16(tbase + c, g0);
            tmem_ld16(tbase + c + 16, g1);
            tmem_ld16(tbase + BN_OUT + c, u0);
            tmem_ld16(tbase + BN_OUT + c + 16, u1);
            tmem_ld_wait();
            reg_fence(g0);
            reg_fence(g1);
            reg_fence(u0);
            reg_fence(u1);
            if (col >= Nout) continue;  // warp-uniform
            uint32_t hp[16], gp[16], up[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const uint32_t *gs = i < 8 ? g0 : g1;
                const uint32_t *us = i < 8 ? u0 : u1;
                const int k = 2 * (i & 7);
                const float ga = __uint_as_float(gs[k]), gb = __uint_as_float(gs[k + 1]);
                const float ua = __uint_as_float(us[k]), ub = __uint_as_float(us[k + 1]);
                hp[i] = pack_bf16x2(__fdividef(ga, 1.0f + __expf(-ga)) * ua,
                                    __fdividef(gb, 1.0f + __expf(-gb)) * ub);
                gp[i] = pack_bf16x2(ga, gb);
                up[i] = pack_bf16x2(ua, ub);
            }
            warp_store_bf16_32x32(blk, hp, mo, col, row0, lane);
            if (save) {
                warp_store_bf16_32x32(blk, gp, mg, col, row0, lane);
                warp_store_bf16_32x32(blk, up, mu, col, row0, lane);
            }
        } else {
            uint32_t r0[16], r1[16];
            tmem_ld16(tbase + c, r0);
            tmem_ld16(tbase + c + 16, r1);
            tmem_ld_wait();
            reg_fence(r0);
            reg_fence(r1);
            if (col >= Nout) continue;  // warp-uniform
            uint32_t p[16];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                p[i] = pack_bf16x2(__uint_as_float(r0[2 * i]), __uint_as_float(r0[2 * i + 1]));
                p[8 + i] = pack_bf16x2(__uint_as_float(r1[2 * i]), __uint_as_float(r1[2 * i + 1]));
            }
            warp_store_bf16_32x32(blk, p, mo, col, row0, lane);
        }
    }
}

// ---------------------------------------------------------- swap-AB tiles
//
// An expert's last tile with at most SWAP_MAX valid rows runs as M = 256
// weight rows (128 per CTA) by N = n_sw token columns (the valid rows rounded
// up to 32; the leader holds tokens 0..n_sw/2-1, the peer the rest).  F1: each
// CTA's 128 A rows are the gate rows (0-63) and the up rows (64-127) of the
// same 64 hidden units, loaded as two 64-row boxes; the up values of TMEM lane
// quadrants 2-3 reach the gate lanes of quadrants 0-1 through the up warp's
// staging block (a named barrier per warp pair).  F2: each CTA's A rows are
// 128 rows of W_down (output features).  Few, large TMA boxes per stage
// matter: the copy engine's cost is per request.
constexpr int SWAP_MAX = 128;
constexpr int SW_BOX = 32;  // token rows per B load of a swap tile

__device__ __forceinline__ int swap_cols(int rows) { return (rows + 31) & ~31; }

__device__ __forceinline__ uint16_t bf16_bits(float v) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// F1 epilogue of a swap tile for one warp of a gate/up warp pair: accumulator
// columns (tokens) [c0, c1).  An up warp (quadrant 2-3) passes its values
// through `xbuf` (its own 2 KB staging block); the gate warp (quadrant 0-1)
// computes H = silu(G) * U for hidden unit `hid` and stores it per token.
__device__ __forceinline__ void epilogue_swap_swiglu(uint32_t tbase, int c0, int c1,
                                                     int rows_valid, int64_t row0, bool gate_warp,
                                                     float *xbuf, int bar_id, int hid, int Nout,
                                                     int lane, uint16_t *__restrict__ out,
                                                     uint16_t *__restrict__ g_save,
                                                     uint16_t *__restrict__ u_save) {
    if (!gate_warp) {
        if (lane == 0) bulk_wait_read<0>();  // an earlier TMA store from the block is done
        __syncwarp();
    }
    for (int c = c0; c < c1; c += 16) {
        uint32_t v[16];
        tmem_ld16(tbase + c, v);
        tmem_ld_wait();
        reg_fence(v);
        if (!gate_warp) {
#pragma unroll
            for (int i = 0; i < 16; ++i) xbuf[i * 32 + lane] = __uint_as_float(v[i]);
            named_bar_sync(bar_id, 64);  // up values ready
            named_bar_sync(bar_id, 64);  // gate warp done reading
            continue;
        }
        float u[16];
        named_bar_sync(bar_id, 64);
#pragma unroll
        for (int i = 0; i < 16; ++i) u[i] = xbuf[i * 32 + lane];
        named_bar_sync(bar_id, 64);
        if (hid < Nout) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                if (c + i >= rows_valid) break;
                const float g = __uint_as_float(v[i]);
                const int64_t at = (row0 + c + i) * Nout + hid;
                out[at] = bf16_bits(__fdividef(g, 1.0f + __expf(-g)) * u[i]);
                if (g_save) {
                    g_save[at] = bf16_bits(g);
                    u_save[at] = bf16_bits(u[i]);
                }
            }
        }
    }
}

// F2 epilogue of a swap tile for one warp: output feature `feat` of this lane,
// accumulator columns (tokens) [c0, c1).
__device__ __forceinline__ void epilogue_swap_store(uint32_t tbase, int c0, int c1,
                                                    int rows_valid, int64_t row0, int feat,
                                                    int Nout, uint16_t *__restrict__ out) {
    for (int c = c0; c < c1; c += 16) {
        uint32_t v[16];
        tmem_ld16(tbase + c, v);
        tmem_ld_wait();
        reg_fence(v);
        if (feat < Nout) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                if (c + i >= rows_valid) break;
                out[(row0 + c + i) * Nout + feat] = bf16_bits(__uint_as_float(v[i]));
            }
        }
    }
}

// ------------------------------------------------------------ CTA-pair kernel
//
// Two CTAs of a cluster compute one 256-row x 256-column tile with
// tcgen05.mma.cta_group::2 (M = 256, N = 256): each CTA holds its own 128 rows
// of A and one half of B (F1: the gate rows in the leader, the up rows in the
// peer; F2: columns 0-127 / 128-255), so each SM stages and reads 32 KB per
// k-block instead of 48 KB, and six stages fit.  The leader (rank 0) issues the
// MMAs; both CTAs' TMA loads complete on the leader's full barrier; the
// leader's commits release a stage, and announce an accumulator, in both CTAs
// at once; both CTAs' epilogue warps release the accumulator on the leader's
// barrier.  Each CTA's TMEM holds its own 128 accumulator rows.
constexpr int P_STAGES = 6;
constexpr int P_B_BYTES = (MMA_N / 2) * BK * 2;   // this CTA's half of B
constexpr int P_STAGE_BYTES = A_BYTES + P_B_BYTES;  // 32 KB
constexpr int P_EPI_WARPS = kEpiThreads / 32;

struct alignas(8) PairBars {
    uint64_t full[P_STAGES];
    uint64_t empty[P_STAGES];
    uint64_t gfull[P_STAGES];  // GATHER: this CTA's A rows of the stage landed
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint32_t tmem_base;
    int abort;
};

constexpr int P_STG_BYTES = P_EPI_WARPS * 2048;  // one 32 x 32 bf16 store block per epilogue warp

// ... + tile_start [N + 1] and the expert counts [N] (copied once, so that the
// MMA issuer reads no global memory between tiles)
constexpr size_t smem_bytes_pair(int N) {
    return 1024 + (size_t)P_STAGES * P_STAGE_BYTES + P_STG_BYTES + sizeof(PairBars) +
           sizeof(int32_t) * (2 * N + 1) + 16;
}

// GATHER: A is not the packed buffer but the token rows themselves.  The two
// gather warps of each CTA fetch packed row r of its 128 from x[row_token[r]]
// with 16-byte cp.async (thread t: rows t/8 + 8i, 16-byte chunk t%8 of the
// k-block, written to the 128-byte swizzled position), so one warp
// instruction moves four whole 128-byte rows; each thread's copies of a stage
// arrive on the CTA's gfull barrier when they land, so the gather threads
// never wait for their own copies and keep every free stage in flight.  Lane
// 1 of warp 0 forwards each stage in order: it waits for gfull, fences the
// rows to the async proxy (the tensor core reads them there) and arrives on
// the leader's full barrier, which thus counts the leader's expect_tx (B by
// TMA) and the two CTAs' forwards.  Rows past the expert's count read token
// 0; their accumulator rows are never stored.
__device__ __forceinline__ void cp_async16_s(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

// Swap tiles: tm_sa0 / tm_sa1 are the A maps of a swap tile (F1: W_gate and
// W_up with 64-row boxes; F2: W_down with 128-row boxes, tm_sa1 unused) and
// tm_sb the B map (the packed rows with 32-row boxes).  GATHER runs no swap
// tiles.
template <int EPI, bool GATHER>
__global__ void __launch_bounds__(pair_threads<GATHER>(), 1)
grouped_gemm_pair(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b0,
                  const __grid_constant__ CUtensorMap tm_b1, const __grid_constant__ CUtensorMap tm_o,
                  const __grid_constant__ CUtensorMap tm_g, const __grid_constant__ CUtensorMap tm_u,
                  const __grid_constant__ CUtensorMap tm_sa0, const __grid_constant__ CUtensorMap tm_sa1,
                  const __grid_constant__ CUtensorMap tm_sb,
                  int N, int Kdim, int Nout,
                  const int32_t *__restrict__ count, const int32_t *__restrict__ offset,
                  const int32_t *__restrict__ row_token, const uint16_t *__restrict__ x_rows,
                  uint16_t *__restrict__ out,
                  uint16_t *__restrict__ g_save, uint16_t *__restrict__ u_save, int *status) {
    pdl_enter();
    constexpr int BN_OUT = EPI == EPI_SWIGLU ? MMA_N / 2 : MMA_N;
    constexpr int PM = 2 * BM;  // rows per pair tile
    constexpr bool kSwap = !GATHER;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *stage_out = smem + (size_t)P_STAGES * P_STAGE_BYTES;  // [8 warps][2 KB]
    PairBars *bars = reinterpret_cast<PairBars *>(stage_out + P_STG_BYTES);
    int32_t *tile_start = reinterpret_cast<int32_t *>(bars + 1);
    int32_t *cnt = tile_start + N + 1;  // expert_count, copied
    volatile int *abort = &bars->abort;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const int unit0 = (int)blockIdx.x / 2, units = (int)gridDim.x / 2;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntn = (Nout + BN_OUT - 1) / BN_OUT;
    const int nk = (Kdim + BK - 1) / BK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < P_STAGES; ++s) {
            mbar_init(smem_u32(&bars->full[s]), GATHER ? 3 : 1);
            mbar_init(smem_u32(&bars->empty[s]), 1);
            mbar_init(smem_u32(&bars->gfull[s]), kGatherThreads);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&bars->tfull[b]), 1);
            mbar_init(smem_u32(&bars->tempty[b]), 2 * P_EPI_WARPS);
        }
        bars->abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        // tile_start[e] = pair tiles of experts < e
        int carry = 0;
        for (int base = 0; base < N; base += 32) {
            const int e = base + lane;
            const int c = e < N ? count[e] : 0;
            if (e < N) cnt[e] = c;
            const int v = ((c + PM - 1) / PM) * ntn;
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
    if (warp == 1) tmem_alloc_pair(smem_u32(&bars->tmem_base), TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // barriers of both CTAs exist before any remote arrival
    tc_fence_after();
    const uint32_t tmem_base = bars->tmem_base;
    const int total = tile_start[N];

    auto map_pair = [&](int g) {
        int lo = 0, hi = N - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (tile_start[mid] <= g) lo = mid;
            else hi = mid - 1;
        }
        const int mt = (cnt[lo] + PM - 1) / PM;
        const int local = g - tile_start[lo];
        return TileMap{lo, local % mt, local / mt};
    };

    if (warp == 0) {
        // -------------------------------------------- TMA producer (both CTAs)
        if (lane == 0) {
            tma_prefetch_desc(&tm_a);
            tma_prefetch_desc(rank && EPI == EPI_SWIGLU ? &tm_b1 : &tm_b0);
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool ok = true;
            for (int g = unit0; g < total && ok; g += units) {
                const TileMap t = map_pair(g);
                const int rows_valid = cnt[t.e] - t.m * PM;
                const bool swap = kSwap && rows_valid <= SWAP_MAX;
                const int n_sw = swap_cols(rows_valid);
                const int sw_loads = (n_sw / 2 + SW_BOX - 1) / SW_BOX;
                const int a_row = offset[t.e] + t.m * PM + (int)rank * BM;
                const int b_row = EPI == EPI_SWIGLU ? t.e * Nout + t.n * BN_OUT
                                                    : t.e * Nout + t.n * BN_OUT + (int)rank * (MMA_N / 2);
                const CUtensorMap *mb = rank && EPI == EPI_SWIGLU ? &tm_b1 : &tm_b0;
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait(smem_u32(&bars->empty[stage]), phase ^ 1, status, abort)) {
                        ok = false;
                        break;
                    }
                    const uint32_t own_full = smem_u32(&bars->full[stage]);
                    const uint32_t full = cluster_map(own_full, 0);
                    const uint32_t sa = smem_u32(smem + (size_t)stage * P_STAGE_BYTES);
                    const uint32_t sb = sa + A_BYTES;
                    if (swap) {
                        if (leader)
                            mbar_arrive_expect_tx(own_full, 2 * (A_BYTES + sw_loads * SW_BOX * BK * 2));
                        if (EPI == EPI_SWIGLU) {
                            const int hrow = t.e * Nout + t.n * BN_OUT + 64 * (int)rank;
                            tma_load_2d_pair(sa, &tm_sa0, full, kb * BK, hrow);
                            tma_load_2d_pair(sa + 64 * 128, &tm_sa1, full, kb * BK, hrow);
                        } else {
                            tma_load_2d_pair(sa, &tm_sa0, full, kb * BK,
                                             t.e * Nout + t.n * MMA_N + BM * (int)rank);
                        }
                        const int trow = offset[t.e] + t.m * PM + (int)rank * (n_sw / 2);
                        for (int i = 0; i < sw_loads; ++i)
                            tma_load_2d_pair(sb + (uint32_t)(i * SW_BOX) * 128, &tm_sb, full,
                                             kb * BK, trow + i * SW_BOX);
                    } else {
                        if (leader)
                            mbar_arrive_expect_tx(own_full,
                                                  GATHER ? 2 * P_B_BYTES : 2 * P_STAGE_BYTES);
                        if (!GATHER) tma_load_2d_pair(sa, &tm_a, full, kb * BK, a_row);
                        tma_load_2d_pair(sb, mb, full, kb * BK, b_row);
                    }
                    ++issued;
                    if (++stage == P_STAGES) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok && leader) {
                // the leader's full barriers count both CTAs' copies: let the
                // ones already issued land before the pair leaves
                for (int s = 0; s < P_STAGES; ++s) {
                    volatile int no_abort = 0;
                    mbar_wait(smem_u32(&bars->full[s]), phase ^ (s >= stage ? 1 : 0), status,
                              &no_abort);
                }
            }
            // every release of every stage (the leader's commits) has arrived
            for (int s = 0; s < P_STAGES; ++s) {
                const int uses = issued / P_STAGES + (s < issued % P_STAGES ? 1 : 0);
                if (uses > 0)
                    mbar_wait(smem_u32(&bars->empty[s]), (uint32_t)((uses - 1) & 1), status,
                              abort);
            }
        } else if (GATHER && lane == 1) {
            // forwarder: the gathered rows of each stage, in order, to the
            // leader's full barrier once they have landed
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int g = unit0; g < total && ok; g += units) {
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait(smem_u32(&bars->gfull[stage]), phase, status, abort)) {
                        ok = false;
                        break;
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    mbar_arrive_cluster(cluster_map(smem_u32(&bars->full[stage]), 0));
                    if (++stage == P_STAGES) { stage = 0; phase ^= 1; }
                }
            }
        }
    } else if (warp == 1) {
        // --------------------------------------------- MMA issuer (leader only)
        if (lane == 0 && leader) {
            constexpr uint32_t idesc = idesc_bf16_f32(PM, MMA_N);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int g = unit0; g < total && ok; g += units) {
                uint32_t tdesc = idesc;
                if (kSwap) {
                    const TileMap t = map_pair(g);
                    const int rows_valid = cnt[t.e] - t.m * PM;
                    if (rows_valid <= SWAP_MAX) tdesc = idesc_bf16_f32(PM, swap_cols(rows_valid));
                }
                if (!mbar_wait(smem_u32(&bars->tempty[acc]), acc_phase ^ 1, status, abort)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * ACC_COLS);
                for (int kb = 0; kb < nk; ++kb) {
                    // GATHER: the peer's rows are released at cluster scope
                    if (!mbar_wait<GATHER>(smem_u32(&bars->full[stage]), phase, status, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + (size_t)stage * P_STAGE_BYTES);
                    const uint32_t sb = sa + A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        tc_mma_bf16_pair(d_tmem, sw128_kmajor_desc(sa + kk * 32),
                                         sw128_kmajor_desc(sb + kk * 32), tdesc,
                                         (kb | kk) != 0 ? 1u : 0u);
                    }
                    tc_commit_pair(smem_u32(&bars->empty[stage]));
                    if (++stage == P_STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                tc_commit_pair(smem_u32(&bars->tfull[acc]));
                if (++acc == 2) { acc = 0; acc_phase ^= 1; }
            }
        }
    } else if (GATHER && warp >= 2 + P_EPI_WARPS) {
        // ------------------------------------------- A-row gather (both CTAs)
        const int gt = threadIdx.x - 32 * (2 + P_EPI_WARPS);  // 0..63
        const int chunk = gt & 7;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int g = unit0; g < total && ok; g += units) {
            const TileMap t = map_pair(g);
            const int a_row = offset[t.e] + t.m * PM + (int)rank * BM;
            const int valid_end = offset[t.e] + cnt[t.e];
            const uint16_t *src[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int r = a_row + gt / 8 + 8 * i;
                src[i] = x_rows + (int64_t)(r < valid_end ? row_token[r] : 0) * Kdim + chunk * 8;
            }
            for (int kb = 0; kb < nk; ++kb) {
                if (!mbar_wait(smem_u32(&bars->empty[stage]), phase ^ 1, status, abort)) {
                    ok = false;
                    break;
                }
                const uint32_t sa = smem_u32(smem + (size_t)stage * P_STAGE_BYTES);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int row = gt / 8 + 8 * i;
                    cp_async16_s(sa + (uint32_t)row * 128 + (uint32_t)((chunk ^ (row & 7)) << 4),
                                 src[i] + kb * BK);
                }
                cp_async_arrive_noinc(smem_u32(&bars->gfull[stage]));
                if (++stage == P_STAGES) { stage = 0; phase ^= 1; }
            }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
    } else {
        // ----------------------------------------------- epilogue (both CTAs)
        const int quad = warp & 3;
        const int half = (warp - 2) >> 2;
        const int row_in_tile = (int)rank * BM + quad * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int g = unit0; g < total; g += units) {
            const TileMap t = map_pair(g);
            const int rows_valid = cnt[t.e] - t.m * PM;
            const bool row_ok = row_in_tile < rows_valid;
            const int64_t row = (int64_t)offset[t.e] + t.m * PM + row_in_tile;
            if (!mbar_wait(smem_u32(&bars->tfull[acc]), acc_phase, status, abort)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + ((uint32_t)(quad * 32) << 16) + acc * ACC_COLS;
            if (kSwap && rows_valid <= SWAP_MAX) {
                const int n_sw = swap_cols(rows_valid);
                const int c0 = half * (n_sw / 2), c1 = c0 + n_sw / 2;
                const int64_t row0 = (int64_t)offset[t.e] + t.m * PM;
                if (EPI == EPI_SWIGLU) {
                    // gate warps (quadrants 0-1) pair with the up warps two below them
                    const bool gate_warp = quad < 2;
                    const int xwarp = gate_warp ? warp - 2 : warp;
                    epilogue_swap_swiglu(tbase, c0, c1, rows_valid, row0, gate_warp,
                                         reinterpret_cast<float *>(stage_out + (xwarp - 2) * 2048),
                                         1 + (quad & 1) + 2 * half,
                                         t.n * BN_OUT + 64 * (int)rank + 32 * (quad & 1) + lane,
                                         Nout, lane, out, g_save, u_save);
                } else {
                    epilogue_swap_store(tbase, c0, c1, rows_valid, row0,
                                        t.n * MMA_N + BM * (int)rank + 32 * quad + lane, Nout, out);
                }
            } else if (rows_valid - (row_in_tile - lane) >= 32)  // all 32 rows of this warp are valid
                epilogue_tile_tma<EPI>(tbase, half, (int)(row - lane), t.n, Nout,
                                       stage_out + (warp - 2) * 2048, &tm_o, &tm_g, &tm_u,
                                       g_save != nullptr, lane);
            else
                epilogue_tile<EPI>(tbase, half, row_ok, row, t.n, Nout, out, g_save, u_save);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster_relaxed(cluster_map(smem_u32(&bars->tempty[acc]), 0));
            if (++acc == 2) { acc = 0; acc_phase ^= 1; }
        }
        if (lane == 0) bulk_wait<0>();  // stores complete before the CTA ends
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // both CTAs are done with every barrier and every MMA
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

// ---------------------------------------------------------------- host side --

template <int EPI, bool GATHER>
moe_status launch_gemm_pair(const CUtensorMap &a, const CUtensorMap &b0, const CUtensorMap &b1,
                            const CUtensorMap &o, const CUtensorMap &og, const CUtensorMap &ou,
                            const CUtensorMap &sa0, const CUtensorMap &sa1, const CUtensorMap &sb,
                            int N, int Kdim, int Nout, int max_row_tiles, const int32_t *count,
                            const int32_t *offset, const int32_t *row_token,
                            const uint16_t *x_rows, uint16_t *out, uint16_t *gs, uint16_t *us,
                            int *status, cudaStream_t st) {
    const size_t smem = smem_bytes_pair(N);
    static PerDeviceOnce smem_attr;
    if (!device_once(smem_attr, [] {
            return set_smem_limit(grouped_gemm_pair<EPI, GATHER>, smem_bytes_pair(kMaxN));
        }))
        return MOE_ERR_CUDA;
    constexpr int BN_OUT = EPI == EPI_SWIGLU ? MMA_N / 2 : MMA_N;
    const int64_t max_units = (int64_t)((max_row_tiles + 1) / 2 + N) * ((Nout + BN_OUT - 1) / BN_OUT);
    const int64_t pairs = std::min<int64_t>(num_sms() / 2, std::max<int64_t>(max_units, 1));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * pairs));
    cfg.blockDim = dim3(pair_threads<GATHER>());
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    set_pdl_attr(attr[1]);
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, grouped_gemm_pair<EPI, GATHER>, a, b0, b1, o, og, ou, sa0, sa1,
                           sb, N, Kdim, Nout, count, offset, row_token, x_rows, out, gs, us,
                           status) != cudaSuccess)
        return MOE_ERR_CUDA;
    return launch_status();
}

// row_token[route_row[t, k]] = t for every accepted route (the inverse of the
// route map over the packed rows).
__global__ void __launch_bounds__(256)
invert_route_rows(int64_t routes, int K, const int32_t *__restrict__ route_row,
                  int32_t *__restrict__ row_token) {
    pdl_enter();
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= routes) return;
    const int32_t r = route_row[i];
    if (r >= 0) row_token[r] = (int32_t)(i / K);
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
    const int64_t R = buffer_rows(s);
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
        !make_map(&md, w_down, s->h, (uint64_t)s->N * s->d, MMA_N / 2))
        return MOE_ERR_CUDA;
    CUtensorMap oh, og, ou, oy;
    if (!make_map_bf16_store(&oh, h_act, s->h, R) || !make_map_bf16_store(&oy, y_disp, s->d, R) ||
        !make_map_bf16_store(&og, g_save ? g_save : h_act, s->h, R) ||
        !make_map_bf16_store(&ou, u_save ? u_save : h_act, s->h, R))
        return MOE_ERR_CUDA;
    // swap tiles: weights by 64 (F1) or 128 (F2, md) rows, packed rows by 32
    CUtensorMap sg, su, sx, sh;
    if (!make_map(&sg, w_gate, s->d, (uint64_t)s->N * s->h, 64) ||
        !make_map(&su, w_up, s->d, (uint64_t)s->N * s->h, 64) ||
        !make_map(&sx, x_disp, s->d, R, SW_BOX) || !make_map(&sh, h_act, s->h, R, SW_BOX))
        return MOE_ERR_CUDA;
    int *status = static_cast<int *>(ws);
    const int64_t rows = std::min<int64_t>(R, (int64_t)s->T * s->K);
    const int max_row_tiles = (int)((rows + BM - 1) / BM + s->N);
    r = launch_gemm_pair<EPI_SWIGLU, false>(ma, mg, mu, oh, og, ou, sg, su, sx, s->N, s->d, s->h,
                                            max_row_tiles, expert_count, expert_offset, nullptr,
                                            nullptr, h_act, g_save, u_save, status, stream);
    if (r != MOE_OK) return r;
    return launch_gemm_pair<EPI_STORE, false>(mh, md, md, oy, oy, oy, md, md, sh, s->N, s->h,
                                              s->d, max_row_tiles, expert_count, expert_offset,
                                              nullptr, nullptr, y_disp, nullptr, nullptr, status,
                                              stream);
}

MOE_API size_t moe_expert_ffn_gather_workspace_bytes(const moe_shape *s) {
    if (check_shape(s) != MOE_OK) return 0;
    return 256 + (((size_t)buffer_rows(s) * sizeof(int32_t) + 255) & ~(size_t)255);
}

MOE_API moe_status moe_expert_ffn_gather(const moe_shape *s, const moe_bf16 *x,
                                         const int32_t *route_row, const int32_t *expert_count,
                                         const int32_t *expert_offset, const moe_bf16 *w_gate,
                                         const moe_bf16 *w_up, const moe_bf16 *w_down,
                                         moe_bf16 *h_act, moe_bf16 *g_save, moe_bf16 *u_save,
                                         moe_bf16 *y_disp, void *ws, size_t ws_bytes,
                                         cudaStream_t stream) {
    moe_status r = check_shape(s);
    if (r != MOE_OK) return r;
    if (s->d % BK != 0 || s->h % BK != 0) return MOE_ERR_UNSUPPORTED;
    if (!expert_count || !expert_offset || !ws) return MOE_ERR_INVALID_ARG;
    if ((g_save == nullptr) != (u_save == nullptr)) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < moe_expert_ffn_gather_workspace_bytes(s) ||
        (reinterpret_cast<uintptr_t>(ws) & 255u))
        return MOE_ERR_WORKSPACE;
    const int64_t R = buffer_rows(s);
    if (R == 0 || s->T == 0) return MOE_OK;
    if (!x || !route_row || !w_gate || !w_up || !w_down || !h_act || !y_disp)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(route_row) || !aligned16(w_gate) || !aligned16(w_up) ||
        !aligned16(w_down) || !aligned16(h_act) || !aligned16(y_disp) ||
        (g_save && !aligned16(g_save)) || (u_save && !aligned16(u_save)) ||
        !aligned16(expert_count) || !aligned16(expert_offset))
        return MOE_ERR_ALIGNMENT;
    int32_t *row_token = reinterpret_cast<int32_t *>(static_cast<char *>(ws) + 256);
    CUtensorMap mx, mg, mu, mh, md;
    if (!make_map(&mx, x, s->d, s->T, 1) ||
        !make_map(&mg, w_gate, s->d, (uint64_t)s->N * s->h, 128) ||
        !make_map(&mu, w_up, s->d, (uint64_t)s->N * s->h, 128) ||
        !make_map(&mh, h_act, s->h, R, BM) ||
        !make_map(&md, w_down, s->h, (uint64_t)s->N * s->d, MMA_N / 2))
        return MOE_ERR_CUDA;
    CUtensorMap oh, og, ou, oy;
    if (!make_map_bf16_store(&oh, h_act, s->h, R) || !make_map_bf16_store(&oy, y_disp, s->d, R) ||
        !make_map_bf16_store(&og, g_save ? g_save : h_act, s->h, R) ||
        !make_map_bf16_store(&ou, u_save ? u_save : h_act, s->h, R))
        return MOE_ERR_CUDA;
    int *status = static_cast<int *>(ws);
    const int64_t routes = (int64_t)s->T * s->K;
    launch_pdl(invert_route_rows, (unsigned)((routes + 255) / 256), 256, 0, stream, routes, s->K,
               route_row, row_token);
    if ((r = launch_status()) != MOE_OK) return r;
    const int64_t rows = std::min<int64_t>(R, routes);
    const int max_row_tiles = (int)((rows + BM - 1) / BM + s->N);
    CUtensorMap sh;
    if (!make_map(&sh, h_act, s->h, R, SW_BOX)) return MOE_ERR_CUDA;
    r = launch_gemm_pair<EPI_SWIGLU, true>(mx, mg, mu, oh, og, ou, mg, mu, mx, s->N, s->d, s->h,
                                           max_row_tiles,
                                           expert_count, expert_offset, row_token,
                                           reinterpret_cast<const uint16_t *>(x), h_act, g_save,
                                           u_save, status, stream);
    if (r != MOE_OK) return r;
    return launch_gemm_pair<EPI_STORE, false>(mh, md, md, oy, oy, oy, md, md, sh, s->N, s->h,
                                              s->d, max_row_tiles, expert_count, expert_offset,
                                              nullptr, nullptr, y_disp, nullptr, nullptr, status,
                                              stream);
}
