// Grouped expert GEMMs in MXFP8 (steps F1, F2 of the quantized path).
//
// OLMo-core MoE report, "Section 05: Expert Parallelism": 5.4 (the grouped
// GEMM reads the dispatched E4M3 data and E8M0 scales as they arrived, and
// hands back quantized outputs), 5.8 (both expert GEMMs in MXFP8), Figure 14
// (Linear 1 -> SwiGLU -> Linear 2), 5.7; "Section 08: Synchronization-Free
// Training", 8.5 and Table 14 (device offsets, valid rows only).
//
// Same persistent CTA-pair scheme as the bf16 grouped GEMM (grouped_gemm.cu):
// clusters of two CTAs, M = 256 rows across the pair x N = 256 columns,
// warp 0 TMA producer, warp 1 MMA issuer in the leader, warps 2-9 epilogue,
// work list derived on the device from expert_count.  What changes:
//   - operands are E4M3 codes: a k-block is 128 elements = one 128-byte
//     swizzled row, so each 32 KB stage covers twice the K of a bf16 stage;
//   - each stage also carries this CTA's 512-byte A-scale chunk and the B
//     scales of all 256 columns, which every CTA's tensor memory needs, as
//     the weights store them: each B chunk four times over (4 KB).  The
//     issuer copies the A chunk with tcgen05.cp 32x128b.warpx4 and the B
//     scales with one 128x256b copy (lane L gets 16 bytes of each chunk's
//     copy L / 32, so all four lane quadrants hold them), then runs four
//     tcgen05.mma kind::mxf8f6f4 block_scale instructions (K = 32 each), the
//     k-th reading byte k of each scale word;
//   - the fp32 accumulator (256 columns) is single: the scale ring needs the
//     rest of tensor memory.  The epilogue drains all its columns into
//     registers first and frees the accumulator at once (a relaxed arrival,
//     which does not wait for its earlier stores), so the next tile's MMAs
//     overlap the SwiGLU, quantization and stores;
//   - the epilogue quantizes along its rows in blocks of 32: F1 writes the
//     SwiGLU output H as E4M3 codes plus scale chunks (F2's A operand), F2
//     writes Y as codes plus row-major scale rows for the combine.
#include <algorithm>

#include "../../include/moe_mxfp8.h"
#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int XM = 128;                      // rows per CTA
constexpr int XK = 128;                      // fp8 elements per k-block
constexpr int XN = 256;                      // MMA N
constexpr int XPM = 2 * XM;                  // rows per pair tile
constexpr int X_A_BYTES = XM * XK;           // 16 KB
constexpr int X_B_BYTES = (XN / 2) * XK;     // this CTA's half of B, 16 KB
constexpr int X_AB_BYTES = X_A_BYTES + X_B_BYTES;
// A chunk, then the four copies of the B chunk of columns 0-127 and the four
// of columns 128-255 (as the weights store them)
constexpr int X_SF_BYTES = (1 + 2 * kMxWeightCopies) * kMxChunk;
constexpr int X_STAGES = 5;
constexpr int X_EPI_WARPS = 8;
constexpr int X_THREADS = 64 + 32 * X_EPI_WARPS;
constexpr int X_TMEM_COLS = 512;
constexpr int X_SF_COL0 = 256;  // scale words of stage s at columns 256 + 16 s (A: +0..3, B: +4..11)

enum { XEPI_SWIGLU = 0, XEPI_STORE = 1 };

struct alignas(8) MxBars {
    uint64_t full[X_STAGES];
    uint64_t empty[X_STAGES];
    uint64_t tfull;
    uint64_t tempty;
    uint32_t tmem_base;
    int abort;
};

constexpr size_t smem_bytes_mx(int N) {
    return 1024 + (size_t)X_STAGES * (X_AB_BYTES + X_SF_BYTES) + sizeof(MxBars) +
           2 * sizeof(int32_t) * (N + 1) + 16;
}

struct XTile {
    int e, m, n;
};

// 32 fp32 values of one row -> 32 E4M3 codes (8 words) and the E8M0 byte.
__device__ __forceinline__ uint32_t quant32(const float (&v)[32], uint32_t (&w)[8]) {
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) m = fmaxf(m, fabsf(v[i]));
    const int E = mx_exponent(m);
    const float inv = mx_inv_scale(E);
#pragma unroll
    for (int i = 0; i < 8; ++i)
        w[i] = e4m3x4(v[4 * i] * inv, v[4 * i + 1] * inv, v[4 * i + 2] * inv, v[4 * i + 3] * inv);
    return (uint32_t)(E + 127);
}

__device__ __forceinline__ void store32(uint8_t *dst, const uint32_t (&w)[8]) {
    uint4 *p = reinterpret_cast<uint4 *>(dst);
    p[0] = make_uint4(w[0], w[1], w[2], w[3]);
    p[1] = make_uint4(w[4], w[5], w[6], w[7]);
}

template <int EPI>
__global__ void __launch_bounds__(X_THREADS, 1)
grouped_gemm_mx_pair(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b0,
                     const __grid_constant__ CUtensorMap tm_b1,
                     const __grid_constant__ CUtensorMap tm_sfa,
                     const __grid_constant__ CUtensorMap tm_sfb0,
                     const __grid_constant__ CUtensorMap tm_sfb1, int N, int Kdim, int Nout,
                     const int32_t *__restrict__ count, const int32_t *__restrict__ offset,
                     uint8_t *__restrict__ out_q, uint8_t *__restrict__ out_sf, int *status) {
    pdl_enter();
    constexpr int BN_OUT = EPI == XEPI_SWIGLU ? XN / 2 : XN;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *sf_ring = smem + (size_t)X_STAGES * X_AB_BYTES;
    MxBars *bars = reinterpret_cast<MxBars *>(sf_ring + (size_t)X_STAGES * X_SF_BYTES);
    int32_t *tile_start = reinterpret_cast<int32_t *>(bars + 1);
    int32_t *pad_block = tile_start + (N + 1);
    volatile int *abort = &bars->abort;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const int unit0 = (int)blockIdx.x / 2, units = (int)gridDim.x / 2;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntn = (Nout + BN_OUT - 1) / BN_OUT;
    const int nk = Kdim / XK;
    const int wblocks = Nout / 128;  // 128-row blocks of one expert's weight matrix (B)

    if (threadIdx.x == 0) {
        for (int s = 0; s < X_STAGES; ++s) {
            mbar_init(smem_u32(&bars->full[s]), 1);
            mbar_init(smem_u32(&bars->empty[s]), 1);
        }
        mbar_init(smem_u32(&bars->tfull), 1);
        mbar_init(smem_u32(&bars->tempty), 2 * X_EPI_WARPS);
        bars->abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        // tile_start[e] = pair tiles of experts < e; pad_block[e] = 128-row
        // scale blocks of experts < e
        int carry = 0, carry_b = 0;
        for (int base = 0; base < N; base += 32) {
            const int e = base + lane;
            const int c = e < N ? count[e] : 0;
            const int v = ((c + XPM - 1) / XPM) * ntn;
            const int vb = (c + 127) / 128;
            int incl = v, incl_b = vb;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int u = __shfl_up_sync(0xFFFFFFFFu, incl, off);
                const int ub = __shfl_up_sync(0xFFFFFFFFu, incl_b, off);
                if (lane >= off) {
                    incl += u;
                    incl_b += ub;
                }
            }
            if (e < N) {
                tile_start[e] = carry + incl - v;
                pad_block[e] = carry_b + incl_b - vb;
            }
            carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
            carry_b += __shfl_sync(0xFFFFFFFFu, incl_b, 31);
        }
        if (lane == 0) {
            tile_start[N] = carry;
            pad_block[N] = carry_b;
        }
    }
    if (warp == 1) tmem_alloc_pair(smem_u32(&bars->tmem_base), X_TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem_base = bars->tmem_base;
    const int total = tile_start[N];

    auto map_tile = [&](int g) {
        int lo = 0, hi = N - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (tile_start[mid] <= g) lo = mid;
            else hi = mid - 1;
        }
        const int mt = (count[lo] + XPM - 1) / XPM;
        const int local = g - tile_start[lo];
        return XTile{lo, local % mt, local / mt};
    };

    if (warp == 0) {
        // ------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0) {
            tma_prefetch_desc(&tm_a);
            tma_prefetch_desc(rank && EPI == XEPI_SWIGLU ? &tm_b1 : &tm_b0);
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool ok = true;
            for (int g = unit0; g < total && ok; g += units) {
                const XTile t = map_tile(g);
                const int a_row = offset[t.e] + t.m * XPM + (int)rank * XM;
                const int b_row = EPI == XEPI_SWIGLU ? t.e * Nout + t.n * BN_OUT
                                                     : t.e * Nout + t.n * BN_OUT + (int)rank * (XN / 2);
                const CUtensorMap *mb = rank && EPI == XEPI_SWIGLU ? &tm_b1 : &tm_b0;
                const int sfa_chunk = (pad_block[t.e] + 2 * t.m + (int)rank) * nk;
                const int sfb0_chunk = EPI == XEPI_SWIGLU ? (t.e * wblocks + t.n) * nk
                                                          : (t.e * wblocks + 2 * t.n) * nk;
                const int sfb1_chunk = EPI == XEPI_SWIGLU ? sfb0_chunk : sfb0_chunk + nk;
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait(smem_u32(&bars->empty[stage]), phase ^ 1, status, abort)) {
                        ok = false;
                        break;
                    }
                    const uint32_t own_full = smem_u32(&bars->full[stage]);
                    const uint32_t full = cluster_map(own_full, 0);
                    const uint32_t sa = smem_u32(smem + (size_t)stage * X_AB_BYTES);
                    const uint32_t sb = sa + X_A_BYTES;
                    const uint32_t ss = smem_u32(sf_ring + (size_t)stage * X_SF_BYTES);
                    if (leader) mbar_arrive_expect_tx(own_full, 2 * (X_AB_BYTES + X_SF_BYTES));
                    tma_load_2d_pair(sa, &tm_a, full, kb * XK, a_row);
                    tma_load_2d_pair(sb, mb, full, kb * XK, b_row);
                    tma_load_2d_pair(ss, &tm_sfa, full, 0, sfa_chunk + kb);
                    tma_load_2d_pair(ss + kMxChunk, &tm_sfb0, full, 0,
                                     (sfb0_chunk + kb) * kMxWeightCopies);
                    tma_load_2d_pair(ss + (1 + kMxWeightCopies) * kMxChunk, &tm_sfb1, full, 0,
                                     (sfb1_chunk + kb) * kMxWeightCopies);
                    ++issued;
                    if (++stage == X_STAGES) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok && leader) {
                for (int s = 0; s < X_STAGES; ++s) {
                    volatile int no_abort = 0;
                    mbar_wait(smem_u32(&bars->full[s]), phase ^ (s >= stage ? 1 : 0), status,
                              &no_abort);
                }
            }
            for (int s = 0; s < X_STAGES; ++s) {
                const int uses = issued / X_STAGES + (s < issued % X_STAGES ? 1 : 0);
                if (uses > 0)
                    mbar_wait(smem_u32(&bars->empty[s]), (uint32_t)((uses - 1) & 1), status, abort);
            }
        }
    } else if (warp == 1) {
        // -------------------------------------------------- MMA issuer (leader only)
        if (lane == 0 && leader) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int g = unit0; g < total && ok; g += units) {
                if (!mbar_wait(smem_u32(&bars->tempty), acc_phase ^ 1, status, abort)) break;
                tc_fence_after();
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait(smem_u32(&bars->full[stage]), phase, status, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + (size_t)stage * X_AB_BYTES);
                    const uint32_t sb = sa + X_A_BYTES;
                    const uint32_t ss = smem_u32(sf_ring + (size_t)stage * X_SF_BYTES);
                    const uint32_t sf_t = tmem_base + (uint32_t)(X_SF_COL0 + 16 * stage);
                    tc_cp_chunk_pair(sf_t, chunk_desc(ss));
                    tc_cp_sfb_pair(sf_t + 4, sfb_desc(ss + kMxChunk));
#pragma unroll
                    for (int kk = 0; kk < XK / 32; ++kk)
                        tc_mma_mxf8_pair(tmem_base, sw128_kmajor_desc(sa + kk * 32),
                                         sw128_kmajor_desc(sb + kk * 32), idesc_mxf8(XPM, XN, kk),
                                         sf_t, sf_t + 4, (kb | kk) != 0 ? 1u : 0u);
                    tc_commit_pair(smem_u32(&bars->empty[stage]));
                    if (++stage == X_STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                tc_commit_pair(smem_u32(&bars->tfull));
                acc_phase ^= 1;
            }
        }
    } else {
        // --------------------------------------------------- epilogue (both CTAs)
        const int quad = warp & 3;
        const int half = (warp - 2) >> 2;
        const int r_in = quad * 32 + lane;  // row within this CTA's 128
        uint32_t acc_phase = 0;
        for (int g = unit0; g < total; g += units) {
            const XTile t = map_tile(g);
            const int rows_valid = count[t.e] - t.m * XPM;
            const bool row_ok = (int)rank * XM + r_in < rows_valid;
            const int64_t row = (int64_t)offset[t.e] + t.m * XPM + (int)rank * XM + r_in;
            if (!mbar_wait(smem_u32(&bars->tfull), acc_phase, status, abort)) break;
            tc_fence_after();
            const uint32_t tq = tmem_base + ((uint32_t)(quad * 32) << 16);
            uint32_t v[8][16];
            if (EPI == XEPI_SWIGLU) {
                // gate columns [64 half, +64) and the up columns 128 further
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    tmem_ld16(tq + half * 64 + 16 * j, v[j]);
                    tmem_ld16(tq + 128 + half * 64 + 16 * j, v[4 + j]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 8; ++j) tmem_ld16(tq + half * 128 + 16 * j, v[j]);
            }
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 8; ++j) reg_fence(v[j]);
            tc_fence_before();
            __syncwarp();
            // relaxed: the loads above have completed (tcgen05.wait::ld), and
            // the previous tile's stores need not be complete before the MMA
            // of the next tile may overwrite the accumulator
            if (lane == 0) mbar_arrive_cluster_relaxed(cluster_map(smem_u32(&bars->tempty), 0));
            acc_phase ^= 1;
            if (!row_ok) continue;
            if (EPI == XEPI_SWIGLU) {
                const int col0 = t.n * BN_OUT + half * 64;  // first of this warp's 64 H columns
                if (col0 >= Nout) continue;
                uint32_t sbytes = 0;
#pragma unroll
                for (int b = 0; b < 2; ++b) {
                    float hv[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float gg = __uint_as_float(v[2 * b + i / 16][i % 16]);
                        const float uu = __uint_as_float(v[4 + 2 * b + i / 16][i % 16]);
                        hv[i] = __fdividef(gg, 1.0f + __expf(-gg)) * uu;
                    }
                    uint32_t w[8];
                    sbytes |= quant32(hv, w) << (8 * b);
                    store32(out_q + row * Nout + col0 + 32 * b, w);
                }
                // H scale chunk: block pad_block[e] + 2m + rank, row r_in, blocks col0/32, +1
                const int64_t blk = pad_block[t.e] + 2 * t.m + (int)rank;
                *reinterpret_cast<uint16_t *>(out_sf + mx_chunk_byte(blk, Nout, r_in, col0 / 32)) =
                    (uint16_t)sbytes;
            } else {
                const int col0 = t.n * BN_OUT + half * 128;  // first of this warp's 128 Y columns
                if (col0 >= Nout) continue;
                uint32_t sbytes = 0;
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    float yv[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) yv[i] = __uint_as_float(v[2 * b + i / 16][i % 16]);
                    uint32_t w[8];
                    sbytes |= quant32(yv, w) << (8 * b);
                    store32(out_q + row * Nout + col0 + 32 * b, w);
                }
                *reinterpret_cast<uint32_t *>(out_sf + row * (Nout / 32) + col0 / 32) = sbytes;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, X_TMEM_COLS);
    }
}

template <int EPI>
moe_status launch_gemm_mx(const CUtensorMap &a, const CUtensorMap &b0, const CUtensorMap &b1,
                          const CUtensorMap &sfa, const CUtensorMap &sfb0, const CUtensorMap &sfb1,
                          int N, int Kdim, int Nout, int max_row_tiles, const int32_t *count,
                          const int32_t *offset, uint8_t *out_q, uint8_t *out_sf, int *status,
                          cudaStream_t st) {
    static PerDeviceOnce smem_attr;
    if (!device_once(smem_attr, [] {
            return set_smem_limit(grouped_gemm_mx_pair<EPI>, smem_bytes_mx(kMaxN));
        }))
        return MOE_ERR_CUDA;
    constexpr int BN_OUT = EPI == XEPI_SWIGLU ? XN / 2 : XN;
    const int64_t max_units = (int64_t)((max_row_tiles + 1) / 2 + N) * ((Nout + BN_OUT - 1) / BN_OUT);
    const int64_t pairs = std::min<int64_t>(num_sms() / 2, std::max<int64_t>(max_units, 1));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * pairs));
    cfg.blockDim = dim3(X_THREADS);
    cfg.dynamicSmemBytes = smem_bytes_mx(N);
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    set_pdl_attr(attr[1]);
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, grouped_gemm_mx_pair<EPI>, a, b0, b1, sfa, sfb0, sfb1, N, Kdim,
                           Nout, count, offset, out_q, out_sf, status) != cudaSuccess)
        return MOE_ERR_CUDA;
    return launch_status();
}

}  // namespace
}  // namespace moe

using namespace moe;

MOE_API moe_status moe_expert_ffn_mxfp8(const moe_shape *s, const uint8_t *x_q, const uint8_t *x_sf,
                                        const int32_t *expert_count, const int32_t *expert_offset,
                                        const uint8_t *w_gate_q, const uint8_t *w_gate_sf,
                                        const uint8_t *w_up_q, const uint8_t *w_up_sf,
                                        const uint8_t *w_down_q, const uint8_t *w_down_sf,
                                        uint8_t *h_q, uint8_t *h_sf, uint8_t *y_q,
                                        uint8_t *y_scale, void *ws, size_t ws_bytes,
                                        cudaStream_t stream) {
    moe_status r = check_shape(s);
    if (r != MOE_OK) return r;
    if (s->d % 128 != 0 || s->h % 128 != 0) return MOE_ERR_UNSUPPORTED;
    if (!expert_count || !expert_offset || !ws) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < 256 || (reinterpret_cast<uintptr_t>(ws) & 255u)) return MOE_ERR_WORKSPACE;
    const int64_t R = buffer_rows(s);
    if (R == 0 || s->T == 0) return MOE_OK;
    if (!x_q || !x_sf || !w_gate_q || !w_gate_sf || !w_up_q || !w_up_sf || !w_down_q ||
        !w_down_sf || !h_q || !h_sf || !y_q || !y_scale)
        return MOE_ERR_INVALID_ARG;
    if (!aligned16(x_q) || !aligned16(x_sf) || !aligned16(w_gate_q) || !aligned16(w_gate_sf) ||
        !aligned16(w_up_q) || !aligned16(w_up_sf) || !aligned16(w_down_q) ||
        !aligned16(w_down_sf) || !aligned16(h_q) || !aligned16(h_sf) || !aligned16(y_q) ||
        !aligned16(y_scale) || !aligned16(expert_count) || !aligned16(expert_offset))
        return MOE_ERR_ALIGNMENT;
    const int d = s->d, h = s->h, N = s->N;
    const uint64_t act_blocks = (uint64_t)((R + 127) / 128 + N);
    CUtensorMap ma, mg, mu, mh, md, sx, sg, su, sh, sd;
    if (!make_map_u8(&ma, x_q, d, R, XM) || !make_map_u8(&mg, w_gate_q, d, (uint64_t)N * h, 128) ||
        !make_map_u8(&mu, w_up_q, d, (uint64_t)N * h, 128) || !make_map_u8(&mh, h_q, h, R, XM) ||
        !make_map_u8(&md, w_down_q, h, (uint64_t)N * d, XN / 2) ||
        !make_map_chunks(&sx, x_sf, act_blocks * (d / 128)) ||
        !make_map_chunks(&sg, w_gate_sf, (uint64_t)N * (h / 128) * (d / 128) * kMxWeightCopies,
                         kMxWeightCopies) ||
        !make_map_chunks(&su, w_up_sf, (uint64_t)N * (h / 128) * (d / 128) * kMxWeightCopies,
                         kMxWeightCopies) ||
        !make_map_chunks(&sh, h_sf, act_blocks * (h / 128)) ||
        !make_map_chunks(&sd, w_down_sf, (uint64_t)N * (d / 128) * (h / 128) * kMxWeightCopies,
                         kMxWeightCopies))
        return MOE_ERR_CUDA;
    int *status = static_cast<int *>(ws);
    const int64_t rows = std::min<int64_t>(R, (int64_t)s->T * s->K);
    const int max_row_tiles = (int)((rows + XM - 1) / XM + N);
    r = launch_gemm_mx<XEPI_SWIGLU>(ma, mg, mu, sx, sg, su, N, d, h, max_row_tiles, expert_count,
                                    expert_offset, h_q, h_sf, status, stream);
    if (r != MOE_OK) return r;
    return launch_gemm_mx<XEPI_STORE>(mh, md, md, sh, sd, sd, N, h, d, max_row_tiles, expert_count,
                                      expert_offset, y_q, y_scale, status, stream);
}
