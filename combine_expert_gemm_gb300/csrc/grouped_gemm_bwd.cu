// Grouped expert backward (step B2): data gradients and weight gradients of
// the bias-free SwiGLU experts over the packed capacity buffers.
//
// OLMo-core MoE report, "Section 05: Expert Parallelism", 5.7 (expert backward
// receives the real per-expert row offsets; the weight-gradient GEMM skips the
// unwritten tail of the capacity buffer); Figure 14 (Linear 1 -> SwiGLU ->
// Linear 2); "Section 08: Synchronization-Free Training", 8.5 (grouped GEMMs
// driven by device offsets).  For expert e with rows X, saved G, U, H and
// output gradient dY (all [rows, .]):
//   dH = dY W_down                           (dgrad, M = rows, K = d)
//   dU = dH * silu(G),  dG = dH * U * silu'(G)  (fused into the dH epilogue)
//   dX = dG W_gate + dU W_up                  (dgrad, M = rows, K = 2h)
//   dW_down = dY^T H                          (wgrad, K = rows of e)
//   dW_gate = dG^T X,  dW_up = dU^T X         (wgrad, K = rows of e)
//
// Every kernel runs on CTA pairs like the forward kernel: 256 x 256 output
// tiles, one tcgen05.mma.cta_group::2 per K-step, each CTA holding its own 128
// rows of A and half of B, 32 KB per k-block in a 6-stage ring; persistent,
// 128-byte swizzle, one thread of the leader issuing MMAs into a double-
// buffered TMEM accumulator, eight epilogue warps per CTA whose full 32-row
// output blocks leave through swizzled shared memory by TMA store.  The backward
// operands that are transposed relative to their storage (weights in dgrad,
// activations in wgrad) are read MN-major: a TMA box of 64 M/N elements x 64 K
// rows lands as 64 swizzled 128-byte rows and the MMA descriptor walks it with
// K rows 128 B apart, 8-row groups 1 KB apart and 64-element M/N blocks 8 KB
// apart; each CTA's two blocks of a k-block arrive by one 3-D box.  No
// transposed copy of anything is made.
//
// In wgrad the reduction runs over an expert's rows, so the last k-block of a
// tile can reach into the next expert's rows or the tail (which may hold NaN).
// That block loads through copies of its maps whose row extent ends at the
// expert's last row, so the copy engine fills the rows past it with zeros; the
// leader issues only the 16-row MMA steps that hold valid rows.
#include <algorithm>

#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int MMA_N = 256;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = MMA_N * BK * 2;
constexpr int BLK = 64 * BK * 2;  // one MN-major 64 x 64 block: 8 KB

// 3-D view of a row-major [rows, inner] bf16 matrix (inner a multiple
// of 64) as [inner / 64 blocks][rows][64]: one box of 64 x box_rows x 2
// blocks lands two 64-column blocks of box_rows rows, each 128-byte
// swizzled, exactly where two boxes of make_map at columns x and x + 64 would
// (the swizzle follows the smem row, and a block is a whole number of 8-row
// groups), with one request instead of two.  A block index past the last
// reads as zeros.  Returns false if inner is not a multiple of 64 or the
// driver refuses the map.
inline bool make_map_mn2(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows,
                         uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn || inner % 64 != 0) return false;
    const cuuint64_t dims[3] = {64, rows, inner / 64};
    const cuuint64_t strides[2] = {inner * 2, 128};
    const cuuint32_t box[3] = {64, box_rows, 2};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Load of a 3-D map (make_map_mn2): blocks z and z + 1 of rows y.. into this
// CTA's shared memory, completing on the pair leader's barrier (a cluster
// address).
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap *map,
                                                 uint32_t bar, int32_t x, int32_t y, int32_t z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

constexpr int ACC_COLS = 256;
constexpr int TMEM_COLS = 512;

enum { DGRAD_DH = 0, DGRAD_DX = 1, WGRAD_DOWN = 2, WGRAD_GATEUP = 3 };

template <int MODE>
struct ModeT {
    static constexpr int threads = 64 + 256;  // producer, MMA, 8 epilogue warps
};

// Shared-memory descriptor of an MN-major operand tile (128-byte swizzle):
// each 128-byte row holds 64 M/N elements of one K index; K rows are 128 B
// apart, 8-row groups 1024 B apart (stride-dimension offset), 64-element M/N
// blocks 8 KB apart (leading-dimension offset).
__device__ __forceinline__ uint64_t sw128_mnmajor_desc(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);
    d |= (uint64_t)(BLK >> 4) << 16;
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)2u << 61;
    return d;
}

__host__ __device__ constexpr uint32_t idesc_bf16_f32_major(int M, int N, int a_mn, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

constexpr int kEpiThreads = 256;                      // 8 epilogue warps

struct Params {
    int N, d, h;
    int ntn;       // output column tiles of 256
    int mtn;       // wgrad: output row tiles of 256 (both halves for gate/up)
    const int32_t *count, *offset;
    const uint16_t *g_save, *u_save;  // DGRAD_DH epilogue inputs
    uint16_t *out0, *out1;            // DH: dG, dU; DX: dx_disp
    float *fout0, *fout1;             // wgrad: dW (down) or (gate, up)
    CUtensorMap *map_slots;           // wgrad: kMapSlots x 2 bounded map copies per CTA
    int rows;                         // R: rows of every row buffer (the maps' extent)
    int *status;
};

struct Tile {
    int e, m, n;
};

// wgrad work unit g: expert-major, output-row tiles fastest.
__device__ __forceinline__ Tile map_wgrad_tile(int g, const Params &p) {
    const int tpe = p.mtn * p.ntn;
    const int e = g / tpe, l = g % tpe;
    return Tile{e, l % p.mtn, l / p.mtn};
}

template <int MODE>
__device__ __forceinline__ int k_blocks(const Params &p, int cnt) {
    if (MODE == DGRAD_DH) return p.d / BK;
    if (MODE == DGRAD_DX) return 2 * p.h / BK;
    return (cnt + BK - 1) / BK;
}

// Epilogue of a dgrad tile for one warp: 32 rows (TMEM lanes) and one half of
// the 256 columns, in 32-column chunks.  DGRAD_DH: dU = dH * silu(G) and
// dG = dH * U * silu'(G) from the saved G, U; DGRAD_DX: a bf16 copy of dX.
// When all 32 rows of the warp are valid each output chunk goes through the
// warp's 2 KB shared-memory block and out by one TMA instruction; otherwise
// the valid rows store their own 64 bytes.  DGRAD_DH: the saved G, U of the next chunk are fetched
// while the current one is computed (slots gq/uq[ch & 1]); the first chunk's
// were fetched into slot 0 by the caller before the accumulator was ready.
template <int MODE>
__device__ __forceinline__ void dgrad_epilogue_tma(uint32_t tbase, int half, int64_t row, int row0,
                                                   int n, const Params &p, uint8_t *blk,
                                                   const CUtensorMap *m0, const CUtensorMap *m1,
                                                   uint4 (&gq)[2][4], uint4 (&uq)[2][4], bool full,
                                                   bool row_ok, int lane) {
    constexpr int NCH = (MMA_N / 2) / 32;
    const int width = MODE == DGRAD_DH ? p.h : p.d;
    // a 32-column bf16 chunk of this lane's row: the warp's TMA block when all
    // 32 rows are valid, else four 16-byte stores of the valid rows
    auto put = [&](const uint32_t (&w)[16], const CUtensorMap *m, uint16_t *base, int ld, int col) {
        if (full) {
            warp_store_bf16_32x32(blk, w, m, col, row0, lane);
        } else if (row_ok) {
            uint4 *dst = reinterpret_cast<uint4 *>(base + row * ld + col);
#pragma unroll
            for (int q = 0; q < 4; ++q) dst[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
        }
    };
#pragma unroll
    for (int ch = 0; ch < NCH; ++ch) {
        const int c = half * (MMA_N / 2) + ch * 32;
        if (MODE == DGRAD_DH && ch + 1 < NCH) {
            const int ncol = n * MMA_N + c + 32;
            if (ncol < width && row_ok) {
                const uint4 *gp = reinterpret_cast<const uint4 *>(p.g_save + row * p.h + ncol);
                const uint4 *up = reinterpret_cast<const uint4 *>(p.u_save + row * p.h + ncol);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    gq[(ch + 1) & 1][i] = __ldcs(gp + i);
                    uq[(ch + 1) & 1][i] = __ldcs(up + i);
                }
            }
        }
        uint32_t r0[16], r1[16];
        tmem_ld16(tbase + c, r0);
        tmem_ld16(tbase + c + 16, r1);
        tmem_ld_wait();
        reg_fence(r0);
        reg_fence(r1);
        const int col = n * MMA_N + c;
        if (col >= width) continue;  // warp-uniform
        if (MODE == DGRAD_DH) {
            const uint32_t *gw = reinterpret_cast<const uint32_t *>(gq[ch & 1]);
            const uint32_t *uw = reinterpret_cast<const uint32_t *>(uq[ch & 1]);
            uint32_t dg[16], du[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float rg[2], ru[2];
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const float z = hf ? bf16_hi(gw[i]) : bf16_lo(gw[i]);
                    const float u = hf ? bf16_hi(uw[i]) : bf16_lo(uw[i]);
                    const uint32_t rv = i < 8 ? r0[2 * i + hf] : r1[2 * (i - 8) + hf];
                    const float dh = __uint_as_float(rv);
                    const float sg = __fdividef(1.0f, 1.0f + __expf(-z));
                    ru[hf] = dh * (z * sg);
                    rg[hf] = dh * u * sg * (1.0f + z * (1.0f - sg));
                }
                dg[i] = pack_bf16x2(rg[0], rg[1]);
                du[i] = pack_bf16x2(ru[0], ru[1]);
            }
            put(dg, m0, p.out0, p.h, col);
            put(du, m1, p.out1, p.h, col);
        } else {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                pk[i] = pack_bf16x2(__uint_as_float(r0[2 * i]), __uint_as_float(r0[2 * i + 1]));
                pk[8 + i] = pack_bf16x2(__uint_as_float(r1[2 * i]), __uint_as_float(r1[2 * i + 1]));
            }
            put(pk, m0, p.out0, p.d, col);
        }
    }
}

// --------------------------------------------------------- CTA-pair dgrad
//
// dH and dX on CTA pairs, as in the forward kernel: each 256-row x 256-column
// tile is one tcgen05.mma.cta_group::2 per K-step; each CTA holds its own 128
// rows of A (K-major) and half of B (two 64-column MN-major blocks of the
// transposed weight), 32 KB per k-block in a 6-stage ring.  The leader issues
// the MMAs; both CTAs' loads complete on the leader's full barrier; the
// leader's commits release stages and accumulators in both CTAs.
constexpr int P_STAGES = 6;
constexpr int P_STAGE_BYTES = A_BYTES + B_BYTES / 2;  // 32 KB
constexpr int P_EPI_WARPS = kEpiThreads / 32;

struct alignas(8) PairBars {
    uint64_t full[P_STAGES];
    uint64_t empty[P_STAGES];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint32_t tmem_base;
    int abort;
};

constexpr int P_STG_BYTES = P_EPI_WARPS * 2048;  // one 32 x 32 bf16 store block per epilogue warp

constexpr size_t smem_bytes_pair(int N) {
    return 1024 + (size_t)P_STAGES * P_STAGE_BYTES + P_STG_BYTES + sizeof(PairBars) +
           sizeof(int32_t) * (N + 1) + 16;
}

template <int MODE>
__global__ void __launch_bounds__(ModeT<MODE>::threads, 1)
grouped_dgrad_pair(const __grid_constant__ CUtensorMap tm_a0, const __grid_constant__ CUtensorMap tm_a1,
                   const __grid_constant__ CUtensorMap tm_b0, const __grid_constant__ CUtensorMap tm_b1,
                   const __grid_constant__ CUtensorMap tm_o0, const __grid_constant__ CUtensorMap tm_o1,
                   const Params p) {
    pdl_enter();
    static_assert(MODE == DGRAD_DH || MODE == DGRAD_DX, "dgrad only");
    constexpr int PM = 2 * BM;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *stage_out = smem + (size_t)P_STAGES * P_STAGE_BYTES;  // [8 warps][2 KB]
    PairBars *bars = reinterpret_cast<PairBars *>(stage_out + P_STG_BYTES);
    int32_t *tile_start = reinterpret_cast<int32_t *>(bars + 1);
    volatile int *abort = &bars->abort;
    int *status = p.status;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const int unit0 = (int)blockIdx.x / 2, units = (int)gridDim.x / 2;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < P_STAGES; ++s) {
            mbar_init(smem_u32(&bars->full[s]), 1);
            mbar_init(smem_u32(&bars->empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&bars->tfull[b]), 1);
            mbar_init(smem_u32(&bars->tempty[b]), 2 * P_EPI_WARPS);
        }
        bars->abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        int carry = 0;
        for (int base = 0; base < p.N; base += 32) {
            const int e = base + lane;
            const int v = e < p.N ? ((p.count[e] + PM - 1) / PM) * p.ntn : 0;
            int incl = v;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int u = __shfl_up_sync(0xFFFFFFFFu, incl, off);
                if (lane >= off) incl += u;
            }
            if (e < p.N) tile_start[e] = carry + incl - v;
            carry += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
        if (lane == 0) tile_start[p.N] = carry;
    }
    if (warp == 1) tmem_alloc_pair(smem_u32(&bars->tmem_base), TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem_base = bars->tmem_base;
    const int total = tile_start[p.N];
    const int nk = k_blocks<MODE>(p, 0);
    const int hb = p.h / BK;

    auto map_pair = [&](int g) {
        int lo = 0, hi = p.N - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (tile_start[mid] <= g) lo = mid;
            else hi = mid - 1;
        }
        const int mt = (p.count[lo] + PM - 1) / PM;
        const int l = g - tile_start[lo];
        return Tile{lo, l % mt, l / mt};
    };

    if (warp == 0) {
        if (lane == 0) {
            tma_prefetch_desc(&tm_a0);
            tma_prefetch_desc(&tm_b0);
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            bool ok = true;
            for (int g = unit0; g < total && ok; g += units) {
                const Tile t = map_pair(g);
                const int a_row = p.offset[t.e] + t.m * PM + (int)rank * BM;
                const int ncol = t.n * MMA_N + (int)rank * (MMA_N / 2);
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait(smem_u32(&bars->empty[stage]), phase ^ 1, status, abort)) {
                        ok = false;
                        break;
                    }
                    const uint32_t own_full = smem_u32(&bars->full[stage]);
                    const uint32_t full = cluster_map(own_full, 0);
                    const uint32_t sa = smem_u32(smem + (size_t)stage * P_STAGE_BYTES);
                    const uint32_t sb = sa + A_BYTES;
                    if (leader) mbar_arrive_expect_tx(own_full, 2 * P_STAGE_BYTES);
                    const bool up = MODE == DGRAD_DX && kb >= hb;
                    const int kk = up ? kb - hb : kb;
                    const int brow = MODE == DGRAD_DH ? t.e * p.d + kb * BK : t.e * p.h + kk * BK;
                    tma_load_2d_pair(sa, up ? &tm_a1 : &tm_a0, full, kk * BK, a_row);
                    // both 64-column blocks of this CTA's half of B (make_map_mn2)
                    tma_load_3d_pair(sb, up ? &tm_b1 : &tm_b0, full, 0, brow, ncol / 64);
                    ++issued;
                    if (++stage == P_STAGES) { stage = 0; phase ^= 1; }
                }
            }
            if (!ok && leader) {
                for (int s = 0; s < P_STAGES; ++s) {
                    volatile int no_abort = 0;
                    mbar_wait(smem_u32(&bars->full[s]), phase ^ (s >= stage ? 1 : 0), status,
                              &no_abort);
                }
            }
            for (int s = 0; s < P_STAGES; ++s) {
                const int uses = issued / P_STAGES + (s < issued % P_STAGES ? 1 : 0);
                if (uses > 0)
                    mbar_wait(smem_u32(&bars->empty[s]), (uint32_t)((uses - 1) & 1), status, abort);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            constexpr uint32_t idesc = idesc_bf16_f32_major(PM, MMA_N, 0, 1);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int g = unit0; g < total && ok; g += units) {
                if (!mbar_wait(smem_u32(&bars->tempty[acc]), acc_phase ^ 1, status, abort)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * ACC_COLS);
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait(smem_u32(&bars->full[stage]), phase, status, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + (size_t)stage * P_STAGE_BYTES);
                    const uint32_t sb = sa + A_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        tc_mma_bf16_pair(d_tmem, sw128_kmajor_desc(sa + kk * 32),
                                         sw128_mnmajor_desc(sb + kk * 2048), idesc,
                                         (kb | kk) != 0 ? 1u : 0u);
                    tc_commit_pair(smem_u32(&bars->empty[stage]));
                    if (++stage == P_STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                tc_commit_pair(smem_u32(&bars->tfull[acc]));
                if (++acc == 2) { acc = 0; acc_phase ^= 1; }
            }
        }
    } else {
        const int quad = warp & 3;
        const int half = (warp - 2) >> 2;
        const int rit = (int)rank * BM + quad * 32 + lane;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int g = unit0; g < total; g += units) {
            const Tile t = map_pair(g);
            const int cnt = p.count[t.e], off = p.offset[t.e];
            const bool row_ok = rit < cnt - t.m * PM;
            const int64_t row = (int64_t)off + t.m * PM + rit;
            const bool full_block = cnt - t.m * PM - (rit - lane) >= 32;  // all 32 rows valid
            uint4 gq[2][4], uq[2][4];
            if (MODE == DGRAD_DH && row_ok) {
                // the first chunk's saved G, U, fetched before the accumulator is ready
                const int col = t.n * MMA_N + half * (MMA_N / 2);
                if (col < p.h) {
                    const uint4 *gp = reinterpret_cast<const uint4 *>(p.g_save + row * p.h + col);
                    const uint4 *up = reinterpret_cast<const uint4 *>(p.u_save + row * p.h + col);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        gq[0][i] = __ldcs(gp + i);
                        uq[0][i] = __ldcs(up + i);
                    }
                }
            }
            if (!mbar_wait(smem_u32(&bars->tfull[acc]), acc_phase, status, abort)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + ((uint32_t)(quad * 32) << 16) + acc * ACC_COLS;
            dgrad_epilogue_tma<MODE>(tbase, half, row, (int)(row - lane), t.n, p,
                                     stage_out + (warp - 2) * 2048, &tm_o0, &tm_o1, gq, uq,
                                     full_block, row_ok, lane);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster_relaxed(cluster_map(smem_u32(&bars->tempty[acc]), 0));
            if (++acc == 2) { acc = 0; acc_phase ^= 1; }
        }
        if (lane == 0) bulk_wait<0>();  // stores complete before the CTA ends
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

template <int MODE>
moe_status launch_dgrad_pair(const CUtensorMap &a0, const CUtensorMap &a1, const CUtensorMap &b0,
                             const CUtensorMap &b1, const CUtensorMap &o0, const CUtensorMap &o1,
                             const Params &p, int max_units, cudaStream_t st) {
    const size_t smem = smem_bytes_pair(p.N);
    static PerDeviceOnce smem_attr;
    if (!device_once(smem_attr, [] {
            return set_smem_limit(grouped_dgrad_pair<MODE>, smem_bytes_pair(kMaxN));
        }))
        return MOE_ERR_CUDA;
    const int pairs = std::min(num_sms() / 2, std::max(max_units, 1));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * pairs));
    cfg.blockDim = dim3(ModeT<MODE>::threads);
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
    if (cudaLaunchKernelEx(&cfg, grouped_dgrad_pair<MODE>, a0, a1, b0, b1, o0, o1, p) != cudaSuccess)
        return MOE_ERR_CUDA;
    return launch_status();
}

// --------------------------------------------------------- CTA-pair wgrad
//
// dW tiles of 256 output rows x 256 output columns, one tcgen05.mma
// cta_group::2 per 16 rows of the expert: each CTA holds its own 128 output
// rows of A and 128 output columns of B, both MN-major (two 64 x 64 blocks
// each), 32 KB per k-block in the 6-stage ring; both CTAs' copies complete on
// the leader's full barrier, as in the dgrad kernel.  The reduction runs over
// the expert's rows, and a tile's last k-block may reach into the next
// expert's rows or the unwritten tail.  That block is loaded through copies
// of the two maps whose row extent ends at the expert's last row, so the rows
// past it arrive as zeros: the producer warp writes the copies into this
// CTA's ring of kMapSlots global slots (tensormap.replace on a shared-memory
// copy of the kernel's map, then a release copy to the tensormap proxy) and
// acquires them before the load.  A slot is rewritten kMapSlots tiles later,
// when the producer has long since waited for the stage its load filled.
constexpr int WG_STAGES = 6;
constexpr int kMapSlots = WG_STAGES + 2;
constexpr int kMaxWgradCtas = 512;
constexpr size_t kMapSlotBytes = (size_t)kMaxWgradCtas * kMapSlots * 2 * sizeof(CUtensorMap);

struct alignas(128) WgradBars {
    CUtensorMap stage_map[2];   // the producer's copies being bounded (A, B)
    uint64_t full[WG_STAGES];   // leader: both CTAs' copies of a k-block landed
    uint64_t empty[WG_STAGES];  // the leader's MMAs are done with the stage
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint32_t tmem_base;
    int abort;
};

constexpr int WG_THREADS = 64 + kEpiThreads;

constexpr int WG_STG_BYTES = P_EPI_WARPS * 32 * 32 * 4;  // one 32 x 32 fp32 block per warp

constexpr size_t smem_bytes_wgrad_pair() {
    return 1024 + (size_t)WG_STAGES * P_STAGE_BYTES + WG_STG_BYTES + sizeof(WgradBars) + 16;
}

// Row extent (dimension 1) of the map copy at smem address `map`.
__device__ __forceinline__ void tmap_set_rows(uint32_t map, int rows) {
    asm volatile("tensormap.replace.tile.global_dim.shared::cta.b1024.b32 [%0], 1, %1;" ::"r"(map),
                 "r"(rows)
                 : "memory");
}
// The whole warp: copies the 128-byte map at smem `src` to global `dst` and
// releases it to the tensormap proxy at GPU scope.
__device__ __forceinline__ void tmap_publish(CUtensorMap *dst, uint32_t src) {
    asm volatile(
        "tensormap.cp_fenceproxy.global.shared::cta.tensormap::generic.release.gpu.sync.aligned"
        " [%0], [%1], 128;" ::"l"(dst),
        "r"(src)
        : "memory");
}
// The thread about to load through the map at `map` acquires its contents.
__device__ __forceinline__ void tmap_acquire(const CUtensorMap *map) {
    asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(map) : "memory");
}

template <int MODE>
__global__ void __launch_bounds__(WG_THREADS, 1)
grouped_wgrad_pair(const __grid_constant__ CUtensorMap tm_a0, const __grid_constant__ CUtensorMap tm_a1,
                   const __grid_constant__ CUtensorMap tm_b0, const __grid_constant__ CUtensorMap tm_o0,
                   const __grid_constant__ CUtensorMap tm_o1, const Params p) {
    pdl_enter();
    static_assert(MODE == WGRAD_DOWN || MODE == WGRAD_GATEUP, "wgrad only");
    constexpr int PM = 2 * BM;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *stage_out = smem + (size_t)WG_STAGES * P_STAGE_BYTES;
    WgradBars *bars =
        reinterpret_cast<WgradBars *>(smem + (size_t)WG_STAGES * P_STAGE_BYTES + WG_STG_BYTES);
    volatile int *abort = &bars->abort;
    int *status = p.status;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const int unit0 = (int)blockIdx.x / 2, units = (int)gridDim.x / 2;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < WG_STAGES; ++s) {
            mbar_init(smem_u32(&bars->full[s]), 1);
            mbar_init(smem_u32(&bars->empty[s]), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(smem_u32(&bars->tfull[b]), 1);
            mbar_init(smem_u32(&bars->tempty[b]), 2 * P_EPI_WARPS);
        }
        bars->abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc_pair(smem_u32(&bars->tmem_base), TMEM_COLS);
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem_base = bars->tmem_base;
    const int total = p.N * p.mtn * p.ntn;
    const int mt_half = (p.h + PM - 1) / PM;  // gate/up: 256-row tiles per half

    if (warp == 0) {
        // ------------------------------------- TMA producer (the whole warp
        // bounds the maps; lane 0 waits and loads)
        if (lane == 0) {
            tma_prefetch_desc(&tm_a0);
            tma_prefetch_desc(&tm_b0);
        }
        CUtensorMap *slots = p.map_slots + (size_t)blockIdx.x * kMapSlots * 2;
        const uint32_t sm_a = smem_u32(&bars->stage_map[0]), sm_b = smem_u32(&bars->stage_map[1]);
        int stage = 0;
        uint32_t phase = 0;
        int issued = 0, slot = 0;
        bool ok = true;
        for (int g = unit0; g < total && ok; g += units) {
            const Tile t = map_wgrad_tile(g, p);
            const int cnt = p.count[t.e], off = p.offset[t.e];
            const int nk = k_blocks<MODE>(p, cnt);
            if (nk == 0) continue;
            const bool up = MODE == WGRAD_GATEUP && t.m >= mt_half;
            const int mcol = (up ? t.m - mt_half : t.m) * PM + (int)rank * BM;
            const int ncol = t.n * MMA_N + (int)rank * (MMA_N / 2);
            const CUtensorMap *ma = up ? &tm_a1 : &tm_a0;
            CUtensorMap *ga = slots + 2 * slot, *gb = ga + 1;
            if (++slot == kMapSlots) slot = 0;
            if (lane == 0) {
                // never past the buffer's own extent, whatever the counts say
                const int end = max(1, min(off + cnt, p.rows));
                bars->stage_map[0] = *ma;
                bars->stage_map[1] = tm_b0;
                tmap_set_rows(sm_a, end);
                tmap_set_rows(sm_b, end);
            }
            __syncwarp();
            tmap_publish(ga, sm_a);
            tmap_publish(gb, sm_b);
            __syncwarp();
            if (lane == 0) {
                tmap_acquire(ga);
                tmap_acquire(gb);
                for (int kb = 0; kb < nk; ++kb) {
                    if (!mbar_wait(smem_u32(&bars->empty[stage]), phase ^ 1, status, abort)) {
                        ok = false;
                        break;
                    }
                    const uint32_t own_full = smem_u32(&bars->full[stage]);
                    const uint32_t full = cluster_map(own_full, 0);
                    const uint32_t sa = smem_u32(smem + (size_t)stage * P_STAGE_BYTES);
                    const uint32_t sb = sa + A_BYTES;
                    const int row = off + kb * BK;
                    const bool last = kb == nk - 1;  // rows past the expert load as zeros
                    if (leader) mbar_arrive_expect_tx(own_full, 2 * P_STAGE_BYTES);
                    tma_load_3d_pair(sa, last ? ga : ma, full, 0, row, mcol / 64);
                    tma_load_3d_pair(sb, last ? gb : &tm_b0, full, 0, row, ncol / 64);
                    ++issued;
                    if (++stage == WG_STAGES) { stage = 0; phase ^= 1; }
                }
            }
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
        }
        if (lane == 0) {
            if (!ok && leader) {
                // the leader's full barriers count both CTAs' copies: let the
                // ones already issued land before the pair leaves
                for (int s = 0; s < WG_STAGES; ++s) {
                    volatile int no_abort = 0;
                    mbar_wait(smem_u32(&bars->full[s]), phase ^ (s >= stage ? 1 : 0), status,
                              &no_abort);
                }
            }
            // the leader's MMAs read this CTA's stages: wait until every use
            // of every stage has been released before leaving
            for (int s = 0; s < WG_STAGES; ++s) {
                const int uses = issued / WG_STAGES + (s < issued % WG_STAGES ? 1 : 0);
                if (uses > 0)
                    mbar_wait(smem_u32(&bars->empty[s]), (uint32_t)((uses - 1) & 1), status, abort);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------- MMA issuer (leader)
        if (leader && lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32_major(PM, MMA_N, 1, 1);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int g = unit0; g < total && ok; g += units) {
                const Tile t = map_wgrad_tile(g, p);
                const int cnt = p.count[t.e];
                const int nk = k_blocks<MODE>(p, cnt);
                if (!mbar_wait(smem_u32(&bars->tempty[acc]), acc_phase ^ 1, status, abort)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * ACC_COLS);
                for (int kb = 0; kb < nk; ++kb) {
                    // the last block's steps cover its valid rows (the rest are zeros)
                    const int steps = kb == nk - 1 ? (cnt - kb * BK + 15) / 16 : BK / 16;
                    if (!mbar_wait(smem_u32(&bars->full[stage]), phase, status, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + (size_t)stage * P_STAGE_BYTES);
                    const uint32_t sb = sa + A_BYTES;
                    for (int kk = 0; kk < steps; ++kk)
                        tc_mma_bf16_pair(d_tmem, sw128_mnmajor_desc(sa + kk * 2048),
                                         sw128_mnmajor_desc(sb + kk * 2048), idesc,
                                         (kb | kk) != 0 ? 1u : 0u);
                    tc_commit_pair(smem_u32(&bars->empty[stage]));
                    if (++stage == WG_STAGES) { stage = 0; phase ^= 1; }
                }
                if (!ok) break;
                tc_commit_pair(smem_u32(&bars->tfull[acc]));
                if (++acc == 2) { acc = 0; acc_phase ^= 1; }
            }
        }
    } else {
        // --------------------------------------------------------- epilogue
        const int quad = warp & 3;
        const int half = (warp - 2) >> 2;  // which 128 of the 256 columns
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int g = unit0; g < total; g += units) {
            const Tile t = map_wgrad_tile(g, p);
            const int cnt = p.count[t.e];
            if (!mbar_wait(smem_u32(&bars->tfull[acc]), acc_phase, status, abort)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + ((uint32_t)(quad * 32) << 16) + acc * ACC_COLS;
            {
                // weight gradient, fp32; an expert without rows gets zeros.  Each
                // 32 x 32 block is written to this warp's shared-memory block in
                // the 128-byte swizzled layout and stored by one TMA instruction
                // (rows past the matrix are clipped by the map).
                const bool up = MODE == WGRAD_GATEUP && t.m >= mt_half;
                const int mbase = (up ? t.m - mt_half : t.m) * PM + (int)rank * BM + quad * 32;
                const int width = MODE == WGRAD_DOWN ? p.h : p.d;
                const int mlim = MODE == WGRAD_DOWN ? p.d : p.h;
                const CUtensorMap *om = up ? &tm_o1 : &tm_o0;
                uint8_t *blk = stage_out + (warp - 2) * 4096;
                const uint32_t blk_s = smem_u32(blk);
                for (int c = half * (MMA_N / 2); c < (half + 1) * (MMA_N / 2); c += 32) {
                    uint32_t r0[16], r1[16];
                    tmem_ld16(tbase + c, r0);
                    tmem_ld16(tbase + c + 16, r1);
                    tmem_ld_wait();
                    reg_fence(r0);
                    reg_fence(r1);
                    const int col0 = t.n * MMA_N + c;
                    if (col0 >= width || mbase >= mlim) continue;  // warp-uniform
                    // the previous store from this block has finished reading it
                    if (lane == 0) bulk_wait_read<0>();
                    __syncwarp();
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const uint32_t *src = q < 4 ? &r0[4 * q] : &r1[4 * (q - 4)];
                        const uint4 v = cnt ? make_uint4(src[0], src[1], src[2], src[3])
                                            : make_uint4(0, 0, 0, 0);
                        *reinterpret_cast<uint4 *>(blk + lane * 128 + ((q ^ (lane & 7)) * 16)) = v;
                    }
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d(om, blk_s, col0, mbase, t.e);
                        bulk_commit();
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster_relaxed(cluster_map(smem_u32(&bars->tempty[acc]), 0));
            if (++acc == 2) { acc = 0; acc_phase ^= 1; }
        }
        if (lane == 0) bulk_wait<0>();  // stores complete before the CTA ends
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

template <int MODE>
moe_status launch_wgrad_pair(const CUtensorMap &a0, const CUtensorMap &a1, const CUtensorMap &b0,
                             const CUtensorMap &o0, const CUtensorMap &o1, const Params &p,
                             int max_units, cudaStream_t st) {
    const size_t smem = smem_bytes_wgrad_pair();
    static PerDeviceOnce smem_attr;
    if (!device_once(smem_attr, [smem] { return set_smem_limit(grouped_wgrad_pair<MODE>, smem); }))
        return MOE_ERR_CUDA;
    // at most kMaxWgradCtas CTAs: the workspace holds that many map rings
    const int pairs = std::min(std::min(num_sms(), kMaxWgradCtas) / 2, std::max(max_units, 1));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * pairs));
    cfg.blockDim = dim3(WG_THREADS);
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
    if (cudaLaunchKernelEx(&cfg, grouped_wgrad_pair<MODE>, a0, a1, b0, o0, o1, p) != cudaSuccess)
        return MOE_ERR_CUDA;
    return launch_status();
}

inline size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

}  // namespace
}  // namespace moe

using namespace moe;

MOE_API size_t moe_expert_ffn_backward_workspace_bytes(const moe_shape *s) {
    if (check_shape(s) != MOE_OK) return 0;
    const size_t R = (size_t)buffer_rows(s);
    return 256 + 2 * align256(R * s->h * 2) + kMapSlotBytes;
}

MOE_API moe_status moe_expert_ffn_backward(
    const moe_shape *s, const moe_bf16 *x_disp, const int32_t *expert_count,
    const int32_t *expert_offset, const moe_bf16 *w_gate, const moe_bf16 *w_up,
    const moe_bf16 *w_down, const moe_bf16 *g_save, const moe_bf16 *u_save, const moe_bf16 *h_act,
    const moe_bf16 *dy_disp, moe_bf16 *dx_disp, float *dw_gate, float *dw_up, float *dw_down,
    void *ws, size_t ws_bytes, cudaStream_t stream) {
    moe_status r = check_shape(s);
    if (r != MOE_OK) return r;
    if (s->d % BK != 0 || s->h % BK != 0) return MOE_ERR_UNSUPPORTED;
    if (!expert_count || !expert_offset || !ws || !w_gate || !w_up || !w_down || !dw_gate ||
        !dw_up || !dw_down)
        return MOE_ERR_INVALID_ARG;
    const int64_t R = buffer_rows(s);
    if (R > 0 && (!x_disp || !g_save || !u_save || !h_act || !dy_disp || !dx_disp))
        return MOE_ERR_INVALID_ARG;
    if (ws_bytes < moe_expert_ffn_backward_workspace_bytes(s) ||
        (reinterpret_cast<uintptr_t>(ws) & 255u))
        return MOE_ERR_WORKSPACE;
    const void *ptrs[] = {x_disp, w_gate, w_up, w_down, g_save, u_save, h_act, dy_disp, dx_disp,
                          dw_gate, dw_up, dw_down, expert_count, expert_offset};
    for (const void *q : ptrs)
        if (!aligned16(q)) return MOE_ERR_ALIGNMENT;

    Params p{};
    p.N = s->N;
    p.d = s->d;
    p.h = s->h;
    p.count = expert_count;
    p.offset = expert_offset;
    p.status = static_cast<int *>(ws);
    p.rows = (int)buffer_rows(s);
    uint16_t *dG = reinterpret_cast<uint16_t *>(static_cast<char *>(ws) + 256);
    uint16_t *dU = reinterpret_cast<uint16_t *>(static_cast<char *>(ws) + 256 +
                                                align256((size_t)R * s->h * 2));
    p.map_slots = reinterpret_cast<CUtensorMap *>(static_cast<char *>(ws) + 256 +
                                                  2 * align256((size_t)R * s->h * 2));
    const int64_t rows = std::min<int64_t>(R, (int64_t)s->T * s->K);
    const int row_tiles = (int)((rows + BM - 1) / BM + s->N);
    const int wg_mt = 2 * ((s->h + 2 * BM - 1) / (2 * BM));

    if (R == 0) {
        // no rows at all: every weight gradient is zero; the weight-gradient
        // kernels need row buffers for their maps, so the outputs are cleared
        // directly.
        const size_t hd = (size_t)s->N * s->h * s->d * sizeof(float);
        if (cudaMemsetAsync(dw_gate, 0, hd, stream) != cudaSuccess ||
            cudaMemsetAsync(dw_up, 0, hd, stream) != cudaSuccess ||
            cudaMemsetAsync(dw_down, 0, hd, stream) != cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_OK;
    }

    CUtensorMap dy_k, wd_mn, dg_k, du_k, wg_mn, wu_mn, dy_mn, h_mn, dg_mn, du_mn, x_mn;
    const uint64_t Nd = (uint64_t)s->N * s->d, Nh = (uint64_t)s->N * s->h;
    // MN-major operands as 3-D two-block maps (d and h are multiples of 64
    // here): each CTA's two 64-column blocks of a k-block arrive by one request
    // instead of two, about 1% off the expert backward on the training layer
    if (!make_map(&dy_k, dy_disp, s->d, R, BM) || !make_map(&dg_k, dG, s->h, R, BM) ||
        !make_map(&du_k, dU, s->h, R, BM) || !make_map_mn2(&wd_mn, w_down, s->h, Nd, 64) ||
        !make_map_mn2(&wg_mn, w_gate, s->d, Nh, 64) || !make_map_mn2(&wu_mn, w_up, s->d, Nh, 64) ||
        !make_map_mn2(&dy_mn, dy_disp, s->d, R, 64) || !make_map_mn2(&h_mn, h_act, s->h, R, 64) ||
        !make_map_mn2(&dg_mn, dG, s->h, R, 64) || !make_map_mn2(&du_mn, dU, s->h, R, 64) ||
        !make_map_mn2(&x_mn, x_disp, s->d, R, 64))
        return MOE_ERR_CUDA;
    CUtensorMap o_dg, o_du, o_dx;
    if (!make_map_bf16_store(&o_dg, dG, s->h, R) || !make_map_bf16_store(&o_du, dU, s->h, R) ||
        !make_map_bf16_store(&o_dx, dx_disp, s->d, R))
        return MOE_ERR_CUDA;
    CUtensorMap o_down, o_gate, o_up;
    if (!make_map_f32_3d(&o_down, dw_down, s->h, s->d, s->N) ||
        !make_map_f32_3d(&o_gate, dw_gate, s->d, s->h, s->N) ||
        !make_map_f32_3d(&o_up, dw_up, s->d, s->h, s->N))
        return MOE_ERR_CUDA;

    // dH = dY W_down, then dG, dU
    p.ntn = (s->h + MMA_N - 1) / MMA_N;
    p.g_save = g_save;
    p.u_save = u_save;
    p.out0 = dG;
    p.out1 = dU;
    const int pair_tiles = (row_tiles + 1) / 2 + s->N;
    r = launch_dgrad_pair<DGRAD_DH>(dy_k, dy_k, wd_mn, wd_mn, o_dg, o_du, p, pair_tiles * p.ntn,
                                    stream);
    if (r != MOE_OK) return r;
    // dX = dG W_gate + dU W_up
    p.ntn = (s->d + MMA_N - 1) / MMA_N;
    p.out0 = dx_disp;
    p.out1 = nullptr;
    r = launch_dgrad_pair<DGRAD_DX>(dg_k, du_k, wg_mn, wu_mn, o_dx, o_dx, p, pair_tiles * p.ntn,
                                    stream);
    if (r != MOE_OK) return r;
    // dW_down = dY^T H
    p.mtn = (s->d + 2 * BM - 1) / (2 * BM);
    p.ntn = (s->h + MMA_N - 1) / MMA_N;
    p.fout0 = dw_down;
    p.fout1 = nullptr;
    r = launch_wgrad_pair<WGRAD_DOWN>(dy_mn, dy_mn, h_mn, o_down, o_down, p, s->N * p.mtn * p.ntn,
                                      stream);
    if (r != MOE_OK) return r;
    // dW_gate = dG^T X, dW_up = dU^T X
    p.mtn = wg_mt;
    p.ntn = (s->d + MMA_N - 1) / MMA_N;
    p.fout0 = dw_gate;
    p.fout1 = dw_up;
    return launch_wgrad_pair<WGRAD_GATEUP>(dg_mn, du_mn, x_mn, o_gate, o_up, p,
                                           s->N * p.mtn * p.ntn, stream);
}
