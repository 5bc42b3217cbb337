// Shared host and device helpers of the sm_103a kernels: status handling,
// shape validation, and thin inline-PTX wrappers for mbarrier, TMA (bulk
// tensor copies) and the tcgen05 tensor-core / tensor-memory instructions.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>
#include <mutex>

#include "../../include/moe.h"

#define MOE_API extern "C" __attribute__((visibility("default")))

namespace moe {

constexpr int kMaxK = 16;
constexpr int kMaxN = 1024;
// Bounded waits: a kernel that waits longer than this on a barrier records
// MOE_ERR_DEVICE_TIMEOUT in its status word and leaves its loops.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// ------------------------------------------------------------------ host --

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline moe_status check_shape(const moe_shape *s) {
    if (!s) return MOE_ERR_INVALID_ARG;
    if (s->T < 0 || s->cap < 0 || s->d <= 0 || s->h <= 0) return MOE_ERR_INVALID_ARG;
    if (s->K < 1 || s->K > kMaxK || s->N < s->K || s->N > kMaxN) return MOE_ERR_INVALID_ARG;
    if ((int64_t)s->T * s->K >= (int64_t)1 << 31) return MOE_ERR_INVALID_ARG;
    if ((int64_t)s->T * s->d >= (int64_t)1 << 40) return MOE_ERR_INVALID_ARG;
    if (s->d % 8 != 0 || s->h % 8 != 0) return MOE_ERR_ALIGNMENT;
    return MOE_OK;
}

// Rows of every capacity buffer: the packed prefix holds at most cap rows per
// expert and at most one row per route, so min(N * cap, T * K) rows suffice.
inline int64_t buffer_rows(const moe_shape *s) {
    const int64_t a = (int64_t)s->N * s->cap, b = (int64_t)s->T * s->K;
    return a < b ? a : b;
}

// ---- programmatic dependent launch ----------------------------------------
//
// Every kernel of the library is launched with programmatic stream
// serialization allowed (launch_pdl, or the same attribute beside a cluster
// dimension).  Its first statement is pdl_enter(): wait until the grid before
// it in the stream has completed and its memory is visible, then let the next
// grid launch.  The next grid's CTAs are thus scheduled, up to their own
// wait, while this grid runs, which hides the launch gap between kernels.
// The wait comes before any memory access and before any early return, so a
// grid never completes ahead of its predecessor.
__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

inline void set_pdl_attr(cudaLaunchAttribute &a) {
    a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    a.val.programmaticStreamSerializationAllowed = 1;
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t st, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    set_pdl_attr(attr[0]);
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

inline moe_status launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

inline int num_sms() {
    static std::atomic<int> cache[64];  // per device; 0 = not read yet
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) dev = 0;
    std::atomic<int> *c = dev < 64 ? &cache[dev] : nullptr;
    int n = c ? c->load(std::memory_order_relaxed) : 0;
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 1;
        if (c) c->store(n, std::memory_order_relaxed);
    }
    return n;
}

// Router term of the input gradient (rowwise.cu): dlogit and dx (+)= sum_k
// dlogit_k W_r[e_k]; fused with the dispatch backward when add is false.
moe_status launch_router_dx(const moe_shape *s, const moe_bf16 *dx_disp, const int32_t *route_row,
                            const float *w_router, const int32_t *topk_idx,
                            const float *topk_gate, const float *dgate, float *dlogit, float *dx,
                            bool add, cudaStream_t stream);

// ---- host: one-time kernel attributes ------------------------------------

// A kernel attribute such as the dynamic shared-memory limit belongs to the
// device that was current when it was set.  device_once(o, fn) runs fn (which
// returns true on success) once per device for the state o, also when several
// host threads make their first call at the same time; devices past 63 are
// refused.
struct PerDeviceOnce {
    std::atomic<uint64_t> done{0};  // bit d: fn succeeded on device d
    std::mutex mu;
};

template <typename Fn>
inline bool device_once(PerDeviceOnce &o, Fn &&fn) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    const uint64_t bit = 1ull << dev;
    if (o.done.load(std::memory_order_acquire) & bit) return true;
    std::lock_guard<std::mutex> lock(o.mu);
    if (o.done.load(std::memory_order_relaxed) & bit) return true;
    if (!fn()) return false;
    o.done.fetch_or(bit, std::memory_order_release);
    return true;
}

// Raises kernel's dynamic shared-memory limit to bytes on the current device.
template <typename K>
inline bool set_smem_limit(K *kernel, size_t bytes) {
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) ==
           cudaSuccess;
}

// ---- host: TMA descriptors -----------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// 2-D bf16 map over a row-major [rows, inner] matrix; box 64 (inner) x
// box_rows, 128-byte swizzle.  The box's 64 inner elements are one 128-byte
// smem row; a K-major operand has K inner, an MN-major operand has M or N
// inner.
inline bool make_map(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows,
                     uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {inner * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D bf16 map over a row-major [rows, inner] matrix for TMA stores of
// 32 x 32 blocks, 64-byte swizzle (a 32-element bf16 row is 64 bytes).
inline bool make_map_bf16_store(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {inner * 2};
    const cuuint32_t box[2] = {32, 32};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D fp32 map over [planes, rows, inner] (row-major, planes of rows x inner)
// for TMA stores of 32 x 32 blocks, 128-byte swizzle: a block never crosses a
// plane, and rows past `rows` or columns past `inner` are clipped.
inline bool make_map_f32_3d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows,
                            uint64_t planes) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {inner, rows, planes};
    const cuuint64_t strides[2] = {inner * 4, inner * rows * 4};
    const cuuint32_t box[3] = {32, 32, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---- host: MXFP8 -----------------------------------------------------------
//
// Scale chunks.  Every MXFP8 operand of the tensor cores (dispatched rows,
// SwiGLU outputs, weights) keeps its E8M0 scales in 512-byte chunks, one per
// 128 rows x 128 columns (4 blocks of 32): the scale of row r (0-127 within
// the 128-row block) and block b (0-3 within the 128 columns) sits at byte
// (r % 32) * 16 + (r / 32) * 4 + b.  This is the order tcgen05.cp 32x128b.warpx4
// copies into tensor memory and the block-scaled MMA reads there: row r's
// scales at TMEM lane r, column r / 32, byte b.  Chunk (block128, kgroup) of an
// operand with K columns starts at (block128 * K / 128 + kgroup) * 512.
// Weights number their 128-row blocks e * rows / 128 + row / 128; packed
// capacity-buffer rows number them per expert from that expert's first row:
// block128 = pad_block[e] + (r - offset[e]) / 128, pad_block[e] = the sum of
// ceil(count[e'] / 128) over e' < e (each expert starts a fresh block).
constexpr int kMxBlock = 32;
constexpr int kMxChunk = 512;

__host__ __device__ inline int64_t mx_chunk_byte(int64_t block128, int kcols, int r_in, int kb) {
    return (block128 * (kcols / 128) + kb / 4) * kMxChunk + (r_in % 32) * 16 + (r_in / 32) * 4 +
           (kb % 4);
}

// Weight scales are stored with every chunk written four times in a row
// (2 KB per 128-row block and 128-column group): the GEMM stages the four
// copies of two chunks with two TMA boxes and moves them into tensor memory,
// already replicated for the four lane quadrants, with one 128x256b copy.
constexpr int kMxWeightCopies = 4;

__host__ __device__ inline int64_t mx_wchunk_byte(int64_t block128, int kcols, int r_in, int kb,
                                                  int copy) {
    return ((block128 * (kcols / 128) + kb / 4) * kMxWeightCopies + copy) * kMxChunk +
           (r_in % 32) * 16 + (r_in / 32) * 4 + (kb % 4);
}

// Bytes of the scale-chunk array of a packed capacity buffer with k columns:
// sum over experts of ceil(count / 128) <= R / 128 + N blocks.
inline size_t mx_act_scale_bytes(int64_t R, int N, int k) {
    return (size_t)((R + 127) / 128 + N) * (size_t)(k / 128) * kMxChunk;
}

// 2-D uint8 map over a row-major [rows, inner] fp8 matrix; box 128 x
// box_rows, 128-byte swizzle (one 128-element row per 128-byte smem row).
inline bool make_map_u8(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows,
                        uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {inner};
    const cuuint32_t box[2] = {128, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Map over a scale-chunk array viewed as [chunks, 128] uint32: one box is
// box_chunks consecutive 512-byte chunks; chunks past the end read as zero.
inline bool make_map_chunks(CUtensorMap *m, const void *base, uint64_t chunks,
                            uint32_t box_chunks = 1) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {128, chunks};
    const cuuint64_t strides[1] = {kMxChunk};
    const cuuint32_t box[2] = {128, box_chunks};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---------------------------------------------------------------- device --

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 -> packed bf16 pair (round to nearest even); lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- cp.async (16-byte global -> shared copies, per thread) ---------------

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
    asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---- mbarrier ------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// The same test with acquire semantics at cluster scope, for a phase that
// other CTAs of the cluster complete with release arrivals covering their
// own shared-memory writes.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete.  Returns false (and
// records MOE_ERR_DEVICE_TIMEOUT in *status) if it has not completed within
// limit_ns (kWaitLimitNs by default), or at once if *abort is already set.
template <bool CLUSTER = false>
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int *status,
                                          volatile int *abort,
                                          unsigned long long limit_ns = kWaitLimitNs) {
    auto test = [&] {
        return CLUSTER ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
    };
    if (test()) return true;
    unsigned long long t0 = global_ns();
    for (uint32_t i = 1;; ++i) {
        if (test()) return true;
        if ((i & 63u) == 0) {
            if (*abort) return false;
            if (global_ns() - t0 > limit_ns) {
                atomicExch(status, (int)MOE_ERR_DEVICE_TIMEOUT);
                *abort = 1;
                return false;
            }
        }
    }
}

// ---- TMA -----------------------------------------------------------------

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, uint32_t src, int32_t x,
                                             int32_t y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(src)
                 : "memory");
}

// TMA store of a 3-D box from this CTA's shared memory (bulk-group
// completion: commit, then wait before the source is reused or the CTA ends).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, uint32_t src, int32_t x,
                                             int32_t y, int32_t z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(x), "r"(y), "r"(z), "r"(src)
        : "memory");
}
__device__ __forceinline__ void bulk_commit() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until at most N committed bulk groups of this thread still read
// shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait() {
    asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// One warp stores a 32-row x 32-column bf16 block: lane r holds its row as 16
// packed bf16 pairs.  The row goes into the warp's 2 KB block of shared memory
// (512-byte aligned) in the 64-byte swizzled layout, and lane 0 stores the
// block with one TMA instruction at (x, y) of the map.  The block is reused:
// the previous store from it must have finished reading first.
__device__ __forceinline__ void warp_store_bf16_32x32(uint8_t *blk, const uint32_t (&w)[16],
                                                      const CUtensorMap *map, int x, int y,
                                                      int lane) {
    if (lane == 0) bulk_wait_read<0>();
    __syncwarp();
#pragma unroll
    for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4 *>(blk + lane * 64 + ((q ^ ((lane >> 1) & 3)) * 16)) =
            make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncwarp();
    if (lane == 0) {
        tma_store_2d(map, smem_u32(blk), x, y);
        bulk_commit();
    }
}


__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---- clusters ------------------------------------------------------------

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// All threads of every CTA in the cluster arrive, then wait.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// ---- tcgen05 ---------------------------------------------------------------

// Shared-memory matrix descriptor of a K-major operand tile stored with the
// 128-byte swizzle: rows of 128 bytes (64 bf16), 8-row atoms 1024 bytes apart.
// Fields: start address >> 4 (bits 0-13), leading-dimension offset >> 4
// (bits 16-29, unused for this layout: 1), stride-dimension offset >> 4
// (bits 32-45: 1024 B), descriptor version 1 (bits 46-48), swizzle mode
// 128 B = 2 (bits 61-63).
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);
    d |= (uint64_t)1u << 16;
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= (uint64_t)1u << 46;
    d |= (uint64_t)2u << 61;
    return d;
}

// Instruction descriptor for kind::f16 with bf16 A and B, fp32 accumulator,
// both operands K-major: D format F32 (bits 4-5 = 1), A format BF16 (bits 7-9
// = 1), B format BF16 (bits 10-12 = 1), N >> 3 (bits 17-22), M >> 4 (bits 24-28).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
           ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives once on the mbarrier when every tcgen05.mma issued so far by this
// thread has completed.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Warp-wide: allocate `ncols` TMEM columns; the base address lands in *dst_smem.
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     dst_smem),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// ---- CTA pairs (tcgen05 cta_group::2) ---------------------------------------

// Address of the same shared-memory object in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t smem_addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
    return r;
}

// Arrive on an mbarrier that may live in another CTA of the cluster.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}

// The same arrival without release semantics, for signals that order no
// memory operation (an epilogue freeing an accumulator whose tcgen05.ld have
// completed): a release arrival would first wait for the thread's earlier
// global stores to complete.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}

// TMA load into this CTA's shared memory whose completion is signalled on an
// mbarrier of the pair's leader CTA (bar is a cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map,
                                                 uint32_t bar, int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// Gather of four rows (r0..r3, any rows of the tensor) x one 64-element box
// into this CTA's shared memory, completion signalled on the pair leader's
// mbarrier (bar is a cluster address).  The map's box is one row high; the
// four rows land as four consecutive 128-byte rows.
__device__ __forceinline__ void tma_gather4_pair(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                                 int32_t x, int32_t r0, int32_t r1, int32_t r2,
                                                 int32_t r3) {
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile::gather4.mbarrier::"
        "complete_tx::bytes [%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(bar)
        : "memory");
}

// MMA over the CTA pair: A rows 0-127 / 128-255 and B columns 0-N/2 / N/2-N
// come from the leader's / peer's shared memory at the same offsets; the
// accumulator rows land in each CTA's own tensor memory.
__device__ __forceinline__ void tc_mma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                 uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrives on the mbarrier at this offset in both CTAs of the pair when every
// cta_group::2 MMA issued so far by this thread has completed.
__device__ __forceinline__ void tc_commit_pair(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar), "h"((uint16_t)0x3)
        : "memory");
}

// Pair-wide TMEM allocation: both CTAs' allocating warps execute it and get
// the same column address.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     dst_smem),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// Warp-wide: each lane starts reading 16 consecutive fp32 columns of its TMEM
// lane into r.  The values are valid only after tmem_ld_wait(r...) below.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// Waits for this thread's outstanding tcgen05.ld, then passes each register
// through an empty volatile asm so that no use of it can be scheduled before
// the wait.
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void reg_fence(uint32_t (&r)[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) asm volatile("" : "+r"(r[i]));
}

// ---- MXFP8 ----------------------------------------------------------------

// Shared exponent of a block from its largest magnitude (finite, >= 0):
// floor(log2 amax) - 8, clamped below at -127 (zero and fp32 subnormals land
// there).  The E8M0 byte is the result + 127.
__device__ __forceinline__ int mx_exponent(float amax) {
    const int ef = (int)((__float_as_uint(amax) >> 23) & 0xFFu);
    return ef - 135 < -127 ? -127 : ef - 135;
}

// 2^-E as an fp32 multiplier (E in [-127, 119], so the result is normal).
__device__ __forceinline__ float mx_inv_scale(int E) {
    return __uint_as_float((uint32_t)(127 - E) << 23);
}

// Four fp32 values -> four E4M3 codes (round to nearest even, saturating at
// 448), a0 in the lowest byte.
__device__ __forceinline__ uint32_t e4m3x4(float a0, float a1, float a2, float a3) {
    uint16_t lo, hi;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(a1), "f"(a0));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(a3), "f"(a2));
    return (uint32_t)lo | ((uint32_t)hi << 16);
}

// Two E4M3 codes (c0 in the low byte) -> their exact fp32 values.
__device__ __forceinline__ float2 e4m3x2_to_f32(uint16_t c) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(c));
    const __half2 hv = *reinterpret_cast<const __half2 *>(&h2);
    return __half22float2(hv);
}

// 2^(s - 127) for an E8M0 byte s < 255 (s = 0 gives the subnormal 2^-127).
__device__ __forceinline__ float e8m0_value(uint32_t s) {
    return s == 0 ? __uint_as_float(0x00400000u) : __uint_as_float(s << 23);
}

// Instruction descriptor for kind::mxf8f6f4 with E4M3 A and B, E8M0 scales
// (bit 23), both operands K-major: B's scale byte (bits 4-5), N >> 3 (bits
// 17-22), M >> 4 (bits 24-28), A's scale byte (bits 29-30).  The byte picks
// which of the four blocks held in each 32-bit TMEM scale word this MMA uses.
__host__ __device__ constexpr uint32_t idesc_mxf8(int M, int N, int sf_byte) {
    return ((uint32_t)sf_byte << 4) | ((uint32_t)(N >> 3) << 17) | (1u << 23) |
           ((uint32_t)(M >> 4) << 24) | ((uint32_t)sf_byte << 29);
}

// Block-scaled MMA over the CTA pair: as tc_mma_bf16_pair, with each CTA's
// A scales at TMEM address sfa and the B scales of all N columns at sfb.
__device__ __forceinline__ void tc_mma_mxf8_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                 uint32_t idesc, uint32_t sfa, uint32_t sfb,
                                                 uint32_t accumulate) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
        " tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X"
        " [%0], %1, %2, %3, [%4], [%5], p;\n}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
}

// Shared-memory descriptor of one 512-byte scale chunk: 32 rows of 16 bytes,
// no swizzle, 8-row groups 128 bytes apart.
__device__ __forceinline__ uint64_t chunk_desc(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);
    d |= (uint64_t)(128u >> 4) << 16;
    d |= (uint64_t)(128u >> 4) << 32;
    d |= (uint64_t)1u << 46;
    return d;
}

// Shared-memory descriptor of the eight B-scale chunks of a stage: the low
// 256 columns' chunk four times (2 KB), then the high columns' chunk four
// times; row L of a 128x256b copy reads 16 bytes at 16 L of each half.
__device__ __forceinline__ uint64_t sfb_desc(uint32_t smem_addr) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);
    d |= (uint64_t)(2048u >> 4) << 16;
    d |= (uint64_t)(128u >> 4) << 32;
    d |= (uint64_t)1u << 46;
    return d;
}

// Issued by the pair's leader: 128 lanes x 32 bytes from each CTA's shared
// memory at this offset into its own tensor memory (eight columns).
__device__ __forceinline__ void tc_cp_sfb_pair(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::2.128x256b [%0], %1;" ::"r"(taddr), "l"(sdesc)
                 : "memory");
}

// Issued by the pair's leader: each CTA's chunk at this shared-memory offset
// goes to its own tensor memory, 32 lanes x 4 columns copied to all four lane
// quadrants (ordered before later tcgen05.mma of the same thread).
__device__ __forceinline__ void tc_cp_chunk_pair(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
                 : "memory");
}

}  // namespace moe
