// Host-side entry points shared by every step: status strings and the
// device status word of a workspace.
#include "moe_common.cuh"

using namespace moe;

MOE_API const char *moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG: bad shape or null pointer";
        case MOE_ERR_ALIGNMENT: return "MOE_ERR_ALIGNMENT: pointer not 16-byte aligned or d/h not a multiple of 8";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE: workspace missing, misaligned or too small";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA: a CUDA call or kernel launch failed";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED: shape outside what the kernels handle";
        case MOE_ERR_DEVICE_TIMEOUT: return "MOE_ERR_DEVICE_TIMEOUT: a bounded wait inside a kernel expired";
        case MOE_ERR_DEVICE_ROUTE_RANGE: return "MOE_ERR_DEVICE_ROUTE_RANGE: a checked call skipped a route row outside the capacity buffers";
    }
    return "unknown moe_status";
}

MOE_API int64_t moe_buffer_rows(const moe_shape *s) {
    if (check_shape(s) != MOE_OK) return -1;
    return buffer_rows(s);
}

MOE_API moe_status moe_read_device_error(void *ws, int32_t *code_out, cudaStream_t stream) {
    if (!ws || !code_out) return MOE_ERR_INVALID_ARG;
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return MOE_ERR_CUDA;
    if (cudaMemsetAsync(ws, 0, sizeof(int32_t), stream) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
    *code_out = v;
    return MOE_OK;
}

namespace {

// Waits, with the bounded wait every kernel uses, on an mbarrier whose phase
// nothing completes; the wait gives up after limit_ns and records the timeout.
__global__ void selftest_wait_timeout(int *status, unsigned long long limit_ns) {
    pdl_enter();
    __shared__ uint64_t bar;
    __shared__ int abort;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, status, &abort, limit_ns);
}

}  // namespace

MOE_API moe_status moe_selftest_wait_timeout(void *ws, uint64_t limit_ns, cudaStream_t stream) {
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return MOE_ERR_WORKSPACE;
    if (limit_ns == 0 || limit_ns > 100000000ull) return MOE_ERR_INVALID_ARG;
    launch_pdl(selftest_wait_timeout, 1, 32, 0, stream, static_cast<int *>(ws), limit_ns);
    return launch_status();
}
