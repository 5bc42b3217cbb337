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
    }
    return "unknown moe_status";
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
