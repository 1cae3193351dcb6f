// api.cu -- device error word and status helpers of the C ABI.
#include "common.cuh"

namespace moe {
__device__ unsigned int g_device_errors = 0u;
}

extern "C" moe_status moe_get_device_errors(uint32_t* flags_out, int clear) {
    unsigned int v = 0;
    if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemcpyFromSymbol(&v, moe::g_device_errors, sizeof(v)) != cudaSuccess) return MOE_ERR_CUDA;
    if (clear) {
        unsigned int z = 0;
        if (cudaMemcpyToSymbol(moe::g_device_errors, &z, sizeof(z)) != cudaSuccess) return MOE_ERR_CUDA;
    }
    if (flags_out) *flags_out = v;
    return v ? MOE_ERR_DEVICE : MOE_OK;
}

extern "C" const char* moe_status_string(moe_status status) {
    switch (status) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
        case MOE_ERR_ALIGNMENT: return "MOE_ERR_ALIGNMENT";
        case MOE_ERR_DEVICE: return "MOE_ERR_DEVICE";
    }
    return "MOE_ERR_UNKNOWN";
}
