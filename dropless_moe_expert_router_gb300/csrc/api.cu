// api.cu -- device error word, status helpers and the bounded-wait self-test of the C ABI.
#include "common.cuh"
#include "sm100_ptx.cuh"

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

extern "C" moe_status moe_host_mapped_pointer(const void* host_ptr, void** dev_ptr) {
    if (!host_ptr || !dev_ptr) return MOE_ERR_INVALID_ARG;
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, host_ptr) != cudaSuccess) {
        cudaGetLastError();   // not an error state of the context
        return MOE_ERR_UNSUPPORTED;
    }
    if (attr.type != cudaMemoryTypeHost || attr.devicePointer == nullptr) return MOE_ERR_UNSUPPORTED;
    // the device address of this byte (attr.devicePointer is that of host_ptr itself)
    *dev_ptr = attr.devicePointer;
    return MOE_OK;
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

namespace moe {
namespace {
// One warp waits on an mbarrier that nothing ever arrives on, with the same
// bounded wait the grouped GEMM uses; the wait gives up after limit_ns, sets
// MOE_DEVERR_TIMEOUT and the kernel returns normally.
__global__ void bounded_wait_selftest_kernel(uint64_t limit_ns) {
    __shared__ uint64_t bar;
    __shared__ uint32_t abort_flag;
    if (threadIdx.x == 0) {
        ptx::mbar_init(&bar, 1);
        abort_flag = 0u;
        ptx::fence_mbar_init();
    }
    __syncwarp();
    ptx::wait_parity(&bar, 0u, &abort_flag, limit_ns);
}
}  // namespace
}  // namespace moe

extern "C" moe_status moe_debug_bounded_wait_selftest(uint32_t limit_us, moe_stream_t stream) {
    if (limit_us == 0 || limit_us > 1000000u) return MOE_ERR_INVALID_ARG;
    moe::bounded_wait_selftest_kernel<<<1, 32, 0, moe_host::as_stream(stream)>>>((uint64_t)limit_us * 1000ull);
    return moe_host::launch_status();
}
