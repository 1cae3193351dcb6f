// nvfp4.cu -- NVFP4 operands: the tensor amax (moe_amax_bf16) and the row-wise quantiser
// (moe_quant_nvfp4).
//
// NVFP4 is named as a planned addition in "Dropless MoE acceleration in JAX with NVIDIA
// Transformer Engine", section "Measured training impact with JAX + Transformer Engine" (and in
// "NVIDIA says its JAX stack makes dropless MoE training 10x faster", "What to watch"); neither
// page defines it. NVIDIA's published format is taken: E2M1 elements, 16 consecutive elements
// along a row sharing one E4M3 decode scale, and one fp32 tensor encode scale
// S = 448 * 6 / amax(tensor) so that the block scales use E4M3's range; a value decodes as
// e2m1 * e4m3(scale) / S. Encoder decisions in fp32 (one rounding per operation):
//   scale = E4M3((amax_block / 6) * S),  code = E2M1(x * (S / e4m3(scale))).
// Both kernels are HBM-bound streams: the amax reads the tensor once (one atomic per CTA), the
// quantiser reads it once more and writes 9/16 of a byte per element.
#include "common.cuh"

namespace moe {
namespace {

__device__ __forceinline__ long long valid_rows_of(long long rows, const int32_t* valid_rows) {
    if (valid_rows == nullptr) return rows;
    const long long v = (long long)__ldg(valid_rows);
    return v < 0 ? 0 : (v < rows ? v : rows);
}

// max |x| over the first valid rows of x [rows, cols] bf16 (cols % 8 == 0) into *amax, which the
// caller zeroed; non-negative floats order like their bit patterns, so an unsigned atomicMax works.
__global__ void __launch_bounds__(256) amax_bf16_kernel(const uint4* __restrict__ x, long long rows, int cols,
                                                        const int32_t* __restrict__ valid_rows,
                                                        float* __restrict__ amax) {
    const long long n = valid_rows_of(rows, valid_rows) * (long long)(cols / 8);
    float m = 0.0f;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        float f[8];
        bf16x8_to_f32(__ldg(x + i), f);
#pragma unroll
        for (int j = 0; j < 8; j++) m = fmaxf(m, fabsf(f[j]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, o));
    __shared__ float wmax[8];
    if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float b = 0.0f;
        for (int w = 0; w < (int)(blockDim.x >> 5); w++) b = fmaxf(b, wmax[w]);
        if (b > 0.0f) atomicMax(reinterpret_cast<unsigned int*>(amax), __float_as_uint(b));
    }
}

// One thread per 16-element block: two 16-byte loads, 8 bytes of codes and one scale byte out.
__global__ void __launch_bounds__(256) quant_nvfp4_kernel(const uint4* __restrict__ x, long long rows, int cols,
                                                          const int32_t* __restrict__ valid_rows,
                                                          const float* __restrict__ amax, uint2* __restrict__ q,
                                                          uint8_t* __restrict__ scales) {
    const float S = nvfp4_encode_scale(__ldg(amax));
    __shared__ float s_rs[256];
    for (int i = threadIdx.x; i < 256; i += blockDim.x) s_rs[i] = nvfp4_rs_entry(S, (uint32_t)i);
    __syncthreads();
    const int bpr = cols / 16;
    const long long nb = valid_rows_of(rows, valid_rows) * (long long)bpr;
    for (long long b = (long long)blockIdx.x * blockDim.x + threadIdx.x; b < nb; b += (long long)gridDim.x * blockDim.x) {
        float f[16];
        bf16x8_to_f32(__ldg(x + 2 * b), f);
        bf16x8_to_f32(__ldg(x + 2 * b + 1), f + 8);
        uint32_t sb;
        q[b] = nvfp4_block(f, S, s_rs, &sb);
        scales[b] = (uint8_t)sb;
    }
}

int sm_count_nv() {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}

int grid_for(long long work, int per_sm) {
    const long long blocks = (work + 255) / 256;
    const long long cap = (long long)sm_count_nv() * per_sm;
    return (int)(blocks < 1 ? 1 : (blocks < cap ? blocks : cap));
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_amax_bf16(const void* x, long long rows, int cols, const int32_t* valid_rows, float* amax,
                                    moe_stream_t stream) {
    using namespace moe;
    if (rows < 0 || cols < 8 || (cols % 8) != 0 || !amax) return MOE_ERR_INVALID_ARG;
    if (rows > 0 && !x) return MOE_ERR_INVALID_ARG;
    if (!moe_host::aligned(x, 16) || !moe_host::aligned(amax, 4) || !moe_host::aligned(valid_rows, 4))
        return MOE_ERR_ALIGNMENT;
    cudaStream_t s = moe_host::as_stream(stream);
    if (cudaMemsetAsync(amax, 0, sizeof(float), s) != cudaSuccess) return MOE_ERR_CUDA;
    if (rows == 0) return MOE_OK;
    amax_bf16_kernel<<<grid_for(rows * (cols / 8), 8), 256, 0, s>>>(static_cast<const uint4*>(x), rows, cols,
                                                                    valid_rows, amax);
    return moe_host::launch_status();
}

extern "C" moe_status moe_quant_nvfp4(const void* x, long long rows, int cols, const int32_t* valid_rows,
                                      const float* amax, uint8_t* q, uint8_t* scales, moe_stream_t stream) {
    using namespace moe;
    if (rows < 0 || cols < 16 || (cols % 16) != 0) return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    if (!x || !amax || !q || !scales) return MOE_ERR_INVALID_ARG;
    if (!moe_host::aligned(x, 16) || !moe_host::aligned(q, 8) || !moe_host::aligned(amax, 4) ||
        !moe_host::aligned(valid_rows, 4))
        return MOE_ERR_ALIGNMENT;
    cudaStream_t s = moe_host::as_stream(stream);
    quant_nvfp4_kernel<<<grid_for(rows * (cols / 16), 8), 256, 0, s>>>(
        static_cast<const uint4*>(x), rows, cols, valid_rows, amax, reinterpret_cast<uint2*>(q), scales);
    return moe_host::launch_status();
}
