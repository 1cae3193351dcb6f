// common.cuh -- shared device helpers of the GB300 dropless-MoE library.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "moe_gb300.h"

namespace moe {

constexpr unsigned FULL = 0xffffffffu;

// Device error word (MOE_DEVERR_* bits); one per device, read by moe_get_device_errors.
extern __device__ unsigned int g_device_errors;

__device__ __forceinline__ void raise_device_error(unsigned bits) { atomicOr(&g_device_errors, bits); }

__device__ __forceinline__ unsigned lane_id() { return threadIdx.x & 31u; }

// Programmatic dependent launch. A kernel launched with programmatic stream serialization may
// start while the kernel before it on the stream is still running: pdl_wait() returns once
// that kernel has completed and its writes are visible (immediately for a kernel launched the
// ordinary way), so such a kernel calls it before it touches anything another kernel wrote.
// pdl_trigger() lets the next kernel on the stream start early (it still waits for this one
// to complete before reading what it writes).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// Read an expert id of either width.
__device__ __forceinline__ int load_id(const void* ids, long long i, bool i16) {
    return i16 ? (int)((const int16_t*)ids)[i] : ((const int32_t*)ids)[i];
}

// ---------------------------------------------------------------- MXFP8 block rule
// E8M0 byte of a block with absolute maximum `amax` (finite, >= 0):
// floor(log2(amax)) - 8 + 127, clamped to [0, 254]; 127 for amax == 0.
__device__ __forceinline__ int e8m0_scale_byte(float amax) {
    if (amax == 0.0f) return 127;
    unsigned u = __float_as_uint(amax);
    int ebits = (int)((u >> 23) & 0xffu);
    int fl;  // floor(log2(amax))
    if (ebits != 0) {
        fl = ebits - 127;
    } else {  // subnormal: mantissa m, amax = m * 2^-149, leading one at bit p -> 2^(p-149)
        fl = (31 - __clz((int)(u & 0x7fffffu))) - 149;
    }
    int b = fl - 8 + 127;
    return b < 0 ? 0 : (b > 254 ? 254 : b);
}

// 2^(127 - byte) as a float; exact for byte in [0, 253].
__device__ __forceinline__ float e8m0_inv_scale(int byte) {
    return __uint_as_float((unsigned)(254 - byte) << 23);
}

// Two floats -> two E4M3 codes (round to nearest even, saturate to +-448), packed lo|hi<<8.
__device__ __forceinline__ unsigned short f32x2_to_e4m3x2(float lo, float hi) {
    return (unsigned short)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

// ---------------------------------------------------------------- NVFP4 block rule
// Tensor encode scale S = 448 * 6 / amax (fp32, one rounding; 1 for amax == 0; at most FLT_MAX).
__device__ __forceinline__ float nvfp4_encode_scale(float amax) {
    if (!(amax > 0.0f)) return 1.0f;
    const float s = __fdiv_rn(2688.0f, amax);
    return s > 3.40282347e38f ? 3.40282347e38f : s;
}

// E2M1 codes of 8 values, element i in bits 4i..4i+3: each rounded to nearest on the grid
// 0, .5, 1, 1.5, 2, 3, 4, 6 (ties to the even code), saturating to 6, sign kept -- the
// conversion instruction's round-to-nearest-even with saturation to the largest finite
// value. The instruction puts its first source in the high nibble.
__device__ __forceinline__ uint32_t e2m1x8(const float* v) {
    uint32_t r;
    asm("{\n .reg .b8 q0, q1, q2, q3;\n"
        " cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n"
        " cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n"
        " cvt.rn.satfinite.e2m1x2.f32 q2, %6, %5;\n"
        " cvt.rn.satfinite.e2m1x2.f32 q3, %8, %7;\n"
        " mov.b32 %0, {q0, q1, q2, q3};\n}"
        : "=r"(r)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return r;
}

// Value of an E4M3 byte (exact).
__device__ __forceinline__ float e4m3_value(uint32_t byte) {
    const __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)byte, __NV_E4M3);
    return __half2float(__half(h));
}

// The elements' multiplier of the NVFP4 rule for a block whose E4M3 decode scale is the byte b:
// S / decode(b), one correctly rounded division; 0 where the decode is not positive (the block
// is then all zero codes). A kernel fills a table of the 256 bytes once per CTA.
__device__ __forceinline__ float nvfp4_rs_entry(float S, uint32_t b) {
    const float ds = e4m3_value(b);
    return ds > 0.0f ? __fdiv_rn(S, ds) : 0.0f;
}

// Encode one NVFP4 block of 16 values with tensor encode scale S: returns the 16 packed codes
// (element i in bits 4i..4i+3) and, in *sbyte, the E4M3 decode scale E4M3((amax / 6) * S).
// rs_tab: nvfp4_rs_entry(S, b) for every byte b.
__device__ __forceinline__ uint2 nvfp4_block(const float* f, float S, const float* rs_tab, uint32_t* sbyte) {
    float am = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; i++) am = fmaxf(am, fabsf(f[i]));
    const float sbf = __fmul_rn(__fdiv_rn(am, 6.0f), S);
    const uint32_t sb = (uint32_t)f32x2_to_e4m3x2(sbf, 0.0f) & 0xffu;
    const float rs = rs_tab[sb];
    uint2 out = make_uint2(0u, 0u);
    if (rs > 0.0f) {
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; i++) v[i] = __fmul_rn(f[i], rs);
        out = make_uint2(e2m1x8(v), e2m1x8(v + 8));
    }
    *sbyte = sb;
    return out;
}

// One NVFP4 block of 16 values held by two adjacent lanes (8 each, the even lane first; both
// lanes must call): this lane's 8 packed codes, and in *sbyte the block's E4M3 scale. The same
// arithmetic as nvfp4_block.
__device__ __forceinline__ uint32_t nvfp4_pair(const float* f, float S, const float* rs_tab, uint32_t* sbyte) {
    float am = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; i++) am = fmaxf(am, fabsf(f[i]));
    am = fmaxf(am, __shfl_xor_sync(FULL, am, 1));
    const float sbf = __fmul_rn(__fdiv_rn(am, 6.0f), S);
    const uint32_t sb = (uint32_t)f32x2_to_e4m3x2(sbf, 0.0f) & 0xffu;
    const float rs = rs_tab[sb];
    uint32_t out = 0u;
    if (rs > 0.0f) {
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; i++) v[i] = __fmul_rn(f[i], rs);
        out = e2m1x8(v);
    }
    *sbyte = sb;
    return out;
}

// 8 bf16 (one uint4) -> floats.
__device__ __forceinline__ void bf16x8_to_f32(const uint4& v, float* f) {
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; i++) {
        float2 t = __bfloat1622float2(p[i]);
        f[2 * i] = t.x;
        f[2 * i + 1] = t.y;
    }
}

__device__ __forceinline__ uint4 f32_to_bf16x8(const float* f) {
    uint4 v;
    __nv_bfloat162* p = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
    for (int i = 0; i < 4; i++) p[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
    return v;
}

// Quantise the 8 floats one lane holds, where four consecutive lanes hold one
// 32-element block: returns the 8 E4M3 codes and (in *sbyte) the block's scale byte.
__device__ __forceinline__ uint2 quant8_in_quad(const float* f, int* sbyte) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; i++) amax = fmaxf(amax, fabsf(f[i]));
    amax = fmaxf(amax, __shfl_xor_sync(FULL, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(FULL, amax, 2));
    int sb = e8m0_scale_byte(amax);
    float inv = e8m0_inv_scale(sb);
    uint2 out;
    out.x = (unsigned)f32x2_to_e4m3x2(f[0] * inv, f[1] * inv) |
            ((unsigned)f32x2_to_e4m3x2(f[2] * inv, f[3] * inv) << 16);
    out.y = (unsigned)f32x2_to_e4m3x2(f[4] * inv, f[5] * inv) |
            ((unsigned)f32x2_to_e4m3x2(f[6] * inv, f[7] * inv) << 16);
    *sbyte = sb;
    return out;
}

}  // namespace moe

// Host-side helpers shared by the entry points.
namespace moe_host {

inline bool aligned(const void* p, size_t a) { return ((uintptr_t)p % a) == 0; }

inline moe_status launch_status() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

inline cudaStream_t as_stream(moe_stream_t s) { return (cudaStream_t)s; }

// Launch with programmatic stream serialization: the kernel may start before the previous
// kernel on the stream completes, so it must call moe::pdl_wait() before reading anything that
// kernel (or any earlier one) wrote.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

}  // namespace moe_host
