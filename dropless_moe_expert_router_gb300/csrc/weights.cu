// weights.cu -- one-time packing of the expert weights for the grouped GEMMs
// (outside the hot path; the analogue of pre-fused MoE weights in the MaxText
// recipe named on "Dropless MoE acceleration in JAX with NVIDIA Transformer
// Engine", section "How to get started and reproduce results").
//
// Logical weights: W1, W3 [E][H][F], W2 [E][F][H] (bf16, row-major).
// Forward:   W13 [E][2F][H]  rows [256 j, 256 j + 128) = W1^T columns 128 j.., the
//                            next 128 = W3^T: one 256-wide output tile holds
//                            matching gate and up columns;
//            W2p [E][H][F]   = W2^T.
// Backward:  W2b [E][F][H]   = W2 (the dh = dy W2^T product contracts over H);
//            W13t [E][H][2F] row h = W1[e][h] and W3[e][h] interleaved per 128
//                            columns (the dx = [da|db] W13 product contracts over 2F).
// MXFP8 packs quantise every packed row along its contraction dimension in
// blocks of 32 (E4M3 payload, E8M0 scale per block, the rule of permute.cu).
#include "common.cuh"

namespace moe {
namespace {

__device__ __forceinline__ int w13_row(int f, int half) { return (f / 128) * 256 + half * 128 + (f % 128); }

// in [E][rows][cols] bf16 -> out [E][out_rows][rows] with out row = map(col).
template <int MODE>  // 0: W13 half 0 (W1), 1: W13 half 1 (W3), 2: W2
__global__ void pack_bf16_kernel(const __nv_bfloat16* __restrict__ in, int rows, int cols,
                                 __nv_bfloat16* __restrict__ out) {
    __shared__ __nv_bfloat16 tile[32][33];
    const int e = blockIdx.z;
    const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
    const __nv_bfloat16* src = in + (size_t)e * rows * cols;
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        int r = r0 + i, c = c0 + threadIdx.x;
        if (r < rows && c < cols) tile[i][threadIdx.x] = src[(size_t)r * cols + c];
    }
    __syncthreads();
    const int out_rows = MODE == 2 ? cols : 2 * cols;
    __nv_bfloat16* dst = out + (size_t)e * out_rows * rows;
    for (int i = threadIdx.y; i < 32; i += blockDim.y) {
        int c = c0 + i, r = r0 + threadIdx.x;
        if (r < rows && c < cols) {
            int orow = MODE == 2 ? c : w13_row(c, MODE);
            dst[(size_t)orow * rows + r] = tile[threadIdx.x][i];
        }
    }
}

// MXFP8 forward packing: transpose as above and quantise each packed row along
// its contraction dimension (the source's rows) in blocks of 32. Block (32
// source rows x 32 source columns); thread x owns one source column.
template <int MODE>
__global__ void pack_mxfp8_kernel(const __nv_bfloat16* __restrict__ in, int rows, int cols,
                                  uint8_t* __restrict__ q, uint8_t* __restrict__ s) {
    const int e = blockIdx.z;
    const int r0 = blockIdx.y * 32;
    const int c = blockIdx.x * 32 + threadIdx.x;
    if (c >= cols) return;
    const __nv_bfloat16* src = in + (size_t)e * rows * cols;
    float v[32];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; i++) {
        v[i] = __bfloat162float(src[(size_t)(r0 + i) * cols + c]);
        amax = fmaxf(amax, fabsf(v[i]));
    }
    const int sb = e8m0_scale_byte(amax);
    const float inv = e8m0_inv_scale(sb);
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; i++)
        w[i] = (uint32_t)f32x2_to_e4m3x2(v[4 * i] * inv, v[4 * i + 1] * inv) |
               ((uint32_t)f32x2_to_e4m3x2(v[4 * i + 2] * inv, v[4 * i + 3] * inv) << 16);
    const int out_rows = MODE == 2 ? cols : 2 * cols;
    const int orow = MODE == 2 ? c : w13_row(c, MODE);
    uint8_t* qrow = q + ((size_t)e * out_rows + orow) * rows + r0;
    uint4* d = reinterpret_cast<uint4*>(qrow);
    d[0] = make_uint4(w[0], w[1], w[2], w[3]);
    d[1] = make_uint4(w[4], w[5], w[6], w[7]);
    s[((size_t)e * out_rows + orow) * (rows / 32) + r0 / 32] = (uint8_t)sb;
}

// Backward packing without transposition: warp per packed row, 8 elements per
// lane per step (four lanes form one 32-element MXFP8 block).
//   INTERLEAVE = false: out row (e, f) = W2[e][f][:]              (ncols = H)
//   INTERLEAVE = true:  out row (e, h) = W1[e][h] | W3[e][h] per 128 (ncols = 2F)
template <bool FP8, bool INTERLEAVE>
__global__ void __launch_bounds__(256) pack_rows_kernel(const __nv_bfloat16* __restrict__ src1,
                                                        const __nv_bfloat16* __restrict__ src3, long long nrows,
                                                        int ncols, int src_cols, void* __restrict__ out,
                                                        uint8_t* __restrict__ scales) {
    const int lane = (int)lane_id();
    const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
    const int n8 = ncols / 8;
    for (long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; row < nrows; row += nwarps) {
        for (int j0 = 0; j0 < n8; j0 += 32) {
            const int j = j0 + lane;      // 8-element chunk; n8 is a multiple of 4 so quads are whole
            const bool in = j < n8;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (in) {
                const int c = 8 * j;
                if (INTERLEAVE) {
                    const int blk = c / 256, half = (c % 256) / 128, i = c % 128;
                    const __nv_bfloat16* s = half ? src3 : src1;
                    v = *reinterpret_cast<const uint4*>(s + row * src_cols + blk * 128 + i);
                } else {
                    v = *reinterpret_cast<const uint4*>(src1 + row * src_cols + c);
                }
            }
            if (FP8) {
                float f[8];
                bf16x8_to_f32(v, f);
                int sb;
                uint2 qv = quant8_in_quad(f, &sb);
                if (in) {
                    reinterpret_cast<uint2*>(out)[row * n8 + j] = qv;
                    if ((lane & 3) == 0) scales[row * (ncols / 32) + j / 4] = (uint8_t)sb;
                }
            } else if (in) {
                reinterpret_cast<uint4*>(out)[row * n8 + j] = v;
            }
        }
    }
}

int sm_count() {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}

}  // namespace
}  // namespace moe

extern "C" size_t moe_packed_weights_bytes(int E, int H, int F, moe_dtype dtype, int which) {
    if (E < 1 || H < 1 || F < 1) return 0;
    const size_t n13 = (size_t)E * 2 * F * H, n2 = (size_t)E * H * F;
    const bool fp8 = dtype == MOE_MXFP8;
    switch (which) {
        case 0: return n13 * (fp8 ? 1 : 2);
        case 1: return fp8 ? n13 / 32 : 0;
        case 2: return n2 * (fp8 ? 1 : 2);
        case 3: return fp8 ? n2 / 32 : 0;
    }
    return 0;
}

extern "C" moe_status moe_prepare_weights(const void* w1, const void* w3, const void* w2, int E, int H, int F,
                                          moe_dtype dtype, void* w13_packed, uint8_t* w13_scales,
                                          void* w2_packed, uint8_t* w2_scales, moe_stream_t stream) {
    using namespace moe;
    if (E < 1 || H < 128 || F < 128 || (H % 128) || (F % 128)) return MOE_ERR_INVALID_ARG;
    if (dtype != MOE_BF16 && dtype != MOE_MXFP8) return MOE_ERR_INVALID_ARG;
    if (!w1 || !w3 || !w2 || !w13_packed || !w2_packed) return MOE_ERR_INVALID_ARG;
    if (dtype == MOE_MXFP8 && (!w13_scales || !w2_scales)) return MOE_ERR_INVALID_ARG;
    if (!moe_host::aligned(w13_packed, 16) || !moe_host::aligned(w2_packed, 16)) return MOE_ERR_ALIGNMENT;
    cudaStream_t s = moe_host::as_stream(stream);
    const __nv_bfloat16* W1 = (const __nv_bfloat16*)w1;
    const __nv_bfloat16* W3 = (const __nv_bfloat16*)w3;
    const __nv_bfloat16* W2 = (const __nv_bfloat16*)w2;
    if (dtype == MOE_BF16) {
        dim3 blk(32, 8);
        dim3 g13((F + 31) / 32, (H + 31) / 32, E), g2((H + 31) / 32, (F + 31) / 32, E);
        pack_bf16_kernel<0><<<g13, blk, 0, s>>>(W1, H, F, (__nv_bfloat16*)w13_packed);
        pack_bf16_kernel<1><<<g13, blk, 0, s>>>(W3, H, F, (__nv_bfloat16*)w13_packed);
        pack_bf16_kernel<2><<<g2, blk, 0, s>>>(W2, F, H, (__nv_bfloat16*)w2_packed);
    } else {
        dim3 g13((F + 31) / 32, H / 32, E), g2((H + 31) / 32, F / 32, E);
        pack_mxfp8_kernel<0><<<g13, 32, 0, s>>>(W1, H, F, (uint8_t*)w13_packed, w13_scales);
        pack_mxfp8_kernel<1><<<g13, 32, 0, s>>>(W3, H, F, (uint8_t*)w13_packed, w13_scales);
        pack_mxfp8_kernel<2><<<g2, 32, 0, s>>>(W2, F, H, (uint8_t*)w2_packed, w2_scales);
    }
    return moe_host::launch_status();
}

extern "C" moe_status moe_prepare_weights_bwd(const void* w1, const void* w3, const void* w2, int E, int H, int F,
                                              moe_dtype dtype, void* w2_bwd, uint8_t* w2_bwd_scales, void* w13t,
                                              uint8_t* w13t_scales, moe_stream_t stream) {
    using namespace moe;
    if (E < 1 || H < 128 || F < 128 || (H % 128) || (F % 128)) return MOE_ERR_INVALID_ARG;
    if (dtype != MOE_BF16 && dtype != MOE_MXFP8) return MOE_ERR_INVALID_ARG;
    if (!w1 || !w3 || !w2 || !w2_bwd || !w13t) return MOE_ERR_INVALID_ARG;
    const bool fp8 = dtype == MOE_MXFP8;
    if (fp8 && (!w2_bwd_scales || !w13t_scales)) return MOE_ERR_INVALID_ARG;
    if (!moe_host::aligned(w1, 16) || !moe_host::aligned(w3, 16) || !moe_host::aligned(w2, 16) ||
        !moe_host::aligned(w2_bwd, 16) || !moe_host::aligned(w13t, 16))
        return MOE_ERR_ALIGNMENT;
    cudaStream_t s = moe_host::as_stream(stream);
    const __nv_bfloat16* W1 = (const __nv_bfloat16*)w1;
    const __nv_bfloat16* W3 = (const __nv_bfloat16*)w3;
    const __nv_bfloat16* W2 = (const __nv_bfloat16*)w2;
    const int blocks = sm_count() * 8;
    if (fp8) {
        pack_rows_kernel<true, false><<<blocks, 256, 0, s>>>(W2, nullptr, (long long)E * F, H, H, w2_bwd,
                                                             w2_bwd_scales);
        pack_rows_kernel<true, true><<<blocks, 256, 0, s>>>(W1, W3, (long long)E * H, 2 * F, F, w13t, w13t_scales);
    } else {
        pack_rows_kernel<false, false><<<blocks, 256, 0, s>>>(W2, nullptr, (long long)E * F, H, H, w2_bwd, nullptr);
        pack_rows_kernel<false, true><<<blocks, 256, 0, s>>>(W1, W3, (long long)E * H, 2 * F, F, w13t, nullptr);
    }
    return moe_host::launch_status();
}
