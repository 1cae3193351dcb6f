// transpose.cu -- group-padded transposition (and group-aware column-wise MXFP8
// quantisation) of permuted operands for the weight-gradient GEMMs.
//
// The weight gradient of expert e contracts over that expert's rows:
// dW[e] = A_e^T B_e ("Dropless MoE acceleration in JAX with NVIDIA Transformer
// Engine": grouped GEMMs on variable-length groups, in a training step; MXFP8
// operands are quantised "group-aware", so 32-row blocks never cross a group).
// For the tensor cores both operands are made K-major along that contraction:
//   xT[c][P_e + i] = x[row(off[e] + i)][c],  i < m_e,
// with P_e = 128 * (e + off[e] / 128), zeros for i in [m_e, 128 * ceil(m_e / 128)).
// P_e is a multiple of 128 and P_e + 128 * ceil(m_e / 128) <= P_{e+1}, so every
// k-block a GEMM reads for expert e lies inside e's padded range and its tail
// is zero: a ragged contraction needs no masking. Total padded length
// Kpad = 128 * (E + ceil(R_cap / 128) + 1).
// MXFP8: each 32-row block of a group (blocks start at the group's first row;
// a partial block takes its amax over its valid rows) gives one E8M0 scale
// per column, stored at xT_scales[c][P_e / 32 + b]; all-padding blocks get
// scale byte 127 and zero payloads.
// Optionally the rows are gathered: row(r) = src_rows[r] (e.g. perm_src, to
// read the tokens x [T, C] directly instead of a permuted copy).
#include "common.cuh"

namespace moe {
namespace {

constexpr int TR_ROWS = 128;  // padded rows per block
constexpr int TR_COLS = 64;   // columns per block

// Last e with e + goff[e] / 128 <= pb (the function is strictly increasing in e),
// by a 32-way search of one warp: each round narrows [lo, hi] by a factor of 32.
__device__ __forceinline__ int find_group_warp(const int* __restrict__ goff, int E, int pb, int lane) {
    int lo = 0, hi = E - 1;
    while (hi > lo) {
        const int step = (hi - lo + 32) / 32;       // ceil(len / 32); candidates lo, lo + step, ... (lane 0 = lo, always true)
        const int cand = min(lo + lane * step, hi);
        const bool ok = cand + __ldg(goff + cand) / 128 <= pb;
        const unsigned m = __ballot_sync(FULL, ok);
        const int k = 31 - __clz(m);                  // last candidate that qualifies
        const int nlo = min(lo + k * step, hi);
        hi = min(hi, nlo + step - 1);
        lo = nlo;
        if (step == 1) break;
    }
    return lo;
}

// Block = one 128-row block of the padded axis x CHUNKS column chunks of 64.
template <bool FP8, int CHUNKS>
__global__ void __launch_bounds__(256) grouped_transpose_kernel(const __nv_bfloat16* __restrict__ x,
                                                                const int* __restrict__ src_rows, int C,
                                                                const int* __restrict__ goff, int E, int kpad,
                                                                void* __restrict__ xT,
                                                                uint8_t* __restrict__ xT_scales) {
    __shared__ __align__(16) __nv_bfloat16 tile[TR_ROWS][TR_COLS + 8];  // rows of 144 B: 16-byte vector access
    __shared__ int s_base, s_valid;
    __shared__ int s_src[TR_ROWS];
    const int pb = blockIdx.x;  // 128-row block of the padded axis
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        const int e = find_group_warp(goff, E, pb, lane);
        const int g0 = __ldg(goff + e), g1 = __ldg(goff + e + 1);
        const int b = pb - (e + g0 / 128);
        const int base = g0 + TR_ROWS * b;          // first source row of this block
        const int valid = (b >= 0 && TR_ROWS * b < g1 - g0) ? min(TR_ROWS, g1 - g0 - TR_ROWS * b) : -1;
        if (lane == 0) {
            s_base = base;
            s_valid = valid;
        }
        if (valid > 0)
            for (int r = lane; r < valid; r += 32)
                s_src[r] = src_rows ? __ldg(src_rows + base + r) : base + r;
    }
    __syncthreads();
    const int valid = s_valid;
    if (valid < 0) return;  // padding that no GEMM reads
    const long long kcol = (long long)TR_ROWS * pb;  // first padded column of this block
    for (int ck = 0; ck < CHUNKS; ck++) {
        const int c0 = (blockIdx.y * CHUNKS + ck) * TR_COLS;
        if (ck > 0) __syncthreads();   // the previous chunk's readers are done with the tile
        // load 128 rows x 64 columns (16-byte chunks; rows past the group are zeros)
        for (int i = threadIdx.x; i < TR_ROWS * (TR_COLS / 8); i += blockDim.x) {
            const int r = i / (TR_COLS / 8), ch = i % (TR_COLS / 8);
            uint4 v = make_uint4(0, 0, 0, 0);
            const int c = c0 + ch * 8;
            if (r < valid && c < C) v = *reinterpret_cast<const uint4*>(x + (long long)s_src[r] * C + c);
            *reinterpret_cast<uint4*>(&tile[r][ch * 8]) = v;
        }
        __syncthreads();
        if (!FP8) {
            // out row c: 128 bf16 = 16 chunks of 8
            for (int i = threadIdx.x; i < TR_COLS * (TR_ROWS / 8); i += blockDim.x) {
                const int cc = i / (TR_ROWS / 8), ch = i % (TR_ROWS / 8);
                const int c = c0 + cc;
                if (c >= C) continue;
                float f[8];
#pragma unroll
                for (int j = 0; j < 8; j++) f[j] = __bfloat162float(tile[ch * 8 + j][cc]);
                reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(xT) + (long long)c * kpad + kcol)[ch] =
                    f32_to_bf16x8(f);
            }
        } else {
            // thread = (column, 32-row block)
            const int cc = threadIdx.x % TR_COLS, sbk = threadIdx.x / TR_COLS;  // sbk in [0, 4)
            const int c = c0 + cc;
            if (c < C) {
                float v[32];
                float amax = 0.0f;
#pragma unroll
                for (int i = 0; i < 32; i++) {
                    v[i] = __bfloat162float(tile[32 * sbk + i][cc]);
                    amax = fmaxf(amax, fabsf(v[i]));
                }
                const int sb = e8m0_scale_byte(amax);
                const float inv = e8m0_inv_scale(sb);
                uint32_t w[8];
#pragma unroll
                for (int i = 0; i < 8; i++)
                    w[i] = (uint32_t)f32x2_to_e4m3x2(v[4 * i] * inv, v[4 * i + 1] * inv) |
                           ((uint32_t)f32x2_to_e4m3x2(v[4 * i + 2] * inv, v[4 * i + 3] * inv) << 16);
                uint4* d =
                    reinterpret_cast<uint4*>(static_cast<uint8_t*>(xT) + (long long)c * kpad + kcol + 32 * sbk);
                d[0] = make_uint4(w[0], w[1], w[2], w[3]);
                d[1] = make_uint4(w[4], w[5], w[6], w[7]);
                xT_scales[(long long)c * (kpad / 32) + kcol / 32 + sbk] = (uint8_t)sb;
            }
        }
    }
}

}  // namespace
}  // namespace moe

extern "C" size_t moe_grouped_transpose_kpad(int R_cap, int E);

extern "C" moe_status moe_grouped_transpose(const void* x, const int32_t* src_rows, int R_cap, int C,
                                            const int32_t* group_offsets, int E, moe_dtype out_dtype, void* xT,
                                            uint8_t* xT_scales, moe_stream_t stream) {
    using namespace moe;
    if (R_cap < 0 || C < TR_COLS || (C % TR_COLS) || E < 1 || !group_offsets) return MOE_ERR_INVALID_ARG;
    if (out_dtype != MOE_BF16 && out_dtype != MOE_MXFP8) return MOE_ERR_INVALID_ARG;
    const bool fp8 = out_dtype == MOE_MXFP8;
    if (R_cap == 0) return MOE_OK;
    if (!x || !xT || (fp8 && !xT_scales)) return MOE_ERR_INVALID_ARG;
    if (!moe_host::aligned(x, 16) || !moe_host::aligned(xT, 16)) return MOE_ERR_ALIGNMENT;
    const size_t kpad = moe_grouped_transpose_kpad(R_cap, E);
    if (kpad / TR_ROWS > 0x7fffffffULL) return MOE_ERR_UNSUPPORTED;
    cudaStream_t s = moe_host::as_stream(stream);
    const unsigned gx = (unsigned)(kpad / TR_ROWS);
    const auto* xb = (const __nv_bfloat16*)x;
    if (C % (4 * TR_COLS) == 0) {
        dim3 grid(gx, (unsigned)(C / (4 * TR_COLS)));
        if (fp8) grouped_transpose_kernel<true, 4><<<grid, 256, 0, s>>>(xb, src_rows, C, group_offsets, E, (int)kpad, xT, xT_scales);
        else grouped_transpose_kernel<false, 4><<<grid, 256, 0, s>>>(xb, src_rows, C, group_offsets, E, (int)kpad, xT, nullptr);
    } else {
        dim3 grid(gx, (unsigned)(C / TR_COLS));
        if (fp8) grouped_transpose_kernel<true, 1><<<grid, 256, 0, s>>>(xb, src_rows, C, group_offsets, E, (int)kpad, xT, xT_scales);
        else grouped_transpose_kernel<false, 1><<<grid, 256, 0, s>>>(xb, src_rows, C, group_offsets, E, (int)kpad, xT, nullptr);
    }
    return moe_host::launch_status();
}
