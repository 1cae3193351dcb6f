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

// Shared tile: row r starts at element r * 72 + (r / 32) * 16 -- rows of 144 bytes (16-byte
// vector access) and an 8-word skew per 32 rows, so that the column reads of the quantiser
// (4 columns x the four 32-row blocks per warp instruction) fall in 16 distinct banks.
constexpr int TR_STRIDE = TR_COLS + 8;
constexpr int TR_TILE = TR_ROWS * TR_STRIDE + (TR_ROWS / 32) * 16;
__device__ __forceinline__ int tr_row(int r) { return r * TR_STRIDE + (r >> 5) * 16; }

// 16-byte asynchronous global -> shared copies (the next column chunk streams in while the
// current one is quantised and stored).
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

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
template <bool FP8, int CHUNKS, bool SCALE_WORDS>
__global__ void __launch_bounds__(256) grouped_transpose_kernel(const __nv_bfloat16* __restrict__ x,
                                                                const int* __restrict__ src_rows, int C,
                                                                const int* __restrict__ goff, int E, int kpad,
                                                                void* __restrict__ xT,
                                                                uint8_t* __restrict__ xT_scales) {
    __shared__ __align__(16) __nv_bfloat16 tiles[2][TR_TILE];   // double buffer over the column chunks
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
    // load 128 rows x 64 columns of chunk ck into buffer ck & 1 (16-byte pieces; rows past the group are zeros)
    auto issue = [&](int ck) {
        __nv_bfloat16* t = tiles[ck & 1];
        const int c0 = (blockIdx.y * CHUNKS + ck) * TR_COLS;
        for (int i = threadIdx.x; i < TR_ROWS * (TR_COLS / 8); i += blockDim.x) {
            const int r = i / (TR_COLS / 8), ch = i % (TR_COLS / 8);
            const int c = c0 + ch * 8;
            void* dst = &t[tr_row(r) + ch * 8];
            if (r < valid && c < C) cp_async16(dst, x + (long long)s_src[r] * C + c);
            else *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
        }
        cp_async_commit();
    };
    issue(0);
    for (int ck = 0; ck < CHUNKS; ck++) {
        const int c0 = (blockIdx.y * CHUNKS + ck) * TR_COLS;
        const __nv_bfloat16* tile = tiles[ck & 1];
        if (ck + 1 < CHUNKS) {
            issue(ck + 1);            // its buffer's previous readers finished at the end of iteration ck - 1
            cp_async_wait<1>();       // chunk ck has landed (this thread's part)
        } else {
            cp_async_wait<0>();
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
                for (int j = 0; j < 8; j++) f[j] = __bfloat162float(tile[tr_row(ch * 8 + j) + cc]);
                reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(xT) + (long long)c * kpad + kcol)[ch] =
                    f32_to_bf16x8(f);
            }
        } else {
            // thread = (column cc = t / 4, 32-row block sbk = t % 4): the four threads of a column
            // write its 128 contiguous output bytes, and one word holds its four scale bytes
            const int cc = threadIdx.x >> 2, sbk = threadIdx.x & 3;
            const int c = c0 + cc;
            float v[32];
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 32; i++) {
                v[i] = __bfloat162float(tile[tr_row(32 * sbk + i) + cc]);
                amax = fmaxf(amax, fabsf(v[i]));
            }
            const int sb = e8m0_scale_byte(amax);
            const float inv = e8m0_inv_scale(sb);
            uint32_t w[8];
#pragma unroll
            for (int i = 0; i < 8; i++)
                w[i] = (uint32_t)f32x2_to_e4m3x2(v[4 * i] * inv, v[4 * i + 1] * inv) |
                       ((uint32_t)f32x2_to_e4m3x2(v[4 * i + 2] * inv, v[4 * i + 3] * inv) << 16);
            uint32_t sw = (uint32_t)sb << (8 * sbk);
            sw |= __shfl_xor_sync(FULL, sw, 1);
            sw |= __shfl_xor_sync(FULL, sw, 2);
            if (c < C) {
                uint4* d =
                    reinterpret_cast<uint4*>(static_cast<uint8_t*>(xT) + (long long)c * kpad + kcol + 32 * sbk);
                d[0] = make_uint4(w[0], w[1], w[2], w[3]);
                d[1] = make_uint4(w[4], w[5], w[6], w[7]);
                uint8_t* srow = xT_scales + (long long)c * (kpad / 32) + kcol / 32;
                if (SCALE_WORDS) {
                    if (sbk == 0) *reinterpret_cast<uint32_t*>(srow) = sw;
                } else {
                    srow[sbk] = (uint8_t)sb;
                }
            }
        }
        __syncthreads();   // this buffer is refilled by the issue of iteration ck + 1
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
    // scale rows start at multiples of 4 bytes (kpad / 32 and kcol / 32 are): word stores when the base allows
    const bool words = fp8 && moe_host::aligned(xT_scales, 4);
#define MOE_TRANSPOSE(f8, ch, sw)                                                                          \
    grouped_transpose_kernel<f8, ch, sw><<<grid, 256, 0, s>>>(xb, src_rows, C, group_offsets, E, (int)kpad, xT, \
                                                              f8 ? xT_scales : nullptr)
    if (C % (4 * TR_COLS) == 0) {
        dim3 grid(gx, (unsigned)(C / (4 * TR_COLS)));
        if (!fp8) MOE_TRANSPOSE(false, 4, false);
        else if (words) MOE_TRANSPOSE(true, 4, true);
        else MOE_TRANSPOSE(true, 4, false);
    } else {
        dim3 grid(gx, (unsigned)(C / TR_COLS));
        if (!fp8) MOE_TRANSPOSE(false, 1, false);
        else if (words) MOE_TRANSPOSE(true, 1, true);
        else MOE_TRANSPOSE(true, 1, false);
    }
#undef MOE_TRANSPOSE
    return moe_host::launch_status();
}
