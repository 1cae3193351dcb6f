// combine.cu -- probability-weighted unpermute/combine back to token order.
//
// "Dropless MoE acceleration in JAX with NVIDIA Transformer Engine", section
// "Optimization 2": after the experts ran, results are routed back and
// accumulated in token order; "Sparser MoE end-to-end", section "Remove work
// that has no selected route": combine pulls and reduces, and visits only the
// selected slots of each token.
//
// One warp per token: a ballot over the token's K route slots (row_map >= 0)
// gives the rows to pull; each lane owns 16-byte column chunks and accumulates
// probs[t,k] * y_perm[row, chunk] in fp32, in ascending k, then rounds to bf16.
// RB routes are pulled at a time (all their loads issued before any of them is
// accumulated), so a token costs about K / RB memory latencies, not K.
#include "common.cuh"

namespace moe {
namespace {

// KC * 32 route slots per token, CHUNKS 16-byte chunks per lane and route, RB routes in flight.
// UNIT: every weight is 1 (the permute backward: the sum of a token's rows); probs is not read.
// (four blocks per SM, 64 registers, where that needs no spills: KC * CHUNKS <= 4)
template <int KC, int CHUNKS, int RB, bool UNIT = false>
__global__ void __launch_bounds__(256, KC * CHUNKS <= 4 ? 4 : 1) combine_kernel(const uint4* __restrict__ y_perm,
                                                      const int* __restrict__ row_map,
                                                      const float* __restrict__ probs, int T, int K, int H,
                                                      uint4* __restrict__ y) {
    const int lane = (int)lane_id();
    const int nwarps_total = (gridDim.x * blockDim.x) >> 5;
    const int H8 = H >> 3;
    for (long long t = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += nwarps_total) {
        int rows[KC];
        float p[KC];
        unsigned mask[KC];
#pragma unroll
        for (int c = 0; c < KC; c++) {
            int k = c * 32 + lane;
            int r = -1;
            float pk = 0.0f;
            if (k < K) {
                r = __ldg(row_map + t * K + k);
                pk = UNIT ? 1.0f : __ldg(probs + t * K + k);
            }
            rows[c] = r;
            p[c] = pk;
            mask[c] = __ballot_sync(FULL, r >= 0);
        }
        for (int j0 = 0; j0 < H8; j0 += 32 * CHUNKS) {
            float acc[CHUNKS][8];
#pragma unroll
            for (int u = 0; u < CHUNKS; u++)
#pragma unroll
                for (int i = 0; i < 8; i++) acc[u][i] = 0.0f;
#pragma unroll
            for (int c = 0; c < KC; c++) {
                unsigned m = mask[c];
                while (m) {
                    // the next (up to) RB selected slots, in ascending k (warp-uniform)
                    int rr[RB];
                    float pp[RB];
                    bool on[RB];
#pragma unroll
                    for (int q = 0; q < RB; q++) {
                        on[q] = m != 0u;
                        const int b = on[q] ? __ffs(m) - 1 : 0;
                        if (on[q]) m &= m - 1;
                        rr[q] = __shfl_sync(FULL, rows[c], b);
                        pp[q] = __shfl_sync(FULL, p[c], b);
                    }
                    uint4 v[RB][CHUNKS];
#pragma unroll
                    for (int q = 0; q < RB; q++)
#pragma unroll
                        for (int u = 0; u < CHUNKS; u++) {
                            const int j = j0 + u * 32 + lane;
                            v[q][u] = on[q] && j < H8 ? __ldg(y_perm + (long long)rr[q] * H8 + j)
                                                      : make_uint4(0, 0, 0, 0);
                        }
#pragma unroll
                    for (int q = 0; q < RB; q++) {
                        if (!on[q]) break;
#pragma unroll
                        for (int u = 0; u < CHUNKS; u++) {
                            float f[8];
                            bf16x8_to_f32(v[q][u], f);
#pragma unroll
                            for (int i = 0; i < 8; i++) acc[u][i] = fmaf(pp[q], f[i], acc[u][i]);
                        }
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < CHUNKS; u++) {
                const int j = j0 + u * 32 + lane;
                if (j < H8) y[t * H8 + j] = f32_to_bf16x8(acc[u]);
            }
        }
    }
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_unpermute_combine(const void* y_perm, const int32_t* row_map, const float* probs,
                                            int T, int K, int H, void* y, moe_stream_t stream) {
    using namespace moe;
    if (T < 0 || K < 1 || K > 128 || H < 8 || (H % 8) != 0) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!y_perm || !row_map || !probs || !y) return MOE_ERR_INVALID_ARG;
    if (!moe_host::aligned(y_perm, 16) || !moe_host::aligned(y, 16) || !moe_host::aligned(row_map, 4) ||
        !moe_host::aligned(probs, 4))
        return MOE_ERR_ALIGNMENT;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    long long blocks = ((long long)T + 7) / 8;
    const long long cap = (long long)sms * 16;
    if (blocks > cap) blocks = cap;
    cudaStream_t s = moe_host::as_stream(stream);
    const int KC = (K + 31) / 32;
    const int H8 = H / 8;
    const int CH = H8 >= 128 ? 4 : (H8 >= 64 ? 2 : 1);  // no more chunks than a row has per lane
    const uint4* yp = (const uint4*)y_perm;
    uint4* yo = (uint4*)y;
#define MOE_COMBINE(kc, ch) \
    combine_kernel<kc, ch, (ch == 4 ? 2 : 4)><<<(int)blocks, 256, 0, s>>>(yp, row_map, probs, T, K, H, yo)
    if (KC == 1) {
        if (CH == 4) MOE_COMBINE(1, 4); else if (CH == 2) MOE_COMBINE(1, 2); else MOE_COMBINE(1, 1);
    } else if (KC == 2) {
        if (CH == 4) MOE_COMBINE(2, 4); else if (CH == 2) MOE_COMBINE(2, 2); else MOE_COMBINE(2, 1);
    } else {
        if (CH == 4) MOE_COMBINE(4, 4); else if (CH == 2) MOE_COMBINE(4, 2); else MOE_COMBINE(4, 1);
    }
#undef MOE_COMBINE
    return moe_host::launch_status();
}

// ---------------------------------------------------------------------------
// Backward of the combine and of the permute (the adjoints of the forward maps;
// the pages give the forwards -- [TEJAX] "Optimization 2", [SPARSER] "Remove
// work that has no selected route" -- and name training, not these steps).
// ---------------------------------------------------------------------------
namespace moe {
namespace {

// Combine backward, one warp per token: for each valid route (t, k) with row r,
// dy_perm[r] = bf16(p[t,k] * dy[t]) and dprobs[t,k] = <dy[t], y_perm[r]> (fp32).
// RB routes at a time; per 32-chunk slice of the row each lane loads one 16-byte
// chunk of dy and of each route's y_perm row, writes the scaled dy chunks and
// accumulates the routes' partial dot products, reduced at the end. Q: the bf16
// dy_perm values are also quantised to MXFP8 along the row (1x32 blocks, four
// lanes per block), the codes and scales of the next GEMM's operand.
template <int KC, int RB, bool Q>
__global__ void __launch_bounds__(256, KC == 1 ? 3 : 1) combine_backward_kernel(const uint4* __restrict__ dy,
                                                               const uint4* __restrict__ y_perm,
                                                               const int* __restrict__ row_map,
                                                               const float* __restrict__ probs, int T, int K,
                                                               int H, uint4* __restrict__ dy_perm,
                                                               float* __restrict__ dprobs,
                                                               uint2* __restrict__ q,
                                                               uint8_t* __restrict__ qs) {
    const int lane = (int)lane_id();
    const int nwarps_total = (gridDim.x * blockDim.x) >> 5;
    const int H8 = H >> 3;
    for (long long t = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += nwarps_total) {
        int rows[KC];
        float p[KC];
        unsigned mask[KC];
#pragma unroll
        for (int c = 0; c < KC; c++) {
            const int k = c * 32 + lane;
            int r = -1;
            float pk = 0.0f;
            if (k < K) {
                r = __ldg(row_map + t * K + k);
                pk = __ldg(probs + t * K + k);
                if (r < 0) dprobs[t * K + k] = 0.0f;       // invalid route: no gradient
            }
            rows[c] = r;
            p[c] = pk;
            mask[c] = __ballot_sync(FULL, r >= 0);
        }
        const uint4* g = dy + t * H8;
#pragma unroll
        for (int c = 0; c < KC; c++) {
            unsigned m = mask[c];
            while (m) {
                int rr[RB], kk[RB];
                float pp[RB], dot[RB];
                bool on[RB];
#pragma unroll
                for (int qq = 0; qq < RB; qq++) {
                    on[qq] = m != 0u;
                    const int b = on[qq] ? __ffs(m) - 1 : 0;
                    if (on[qq]) m &= m - 1;
                    rr[qq] = __shfl_sync(FULL, rows[c], b);
                    pp[qq] = __shfl_sync(FULL, p[c], b);
                    kk[qq] = c * 32 + b;
                    dot[qq] = 0.0f;
                }
                for (int j0 = 0; j0 < H8; j0 += 32) {   // warp-uniform (the quantiser's quads)
                    const int j = j0 + lane;
                    const bool in = j < H8;
                    float gv[8];
                    bf16x8_to_f32(in ? __ldg(g + j) : make_uint4(0, 0, 0, 0), gv);
                    uint4 v[RB];
#pragma unroll
                    for (int qq = 0; qq < RB; qq++)
                        v[qq] = on[qq] && in ? __ldg(y_perm + (long long)rr[qq] * H8 + j) : make_uint4(0, 0, 0, 0);
#pragma unroll
                    for (int qq = 0; qq < RB; qq++) {
                        if (!on[qq]) continue;                 // warp-uniform
                        float yv[8], o[8];
                        bf16x8_to_f32(v[qq], yv);
#pragma unroll
                        for (int i = 0; i < 8; i++) {
                            dot[qq] = fmaf(gv[i], yv[i], dot[qq]);
                            o[i] = pp[qq] * gv[i];
                        }
                        const uint4 ob = f32_to_bf16x8(o);
                        if (in) __stcs(dy_perm + (long long)rr[qq] * H8 + j, ob);
                        if constexpr (Q) {
                            float f[8];
                            bf16x8_to_f32(ob, f);               // the stored bf16 values
                            int sb;
                            const uint2 code = quant8_in_quad(f, &sb);
                            if (in) {
                                q[(long long)rr[qq] * H8 + j] = code;
                                if ((lane & 3) == 0) qs[(long long)rr[qq] * (H >> 5) + (j >> 2)] = (uint8_t)sb;
                            }
                        }
                    }
                }
#pragma unroll
                for (int qq = 0; qq < RB; qq++) {
                    float d = dot[qq];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(FULL, d, o);
                    if (on[qq] && lane == 0) dprobs[t * K + kk[qq]] = d;
                }
            }
        }
    }
}

int device_sms() {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_permute_backward(const void* dx_perm, const int32_t* row_map, int T, int K, int H,
                                           void* dx, moe_stream_t stream) {
    using namespace moe;
    if (T < 0 || K < 1 || K > 128 || H < 8 || (H % 8) != 0) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!dx_perm || !row_map || !dx) return MOE_ERR_INVALID_ARG;
    if (!moe_host::aligned(dx_perm, 16) || !moe_host::aligned(dx, 16) || !moe_host::aligned(row_map, 4))
        return MOE_ERR_ALIGNMENT;
    long long blocks = ((long long)T + 7) / 8;
    const long long cap = (long long)device_sms() * 16;
    if (blocks > cap) blocks = cap;
    cudaStream_t s = moe_host::as_stream(stream);
    const int KC = (K + 31) / 32;
    const int H8 = H / 8;
    const int CH = H8 >= 128 ? 4 : (H8 >= 64 ? 2 : 1);
    const uint4* xp = (const uint4*)dx_perm;
    uint4* xo = (uint4*)dx;
#define MOE_PERMUTE_BWD(kc, ch) \
    combine_kernel<kc, ch, (ch == 4 ? 2 : 4), true><<<(int)blocks, 256, 0, s>>>(xp, row_map, nullptr, T, K, H, xo)
    if (KC == 1) {
        if (CH == 4) MOE_PERMUTE_BWD(1, 4); else if (CH == 2) MOE_PERMUTE_BWD(1, 2); else MOE_PERMUTE_BWD(1, 1);
    } else if (KC == 2) {
        if (CH == 4) MOE_PERMUTE_BWD(2, 4); else if (CH == 2) MOE_PERMUTE_BWD(2, 2); else MOE_PERMUTE_BWD(2, 1);
    } else {
        if (CH == 4) MOE_PERMUTE_BWD(4, 4); else if (CH == 2) MOE_PERMUTE_BWD(4, 2); else MOE_PERMUTE_BWD(4, 1);
    }
#undef MOE_PERMUTE_BWD
    return moe_host::launch_status();
}

extern "C" moe_status moe_unpermute_combine_backward(const void* dy, const void* y_perm, const int32_t* row_map,
                                                     const float* probs, int T, int K, int H, void* dy_perm,
                                                     float* dprobs, uint8_t* dy_perm_q, uint8_t* dy_perm_scales,
                                                     moe_stream_t stream) {
    using namespace moe;
    if (T < 0 || K < 1 || K > 128 || H < 8 || (H % 8) != 0) return MOE_ERR_INVALID_ARG;
    const bool quant = dy_perm_q != nullptr || dy_perm_scales != nullptr;
    if (quant && (!dy_perm_q || !dy_perm_scales || (H % 32) != 0)) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!dy || !y_perm || !row_map || !probs || !dy_perm || !dprobs) return MOE_ERR_INVALID_ARG;
    if (!moe_host::aligned(dy, 16) || !moe_host::aligned(y_perm, 16) || !moe_host::aligned(dy_perm, 16) ||
        !moe_host::aligned(row_map, 4) || !moe_host::aligned(probs, 4) || !moe_host::aligned(dprobs, 4) ||
        (quant && !moe_host::aligned(dy_perm_q, 8)))
        return MOE_ERR_ALIGNMENT;
    long long blocks = ((long long)T + 7) / 8;
    const long long cap = (long long)device_sms() * 16;
    if (blocks > cap) blocks = cap;
    cudaStream_t s = moe_host::as_stream(stream);
    const int KC = (K + 31) / 32;
#define MOE_COMBINE_BWD(kc, qz)                                                                          \
    combine_backward_kernel<kc, 4, qz><<<(int)blocks, 256, 0, s>>>((const uint4*)dy, (const uint4*)y_perm, \
                                                                   row_map, probs, T, K, H, (uint4*)dy_perm, \
                                                                   dprobs, (uint2*)dy_perm_q, dy_perm_scales)
    if (quant) {
        if (KC == 1) MOE_COMBINE_BWD(1, true);
        else if (KC == 2) MOE_COMBINE_BWD(2, true);
        else MOE_COMBINE_BWD(4, true);
    } else {
        if (KC == 1) MOE_COMBINE_BWD(1, false);
        else if (KC == 2) MOE_COMBINE_BWD(2, false);
        else MOE_COMBINE_BWD(4, false);
    }
#undef MOE_COMBINE_BWD
    return moe_host::launch_status();
}
