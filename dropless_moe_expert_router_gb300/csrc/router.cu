// router.cu -- router top-K kernels and the moe_route_topk entry point.
//
// Two paths ("Sparser MoE end-to-end", section "Preserve a compact route"):
//  * small E and K: a warp (or a group of G lanes of a warp) per row keeps the
//    logits in registers and runs K rounds of a segmented arg-max;
//  * large E and K (e.g. 2,304 experts, top-36): radix select -- three bounded
//    histogram passes (11/11/10-bit digits of an order-preserving key) find the
//    exact K-th largest key, only candidates matching the narrowed prefix are
//    counted after the first pass, and the K winners are ranked in a final
//    O(K^2 / 32) step instead of K full-row scans.
// Output: ids [T, K] (selection order: descending logit, lower index on ties),
// probs [T, K] fp32 (softmax over all E logits at the selected ids, or over the
// K selected logits with MOE_ROUTE_RENORM).
#include "common.cuh"

#include <math.h>

namespace moe {
namespace {

constexpr int RADIX_WARPS = 4;    // warps (rows in flight) per block of the radix kernel
constexpr int KMAX = 128;         // largest K of the radix kernel (list in shared memory)

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, o));
    return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
    return v;
}

__device__ __forceinline__ void store_route(void* ids, bool i16, long long i, int id) {
    if (i16) ((int16_t*)ids)[i] = (int16_t)id;
    else ((int32_t*)ids)[i] = id;
}

// "a beats b": larger logit, then lower index; unavailable entries lose to all.
__device__ __forceinline__ bool beats(bool aa, float av, int ai, bool ba, float bv, int bi) {
    if (aa != ba) return aa;
    if (av != bv) return av > bv;
    return ai < bi;
}

// ---------------------------------------------------------------------------
// Small path: G lanes per row (32 / G rows per warp), V logits per lane
// (expert index = i * G + lane_in_group). E <= G * V, K <= 16.
// ---------------------------------------------------------------------------
template <int G, int V>
__global__ void __launch_bounds__(256) route_small_kernel(const float* __restrict__ logits, int T, int E,
                                                          int K, void* ids, bool i16,
                                                          float* __restrict__ probs, bool renorm) {
    const int lane = (int)lane_id();
    const int gl = lane % G;
    const long long gwarp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const long long t = gwarp * (32 / G) + lane / G;
    const bool row_ok = t < T;

    float v[V];
    bool avail[V];
    int rank[V];
#pragma unroll
    for (int i = 0; i < V; i++) {
        int e = i * G + gl;
        avail[i] = row_ok && e < E;
        v[i] = avail[i] ? __ldg(logits + t * E + e) : -INFINITY;
        rank[i] = -1;
    }
    // row maximum
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < V; i++) m = fmaxf(m, v[i]);
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, o));

    // K rounds of segmented arg-max
    for (int k = 0; k < K; k++) {
        bool ba = false;
        float bv = -INFINITY;
        int bi = 0x7fffffff;
#pragma unroll
        for (int i = 0; i < V; i++) {
            int e = i * G + gl;
            if (beats(avail[i], v[i], e, ba, bv, bi)) { ba = avail[i]; bv = v[i]; bi = e; }
        }
#pragma unroll
        for (int o = G / 2; o > 0; o >>= 1) {
            bool oa = __shfl_xor_sync(FULL, ba, o);
            float ov = __shfl_xor_sync(FULL, bv, o);
            int oi = __shfl_xor_sync(FULL, bi, o);
            if (beats(oa, ov, oi, ba, bv, bi)) { ba = oa; bv = ov; bi = oi; }
        }
#pragma unroll
        for (int i = 0; i < V; i++)
            if (avail[i] && i * G + gl == bi) { avail[i] = false; rank[i] = k; }
    }
    // denominators
    float den = 0.0f;
#pragma unroll
    for (int i = 0; i < V; i++) {
        int e = i * G + gl;
        bool real = row_ok && e < E;
        if (real && (!renorm || rank[i] >= 0)) den += expf(v[i] - m);
    }
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) den += __shfl_xor_sync(FULL, den, o);
    if (!row_ok) return;
#pragma unroll
    for (int i = 0; i < V; i++) {
        if (rank[i] >= 0) {
            long long o = t * K + rank[i];
            store_route(ids, i16, o, i * G + gl);
            probs[o] = expf(v[i] - m) / den;
        }
    }
}

// ---------------------------------------------------------------------------
// Radix path: one warp per row, V = ceil(E/32) logits per lane in registers
// (expert index = i * 32 + lane, so every load is a coalesced 128-byte line).
// ---------------------------------------------------------------------------

// Order-preserving key: larger float -> larger unsigned; -0 and +0 map to one key.
__device__ __forceinline__ unsigned f2key(float f) {
    unsigned u = __float_as_uint(f);
    if ((u << 1) == 0) u = 0;  // -0 -> +0
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key2f(unsigned k) {
    return (k & 0x80000000u) ? __uint_as_float(k & 0x7fffffffu) : __uint_as_float(~k);
}

// Inclusive suffix sum over lanes (lane l gets sum of lanes >= l).
__device__ __forceinline__ unsigned suffix_sum(unsigned v, int lane) {
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        unsigned o = __shfl_down_sync(FULL, v, d);
        if (lane + d < 32) v += o;
    }
    return v;
}

// Find the bin holding the rem-th largest element of a histogram of nb bins
// (nb = 2048 or 1024) in shared memory. Returns the bin; *above = number of
// elements in higher bins.
__device__ __forceinline__ int find_bin(const unsigned* hist, int nb, unsigned rem, int lane,
                                        unsigned* above) {
    const int per = nb / 32;                    // bins per lane at the first level
    unsigned s = 0;
    for (int j = 0; j < per; j++) s += hist[lane * per + j];
    unsigned suf = suffix_sum(s, lane);
    unsigned nxt = __shfl_down_sync(FULL, suf, 1);
    if (lane == 31) nxt = 0;
    int L = __ffs(__ballot_sync(FULL, suf >= rem && nxt < rem)) - 1;
    unsigned aboveL = __shfl_sync(FULL, nxt, L);
    // second level: lane L's `per` bins, per/32 to a lane
    const int q = per / 32;
    unsigned s2 = 0;
    for (int j = 0; j < q; j++) s2 += hist[L * per + lane * q + j];
    unsigned suf2 = suffix_sum(s2, lane);
    unsigned nxt2 = __shfl_down_sync(FULL, suf2, 1);
    if (lane == 31) nxt2 = 0;
    int L2 = __ffs(__ballot_sync(FULL, aboveL + suf2 >= rem && aboveL + nxt2 < rem)) - 1;
    unsigned acc = aboveL + __shfl_sync(FULL, nxt2, L2);
    int base = L * per + L2 * q;
    int bin = base;
    for (int j = q - 1; j >= 0; j--) {
        unsigned c = hist[base + j];
        if (acc + c >= rem) { bin = base + j; break; }
        acc += c;
    }
    *above = acc;
    return bin;
}

template <int V>
__global__ void __launch_bounds__(RADIX_WARPS * 32) route_radix_kernel(const float* __restrict__ logits,
                                                                       int T, int E, int K, void* ids,
                                                                       bool i16, float* __restrict__ probs,
                                                                       bool renorm) {
    __shared__ unsigned s_hist[RADIX_WARPS][2048];
    __shared__ unsigned s_key[RADIX_WARPS][KMAX];
    __shared__ int s_idx[RADIX_WARPS][KMAX];
    const int warp = threadIdx.x >> 5;
    const int lane = (int)lane_id();
    unsigned* hist = s_hist[warp];
    unsigned* lkey = s_key[warp];
    int* lidx = s_idx[warp];

    for (long long t = (long long)blockIdx.x * RADIX_WARPS + warp; t < T;
         t += (long long)gridDim.x * RADIX_WARPS) {
        const float* row = logits + t * E;
        unsigned key[V];
        float m = -INFINITY;
#pragma unroll
        for (int i = 0; i < V; i++) {
            int e = i * 32 + lane;
            float x = (e < E) ? __ldg(row + e) : -INFINITY;
            key[i] = (e < E) ? f2key(x) : 0u;   // absent slots: key 0, below every real key
            m = fmaxf(m, x);
        }
        m = warp_max(m);
        float den = 0.0f;
        if (!renorm) {
#pragma unroll
            for (int i = 0; i < V; i++)
                if (i * 32 + lane < E) den += expf(key2f(key[i]) - m);
            den = warp_sum(den);
        }

        // three histogram passes over 11/11/10-bit digits, each restricted to the
        // keys that match the prefix found so far
        unsigned prefix = 0, pmask = 0, rem = (unsigned)K;
#pragma unroll 1
        for (int p = 0; p < 3; p++) {
            const int sh = p == 0 ? 21 : (p == 1 ? 10 : 0);
            const int nbits = p == 2 ? 10 : 11;
            const int nb = 1 << nbits;
            const unsigned dmask = (unsigned)nb - 1u;
            for (int b = lane; b < nb; b += 32) hist[b] = 0u;
            __syncwarp();
#pragma unroll
            for (int i = 0; i < V; i++)
                if (key[i] != 0u && (key[i] & pmask) == prefix) atomicAdd(&hist[(key[i] >> sh) & dmask], 1u);
            __syncwarp();
            unsigned above;
            int bin = find_bin(hist, nb, rem, lane, &above);
            rem -= above;
            prefix |= (unsigned)bin << sh;
            pmask |= dmask << sh;
            __syncwarp();
        }
        // prefix is now the exact K-th largest key; take every key above it and
        // the `rem` lowest-index keys equal to it
        const unsigned tau = prefix;
        unsigned tie_left = rem;
        int base = 0;
#pragma unroll
        for (int i = 0; i < V; i++) {
            int e = i * 32 + lane;
            bool real = e < E;
            bool gt = real && key[i] > tau;
            bool eq = real && key[i] == tau;
            unsigned meq = __ballot_sync(FULL, eq);
            unsigned r = (unsigned)__popc(meq & lanemask_lt());
            bool take = gt || (eq && r < tie_left);
            unsigned ne = (unsigned)__popc(meq);
            tie_left -= ne < tie_left ? ne : tie_left;
            unsigned mt = __ballot_sync(FULL, take);
            if (take) {
                int pos = base + __popc(mt & lanemask_lt());
                lkey[pos] = key[i];
                lidx[pos] = e;
            }
            base += __popc(mt);
        }
        __syncwarp();
        if (renorm) {
            for (int j = lane; j < K; j += 32) den += expf(key2f(lkey[j]) - m);
            den = warp_sum(den);
        }
        // rank the K winners: descending key, ascending index
        for (int j = lane; j < K; j += 32) {
            unsigned kj = lkey[j];
            int ij = lidx[j];
            int rk = 0;
            for (int j2 = 0; j2 < K; j2++) {
                unsigned k2 = lkey[j2];
                rk += (k2 > kj) || (k2 == kj && lidx[j2] < ij);
            }
            long long o = t * K + rk;
            store_route(ids, i16, o, ij);
            probs[o] = expf(key2f(kj) - m) / den;
        }
        __syncwarp();
    }
}

template <int G, int V>
cudaError_t launch_small(const float* logits, int T, int E, int K, void* ids, bool i16, float* probs,
                         bool renorm, cudaStream_t s) {
    const int rows_per_block = 8 * (32 / G);
    int blocks = (T + rows_per_block - 1) / rows_per_block;
    route_small_kernel<G, V><<<blocks, 256, 0, s>>>(logits, T, E, K, ids, i16, probs, renorm);
    return cudaGetLastError();
}

template <int V>
cudaError_t launch_radix(const float* logits, int T, int E, int K, void* ids, bool i16, float* probs,
                         bool renorm, cudaStream_t s) {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    long long need = ((long long)T + RADIX_WARPS - 1) / RADIX_WARPS;
    long long cap = (long long)sms * 8;
    int blocks = (int)(need < cap ? need : cap);
    route_radix_kernel<V><<<blocks, RADIX_WARPS * 32, 0, s>>>(logits, T, E, K, ids, i16, probs, renorm);
    return cudaGetLastError();
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_route_topk(const float* logits, int T, int E, int K, void* ids,
                                     moe_dtype id_dtype, float* probs, unsigned flags,
                                     moe_stream_t stream) {
    using namespace moe;
    if (T < 0 || E < 1 || K < 1 || K > E) return MOE_ERR_INVALID_ARG;
    if (id_dtype != MOE_I16 && id_dtype != MOE_I32) return MOE_ERR_INVALID_ARG;
    if (id_dtype == MOE_I16 && E > 32767) return MOE_ERR_INVALID_ARG;
    if (flags & ~MOE_ROUTE_RENORM) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!logits || !ids || !probs) return MOE_ERR_INVALID_ARG;
    if (!moe_host::aligned(logits, 4) || !moe_host::aligned(probs, 4) ||
        !moe_host::aligned(ids, id_dtype == MOE_I16 ? 2 : 4))
        return MOE_ERR_ALIGNMENT;
    const bool i16 = id_dtype == MOE_I16;
    const bool renorm = (flags & MOE_ROUTE_RENORM) != 0;
    cudaStream_t s = moe_host::as_stream(stream);
    cudaError_t err;
    if (E <= 256 && K <= 16) {
        if (E <= 1) err = launch_small<1, 1>(logits, T, E, K, ids, i16, probs, renorm, s);
        else if (E <= 2) err = launch_small<2, 1>(logits, T, E, K, ids, i16, probs, renorm, s);
        else if (E <= 4) err = launch_small<4, 1>(logits, T, E, K, ids, i16, probs, renorm, s);
        else if (E <= 8) err = launch_small<8, 1>(logits, T, E, K, ids, i16, probs, renorm, s);
        else if (E <= 16) err = launch_small<16, 1>(logits, T, E, K, ids, i16, probs, renorm, s);
        else if (E <= 32) err = launch_small<32, 1>(logits, T, E, K, ids, i16, probs, renorm, s);
        else if (E <= 64) err = launch_small<32, 2>(logits, T, E, K, ids, i16, probs, renorm, s);
        else if (E <= 128) err = launch_small<32, 4>(logits, T, E, K, ids, i16, probs, renorm, s);
        else err = launch_small<32, 8>(logits, T, E, K, ids, i16, probs, renorm, s);
    } else {
        if (K > KMAX || E > 4096) return MOE_ERR_UNSUPPORTED;
        if (E <= 256) err = launch_radix<8>(logits, T, E, K, ids, i16, probs, renorm, s);
        else if (E <= 512) err = launch_radix<16>(logits, T, E, K, ids, i16, probs, renorm, s);
        else if (E <= 1024) err = launch_radix<32>(logits, T, E, K, ids, i16, probs, renorm, s);
        else if (E <= 2304) err = launch_radix<72>(logits, T, E, K, ids, i16, probs, renorm, s);
        else err = launch_radix<128>(logits, T, E, K, ids, i16, probs, renorm, s);
    }
    return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" size_t moe_route_ids_bytes(int T, int K, moe_dtype id_dtype) {
    if (T < 0 || K < 0) return 0;
    return (size_t)T * (size_t)K * (id_dtype == MOE_I16 ? 2u : 4u);
}

extern "C" size_t moe_route_probs_bytes(int T, int K) {
    if (T < 0 || K < 0) return 0;
    return (size_t)T * (size_t)K * 4u;
}
