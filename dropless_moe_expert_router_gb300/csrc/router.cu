// router.cu -- router top-K kernels and the moe_route_topk entry point.
//
// Two paths ("Sparser MoE end-to-end", section "Preserve a compact route"):
//  * small E and K: a warp (or a group of G lanes of a warp) per row keeps the
//    logits in registers and runs K rounds of a segmented arg-max;
//  * large E and K (e.g. 2,304 experts, top-36): radix/threshold select -- a
//    bounded histogram pass over the top 11 bits of an order-preserving key
//    finds the bin of the K-th largest key, the candidates in that bin are
//    ranked directly (further 11- and 10-bit passes narrow the range only when
//    the bin is crowded), and the K winners are ranked in a final step; no
//    full-row scan per selected expert.
// Output: ids [T, K] (selection order: descending logit, lower index on ties),
// probs [T, K] fp32 (softmax over all E logits at the selected ids, or over the
// K selected logits with MOE_ROUTE_RENORM).
#include "common.cuh"

#include <math.h>

namespace moe {
namespace {

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

// ---------------------------------------------------------------------------
// Radix path, one CTA (256 threads) per row: V logits per thread, expert index
// e = i * 256 + tid (coalesced loads). The first histogram pass (top 11 bits of
// the key) finds the bin that holds the K-th largest key; the keys in that bin
// (normally a few dozen) are compacted and ranked directly. Only if that bin
// holds more than CAND_MAX keys do the next passes (11 and 10 bits) narrow it
// further, down to the exact K-th key.
// ---------------------------------------------------------------------------
constexpr int RT = 256;           // threads per row
constexpr int RW = RT / 32;       // warps per row
constexpr int CAND_MAX = 256;     // candidates ranked directly

struct RadixSmem {
    unsigned hist[2048];          // skewed: bin d at (d % 8) * 256 + d / 8
    unsigned cand_key[CAND_MAX];
    int cand_idx[CAND_MAX];
    unsigned list_key[KMAX];
    int list_idx[KMAX];
    float red[RW];
    unsigned ured[RW];
    int n_cand, n_list;
    unsigned bin, above;
};

__device__ __forceinline__ float block_max(float v, RadixSmem& sm) {
    v = warp_max(v);
    __syncthreads();
    if (lane_id() == 0) sm.red[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = sm.red[0];
#pragma unroll
    for (int w = 1; w < RW; w++) r = fmaxf(r, sm.red[w]);
    return r;
}
__device__ __forceinline__ float block_sum(float v, RadixSmem& sm) {
    v = warp_sum(v);
    __syncthreads();
    if (lane_id() == 0) sm.red[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = 0.0f;
#pragma unroll
    for (int w = 0; w < RW; w++) r += sm.red[w];
    return r;
}

// One histogram pass over keys matching (key & pmask) == prefix, on the digit
// (key >> sh) & (nb - 1); nb = 2048 or 1024. Sets sm.bin to the digit holding
// the rem-th largest matching key and sm.above to the matching keys in higher
// digits. Each thread owns nb / 256 consecutive digits.
template <int V>
__device__ void radix_pass(const unsigned (&key)[V], unsigned prefix, unsigned pmask, int sh, int nb,
                           unsigned rem, RadixSmem& sm) {
    const int tid = threadIdx.x, lane = (int)lane_id(), warp = tid >> 5;
    const int per = nb / RT;                       // 8 or 4 digits per thread
    const int pshift = per == 8 ? 3 : 2;
    for (int b = tid; b < nb; b += RT) sm.hist[b] = 0u;
    __syncthreads();
    const unsigned dmask = (unsigned)nb - 1u;
#pragma unroll
    for (int i = 0; i < V; i++)
        if (key[i] != 0u && (key[i] & pmask) == prefix) {
            const int d = (int)((key[i] >> sh) & dmask);
            atomicAdd(&sm.hist[((d & (per - 1)) << 8) + (d >> pshift)], 1u);
        }
    __syncthreads();
    unsigned s = 0;
    for (int j = 0; j < per; j++) s += sm.hist[j * RT + tid];
    // block suffix sum over threads (thread t: sum of threads >= t)
    unsigned suf = suffix_sum(s, lane);
    if (lane == 0) sm.ured[warp] = suf;             // warp total
    __syncthreads();
    unsigned later = 0;
    for (int w = warp + 1; w < RW; w++) later += sm.ured[w];
    suf += later;
    const unsigned nxt = suf - s;                   // sum of threads > t
    if (suf >= rem && nxt < rem) {                  // exactly one thread
        unsigned acc = nxt;
        int d = tid * per;
        for (int j = per - 1; j >= 0; j--) {
            const unsigned c = sm.hist[j * RT + tid];
            if (acc + c >= rem) { d = tid * per + j; break; }
            acc += c;
        }
        sm.bin = (unsigned)d;
        sm.above = acc;
    }
    __syncthreads();
}

template <int V>
__global__ void __launch_bounds__(RT, 5) route_radix_kernel(const float* __restrict__ logits, int T, int E,
                                                            int K, void* ids, bool i16, float* __restrict__ probs,
                                                            bool renorm) {
    __shared__ RadixSmem sm;
    const int tid = threadIdx.x, lane = (int)lane_id(), warp = tid >> 5;
    // the next row's logits are loaded while the current row is processed
    float xn[V];
    if (blockIdx.x < T) {
#pragma unroll
        for (int i = 0; i < V; i++) {
            const int e = i * RT + tid;
            xn[i] = (e < E) ? __ldg(logits + (long long)blockIdx.x * E + e) : -INFINITY;
        }
    }
    for (long long t = blockIdx.x; t < T; t += gridDim.x) {
        unsigned key[V];
        float m = -INFINITY;
#pragma unroll
        for (int i = 0; i < V; i++) {
            const int e = i * RT + tid;
            key[i] = (e < E) ? f2key(xn[i]) : 0u;   // absent slots: key 0, below every real key
            m = fmaxf(m, xn[i]);
        }
        const long long tn = t + gridDim.x;
        if (tn < T) {
#pragma unroll
            for (int i = 0; i < V; i++) {
                const int e = i * RT + tid;
                xn[i] = (e < E) ? __ldg(logits + tn * E + e) : -INFINITY;
            }
        }
        m = block_max(m, sm);
        float den = 0.0f;
        if (!renorm) {
#pragma unroll
            for (int i = 0; i < V; i++)
                if (key[i] != 0u) den += expf(key2f(key[i]) - m);
            den = block_sum(den, sm);
        }
        if (tid == 0) { sm.n_cand = 0; sm.n_list = 0; }
        // narrow the K-th key until its bin is small enough to rank directly
        unsigned prefix = 0, pmask = 0, rem = (unsigned)K;
        bool exact = false;
#pragma unroll 1
        for (int p = 0; p < 3; p++) {
            const int sh = p == 0 ? 21 : (p == 1 ? 10 : 0);
            const int nb = p == 2 ? 1024 : 2048;
            radix_pass<V>(key, prefix, pmask, sh, nb, rem, sm);
            rem -= sm.above;
            prefix |= sm.bin << sh;
            pmask |= ((unsigned)nb - 1u) << sh;
            const unsigned cnt = sm.hist[((sm.bin & (nb / RT - 1)) << 8) + (sm.bin >> (nb == 2048 ? 3 : 2))];
            if (p == 2) exact = true;
            else if (cnt <= CAND_MAX) break;
            __syncthreads();   // sm.bin / sm.hist reused by the next pass
        }
        // keys above the prefix go straight to the list; keys matching it are candidates
#pragma unroll
        for (int i = 0; i < V; i++) {
            const unsigned k = key[i];
            if (k == 0u) continue;
            const unsigned km = k & pmask;
            if (km > prefix) {
                const int pos = atomicAdd(&sm.n_list, 1);
                sm.list_key[pos] = k;
                sm.list_idx[pos] = i * RT + tid;
            } else if (km == prefix && !exact) {
                const int pos = atomicAdd(&sm.n_cand, 1);
                sm.cand_key[pos] = k;
                sm.cand_idx[pos] = i * RT + tid;
            }
        }
        if (exact) {
            // prefix is the K-th key itself: take the `rem` lowest-index keys equal to it, in index order
            unsigned taken = 0;
#pragma unroll
            for (int i = 0; i < V; i++) {
                const bool eq = key[i] == prefix && key[i] != 0u;
                const unsigned bal = __ballot_sync(FULL, eq);
                __syncthreads();
                if (lane == 0) sm.ured[warp] = __popc(bal);
                __syncthreads();
                unsigned before = taken;
                for (int w = 0; w < warp; w++) before += sm.ured[w];
                unsigned tot = taken;
                for (int w = 0; w < RW; w++) tot += sm.ured[w];
                const unsigned r = before + __popc(bal & lanemask_lt());
                if (eq && r < rem) {
                    const int pos = atomicAdd(&sm.n_list, 1);
                    sm.list_key[pos] = key[i];
                    sm.list_idx[pos] = i * RT + tid;
                }
                taken = tot;
            }
        }
        __syncthreads();
        if (!exact) {
            // rank the candidates (descending key, ascending index); the first rem join the list
            const int nc = sm.n_cand;
            for (int c = tid; c < nc; c += RT) {
                const unsigned kc = sm.cand_key[c];
                const int ic = sm.cand_idx[c];
                unsigned r = 0;
                for (int j = 0; j < nc; j++) {
                    const unsigned kj = sm.cand_key[j];
                    r += (kj > kc) || (kj == kc && sm.cand_idx[j] < ic);
                }
                if (r < rem) {
                    const int pos = atomicAdd(&sm.n_list, 1);
                    sm.list_key[pos] = kc;
                    sm.list_idx[pos] = ic;
                }
            }
            __syncthreads();
        }
        // the list holds exactly K keys: rank them and write ids / probs in order
        if (renorm) {
            float d = 0.0f;
            for (int j = tid; j < K; j += RT) d += expf(key2f(sm.list_key[j]) - m);
            den = block_sum(d, sm);
        }
        for (int j = tid; j < K; j += RT) {
            const unsigned kj = sm.list_key[j];
            const int ij = sm.list_idx[j];
            int rk = 0;
            for (int j2 = 0; j2 < K; j2++) {
                const unsigned k2 = sm.list_key[j2];
                rk += (k2 > kj) || (k2 == kj && sm.list_idx[j2] < ij);
            }
            const long long o = t * K + rk;
            store_route(ids, i16, o, ij);
            probs[o] = expf(key2f(kj) - m) / den;
        }
        __syncthreads();   // shared state is reused by the next row
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
    const long long cap = (long long)sms * 5;   // resident CTAs per SM at 48 registers: one wave
    const int blocks = (int)(T < cap ? T : cap);
    route_radix_kernel<V><<<blocks, RT, 0, s>>>(logits, T, E, K, ids, i16, probs, renorm);
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
        if (K > KMAX || E > 8192) return MOE_ERR_UNSUPPORTED;
        if (E <= 256) err = launch_radix<1>(logits, T, E, K, ids, i16, probs, renorm, s);
        else if (E <= 512) err = launch_radix<2>(logits, T, E, K, ids, i16, probs, renorm, s);
        else if (E <= 1024) err = launch_radix<4>(logits, T, E, K, ids, i16, probs, renorm, s);
        else if (E <= 2304) err = launch_radix<9>(logits, T, E, K, ids, i16, probs, renorm, s);
        else if (E <= 4096) err = launch_radix<16>(logits, T, E, K, ids, i16, probs, renorm, s);
        else err = launch_radix<32>(logits, T, E, K, ids, i16, probs, renorm, s);
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
