// router_sigmoid.cu -- sigmoid-score routing with a per-expert selection bias, and its
// backward: moe_route_sigmoid_topk and moe_route_sigmoid_topk_backward.
//
// "Sparser MoE end-to-end", sections "The workload changes the bottleneck" (the router's
// score transformation, top-k selection and router backward) and "Preserve a compact
// route" (bias statistics carried with compact [T, K] routes). The pages name these
// without defining them; the DeepSeek-style reading is taken:
//   score s_e = 1 / (1 + exp(-l_e)), selection key s_e + b_e (fp32), ids = the K largest
//   keys in descending order (lower index first on equal keys), probs = s at the ids, or
//   renormalised over the K selected scores. The bias steers only the selection; its
//   statistics (valid routes per expert) are what moe_permute writes as group_sizes.
//
// One warp per row. Lane l keeps the scores and keys of experts e = 32 i + l (i < NV) in
// registers; each of the K rounds takes the lanes' best keys and an arg-max across the
// warp (5 shuffle steps), and the winner's lane retires it. Rows are read once, coalesced.
//
// Exact selection. The ids are those of the logistic rounded once to fp32 from its exact
// value (a reference that rounds the exact score once). Double arithmetic is scarce on this
// part, so it is spent only where the decision needs it. A first pass ranks fp32 keys from
// expf (a few ulp from the exact ones) and takes the K largest and the next one: when every
// gap between these K + 1 keys exceeds a margin (2^-18 max(1, |key|): nearly three times the
// largest gap two keys a few ulp from exact can show -- expf is within 2 ulp, the add and the
// division round once each), the exact keys have the same K largest in the same order, and the first pass
// is the answer (probs from the fp32 scores, within a few ulp). Otherwise every expert whose
// fp32 key is within the margin of the K-th (tau) is a candidate -- no other can be among the
// K largest exact keys, as the first pass's K winners' exact keys all beat every other
// expert's -- the candidates get their exactly rounded scores and a second pass ranks them.
#include "common.cuh"

#include <math.h>

namespace moe {
namespace {

constexpr int SIG_KMAX = 64;       // K <= 64: two output slots per lane
constexpr int SIG_NVMAX = 32;      // E <= 1024: at most 32 experts per lane

// "a beats b": available first, then the larger key, then the lower expert index.
__device__ __forceinline__ bool key_beats(bool aa, float av, int ai, bool ba, float bv, int bi) {
    if (aa != ba) return aa;
    if (av != bv) return av > bv;
    return ai < bi;
}

__device__ __forceinline__ float logistic(float x) { return 1.0f / (1.0f + expf(-x)); }

// The logistic function evaluated in double and rounded once to fp32.
__device__ __forceinline__ float logistic_rn(float x) {
    return __double2float_rn(1.0 / (1.0 + exp(-(double)x)));
}

// One selection round over the lanes' available slots: the warp-wide winner (largest key,
// lower expert index on equal keys); bi = 0x7fffffff when no slot is available anywhere.
template <int NV>
__device__ __forceinline__ void warp_best(const float (&key)[NV], uint32_t avail, int lane, bool& ba, float& bv,
                                          int& bi) {
    ba = false;
    bv = 0.0f;
    bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < NV; i++) {          // strict comparison over ascending i: lower index on ties
        const bool a = (avail >> i) & 1u;
        if (a && (!ba || key[i] > bv)) {
            ba = true;
            bv = key[i];
            bi = i * 32 + lane;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const bool oa = __shfl_xor_sync(FULL, (int)ba, o) != 0;
        const float ov = __shfl_xor_sync(FULL, bv, o);
        const int oi = __shfl_xor_sync(FULL, bi, o);
        if (key_beats(oa, ov, oi, ba, bv, bi)) {
            ba = oa;
            bv = ov;
            bi = oi;
        }
    }
}

__device__ __forceinline__ void store_route_id(void* ids, bool i16, long long i, int id) {
    if (i16) static_cast<int16_t*>(ids)[i] = (int16_t)id;
    else static_cast<int32_t*>(ids)[i] = id;
}

template <int NV>
__global__ void __launch_bounds__(256) route_sigmoid_kernel(const float* __restrict__ logits,
                                                            const float* __restrict__ bias, int T, int E,
                                                            int K, void* __restrict__ ids, bool i16,
                                                            float* __restrict__ probs, bool renorm) {
    pdl_trigger();   // the permute that follows may launch now (it waits for the routes)
    const int lane = (int)lane_id();
    const int nwarps_total = (gridDim.x * blockDim.x) >> 5;
    // the bias of this lane's experts (the same for every row)
    float b[NV];
#pragma unroll
    for (int i = 0; i < NV; i++) {
        const int e = i * 32 + lane;
        b[i] = (bias != nullptr && e < E) ? __ldg(bias + e) : 0.0f;
    }
    for (long long t = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += nwarps_total) {
        const float* l = logits + t * E;
        float s[NV], key[NV];
        uint32_t avail = 0u;
#pragma unroll
        for (int i = 0; i < NV; i++) {
            const int e = i * 32 + lane;
            s[i] = 0.0f;
            key[i] = 0.0f;
            if (e < E) {
                s[i] = logistic(__ldg(l + e));
                key[i] = __fadd_rn(s[i], b[i]);
                avail |= 1u << i;
            }
        }
        // K rounds of selection over the available slots: the winners in order, their scores
        // (handed over by the winner's lane) and the sum of those scores
        float out_s0 = 0.0f, out_s1 = 0.0f;
        int out_e0 = 0, out_e1 = 0;
        float Z = 0.0f;
        auto take = [&](int k, int bi, uint32_t& left) {
            const int slot = bi >> 5;
            float mine = 0.0f;
#pragma unroll
            for (int i = 0; i < NV; i++)
                if (i == slot) mine = s[i];
            const float sw = __shfl_sync(FULL, mine, bi & 31);
            if (lane == (bi & 31)) left &= ~(1u << slot);
            Z += sw;                                      // same order in every lane
            if (lane == (k & 31)) {
                if (k < 32) {
                    out_s0 = sw;
                    out_e0 = bi;
                } else {
                    out_s1 = sw;
                    out_e1 = bi;
                }
            }
        };
        // first pass on the fp32 keys: the K largest in order, and the next one; when two of
        // these K + 1 keys are within the margin of each other, the row takes the exact pass
        float tau = 0.0f, prev = 0.0f;
        bool near = false;
        {
            uint32_t left = avail;
            const int rounds = K < E ? K + 1 : K;
            for (int k = 0; k < rounds; k++) {
                bool ba;
                float bv;
                int bi;
                warp_best<NV>(key, left, lane, ba, bv, bi);   // the same in every lane
                if (k > 0 && prev - bv <= fmaxf(1.0f, fmaxf(fabsf(prev), fabsf(bv))) * (1.0f / 262144.0f))
                    near = true;
                prev = bv;
                if (k == K) break;
                tau = bv;
                take(k, bi, left);
            }
        }
        if (near) {
            // candidates: fp32 keys within the margin of tau, given their exactly rounded scores
            const float margin = fmaxf(1.0f, fabsf(tau)) * (1.0f / 262144.0f);
            const bool all_cand = !isfinite(tau);
#pragma unroll
            for (int i = 0; i < NV; i++) {
                if (!((avail >> i) & 1u)) continue;
                if (all_cand || key[i] >= tau - margin) {
                    s[i] = logistic_rn(__ldg(l + i * 32 + lane));
                    key[i] = __fadd_rn(s[i], b[i]);
                } else {
                    avail &= ~(1u << i);
                }
            }
            Z = 0.0f;
            for (int k = 0; k < K; k++) {       // second pass: the candidates' exact keys
                bool ba;
                float bv;
                int bi;
                // at least K candidates, so a winner always exists
                warp_best<NV>(key, avail, lane, ba, bv, bi);
                take(k, bi, avail);
            }
        }
        const float inv = renorm ? 1.0f / Z : 1.0f;
        if (lane < K) {
            store_route_id(ids, i16, t * K + lane, out_e0);
            probs[t * K + lane] = renorm ? out_s0 * inv : out_s0;
        }
        if (lane + 32 < K) {
            store_route_id(ids, i16, t * K + lane + 32, out_e1);
            probs[t * K + lane + 32] = renorm ? out_s1 * inv : out_s1;
        }
    }
}

// Backward, one warp per row, selection held fixed (set semantics: a repeated id counts
// once, its slots' gradients summed; invalid ids are skipped). G_e, s_e = logistic(l_e),
// Z = sum over the selected experts of s_e, p_e = s_e / Z, c = sum of G_e p_e:
//   dlogits[t,e] = G_e s_e (1 - s_e)                 without renormalisation
//   dlogits[t,e] = s_e (1 - s_e) (G_e - c) / Z       with it
// for selected e, 0 elsewhere.
template <int KC>
__global__ void __launch_bounds__(256) route_sigmoid_backward_kernel(const float* __restrict__ logits,
                                                                     const void* __restrict__ ids, bool i16,
                                                                     const float* __restrict__ dprobs, int T,
                                                                     int E, int K, bool renorm,
                                                                     float* __restrict__ dlogits) {
    const int lane = (int)lane_id();
    const int nwarps_total = (gridDim.x * blockDim.x) >> 5;
    for (long long t = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += nwarps_total) {
        const float* l = logits + t * E;
        float* out = dlogits + t * E;
        int id[KC];
        float g[KC];
        bool first[KC];
#pragma unroll
        for (int c = 0; c < KC; c++) {
            const int k = c * 32 + lane;
            int e = -1;
            float gk = 0.0f;
            if (k < K) {
                e = i16 ? (int)reinterpret_cast<const int16_t*>(ids)[t * K + k]
                        : reinterpret_cast<const int32_t*>(ids)[t * K + k];
                if (e < 0 || e >= E) e = -1;
                gk = e >= 0 ? __ldg(dprobs + t * K + k) : 0.0f;
            }
            id[c] = e;
            g[c] = gk;
            first[c] = e >= 0;
        }
        // G_e gathered on each expert's first slot; later slots of the same expert step aside
#pragma unroll
        for (int c2 = 0; c2 < KC; c2++)
            for (int b = 0; b < 32; b++) {
                if (c2 * 32 + b >= K) break;          // warp-uniform
                const int e2 = __shfl_sync(FULL, id[c2], b);
                const float g2 = __shfl_sync(FULL, g[c2], b);
                const int k2 = c2 * 32 + b;
#pragma unroll
                for (int c = 0; c < KC; c++) {
                    const int k = c * 32 + lane;
                    if (id[c] >= 0 && e2 == id[c] && k2 != k) {
                        if (k2 < k) first[c] = false;
                        else g[c] += g2;
                    }
                }
            }
        float se[KC];
        float Z = 0.0f;
#pragma unroll
        for (int c = 0; c < KC; c++) {
            se[c] = first[c] ? logistic(__ldg(l + id[c])) : 0.0f;
            Z += se[c];
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) Z += __shfl_xor_sync(FULL, Z, o);
        const float invZ = Z > 0.0f ? 1.0f / Z : 0.0f;
        float cs = 0.0f;
#pragma unroll
        for (int c = 0; c < KC; c++) cs += first[c] ? g[c] * se[c] * invZ : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) cs += __shfl_xor_sync(FULL, cs, o);
        for (int e = lane; e < E; e += 32) out[e] = 0.0f;
        __syncwarp();
#pragma unroll
        for (int c = 0; c < KC; c++)
            if (first[c]) {
                const float w = se[c] * (1.0f - se[c]);
                out[id[c]] = renorm ? w * (g[c] - cs) * invZ : g[c] * w;
            }
        __syncwarp();
    }
}

int sm_count() {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}

template <int NV>
void launch_sigmoid(const float* logits, const float* bias, int T, int E, int K, void* ids, bool i16,
                    float* probs, bool renorm, cudaStream_t s) {
    long long blocks = ((long long)T + 7) / 8;
    const long long cap = (long long)sm_count() * 8;
    if (blocks > cap) blocks = cap;
    route_sigmoid_kernel<NV><<<(int)blocks, 256, 0, s>>>(logits, bias, T, E, K, ids, i16, probs, renorm);
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_route_sigmoid_topk(const float* logits, const float* expert_bias, int T, int E, int K,
                                             void* ids, moe_dtype id_dtype, float* probs, unsigned flags,
                                             moe_stream_t stream) {
    using namespace moe;
    if (T < 0 || E < 1 || K < 1 || K > E) return MOE_ERR_INVALID_ARG;
    if (id_dtype != MOE_I16 && id_dtype != MOE_I32) return MOE_ERR_INVALID_ARG;
    if (id_dtype == MOE_I16 && E > 32767) return MOE_ERR_INVALID_ARG;
    if (flags & ~MOE_ROUTE_RENORM) return MOE_ERR_INVALID_ARG;
    if (E > 32 * SIG_NVMAX || K > SIG_KMAX) return MOE_ERR_UNSUPPORTED;
    if (T == 0) return MOE_OK;
    if (!logits || !ids || !probs) return MOE_ERR_INVALID_ARG;
    if (!moe_host::aligned(logits, 4) || !moe_host::aligned(probs, 4) ||
        (expert_bias && !moe_host::aligned(expert_bias, 4)) ||
        !moe_host::aligned(ids, id_dtype == MOE_I16 ? 2 : 4))
        return MOE_ERR_ALIGNMENT;
    const bool i16 = id_dtype == MOE_I16;
    const bool renorm = (flags & MOE_ROUTE_RENORM) != 0;
    cudaStream_t s = moe_host::as_stream(stream);
    const int nv = (E + 31) / 32;
    if (nv <= 1) launch_sigmoid<1>(logits, expert_bias, T, E, K, ids, i16, probs, renorm, s);
    else if (nv <= 2) launch_sigmoid<2>(logits, expert_bias, T, E, K, ids, i16, probs, renorm, s);
    else if (nv <= 4) launch_sigmoid<4>(logits, expert_bias, T, E, K, ids, i16, probs, renorm, s);
    else if (nv <= 8) launch_sigmoid<8>(logits, expert_bias, T, E, K, ids, i16, probs, renorm, s);
    else if (nv <= 16) launch_sigmoid<16>(logits, expert_bias, T, E, K, ids, i16, probs, renorm, s);
    else launch_sigmoid<32>(logits, expert_bias, T, E, K, ids, i16, probs, renorm, s);
    return moe_host::launch_status();
}

extern "C" moe_status moe_route_sigmoid_topk_backward(const float* logits, const void* ids, moe_dtype id_dtype,
                                                      const float* dprobs, int T, int E, int K, unsigned flags,
                                                      float* dlogits, moe_stream_t stream) {
    using namespace moe;
    if (T < 0 || E < 1 || K < 1 || K > E || K > 128) return MOE_ERR_INVALID_ARG;
    if (id_dtype != MOE_I16 && id_dtype != MOE_I32) return MOE_ERR_INVALID_ARG;
    if (flags & ~MOE_ROUTE_RENORM) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!logits || !ids || !dprobs || !dlogits) return MOE_ERR_INVALID_ARG;
    if (!moe_host::aligned(logits, 4) || !moe_host::aligned(dprobs, 4) || !moe_host::aligned(dlogits, 4) ||
        !moe_host::aligned(ids, id_dtype == MOE_I16 ? 2 : 4))
        return MOE_ERR_ALIGNMENT;
    long long blocks = ((long long)T + 7) / 8;
    const long long cap = (long long)sm_count() * 16;
    if (blocks > cap) blocks = cap;
    cudaStream_t s = moe_host::as_stream(stream);
    const bool i16 = id_dtype == MOE_I16;
    const bool renorm = (flags & MOE_ROUTE_RENORM) != 0;
    const int KC = (K + 31) / 32;
#define MOE_SIG_BWD(kc)                                                                                    \
    route_sigmoid_backward_kernel<kc><<<(int)blocks, 256, 0, s>>>(logits, ids, i16, dprobs, T, E, K, renorm, \
                                                                  dlogits)
    if (KC == 1) MOE_SIG_BWD(1);
    else if (KC == 2) MOE_SIG_BWD(2);
    else MOE_SIG_BWD(4);
#undef MOE_SIG_BWD
    return moe_host::launch_status();
}
