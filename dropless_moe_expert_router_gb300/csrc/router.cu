// router.cu -- router top-K kernels and the moe_route_topk entry point.
//
// Three paths ("Sparser MoE end-to-end", section "Preserve a compact route"):
//  * small E and K: a warp (or a group of G lanes of a warp) per row keeps the
//    logits in registers and runs K rounds of a segmented arg-max;
//  * large E and K with E % 4 == 0, E <= 2,304 (e.g. 2,304 experts, top-36):
//    threshold select, one warp per row -- a threshold from the lanes' own top
//    values bounds the K-th largest logit from below, the few logits above it
//    are ranked directly, and a warp-level exact search takes over for rows
//    with heavy ties;
//  * other large shapes: radix/threshold select, one CTA per row -- a bounded
//    histogram pass over the top 11 bits of an order-preserving key finds the
//    bin of the K-th largest key, the candidates in that bin are ranked
//    directly (further 11- and 10-bit passes narrow the range only when the
//    bin is crowded), and the K winners are ranked in a final step.
// No path scans the full row once per selected expert.
// Output: ids [T, K] (selection order: descending logit, lower index on ties),
// probs [T, K] fp32 (softmax over all E logits at the selected ids, or over the
// K selected logits with MOE_ROUTE_RENORM).
#include "common.cuh"
#include "sm100_ptx.cuh"

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
// (expert index = i * G + lane_in_group). E <= G * V, K <= 16. With one logit
// per lane each lane ranks its logit against the row's G in one pass; with
// more, K rounds of a segmented arg-max.
// ---------------------------------------------------------------------------
template <int G, int V>
__global__ void __launch_bounds__(256) route_small_kernel(const float* __restrict__ logits, int T, int E,
                                                          int K, void* ids, bool i16,
                                                          float* __restrict__ probs, bool renorm) {
    pdl_trigger();   // the permute that follows may launch now (it waits for the routes)
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

    if constexpr (V == 1) {
        // one logit per lane: its rank among the row's G logits (larger first, lower index
        // on ties) in one pass of G compares; a rank below K is the output slot
        const int e = gl;
        int r = 0;
        for (int j = 0; j < G; j++) {
            const bool oa = __shfl_sync(FULL, avail[0], (lane & ~(G - 1)) + j);
            const float ov = __shfl_sync(FULL, v[0], (lane & ~(G - 1)) + j);
            r += beats(oa, ov, j, avail[0], v[0], e) ? 1 : 0;
        }
        if (avail[0] && r < K) rank[0] = r;
    } else {
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
    pdl_trigger();   // the permute that follows may launch now (it waits for the routes)
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

// ---------------------------------------------------------------------------
// Filter path, one warp per row (rows 16-byte aligned, E % 4 == 0, E <= 128 NV4):
// lane l holds the float4s q = j*32 + l of its row (expert e = 4 q + c) and keeps
// its P largest logits. A 16-step search over the top 16 bits of the order-
// preserving key of those 32 P values gives a threshold tau with at least K
// logits >= tau (the K-th largest of a subset of the row is a lower bound of the
// row's K-th largest) and, normally, only a few more. The logits >= tau are
// compacted to shared memory and ranked directly; a winner's rank is its output
// slot. A row with more than FCAND logits >= tau (heavy ties) takes the exact
// path instead: a 32-step search for the K-th largest key, the larger logits
// ranked, and the logits equal to it taken in expert order.
// ---------------------------------------------------------------------------
constexpr int FW = 8;             // warps (rows in flight) per CTA
constexpr int FCAND = 256;        // candidates per warp ranked directly

// Shared memory of one CTA: per warp a row buffer (4 * 128 * NV4 bytes, filled by
// a bulk copy one row ahead), the candidate list and its ranks, a counter and an
// mbarrier.
struct FilterWarp {
    unsigned long long cand[FCAND];   // (logit, expert) as a pair, then as a 64-bit rank key
    int rank[FCAND];
    uint64_t bar;
    int n;
    uint32_t abort_flag;
};
template <int NV4>
constexpr size_t filter_smem_bytes() {
    return (size_t)FW * (512 * NV4 + sizeof(FilterWarp));
}

constexpr float LOG2E = 1.4426950408889634f;

// 2^y by the hardware approximation (relative error about 2^-22); exp(x - m) is
// taken as 2^(x log2(e) - m log2(e)) with one rounding for the exponent.
__device__ __forceinline__ float ex2_approx(float y) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(y));
    return r;
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Packed pair arithmetic (two fp32 lanes in one 64-bit register).
__device__ __forceinline__ unsigned long long f2_pack(float lo, float hi) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(unsigned long long v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b,
                                                     unsigned long long c) {
    unsigned long long r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b) {
    unsigned long long r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// A candidate as a unique 64-bit key: order-preserving logit key above, the
// complement of the expert index below, so that a larger key is a better route
// (larger logit, then lower index).
__device__ __forceinline__ unsigned long long cand_pack(float x, int e) {
    return ((unsigned long long)__float_as_uint(x) << 32) | (unsigned)e;
}
__device__ __forceinline__ unsigned long long cand_key(unsigned long long pair) {
    const unsigned k = f2key(__uint_as_float((unsigned)(pair >> 32)));
    return ((unsigned long long)k << 32) | (0xffffffffu - (unsigned)pair);
}
__device__ __forceinline__ float key_logit(unsigned long long key) { return key2f((unsigned)(key >> 32)); }
__device__ __forceinline__ int key_expert(unsigned long long key) { return (int)(0xffffffffu - (unsigned)key); }

// Turns the warp's n (logit, expert) pairs into rank keys and ranks them, two per
// lane per sweep over the list; returns this lane's share of sum exp(logit - m)
// over the candidates ranked below `limit` (mb = m log2(e)).
__device__ __forceinline__ float rank_candidates(unsigned long long* cand, int* rk, int n, int limit, float mb) {
    for (int c = (int)lane_id(); c < n; c += 32) cand[c] = cand_key(cand[c]);
    __syncwarp();
    float d = 0.0f;
    for (int c0 = (int)lane_id(); c0 < n; c0 += 64) {
        const int c1 = c0 + 32;
        const unsigned long long ka = cand[c0];
        const unsigned long long kb = c1 < n ? cand[c1] : ~0ull;
        int ra = 0, rb = 0;
#pragma unroll 4
        for (int q = 0; q < n; q++) {
            const unsigned long long o = cand[q];
            ra += o > ka;
            rb += o > kb;
        }
        rk[c0] = ra;
        if (ra < limit) d += ex2_approx(fmaf(key_logit(ka), LOG2E, -mb));
        if (c1 < n) {
            rk[c1] = rb;
            if (rb < limit) d += ex2_approx(fmaf(key_logit(kb), LOG2E, -mb));
        }
    }
    return d;
}

__device__ __forceinline__ void write_ranked(const unsigned long long* cand, const int* rk, int n, int limit,
                                             long long t, int K, void* ids, bool i16, float* probs, float mb,
                                             float inv_den) {
    for (int c = (int)lane_id(); c < n; c += 32) {
        const int r = rk[c];
        if (r < limit) {
            const long long o = t * K + r;
            store_route(ids, i16, o, key_expert(cand[c]));
            probs[o] = ex2_approx(fmaf(key_logit(cand[c]), LOG2E, -mb)) * inv_den;
        }
    }
}

// G: group maxima per lane for the threshold (32 G >= K); element (j, c) of a lane
// belongs to group (4 j + c) mod G.
// FULL: E == 128 NV4, so every lane holds all NV4 float4 slots of a row (no absent slots).
template <int NV4, int G, bool FULL>
__global__ void __launch_bounds__(FW * 32, 2) route_filter_kernel(const float* __restrict__ logits, int T, int E,
                                                                  int K, void* ids, bool i16,
                                                                  float* __restrict__ probs, bool renorm) {
    pdl_trigger();   // the permute that follows may launch now (it waits for the routes)
    extern __shared__ __align__(16) uint8_t fsm[];
    const int lane = (int)lane_id(), w = (int)(threadIdx.x >> 5);
    float* rowbuf = reinterpret_cast<float*>(fsm) + (size_t)w * 128 * NV4;
    FilterWarp& fw = reinterpret_cast<FilterWarp*>(fsm + (size_t)FW * 512 * NV4)[w];
    unsigned long long* cand = fw.cand;
    int* rk = fw.rank;
    const int E4 = E >> 2;
    const uint32_t row_bytes = 4u * (uint32_t)E;
    const int nq = E4 > lane ? (E4 - lane + 31) / 32 : 0;   // float4s of the row this lane holds
    const long long nwarps = (long long)gridDim.x * FW;
    long long t = (long long)blockIdx.x * FW + w;
    if (lane == 0) {
        ptx::mbar_init(&fw.bar, 1);
        fw.abort_flag = 0u;
        ptx::fence_mbar_init();
        if (t < T) {
            ptx::mbar_arrive_expect_tx(&fw.bar, row_bytes);
            ptx::bulk_load(rowbuf, logits + t * E, row_bytes, &fw.bar);
        }
    }
    __syncwarp();
    uint32_t phase = 0;
    for (; t < T; t += nwarps) {
        if (!ptx::wait_parity(&fw.bar, phase, &fw.abort_flag)) break;
        phase ^= 1u;
        // absent slots (past E) hold -inf: no group maximum, exp or threshold test is changed by them
        float x[NV4][4];
        const float4* rb = reinterpret_cast<const float4*>(rowbuf);
#pragma unroll
        for (int j = 0; j < NV4; j++) {
            const float4 f =
                FULL || j < nq ? rb[j * 32 + lane] : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
            x[j][0] = f.x;
            x[j][1] = f.y;
            x[j][2] = f.z;
            x[j][3] = f.w;
        }
        float gm[G];
#pragma unroll
        for (int g = 0; g < G; g++) gm[g] = -INFINITY;
        constexpr int GS = G / 4;                 // slot j + GS is in the same group as slot j
#pragma unroll
        for (int j0 = 0; j0 < NV4; j0 += 2 * GS)
#pragma unroll
            for (int j = j0; j < j0 + GS && j < NV4; j++)
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    const int g = (4 * j + c) % G;
                    gm[g] = j + GS < NV4 ? max3f(gm[g], x[j][c], x[j + GS][c]) : fmaxf(gm[g], x[j][c]);
                }
        float m = gm[0];
#pragma unroll
        for (int g = 1; g < G; g++) m = fmaxf(m, gm[g]);
        m = warp_max(m);
        const float mb = m * LOG2E;
        float den = 0.0f;
        if (!renorm) {
            // sum of 2^(x log2 e - m log2 e), the exponent arguments and sums formed in pairs
            const unsigned long long l2 = f2_pack(LOG2E, LOG2E), nm = f2_pack(-mb, -mb);
            unsigned long long d01 = 0ull, d23 = 0ull;
#pragma unroll
            for (int j = 0; j < NV4; j++) {
                float y0, y1, y2, y3;
                f2_unpack(f2_fma(f2_pack(x[j][0], x[j][1]), l2, nm), y0, y1);
                f2_unpack(f2_fma(f2_pack(x[j][2], x[j][3]), l2, nm), y2, y3);
                d01 = f2_add(d01, f2_pack(ex2_approx(y0), ex2_approx(y1)));
                d23 = f2_add(d23, f2_pack(ex2_approx(y2), ex2_approx(y3)));
            }
            float a0, a1, a2, a3;
            f2_unpack(d01, a0, a1);
            f2_unpack(d23, a2, a3);
            den = warp_sum((a0 + a1) + (a2 + a3));
        }
        // threshold: the largest 16-bit key prefix that at least K of the 32 G group maxima reach
        // (the K-th largest of a subset of the row is at most the row's K-th largest)
        unsigned ck[G];
#pragma unroll
        for (int g = 0; g < G; g++) ck[g] = f2key(gm[g]);
        // key bits shared by every group maximum are bits of the answer: start below them
        unsigned kmin = ck[0], kmax = ck[0];
#pragma unroll
        for (int g = 1; g < G; g++) {
            kmin = min(kmin, ck[g]);
            kmax = max(kmax, ck[g]);
        }
        kmin = __reduce_min_sync(FULL, kmin);
        kmax = __reduce_max_sync(FULL, kmax);
        const unsigned diff16 = (kmin ^ kmax) >> 16;
        unsigned pre = kmin >> 16;
        int b0 = -2;                              // lower bit of the first two-bit step
        if (diff16) {
            b0 = (31 - __clz(diff16)) & ~1;
            pre &= ~((2u << b0) - 1u);            // bits b0 .. 0 are searched (b0 + 1 is kept or found again)
        }
#pragma unroll 1
        for (int b = b0; b >= 0; b -= 2) {       // two bits a step: three independent counts
            const unsigned t1 = (pre | (1u << b)) << 16, t2 = (pre | (2u << b)) << 16,
                           t3 = (pre | (3u << b)) << 16;
            unsigned c1 = 0, c2 = 0, c3 = 0;
#pragma unroll
            for (int g = 0; g < G; g++) {
                c1 += ck[g] >= t1;
                c2 += ck[g] >= t2;
                c3 += ck[g] >= t3;
            }
            c1 = __reduce_add_sync(FULL, c1);
            c2 = __reduce_add_sync(FULL, c2);
            c3 = __reduce_add_sync(FULL, c3);
            const unsigned uk = (unsigned)K;
            pre |= (c3 >= uk ? 3u : c2 >= uk ? 2u : c1 >= uk ? 1u : 0u) << b;
        }
        // at or below the key of -inf the test would admit -inf (and absent) slots: exact path
        const bool low = pre < 0x80u;
        const float tau = low ? INFINITY : key2f(pre << 16);
        // this lane's logits >= tau as a bit mask over its slots (bit 4 j + c), and their count
        constexpr int NW = (4 * NV4 + 31) / 32;
        unsigned mk[NW];
#pragma unroll
        for (int i = 0; i < NW; i++) mk[i] = 0u;
#pragma unroll
        for (int j = 0; j < NV4; j++)
#pragma unroll
            for (int c = 0; c < 4; c++)
                if (x[j][c] >= tau) mk[(4 * j + c) >> 5] |= 1u << ((4 * j + c) & 31);
        int cnt = 0;
#pragma unroll
        for (int i = 0; i < NW; i++) cnt += __popc(mk[i]);
        int incl = cnt;
#pragma unroll
        for (int dd = 1; dd < 32; dd <<= 1) {
            const int o = __shfl_up_sync(FULL, incl, dd);
            if (lane >= dd) incl += o;
        }
        const int n = __shfl_sync(FULL, incl, 31);
        const bool direct = !low && n <= FCAND;
        int a = 0;                                        // exact path: logits above the K-th
        if (direct) {
            // the candidates, read back from the row buffer at the set bits
            int pos = incl - cnt;
#pragma unroll
            for (int i = 0; i < NW; i++) {
                unsigned bits = mk[i];
                while (bits) {
                    const int bslot = 32 * i + __ffs(bits) - 1;
                    bits &= bits - 1u;
                    const int e = 128 * (bslot >> 2) + 4 * lane + (bslot & 3);
                    cand[pos++] = cand_pack(rowbuf[e], e);
                }
            }
        } else {
            // exact path over the row buffer: the K-th largest key by a search over all 32 key bits
            unsigned kk = 0;
#pragma unroll 1
            for (int b = 31; b >= 0; b--) {
                const unsigned trial = kk | (1u << b);
                unsigned c = 0;
                if (trial <= 0x007fffffu) {
                    c = (unsigned)K;                      // at or below the key of -inf: every logit
                } else {
                    const float f = key2f(trial);         // above the key of +inf: NaN, no logit
#pragma unroll 4
                    for (int e = lane; e < E; e += 32) c += rowbuf[e] >= f;
                    c = __reduce_add_sync(FULL, c);
                }
                if (c >= (unsigned)K) kk = trial;
            }
            const float fk = key2f(kk);                   // the K-th largest logit
            const float ek = ex2_approx(fmaf(fk, LOG2E, -mb));
            if (lane == 0) fw.n = 0;
            __syncwarp();
            float d = 0.0f;
            for (int e = lane; e < E; e += 32) {
                const float v = rowbuf[e];
                if (v > fk) {                             // fewer than K such logits
                    cand[atomicAdd(&fw.n, 1)] = cand_pack(v, e);
                    d += ex2_approx(fmaf(v, LOG2E, -mb));
                }
            }
            __syncwarp();
            a = fw.n;
            const int rem = K - a;                        // logits equal to fk that are taken, in expert order
            if (renorm) den = warp_sum(d) + (float)rem * ek;
            const float pk = ek / den;
            int taken = 0;
            for (int e0 = 0; e0 < E && taken < rem; e0 += 32) {
                const int e = e0 + lane;
                const bool eq = e < E && rowbuf[e] == fk;
                const unsigned bal = __ballot_sync(FULL, eq);
                const int ord = taken + __popc(bal & lanemask_lt());
                if (eq && ord < rem) {
                    const long long o = t * K + a + ord;
                    store_route(ids, i16, o, e);
                    probs[o] = pk;
                }
                taken += __popc(bal);
            }
        }
        // the row buffer is free: start the copy of this warp's next row
        __syncwarp();
        if (lane == 0 && t + nwarps < T) {
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive_expect_tx(&fw.bar, row_bytes);
            ptx::bulk_load(rowbuf, logits + (t + nwarps) * E, row_bytes, &fw.bar);
        }
        if (direct) {
            const float d = rank_candidates(cand, rk, n, K, mb);
            if (renorm) den = warp_sum(d);
            __syncwarp();
            write_ranked(cand, rk, n, K, t, K, ids, i16, probs, mb, 1.0f / den);
        } else {
            rank_candidates(cand, rk, a, K, mb);
            __syncwarp();
            write_ranked(cand, rk, a, K, t, K, ids, i16, probs, mb, 1.0f / den);
        }
        __syncwarp();   // the warp's shared lists are reused by its next row
    }
}

template <int NV4, int G, bool FULL>
cudaError_t launch_filter(const float* logits, int T, int E, int K, void* ids, bool i16, float* probs,
                          bool renorm, cudaStream_t s) {
    constexpr size_t smem = filter_smem_bytes<NV4>();
    static int resident = 0;                      // one wave of CTAs: SMs x resident CTAs per SM
    if (!resident) {
        int dev = 0, sms = 0, per = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        cudaError_t e = cudaFuncSetAttribute(route_filter_kernel<NV4, G, FULL>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, route_filter_kernel<NV4, G, FULL>, FW * 32, smem);
        resident = sms * (per > 0 ? per : 1);
    }
    const long long need = ((long long)T + FW - 1) / FW;
    const int blocks = (int)(need < resident ? need : resident);
    route_filter_kernel<NV4, G, FULL><<<blocks, FW * 32, smem, s>>>(logits, T, E, K, ids, i16, probs, renorm);
    return cudaGetLastError();
}

template <int NV4>
cudaError_t launch_filter_k(const float* logits, int T, int E, int K, void* ids, bool i16, float* probs,
                            bool renorm, cudaStream_t s) {
    const bool full = E == 128 * NV4;
    if (K <= 128 && K > 64)
        return full ? launch_filter<NV4, 8, true>(logits, T, E, K, ids, i16, probs, renorm, s)
                    : launch_filter<NV4, 8, false>(logits, T, E, K, ids, i16, probs, renorm, s);
    return full ? launch_filter<NV4, 4, true>(logits, T, E, K, ids, i16, probs, renorm, s)
                : launch_filter<NV4, 4, false>(logits, T, E, K, ids, i16, probs, renorm, s);
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
    } else if (E % 4 == 0 && E <= 2304 && K <= KMAX && moe_host::aligned(logits, 16)) {
        if (E <= 256) err = launch_filter_k<2>(logits, T, E, K, ids, i16, probs, renorm, s);
        else if (E <= 512) err = launch_filter_k<4>(logits, T, E, K, ids, i16, probs, renorm, s);
        else if (E <= 1024) err = launch_filter_k<8>(logits, T, E, K, ids, i16, probs, renorm, s);
        else err = launch_filter_k<18>(logits, T, E, K, ids, i16, probs, renorm, s);
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

// ---------------------------------------------------------------------------
// Router backward ("Sparser MoE end-to-end", sections "The workload changes the
// bottleneck" and "Preserve a compact route": a router backward kernel beside
// the forward; the pages do not define it). The gradient of the forward's
// probabilities with respect to the logits, the selection held fixed: for row
// t with selected set S (valid ids), g[k] = dprobs[t,k], G_e = sum of g[k] over
// the k with ids[t,k] = e, p the softmax over all E (or, renormalised, over S,
// 0 off S) and s = sum over valid k of g[k] p_{ids[t,k]}:
//   dlogits[t,e] = p_e (G_e - s)   (0 off S when renormalised).
// One warp per row: the row maximum and the denominator, s from the selected
// slots, then every dlogit is written as -p_e s and the selected ones are
// overwritten (by the lane of each id's first occurrence) with p_e (G_e - s).
// ---------------------------------------------------------------------------
namespace moe {
namespace {

template <int KC>
__global__ void __launch_bounds__(256) route_backward_kernel(const float* __restrict__ logits,
                                                             const void* __restrict__ ids, bool i16,
                                                             const float* __restrict__ dprobs, int T, int E,
                                                             int K, bool renorm, float* __restrict__ dlogits) {
    const int lane = (int)lane_id();
    const int nwarps_total = (gridDim.x * blockDim.x) >> 5;
    for (long long t = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += nwarps_total) {
        const float* l = logits + t * E;
        float* out = dlogits + t * E;
        // the route slots of this row: id (or -1), gradient, and whether it is the id's first occurrence
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
        // G_e accumulated on the first occurrence; later duplicates contribute and step aside
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
                        else g[c] += g2;      // a later slot of the same expert: its gradient joins
                    }
                }
            }
        // row maximum over all E (as in the forward)
        float m = -INFINITY;
        for (int e = lane; e < E; e += 32) m = fmaxf(m, __ldg(l + e));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, o));
        // denominator: all E, or the selected set (each expert once)
        float den = 0.0f;
        if (!renorm) {
            for (int e = lane; e < E; e += 32) den += __expf(__ldg(l + e) - m);
        } else {
#pragma unroll
            for (int c = 0; c < KC; c++)
                if (first[c]) den += __expf(__ldg(l + id[c]) - m);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(FULL, den, o);
        const float inv = 1.0f / den;
        // s = sum over the selected experts of G_e p_e (first occurrences carry G_e)
        float sp = 0.0f;
        float pe[KC];
#pragma unroll
        for (int c = 0; c < KC; c++) {
            pe[c] = first[c] ? __expf(__ldg(l + id[c]) - m) * inv : 0.0f;
            sp += first[c] ? g[c] * pe[c] : 0.0f;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sp += __shfl_xor_sync(FULL, sp, o);
        // every dlogit: -p_e s (0 off the selection when renormalised) ...
        for (int e = lane; e < E; e += 32) out[e] = renorm ? 0.0f : -(__expf(__ldg(l + e) - m) * inv) * sp;
        __syncwarp();
        // ... the selected ones: p_e (G_e - s)
#pragma unroll
        for (int c = 0; c < KC; c++)
            if (first[c]) out[id[c]] = pe[c] * (g[c] - sp);
        __syncwarp();
    }
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_route_topk_backward(const float* logits, const void* ids, moe_dtype id_dtype,
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
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    long long blocks = ((long long)T + 7) / 8;
    const long long cap = (long long)sms * 16;
    if (blocks > cap) blocks = cap;
    cudaStream_t s = moe_host::as_stream(stream);
    const bool i16 = id_dtype == MOE_I16;
    const bool renorm = (flags & MOE_ROUTE_RENORM) != 0;
    const int KC = (K + 31) / 32;
#define MOE_ROUTE_BWD(kc) \
    route_backward_kernel<kc><<<(int)blocks, 256, 0, s>>>(logits, ids, i16, dprobs, T, E, K, renorm, dlogits)
    if (KC == 1) MOE_ROUTE_BWD(1);
    else if (KC == 2) MOE_ROUTE_BWD(2);
    else MOE_ROUTE_BWD(4);
#undef MOE_ROUTE_BWD
    return moe_host::launch_status();
}
