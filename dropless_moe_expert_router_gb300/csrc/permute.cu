// permute.cu -- dropless dispatch into expert-contiguous order, the standalone
// group-aware MXFP8 quantiser, and their entry points.
//
// The permutation is a deterministic device-side counting sort of the T*K
// routes by expert ("Dropless MoE acceleration in JAX with NVIDIA Transformer
// Engine", sections "Dropless vs capacity-based MoE" and "Optimization 1":
// every route is kept, group sizes never leave the device; "Sparser MoE
// end-to-end", section "Remove work that has no selected route": local
// processing visits only the selected slots of a token, found by a warp ballot):
//
//   1. rank    small E (TT = 128 tokens): a warp per tile walks the tile's routes in
//              flattened order, 32 at a time (16 such rows of ids loaded ahead, one
//              memory latency per 512 routes); __match_any groups the lanes of one
//              expert, so each valid route gets its rank among the tile's earlier
//              routes of the same expert. Large E (TT = 64 tokens): a CTA per tile
//              sets each route's token bit in its expert's 64-bit token mask and
//              counts the expert's routes (shared-memory atomics, order-free); a
//              route's rank is the population of its expert's mask below its token
//              (a tile where a token lists an expert twice is ranked in flattened
//              order by one warp instead). Both write per-(expert, tile) counts to
//              the workspace table [E][tiles] and the tile-local rank into row_map.
//   2. scan    (warp per expert, then the last block to finish): exclusive scan
//              of each expert's counts over tiles -> per-tile bases, group_sizes;
//              the last block scans group_sizes -> group_offsets. When the table
//              is small (E * tiles <= 2048) this step is not a kernel of its own:
//              every scatter block scans the table in shared memory first.
//   3. scatter (warp per token): row = group_offsets[e] + base[e][tile] + rank;
//              a ballot over the token's valid slots gives the destinations,
//              the token row is read once and stored to each of them with 16-byte
//              vectors (optionally quantised to MXFP8 on the way).
// Rows within an expert end up in ascending t*K + k order, independent of
// scheduling.
#include "common.cuh"

namespace moe {
namespace {

constexpr int SCAN_THREADS = 1024;

inline int tile_tokens(int E) { return E > 64 ? 64 : 128; }

struct PermuteWs {
    int* table;        // [E][tiles]
    unsigned* ticket;  // completion counter of the scan kernel
};

inline size_t align16(size_t n) { return (n + 15) & ~(size_t)15; }

inline PermuteWs carve(void* ws, int E, int tiles) {
    PermuteWs w;
    w.table = (int*)ws;
    w.ticket = (unsigned*)((char*)ws + align16((size_t)E * (size_t)tiles * sizeof(int)));
    return w;
}

// ---------------------------------------------------------------- 1. rank
__global__ void perm_rank_kernel(const void* __restrict__ ids, bool i16, int T, int K, int E, int TT,
                                 int tiles, int* __restrict__ table, int* __restrict__ row_map,
                                 unsigned* __restrict__ ticket) {
    extern __shared__ int s_cnt[];  // [warps][E]
    const int warp = threadIdx.x >> 5, lane = (int)lane_id();
    const int nwarps = blockDim.x >> 5;
    int* cnt = s_cnt + (size_t)warp * E;
    pdl_wait();        // the ids (and everything before this kernel) are complete
    pdl_trigger();     // the scan / scatter may launch now; they wait for this kernel's writes
    if (blockIdx.x == 0 && threadIdx.x == 0) *ticket = 0u;
    const int tile = blockIdx.x * nwarps + warp;
    if (tile >= tiles) return;
    for (int e = lane; e < E; e += 32) cnt[e] = 0;
    __syncwarp();
    const long long i0 = (long long)tile * TT * K;
    long long i1 = (long long)(tile + 1) * TT * K;
    const long long nroutes = (long long)T * K;
    if (i1 > nroutes) i1 = nroutes;
    // U rows of 32 routes are loaded before any is ranked: one memory latency per 32 U routes
    constexpr int U = 16;
    for (long long c0 = i0; c0 < i1; c0 += 32 * U) {
        int ev[U];
#pragma unroll
        for (int u = 0; u < U; u++) {
            const long long i = c0 + u * 32 + lane;
            ev[u] = i < i1 ? load_id(ids, i, i16) : -1;
        }
#pragma unroll
        for (int u = 0; u < U; u++) {
            if (c0 + u * 32 >= i1) break;   // warp-uniform
            const long long i = c0 + u * 32 + lane;
            int e = ev[u];
            if (i < i1 && (e < -1 || e >= E)) {
                raise_device_error(MOE_DEVERR_BAD_ID);
                e = -1;
            }
            const unsigned grp = __match_any_sync(FULL, e);
            const int leader = __ffs(grp) - 1;
            const int rk = __popc(grp & lanemask_lt());
            int old = 0;
            if (lane == leader && e >= 0) {
                old = cnt[e];
                cnt[e] = old + __popc(grp);
            }
            old = __shfl_sync(FULL, old, leader);
            if (i < i1) row_map[i] = (e >= 0) ? old + rk : -1;
            __syncwarp();
        }
    }
    for (int e = lane; e < E; e += 32) table[(size_t)e * tiles + tile] = cnt[e];
}

// Large E (TT = 64 tokens): one CTA per tile. Every valid route sets its token's bit in its
// expert's 64-bit token mask and adds one to its expert's count, by shared-memory atomics whose
// order does not matter. When no token of the tile lists an expert twice (every count equals its
// mask's population), a route's rank among the tile's earlier routes of its expert is the number
// of the expert's tokens before its own: the rank the flattened order gives. A tile where a token
// lists an expert twice is ranked again by one warp walking its routes in flattened order, as
// the small-E kernel does.
constexpr int RANK_MASK_THREADS = 1024;

inline size_t rank_mask_smem(int E) { return ((size_t)E * 12 + 15) & ~(size_t)15; }   // masks, counts

template <int MAXR>   // routes per thread: TT * K / RANK_MASK_THREADS rounded up
__global__ void __launch_bounds__(RANK_MASK_THREADS) perm_rank_mask_kernel(const void* __restrict__ ids, bool i16,
                                                                          int T, int K, int E, int TT, int tiles,
                                                                          int* __restrict__ table,
                                                                          int* __restrict__ row_map,
                                                                          unsigned* __restrict__ ticket) {
    extern __shared__ __align__(16) uint8_t s_rm[];
    unsigned long long* mask = reinterpret_cast<unsigned long long*>(s_rm);   // [E]
    unsigned* cnt = reinterpret_cast<unsigned*>(s_rm + (size_t)E * 8);        // [E]
    pdl_wait();        // the ids (and everything before this kernel) are complete
    pdl_trigger();     // the scan / scatter may launch now; they wait for this kernel's writes
    if (blockIdx.x == 0 && threadIdx.x == 0) *ticket = 0u;
    const int tile = blockIdx.x;
    const long long i0 = (long long)tile * TT * K;
    long long i1 = i0 + (long long)TT * K;
    const long long nroutes = (long long)T * K;
    if (i1 > nroutes) i1 = nroutes;
    const int n = (int)(i1 - i0);
    int ev[MAXR];
#pragma unroll
    for (int r = 0; r < MAXR; r++) {
        const int j = r * RANK_MASK_THREADS + (int)threadIdx.x;
        int e = j < n ? load_id(ids, i0 + j, i16) : -1;
        if (j < n && (e < -1 || e >= E)) {
            raise_device_error(MOE_DEVERR_BAD_ID);
            e = -1;
        }
        ev[r] = e;
    }
    const int n16 = (int)(((size_t)E * 12 + 15) / 16);
    for (int i = threadIdx.x; i < n16; i += blockDim.x) reinterpret_cast<uint4*>(s_rm)[i] = make_uint4(0, 0, 0, 0);
    // token of route j within the tile, j / K: the high word of j * ceil(2^32 / K) (exact for
    // j < 2^32 / K; K = 1 is j itself)
    const unsigned kinv = K > 1 ? 0xffffffffu / (unsigned)K + 1u : 0u;
    auto token_of = [&](unsigned j) { return K > 1 ? __umulhi(j, kinv) : j; };
    __syncthreads();   // the masks and counts are zero
#pragma unroll
    for (int r = 0; r < MAXR; r++) {
        if (ev[r] >= 0) {
            const unsigned j = (unsigned)(r * RANK_MASK_THREADS) + threadIdx.x;
            atomicOr(&mask[ev[r]], 1ull << token_of(j));
            atomicAdd(&cnt[ev[r]], 1u);
        }
    }
    __syncthreads();
    // the tile's counts to the table; a token listing an expert twice leaves a count above the
    // population of that expert's mask
    int dup = 0;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const unsigned c = cnt[e];
        dup |= c != (unsigned)__popcll(mask[e]);
        table[(size_t)e * tiles + tile] = (int)c;
    }
    if (!__syncthreads_or(dup)) {
#pragma unroll
        for (int r = 0; r < MAXR; r++) {
            const unsigned j = (unsigned)(r * RANK_MASK_THREADS) + threadIdx.x;
            if ((int)j < n)
                row_map[i0 + j] = ev[r] >= 0 ? __popcll(mask[ev[r]] & ((1ull << token_of(j)) - 1ull)) : -1;
        }
        return;
    }
    // a token lists an expert twice: warp 0 ranks the tile's routes in flattened order
    if (threadIdx.x >= 32) return;
    const int lane = (int)threadIdx.x;
    for (int e = lane; e < E; e += 32) cnt[e] = 0u;
    __syncwarp();
    for (int c0 = 0; c0 < n; c0 += 32) {
        const int j = c0 + lane;
        int e = j < n ? load_id(ids, i0 + j, i16) : -1;
        if (e < -1 || e >= E) e = -1;                  // (flagged above)
        const unsigned grp = __match_any_sync(FULL, e);
        const int leader = __ffs(grp) - 1;
        unsigned old = 0u;
        if (lane == leader && e >= 0) {
            old = cnt[e];
            cnt[e] = old + (unsigned)__popc(grp);
        }
        old = __shfl_sync(FULL, old, leader);
        if (j < n) row_map[i0 + j] = e >= 0 ? (int)old + __popc(grp & lanemask_lt()) : -1;
        __syncwarp();
    }
}

// ---------------------------------------------------------------- 2. scan
__global__ void __launch_bounds__(SCAN_THREADS) perm_scan_kernel(int E, int tiles, int* __restrict__ table,
                                                                 int* __restrict__ group_sizes,
                                                                 int* __restrict__ group_offsets,
                                                                 unsigned* __restrict__ ticket) {
    __shared__ int s_warp[SCAN_THREADS / 32];
    __shared__ bool s_last;
    const int warp = threadIdx.x >> 5, lane = (int)lane_id();
    const int nwarps = SCAN_THREADS / 32;
    pdl_wait();        // the rank kernel's table is complete
    pdl_trigger();
    // (a) warp per expert: exclusive scan of its per-tile counts, in place; SCAN_CHUNKS rows of
    // 32 counts are loaded before any is scanned (one memory round trip per 32 SCAN_CHUNKS)
    constexpr int SCAN_CHUNKS = 8;
    for (int e = blockIdx.x * nwarps + warp; e < E; e += gridDim.x * nwarps) {
        int* row = table + (size_t)e * tiles;
        int carry = 0;
        for (int j0 = 0; j0 < tiles; j0 += 32 * SCAN_CHUNKS) {
            int v[SCAN_CHUNKS];
#pragma unroll
            for (int c = 0; c < SCAN_CHUNKS; c++) {
                const int j = j0 + 32 * c + lane;
                v[c] = j < tiles ? __ldcg(row + j) : 0;
            }
#pragma unroll
            for (int c = 0; c < SCAN_CHUNKS; c++) {
                const int j = j0 + 32 * c + lane;
                int inc = v[c];
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const int o = __shfl_up_sync(FULL, inc, d);
                    if (lane >= d) inc += o;
                }
                if (j < tiles) row[j] = carry + inc - v[c];
                carry += __shfl_sync(FULL, inc, 31);
            }
        }
        if (lane == 0) group_sizes[e] = carry;
    }
    // (b) the last block to finish scans group_sizes -> group_offsets
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = (atomicAdd(ticket, 1u) == gridDim.x - 1);
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const int per = (E + SCAN_THREADS - 1) / SCAN_THREADS;
    const int b0 = threadIdx.x * per;
    int local = 0;
    for (int j = 0; j < per; j++)
        if (b0 + j < E) local += __ldcg(group_sizes + b0 + j);
    int inc = local;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        int o = __shfl_up_sync(FULL, inc, d);
        if (lane >= d) inc += o;
    }
    if (lane == 31) s_warp[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        int w = s_warp[lane];
        int wi = w;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            int o = __shfl_up_sync(FULL, wi, d);
            if (lane >= d) wi += o;
        }
        s_warp[lane] = wi - w;  // exclusive prefix of warp totals
    }
    __syncthreads();
    int run = s_warp[warp] + inc - local;
    for (int j = 0; j < per; j++) {
        if (b0 + j < E) {
            group_offsets[b0 + j] = run;
            run += __ldcg(group_sizes + b0 + j);
        }
    }
    if (threadIdx.x == SCAN_THREADS - 1) group_offsets[E] = s_warp[warp] + inc;
}

// ---------------------------------------------------------------- 3. scatter
// Up to KC*32 routes per token (K <= 128). SCAN: the count table is small (E * tiles <=
// SCAN_IN_BLOCK_MAX): every block scans it in shared memory itself (the work of step 2),
// and block 0 publishes group_sizes and group_offsets.
constexpr int SCAN_IN_BLOCK_MAX = 2048;   // larger tables: the scatter is long and wants the full grid

// The table and the offsets fit the default 48 KB of dynamic shared memory.
inline bool scan_in_block(int E, long long tiles) {
    return (long long)E * tiles <= SCAN_IN_BLOCK_MAX && ((long long)E * tiles + E + 1) * 4 <= 48 * 1024;
}

// FUSE: 0 bf16 rows; 1 MXFP8 rows (E4M3 + one E8M0 byte per 32, quads of lanes); 2 NVFP4 rows
// (packed E2M1 + one E4M3 byte per 16, pairs of lanes) with the encode scale of the device *amax.
// (MXFP8 with the scan in every block: held to 64 registers, four blocks per SM in its one wave)
template <int KC, int FUSE, bool SCAN>
__global__ void __launch_bounds__(256, FUSE == 1 && SCAN ? 4 : 1)
    perm_scatter_kernel(const uint4* __restrict__ x, int T, int H,
                                                           const void* __restrict__ ids, bool i16, int K, int E,
                                                           int TT, int tiles, const int* __restrict__ table,
                                                           int* __restrict__ group_sizes,
                                                           int* __restrict__ group_offsets,
                                                           int* __restrict__ row_map, int* __restrict__ perm_src,
                                                           void* __restrict__ x_perm,
                                                           uint8_t* __restrict__ scales,
                                                           const float* __restrict__ amax) {
    extern __shared__ int s_dyn[];  // SCAN: table [E][tiles], then offsets [E + 1]
    const int lane = (int)lane_id();
    const int nwarps_total = (gridDim.x * blockDim.x) >> 5;
    int* s_tab = s_dyn;
    int* s_off = s_dyn + (SCAN ? E * tiles : 0);
    pdl_wait();        // launched early: the rank (and scan) kernels' writes are complete from here
    if constexpr (SCAN) {
        const int warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
        for (int i = threadIdx.x; i < E * tiles; i += blockDim.x) s_tab[i] = __ldcg(table + i);
        __syncthreads();
        // warp per expert: exclusive scan of its per-tile counts (in place), its total
        for (int e = warp; e < E; e += nwarps) {
            int* row = s_tab + (size_t)e * tiles;
            int carry = 0;
            for (int j0 = 0; j0 < tiles; j0 += 32) {
                const int j = j0 + lane;
                const int v = j < tiles ? row[j] : 0;
                int inc = v;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const int o = __shfl_up_sync(FULL, inc, d);
                    if (lane >= d) inc += o;
                }
                if (j < tiles) row[j] = carry + inc - v;
                carry += __shfl_sync(FULL, inc, 31);
            }
            if (lane == 0) s_off[e] = carry;
        }
        __syncthreads();
        // exclusive scan of the totals (warp 0, a contiguous run of experts per lane)
        if (warp == 0) {
            const int per = (E + 31) / 32, b0 = lane * per;
            int local = 0;
            for (int j = 0; j < per; j++)
                if (b0 + j < E) local += s_off[b0 + j];
            int inc = local;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int o = __shfl_up_sync(FULL, inc, d);
                if (lane >= d) inc += o;
            }
            int run = inc - local;
            for (int j = 0; j < per; j++)
                if (b0 + j < E) {
                    const int v = s_off[b0 + j];
                    s_off[b0 + j] = run;
                    run += v;
                }
            if (lane == 31) s_off[E] = inc;
        }
        __syncthreads();
        if (blockIdx.x == 0) {
            for (int e = threadIdx.x; e <= E; e += blockDim.x) {
                group_offsets[e] = s_off[e];
                if (e < E) group_sizes[e] = s_off[e + 1] - s_off[e];
            }
        }
    }
    const int H8 = H >> 3;     // 16-byte chunks per row
    const int iters = (H8 + 31) >> 5;
    float S = 1.0f;
    __shared__ float s_rs[FUSE == 2 ? 256 : 1];   // NVFP4: the elements' multiplier per scale byte
    if constexpr (FUSE == 2) {
        S = nvfp4_encode_scale(__ldg(amax));
        for (int i = threadIdx.x; i < 256; i += blockDim.x) s_rs[i] = nvfp4_rs_entry(S, (uint32_t)i);
        __syncthreads();
    }
    for (long long t = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += nwarps_total) {
        const int tile = (int)(t / TT);
        int rows[KC];
        unsigned mask[KC];
#pragma unroll
        for (int c = 0; c < KC; c++) {
            int k = c * 32 + lane;
            int r = -1;
            if (k < K) {
                long long i = t * K + k;
                int lr = row_map[i];
                if (lr >= 0) {
                    int e = load_id(ids, i, i16);
                    r = SCAN ? s_off[e] + s_tab[(size_t)e * tiles + tile] + lr
                             : group_offsets[e] + table[(size_t)e * tiles + tile] + lr;
                    perm_src[r] = (int)t;
                }
                row_map[i] = r;
            }
            rows[c] = r;
            mask[c] = __ballot_sync(FULL, r >= 0);
        }
        const uint4* src = x + t * H8;
        // U 16-byte chunks per lane in flight before the stores (memory-level parallelism)
        constexpr int U = FUSE == 2 ? 2 : 4;   // (NVFP4: two, for four blocks per SM within 64 registers)
        for (int it0 = 0; it0 < iters; it0 += U) {
            uint4 v[U];
            bool in[U];
#pragma unroll
            for (int u = 0; u < U; u++) {
                const int j = (it0 + u) * 32 + lane;
                in[u] = (it0 + u < iters) && j < H8;
                v[u] = in[u] ? __ldg(src + j) : make_uint4(0, 0, 0, 0);
            }
            if constexpr (FUSE == 0) {
#pragma unroll
                for (int c = 0; c < KC; c++) {
                    unsigned m = mask[c];
                    while (m) {
                        const int b = __ffs(m) - 1;
                        m &= m - 1;
                        const int r = __shfl_sync(FULL, rows[c], b);
                        uint4* dst = reinterpret_cast<uint4*>(x_perm) + (long long)r * H8 + lane;
#pragma unroll
                        for (int u = 0; u < U; u++)
                            if (in[u]) dst[(it0 + u) * 32] = v[u];
                    }
                }
            } else if constexpr (FUSE == 2) {
                uint32_t qv[U], sb[U];
#pragma unroll
                for (int u = 0; u < U; u++) {
                    if (it0 + u < iters) {  // warp-uniform: the pair shuffles see every lane
                        float f[8];
                        bf16x8_to_f32(v[u], f);
                        qv[u] = nvfp4_pair(f, S, s_rs, &sb[u]);
                    }
                }
#pragma unroll
                for (int c = 0; c < KC; c++) {
                    unsigned m = mask[c];
                    while (m) {
                        const int b = __ffs(m) - 1;
                        m &= m - 1;
                        const int r = __shfl_sync(FULL, rows[c], b);
#pragma unroll
                        for (int u = 0; u < U; u++) {
                            if (in[u]) {
                                const int j = (it0 + u) * 32 + lane;
                                reinterpret_cast<uint32_t*>(x_perm)[(long long)r * H8 + j] = qv[u];
                                if ((lane & 1) == 0) scales[(long long)r * (H >> 4) + (j >> 1)] = (uint8_t)sb[u];
                            }
                        }
                    }
                }
            } else {
                uint2 qv[U];
                int sb[U];
#pragma unroll
                for (int u = 0; u < U; u++) {
                    if (it0 + u < iters) {  // warp-uniform: the quad shuffles see every lane
                        float f[8];
                        bf16x8_to_f32(v[u], f);
                        qv[u] = quant8_in_quad(f, &sb[u]);
                    }
                }
#pragma unroll
                for (int c = 0; c < KC; c++) {
                    unsigned m = mask[c];
                    while (m) {
                        const int b = __ffs(m) - 1;
                        m &= m - 1;
                        const int r = __shfl_sync(FULL, rows[c], b);
#pragma unroll
                        for (int u = 0; u < U; u++) {
                            if (in[u]) {
                                const int j = (it0 + u) * 32 + lane;
                                reinterpret_cast<uint2*>(x_perm)[(long long)r * H8 + j] = qv[u];
                                if ((lane & 3) == 0) scales[(long long)r * (H >> 5) + (j >> 2)] = (uint8_t)sb[u];
                            }
                        }
                    }
                }
            }
        }
    }
}

// max |x| over the tokens with at least one valid route (0 <= id < E): the amax of the rows the
// permute copies. Warp per token; *amax zeroed by the caller; one atomic per CTA.
__global__ void __launch_bounds__(256) amax_routed_kernel(const uint4* __restrict__ x, int T, int H,
                                                          const void* __restrict__ ids, bool i16, int K, int E,
                                                          float* __restrict__ amax) {
    const int lane = (int)lane_id();
    const int nwarps_total = (gridDim.x * blockDim.x) >> 5;
    const int H8 = H >> 3;
    float m = 0.0f;
    for (long long t = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += nwarps_total) {
        bool routed = false;
        for (int k = lane; k < K; k += 32) {
            const int e = load_id(ids, t * K + k, i16);
            routed |= e >= 0 && e < E;
        }
        if (!__any_sync(FULL, routed)) continue;        // warp-uniform
        const uint4* src = x + t * H8;
        for (int j = lane; j < H8; j += 32) {
            float f[8];
            bf16x8_to_f32(__ldg(src + j), f);
#pragma unroll
            for (int i = 0; i < 8; i++) m = fmaxf(m, fabsf(f[i]));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL, m, o));
    __shared__ float wmax[8];
    if (lane == 0) wmax[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float b = 0.0f;
        for (int w = 0; w < (int)(blockDim.x >> 5); w++) b = fmaxf(b, wmax[w]);
        if (b > 0.0f) atomicMax(reinterpret_cast<unsigned int*>(amax), __float_as_uint(b));
    }
}

// ---------------------------------------------------------------- standalone quantiser
// Row-wise: warp per row, rows < R only.
__global__ void __launch_bounds__(256) quant_rows_kernel(const uint4* __restrict__ x, int R_cap, int H,
                                                         const int* __restrict__ group_offsets, int E,
                                                         uint2* __restrict__ q, uint8_t* __restrict__ scales) {
    const int lane = (int)lane_id();
    const int R = __ldg(group_offsets + E);
    const int nwarps_total = (gridDim.x * blockDim.x) >> 5;
    const int H8 = H >> 3;
    const int iters = (H8 + 31) >> 5;
    for (long long r = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < R && r < R_cap;
         r += nwarps_total) {
        for (int it = 0; it < iters; it++) {
            const int j = it * 32 + lane;
            const bool in = j < H8;
            uint4 v = in ? __ldg(x + r * H8 + j) : make_uint4(0, 0, 0, 0);
            float f[8];
            bf16x8_to_f32(v, f);
            int sb;
            uint2 qv = quant8_in_quad(f, &sb);
            if (in) {
                q[r * H8 + j] = qv;
                if ((lane & 3) == 0) scales[r * (H >> 5) + (j >> 2)] = (uint8_t)sb;
            }
        }
    }
}

// Column-wise, group-aware: block (srow, column chunk of 256). Scale row srow
// belongs to the group e with e + off[e]/32 <= srow < (e+1) + off[e+1]/32;
// its block index within the group is b = srow - e - off[e]/32.
__global__ void __launch_bounds__(256) quant_cols_kernel(const __nv_bfloat16* __restrict__ x, int H,
                                                         const int* __restrict__ group_offsets, int E,
                                                         uint8_t* __restrict__ q, uint8_t* __restrict__ scales) {
    __shared__ int s_e;
    const int srow = blockIdx.x;
    if (threadIdx.x == 0) {
        int lo = 0, hi = E - 1;  // last e with e + off[e]/32 <= srow
        while (lo < hi) {
            int mid = (lo + hi + 1) >> 1;
            if (mid + __ldg(group_offsets + mid) / 32 <= srow) lo = mid;
            else hi = mid - 1;
        }
        s_e = lo;
    }
    __syncthreads();
    const int e = s_e;
    const int off0 = __ldg(group_offsets + e), off1 = __ldg(group_offsets + e + 1);
    const int b = srow - e - off0 / 32;
    if (b < 0) return;
    const int r0 = off0 + 32 * b;
    if (r0 >= off1) return;
    const int n = min(32, off1 - r0);
    const int col = blockIdx.y * blockDim.x + threadIdx.x;
    if (col >= H) return;
    float v[32];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; i++) {
        v[i] = i < n ? __bfloat162float(x[(long long)(r0 + i) * H + col]) : 0.0f;
        amax = fmaxf(amax, fabsf(v[i]));
    }
    const int sb = e8m0_scale_byte(amax);
    const float inv = e8m0_inv_scale(sb);
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
        unsigned short two = f32x2_to_e4m3x2(v[i] * inv, v[i + 1] * inv);
        if (i < n) q[(long long)(r0 + i) * H + col] = (uint8_t)(two & 0xff);
        if (i + 1 < n) q[(long long)(r0 + i + 1) * H + col] = (uint8_t)(two >> 8);
    }
    scales[(long long)srow * H + col] = (uint8_t)sb;
}

int sm_count() {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}

int rank_warps_per_block(int E) {
    int w = (48 * 1024) / (E * 4);
    return w < 1 ? 1 : (w > 8 ? 8 : w);
}

}  // namespace
}  // namespace moe

extern "C" int moe_permute_kernel_launches(int T, int K, int E) {
    using namespace moe;
    if (T < 0 || K < 1 || E < 1) return -1;
    if (T == 0) return 0;
    const int TT = tile_tokens(E);
    const long long tiles = ((long long)T + TT - 1) / TT;
    return scan_in_block(E, tiles) ? 2 : 3;
}

extern "C" size_t moe_permute_workspace_size(int T, int K, int E) {
    using namespace moe;
    if (T < 0 || K < 1 || E < 1) return 0;
    const int TT = tile_tokens(E);
    const long long tiles = ((long long)T + TT - 1) / TT;
    return align16((size_t)E * (size_t)(tiles > 0 ? tiles : 1) * sizeof(int)) + 16;
}

// The permute's argument checks other than the workspace's (shapes, dtypes, pointers,
// alignment), in the order every permute entry point reports them.
static moe_status permute_check_args(const void* x, int T, int H, const void* ids, moe_dtype id_dtype, int K,
                                     int E, const void* x_perm, const uint8_t* x_perm_scales,
                                     const int32_t* group_sizes, const int32_t* group_offsets,
                                     const int32_t* row_map, const int32_t* perm_src, bool fuse) {
    if (T < 0 || H < 32 || (H % 32) != 0 || K < 1 || E < 1 || K > E || K > 128) return MOE_ERR_INVALID_ARG;
    if (id_dtype != MOE_I16 && id_dtype != MOE_I32) return MOE_ERR_INVALID_ARG;
    if (!group_sizes || !group_offsets) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!x || !ids || !x_perm || !row_map || !perm_src)) return MOE_ERR_INVALID_ARG;
    if (fuse && T > 0 && !x_perm_scales) return MOE_ERR_INVALID_ARG;
    // (large E: the count kernel keeps a 64-bit token mask and a count per expert in shared memory)
    if ((long long)E * 4 > 227 * 1024 || (E > 64 && moe::rank_mask_smem(E) > 227 * 1024)) return MOE_ERR_UNSUPPORTED;
    if (!moe_host::aligned(x, 16) || !moe_host::aligned(x_perm, fuse ? 8 : 16) || !moe_host::aligned(row_map, 4) ||
        !moe_host::aligned(perm_src, 4) || !moe_host::aligned(group_sizes, 4) ||
        !moe_host::aligned(group_offsets, 4))
        return MOE_ERR_ALIGNMENT;
    return MOE_OK;
}

// fuse_mode: 0 bf16 rows, 1 MXFP8, 2 NVFP4 (with the device amax already computed on the stream)
static moe_status permute_impl(const void* x, int T, int H, const void* ids, moe_dtype id_dtype, int K, int E,
                               void* x_perm, uint8_t* x_perm_scales, int32_t* group_sizes, int32_t* group_offsets,
                               int32_t* row_map, int32_t* perm_src, int fuse_mode, const float* amax,
                               void* workspace, size_t workspace_bytes, moe_stream_t stream) {
    using namespace moe;
    const moe_status arg = permute_check_args(x, T, H, ids, id_dtype, K, E, x_perm, x_perm_scales, group_sizes,
                                              group_offsets, row_map, perm_src, fuse_mode != 0);
    if (arg != MOE_OK) return arg;
    if (!workspace || workspace_bytes < moe_permute_workspace_size(T, K, E)) return MOE_ERR_WORKSPACE;
    if (!moe_host::aligned(workspace, 16)) return MOE_ERR_ALIGNMENT;
    cudaStream_t s = moe_host::as_stream(stream);
    const bool i16 = id_dtype == MOE_I16;
    const int TT = tile_tokens(E);
    const int tiles = T > 0 ? (T + TT - 1) / TT : 1;
    PermuteWs w = carve(workspace, E, tiles);

    if (T == 0) {  // empty batch: all groups empty
        if (cudaMemsetAsync(group_sizes, 0, sizeof(int) * (size_t)E, s) != cudaSuccess) return MOE_ERR_CUDA;
        if (cudaMemsetAsync(group_offsets, 0, sizeof(int) * (size_t)(E + 1), s) != cudaSuccess)
            return MOE_ERR_CUDA;
        return MOE_OK;
    }
    // 1. rank
    if (E > 64) {
        // large E: a CTA per tile of 64 tokens (at most 64 * 128 routes, 8 per thread)
        const size_t smem = rank_mask_smem(E);
        const int per = (int)(((long long)TT * K + RANK_MASK_THREADS - 1) / RANK_MASK_THREADS);
#define MOE_RANK_MASK(mr)                                                                                         \
    do {                                                                                                           \
        if (smem > 48 * 1024 && cudaFuncSetAttribute(perm_rank_mask_kernel<mr>,                                    \
                                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=  \
                                    cudaSuccess)                                                                   \
            return MOE_ERR_CUDA;                                                                                   \
        if (moe_host::launch_pdl(perm_rank_mask_kernel<mr>, dim3(tiles), dim3(RANK_MASK_THREADS), smem, s, ids,   \
                                 i16, T, K, E, TT, tiles, w.table, row_map, w.ticket) != cudaSuccess)              \
            return MOE_ERR_CUDA;                                                                                   \
    } while (0)
        if (per <= 1) MOE_RANK_MASK(1);
        else if (per <= 2) MOE_RANK_MASK(2);
        else if (per <= 3) MOE_RANK_MASK(3);
        else if (per <= 4) MOE_RANK_MASK(4);
        else MOE_RANK_MASK(8);
#undef MOE_RANK_MASK
    } else {
        const int wpb = rank_warps_per_block(E);
        const size_t smem = (size_t)wpb * E * sizeof(int);
        if (smem > 48 * 1024) {
            if (cudaFuncSetAttribute(perm_rank_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
                cudaSuccess)
                return MOE_ERR_CUDA;
        }
        if (moe_host::launch_pdl(perm_rank_kernel, dim3((tiles + wpb - 1) / wpb), dim3(wpb * 32), smem, s, ids, i16,
                                 T, K, E, TT, tiles, w.table, row_map, w.ticket) != cudaSuccess)
            return MOE_ERR_CUDA;
    }
    if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
    // 2. scan (a separate kernel only when the count table is too large for one block's shared memory)
    const int cap = sm_count();
    const bool in_block = scan_in_block(E, tiles);
    if (!in_block) {
        const int experts_per_block = SCAN_THREADS / 32;
        int sblocks = (E + experts_per_block - 1) / experts_per_block;
        if (sblocks > cap) sblocks = cap;
        if (moe_host::launch_pdl(perm_scan_kernel, dim3(sblocks), dim3(SCAN_THREADS), 0, s, E, tiles, w.table,
                                 group_sizes, group_offsets, w.ticket) != cudaSuccess)
            return MOE_ERR_CUDA;
    }
    // 3. scatter: warp per token (with the scan in every block: one wave of blocks, as many as
    //    the SMs hold at once, each warp taking several tokens, so the scan of each block is
    //    spread over more rows)
    const long long warps_needed = T;
    const long long blocks_needed = (warps_needed + 7) / 8;
    const int KC = (K + 31) / 32;
    const size_t ssmem = in_block ? ((size_t)E * tiles + E + 1) * sizeof(int) : 0;
#define MOE_SCATTER(kc, fz, sc)                                                                                  \
    do {                                                                                                          \
        int per_sm = 4;                                                                                           \
        if (sc && cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, perm_scatter_kernel<kc, fz, sc>, 256,    \
                                                                ssmem) != cudaSuccess)                            \
            return MOE_ERR_CUDA;                                                                                  \
        const long long bcap = (long long)cap * (sc ? (per_sm > 0 ? per_sm : 1) : 16);                            \
        const long long blocks = blocks_needed < bcap ? blocks_needed : bcap;                                     \
        if (moe_host::launch_pdl(perm_scatter_kernel<kc, fz, sc>, dim3((unsigned)blocks), dim3(256), ssmem, s,  \
                                 (const uint4*)x, T, H, ids, i16, K, E, TT, tiles, (const int*)w.table,          \
                                 group_sizes, group_offsets, row_map, perm_src, x_perm, x_perm_scales, amax) !=   \
            cudaSuccess)                                                                                          \
            return MOE_ERR_CUDA;                                                                                  \
    } while (0)
#define MOE_SCATTER_KC(fz, sc)        \
    if (KC == 1) MOE_SCATTER(1, fz, sc); \
    else if (KC == 2) MOE_SCATTER(2, fz, sc); \
    else MOE_SCATTER(4, fz, sc);
    if (fuse_mode == 1) {
        if (in_block) { MOE_SCATTER_KC(1, true) } else { MOE_SCATTER_KC(1, false) }
    } else if (fuse_mode == 2) {
        if (in_block) { MOE_SCATTER_KC(2, true) } else { MOE_SCATTER_KC(2, false) }
    } else {
        if (in_block) { MOE_SCATTER_KC(0, true) } else { MOE_SCATTER_KC(0, false) }
    }
#undef MOE_SCATTER_KC
#undef MOE_SCATTER
    return moe_host::launch_status();
}

extern "C" moe_status moe_permute(const void* x, int T, int H, const void* ids, moe_dtype id_dtype, int K,
                                  int E, void* x_perm, uint8_t* x_perm_scales, int32_t* group_sizes,
                                  int32_t* group_offsets, int32_t* row_map, int32_t* perm_src,
                                  unsigned flags, void* workspace, size_t workspace_bytes,
                                  moe_stream_t stream) {
    if (flags & ~MOE_PERMUTE_FUSE_MXFP8) return MOE_ERR_INVALID_ARG;
    return permute_impl(x, T, H, ids, id_dtype, K, E, x_perm, x_perm_scales, group_sizes, group_offsets, row_map,
                        perm_src, (flags & MOE_PERMUTE_FUSE_MXFP8) ? 1 : 0, nullptr, workspace, workspace_bytes,
                        stream);
}

extern "C" moe_status moe_permute_nvfp4(const void* x, int T, int H, const void* ids, moe_dtype id_dtype, int K,
                                        int E, float* x_amax, void* x_perm_q, uint8_t* x_perm_scales,
                                        int32_t* group_sizes, int32_t* group_offsets, int32_t* row_map,
                                        int32_t* perm_src, void* workspace, size_t workspace_bytes,
                                        moe_stream_t stream) {
    using namespace moe;
    if (T < 0 || H < 32 || (H % 32) != 0 || K < 1 || E < 1 || K > E || K > 128) return MOE_ERR_INVALID_ARG;
    if (id_dtype != MOE_I16 && id_dtype != MOE_I32) return MOE_ERR_INVALID_ARG;
    if (!x_amax || (T > 0 && (!x || !ids || !x_perm_scales))) return MOE_ERR_INVALID_ARG;
    if (!moe_host::aligned(x_amax, 4) || !moe_host::aligned(x, 16)) return MOE_ERR_ALIGNMENT;
    cudaStream_t s = moe_host::as_stream(stream);
    // 0. the amax of the routed tokens' rows (= of the rows the scatter writes)
    if (cudaMemsetAsync(x_amax, 0, sizeof(float), s) != cudaSuccess) return MOE_ERR_CUDA;
    if (T > 0) {
        long long blocks = ((long long)T + 7) / 8;
        const long long cap = (long long)sm_count() * 8;
        if (blocks > cap) blocks = cap;
        amax_routed_kernel<<<(int)blocks, 256, 0, s>>>((const uint4*)x, T, H, ids, id_dtype == MOE_I16, K, E, x_amax);
        if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
    }
    return permute_impl(x, T, H, ids, id_dtype, K, E, x_perm_q, x_perm_scales, group_sizes, group_offsets, row_map,
                        perm_src, 2, x_amax, workspace, workspace_bytes, stream);
}

extern "C" moe_status moe_quant_mxfp8_grouped(const void* x, int R_cap, int H, const int32_t* group_offsets,
                                              int E, uint8_t* q, uint8_t* scales, unsigned flags,
                                              moe_stream_t stream) {
    using namespace moe;
    if (R_cap < 0 || H < 32 || (H % 32) != 0 || E < 1) return MOE_ERR_INVALID_ARG;
    if (flags & ~MOE_QUANT_COLWISE) return MOE_ERR_INVALID_ARG;
    if (R_cap == 0) return MOE_OK;
    if (!x || !group_offsets || !q || !scales) return MOE_ERR_INVALID_ARG;
    if (!moe_host::aligned(x, 16) || !moe_host::aligned(q, 8) || !moe_host::aligned(group_offsets, 4))
        return MOE_ERR_ALIGNMENT;
    cudaStream_t s = moe_host::as_stream(stream);
    if (flags & MOE_QUANT_COLWISE) {
        const long long srows = (long long)E + R_cap / 32 + 1;
        if (srows > 0x7fffffffLL) return MOE_ERR_UNSUPPORTED;
        dim3 grid((unsigned)srows, (unsigned)((H + 255) / 256));
        quant_cols_kernel<<<grid, 256, 0, s>>>((const __nv_bfloat16*)x, H, group_offsets, E, q, scales);
    } else {
        long long blocks = ((long long)R_cap + 7) / 8;
        const long long bcap = (long long)sm_count() * 16;
        if (blocks > bcap) blocks = bcap;
        quant_rows_kernel<<<(int)blocks, 256, 0, s>>>((const uint4*)x, R_cap, H, group_offsets, E, (uint2*)q,
                                                      scales);
    }
    return moe_host::launch_status();
}

// ---------------------------------------------------------------------------
// moe_permute_noalloc: moe_permute for callers that may not allocate device
// memory. Its scratch (the per-expert, per-token-tile count table and the scan's
// completion counter) lives in this file-scope array instead of a caller
// workspace. Every GPU that loads the library holds the array until the process
// exits; all calls on a device share it.
// ---------------------------------------------------------------------------
namespace moe {
namespace {

constexpr size_t NOALLOC_SCRATCH_BYTES = (size_t)4 << 20;  // 4 MiB
static __device__ __align__(256) uint8_t g_permute_scratch[NOALLOC_SCRATCH_BYTES];

// Device address of g_permute_scratch on the current device. Host code cannot use the
// array's name as a device address; the runtime gives it per device. It is asked on every
// call (a lookup once the module is loaded), so no address outlives a device reset or a
// context teardown. The first call on a device may load the module: make it before any
// stream capture.
moe_status noalloc_scratch(void** out) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
    *out = p;
    return MOE_OK;
}

}  // namespace
}  // namespace moe

extern "C" size_t moe_permute_noalloc_max_scratch(void) { return moe::NOALLOC_SCRATCH_BYTES; }

extern "C" moe_status moe_permute_noalloc(const void* x, int T, int H, const void* ids, moe_dtype id_dtype, int K,
                                          int E, void* x_perm, uint8_t* x_perm_scales, int32_t* group_sizes,
                                          int32_t* group_offsets, int32_t* row_map, int32_t* perm_src,
                                          unsigned flags, moe_stream_t stream) {
    if (flags & ~MOE_PERMUTE_FUSE_MXFP8) return MOE_ERR_INVALID_ARG;
    const moe_status arg = permute_check_args(x, T, H, ids, id_dtype, K, E, x_perm, x_perm_scales, group_sizes,
                                              group_offsets, row_map, perm_src, (flags & MOE_PERMUTE_FUSE_MXFP8) != 0);
    if (arg != MOE_OK) return arg;
    if (moe_permute_workspace_size(T, K, E) > moe::NOALLOC_SCRATCH_BYTES) return MOE_ERR_WORKSPACE;
    void* scratch = nullptr;
    moe_status st = moe::noalloc_scratch(&scratch);
    if (st != MOE_OK) return st;
    // The scratch needs no clearing: the rank kernel writes every table entry it
    // later reads and resets the completion counter before the scan kernel runs.
    return moe_permute(x, T, H, ids, id_dtype, K, E, x_perm, x_perm_scales, group_sizes, group_offsets, row_map,
                       perm_src, flags, scratch, moe::NOALLOC_SCRATCH_BYTES, stream);
}
