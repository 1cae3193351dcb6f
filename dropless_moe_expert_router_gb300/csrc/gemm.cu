// gemm.cu -- persistent ragged grouped GEMM on tcgen05 tensor cores: the
// forward SwiGLU expert MLP (two launches), its activation gradient (two
// launches) and its weight gradient.
//
// "Dropless MoE acceleration in JAX with NVIDIA Transformer Engine", section
// "Optimization 1: Grouped GEMM": one kernel covers every expert with its actual
// token count and computes only valid regions; the token counts stay on the
// device (no device-to-host copy, so the call can live in a CUDA graph); on
// Blackwell the expert matmuls can use MXFP8 block scaling. The same page's
// MoE-layer figure: the grouped MLP is two grouped GEMMs on variable-length
// groups; its "Measured training impact" is a training step, so the grouped
// backward GEMMs run on the same ragged groups.
//
// One kernel template, four modes:
//   UP     A = x_perm [R_cap, H] (rows grouped by expert), B = W13 packed
//          [E][2F][H]; epilogue: h = silu(a) * b (bf16 or MXFP8), optionally the
//          bf16 pre-activations (a | b) and a bf16 copy of h for the backward.
//   DOWN   A = h or dab [R_cap, K], B = W2p [E][H][F] or W13t [E][H][2F];
//          epilogue: plain bf16 store (y_perm, or dx).
//   DGRAD  A = dy_perm [R_cap, H], B = W2 [E][F][H]; epilogue: SwiGLU backward
//          da = dh * b * silu'(a), db = dh * silu(a) with the saved (a | b),
//          stored bf16 in the same interleaved layout.
//   WGRAD  contraction over each expert's rows: A = aT [M][Kpad], B = bT [N][Kpad]
//          (transposed, group-padded operands, zero past each group's end);
//          output dW[e] [M][N] bf16, or split into two [M][N/2] halves.
//
// Design (one CTA per SM, persistent, warp-specialised; 320 threads):
//   warp 0     TMA producer: A tile [128 rows x 128 B] and B tile [256 rows x 128 B]
//              per k-block into a 4-stage shared-memory ring (128-byte swizzle);
//              MXFP8 adds one TMA box of 16 E8M0 scale bytes per A and B row.
//   warp 1     allocates TMEM and issues tcgen05.mma (M=128, N=256) from one
//              lane; each k-block's commit frees its ring stage, each tile's
//              commit hands the accumulator to the epilogue. For MXFP8 the warp
//              first rearranges the k-block's scale words into the layout
//              tcgen05.cp expects and copies them to TMEM.
//   warp 10    (MXFP8) rearranges each landed slot of scales (four k-blocks) for tcgen05.cp.
//   warps 2-9  epilogue: two warps per TMEM lane quarter, each copying its half of
//              the fp32 accumulator columns to registers with tcgen05.ld and
//              handing TMEM back before the mode's math and stores (so with one
//              accumulator, as for MXFP8, the next tile's MMAs start at once).
// Tiles are scheduled on the device: every CTA reads group_offsets and walks
// the tile list with a static stride of gridDim.x. Row-grouped modes count
// ceil(m_e / 128) row tiles per expert and order tiles expert-major, then
// output column tile, then row tile (one weight tile is consumed by all row
// tiles of its expert while it is hot in L2); a row tile that runs past its
// group reads the next group's rows (or TMA zero fill past R_cap) and those
// accumulator rows are never stored. WGRAD tiles are (expert, N tile, M tile)
// with ceil(m_e / BK) k-blocks each; an expert without rows stores zeros.
// No padding of the data, no dropping.
//
// BF16: kind::f16, two TMEM accumulators (2 x 256 columns) so the epilogue of
// tile i overlaps the main loop of tile i+1. When groups are large, a tile is
// 256 rows computed by a cluster of two CTAs (tcgen05 cta_group::2): each CTA
// loads its 128 A rows and half of the B tile, the even CTA issues the MMAs
// into both CTAs' TMEM and its barriers collect both CTAs' loads and
// epilogues; the smaller stage (32 KB) allows a 6-deep ring.
// MXFP8: kind::mxf8f6f4.block_scale (E4M3 x E4M3, UE8M0 scale per 32
// elements); one accumulator plus per-stage scale-factor columns in TMEM.
#include "common.cuh"
#include "sm100_ptx.cuh"

#include <cudaTypedefs.h>

namespace moe {
namespace {

constexpr int BM = 128;          // rows per tile and CTA (MMA M per CTA)
constexpr int BN = 256;          // output columns per tile (MMA N)
constexpr int NUM_THREADS = 352;     // warp 0 TMA, warp 1 MMA, warps 2-9 epilogue, warp 10 scales (MXFP8)
constexpr int TMEM_COLS = 512;

enum { MODE_UP = 0, MODE_DOWN = 1, MODE_DGRAD = 2, MODE_WGRAD = 3 };

// PAIR: a tile is computed by a cluster of two CTAs with tcgen05 cta_group::2 --
// M = 256 rows (128 per CTA), and each CTA loads only its half of the B tile,
// so a stage is 32 KB and the ring is 6 stages deep.
template <bool FP8, bool PAIR = false, bool NV4 = false>
struct Cfg {
    static_assert(!(FP8 && PAIR), "MXFP8 uses single-CTA tiles");
    static_assert(!NV4 || FP8, "NVFP4 runs on the block-scaled 8-bit machinery");
    static constexpr int BK = FP8 ? 128 : 64;       // elements per k-block (128 bytes per row)
    static constexpr int UMMA_K = FP8 ? 32 : 16;    // elements per MMA instruction
    static constexpr int KSTEPS = BK / UMMA_K;      // MMAs per k-block (4)
    static constexpr int TM = PAIR ? 2 * BM : BM;   // rows of a tile (both CTAs of a pair)
    static constexpr int B_ROWS = PAIR ? BN / 2 : BN;  // B rows this CTA loads
    static constexpr int A_BYTES = BM * 128;
    static constexpr int B_BYTES = B_ROWS * 128;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = PAIR ? 6 : 4;
    // MXFP8 scales: one TMA box of 16 scale bytes (a group of four k-blocks) per operand row,
    // loaded once per group by the scale warp, up to SF_SLOTS groups ahead of the MMA warp,
    // into a ring of slots beside the operand stages; A rows first, then B rows. The scale
    // warp rearranges a landed slot in place into four k-block chunks of SF_CHUNK bytes
    // (A 512, B 2 x 512) laid out for tcgen05.cp.
    static constexpr int SF_SLOTS = FP8 ? 3 : 0;
    static constexpr int SF_SLOT_BYTES = FP8 ? (BM + BN) * 16 : 0;
    static constexpr int SF_CHUNK = 3 * 512;
    static constexpr int RING_BYTES = STAGES * STAGE_BYTES + SF_SLOTS * SF_SLOT_BYTES;
    static constexpr int ACC_STAGES = FP8 ? 1 : 2;
    // TMEM columns of one stage's scales: MXFP8 4 A + 8 B for the whole k-block (the four MMAs pick
    // a byte each); NVFP4 the same 12 for each of the four MMAs (each takes a whole word: four
    // E4M3 scales of 16 elements)
    static constexpr int SF_COLS = NV4 ? 48 : 12;
    // k-blocks one 16-byte scale box per row covers: MXFP8 four (4 x 128 / 32), NVFP4 one (256 / 16)
    static constexpr int SF_GROUP = NV4 ? 1 : 4;
    static constexpr int THREADS = FP8 ? NUM_THREADS : NUM_THREADS - 32;  // the scale warp exists for MXFP8 only
};

struct GemmArgs {
    const int* goff;             // [E+1] group offsets (device)
    int E;
    int Kdim;                    // contraction length (row-grouped modes)
    int N;                       // B rows per expert (row-grouped) / B rows (WGRAD)
    int n_tiles;                 // N / BN
    int R_cap;                   // rows of A (row-grouped)
    void* out;                   // output (see the mode)
    int ldo;                     // output row stride in elements
    uint8_t* out_scales;         // UP + MXFP8: h scales [R_cap, ldo/32]; DGRAD: optional dab scales
    uint8_t* out_q;              // DGRAD: optional row-wise MXFP8 codes of dab [R_cap, ldo]
    const uint8_t* a_scales;     // MXFP8 scales of A: [rows of A][sf_row_bytes]
    const uint8_t* b_scales;     // MXFP8 scales of B
    int sf_row_bytes;            // scale bytes per operand row (= contraction length / 32)
    __nv_bfloat16* ab;           // UP: optional (a | b) save; DGRAD: the saved (a | b) input
    __nv_bfloat16* h_bf16;       // UP + MXFP8: optional bf16 copy of h
    int M;                       // WGRAD: rows of aT (multiple of BM)
    int m_tiles;                 // WGRAD: M / BM
    void* out2;                  // WGRAD split: second half [E][M][N/2]
    int st32;                    // every output row segment is 32-byte aligned: 32-byte stores
    const float* a_amax;         // NVFP4: device amax of A's tensor (its encode scale 448 * 6 / amax)
    const float* b_amax;         // NVFP4: device amax of B's tensor
    float* out_amax;             // NVFP4 UP: device amax of the bf16 h written (zeroed by the caller)
};

template <bool FP8, bool PAIR = false>
constexpr size_t smem_bytes_for(int E) {
    using C = Cfg<FP8, PAIR>;
    return 1024 /* alignment slack */ + (size_t)C::RING_BYTES + 256 /* barriers, flags */ +
           (size_t)C::THREADS * 4 + (size_t)2 * (E + 1) * 4;
}

// One 1x32 MXFP8 block held by one thread: E8M0 scale byte from the block's amax,
// E4M3 codes (RNE, saturating) of v / 2^(byte - 127) packed four per word.
__device__ __forceinline__ int quant32_in_thread(const float* v, uint32_t* w) {
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 32; i++) amax = fmaxf(amax, fabsf(v[i]));
    const int sbyte = e8m0_scale_byte(amax);
    const float inv = e8m0_inv_scale(sbyte);
#pragma unroll
    for (int i = 0; i < 8; i++)
        w[i] = (uint32_t)f32x2_to_e4m3x2(v[4 * i] * inv, v[4 * i + 1] * inv) |
               ((uint32_t)f32x2_to_e4m3x2(v[4 * i + 2] * inv, v[4 * i + 3] * inv) << 16);
    return sbyte;
}

struct TileInfo {
    int e, m, n;
    int row0, rows;      // this CTA's first output row and its rows inside the group (may be <= 0)
    int a_row, b_row;    // operand rows this CTA loads
    int k0, nkb;         // first contraction element and number of k-blocks
};

// Row-grouped modes: tile -> (expert, column tile, row tile of C::TM rows).
template <bool FP8, bool PAIR>
__device__ __forceinline__ TileInfo decode_rows(int tile, const int* s_mtp, const int* s_goff, const GemmArgs& p,
                                                int rank) {
    using C = Cfg<FP8, PAIR>;
    const int q = tile / p.n_tiles;
    int lo = 0, hi = p.E - 1;  // last e with s_mtp[e] <= q (never an empty expert)
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (s_mtp[mid] <= q) lo = mid;
        else hi = mid - 1;
    }
    const int mt = s_mtp[lo + 1] - s_mtp[lo];
    const int local = tile - s_mtp[lo] * p.n_tiles;
    TileInfo t;
    t.e = lo;
    t.n = local / mt;
    t.m = local - t.n * mt;
    t.row0 = s_goff[lo] + t.m * C::TM + BM * rank;
    t.rows = min(BM, s_goff[lo + 1] - t.row0);
    t.a_row = t.row0;
    t.b_row = lo * p.N + t.n * BN + C::B_ROWS * rank;
    t.k0 = 0;
    t.nkb = p.Kdim / C::BK;
    return t;
}

// WGRAD: tile -> (expert, N tile, M tile); the expert's rows sit at
// [128 * (e + goff[e] / 128), + m_e) of the padded contraction axis.
template <bool FP8, bool PAIR>
__device__ __forceinline__ TileInfo decode_wgrad(int tile, const int* s_goff, const GemmArgs& p, int rank) {
    using C = Cfg<FP8, PAIR>;
    const int per = p.m_tiles * p.n_tiles;
    TileInfo t;
    t.e = tile / per;
    const int local = tile - t.e * per;
    t.n = local / p.m_tiles;
    t.m = local - t.n * p.m_tiles;
    const int g0 = s_goff[t.e], m_e = s_goff[t.e + 1] - g0;
    t.row0 = t.m * C::TM + BM * rank;
    t.rows = BM;
    t.a_row = t.row0;
    t.b_row = t.n * BN + C::B_ROWS * rank;
    t.k0 = 128 * (t.e + g0 / 128);
    t.nkb = (m_e + C::BK - 1) / C::BK;
    return t;
}

template <int MODE, bool FP8, bool PAIR>
__device__ __forceinline__ TileInfo decode(int tile, const int* s_mtp, const int* s_goff, const GemmArgs& p,
                                           int rank) {
    if constexpr (MODE == MODE_WGRAD) return decode_wgrad<FP8, PAIR>(tile, s_goff, p, rank);
    else return decode_rows<FP8, PAIR>(tile, s_mtp, s_goff, p, rank);
}

// First contraction element of a tile, in units of 128 elements (WGRAD: the
// expert's padded start; row-grouped modes: 0).
template <int MODE>
__device__ __forceinline__ int tile_k0_div128(const GemmArgs& p, int tile, const int* s_goff) {
    if constexpr (MODE == MODE_WGRAD) {
        const int e = tile / (p.m_tiles * p.n_tiles);
        return e + s_goff[e] / 128;
    } else {
        return 0;
    }
}

__device__ __forceinline__ float silu_f(float a) { return __fdividef(a, 1.0f + __expf(-a)); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Epilogue outputs are streamed (evict-first in L2): the operand tiles that the other CTAs
// are about to re-read stay resident instead.
// One 32-byte global store (dst 32-byte aligned): a whole sector per thread.
__device__ __forceinline__ void st_global_32B(void* dst, const uint32_t* w) {
    asm volatile("st.global.cs.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

// 32 bytes from w[0..8) at dst: one 32-byte store when st32, else two 16-byte stores.
__device__ __forceinline__ void store_32B(void* dst, const uint32_t* w, bool st32) {
    if (st32) {
        st_global_32B(dst, w);
    } else {
        uint4* d = reinterpret_cast<uint4*>(dst);
        __stcs(d, make_uint4(w[0], w[1], w[2], w[3]));
        __stcs(d + 1, make_uint4(w[4], w[5], w[6], w[7]));
    }
}

// 32 fp32 values -> 32 bf16 (64 bytes).
__device__ __forceinline__ void store_bf16x32(void* dst, const float* v, bool st32) {
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; i++) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
    store_32B(dst, w, st32);
    store_32B(static_cast<uint8_t*>(dst) + 32, w + 8, st32);
}

__device__ __forceinline__ void load_bf16x32(const void* src, float* v) {
    const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
    for (int i = 0; i < 4; i++) bf16x8_to_f32(s[i], v + 8 * i);
}

template <int MODE, bool FP8, bool PAIR, bool NV4 = false>
__global__ void __launch_bounds__(Cfg<FP8, PAIR>::THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                        const GemmArgs p) {
    using C = Cfg<FP8, PAIR, NV4>;
    constexpr int STAGES = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ring = smem;  // STAGES x [A | B]
    uint8_t* sfring = ring + (size_t)STAGES * C::STAGE_BYTES;  // MXFP8: SF_SLOTS x [A scales | B scales]
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + (size_t)C::RING_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* done = tempty + 2;
    uint64_t* sf_full = done + 1;   // MXFP8 scale slots: landed / rearranged / free again
    uint64_t* sf_ready = sf_full + 3;
    uint64_t* sf_empty = sf_ready + 3;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sf_empty + 3);
    volatile uint32_t* s_abort = s_tmem + 1;
    int* s_part = reinterpret_cast<int*>(smem + (size_t)C::RING_BYTES + 256);
    int* s_goff = s_part + C::THREADS;
    int* s_mtp = s_goff + (p.E + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int E = p.E;
    // CTA pairs: rank within the pair; the even CTA (rank 0) issues the MMAs and owns
    // the barriers both CTAs' loads and epilogues signal
    const int rank = PAIR ? (int)ptx::cluster_ctarank() : 0;
    const bool leader = rank == 0;
    const int tile0 = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int tile_step = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; s++) {
            ptx::mbar_init(&full[s], 1);
            ptx::mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < 3; s++) {
            ptx::mbar_init(&sf_full[s], 1);
            ptx::mbar_init(&sf_ready[s], 1);
            ptx::mbar_init(&sf_empty[s], 1);
        }
        for (int a = 0; a < 2; a++) {
            ptx::mbar_init(&tfull[a], 1);
            ptx::mbar_init(&tempty[a], PAIR ? 16 : 8);  // one arrival per epilogue warp (of both CTAs of a pair)
        }
        ptx::mbar_init(done, 1);
        *s_abort = 0u;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmB);
        if constexpr (FP8) {
            ptx::prefetch_tmap(&tmSA);
            ptx::prefetch_tmap(&tmSB);
        }
    }
    if constexpr (PAIR) ptx::cluster_sync();  // both CTAs' barriers exist before any cross-CTA signal
    if (warp == 1) {
        if constexpr (PAIR) {
            ptx::tmem_alloc_pair(s_tmem, TMEM_COLS);
            ptx::tmem_relinquish_pair();
        } else {
            ptx::tmem_alloc(s_tmem, TMEM_COLS);
            ptx::tmem_relinquish();
        }
    }
    // group table: offsets, and the exclusive scan of row tiles (C::TM rows) per expert
    for (int e = threadIdx.x; e <= E; e += C::THREADS) s_goff[e] = __ldg(p.goff + e);
    __syncthreads();
    {
        const int per = (E + C::THREADS - 1) / C::THREADS;
        const int b0 = threadIdx.x * per;
        int local = 0;
        for (int j = 0; j < per; j++) {
            int e = b0 + j;
            if (e < E) local += (s_goff[e + 1] - s_goff[e] + C::TM - 1) / C::TM;
        }
        s_part[threadIdx.x] = local;
        __syncthreads();
        if (threadIdx.x == 0) {
            int run = 0;
            for (int i = 0; i < C::THREADS; i++) {
                int v = s_part[i];
                s_part[i] = run;
                run += v;
            }
            s_mtp[E] = run;
        }
        __syncthreads();
        int run = s_part[threadIdx.x];
        for (int j = 0; j < per; j++) {
            int e = b0 + j;
            if (e < E) {
                s_mtp[e] = run;
                run += (s_goff[e + 1] - s_goff[e] + C::TM - 1) / C::TM;
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) ptx::cluster_sync();  // both CTAs' TMEM is allocated
    ptx::tc_fence_after();

    const uint32_t tmem = *s_tmem;
    const int total_tiles = MODE == MODE_WGRAD ? E * p.m_tiles * p.n_tiles : s_mtp[E] * p.n_tiles;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        int stage = 0;
        uint32_t phase = 0;
        int issued = 0;
        bool ok = true;
        for (int tile = tile0; tile < total_tiles && ok; tile += tile_step) {
            const TileInfo ti = decode<MODE, FP8, PAIR>(tile, s_mtp, s_goff, p, rank);
            for (int kb = 0; kb < ti.nkb; kb++) {
                const int k = ti.k0 + kb * C::BK;
                if (!ptx::wait_parity(&empty[stage], phase ^ 1u, s_abort)) { ok = false; break; }
                uint8_t* sa = ring + (size_t)stage * C::STAGE_BYTES;
                uint8_t* sb = sa + C::A_BYTES;
                if (lane == 0) {
                    if constexpr (PAIR) {
                        // the even CTA's full barrier counts both CTAs' bytes
                        if (leader) ptx::mbar_arrive_expect_tx(&full[stage], 2 * C::STAGE_BYTES);
                        const uint32_t bar = ptx::mapa_rank(&full[stage], 0);
                        ptx::tma_load_2d_pair(sa, &tmA, bar, k, ti.a_row);
                        ptx::tma_load_2d_pair(sb, &tmB, bar, k, ti.b_row);
                    } else {
                        ptx::mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
                        ptx::tma_load_2d(sa, &tmA, &full[stage], k, ti.a_row);
                        ptx::tma_load_2d(sb, &tmB, &full[stage], k, ti.b_row);
                    }
                }
                __syncwarp();
                issued++;
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
        if (!ok && !PAIR) {
            // give the loads already issued a bounded chance to land before the CTA exits
            for (int i = 0; i < STAGES && i < issued; i++) {
                if (--stage < 0) { stage = STAGES - 1; phase ^= 1u; }
                volatile uint32_t never = 0u;
                ptx::wait_parity(&full[stage], phase, &never, 100000000ull);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (even CTA of a pair)
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        int sslot = 0;
        uint32_t sphase = 0;
        bool ok = leader;
        for (int tile = tile0; tile < total_tiles && ok; tile += tile_step) {
            const int nkb =
                MODE == MODE_WGRAD ? decode_wgrad<FP8, PAIR>(tile, s_goff, p, rank).nkb : p.Kdim / C::BK;
            const int k0b = tile_k0_div128<MODE>(p, tile, s_goff);
            if (!ptx::wait_parity(&tempty[acc], acc_phase ^ 1u, s_abort)) { ok = false; break; }
            ptx::tc_fence_after();
            const uint32_t d_tmem = tmem + (uint32_t)(acc * BN);
            for (int kb = 0; kb < nkb; kb++) {
                const int gk = k0b + kb;                 // k-block index along the contraction
                if (!ptx::wait_parity(&full[stage], phase, s_abort)) { ok = false; break; }
                // MXFP8: the group's scales, rearranged by the scale warp
                if (FP8 && (NV4 || kb == 0 || (gk & 3) == 0) &&
                    !ptx::wait_parity(&sf_ready[sslot], sphase, s_abort)) {
                    ok = false;
                    break;
                }
                ptx::tc_fence_after();
                uint8_t* sa = ring + (size_t)stage * C::STAGE_BYTES;
                uint8_t* sb = sa + C::A_BYTES;
                const bool group_end = NV4 || kb == nkb - 1 || (gk & 3) == 3;
                if (lane == 0) {
                    const uint32_t a0 = ptx::smem_addr(sa), b0 = ptx::smem_addr(sb);
                    if constexpr (NV4) {
                        // NVFP4: the slot holds this k-block's scales; chunk k (one word per row)
                        // feeds MMA k, which covers 64 elements (32 bytes) of the k-block
                        const uint32_t sf_t = tmem + (uint32_t)(BN + stage * C::SF_COLS);
                        const uint32_t sfa_s = ptx::smem_addr(sfring + (size_t)sslot * C::SF_SLOT_BYTES);
#pragma unroll
                        for (int k = 0; k < C::KSTEPS; k++) {
                            ptx::tc_cp_32x128b_warpx4(sf_t + 12 * k, ptx::sdesc_plain(sfa_s + k * C::SF_CHUNK));
                            ptx::tc_cp_32x128b_warpx4(sf_t + 12 * k + 4,
                                                      ptx::sdesc_plain(sfa_s + k * C::SF_CHUNK + 512));
                            ptx::tc_cp_32x128b_warpx4(sf_t + 12 * k + 8,
                                                      ptx::sdesc_plain(sfa_s + k * C::SF_CHUNK + 1024));
                        }
#pragma unroll
                        for (int k = 0; k < C::KSTEPS; k++)
                            ptx::mma_nvf4(d_tmem, ptx::sdesc_k_sw128(a0 + k * 32), ptx::sdesc_k_sw128(b0 + k * 32),
                                          ptx::idesc_nvf4(BM, BN), sf_t + 12 * k, sf_t + 12 * k + 4, (kb | k) != 0);
                        ptx::tc_commit(&empty[stage]);
                        ptx::tc_commit(&sf_empty[sslot]);
                    } else if constexpr (FP8) {
                        const uint32_t sf_t = tmem + (uint32_t)(BN + stage * C::SF_COLS);
                        const uint32_t sfa_s =
                            ptx::smem_addr(sfring + (size_t)sslot * C::SF_SLOT_BYTES + (gk & 3) * C::SF_CHUNK);
                        ptx::tc_cp_32x128b_warpx4(sf_t, ptx::sdesc_plain(sfa_s));
                        ptx::tc_cp_32x128b_warpx4(sf_t + 4, ptx::sdesc_plain(sfa_s + 512));
                        ptx::tc_cp_32x128b_warpx4(sf_t + 8, ptx::sdesc_plain(sfa_s + 1024));
#pragma unroll
                        for (int k = 0; k < C::KSTEPS; k++)
                            ptx::mma_mxf8(d_tmem, ptx::sdesc_k_sw128(a0 + k * 32), ptx::sdesc_k_sw128(b0 + k * 32),
                                          ptx::idesc_mxf8(BM, BN, k, k), sf_t, sf_t + 4, (kb | k) != 0);
                        ptx::tc_commit(&empty[stage]);
                        if (group_end) ptx::tc_commit(&sf_empty[sslot]);  // the slot's last copies are done
                    } else if constexpr (PAIR) {
#pragma unroll
                        for (int k = 0; k < C::KSTEPS; k++)
                            ptx::mma_f16_pair(d_tmem, ptx::sdesc_k_sw128(a0 + k * 32),
                                              ptx::sdesc_k_sw128(b0 + k * 32), ptx::idesc_bf16(2 * BM, BN),
                                              (kb | k) != 0);
                        ptx::tc_commit_pair(&empty[stage], 0x3);  // frees the stage in both CTAs
                    } else {
#pragma unroll
                        for (int k = 0; k < C::KSTEPS; k++)
                            ptx::mma_f16(d_tmem, ptx::sdesc_k_sw128(a0 + k * 32), ptx::sdesc_k_sw128(b0 + k * 32),
                                         ptx::idesc_bf16(BM, BN), (kb | k) != 0);
                        ptx::tc_commit(&empty[stage]);
                    }
                }
                __syncwarp();
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                if (FP8 && group_end && ++sslot == C::SF_SLOTS) { sslot = 0; sphase ^= 1u; }
            }
            if (!ok) break;
            if (lane == 0) {
                if constexpr (PAIR) ptx::tc_commit_pair(&tfull[acc], 0x3);
                else ptx::tc_commit(&tfull[acc]);
            }
            __syncwarp();
            if (++acc == C::ACC_STAGES) { acc = 0; acc_phase ^= 1u; }
        }
        if (leader) {
            // make sure every MMA issued by this CTA has completed before TMEM is released
            if (lane == 0) {
                if constexpr (PAIR) ptx::tc_commit_pair(done, 0x1);
                else ptx::tc_commit(done);
            }
            __syncwarp();
            volatile uint32_t never = 0u;
            ptx::wait_parity(done, 0u, &never, 100000000ull);
        }
    } else if (FP8 && warp == 10) {
        // ------------------------------------------------------------ scale warp (MXFP8)
        // Loads this CTA's scale groups (the 16 scale bytes per row of a group of four
        // k-blocks), up to SF_SLOTS groups ahead of the MMA warp, and rearranges each landed
        // slot for tcgen05.cp .32x128b: k-block w's chunk at w * SF_CHUNK holds the A rows
        // (word lane*4 + j = row 32 j + lane) and then the B rows 0-127 and 128-255 in the
        // same order. In place, off the MMA warp's critical path. Groups are walked in the
        // MMA warp's order: every tile with k-blocks, a group starting at its first k-block
        // and at every k-block index that is a multiple of four.
        if constexpr (FP8) {
            struct Cursor {
                int tile, kb;
                TileInfo ti;
            };
            auto first_from = [&](int tile) {
                Cursor c;
                c.tile = tile;
                c.kb = 0;
                for (; c.tile < total_tiles; c.tile += tile_step) {
                    c.ti = decode<MODE, FP8, PAIR>(c.tile, s_mtp, s_goff, p, rank);
                    if (c.ti.nkb > 0) break;
                }
                return c;
            };
            auto next_group = [&](Cursor c) {
                c.kb += NV4 ? 1 : 4 - ((c.ti.k0 / C::BK + c.kb) & 3);
                return c.kb < c.ti.nkb ? c : first_from(c.tile + tile_step);
            };
            Cursor ld = first_from(tile0), pr = ld;
            int ld_slot = 0, pr_slot = 0, loaded = 0;   // loaded: issued and not yet rearranged
            uint32_t ld_phase = 0, pr_phase = 0;
            // Neither step blocks the other (non-blocking barrier tests): a load is issued when its
            // slot is free again (the MMA warp finished the group it held) and a landed group is
            // rearranged at once, so the groups after the one in use are always ready or in flight.
            uint64_t t_idle = ptx::globaltimer_ns();
            while (pr.tile < total_tiles) {
                bool progress = false;
                // (every lane polls, so each has acquired what it reads; the branch is taken only
                // when all lanes saw the phase complete, keeping the warp converged)
                if (ld.tile < total_tiles && loaded < C::SF_SLOTS &&
                    __all_sync(FULL, ptx::mbar_test_wait(&sf_empty[ld_slot], ld_phase ^ 1u))) {
                    if (lane == 0) {
                        uint8_t* sf = sfring + (size_t)ld_slot * C::SF_SLOT_BYTES;
                        // scale byte of the group's first element: MXFP8 element / 32 (groups of four
                        // k-blocks, 16-byte aligned); NVFP4 byte index (2 elements) / 8 = element / 16
                        const int kx = NV4 ? (ld.ti.k0 + ld.kb * C::BK) / 8 : ((ld.ti.k0 + ld.kb * C::BK) / 32) & ~15;
                        ptx::mbar_arrive_expect_tx(&sf_full[ld_slot], C::SF_SLOT_BYTES);
                        ptx::tma_load_2d(sf, &tmSA, &sf_full[ld_slot], kx, ld.ti.a_row);
                        ptx::tma_load_2d(sf + BM * 16, &tmSB, &sf_full[ld_slot], kx, ld.ti.b_row);
                    }
                    __syncwarp();
                    loaded++;
                    ld = next_group(ld);
                    if (++ld_slot == C::SF_SLOTS) { ld_slot = 0; ld_phase ^= 1u; }
                    progress = true;
                }
                if (loaded > 0 && __all_sync(FULL, ptx::mbar_test_wait(&sf_full[pr_slot], pr_phase))) {
                    uint8_t* sf = sfring + (size_t)pr_slot * C::SF_SLOT_BYTES;
                    const uint4* la = reinterpret_cast<const uint4*>(sf);
                    const uint4* lb = reinterpret_cast<const uint4*>(sf + BM * 16);
                    uint4 va[4], vb[8];
#pragma unroll
                    for (int j = 0; j < 4; j++) va[j] = la[32 * j + lane];
#pragma unroll
                    for (int j = 0; j < 8; j++) vb[j] = lb[32 * j + lane];
                    __syncwarp();
                    uint4* out = reinterpret_cast<uint4*>(sf);
#pragma unroll
                    for (int w = 0; w < 4; w++) {
                        auto word = [w](const uint4& v) { return w == 0 ? v.x : w == 1 ? v.y : w == 2 ? v.z : v.w; };
                        uint4* chunk = out + w * (C::SF_CHUNK / 16);
                        chunk[lane] = make_uint4(word(va[0]), word(va[1]), word(va[2]), word(va[3]));
                        chunk[32 + lane] = make_uint4(word(vb[0]), word(vb[1]), word(vb[2]), word(vb[3]));
                        chunk[64 + lane] = make_uint4(word(vb[4]), word(vb[5]), word(vb[6]), word(vb[7]));
                    }
                    ptx::fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(&sf_ready[pr_slot]);
                    loaded--;
                    pr = next_group(pr);
                    if (++pr_slot == C::SF_SLOTS) { pr_slot = 0; pr_phase ^= 1u; }
                    progress = true;
                }
                // bounded: give up (and flag it) when nothing has moved for the wait limit
                if (progress) {
                    t_idle = ptx::globaltimer_ns();
                } else if (__nanosleep(64), *s_abort) {
                    break;
                } else if (ptx::globaltimer_ns() - t_idle > ptx::WAIT_LIMIT_NS) {
                    *s_abort = 1u;
                    raise_device_error(MOE_DEVERR_TIMEOUT);
                    break;
                }
            }
            // give the scale loads still in flight a bounded chance to land before the CTA exits
            for (int i = 0; i < loaded; i++) {
                volatile uint32_t never = 0u;
                ptx::wait_parity(&sf_full[pr_slot], pr_phase, &never, 100000000ull);
                if (++pr_slot == C::SF_SLOTS) { pr_slot = 0; pr_phase ^= 1u; }
            }
        }
    } else {
        // ------------------------------------------------------------ epilogue (8 warps)
        // Two warps per TMEM lane quarter, each owning half of the tile's columns. A warp
        // first copies its 128 accumulator columns to registers and hands TMEM back (so the
        // next tile's MMAs can start), then does the math and the stores.
        const int q = warp & 3;                  // TMEM lane quarter of this warp
        const int hf = (warp - 2) >> 2;          // column half of this warp
        const int rit = q * 32 + lane;           // row within this CTA's tile
        int acc = 0;
        uint32_t acc_phase = 0;
        // NVFP4: the accumulator sums decoded products without the two tensors' encode scales;
        // alpha = 1 / (S_A S_B) restores them. h_amax: max |h| of the bf16 h this thread wrote.
        float alpha = 1.0f, h_amax = 0.0f;
        if constexpr (NV4)
            alpha = __fdiv_rn(1.0f, nvfp4_encode_scale(__ldg(p.a_amax))) *
                    __fdiv_rn(1.0f, nvfp4_encode_scale(__ldg(p.b_amax)));
        for (int tile = tile0; tile < total_tiles; tile += tile_step) {
            const TileInfo ti = decode<MODE, FP8, PAIR>(tile, s_mtp, s_goff, p, rank);
            if (!ptx::wait_parity(&tfull[acc], acc_phase, s_abort)) break;
            ptx::tc_fence_after();
            const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
            const bool valid = rit < ti.rows;
            const long long r = (long long)ti.row0 + rit;
            const bool has_acc = !(MODE == MODE_WGRAD && ti.nkb == 0);  // an expert without rows: zeros
            uint32_t v[128];
            if (has_acc) {
                if constexpr (MODE == MODE_UP) {
                    // gate columns [64 hf, 64 hf + 64) and the matching up columns
                    ptx::tmem_ld_x32(tbase + 64 * hf, v);
                    ptx::tmem_ld_x32(tbase + 64 * hf + 32, v + 32);
                    ptx::tmem_ld_x32(tbase + BN / 2 + 64 * hf, v + 64);
                    ptx::tmem_ld_x32(tbase + BN / 2 + 64 * hf + 32, v + 96);
                } else {
#pragma unroll
                    for (int c = 0; c < 4; c++) ptx::tmem_ld_x32(tbase + 128 * hf + 32 * c, v + 32 * c);
                }
                ptx::tmem_wait_ld();
            } else {
#pragma unroll
                for (int i = 0; i < 128; i++) v[i] = 0u;
            }
            ptx::tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if constexpr (PAIR) ptx::mbar_arrive_cluster(ptx::mapa_rank(&tempty[acc], 0));  // even CTA's barrier
                else ptx::mbar_arrive(&tempty[acc]);
            }
            if (++acc == C::ACC_STAGES) { acc = 0; acc_phase ^= 1u; }
            if constexpr (NV4) {
                float* fs = reinterpret_cast<float*>(v);
#pragma unroll
                for (int i = 0; i < 128; i++) fs[i] *= alpha;
            }
            const float* f = reinterpret_cast<const float*>(v);

            if constexpr (MODE == MODE_UP) {
#pragma unroll
                for (int c = 0; c < 2; c++) {
                    const int hcol = ti.n * (BN / 2) + 64 * hf + 32 * c;   // h column
                    if (valid && p.ab) {
                        // saved pre-activations, same interleaved layout as W13 packed
                        __nv_bfloat16* abrow = p.ab + r * (2 * p.ldo) + ti.n * BN + 64 * hf + 32 * c;
                        store_bf16x32(abrow, f + 32 * c, p.st32);
                        store_bf16x32(abrow + BN / 2, f + 64 + 32 * c, p.st32);
                    }
                    // h = silu(a) * b, written over the gate values it no longer needs
                    float* hv = reinterpret_cast<float*>(v) + 32 * c;
#pragma unroll
                    for (int i = 0; i < 32; i++) hv[i] = silu_f(hv[i]) * f[64 + 32 * c + i];
                    if constexpr (FP8 && !NV4) {
                        uint32_t w[8];
                        const int sbyte = quant32_in_thread(hv, w);
                        if (valid) {
                            store_32B(static_cast<uint8_t*>(p.out) + r * p.ldo + hcol, w, p.st32);
                            p.out_scales[r * (p.ldo / 32) + hcol / 32] = (uint8_t)sbyte;
                            if (p.h_bf16) store_bf16x32(p.h_bf16 + r * p.ldo + hcol, hv, p.st32);
                        }
                    } else {
                        if (valid) {
                            store_bf16x32(static_cast<__nv_bfloat16*>(p.out) + r * p.ldo + hcol, hv, p.st32);
                            if constexpr (NV4) {
                                // amax of the bf16 values stored (the next quantisation's tensor scale)
#pragma unroll
                                for (int i = 0; i < 32; i++)
                                    h_amax = fmaxf(h_amax, fabsf(__bfloat162float(__float2bfloat16_rn(hv[i]))));
                            }
                        }
                    }
                }
            } else if constexpr (MODE == MODE_DGRAD) {
                // dh columns fc = n*256 + 128 hf + 32c + i; (a | b) and (da | db) interleaved per 128.
                // The saved (a | b) is read-only here: a chunk's eight 16-byte loads are issued
                // before its math, one memory round trip per chunk of 32 columns.
                if (valid) {
                    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out);
#pragma unroll
                    for (int c = 0; c < 4; c++) {
                        const int fc = ti.n * BN + 128 * hf + 32 * c;
                        const long long off = r * p.ldo + (long long)(fc / 128) * 256 + (fc % 128);
                        const uint4* src = reinterpret_cast<const uint4*>(p.ab + off);
                        uint4 av[4], bv[4];
#pragma unroll
                        for (int sbk = 0; sbk < 4; sbk++) {
                            av[sbk] = __ldg(src + sbk);
                            bv[sbk] = __ldg(src + 16 + sbk);   // + 128 elements
                        }
                        uint32_t wa[16], wb[16];
#pragma unroll
                        for (int sbk = 0; sbk < 4; sbk++) {
                            float a[8], b[8];
                            bf16x8_to_f32(av[sbk], a);
                            bf16x8_to_f32(bv[sbk], b);
#pragma unroll
                            for (int i = 0; i < 8; i += 2) {
                                float da2[2], db2[2];
#pragma unroll
                                for (int u = 0; u < 2; u++) {
                                    const float dh = f[32 * c + 8 * sbk + i + u];
                                    const float sg = __fdividef(1.0f, 1.0f + __expf(-a[i + u]));
                                    da2[u] = dh * b[i + u] * (sg * (1.0f + a[i + u] * (1.0f - sg)));
                                    db2[u] = dh * a[i + u] * sg;
                                }
                                wa[4 * sbk + i / 2] = pack_bf16x2(da2[0], da2[1]);
                                wb[4 * sbk + i / 2] = pack_bf16x2(db2[0], db2[1]);
                            }
                        }
                        store_32B(o + off, wa, p.st32);
                        store_32B(o + off + 16, wa + 8, p.st32);
                        store_32B(o + off + 128, wb, p.st32);
                        store_32B(o + off + 144, wb + 8, p.st32);
                        if (p.out_q) {
                            // row-wise MXFP8 of the bf16 da and db blocks just stored (the dx GEMM's operand)
#pragma unroll
                            for (int half = 0; half < 2; half++) {
                                const uint32_t* src2 = half ? wb : wa;
                                float fv[32];
#pragma unroll
                                for (int i = 0; i < 16; i++) {
                                    fv[2 * i] = __uint_as_float(src2[i] << 16);
                                    fv[2 * i + 1] = __uint_as_float(src2[i] & 0xffff0000u);
                                }
                                uint32_t w[8];
                                const int sbyte = quant32_in_thread(fv, w);
                                const long long qo = off + 128 * half;
                                store_32B(p.out_q + qo, w, p.st32);
                                p.out_scales[qo >> 5] = (uint8_t)sbyte;
                            }
                        }
                    }
                }
            } else if constexpr (MODE == MODE_WGRAD) {
                const long long orow = (long long)ti.e * p.M + ti.row0 + rit;
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    if (p.out2) {  // split: column half 0 of the tile -> out, half 1 -> out2
                        __nv_bfloat16* o = static_cast<__nv_bfloat16*>(hf ? p.out2 : p.out);
                        store_bf16x32(o + orow * (p.N / 2) + ti.n * (BN / 2) + 32 * c, f + 32 * c, p.st32);
                    } else {
                        store_bf16x32(static_cast<__nv_bfloat16*>(p.out) + orow * p.N + ti.n * BN + 128 * hf + 32 * c,
                                      f + 32 * c, p.st32);
                    }
                }
            } else {  // MODE_DOWN
                if (valid) {
#pragma unroll
                    for (int c = 0; c < 4; c++)
                        store_bf16x32(static_cast<__nv_bfloat16*>(p.out) + r * p.ldo + ti.n * BN + 128 * hf + 32 * c,
                                      f + 32 * c, p.st32);
                }
            }
        }
        if constexpr (NV4 && MODE == MODE_UP) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) h_amax = fmaxf(h_amax, __shfl_xor_sync(FULL, h_amax, o));
            if (lane == 0 && h_amax > 0.0f)
                atomicMax(reinterpret_cast<unsigned int*>(p.out_amax), __float_as_uint(h_amax));
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if constexpr (PAIR) ptx::cluster_sync();  // no CTA leaves while its peer may still signal it
    if (warp == 1) {
        ptx::tc_fence_after();
        if constexpr (PAIR) ptx::tmem_dealloc_pair(tmem, TMEM_COLS);
        else ptx::tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// 2-D K-major operand [outer rows][inner elements], box {128 bytes, box_rows}, 128-byte swizzle.
bool make_operand_map(CUtensorMap* m, const void* base, bool fp8, uint64_t inner, uint64_t outer,
                      uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    const uint32_t esz = fp8 ? 1 : 2;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {inner * esz};
    cuuint32_t box[2] = {128u / esz, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                    const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int device_sms() {
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return sms;
}

// MXFP8 scales [rows][row_bytes] (bytes), box {16 bytes, box_rows}, no swizzle.
bool make_scale_map(CUtensorMap* m, const void* base, uint64_t row_bytes, uint64_t rows, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {row_bytes, rows};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {16u, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// A: [a_rows][a_inner], B: [b_rows][a_inner], both K-major.
template <int MODE, bool FP8, bool PAIR, bool NV4 = false>
moe_status launch_gemm(const void* A, uint64_t a_rows, const void* B, uint64_t b_rows, uint64_t inner,
                       GemmArgs a, cudaStream_t s) {
    using C = Cfg<FP8, PAIR, NV4>;
    CUtensorMap tmA, tmB, tmSA, tmSB;
    if (!make_operand_map(&tmA, A, FP8, inner, a_rows, BM)) return MOE_ERR_CUDA;
    if (!make_operand_map(&tmB, B, FP8, inner, b_rows, C::B_ROWS)) return MOE_ERR_CUDA;
    if (FP8) {
        if (!make_scale_map(&tmSA, a.a_scales, (uint64_t)a.sf_row_bytes, a_rows, BM)) return MOE_ERR_CUDA;
        if (!make_scale_map(&tmSB, a.b_scales, (uint64_t)a.sf_row_bytes, b_rows, BN)) return MOE_ERR_CUDA;
    } else {
        tmSA = tmA;
        tmSB = tmB;
    }
    if (MODE == MODE_WGRAD) a.m_tiles = a.M / C::TM;
    {
        // outputs are written in 32-byte row segments (at multiples of 32 elements) when every
        // output base and row pitch allows it
        auto al32 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 31u) == 0; };
        const bool pitch_ok = MODE == MODE_WGRAD ? (a.N % 32 == 0) : (a.ldo % 32 == 0);
        a.st32 = pitch_ok && al32(a.out) && al32(a.out2) && al32(a.ab) && al32(a.h_bf16) ? 1 : 0;
    }
    const size_t smem = smem_bytes_for<FP8, PAIR>(a.E);
    auto kern = grouped_gemm_kernel<MODE, FP8, PAIR, NV4>;
    // raise the kernel's dynamic shared-memory limit once per process and size (not a stream operation,
    // but keeping it out of repeated calls keeps captured launches free of other API calls)
    static int configured_smem = 0;
    if ((int)smem > configured_smem) {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return MOE_ERR_CUDA;
        configured_smem = (int)smem;
    }
    const int sms = device_sms();
    if (!PAIR) {
        kern<<<sms, C::THREADS, smem, s>>>(tmA, tmB, tmSA, tmSB, a);
        return moe_host::launch_status();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(sms / 2 * 2));
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, kern, tmA, tmB, tmSA, tmSB, a) != cudaSuccess) return MOE_ERR_CUDA;
    return moe_host::launch_status();
}

// bf16 tiles are computed by CTA pairs (M = 256) when the groups can fill them:
// row-grouped GEMMs when the mean group (R_cap / E, an upper bound) has at least
// 512 rows, and weight gradients whose M is a multiple of 256; otherwise, and
// for MXFP8, by single CTAs (M = 128).
template <int MODE>
moe_status launch_mode(bool fp8, const void* A, uint64_t a_rows, const void* B, uint64_t b_rows, uint64_t inner,
                       const GemmArgs& a, cudaStream_t s) {
    if (fp8) return launch_gemm<MODE, true, false>(A, a_rows, B, b_rows, inner, a, s);
    const bool pair = MODE == MODE_WGRAD ? (a.M % (2 * BM)) == 0 : (long long)a.R_cap >= 512LL * a.E;
    return pair ? launch_gemm<MODE, false, true>(A, a_rows, B, b_rows, inner, a, s)
                : launch_gemm<MODE, false, false>(A, a_rows, B, b_rows, inner, a, s);
}

moe_status check_common(moe_dtype dtype, const int32_t* group_offsets, int E, int H, int F, int R_cap) {
    if (dtype != MOE_BF16 && dtype != MOE_MXFP8) return MOE_ERR_INVALID_ARG;
    if (E < 1 || H < 128 || F < 128 || R_cap < 0 || !group_offsets) return MOE_ERR_INVALID_ARG;
    if ((H % 256) || (F % 128)) return MOE_ERR_UNSUPPORTED;
    // MXFP8: a row of scales of every contraction (H, F, 2F) is a whole number of 16-byte TMA boxes
    if (dtype == MOE_MXFP8 && ((H % 512) || (F % 512))) return MOE_ERR_UNSUPPORTED;
    if ((dtype == MOE_MXFP8 ? smem_bytes_for<true>(E) : smem_bytes_for<false>(E)) > 227 * 1024)
        return MOE_ERR_UNSUPPORTED;
    if ((long long)E * 2 * F > 0x7fffffffLL || (long long)E * H > 0x7fffffffLL) return MOE_ERR_UNSUPPORTED;
    if ((long long)R_cap * 2 * F > 0x7fffffffffffLL) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

bool al(const void* p, size_t a) { return p == nullptr || moe_host::aligned(p, a); }

}  // namespace
}  // namespace moe

using moe::GemmArgs;

extern "C" moe_status moe_grouped_gemm_up(const void* x_perm, const uint8_t* x_scales, const void* w13_packed,
                                          const uint8_t* w13_scales, moe_dtype dtype,
                                          const int32_t* group_offsets, int E, int H, int F, int R_cap, void* h,
                                          uint8_t* h_scales, void* ab_save, void* h_bf16_save,
                                          moe_stream_t stream) {
    using namespace moe;
    moe_status st = check_common(dtype, group_offsets, E, H, F, R_cap);
    if (st != MOE_OK) return st;
    if (R_cap == 0) return MOE_OK;
    const bool fp8 = dtype == MOE_MXFP8;
    if (!x_perm || !w13_packed || !h || (fp8 && (!x_scales || !w13_scales || !h_scales))) return MOE_ERR_INVALID_ARG;
    if (h_bf16_save && !fp8) return MOE_ERR_INVALID_ARG;
    if (!al(x_perm, 128) || !al(w13_packed, 128) || !al(h, 16) || !al(ab_save, 16) || !al(h_bf16_save, 16) ||
        (fp8 && (!al(x_scales, 16) || !al(w13_scales, 16))))
        return MOE_ERR_ALIGNMENT;
    GemmArgs a{};
    a.goff = group_offsets;
    a.E = E;
    a.Kdim = H;
    a.N = 2 * F;
    a.n_tiles = 2 * F / BN;
    a.R_cap = R_cap;
    a.out = h;
    a.ldo = F;
    a.out_scales = h_scales;
    a.a_scales = x_scales;
    a.b_scales = w13_scales;
    a.sf_row_bytes = H / 32;
    a.ab = static_cast<__nv_bfloat16*>(ab_save);
    a.h_bf16 = static_cast<__nv_bfloat16*>(h_bf16_save);
    return launch_mode<MODE_UP>(fp8, x_perm, (uint64_t)R_cap, w13_packed, (uint64_t)E * 2 * F, (uint64_t)H, a,
                                moe_host::as_stream(stream));
}

// Shared by the forward down projection (A = h, B = W2p, K = F) and the dx
// product of the backward (A = dab, B = W13t, K = 2F): y[r] = A[r] B[e]^T.
static moe_status grouped_down(const void* A, const uint8_t* a_scales, const void* B, const uint8_t* b_scales,
                               moe_dtype dtype, const int32_t* group_offsets, int E, int H, int Kc, int R_cap,
                               void* out, moe_stream_t stream) {
    using namespace moe;
    if (R_cap == 0) return MOE_OK;
    const bool fp8 = dtype == MOE_MXFP8;
    if (!A || !B || !out || (fp8 && (!a_scales || !b_scales))) return MOE_ERR_INVALID_ARG;
    if (!al(A, 128) || !al(B, 128) || !al(out, 16) || (fp8 && (!al(a_scales, 16) || !al(b_scales, 16))))
        return MOE_ERR_ALIGNMENT;
    GemmArgs a{};
    a.goff = group_offsets;
    a.E = E;
    a.Kdim = Kc;
    a.N = H;
    a.n_tiles = H / BN;
    a.R_cap = R_cap;
    a.out = out;
    a.ldo = H;
    a.a_scales = a_scales;
    a.b_scales = b_scales;
    a.sf_row_bytes = Kc / 32;
    return launch_mode<MODE_DOWN>(fp8, A, (uint64_t)R_cap, B, (uint64_t)E * H, (uint64_t)Kc, a,
                                  moe_host::as_stream(stream));
}

// NVFP4 operands are passed to the kernel as bytes (two elements each): a k-block is 128
// bytes = 256 elements, the contraction length and the tensor maps' inner extent are in bytes,
// and each 16-byte scale box per row covers one k-block (16 scales of 16 elements).
static moe_status check_nvfp4(const int32_t* group_offsets, int E, int H, int F, int R_cap) {
    using namespace moe;
    if (E < 1 || H < 256 || F < 256 || R_cap < 0 || !group_offsets) return MOE_ERR_INVALID_ARG;
    if ((H % 256) || (F % 256)) return MOE_ERR_UNSUPPORTED;
    if (smem_bytes_for<true>(E) > 227 * 1024) return MOE_ERR_UNSUPPORTED;
    if ((long long)E * 2 * F > 0x7fffffffLL || (long long)E * H > 0x7fffffffLL) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

extern "C" moe_status moe_grouped_gemm_up_nvfp4(const void* x_q, const uint8_t* x_scales, const float* x_amax,
                                                const void* w13_q, const uint8_t* w13_scales, const float* w13_amax,
                                                const int32_t* group_offsets, int E, int H, int F, int R_cap,
                                                void* h, float* h_amax, void* ab_save, moe_stream_t stream) {
    using namespace moe;
    moe_status st = check_nvfp4(group_offsets, E, H, F, R_cap);
    if (st != MOE_OK) return st;
    if (!x_q || !x_scales || !x_amax || !w13_q || !w13_scales || !w13_amax || !h || !h_amax)
        return MOE_ERR_INVALID_ARG;
    if (!al(x_q, 128) || !al(w13_q, 128) || !al(x_scales, 16) || !al(w13_scales, 16) || !al(h, 16) ||
        !al(ab_save, 16) || !al(x_amax, 4) || !al(w13_amax, 4) || !al(h_amax, 4))
        return MOE_ERR_ALIGNMENT;
    cudaStream_t s = moe_host::as_stream(stream);
    if (cudaMemsetAsync(h_amax, 0, sizeof(float), s) != cudaSuccess) return MOE_ERR_CUDA;
    if (R_cap == 0) return MOE_OK;
    GemmArgs a{};
    a.goff = group_offsets;
    a.E = E;
    a.Kdim = H / 2;
    a.N = 2 * F;
    a.n_tiles = 2 * F / BN;
    a.R_cap = R_cap;
    a.out = h;
    a.ldo = F;
    a.a_scales = x_scales;
    a.b_scales = w13_scales;
    a.sf_row_bytes = H / 16;
    a.ab = static_cast<__nv_bfloat16*>(ab_save);
    a.a_amax = x_amax;
    a.b_amax = w13_amax;
    a.out_amax = h_amax;
    return launch_gemm<MODE_UP, true, false, true>(x_q, (uint64_t)R_cap, w13_q, (uint64_t)E * 2 * F,
                                                    (uint64_t)(H / 2), a, s);
}

extern "C" moe_status moe_grouped_gemm_down_nvfp4(const void* h_q, const uint8_t* h_scales, const float* h_amax,
                                                  const void* w2_q, const uint8_t* w2_scales, const float* w2_amax,
                                                  const int32_t* group_offsets, int E, int H, int F, int R_cap,
                                                  void* y_perm, moe_stream_t stream) {
    using namespace moe;
    moe_status st = check_nvfp4(group_offsets, E, H, F, R_cap);
    if (st != MOE_OK) return st;
    if (R_cap == 0) return MOE_OK;
    if (!h_q || !h_scales || !h_amax || !w2_q || !w2_scales || !w2_amax || !y_perm) return MOE_ERR_INVALID_ARG;
    if (!al(h_q, 128) || !al(w2_q, 128) || !al(h_scales, 16) || !al(w2_scales, 16) || !al(y_perm, 16) ||
        !al(h_amax, 4) || !al(w2_amax, 4))
        return MOE_ERR_ALIGNMENT;
    GemmArgs a{};
    a.goff = group_offsets;
    a.E = E;
    a.Kdim = F / 2;
    a.N = H;
    a.n_tiles = H / BN;
    a.R_cap = R_cap;
    a.out = y_perm;
    a.ldo = H;
    a.a_scales = h_scales;
    a.b_scales = w2_scales;
    a.sf_row_bytes = F / 16;
    a.a_amax = h_amax;
    a.b_amax = w2_amax;
    return launch_gemm<MODE_DOWN, true, false, true>(h_q, (uint64_t)R_cap, w2_q, (uint64_t)E * H, (uint64_t)(F / 2),
                                                      a, moe_host::as_stream(stream));
}

extern "C" moe_status moe_grouped_gemm_down(const void* h, const uint8_t* h_scales, const void* w2_packed,
                                            const uint8_t* w2_scales, moe_dtype dtype,
                                            const int32_t* group_offsets, int E, int H, int F, int R_cap,
                                            void* y_perm, moe_stream_t stream) {
    moe_status st = moe::check_common(dtype, group_offsets, E, H, F, R_cap);
    if (st != MOE_OK) return st;
    return grouped_down(h, h_scales, w2_packed, w2_scales, dtype, group_offsets, E, H, F, R_cap, y_perm, stream);
}

extern "C" moe_status moe_grouped_swiglu_gemm(const void* x_perm, const uint8_t* x_scales,
                                              const void* w13_packed, const uint8_t* w13_scales,
                                              const void* w2_packed, const uint8_t* w2_scales, moe_dtype dtype,
                                              const int32_t* group_offsets, int E, int H, int F, int R_cap,
                                              void* h, uint8_t* h_scales, void* y_perm, moe_stream_t stream) {
    moe_status st = moe_grouped_gemm_up(x_perm, x_scales, w13_packed, w13_scales, dtype, group_offsets, E, H, F,
                                        R_cap, h, h_scales, nullptr, nullptr, stream);
    if (st != MOE_OK) return st;
    return moe_grouped_gemm_down(h, h_scales, w2_packed, w2_scales, dtype, group_offsets, E, H, F, R_cap, y_perm,
                                 stream);
}

extern "C" moe_status moe_grouped_swiglu_dgrad(const void* dy, const uint8_t* dy_scales, const void* w2_bwd,
                                               const uint8_t* w2_bwd_scales, const void* ab, moe_dtype dtype,
                                               const int32_t* group_offsets, int E, int H, int F, int R_cap,
                                               void* dab, uint8_t* dab_q, uint8_t* dab_scales,
                                               moe_stream_t stream) {
    using namespace moe;
    moe_status st = check_common(dtype, group_offsets, E, H, F, R_cap);
    if (st != MOE_OK) return st;
    if ((F % BN) != 0) return MOE_ERR_UNSUPPORTED;
    if (R_cap == 0) return MOE_OK;
    const bool fp8 = dtype == MOE_MXFP8;
    if (!dy || !w2_bwd || !ab || !dab || (fp8 && (!dy_scales || !w2_bwd_scales))) return MOE_ERR_INVALID_ARG;
    if ((dab_q == nullptr) != (dab_scales == nullptr)) return MOE_ERR_INVALID_ARG;
    if (!al(dy, 128) || !al(w2_bwd, 128) || !al(ab, 16) || !al(dab, 16) ||
        (fp8 && (!al(dy_scales, 16) || !al(w2_bwd_scales, 16))) || (dab_q && !al(dab_q, 32)))
        return MOE_ERR_ALIGNMENT;
    GemmArgs a{};
    a.goff = group_offsets;
    a.E = E;
    a.Kdim = H;
    a.N = F;
    a.n_tiles = F / BN;
    a.R_cap = R_cap;
    a.out = dab;
    a.ldo = 2 * F;
    a.a_scales = dy_scales;
    a.b_scales = w2_bwd_scales;
    a.sf_row_bytes = H / 32;
    a.ab = const_cast<__nv_bfloat16*>(static_cast<const __nv_bfloat16*>(ab));
    a.out_q = dab_q;
    a.out_scales = dab_scales;
    return launch_mode<MODE_DGRAD>(fp8, dy, (uint64_t)R_cap, w2_bwd, (uint64_t)E * F, (uint64_t)H, a,
                                   moe_host::as_stream(stream));
}

extern "C" moe_status moe_grouped_gemm_dx(const void* dab, const uint8_t* dab_scales, const void* w13t,
                                          const uint8_t* w13t_scales, moe_dtype dtype, const int32_t* group_offsets,
                                          int E, int H, int F, int R_cap, void* dx, moe_stream_t stream) {
    moe_status st = moe::check_common(dtype, group_offsets, E, H, F, R_cap);
    if (st != MOE_OK) return st;
    return grouped_down(dab, dab_scales, w13t, w13t_scales, dtype, group_offsets, E, H, 2 * F, R_cap, dx, stream);
}

extern "C" size_t moe_grouped_transpose_kpad(int R_cap, int E) {
    if (R_cap < 0 || E < 1) return 0;
    const size_t k = (size_t)128 * ((size_t)E + ((size_t)R_cap + 127) / 128 + 1);
    return (k + 511) / 512 * 512;  // MXFP8 scale rows of whole 16-byte TMA boxes
}

extern "C" moe_status moe_grouped_gemm_wgrad(const void* aT, const uint8_t* aT_scales, const void* bT,
                                             const uint8_t* bT_scales, moe_dtype dtype,
                                             const int32_t* group_offsets, int E, int M, int N, int R_cap,
                                             void* dw, void* dw2, moe_stream_t stream) {
    using namespace moe;
    if (dtype != MOE_BF16 && dtype != MOE_MXFP8) return MOE_ERR_INVALID_ARG;
    if (E < 1 || M < BM || N < BN || R_cap < 0 || !group_offsets) return MOE_ERR_INVALID_ARG;
    if ((M % BM) || (N % BN)) return MOE_ERR_UNSUPPORTED;
    if ((dtype == MOE_MXFP8 ? smem_bytes_for<true>(E) : smem_bytes_for<false>(E)) > 227 * 1024)
        return MOE_ERR_UNSUPPORTED;
    const size_t kpad = moe_grouped_transpose_kpad(R_cap, E);
    if (kpad > 0x7fffffffULL || (long long)E * M > 0x7fffffffLL) return MOE_ERR_UNSUPPORTED;
    const bool fp8 = dtype == MOE_MXFP8;
    if (!aT || !bT || !dw || (fp8 && (!aT_scales || !bT_scales))) return MOE_ERR_INVALID_ARG;
    if (!al(aT, 128) || !al(bT, 128) || !al(dw, 16) || !al(dw2, 16) ||
        (fp8 && (!al(aT_scales, 16) || !al(bT_scales, 16))))
        return MOE_ERR_ALIGNMENT;
    GemmArgs a{};
    a.goff = group_offsets;
    a.E = E;
    a.N = N;
    a.n_tiles = N / BN;
    a.M = M;
    a.m_tiles = M / BM;  // reset per tile height at launch
    a.out = dw;
    a.out2 = dw2;
    a.a_scales = aT_scales;
    a.b_scales = bT_scales;
    a.sf_row_bytes = (int)(kpad / 32);
    return launch_mode<MODE_WGRAD>(fp8, aT, (uint64_t)M, bT, (uint64_t)N, (uint64_t)kpad, a,
                                   moe_host::as_stream(stream));
}
