// gemm.cu -- persistent ragged grouped GEMM on tcgen05 tensor cores, with the
// SwiGLU expert MLP built from two launches, plus one-time weight packing.
//
// "Dropless MoE acceleration in JAX with NVIDIA Transformer Engine", section
// "Optimization 1: Grouped GEMM": one kernel covers every expert with its actual
// token count and computes only valid regions; the token counts stay on the
// device (no device-to-host copy, so the call can live in a CUDA graph); on
// Blackwell the expert matmuls can use MXFP8 block scaling. The same page's
// MoE-layer figure: the grouped MLP is two grouped GEMMs on variable-length
// groups.
//
// Design (one CTA per SM, persistent, warp-specialised; 192 threads):
//   warp 0     TMA producer: A tile [128 rows x 128 B] and B tile [256 rows x 128 B]
//              per k-block into a 4-stage shared-memory ring (128-byte swizzle);
//              MXFP8 adds the per-row E8M0 scale words of the k-block (cp.async
//              straight into the layout tcgen05.cp expects).
//   warp 1     allocates TMEM and issues tcgen05.mma (M=128, N=256) from one
//              lane; each k-block's commit frees its ring stage, each tile's
//              commit hands the accumulator to the epilogue.
//   warps 2-5  epilogue: tcgen05.ld of the fp32 accumulator (each warp owns the
//              32 TMEM lanes of its quarter), SwiGLU (GEMM1) or plain (GEMM2),
//              bf16 (or MXFP8) rows stored for the rows inside the group only.
// Tiles are scheduled on the device: every CTA reads group_offsets, counts
// ceil(m_e / 128) row tiles per expert and walks the tile list
// (expert-major, then output column tile, then row tile, so one weight tile is
// consumed by all row tiles of its expert while it is hot in L2) with a static
// stride of gridDim.x. A row tile that runs past its group reads the next
// group's rows (or TMA zero fill past R_cap); those accumulator rows are
// simply never stored. No padding, no dropping.
//
// BF16: kind::f16, two TMEM accumulators (2 x 256 columns) so the epilogue of
// tile i overlaps the main loop of tile i+1.
// MXFP8: kind::mxf8f6f4.block_scale (E4M3 x E4M3, UE8M0 scale per 32
// elements); one accumulator plus per-stage scale-factor columns in TMEM.
#include "common.cuh"
#include "sm100_ptx.cuh"

#include <cudaTypedefs.h>

namespace moe {
namespace {

constexpr int BM = 128;          // rows per tile (MMA M)
constexpr int BN = 256;          // output columns per tile (MMA N)
constexpr int STAGES = 4;        // shared-memory ring depth
constexpr int NUM_THREADS = 192;
constexpr int TMEM_COLS = 512;

template <bool FP8>
struct Cfg {
    static constexpr int BK = FP8 ? 128 : 64;       // elements per k-block (128 bytes per row)
    static constexpr int UMMA_K = FP8 ? 32 : 16;    // elements per MMA instruction
    static constexpr int KSTEPS = BK / UMMA_K;      // MMAs per k-block (4)
    static constexpr int A_BYTES = BM * 128;
    static constexpr int B_BYTES = BN * 128;
    static constexpr int SFA_BYTES = FP8 ? BM * 4 : 0;   // one 32-bit word (4 scales) per row
    static constexpr int SFB_BYTES = FP8 ? BN * 4 : 0;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
    static constexpr int ACC_STAGES = FP8 ? 1 : 2;
    static constexpr int SF_COLS = 12;              // TMEM columns of one stage's scales (4 A + 8 B)
};

struct GemmArgs {
    const int* goff;             // [E+1] group offsets (device)
    int E;
    int Kdim;                    // contraction length
    int N;                       // B rows per expert
    int n_tiles;                 // N / BN
    int R_cap;                   // rows of A
    void* out;                   // [R_cap, ldo] bf16, or E4M3 codes (MXFP8 h)
    int ldo;
    uint8_t* out_scales;         // [R_cap, ldo/32] (MXFP8 h only)
    const uint8_t* a_scales;     // [R_cap, Kdim/32] (MXFP8)
    const uint8_t* b_scales;     // [E*N, Kdim/32] (MXFP8)
};

template <bool FP8>
constexpr size_t smem_bytes_for(int E) {
    return 1024 /* alignment slack */ + (size_t)STAGES * Cfg<FP8>::STAGE_BYTES + 256 /* barriers, flags */ +
           (size_t)NUM_THREADS * 4 + (size_t)2 * (E + 1) * 4;
}

struct TileInfo {
    int e, m, n, row0, rows;
};

__device__ __forceinline__ TileInfo decode_tile(int tile, const int* s_mtp, const int* s_goff, int E, int n_tiles) {
    const int q = tile / n_tiles;
    int lo = 0, hi = E - 1;  // last e with s_mtp[e] <= q (never an empty expert)
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (s_mtp[mid] <= q) lo = mid;
        else hi = mid - 1;
    }
    const int mt = s_mtp[lo + 1] - s_mtp[lo];
    const int local = tile - s_mtp[lo] * n_tiles;
    TileInfo t;
    t.e = lo;
    t.n = local / mt;
    t.m = local - t.n * mt;
    t.row0 = s_goff[lo] + t.m * BM;
    t.rows = min(BM, s_goff[lo + 1] - t.row0);
    return t;
}

__device__ __forceinline__ float silu_f(float a) { return __fdividef(a, 1.0f + __expf(-a)); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src, bool valid) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(valid ? 4 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(ptx::smem_addr(bar)) : "memory");
}

template <bool SWIGLU, bool FP8>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const GemmArgs p) {
    using C = Cfg<FP8>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* ring = smem;  // STAGES x [A | B | SFA | SFB]
    uint64_t* full = reinterpret_cast<uint64_t*>(ring + (size_t)STAGES * C::STAGE_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* done = tempty + 2;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(done + 1);
    volatile uint32_t* s_abort = s_tmem + 1;
    int* s_part = reinterpret_cast<int*>(smem + (size_t)STAGES * C::STAGE_BYTES + 256);
    int* s_goff = s_part + NUM_THREADS;
    int* s_mtp = s_goff + (p.E + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int E = p.E;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; s++) {
            ptx::mbar_init(&full[s], FP8 ? 1 + 32 : 1);
            ptx::mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; a++) {
            ptx::mbar_init(&tfull[a], 1);
            ptx::mbar_init(&tempty[a], 128);
        }
        ptx::mbar_init(done, 1);
        *s_abort = 0u;
        ptx::fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tmap(&tmA);
        ptx::prefetch_tmap(&tmB);
    }
    if (warp == 1) {
        ptx::tmem_alloc(s_tmem, TMEM_COLS);
        ptx::tmem_relinquish();
    }
    // group table: offsets, and the exclusive scan of row tiles per expert
    for (int e = threadIdx.x; e <= E; e += NUM_THREADS) s_goff[e] = __ldg(p.goff + e);
    __syncthreads();
    {
        const int per = (E + NUM_THREADS - 1) / NUM_THREADS;
        const int b0 = threadIdx.x * per;
        int local = 0;
        for (int j = 0; j < per; j++) {
            int e = b0 + j;
            if (e < E) local += (s_goff[e + 1] - s_goff[e] + BM - 1) / BM;
        }
        s_part[threadIdx.x] = local;
        __syncthreads();
        if (threadIdx.x == 0) {
            int run = 0;
            for (int i = 0; i < NUM_THREADS; i++) {
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
                run += (s_goff[e + 1] - s_goff[e] + BM - 1) / BM;
            }
        }
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();

    const uint32_t tmem = *s_tmem;
    const int total_tiles = s_mtp[E] * p.n_tiles;
    const int num_kb = p.Kdim / C::BK;
    const int kb_bytes_sf = p.Kdim / 32;  // scale bytes per row

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        int stage = 0;
        uint32_t phase = 0;
        int issued = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
            const TileInfo ti = decode_tile(tile, s_mtp, s_goff, E, p.n_tiles);
            const int a_row = ti.row0;
            const int b_row = ti.e * p.N + ti.n * BN;
            for (int kb = 0; kb < num_kb; kb++) {
                if (!ptx::wait_parity(&empty[stage], phase ^ 1u, s_abort)) { ok = false; break; }
                uint8_t* sa = ring + (size_t)stage * C::STAGE_BYTES;
                uint8_t* sb = sa + C::A_BYTES;
                if (lane == 0) {
                    ptx::mbar_arrive_expect_tx(&full[stage], C::A_BYTES + C::B_BYTES);
                    ptx::tma_load_2d(sa, &tmA, &full[stage], kb * C::BK, a_row);
                    ptx::tma_load_2d(sb, &tmB, &full[stage], kb * C::BK, b_row);
                }
                if constexpr (FP8) {
                    // scale words of this k-block, transposed for tcgen05.cp .32x128b:
                    // word (lane*4 + j) of a 512-byte chunk holds row 32*j + lane of the chunk
                    const uint32_t sfa = ptx::smem_addr(sb + C::B_BYTES);
                    const uint32_t sfb = sfa + C::SFA_BYTES;
#pragma unroll
                    for (int j = 0; j < 4; j++) {
                        const int r = a_row + 32 * j + lane;
                        const bool v = r < p.R_cap;
                        cp_async_4(sfa + (lane * 4 + j) * 4,
                                   p.a_scales + (size_t)(v ? r : 0) * kb_bytes_sf + kb * 4, v);
                    }
#pragma unroll
                    for (int c = 0; c < 2; c++)
#pragma unroll
                        for (int j = 0; j < 4; j++) {
                            const int r = b_row + 128 * c + 32 * j + lane;
                            cp_async_4(sfb + c * 512 + (lane * 4 + j) * 4,
                                       p.b_scales + (size_t)r * kb_bytes_sf + kb * 4, true);
                        }
                    cp_async_arrive_noinc(&full[stage]);
                }
                __syncwarp();
                issued++;
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
        }
        if (!ok) {
            // give the loads already issued a bounded chance to land before the CTA exits
            for (int i = 0; i < STAGES && i < issued; i++) {
                if (--stage < 0) { stage = STAGES - 1; phase ^= 1u; }
                volatile uint32_t never = 0u;
                ptx::wait_parity(&full[stage], phase, &never, 100000000ull);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        int stage = 0;
        uint32_t phase = 0;
        int acc = 0;
        uint32_t acc_phase = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
            if (!ptx::wait_parity(&tempty[acc], acc_phase ^ 1u, s_abort)) { ok = false; break; }
            ptx::tc_fence_after();
            const uint32_t d_tmem = tmem + (uint32_t)(acc * BN);
            for (int kb = 0; kb < num_kb; kb++) {
                if (!ptx::wait_parity(&full[stage], phase, s_abort)) { ok = false; break; }
                ptx::tc_fence_after();
                if (lane == 0) {
                    uint8_t* sa = ring + (size_t)stage * C::STAGE_BYTES;
                    uint8_t* sb = sa + C::A_BYTES;
                    const uint32_t a0 = ptx::smem_addr(sa), b0 = ptx::smem_addr(sb);
                    if constexpr (FP8) {
                        ptx::fence_proxy_async_smem();
                        const uint32_t sf_t = tmem + (uint32_t)(BN + stage * C::SF_COLS);
                        const uint32_t sfa_s = ptx::smem_addr(sb + C::B_BYTES);
                        ptx::tc_cp_32x128b_warpx4(sf_t, ptx::sdesc_plain(sfa_s));
                        ptx::tc_cp_32x128b_warpx4(sf_t + 4, ptx::sdesc_plain(sfa_s + C::SFA_BYTES));
                        ptx::tc_cp_32x128b_warpx4(sf_t + 8, ptx::sdesc_plain(sfa_s + C::SFA_BYTES + 512));
#pragma unroll
                        for (int k = 0; k < C::KSTEPS; k++)
                            ptx::mma_mxf8(d_tmem, ptx::sdesc_k_sw128(a0 + k * 32), ptx::sdesc_k_sw128(b0 + k * 32),
                                          ptx::idesc_mxf8(BM, BN, k, k), sf_t, sf_t + 4, (kb | k) != 0);
                    } else {
#pragma unroll
                        for (int k = 0; k < C::KSTEPS; k++)
                            ptx::mma_f16(d_tmem, ptx::sdesc_k_sw128(a0 + k * 32), ptx::sdesc_k_sw128(b0 + k * 32),
                                         ptx::idesc_bf16(BM, BN), (kb | k) != 0);
                    }
                    ptx::tc_commit(&empty[stage]);
                }
                __syncwarp();
                if (++stage == STAGES) { stage = 0; phase ^= 1u; }
            }
            if (!ok) break;
            if (lane == 0) ptx::tc_commit(&tfull[acc]);
            __syncwarp();
            if (++acc == C::ACC_STAGES) { acc = 0; acc_phase ^= 1u; }
        }
        // make sure every MMA issued by this CTA has completed before TMEM is released
        if (lane == 0) ptx::tc_commit(done);
        __syncwarp();
        volatile uint32_t never = 0u;
        ptx::wait_parity(done, 0u, &never, 100000000ull);
    } else {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                 // TMEM lane quarter of this warp
        const int rit = q * 32 + lane;          // row within the tile
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
            const TileInfo ti = decode_tile(tile, s_mtp, s_goff, E, p.n_tiles);
            if (!ptx::wait_parity(&tfull[acc], acc_phase, s_abort)) break;
            ptx::tc_fence_after();
            const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
            const bool valid = rit < ti.rows;
            const long long r = (long long)ti.row0 + rit;
            if constexpr (SWIGLU) {
                const int col0 = ti.n * (BN / 2);
#pragma unroll 1
                for (int c = 0; c < BN / 64; c++) {
                    uint32_t g[32], u[32];
                    ptx::tmem_ld_x32(tbase + 32 * c, g);
                    ptx::tmem_ld_x32(tbase + BN / 2 + 32 * c, u);
                    ptx::tmem_wait_ld();
                    float hv[32];
#pragma unroll
                    for (int i = 0; i < 32; i++) hv[i] = silu_f(__uint_as_float(g[i])) * __uint_as_float(u[i]);
                    if constexpr (FP8) {
                        float amax = 0.0f;
#pragma unroll
                        for (int i = 0; i < 32; i++) amax = fmaxf(amax, fabsf(hv[i]));
                        const int sbyte = e8m0_scale_byte(amax);
                        const float inv = e8m0_inv_scale(sbyte);
                        uint32_t w[8];
#pragma unroll
                        for (int i = 0; i < 8; i++)
                            w[i] = (uint32_t)f32x2_to_e4m3x2(hv[4 * i] * inv, hv[4 * i + 1] * inv) |
                                   ((uint32_t)f32x2_to_e4m3x2(hv[4 * i + 2] * inv, hv[4 * i + 3] * inv) << 16);
                        if (valid) {
                            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(p.out) + r * p.ldo + col0 + 32 * c);
                            dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                            dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                            p.out_scales[r * (p.ldo / 32) + (col0 / 32) + c] = (uint8_t)sbyte;
                        }
                    } else {
                        uint32_t w[16];
#pragma unroll
                        for (int i = 0; i < 16; i++) w[i] = pack_bf16x2(hv[2 * i], hv[2 * i + 1]);
                        if (valid) {
                            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + r * p.ldo +
                                                                  col0 + 32 * c);
#pragma unroll
                            for (int i = 0; i < 4; i++)
                                dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                        }
                    }
                }
            } else {
                const int col0 = ti.n * BN;
#pragma unroll 1
                for (int c = 0; c < BN / 32; c++) {
                    uint32_t v[32];
                    ptx::tmem_ld_x32(tbase + 32 * c, v);
                    ptx::tmem_wait_ld();
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; i++) w[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
                    if (valid) {
                        uint4* dst =
                            reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + r * p.ldo + col0 + 32 * c);
#pragma unroll
                        for (int i = 0; i < 4; i++) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
                    }
                }
            }
            ptx::tc_fence_before();
            ptx::mbar_arrive(&tempty[acc]);
            if (++acc == C::ACC_STAGES) { acc = 0; acc_phase ^= 1u; }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ---------------------------------------------------------------- weight packing
// W1, W3 [E][H][F] -> W13 [E][2F][H] with rows grouped per 256-row tile:
// rows [256 j, 256 j + 128) = W1^T rows f in [128 j, 128 j + 128), the next 128 = W3^T.
// W2 [E][F][H] -> W2p [E][H][F] (= W2^T per expert).
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

// MXFP8 packing: transpose as above and quantise each packed row along its
// contraction dimension (the source's rows) in blocks of 32. Block (32 source
// rows x 32 source columns); thread x owns one source column.
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

template <bool SWIGLU, bool FP8>
moe_status launch_gemm(const void* A, const void* B, const GemmArgs& a, cudaStream_t s) {
    CUtensorMap tmA, tmB;
    if (!make_operand_map(&tmA, A, FP8, (uint64_t)a.Kdim, (uint64_t)a.R_cap, BM)) return MOE_ERR_CUDA;
    if (!make_operand_map(&tmB, B, FP8, (uint64_t)a.Kdim, (uint64_t)a.E * a.N, BN)) return MOE_ERR_CUDA;
    const size_t smem = smem_bytes_for<FP8>(a.E);
    if (cudaFuncSetAttribute(grouped_gemm_kernel<SWIGLU, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
        return MOE_ERR_CUDA;
    grouped_gemm_kernel<SWIGLU, FP8><<<device_sms(), NUM_THREADS, smem, s>>>(tmA, tmB, a);
    return moe_host::launch_status();
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

static moe_status check_gemm_common(moe_dtype dtype, const int32_t* group_offsets, int E, int H, int F,
                                    int R_cap) {
    using namespace moe;
    if (dtype != MOE_BF16 && dtype != MOE_MXFP8) return MOE_ERR_INVALID_ARG;
    if (E < 1 || H < 128 || F < 128 || R_cap < 0 || !group_offsets) return MOE_ERR_INVALID_ARG;
    if ((H % 256) || (F % 128)) return MOE_ERR_UNSUPPORTED;
    if (smem_bytes_for<true>(E) > 227 * 1024) return MOE_ERR_UNSUPPORTED;
    if ((long long)E * 2 * F > 0x7fffffffLL || (long long)E * H > 0x7fffffffLL) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

extern "C" moe_status moe_grouped_gemm_up(const void* x_perm, const uint8_t* x_scales, const void* w13_packed,
                                          const uint8_t* w13_scales, moe_dtype dtype,
                                          const int32_t* group_offsets, int E, int H, int F, int R_cap, void* h,
                                          uint8_t* h_scales, moe_stream_t stream) {
    using namespace moe;
    moe_status st = check_gemm_common(dtype, group_offsets, E, H, F, R_cap);
    if (st != MOE_OK) return st;
    if (R_cap == 0) return MOE_OK;
    const bool fp8 = dtype == MOE_MXFP8;
    if (!x_perm || !w13_packed || !h || (fp8 && (!x_scales || !w13_scales || !h_scales)))
        return MOE_ERR_INVALID_ARG;
    if (!moe_host::aligned(x_perm, 128) || !moe_host::aligned(w13_packed, 128) || !moe_host::aligned(h, 16) ||
        (fp8 && (!moe_host::aligned(x_scales, 4) || !moe_host::aligned(w13_scales, 4))))
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
    cudaStream_t s = moe_host::as_stream(stream);
    return fp8 ? launch_gemm<true, true>(x_perm, w13_packed, a, s)
               : launch_gemm<true, false>(x_perm, w13_packed, a, s);
}

extern "C" moe_status moe_grouped_gemm_down(const void* h, const uint8_t* h_scales, const void* w2_packed,
                                            const uint8_t* w2_scales, moe_dtype dtype,
                                            const int32_t* group_offsets, int E, int H, int F, int R_cap,
                                            void* y_perm, moe_stream_t stream) {
    using namespace moe;
    moe_status st = check_gemm_common(dtype, group_offsets, E, H, F, R_cap);
    if (st != MOE_OK) return st;
    if ((H % BN) != 0) return MOE_ERR_UNSUPPORTED;
    if (R_cap == 0) return MOE_OK;
    const bool fp8 = dtype == MOE_MXFP8;
    if (!h || !w2_packed || !y_perm || (fp8 && (!h_scales || !w2_scales))) return MOE_ERR_INVALID_ARG;
    if (!moe_host::aligned(h, 128) || !moe_host::aligned(w2_packed, 128) || !moe_host::aligned(y_perm, 16) ||
        (fp8 && (!moe_host::aligned(h_scales, 4) || !moe_host::aligned(w2_scales, 4))))
        return MOE_ERR_ALIGNMENT;
    GemmArgs a{};
    a.goff = group_offsets;
    a.E = E;
    a.Kdim = F;
    a.N = H;
    a.n_tiles = H / BN;
    a.R_cap = R_cap;
    a.out = y_perm;
    a.ldo = H;
    a.a_scales = h_scales;
    a.b_scales = w2_scales;
    cudaStream_t s = moe_host::as_stream(stream);
    return fp8 ? launch_gemm<false, true>(h, w2_packed, a, s) : launch_gemm<false, false>(h, w2_packed, a, s);
}

extern "C" moe_status moe_grouped_swiglu_gemm(const void* x_perm, const uint8_t* x_scales,
                                              const void* w13_packed, const uint8_t* w13_scales,
                                              const void* w2_packed, const uint8_t* w2_scales, moe_dtype dtype,
                                              const int32_t* group_offsets, int E, int H, int F, int R_cap,
                                              void* h, uint8_t* h_scales, void* y_perm, moe_stream_t stream) {
    moe_status st = moe_grouped_gemm_up(x_perm, x_scales, w13_packed, w13_scales, dtype, group_offsets, E, H, F,
                                        R_cap, h, h_scales, stream);
    if (st != MOE_OK) return st;
    return moe_grouped_gemm_down(h, h_scales, w2_packed, w2_scales, dtype, group_offsets, E, H, F, R_cap, y_perm,
                                 stream);
}
