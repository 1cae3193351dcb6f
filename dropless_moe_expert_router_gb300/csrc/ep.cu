// ep.cu -- expert-parallel dispatch metadata: the local expert of each row a rank receives
// (moe_ep_recv_expert_ids).
//
// "Dropless MoE acceleration in JAX with NVIDIA Transformer Engine", section "Optimization 2:
// Expert parallelism to fuse Dispatch and Combine", and "Sparser MoE end-to-end", section
// "Remove work that has no selected route": only selected routes travel; a destination rank
// receives the rows of its own experts. Each source sends, from its expert-contiguous permuted
// order, the rows of the destination's experts; the destination receives them source by
// source and, within a source, expert by expert. With recv_counts[s][j] the rows from source s
// for local expert j, received row r belongs to local expert j of the segment (s, j) that
// holds it; rows past the last segment (spare receive capacity) get -1, which the local
// permute skips as an invalid route.
//
// Every block scans the segment counts into shared memory (64-bit inclusive ends), then labels
// a grid-stride share of the rows by a binary search over the ends. Counts are device data
// (the output of the count exchange), so the host never reads them.
#include "common.cuh"

namespace moe {
namespace {

constexpr int EP_THREADS = 256;
constexpr int EP_MAX_SEGMENTS = 4096;   // G * E_loc: e.g. 72 ranks x 32 local experts = 2304

__global__ void __launch_bounds__(EP_THREADS) ep_recv_ids_kernel(const int32_t* __restrict__ counts, int nseg,
                                                                 int E_loc, long long R_cap,
                                                                 int32_t* __restrict__ ids) {
    __shared__ long long ends[EP_MAX_SEGMENTS];
    __shared__ long long part[EP_THREADS];
    const int tid = threadIdx.x;
    const int per = (nseg + EP_THREADS - 1) / EP_THREADS;
    const int b0 = min(nseg, tid * per), b1 = min(nseg, b0 + per);
    long long local = 0;
    for (int i = b0; i < b1; i++) {
        const int c = __ldg(counts + i);
        if (c < 0) raise_device_error(MOE_DEVERR_BAD_ID);     // read as 0
        local += c > 0 ? c : 0;
    }
    part[tid] = local;
    __syncthreads();
    for (int off = 1; off < EP_THREADS; off <<= 1) {          // inclusive scan of the chunk sums
        const long long v = tid >= off ? part[tid - off] : 0;
        __syncthreads();
        part[tid] += v;
        __syncthreads();
    }
    long long run = part[tid] - local;
    for (int i = b0; i < b1; i++) {
        const int c = __ldg(counts + i);
        run += c > 0 ? c : 0;
        ends[i] = run;
    }
    __syncthreads();
    const long long total = ends[nseg - 1];
    for (long long r = (long long)blockIdx.x * EP_THREADS + tid; r < R_cap; r += (long long)gridDim.x * EP_THREADS) {
        int id = -1;
        if (r < total) {
            int lo = 0, hi = nseg - 1;                          // first segment whose end exceeds r
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (ends[mid] > r) hi = mid;
                else lo = mid + 1;
            }
            id = lo % E_loc;
        }
        ids[r] = id;
    }
}

}  // namespace
}  // namespace moe

extern "C" moe_status moe_ep_recv_expert_ids(const int32_t* recv_counts, int G, int E_loc, long long R_cap,
                                             int32_t* ids, moe_stream_t stream) {
    using namespace moe;
    if (G < 1 || E_loc < 1 || R_cap < 0) return MOE_ERR_INVALID_ARG;
    if ((long long)G * E_loc > EP_MAX_SEGMENTS) return MOE_ERR_UNSUPPORTED;
    if (R_cap == 0) return MOE_OK;
    if (!recv_counts || !ids) return MOE_ERR_INVALID_ARG;
    if (!moe_host::aligned(recv_counts, 4) || !moe_host::aligned(ids, 4)) return MOE_ERR_ALIGNMENT;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    long long blocks = (R_cap + EP_THREADS - 1) / EP_THREADS;
    if (blocks > 2LL * sms) blocks = 2LL * sms;
    ep_recv_ids_kernel<<<(int)blocks, EP_THREADS, 0, moe_host::as_stream(stream)>>>(recv_counts, G * E_loc, E_loc,
                                                                                   R_cap, ids);
    return moe_host::launch_status();
}
