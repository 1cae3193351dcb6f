/*
 * moe_gb300.h -- C ABI of the single-GPU dropless Mixture-of-Experts layer
 * hot path for NVIDIA GB300 (sm_103a).
 *
 * The path: router top-K -> permute (dispatch into expert-contiguous order,
 * optionally quantising to MXFP8 on the way) -> grouped SwiGLU expert MLP
 * (two ragged grouped GEMMs, BF16 or MXFP8) -> probability-weighted
 * unpermute/combine back to token order; plus the grouped backward GEMMs.
 *
 * Sources (cited by page title and section):
 *   [SPARSER] "Sparser MoE end-to-end" (harryzhou2000 blog)
 *   [TEJAX]   "Dropless MoE acceleration in JAX with NVIDIA Transformer Engine"
 *             (news.bpdata.com)
 *   [CLARITY] "NVIDIA's unoptimized DeepSeek-V3 baseline spends 84% of kernel
 *             time moving tokens between GPUs" (theclarity.today)
 *
 * Conventions shared by every entry point:
 *  - Ownership: the caller allocates every buffer (device memory unless stated)
 *    and keeps it alive until the enqueued work has finished. The library never
 *    allocates, never synchronises and never copies device->host in the calls
 *    below, except moe_get_device_errors. Group sizes stay on the device
 *    ([TEJAX] "Optimization 1: Grouped GEMM": shapes must not need the CPU, so
 *    CUDA graphs stay usable); every call is safe to capture in a CUDA graph.
 *  - Streams: work is enqueued on `stream` (a cudaStream_t; NULL = legacy
 *    default stream) and nowhere else.
 *  - Layouts are row-major. bf16 tensors are passed as raw 16-bit payloads.
 *    Device pointers must be 16-byte aligned; operands of the grouped GEMMs
 *    (x_perm, h, packed weights and their scales) must be 128-byte aligned.
 *  - Capacity: permuted buffers have R_cap = T*K rows. Only the first
 *    R = group_offsets[E] rows are written or read; the rest are unspecified.
 *  - Errors: argument checks are synchronous and return a status without
 *    enqueuing anything. A failed launch returns MOE_ERR_CUDA. Conditions found
 *    on the device never trap: they set bits in a device error word that
 *    moe_get_device_errors reads.
 *  - T = 0 (no tokens) is legal and enqueues nothing.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *moe_stream_t;

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* bad shape, null pointer or flag combination */
    MOE_ERR_UNSUPPORTED = 2,   /* legal but not implemented (e.g. H % 128 != 0 for the GEMM) */
    MOE_ERR_WORKSPACE = 3,     /* workspace missing or too small */
    MOE_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
    MOE_ERR_ALIGNMENT = 5,     /* a pointer is not aligned as required */
    MOE_ERR_DEVICE = 6         /* the device error word is non-zero (moe_get_device_errors) */
} moe_status;

typedef enum {
    MOE_I16 = 0,   /* int16 expert ids (E <= 32767) */
    MOE_I32 = 1,   /* int32 expert ids */
    MOE_BF16 = 2,  /* bfloat16 operands */
    MOE_MXFP8 = 3  /* E4M3 payloads with one E8M0 scale byte per 32 elements */
} moe_dtype;

/* flags */
#define MOE_ROUTE_RENORM 1u        /* probs normalised over the K selected experts */
#define MOE_PERMUTE_FUSE_MXFP8 2u  /* permute writes MXFP8 rows instead of bf16 rows */
#define MOE_QUANT_COLWISE 4u       /* group-aware 32x1 blocks along rows (wgrad operands) */

/* device error bits */
#define MOE_DEVERR_BAD_ID 1u       /* an expert id outside [-1, E) was seen (treated as invalid) */
#define MOE_DEVERR_TIMEOUT 2u      /* a bounded wait inside a kernel gave up */

/* ------------------------------------------------------------------------
 * Router top-K ([SPARSER] "Preserve a compact route": radix/threshold
 * selection with bounded histogram passes for large E and K, a separate fast
 * path for small top-k, and routes carried as a dense [T, K] id list rather
 * than a [T, E] map; [TEJAX] "Optimization 2": router kernels assign tokens
 * before dispatch).
 *
 * logits [T, E] fp32. For every row: the K experts with the largest logits,
 * ties to the lower expert index (-0 and +0 are equal), written to ids[T, K]
 * in that order (int16 or int32 per id_dtype); probs[T, K] fp32 is the softmax
 * over all E logits taken at the selected expert, or, with MOE_ROUTE_RENORM,
 * the softmax over the K selected logits. The router never emits -1.
 * Requires 1 <= K <= E, K <= 128, E <= 8192, no NaN
 * logits (NaN rows give unspecified ids). Small E (<= 256) and K (<= 16) use a
 * warp-per-row arg-max path; E % 4 == 0, E <= 2304 with 16-byte aligned logits
 * use a warp-per-row threshold select; the rest use the radix-select path (a
 * CTA per row). All paths give the same ids and the same probs up to fp32
 * rounding order.
 * ------------------------------------------------------------------------ */
moe_status moe_route_topk(const float *logits, int T, int E, int K,
                          void *ids, moe_dtype id_dtype, float *probs,
                          unsigned flags, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Router backward ([SPARSER] "The workload changes the bottleneck" names a
 * router backward among the kernels, "Preserve a compact route" a backward
 * beside the forward; neither defines it). The gradient of moe_route_topk's
 * probs with respect to the logits, the selection held fixed (top-K is
 * piecewise constant): for row t, S = its valid ids (0 <= id < E; others
 * skipped), g[k] = dprobs[t,k], G_e = sum of g[k] over the k with ids[t,k] = e,
 * p the softmax over all E (with MOE_ROUTE_RENORM: over S, and 0 off S),
 * s = sum over valid k of g[k] p_{ids[t,k]}:
 *   dlogits[t,e] = p_e (G_e - s)       (0 off S with MOE_ROUTE_RENORM).
 * logits [T, E] fp32 (the forward's input), ids [T, K] int16/int32, dprobs
 * [T, K] fp32 in; dlogits [T, E] fp32 out (every element written). Same size
 * limits as moe_route_topk (K <= 128); fp32 arithmetic, within 1e-6 absolute
 * of the exact value for logits of the workloads' scale.
 * ------------------------------------------------------------------------ */
moe_status moe_route_topk_backward(const float *logits, const void *ids, moe_dtype id_dtype,
                                   const float *dprobs, int T, int E, int K,
                                   unsigned flags, float *dlogits, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Sigmoid-score routing with a per-expert selection bias ([SPARSER] "The
 * workload changes the bottleneck": the router's score transformation and
 * top-k selection; "Preserve a compact route": bias statistics carried with
 * compact routes; the pages define neither, the DeepSeek-style reading is
 * taken). For every row t and expert e:
 *   s_e = 1 / (1 + exp(-logits[t,e]))      (fp32)
 *   key_e = s_e + expert_bias[e]            (fp32; bias NULL means 0)
 * ids[t, 0..K) = the K largest keys, in descending order, ties to the lower
 * expert index; probs[t,k] = s at ids[t,k], or with MOE_ROUTE_RENORM that
 * score divided by the sum of the K selected scores. The bias steers only the
 * selection; its statistics (valid routes per expert) are the group_sizes that
 * moe_permute writes. logits [T, E] fp32, expert_bias [E] fp32 (optional) in;
 * ids [T, K] int16/int32 and probs [T, K] fp32 out. One warp per row, keys in
 * registers. Requires 1 <= K <= E, E <= 1024 and K <= 64 (else
 * MOE_ERR_UNSUPPORTED), no NaN logits or biases, finite biases. The score is
 * CUDA's fp32 logistic (within 2 ulp of the correctly rounded value), so two
 * keys within a few ulp of each other may be ordered either way.
 * ------------------------------------------------------------------------ */
moe_status moe_route_sigmoid_topk(const float *logits, const float *expert_bias, int T, int E,
                                  int K, void *ids, moe_dtype id_dtype, float *probs,
                                  unsigned flags, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Backward of moe_route_sigmoid_topk's probs with respect to the logits, the
 * selection held fixed. Row t: S = its distinct valid ids, G_e = sum of
 * dprobs[t,k] over the k with ids[t,k] = e, s_e the score above, Z = sum over
 * S of s_e, c = sum over S of G_e s_e / Z:
 *   dlogits[t,e] = G_e s_e (1 - s_e)                  (e in S)
 *   dlogits[t,e] = s_e (1 - s_e) (G_e - c) / Z        (e in S, MOE_ROUTE_RENORM)
 * and 0 off S (the bias has no gradient path). logits [T, E], ids [T, K],
 * dprobs [T, K] in; dlogits [T, E] fp32 out (every element written).
 * Requires 1 <= K <= min(E, 128).
 * ------------------------------------------------------------------------ */
moe_status moe_route_sigmoid_topk_backward(const float *logits, const void *ids, moe_dtype id_dtype,
                                           const float *dprobs, int T, int E, int K,
                                           unsigned flags, float *dlogits, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Permute / dispatch ([TEJAX] "Dropless vs capacity-based MoE": every routed
 * token is processed, nothing dropped or padded; MoE-layer figure: tokens are
 * grouped per expert and combine restores token order; [SPARSER] "Remove work
 * that has no selected route": local processing visits only the selected
 * slots, found by a warp ballot; invalid routes (-1) are preserved).
 *
 * A device-side counting sort of the T*K routes by expert:
 *   group_sizes[E]      number of valid routes per expert (int32)
 *   group_offsets[E+1]  exclusive scan of group_sizes; group_offsets[E] = R
 *   row_map[T, K]       destination row of route (t, k), -1 if invalid (int32)
 *   perm_src[R_cap]     source token of each destination row (int32; rows >= R untouched)
 *   x_perm[R_cap, H]    x_perm[row_map[t,k]] = x[t] bit for bit (bf16), or with
 *                       MOE_PERMUTE_FUSE_MXFP8: E4M3 payload bytes, with
 *   x_perm_scales[R_cap, H/32]  the row-wise 1x32 E8M0 scale bytes (else NULL).
 * Route (t, k) is valid iff 0 <= ids[t,k] < E; ids outside [-1, E) also set
 * MOE_DEVERR_BAD_ID. Within an expert, rows are in ascending t*K + k order
 * (deterministic; no dependence on atomic ordering). The MXFP8 rule: per 32
 * consecutive elements, scale byte = clamp(floor(log2(amax)) - 8 + 127, 0, 254)
 * (127 for an all-zero block), payload = E4M3(x / 2^(byte-127)) rounded to
 * nearest even and saturated to +-448.
 * Requires H % 32 == 0, 1 <= K <= min(E, 128), E <= 19370 (above 64
 * experts the count kernel keeps a 64-bit token mask and a count per expert in
 * shared memory; larger E gets MOE_ERR_UNSUPPORTED), and a workspace of
 * moe_permute_workspace_size(T, K, E) bytes (16-byte aligned; its contents
 * need not be initialised and are overwritten).
 * ------------------------------------------------------------------------ */
size_t moe_permute_workspace_size(int T, int K, int E);

/* Number of kernels moe_permute launches for this shape (2 when the per-expert,
 * per-token-tile count table is small enough to be scanned inside the scatter
 * kernel, else 3; 0 for T == 0; -1 for invalid sizes). Host-only, no GPU work;
 * not an operation of the pages, a count for launch accounting. */
int moe_permute_kernel_launches(int T, int K, int E);

moe_status moe_permute(const void *x, int T, int H,
                       const void *ids, moe_dtype id_dtype, int K, int E,
                       void *x_perm, uint8_t *x_perm_scales,
                       int32_t *group_sizes, int32_t *group_offsets,
                       int32_t *row_map, int32_t *perm_src,
                       unsigned flags, void *workspace, size_t workspace_bytes,
                       moe_stream_t stream);

/* ------------------------------------------------------------------------
 * moe_permute_noalloc: moe_permute without a caller workspace. (The pages
 * describe nothing like it; it exists for callers of this library.)
 *
 * Some callers cannot allocate device memory: a serving process that reserves
 * all of its GPU memory at start-up and forbids any later cudaMalloc, a plug-in
 * whose host application owns the CUDA allocator and offers C code no hook
 * into it, or code that must not risk the implicit device synchronisation
 * cudaMalloc / cudaFree may perform. This entry point takes the same arguments
 * as moe_permute minus the workspace and allocates nothing: its scratch is a
 * static device array of moe_permute_noalloc_max_scratch() bytes (4 MiB),
 * held by every GPU that loads the library until the process exits.
 *  - Its argument checks (shapes, dtypes, null pointers, alignment) come first
 *    and report what moe_permute reports; then it returns MOE_ERR_WORKSPACE,
 *    without enqueuing anything, when moe_permute_workspace_size(T, K, E)
 *    exceeds that maximum.
 *  - Every call looks up the array's device address on the current device
 *    (cudaGetSymbolAddress), so no address outlives a device reset. The first
 *    call on a device may load the library's device code: make that first call
 *    before any stream capture.
 *  - All calls on a device share the one array, and it keeps the last call's
 *    contents (nothing in it needs to start at zero: each call rewrites what it
 *    reads). Calls that overlap on the GPU (other streams, or other host threads
 *    on the same device) race on it: serialise them.
 * Outputs, requirements and errors are otherwise those of moe_permute.
 * ------------------------------------------------------------------------ */
size_t moe_permute_noalloc_max_scratch(void);

moe_status moe_permute_noalloc(const void *x, int T, int H,
                               const void *ids, moe_dtype id_dtype, int K, int E,
                               void *x_perm, uint8_t *x_perm_scales,
                               int32_t *group_sizes, int32_t *group_offsets,
                               int32_t *row_map, int32_t *perm_src,
                               unsigned flags, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Expert-parallel dispatch metadata ([TEJAX] "Optimization 2: Expert
 * parallelism to fuse Dispatch and Combine"; [SPARSER] "Remove work that has
 * no selected route": only selected routes travel, each destination receives
 * the rows of its own experts).
 *
 * G ranks, E_loc experts per rank (rank g owns experts g*E_loc ..
 * g*E_loc + E_loc - 1). Every source rank sends, from its moe_permute order,
 * the rows of the destination's experts (they are contiguous there); the
 * destination receives them source by source and, within a source, expert by
 * expert. recv_counts [G][E_loc] int32 (device): rows received from source s
 * for local expert j (the exchanged group sizes). Writes ids [R_cap] int32
 * (device): the local expert of each received row r, i.e. j of the segment
 * (s, j) that holds r when the segments are laid end to end in that order;
 * rows past the last segment get -1. moe_permute of the received rows with
 * these ids (K = 1, E = E_loc) gives the local experts' contiguous order.
 * Requires G * E_loc <= 4096; a negative count is read as 0 and sets
 * MOE_DEVERR_BAD_ID. Enqueues one kernel; the host never reads the counts.
 * ------------------------------------------------------------------------ */
moe_status moe_ep_recv_expert_ids(const int32_t *recv_counts, int G, int E_loc,
                                  long long R_cap, int32_t *ids, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Group-aware MXFP8 quantisation ([TEJAX] "Transformer Engine building
 * blocks": group-aware MXFP8 quantization feeding the MXFP8 grouped GEMM).
 *
 * x [R_cap, H] bf16, rows [group_offsets[e], group_offsets[e+1]) forming
 * group e; only rows < group_offsets[E] are read or written.
 *  - default (row-wise 1x32): q[R_cap, H] E4M3, scales[R_cap, H/32].
 *  - MOE_QUANT_COLWISE (32x1 along rows, for the weight-gradient GEMMs whose
 *    contraction runs over a group's rows): blocks start at each group's first
 *    row and never cross a group; a partial last block takes its amax over its
 *    valid rows. q[R_cap, H]; scales[E + R_cap/32 + 1, H] where block b of
 *    group e is scale row e + group_offsets[e]/32 + b (rows no block uses are
 *    left untouched).
 * Same scale/payload rule as moe_permute. Requires H % 32 == 0.
 * ------------------------------------------------------------------------ */
moe_status moe_quant_mxfp8_grouped(const void *x, int R_cap, int H,
                                   const int32_t *group_offsets, int E,
                                   uint8_t *q, uint8_t *scales,
                                   unsigned flags, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * NVFP4 operands ([TEJAX] "Measured training impact with JAX + Transformer
 * Engine" and [WITTY] "What to watch" name NVFP4 as a planned addition and do
 * not define it; NVIDIA's published format is taken). Elements E2M1 (0, 0.5,
 * 1, 1.5, 2, 3, 4, 6 and their negatives); 16 consecutive elements of a row
 * share one E4M3 decode scale; the tensor has one fp32 encode scale
 * S = 448 * 6 / amax (1 when amax is 0, at most FLT_MAX); a value decodes as
 * e2m1 * e4m3(scale) / S. Encoder, in fp32 with one rounding per operation:
 *   scale = E4M3(round to nearest even, saturating)((amax_block / 6) * S)
 *   code  = E2M1(round to nearest even, saturating to 6, sign kept)(x * (S / e4m3(scale))),
 *           0 when e4m3(scale) is 0.
 * Packing: element 2i in the low nibble of byte i, 2i+1 in the high nibble.
 *
 * moe_amax_bf16: *amax = max |x| over rows [0, n) of x [rows, cols] bf16, with
 *   n = rows, or min(rows, *valid_rows) when valid_rows (a device int, e.g.
 *   &group_offsets[E]) is given; cols % 8 == 0; amax is zeroed on the stream
 *   first. moe_quant_nvfp4: the same rows of x quantised with the encode scale of
 *   the device *amax: q [rows, cols/2] packed codes (8-byte aligned), scales
 *   [rows, cols/16]; rows past n are not written; cols % 16 == 0.
 * ------------------------------------------------------------------------ */
moe_status moe_amax_bf16(const void *x, long long rows, int cols, const int32_t *valid_rows,
                         float *amax, moe_stream_t stream);
moe_status moe_quant_nvfp4(const void *x, long long rows, int cols, const int32_t *valid_rows,
                           const float *amax, uint8_t *q, uint8_t *scales, moe_stream_t stream);

/* moe_permute_nvfp4: moe_permute (same routing outputs, workspace and rules)
 * whose scatter writes NVFP4 rows: first *x_amax = max |x| over the tokens
 * with at least one valid route (exactly the amax of the rows x_perm
 * receives; zeroed on the stream first), then each row is quantised with that
 * amax's encode scale as it is copied: x_perm_q [T*K, H/2] packed E2M1 (4-byte
 * aligned), x_perm_scales [T*K, H/16] E4M3 -- the bytes moe_quant_nvfp4 would
 * write from the bf16 permuted rows. One kernel more than moe_permute. */
moe_status moe_permute_nvfp4(const void *x, int T, int H, const void *ids, moe_dtype id_dtype,
                             int K, int E, float *x_amax, void *x_perm_q, uint8_t *x_perm_scales,
                             int32_t *group_sizes, int32_t *group_offsets, int32_t *row_map,
                             int32_t *perm_src, void *workspace, size_t workspace_bytes,
                             moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Grouped SwiGLU expert MLP ([TEJAX] "Optimization 1: Grouped GEMM": one
 * kernel covers all experts, each with its actual token count, computing only
 * valid regions, with the counts kept on the device; MoE-layer figure: the
 * grouped MLP is two grouped GEMMs on variable-length groups; "Transformer
 * Engine building blocks": MXFP8 grouped GEMM on Blackwell).
 *
 * For each expert e and each row r in [group_offsets[e], group_offsets[e+1]):
 *   a = x_perm[r] W1[e],  b = x_perm[r] W3[e]       (fp32 accumulation)
 *   h[r] = silu(a) * b    rounded to bf16, or (MXFP8) quantised 1x32 along F
 *   y_perm[r] = h[r] W2[e]  rounded to bf16
 * Rows >= group_offsets[E] are never written. Logical weights: W1, W3 [E, H, F]
 * and W2 [E, F, H] bf16; the GEMMs read them packed once by
 * moe_prepare_weights (outside the hot path):
 *   w13_packed [E][2F][H]: per 256-row tile j, rows 0..127 = columns
 *              128j..128j+127 of W1 transposed, rows 128..255 the same of W3;
 *   w2_packed  [E][H][F] = W2 transposed per expert;
 * bf16, or MXFP8 (E4M3 bytes, plus E8M0 scales [E][2F][H/32] and [E][H][F/32]
 * with blocks of 32 along the contraction dimension).
 * Activations: x_perm [R_cap, H] bf16, or MXFP8 E4M3 with x_scales
 * [R_cap, H/32] (as written by moe_permute with MOE_PERMUTE_FUSE_MXFP8);
 * h [R_cap, F] (caller-allocated intermediate, kept for the backward pass)
 * bf16, or E4M3 with h_scales [R_cap, F/32]; y_perm [R_cap, H] bf16.
 * Requires H % 256 == 0 and F % 128 == 0 (MXFP8: H % 512 == 0 and F % 512 == 0),
 * x_perm, h and the packed weights 128-byte aligned, scales 16-byte aligned,
 * E small enough for the group table to fit in shared memory (bf16: E <= 4200,
 * MXFP8: E <= 1150). moe_grouped_gemm_up / _down run the two halves alone.
 * ------------------------------------------------------------------------ */
size_t moe_packed_weights_bytes(int E, int H, int F, moe_dtype dtype, int which);
/* which: 0 = w13 payload, 1 = w13 scales, 2 = w2 payload, 3 = w2 scales (0 bytes for bf16) */

moe_status moe_prepare_weights(const void *w1, const void *w3, const void *w2, int E, int H, int F,
                               moe_dtype dtype, void *w13_packed, uint8_t *w13_scales,
                               void *w2_packed, uint8_t *w2_scales, moe_stream_t stream);

moe_status moe_grouped_swiglu_gemm(const void *x_perm, const uint8_t *x_scales,
                                   const void *w13_packed, const uint8_t *w13_scales,
                                   const void *w2_packed, const uint8_t *w2_scales, moe_dtype dtype,
                                   const int32_t *group_offsets, int E, int H, int F, int R_cap,
                                   void *h, uint8_t *h_scales, void *y_perm, moe_stream_t stream);

/* moe_grouped_gemm_up also saves, when the pointers are not NULL, what the
 * backward pass needs: ab_save [R_cap, 2F] bf16, the pre-activations a and b in
 * the interleaved layout of w13_packed (per 256 columns: 128 of a, then the
 * same 128 columns of b); h_bf16_save [R_cap, F] bf16, a bf16 copy of h (MXFP8
 * only, for the column-wise quantisation of the weight gradient). */
moe_status moe_grouped_gemm_up(const void *x_perm, const uint8_t *x_scales, const void *w13_packed,
                               const uint8_t *w13_scales, moe_dtype dtype,
                               const int32_t *group_offsets, int E, int H, int F, int R_cap,
                               void *h, uint8_t *h_scales, void *ab_save, void *h_bf16_save,
                               moe_stream_t stream);

moe_status moe_grouped_gemm_down(const void *h, const uint8_t *h_scales, const void *w2_packed,
                                 const uint8_t *w2_scales, moe_dtype dtype,
                                 const int32_t *group_offsets, int E, int H, int F, int R_cap,
                                 void *y_perm, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * The grouped SwiGLU MLP's two GEMMs on NVFP4 operands (tcgen05 kind
 * mxf4nvf4: E2M1 x E2M1 with a UE4M3 scale per 16 elements, fp32
 * accumulation, the two tensors' encode scales divided out in the epilogue).
 * Operands as moe_quant_nvfp4 writes them: x_q [R_cap, H/2] + x_scales
 * [R_cap, H/16] with the device x_amax; weights in the packed layouts of
 * moe_grouped_gemm_up (w13 [E][2F][H]) and down (w2 [E][H][F]) quantised
 * row-wise along the contraction dimension, each stacked tensor with one amax.
 * moe_grouped_gemm_up_nvfp4 writes h [R_cap, F] bf16 = silu(a) * b, the
 * optional ab_save like moe_grouped_gemm_up, and *h_amax = max |h| over the
 * rows it wrote (zeroed on the stream first), which moe_quant_nvfp4 takes to
 * quantise h for moe_grouped_gemm_down_nvfp4 (y_perm [R_cap, H] bf16).
 * Requires H % 256 == 0 and F % 256 == 0 (128-byte k-blocks of 256 elements);
 * operand bases 128-byte aligned, scales 16-byte aligned.
 * ------------------------------------------------------------------------ */
moe_status moe_grouped_gemm_up_nvfp4(const void *x_q, const uint8_t *x_scales, const float *x_amax,
                                     const void *w13_q, const uint8_t *w13_scales, const float *w13_amax,
                                     const int32_t *group_offsets, int E, int H, int F, int R_cap,
                                     void *h, float *h_amax, void *ab_save, moe_stream_t stream);
moe_status moe_grouped_gemm_down_nvfp4(const void *h_q, const uint8_t *h_scales, const float *h_amax,
                                       const void *w2_q, const uint8_t *w2_scales, const float *w2_amax,
                                       const int32_t *group_offsets, int E, int H, int F, int R_cap,
                                       void *y_perm, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Grouped backward of the SwiGLU expert MLP (the training step of [TEJAX]
 * "Measured training impact", on the same ragged groups as the forward).
 *
 * For each expert e and row r of its group, with a, b the saved bf16
 * pre-activations (ab_save of moe_grouped_gemm_up) and dy the gradient of y_perm:
 *   dh = dy W2[e]^T;  da = dh * b * silu'(a);  db = dh * silu(a)
 *       (silu'(a) = s(a) (1 + a (1 - s(a))), s the logistic function)
 *   dx = da W1[e]^T + db W3[e]^T
 *   dW2[e] = h_e^T dy_e;  dW1[e] = x_e^T da_e;  dW3[e] = x_e^T db_e
 * (fp32 accumulation, bf16 outputs). Backward weights, packed once by
 * moe_prepare_weights_bwd: w2_bwd [E][F][H] (= W2) and w13t [E][H][2F] (row h =
 * W1[e][h] and W3[e][h] interleaved per 128 columns), bf16 or MXFP8 with blocks
 * along H and along 2F respectively.
 *
 * moe_grouped_swiglu_dgrad: dy [R_cap, H] (bf16, or MXFP8 row-wise: E4M3 +
 *   dy_scales [R_cap, H/32]) -> dab [R_cap, 2F] bf16 = (da | db) interleaved per
 *   128 columns like ab. Requires F % 256 == 0. Optional (both or neither, NULL
 *   skips): dab_q [R_cap, 2F] E4M3 bytes (32-byte aligned) and dab_scales
 *   [R_cap, 2F/32] E8M0, the row-wise MXFP8 of the bf16 dab (1x32 blocks along
 *   2F, as moe_quant_mxfp8_grouped writes it), for moe_grouped_gemm_dx.
 * moe_grouped_gemm_dx: dab (bf16, or MXFP8 row-wise along 2F) -> dx [R_cap, H] bf16.
 * moe_grouped_transpose: makes a weight-gradient operand: for x [R_cap, C] bf16
 *   (or, with src_rows != NULL, x [*, C] read at row src_rows[r], e.g. the
 *   tokens through perm_src), xT[c][P_e + i] = x[off[e] + i][c] for i < m_e, with
 *   P_e = 128 * (e + off[e] / 128) and zeros up to P_e + 128 * ceil(m_e / 128);
 *   xT is [C][Kpad], Kpad = moe_grouped_transpose_kpad(R_cap, E) (a multiple of
 *   512 at least 128 * (E + ceil(R_cap / 128) + 1)). MXFP8 output:
 *   group-aware 32-row blocks (starting at each group's first row, a partial
 *   block taking its amax over valid rows), E4M3 payload in xT and E8M0 scales
 *   xT_scales[c][P_e / 32 + b] ([C][Kpad/32]). Requires C % 64 == 0.
 * moe_grouped_gemm_wgrad: aT [M][Kpad], bT [N][Kpad] from moe_grouped_transpose
 *   -> dw [E][M][N] bf16 with dw[e] = sum over group e's rows of a^T b; with dw2
 *   != NULL the output is split: columns [256j, 256j+128) of each row go to
 *   dw [E][M][N/2] and [256j+128, 256j+256) to dw2 (so bT = transposed dab gives
 *   dW1 and dW3 in their logical layouts). An expert with no rows gets zeros.
 *   Requires M % 128 == 0, N % 256 == 0.
 * ------------------------------------------------------------------------ */
moe_status moe_prepare_weights_bwd(const void *w1, const void *w3, const void *w2, int E, int H, int F,
                                   moe_dtype dtype, void *w2_bwd, uint8_t *w2_bwd_scales,
                                   void *w13t, uint8_t *w13t_scales, moe_stream_t stream);

moe_status moe_grouped_swiglu_dgrad(const void *dy, const uint8_t *dy_scales, const void *w2_bwd,
                                    const uint8_t *w2_bwd_scales, const void *ab, moe_dtype dtype,
                                    const int32_t *group_offsets, int E, int H, int F, int R_cap,
                                    void *dab, uint8_t *dab_q, uint8_t *dab_scales,
                                    moe_stream_t stream);

moe_status moe_grouped_gemm_dx(const void *dab, const uint8_t *dab_scales, const void *w13t,
                               const uint8_t *w13t_scales, moe_dtype dtype,
                               const int32_t *group_offsets, int E, int H, int F, int R_cap,
                               void *dx, moe_stream_t stream);

size_t moe_grouped_transpose_kpad(int R_cap, int E);

moe_status moe_grouped_transpose(const void *x, const int32_t *src_rows, int R_cap, int C,
                                 const int32_t *group_offsets, int E, moe_dtype out_dtype,
                                 void *xT, uint8_t *xT_scales, moe_stream_t stream);

moe_status moe_grouped_gemm_wgrad(const void *aT, const uint8_t *aT_scales, const void *bT,
                                  const uint8_t *bT_scales, moe_dtype dtype,
                                  const int32_t *group_offsets, int E, int M, int N, int R_cap,
                                  void *dw, void *dw2, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Unpermute / combine ([TEJAX] "Optimization 2": results are routed back and
 * accumulated; [SPARSER] "Remove work that has no selected route": combine is a
 * pull-and-reduce over each token's selected rows).
 *
 * y[t, :] = bf16( sum over k = 0..K-1 with row_map[t,k] >= 0 of
 *                 probs[t,k] * y_perm[row_map[t,k], :] )
 * accumulated in fp32 in ascending k; a token with no valid route gets zeros.
 * y_perm [R_cap, H] bf16, row_map [T, K] int32, probs [T, K] fp32, y [T, H] bf16.
 * Requires H % 8 == 0.
 * ------------------------------------------------------------------------ */
moe_status moe_unpermute_combine(const void *y_perm, const int32_t *row_map,
                                 const float *probs, int T, int K, int H,
                                 void *y, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Combine backward: the adjoint of moe_unpermute_combine (the chain rule
 * through y[t] = sum_k p[t,k] y_perm[row_map[t,k]]; the pages give the
 * forward, [TEJAX] "Optimization 2", and name training, not this step).
 * For every valid route (t, k) with row r = row_map[t,k]:
 *   dy_perm[r]   = bf16(p[t,k] * dy[t])                  (one rounding)
 *   dprobs[t,k]  = sum_j dy[t,j] * y_perm[r,j]            (fp32 accumulation)
 * and dprobs[t,k] = 0 for invalid routes. dy [T, H] bf16, y_perm [R_cap, H]
 * bf16 (the forward's), row_map [T, K], probs [T, K] fp32 in; dy_perm
 * [R_cap, H] bf16 (rows no route maps to are not written) and dprobs [T, K]
 * fp32 out. Requires H % 8 == 0, 1 <= K <= 128; 16-byte aligned rows.
 * Optional (both or neither; NULL skips): dy_perm_q [R_cap, H] E4M3 bytes
 * (8-byte aligned) and dy_perm_scales [R_cap, H/32] E8M0 bytes, the row-wise
 * MXFP8 quantisation (1x32 blocks along H, as moe_quant_mxfp8_grouped writes
 * it) of the bf16 dy_perm values, for the next grouped GEMM; requires
 * H % 32 == 0. Same rows written as dy_perm.
 * ------------------------------------------------------------------------ */
moe_status moe_unpermute_combine_backward(const void *dy, const void *y_perm,
                                          const int32_t *row_map, const float *probs,
                                          int T, int K, int H, void *dy_perm,
                                          float *dprobs, uint8_t *dy_perm_q,
                                          uint8_t *dy_perm_scales, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Permute backward: the adjoint of moe_permute's row copies, dx[t] = bf16(sum
 * over the valid k, ascending, of dx_perm[row_map[t,k]]) with fp32
 * accumulation; tokens without a valid route get 0. dx_perm [R_cap, H] bf16,
 * row_map [T, K] in; dx [T, H] bf16 out. Requires H % 8 == 0, 1 <= K <= 128.
 * ------------------------------------------------------------------------ */
moe_status moe_permute_backward(const void *dx_perm, const int32_t *row_map,
                                int T, int K, int H, void *dx, moe_stream_t stream);

/* ------------------------------------------------------------------------
 * Device error word. Copies the word to *flags_out (synchronising the device)
 * and clears it when `clear` is non-zero. Not for the hot path. Returns
 * MOE_ERR_DEVICE when the word was non-zero.
 * ------------------------------------------------------------------------ */
moe_status moe_get_device_errors(uint32_t *flags_out, int clear);

/* Self-test of the bounded waits the grouped GEMM uses for its pipeline barriers:
 * launches one warp that waits on a barrier nothing arrives on; after limit_us
 * microseconds (1 .. 1,000,000) the wait gives up, sets MOE_DEVERR_TIMEOUT in the
 * device error word and the kernel returns, leaving the context usable. */
moe_status moe_debug_bounded_wait_selftest(uint32_t limit_us, moe_stream_t stream);

/* Human-readable name of a status code (static storage). */
const char *moe_status_string(moe_status status);

/* Device address of page-locked host memory (cudaHostAlloc / pinned): on systems with a
 * unified address space the library's kernels can read their inputs from, and write their
 * outputs to, such memory directly (moe_permute's x, moe_unpermute_combine's y), so a caller
 * whose tensors live on the host needs no separate copy in or out. Writes *dev_ptr and returns
 * MOE_OK when host_ptr lies in page-locked memory the current device can address,
 * MOE_ERR_UNSUPPORTED otherwise (plain pageable memory, no mapping), MOE_ERR_INVALID_ARG for
 * null pointers. No work is enqueued. (The pages describe no such call.) */
moe_status moe_host_mapped_pointer(const void *host_ptr, void **dev_ptr);

/* Byte sizes of the compact route ([SPARSER] "Preserve a compact route":
 * [T, K] ids instead of a [T, E] map): ids of the given dtype, and fp32 probs. */
size_t moe_route_ids_bytes(int T, int K, moe_dtype id_dtype);
size_t moe_route_probs_bytes(int T, int K);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
