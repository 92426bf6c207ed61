/*
 * moe.h -- C ABI of the GB300 (sm_103a) MoE layer local data path.
 *
 * The layer, per token t of x[T, D] (page "Expert Parallelism (EP)",
 * llm-infra-atlas, section 1 "MoE layer forward path"):
 *   1. gating logits  l = x . W_g^T (+ b)                     [T, E]
 *   2. top-k experts and their routing weights (softmax or sigmoid scores,
 *      optionally renormalised over the chosen k)
 *   3. tokens_per_expert and the dispatch permute into an expert-contiguous
 *      layout whose segments are padded to the GEMM M tile (same page,
 *      section 2, the layout contract between dispatch and grouped GEMM)
 *   4. m-grouped expert FFN, SwiGLU form: h = SiLU(X_e w1_e^T) * (X_e w3_e^T),
 *      y = h w2_e^T, with GroupedExperts weights w1/w3 [E, H, D] and
 *      w2 [E, D, H] (page "Expert Tensor Parallel design", HyperParallel
 *      issue 104, section 4.3)
 *   5. unpermute with the top-k weighted reduce back to token order
 *      (page "Expert Parallelism (EP)", section 1, combine post-process).
 *
 * Shards.  A call may cover an expert range [e_first, e_first + E_local) and
 * one H shard of width H_local (w1/w3 split on dim 1, w2 on dim 2: "Expert
 * Tensor Parallel design", section 4.3).  Its output is then a partial sum;
 * the partials of all shards add up to the layer output (row-parallel
 * identity Y = sum_t Y_partial^(t), page "NCCL course 32", section "Tensor
 * Parallel matrix split").  The library itself never communicates.
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller, dense,
 *     row-major, and 16-byte aligned.  The library allocates nothing.
 *   - Element type of x, W_g, weights, x_perm, h and out is cfg->dtype
 *     (MOE_F32 or MOE_BF16).  y_perm (the second GEMM's result per routed
 *     row) is fp32 for MOE_F32 and fp16 for MOE_BF16: the fp32 accumulator
 *     rounded once to nearest-even fp16, which keeps 3 more significant bits
 *     than bf16 at half the bytes of fp32.  Router bias, logits and topk_w
 *     are always fp32; indices are int32.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL means the
 *     legacy default stream) and performs no host synchronisation.
 *   - Host-side argument errors are returned before anything is launched.
 *     A failed launch returns MOE_ERR_CUDA.  Problems only the device can
 *     see (an expert id out of range, a NaN logit, masked capacity exceeded,
 *     a bounded wait that ran out) set bits in a status word inside the
 *     workspace; the kernels then skip the offending row instead of
 *     touching memory out of bounds.  moe_get_device_status() reads it.
 *   - The workspace `ws` (ws_bytes >= the size query of the call) must be
 *     zero-filled once before first use; calls keep it consistent after.
 *     Two calls that share a workspace must not run concurrently.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *moe_stream_t; /* same type as cudaStream_t */

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,  /* bad pointer, size, alignment or enum value */
    MOE_ERR_UNSUPPORTED = 2,  /* valid but not implemented (e.g. dtype mix) */
    MOE_ERR_CAPACITY = 3,     /* masked layout: an expert got > capacity rows */
    MOE_ERR_CUDA = 4,         /* a CUDA runtime / launch error */
    MOE_ERR_TIMEOUT = 5,      /* a bounded device wait ran out */
    MOE_ERR_BAD_ROUTING = 6,  /* expert id out of range, NaN logit, bad offsets */
    MOE_ERR_WORKSPACE = 7     /* workspace missing, misaligned or too small */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;
typedef enum { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 } moe_score;
typedef enum { MOE_LAYOUT_CONTIGUOUS = 0, MOE_LAYOUT_MASKED = 1 } moe_layout;

/*
 * Problem description shared by every call.
 *   T        tokens (rows of x), >= 0
 *   D        model dim, multiple of 8 (bf16: 16-byte rows for TMA)
 *   H_local  expert hidden width held by this call (H, or H/tp for an H
 *            shard), multiple of 8
 *   E        total number of experts (router width), 1..1024
 *   k        experts per token, 1..min(E, 32)
 *   e_first, E_local  local expert range, 0 <= e_first, e_first+E_local <= E
 *   dtype    moe_dtype; score moe_score; renorm 0/1 (renormalise the k
 *            chosen scores to sum to one)
 *   layout   moe_layout
 *   align_m  contiguous layout: each expert segment is padded up to a
 *            multiple of align_m rows (the GEMM M tile is 128; the bf16
 *            grouped GEMM is fastest when align_m is a multiple of 128)
 *   capacity masked layout: rows reserved per local expert (segment i
 *            starts at i*capacity); ignored for the contiguous layout
 *   n_group, topk_group  group-limited routing ("Expert Parallelism (EP)",
 *            section 3, DeepSeek-V3 style): with n_group > 1 the E experts
 *            form n_group equal groups of consecutive indices and a token
 *            may only choose experts of its topk_group best groups; a group
 *            scores the fp32 sum of its k/topk_group largest keys (added in
 *            selection order), ties to the lower group.  Requires
 *            E % n_group == 0, n_group <= 32, 1 <= topk_group <= n_group and
 *            topk_group <= k <= topk_group * E / n_group.  n_group 0 or 1:
 *            plain top-k (topk_group ignored).
 */
typedef struct {
    int32_t T, D, H_local, E, k;
    int32_t e_first, E_local;
    int32_t dtype, score, renorm, layout;
    int32_t align_m, capacity;
    int32_t n_group, topk_group;
} moe_config;

/* Human-readable name of a status code (static storage, never NULL). */
const char *moe_status_string(int32_t status);

/* Text of the last host-side error of the calling thread ("" if none). */
const char *moe_last_error_string(void);

/* ABI version: major * 10000 + minor * 100 + patch.  2.0.0 made y_perm of
 * bf16 layers fp16 (it was fp32 in 1.x). */
int32_t moe_abi_version(void);

/*
 * Kernels this library has launched in the calling process so far (all
 * threads, all devices; a launch counts when it was issued, whether or not
 * the kernel has run yet).  Instrumentation only: read it before and after
 * a region to count the region's launches.  Never fails.
 */
uint64_t moe_kernel_launches(void);

/* MOE_OK if cfg describes a problem every call below accepts. */
moe_status moe_validate_config(const moe_config *cfg);

/*
 * Rows of the permuted buffers x_perm / h / y_perm:
 *   contiguous: T * min(k, E_local) + E_local * (align_m - 1)
 *   masked:     E_local * capacity
 * Returns -1 if cfg is invalid.
 */
int64_t moe_rows_alloc(const moe_config *cfg);

/* Workspace bytes for the step calls (route, permute, grouped, combine). */
int64_t moe_workspace_size(const moe_config *cfg);

/* Workspace bytes for moe_layer_forward (includes every intermediate). */
int64_t moe_layer_workspace_size(const moe_config *cfg);

/*
 * Step 1+2: router logits, top-k and routing weights
 * ("Expert Parallelism (EP)", section 1: router.gating, routing).
 *   x [T, D] (dtype), wg [E, D] (dtype), bias [E] fp32 or NULL.
 *   logits_out [T, E] fp32 or NULL: the selection key l = x.wg^T + b
 *     accumulated in fp32.
 *   topk_idx [T, k] int32: chosen experts in selection order -- larger key
 *     first, equal keys by lower expert index, NaN after every number.
 *   topk_w [T, k] fp32: softmax over all E (or sigmoid) of the key at the
 *     chosen experts, divided by their sum when cfg->renorm.
 * A NaN key sets MOE_ERR_BAD_ROUTING in the status word.
 */
moe_status moe_route_topk(const moe_config *cfg, const void *x, const void *wg,
                          const float *bias, float *logits_out, int32_t *topk_idx,
                          float *topk_w, void *ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Step 3: tokens_per_expert, segment offsets and dispatch permute
 * ("Expert Parallelism (EP)", section 1 preprocess + permute; section 2
 * layout contract).
 *   topk_idx [T, k] int32 (any source; ids outside [0, E) are skipped and
 *     flag MOE_ERR_BAD_ROUTING).
 *   tokens_per_expert [E] int32: count of (t, j) with topk_idx = e, over all
 *     E experts (so it sums to T*k).
 *   seg_offsets [E_local + 1] int32: first row of each local expert's
 *     segment; contiguous: exclusive scan of counts padded to align_m;
 *     masked: i * capacity.
 *   row_of [T, k] int32: row of x_perm holding (t, j), or -1 when expert
 *     topk_idx[t, j] is not local.  Inside a segment rows are in ascending
 *     token order.
 *   token_of_row [rows_alloc] int32: the token of each row, -1 for padding.
 *   x_perm [rows_alloc, D] (dtype): x_perm[row_of[t, j]] = x[t] bit for
 *     bit.  Padding rows are not written (their contents are unspecified).
 * Masked layout: an expert with more than `capacity` tokens keeps its first
 * `capacity` (in token order), the rest get row_of = -1, and the status word
 * gets MOE_ERR_CAPACITY.
 */
moe_status moe_permute(const moe_config *cfg, const void *x, const int32_t *topk_idx,
                       int32_t *tokens_per_expert, int32_t *seg_offsets, int32_t *row_of,
                       int32_t *token_of_row, void *x_perm, void *ws, size_t ws_bytes,
                       moe_stream_t stream);

/*
 * Step 4: m-grouped SwiGLU expert FFN over the permuted layout
 * ("Expert Parallelism (EP)", section 1 routed_experts_compute and section
 * 2 m-grouped GEMM; weight shapes "Expert Tensor Parallel design" 4.3).
 *   x_perm [rows_alloc, D], seg_offsets [E_local + 1],
 *   tokens_per_expert [E] (the global counts; local expert i reads entry
 *     e_first + i; valid rows of segment i are the first
 *     min(count, seg_offsets[i+1] - seg_offsets[i])).
 *   w1, w3 [E_local, H_local, D]; w2 [E_local, D, H_local] (dtype).
 *   h [rows_alloc, H_local] (dtype, written for valid rows):
 *     h = SiLU(x_perm w1^T) * (x_perm w3^T), fp32 accumulation, one rounding.
 *   y_perm [rows_alloc, D] (written for valid rows): y = h w2^T accumulated
 *     in fp32; stored as that fp32 value for MOE_F32, rounded once to fp16
 *     for MOE_BF16.  A bf16 result that fp16 cannot hold (|y| >= 65520,
 *     which rounds to infinity) is flagged in the status word:
 *     moe_get_device_status then returns MOE_ERR_UNSUPPORTED (the stored
 *     value is +-inf).  The weighted combine widens the fp16 value to fp32.
 *   Rows that hold no token (padding) and rows of other segments are never
 *   written.
 * Segments may have any length; offsets outside [0, rows_alloc] flag
 * MOE_ERR_BAD_ROUTING and the segment is skipped.
 */
moe_status moe_grouped_swiglu(const moe_config *cfg, const void *x_perm,
                              const int32_t *seg_offsets, const int32_t *tokens_per_expert,
                              const void *w1, const void *w3, const void *w2, void *h,
                              void *y_perm, void *ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Step 5: unpermute with the top-k weighted reduce ("Expert Parallelism
 * (EP)", section 1 combine post-process; section 5: the transpose of the
 * dispatch permute).
 *   out[t, :] = sum_{j < k, row_of[t,j] >= 0} topk_w[t, j] * y_perm[row_of[t, j], :]
 * y_perm [rows_alloc, D] (fp32 for MOE_F32, fp16 for MOE_BF16, as
 * moe_grouped_swiglu writes it); summed in fp32 in slot order j, rounded
 * once to dtype into out [T, D].  Tokens with no
 * local expert get zeros.  Rows >= rows_alloc flag MOE_ERR_BAD_ROUTING and
 * are skipped.
 */
moe_status moe_unpermute_combine(const moe_config *cfg, const void *y_perm,
                                 const int32_t *row_of, const float *topk_w, void *out,
                                 void *ws, size_t ws_bytes, moe_stream_t stream);

/*
 * Steps 1-5 in order on one stream, every intermediate carved from ws
 * (ws_bytes >= moe_layer_workspace_size(cfg)).  out [T, D] (dtype) is this
 * call's partial output (the full layer output when the call holds every
 * expert and the whole H).
 */
moe_status moe_layer_forward(const moe_config *cfg, const void *x, const void *wg,
                             const float *bias, const void *w1, const void *w3,
                             const void *w2, void *out, void *ws, size_t ws_bytes,
                             moe_stream_t stream);

/* Workspace bytes for moe_layer_forward_host: the layer workspace plus
 * device staging for x and out. */
int64_t moe_layer_host_workspace_size(const moe_config *cfg);

/*
 * moe_layer_forward with the activations in HOST memory: x_host [T, D] and
 * out_host [T, D] (dtype, row-major) are host pointers; the router and
 * expert weights stay device pointers.  On `stream`, the call copies x_host
 * into device staging carved from ws (one cudaMemcpyAsync) and runs steps
 * 1-5.  When out_host is page-locked memory mapped into the device's
 * address space, the combine writes the output there directly; otherwise it
 * writes device staging that one cudaMemcpyAsync copies back.  out_host
 * holds the result once `stream` has completed.  Page-locked host buffers
 * let the copies run asynchronously; pageable ones work but the copies then
 * synchronise with the host.  ws_bytes >= moe_layer_host_workspace_size(cfg).
 */
moe_status moe_layer_forward_host(const moe_config *cfg, const void *x_host, const void *wg,
                                  const float *bias, const void *w1, const void *w3,
                                  const void *w2, void *out_host, void *ws, size_t ws_bytes,
                                  moe_stream_t stream);

/*
 * A depth-2 pipeline of moe_layer_forward calls with HOST activations (this
 * entry point has no counterpart in the pages; it is how a serving loop
 * keeps the host link and the GPU busy together).  Each submitted call
 * copies its x_host in and its result out, like moe_layer_forward_host, but
 * on two streams of the pipeline: the input copy of a call runs while the
 * previous call computes, and its output copy while the next call computes.
 * Device staging alternates between two slots of x and of out.
 *
 *   moe_host_pipeline_workspace_size: bytes of the caller's workspace (the
 *     layer workspace plus two x slots and two out slots), or -1 for a bad
 *     config.
 *   moe_host_pipeline_create: checks the config and the workspace (device
 *     memory, zero-filled once, 256-byte aligned, ws_bytes >= the size
 *     above) and creates the pipeline's two streams and its events on the
 *     current device.  Allocates no device memory.  *out receives the
 *     handle (NULL on failure).
 *   moe_host_pipeline_submit: queues one call: x_host [T, D] and out_host
 *     [T, D] (dtype, row-major) are host pointers, the weights device
 *     pointers, `stream` the compute stream, the same for every call
 *     between two syncs (the calls share the layer workspace's
 *     intermediates and rely on that stream's order; another stream there
 *     is MOE_ERR_INVALID_ARG).  Returns after queueing.  The
 *     host buffers of every submitted call must stay valid, and x_host
 *     unchanged, until moe_host_pipeline_sync returns; out_host holds the
 *     call's output from then on.  Page-locked buffers let the copies
 *     overlap the compute.
 *   moe_host_pipeline_sync: waits for every submitted call, output copies
 *     included, then returns the workspace status word like
 *     moe_get_device_status (and clears it).
 *   moe_host_pipeline_destroy: waits for the pipeline's streams and frees
 *     its streams, events and handle (NULL is a no-op).
 * Host-side argument errors are returned before anything is queued.
 */
typedef struct moe_host_pipeline moe_host_pipeline;
int64_t moe_host_pipeline_workspace_size(const moe_config *cfg);
moe_status moe_host_pipeline_create(const moe_config *cfg, void *ws, size_t ws_bytes,
                                    moe_host_pipeline **out);
moe_status moe_host_pipeline_submit(moe_host_pipeline *pipe, const void *x_host, const void *wg,
                                    const float *bias, const void *w1, const void *w3,
                                    const void *w2, void *out_host, moe_stream_t stream);
moe_status moe_host_pipeline_sync(moe_host_pipeline *pipe);
void moe_host_pipeline_destroy(moe_host_pipeline *pipe);

/*
 * Training: the forward that keeps what the backward needs, and the backward
 * of the whole layer ("Expert Parallelism (EP)", section 5: the backward runs
 * the forward in mirror -- the combine's backward is a dispatch of the output
 * gradient times the slot weights, the dispatch's backward a combine -- with
 * m-grouped dgrad and k-grouped wgrad GEMMs for the experts and the router
 * differentiated through its score function; the top-k selection itself has
 * no gradient).
 *
 * Supported: bf16, every expert and the whole H on this call (e_first = 0,
 * E_local = E, H_local = H), D and H_local multiples of 64, align_m (masked:
 * capacity) a multiple of 64; otherwise MOE_ERR_UNSUPPORTED.  The workspace
 * (ws_bytes >= moe_layer_train_workspace_size(cfg), -1 when unsupported)
 * holds the forward's intermediates plus the gate/up pre-activations [rows,
 * 2H] and the router logits, and the backward's own buffers.
 */
int64_t moe_layer_train_workspace_size(const moe_config *cfg);

/*
 * moe_layer_forward that also keeps, in ws, the gate and up pre-activations
 * (bf16) and the router logits.  Same output as moe_layer_forward.
 */
moe_status moe_layer_forward_train(const moe_config *cfg, const void *x, const void *wg,
                                   const float *bias, const void *w1, const void *w3,
                                   const void *w2, void *out, void *ws, size_t ws_bytes,
                                   moe_stream_t stream);

/*
 * Gradients of L = sum(dout * out) for the forward last run with
 * moe_layer_forward_train on the same ws and the same x, wg, w1, w3, w2.
 *   dout [T, D] bf16: output gradient; dx [T, D] bf16: input gradient.
 *   dwg [E, D], dbias [E] (or NULL), dw1 / dw3 [E, H, D], dw2 [E, D, H]: fp32,
 *   overwritten.
 * Per token t and slot j (row r, expert e, weight w_j):
 *   gy[r] = w_j dout[t],  dw_j = <dout[t], y_perm[r]>;
 *   dh = gy w2_e,  dg = dh * u * SiLU'(g),  du = dh * SiLU(g),
 *   dx[t] = sum_j (dg w1_e + du w3_e)[r] + (dl[t] wg);
 *   dw2_e = sum_r gy^T h,  dw1_e = sum_r dg^T x,  dw3_e = sum_r du^T x;
 *   dl = the score function's backward of dw (softmax over E or sigmoid,
 *   with renorm), dbias = sum_t dl,  dwg = dl^T x.
 * The backward overwrites the padding rows of the saved x_perm and h with
 * zeros.  Reduction orders are fixed: results are bit-identical run to run.
 * With T = 0 there is nothing to differentiate: dx has no rows, and dwg,
 * dbias, dw1, dw3 and dw2 are set to zero (only their pointers are checked).
 */
moe_status moe_layer_backward(const moe_config *cfg, const void *x, const void *wg,
                              const void *w1, const void *w3, const void *w2, const void *dout,
                              void *dx, float *dwg, float *dbias, float *dw1, float *dw3,
                              float *dw2, void *ws, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_layer_backward with the expert weight gradients dw1, dw3, dw2 in
 * wgrad_dtype: MOE_F32 (the same as moe_layer_backward) or MOE_BF16 (each
 * fp32 sum rounded once to nearest-even bf16: half the bytes of the
 * weight-gradient writes, which bound those GEMMs).  dwg and dbias stay fp32.
 */
moe_status moe_layer_backward_ex(const moe_config *cfg, const void *x, const void *wg,
                                 const void *w1, const void *w3, const void *w2, const void *dout,
                                 void *dx, float *dwg, float *dbias, void *dw1, void *dw3,
                                 void *dw2, int32_t wgrad_dtype, void *ws, size_t ws_bytes,
                                 moe_stream_t stream);

/*
 * FP8 e4m3 dispatch (page "Expert Parallelism (EP)", llm-infra-atlas: the FP8
 * dispatch of its next steps -- dispatched activations as e4m3 values with
 * scales feeding an FP8 grouped GEMM).  The page does not fix the scale
 * granularity; these calls use one binary32 scale per row:
 *   s[r] = max_c |v[r, c]| / 448  (1 for an all-zero row),
 *   q[r, c] = e4m3(v[r, c] / s[r])  (nearest, ties to even, saturating to
 *   +-448; NaN to 0x7f), both divisions correctly rounded binary32;
 *   value(q) * s[r] reconstructs v[r, c] within half an e4m3 step.
 * e4m3 is the "fn" format: bias 7, 3 mantissa bits, no infinities.
 * Per-row scales factor out of a GEMM's K sum, so GEMM1 runs on the codes
 * (tcgen05 kind::f8f6f4, fp32 accumulate) and multiplies its accumulator by
 * s_x[row] * s_w[unit] before SwiGLU; h stays bf16 and GEMM2 stays bf16.
 */

/*
 * Row-wise quantisation of bf16 src [rows, cols] (cols % 16 == 0) into
 * codes dst [rows, cols] (uint8) and scale [rows] (fp32): the form the FP8
 * calls take w1 and w3 in (rows = E_local * H_local, cols = D).  Device
 * pointers; 16-byte aligned src and dst.
 */
moe_status moe_quantize_rows_fp8(const void *src, int64_t rows, int32_t cols, uint8_t *dst,
                                 float *scale, moe_stream_t stream);

/*
 * moe_permute with the dispatched rows quantised: x [T, D] bf16 in;
 * x_perm_q [rows_alloc, D] e4m3 codes and x_scale [rows_alloc] fp32 out
 * (each token's row quantised once, copied to its k rows with its scale).
 * Counts, offsets, row_of and token_of_row exactly as moe_permute.
 * Requires dtype MOE_BF16, D % 16 == 0 and k <= 32 (else MOE_ERR_UNSUPPORTED).
 */
moe_status moe_permute_fp8(const moe_config *cfg, const void *x, const int32_t *topk_idx,
                           int32_t *tokens_per_expert, int32_t *seg_offsets, int32_t *row_of,
                           int32_t *token_of_row, uint8_t *x_perm_q, float *x_scale, void *ws,
                           size_t ws_bytes, moe_stream_t stream);

/*
 * moe_grouped_swiglu with GEMM1 on e4m3 operands:
 *   g = s_x[r] s_w1[e, n] sum_d q_x[r, d] q_w1[e, n, d],  u likewise with w3,
 *   h[r, n] = bf16(SiLU(g) u),  y_perm = fp16(h w2_e^T) (bf16 x bf16, fp32
 *   accumulation, one rounding).
 * x_perm_q / x_scale as moe_permute_fp8 writes them; w1_q, w3_q
 * [E_local, H_local, D] codes with w1_scale, w3_scale [E_local, H_local]
 * (moe_quantize_rows_fp8 of the bf16 weights); w2 bf16 [E_local, D, H_local];
 * h bf16 [rows_alloc, H_local], y_perm fp16 [rows_alloc, D].
 * MOE_ERR_UNSUPPORTED for more local experts than the CTA-pair kernel's
 * shared-memory tile table holds.
 */
moe_status moe_grouped_swiglu_fp8(const moe_config *cfg, const uint8_t *x_perm_q,
                                  const float *x_scale, const int32_t *seg_offsets,
                                  const int32_t *tokens_per_expert, const uint8_t *w1_q,
                                  const float *w1_scale, const uint8_t *w3_q,
                                  const float *w3_scale, const void *w2, void *h, void *y_perm,
                                  void *ws, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_layer_forward with the FP8 dispatch and GEMM1: route (bf16 x, fp32
 * keys, as moe_route_topk), moe_permute_fp8, moe_grouped_swiglu_fp8 and the
 * combine, on one stream.  Workspace: moe_layer_workspace_size (it holds the
 * codes in the x_perm buffer and one scale per row).
 */
moe_status moe_layer_forward_fp8(const moe_config *cfg, const void *x, const void *wg,
                                 const float *bias, const uint8_t *w1_q, const float *w1_scale,
                                 const uint8_t *w3_q, const float *w3_scale, const void *w2,
                                 void *out, void *ws, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_layer_forward with the combine fused into the grouped GEMM's second
 * GEMM ([EP] section 2: the permute / combine fusion that removes a round
 * trip of the routed rows): GEMM2's epilogue multiplies each row's fp32
 * result by its slot weight and adds it into an fp32 [T, D] accumulator
 * (the y_perm buffer of ws) with atomic adds; a last kernel rounds it to
 * the bf16 out.  y_perm is never written.  The sum over a token's slots
 * runs in whatever order the tiles finish, so -- unlike moe_layer_forward --
 * results may differ in the last bits from run to run.  bf16, D % 4 == 0,
 * workspace moe_layer_workspace_size.
 */
moe_status moe_layer_forward_fused(const moe_config *cfg, const void *x, const void *wg,
                                   const float *bias, const void *w1, const void *w3,
                                   const void *w2, void *out, void *ws, size_t ws_bytes,
                                   moe_stream_t stream);

/*
 * The dispatch fused into the first GEMM's operand load ("Expert Parallelism
 * (EP)", section 4: the dispatch folded into the neighbouring kernel so the
 * routed rows skip one HBM round trip; section 2: the expert-contiguous,
 * M-tile-aligned layout the grouped GEMM reads).  The permuted copy x_perm
 * is never made: GEMM1 reads row r of the layout as x[token_of_row[r]].
 *
 * moe_permute_index: moe_permute without the row copy -- the same
 * tokens_per_expert, seg_offsets, row_of and token_of_row, bit for bit, and
 * the same status flags; x and x_perm are not taken.
 */
moe_status moe_permute_index(const moe_config *cfg, const int32_t *topk_idx,
                             int32_t *tokens_per_expert, int32_t *seg_offsets, int32_t *row_of,
                             int32_t *token_of_row, void *ws, size_t ws_bytes,
                             moe_stream_t stream);

/*
 * moe_grouped_swiglu with GEMM1's rows gathered from x [T, D] (bf16) by
 * token_of_row [rows_alloc] (as moe_permute / moe_permute_index write it;
 * -1 rows are read as zeros).  h and y_perm are bit for bit those of
 * moe_grouped_swiglu on the x_perm that moe_permute would have written.
 * bf16 only (MOE_ERR_UNSUPPORTED otherwise); it always runs the CTA-pair
 * kernel, whatever the rows per expert.
 */
moe_status moe_grouped_swiglu_gather(const moe_config *cfg, const void *x,
                                     const int32_t *token_of_row, const int32_t *seg_offsets,
                                     const int32_t *tokens_per_expert, const void *w1,
                                     const void *w3, const void *w2, void *h, void *y_perm,
                                     void *ws, size_t ws_bytes, moe_stream_t stream);

/*
 * moe_layer_forward with the two calls above in place of moe_permute and
 * moe_grouped_swiglu: route, permute_index, grouped_swiglu_gather, combine,
 * on one stream.  The output equals moe_layer_forward's bit for bit.  bf16
 * only; workspace moe_layer_workspace_size (its x_perm region is unused).
 */
moe_status moe_layer_forward_gather(const moe_config *cfg, const void *x, const void *wg,
                                    const float *bias, const void *w1, const void *w3,
                                    const void *w2, void *out, void *ws, size_t ws_bytes,
                                    moe_stream_t stream);

/*
 * moe_permute without a workspace (this entry point has no counterpart in
 * the pages; it exists for callers that cannot allocate device memory).
 *
 * Some callers cannot call cudaMalloc where they dispatch: code running in a
 * memory pool it does not own, plugins handed only their input and output
 * tensors, or latency-critical loops where an allocation's implicit device
 * synchronisation is not acceptable.  This call does the same work as
 * moe_permute (same arguments and outputs, same bit-exact results) but keeps
 * its scratch in a fixed device array of about 1 MiB inside the library, which every
 * GPU that loads the library holds until the process exits.  It allocates
 * nothing.
 *   Limit: 2 * ceil(T / 256) * E <= 262144 (e.g. T = 16384 with E <= 2048);
 *     larger problems return MOE_ERR_UNSUPPORTED before any launch.
 *   device_flags: device int32 that the kernels OR their MOE status flags
 *     into (bad expert id: 1, capacity exceeded: 2), or NULL to drop them.
 *     The caller zeroes it; moe_get_device_status does not see these flags.
 *   The first call on each device looks up the array's device address
 *     (with that device current); make that first call before any stream
 *     capture.  The address is looked up again when the device's current
 *     context is not the one it was taken in (after cudaDeviceReset the
 *     library's module, and the array with it, load anew); a call made
 *     under stream capture after such a reset is not supported.
 *   Every call shares the one array and leaves its contents behind; the
 *     one word that must be zero between calls (a completion ticket) starts
 *     at zero when the library loads and every call returns it to zero.
 *     Calls whose kernels overlap on the GPU
 *     (other streams, other host threads) race on it: order them on one
 *     stream.
 */
moe_status moe_permute_noalloc(const moe_config *cfg, const void *x, const int32_t *topk_idx,
                               int32_t *tokens_per_expert, int32_t *seg_offsets,
                               int32_t *row_of, int32_t *token_of_row, void *x_perm,
                               int32_t *device_flags, moe_stream_t stream);

/*
 * Synchronises `stream`, reads the workspace status word, clears it and
 * returns the most serious flagged condition (MOE_OK if none).  Order:
 * TIMEOUT, then MOE_ERR_CUDA for a kernel that found itself launched
 * without the thread-block cluster it needs (it did no work), then
 * MOE_ERR_UNSUPPORTED for a bf16 expert output beyond fp16's range in
 * y_perm, then CAPACITY, BAD_ROUTING.
 */
moe_status moe_get_device_status(const void *ws, size_t ws_bytes, moe_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H */
