// Internal launchers of the MoE data-path kernels (host side).  Each
// returns the launch's cudaError_t; argument validation is done by the
// C ABI layer before any of these is called.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace moe {

#ifndef MOE_PDL
#define MOE_PDL 1
#endif

// Launch with programmatic stream serialisation (see griddep_wait): the
// kernel may be scheduled while the previous kernel on `stream` drains.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = MOE_PDL ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Sets the text returned by moe_last_error_string() for the calling thread.
void set_last_error(const char *msg);

// Adds n to the count returned by moe_kernel_launches(); every launch site
// calls it once per kernel it issues.
void count_launch(int n = 1);

// TMA tensor maps over bf16 row-major data, 128-byte swizzle, boxes of 64
// columns x box_rows rows (x 1 expert for the 3-D form [experts, rows, cols]).
bool make_tmap_2d(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint32_t box_rows);
bool make_tmap_3d(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint64_t experts,
                  uint32_t box_rows);
// fp32 row-major [rows, cols], box = box_cols x box_rows, 128-byte swizzle.
bool make_tmap_2d_f32(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows,
                      uint32_t box_cols, uint32_t box_rows);
// Row-major [experts, rows, cols] (experts = 0: a 2-D [rows, cols]) of 1-, 2- or
// 4-byte elements (e4m3 codes / bf16 / fp32), box = box_cols x box_rows (x 1), swizzle of
// 32, 64 or 128 bytes (box_cols x element bytes must equal it).
bool make_tmap_tile(CUtensorMap *m, const void *base, int elem_bytes, uint64_t cols, uint64_t rows,
                    uint64_t experts, uint32_t box_cols, uint32_t box_rows, int swizzle_bytes);
int sm_count();  // SMs of the current device (0 on error)

// Raises a kernel's dynamic shared-memory limit to at least `bytes` on the
// current device.  The attribute is set once per (kernel, device) and
// raised only when a larger size is asked for, so launches do not pay for it.
cudaError_t ensure_smem(const void *kernel, size_t bytes);

// Router.  bf16 with E <= kRouterTcMaxE runs on the tensor cores and needs
// router_scratch_floats(T, E, 1) floats of scratch for the split partials;
// everything else (or a missing scratch) runs the fused SIMT kernel.
constexpr int kRouterTcMaxE = 256;
#ifndef MOE_ROUTER_SPLITS
#define MOE_ROUTER_SPLITS 8
#endif
constexpr int kRouterMaxSplits = MOE_ROUTER_SPLITS;
int64_t router_scratch_floats(int T, int E, int is_bf16);
// n_group > 1: group-limited selection (validated by the caller).
cudaError_t launch_router_topk(const void *x, const void *wg, const float *bias, float *logits_out,
                               int *topk_idx, float *topk_w, int T, int D, int E, int k,
                               int score, int renorm, int n_group, int topk_group, int is_bf16,
                               float *scratch, int64_t scratch_floats, int *status,
                               cudaStream_t stream);

// Scratch ints needed by launch_permute: blocks of 256 tokens x E, twice.
int64_t permute_scratch_ints(int T, int E);

cudaError_t launch_permute(const void *x, const int *topk_idx, int *tokens_per_expert,
                           int *seg_offsets, int *row_of, int *token_of_row, void *x_perm,
                           int T, int D, int E, int k, int e_first, int E_local, int layout,
                           int align_m, int capacity, int64_t rows_alloc, int elem_bytes,
                           int *scratch, int *status, cudaStream_t stream,
                           float *x_scale = nullptr,   // set: bf16 x -> e4m3 x_perm + row scales
                           float *zero_out = nullptr);  // set: zero rows [T, D] fp32 (fused combine)

// out[i] = bf16(comb[i]) for the fused combine's fp32 accumulator (n % 4 == 0).
cudaError_t launch_comb_to_bf16(const float *comb, void *out, int64_t n, cudaStream_t stream);

// Row-wise e4m3 quantisation of bf16 rows [rows, cols] (cols % 8 == 0):
// scale[r] = amax / 448 (1 for a zero row), codes = e4m3(x / scale).  With
// row_of [rows, k], row t's codes and scale go to rows row_of[t, j] (the
// dispatch), else to row t.
cudaError_t launch_quantize_rows_e4m3(const void *src, int64_t rows, int cols, const int *row_of,
                                      int k, uint8_t *dst, float *scale, cudaStream_t stream);

// out[t] = sum_j w[t, j] y_perm[row_of[t, j]], fp32 in slot order, rounded
// once; y_perm fp16 with a bf16 out (is_bf16), fp32 with an fp32 out.
cudaError_t launch_combine(const void *y_perm, const int *row_of, const float *topk_w, void *out,
                           int T, int D, int k, int64_t rows_alloc, int is_bf16, int *status,
                           cudaStream_t stream);

// fp32 SIMT grouped SwiGLU (both GEMMs).
cudaError_t launch_grouped_swiglu_f32(const float *x_perm, const int *seg_offsets,
                                      const int *tokens_per_expert, const float *w1,
                                      const float *w3, const float *w2, float *h, float *y_perm,
                                      int D, int H_local, int e_first, int E_local,
                                      int64_t rows_alloc, int *status, cudaStream_t stream);

// Scratch ints of the pair kernel's one-launch schedule (block counters);
// they must be zero before the first call and are left zero by each call.
// The same with GEMM1 on e4m3 operands (kind::f8f6f4): x_perm_q [rows, D]
// and w1_q / w3_q [E_local, H_local, D] codes with one scale per row
// (x_scale [rows], w1_scale / w3_scale [E_local, H_local]); GEMM1's fp32
// accumulator is multiplied by x_scale[row] * w_scale[unit] before SwiGLU.
// GEMM2 stays bf16.  D % 16 == 0.
cudaError_t launch_grouped_swiglu_fp8_pair(const uint8_t *x_perm_q, const float *x_scale,
                                           const int *seg_offsets, const int *tokens_per_expert,
                                           const uint8_t *w1_q, const float *w1_scale,
                                           const uint8_t *w3_q, const float *w3_scale,
                                           const void *w2, void *h, void *y_perm, int D,
                                           int H_local, int e_first, int E_local,
                                           int64_t rows_alloc, int *scratch, int *status,
                                           cudaStream_t stream, bool *launched);
int64_t grouped_pair_scratch_ints(int64_t rows_alloc, int E_local);

// Combine fused into the grouped GEMM's second GEMM: its epilogue adds
// topk_w[t, j] * y for each row r = row_of[t, j] into comb [T, D] (fp32,
// zeroed beforehand) with atomic adds, instead of storing y_perm.  The sum
// over a token's slots then runs in no fixed order.
struct FusedCombine {
    float *comb;
    const int *token_of_row, *row_of;
    const float *topk_w;
    int k;
};

// GEMM1's A rows gathered from the token rows: row r of the grouped layout
// is x[token_of_row[r]] (x: [T, D] bf16), so x_perm need not exist.
struct GatherA {
    const void *x;
    const int *token_of_row;
    int64_t T;
};

// bf16 tcgen05 grouped SwiGLU on CTA pairs (cta_group::2).  With `scratch`
// both GEMMs run in one cooperative launch; without it, or where the device
// refuses a cooperative cluster launch, in two.  Sets *launched to false (and
// returns cudaSuccess) when the device cannot run clusters of two with this
// shared-memory size, so the caller can use the 1-CTA kernel.
cudaError_t launch_grouped_swiglu_bf16_pair(const void *x_perm, const int *seg_offsets,
                                            const int *tokens_per_expert, const void *w1,
                                            const void *w3, const void *w2, void *h, void *y_perm,
                                            int D, int H_local, int e_first, int E_local,
                                            int64_t rows_alloc, int *scratch, int *status,
                                            cudaStream_t stream, bool *launched,
                                            void *gu = nullptr, const FusedCombine *fc = nullptr,
                                            const GatherA *ga = nullptr);

// Backward of the bf16 grouped SwiGLU on CTA pairs: dgu = SwiGLU'(gy . w2_e)
// with the saved gate/up gu, dxp = dgu . [w1_e; w3_e] (fp32), and the weight
// gradients dw1, dw3 [E_local, H, D], dw2 [E_local, D, H] (fp32, or bf16 with
// grad_bf16: the fp32 sums rounded once).  Padding
// rows of x_perm, h and gy are set to zero first.  Needs D and H_local
// multiples of 64 and segments starting on multiples of 64 rows.
cudaError_t launch_grouped_swiglu_bwd(const void *x_perm, const void *h, const void *gu,
                                      const void *gy, const int *seg_offsets,
                                      const int *tokens_per_expert, const int *token_of_row,
                                      const void *w1, const void *w3, const void *w2,
                                      void *dgu, float *dxp, void *dw1, void *dw3, void *dw2,
                                      int D, int H_local, int e_first, int E_local,
                                      int64_t rows_alloc, int *status, cudaStream_t stream,
                                      int grad_bf16 = 0);  // dw1, dw3, dw2 in bf16 (else fp32)
int64_t grouped_bwd_smem(int E_local);

// Backward of the combine: gy[row] = bf16(w * dout[t]) (rows without a token
// untouched) and dw[t, j] = <dout[t], y_perm[row]> (y_perm fp16, as the bf16
// forward stores it).
cudaError_t launch_combine_bwd(const void *dout, const void *y_perm, const int *row_of,
                               const float *topk_w, void *gy, float *dw, int T, int D, int k,
                               int64_t rows_alloc, int is_bf16, int *status, cudaStream_t stream);

// Backward of the dispatch: dx[t] = sum_j dxp[row_of[t, j]] + r[t], where
// r[t] = add[t] when add, else sum_j dl[t, e_j] wg[e_j] (e_j = topk_idx[t, j];
// the router's part of dx when dl is zero off the selected experts), else 0.
cudaError_t launch_dispatch_bwd(const float *dxp, const int *row_of, const float *add,
                                const int *topk_idx, const float *dl, const void *wg, int E,
                                void *dx, int T, int D, int k, int64_t rows_alloc, int is_bf16,
                                cudaStream_t stream);

// dl is dense (every expert's logit gets a gradient) only for a softmax
// over all E without renormalisation; otherwise it is zero off the k
// selected experts of each token.
inline bool router_dl_dense(int score, int renorm) { return score == 0 && !renorm; }

// Floats of scratch launch_router_bwd needs for the split-K partials of
// dwg and dbias (0 when one split suffices).
int64_t router_bwd_scratch_floats(int T, int D, int E);

// The expert-contiguous layout of every expert (seg_off [E + 1], tpe [E],
// token_of_row), with no slot dropped: each (token, selected expert) has a row.
struct RouterSegments {
    const int *seg_off, *tpe, *token_of_row;
};

// Backward of the router from dw: dl [T, E], dbias [E] (or null), dwg [E, D]
// and, when router_dl_dense, the router's part of dx, dx_router [T, D]
// (fp32); otherwise dx_router is left to launch_dispatch_bwd.  With segs and
// dl zero off the selected experts, dwg and dbias are sums over each
// expert's segment instead of a dense GEMM over all T.
cudaError_t launch_router_bwd(const void *x, const void *wg, const float *logits,
                              const int *topk_idx, const float *topk_w, const float *dw, float *dl,
                              float *dx_router, float *dwg, float *dbias, float *scratch, int T,
                              int D, int E, int k, int score, int renorm, int is_bf16,
                              cudaStream_t stream, const RouterSegments *segs = nullptr);

// bf16 tcgen05 grouped SwiGLU (both GEMMs), one CTA per tile.
cudaError_t launch_grouped_swiglu_bf16(const void *x_perm, const int *seg_offsets,
                                       const int *tokens_per_expert, const void *w1,
                                       const void *w3, const void *w2, void *h, void *y_perm,
                                       int D, int H_local, int e_first, int E_local,
                                       int64_t rows_alloc, int *status, cudaStream_t stream);

}  // namespace moe
