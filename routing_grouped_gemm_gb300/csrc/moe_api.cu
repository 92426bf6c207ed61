// C ABI of the MoE layer local data path: argument validation, workspace
// carving and the launch sequence.  Declarations and contracts: moe.h.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "../../include/moe.h"
#include "common.cuh"
#include "launch.h"

#define MOE_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

// 2.0.0: y_perm of bf16 layers is fp16 (fp32 up to 1.5.0)
constexpr int32_t kAbiVersion = 20000;
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;
constexpr int64_t kAlign = 256;

thread_local char g_last_error[256] = "";

int64_t align_up(int64_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

moe_status cuda_fail(cudaError_t e, const char *where) {
    snprintf(g_last_error, sizeof g_last_error, "%s: %s", where, cudaGetErrorString(e));
    return MOE_ERR_CUDA;
}

moe_status arg_fail(const char *why, moe_status st = MOE_ERR_INVALID_ARG) {
    snprintf(g_last_error, sizeof g_last_error, "%s", why);
    return st;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int elem_bytes(const moe_config *c) { return c->dtype == MOE_BF16 ? 2 : 4; }

int64_t rows_alloc_of(const moe_config *c) {
    if (c->layout == MOE_LAYOUT_MASKED) return (int64_t)c->E_local * c->capacity;
    const int64_t kl = c->k < c->E_local ? c->k : c->E_local;
    return (int64_t)c->T * kl + (int64_t)c->E_local * (c->align_m - 1);
}

moe_status validate(const moe_config *c) {
    if (!c) return arg_fail("config is NULL");
    if (c->T < 0) return arg_fail("T < 0");
    if (c->D < 8 || c->D % 8) return arg_fail("D must be a positive multiple of 8");
    if (c->H_local < 8 || c->H_local % 8) return arg_fail("H_local must be a positive multiple of 8");
    if (c->E < 1 || c->E > kMaxExperts) return arg_fail("E must be in 1..1024");
    if (c->k < 1 || c->k > c->E || c->k > kMaxTopK) return arg_fail("k must be in 1..min(E, 32)");
    if (c->e_first < 0 || c->E_local < 0 || c->e_first + c->E_local > c->E)
        return arg_fail("expert range outside [0, E)");
    if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return arg_fail("unknown dtype");
    if (c->score != MOE_SCORE_SOFTMAX && c->score != MOE_SCORE_SIGMOID)
        return arg_fail("unknown score function");
    if (c->renorm != 0 && c->renorm != 1) return arg_fail("renorm must be 0 or 1");
    if (c->layout != MOE_LAYOUT_CONTIGUOUS && c->layout != MOE_LAYOUT_MASKED)
        return arg_fail("unknown layout");
    if (c->layout == MOE_LAYOUT_CONTIGUOUS && (c->align_m < 1 || c->align_m > (1 << 16)))
        return arg_fail("align_m must be in 1..65536");
    if (c->layout == MOE_LAYOUT_MASKED && c->capacity < 0) return arg_fail("capacity < 0");
    if (c->n_group < 0) return arg_fail("n_group < 0");
    if (c->n_group > 1) {
        if (c->n_group > 32 || c->E % c->n_group != 0)
            return arg_fail("n_group must divide E and be at most 32");
        if (c->topk_group < 1 || c->topk_group > c->n_group || c->k < c->topk_group ||
            c->k > c->topk_group * (c->E / c->n_group))
            return arg_fail("topk_group must satisfy 1 <= topk_group <= n_group and "
                            "topk_group <= k <= topk_group * E / n_group");
    }
    if ((int64_t)c->T * c->k >= (int64_t)1 << 31) return arg_fail("T*k too large");
    if (rows_alloc_of(c) >= (int64_t)1 << 31) return arg_fail("permuted rows exceed 2^31");
    return MOE_OK;
}

struct StepWs {
    moe::StatusBlock *status;
    int *scratch;           // permute counting-sort scratch
    float *router_part;     // router split partials (bf16 tensor-core path)
    int64_t router_floats;
    int *grouped;           // grouped GEMM block counters (bf16), zero between calls
};

int64_t permute_ws_bytes(const moe_config *c) {
    return align_up(4 * moe::permute_scratch_ints(c->T, c->E));
}

int64_t router_ws_bytes(const moe_config *c) {
    return align_up(4 * moe::router_scratch_floats(c->T, c->E, c->dtype == MOE_BF16));
}

int64_t grouped_ws_bytes(const moe_config *c) {
    return c->dtype == MOE_BF16
               ? align_up(4 * moe::grouped_pair_scratch_ints(rows_alloc_of(c), c->E_local))
               : 0;
}

int64_t step_ws_bytes(const moe_config *c) {
    return (int64_t)sizeof(moe::StatusBlock) + permute_ws_bytes(c) + router_ws_bytes(c) +
           grouped_ws_bytes(c);
}

moe_status carve_step(const moe_config *c, void *ws, size_t ws_bytes, StepWs *out) {
    if (!ws) return arg_fail("workspace is NULL", MOE_ERR_WORKSPACE);
    if (!aligned(ws, kAlign)) return arg_fail("workspace must be 256-byte aligned", MOE_ERR_WORKSPACE);
    if ((int64_t)ws_bytes < step_ws_bytes(c)) return arg_fail("workspace too small", MOE_ERR_WORKSPACE);
    char *base = static_cast<char *>(ws);
    out->status = reinterpret_cast<moe::StatusBlock *>(base);
    out->scratch = reinterpret_cast<int *>(base + sizeof(moe::StatusBlock));
    out->router_floats = moe::router_scratch_floats(c->T, c->E, c->dtype == MOE_BF16);
    out->router_part = out->router_floats
                           ? reinterpret_cast<float *>(base + sizeof(moe::StatusBlock) +
                                                       permute_ws_bytes(c))
                           : nullptr;
    out->grouped = grouped_ws_bytes(c)
                       ? reinterpret_cast<int *>(base + sizeof(moe::StatusBlock) +
                                                 permute_ws_bytes(c) + router_ws_bytes(c))
                       : nullptr;
    return MOE_OK;
}

struct LayerWs {
    StepWs step;
    int *topk_idx, *tpe, *seg_off, *row_of, *token_of_row;
    float *topk_w;
    void *x_perm, *h, *y_perm;
    float *x_scale;  // FP8 layer: one scale per row of x_perm
};

int64_t layer_ws_layout(const moe_config *c, char *base, LayerWs *L) {
    int64_t off = step_ws_bytes(c);
    const int64_t R = (int64_t)c->T * c->k;
    const int64_t rows = rows_alloc_of(c);
    const int eb = elem_bytes(c);
    auto take = [&](int64_t bytes) -> char * {
        char *p = base ? base + off : nullptr;
        off += align_up(bytes);
        return p;
    };
    char *p_idx = take(4 * R);
    char *p_w = take(4 * R);
    char *p_tpe = take(4 * (int64_t)c->E);
    char *p_seg = take(4 * ((int64_t)c->E_local + 1));
    char *p_row = take(4 * R);
    char *p_tor = take(4 * rows);
    char *p_xp = take(rows * c->D * eb);
    char *p_h = take(rows * c->H_local * eb);
    // y_perm: fp16 for bf16 layers, fp32 for fp32 ones; for bf16 the region
    // also holds moe_layer_forward_fused's fp32 [T, D] accumulator
    char *p_yp = take(c->dtype == MOE_BF16 ? std::max(rows * c->D * 2, (int64_t)c->T * c->D * 4)
                                           : rows * c->D * 4);
    char *p_xs = take(rows * 4);
    if (L) {
        L->x_scale = reinterpret_cast<float *>(p_xs);
        L->topk_idx = reinterpret_cast<int *>(p_idx);
        L->topk_w = reinterpret_cast<float *>(p_w);
        L->tpe = reinterpret_cast<int *>(p_tpe);
        L->seg_off = reinterpret_cast<int *>(p_seg);
        L->row_of = reinterpret_cast<int *>(p_row);
        L->token_of_row = reinterpret_cast<int *>(p_tor);
        L->x_perm = p_xp;
        L->h = p_h;
        L->y_perm = p_yp;
    }
    return off;
}

// Training workspace: the layer workspace, then what the backward needs
// besides it: the gate/up pre-activations gu [rows, 2H] (bf16), the router
// logits [T, E], and the backward's own buffers gy [rows, D] (bf16), dgu
// [rows, 2H] (bf16), dxp [rows, D], dw [T, k], dl [T, E], dx_router [T, D]
// and the router backward's split-K partials (fp32).
struct TrainWs {
    __nv_bfloat16 *gu, *gy, *dgu;
    float *logits, *dxp, *dw, *dl, *dxr, *rsplit;
};

int64_t train_ws_layout(const moe_config *c, char *base, TrainWs *W) {
    int64_t off = layer_ws_layout(c, nullptr, nullptr);
    const int64_t rows = rows_alloc_of(c);
    auto take = [&](int64_t bytes) -> char * {
        char *p = base ? base + off : nullptr;
        off += align_up(bytes);
        return p;
    };
    char *p_gu = take(rows * 2 * c->H_local * 2);
    char *p_lg = take((int64_t)c->T * c->E * 4);
    char *p_gy = take(rows * c->D * 2);
    char *p_dgu = take(rows * 2 * c->H_local * 2);
    char *p_dxp = take(rows * c->D * 4);
    char *p_dw = take((int64_t)c->T * c->k * 4);
    char *p_dl = take((int64_t)c->T * c->E * 4);
    char *p_dxr = take((int64_t)c->T * c->D * 4);
    char *p_rs = take(moe::router_bwd_scratch_floats(c->T, c->D, c->E) * 4);
    if (W) {
        W->gu = reinterpret_cast<__nv_bfloat16 *>(p_gu);
        W->logits = reinterpret_cast<float *>(p_lg);
        W->gy = reinterpret_cast<__nv_bfloat16 *>(p_gy);
        W->dgu = reinterpret_cast<__nv_bfloat16 *>(p_dgu);
        W->dxp = reinterpret_cast<float *>(p_dxp);
        W->dw = reinterpret_cast<float *>(p_dw);
        W->dl = reinterpret_cast<float *>(p_dl);
        W->dxr = reinterpret_cast<float *>(p_dxr);
        W->rsplit = reinterpret_cast<float *>(p_rs);
    }
    return off;
}

// What the training forward and the backward support: bf16, every expert
// and the whole H on this call, dimensions in whole 64-element blocks and
// segments on 64-row boundaries (the k-grouped weight gradients reduce over
// whole 64-row blocks of each segment).
moe_status train_supported(const moe_config *c) {
    if (c->dtype != MOE_BF16) return arg_fail("training path: bf16 only", MOE_ERR_UNSUPPORTED);
    if (c->e_first != 0 || c->E_local != c->E)
        return arg_fail("training path: every expert on this call (no expert range)",
                        MOE_ERR_UNSUPPORTED);
    if (c->D % 64 || c->H_local % 64)
        return arg_fail("training path: D and H_local must be multiples of 64", MOE_ERR_UNSUPPORTED);
    if (c->layout == MOE_LAYOUT_CONTIGUOUS ? c->align_m % 64 != 0 : c->capacity % 64 != 0)
        return arg_fail("training path: align_m (capacity) must be a multiple of 64",
                        MOE_ERR_UNSUPPORTED);
    if (moe::grouped_bwd_smem(c->E_local) > 227 * 1024)
        return arg_fail("training path: too many experts for one CTA's tile table", MOE_ERR_UNSUPPORTED);
    return MOE_OK;
}

bool need16(const void *p) { return p && aligned(p, 16); }

// ---------------------------------------------------------------------
// step implementations (arguments already validated)
// ---------------------------------------------------------------------
moe_status do_route(const moe_config *c, const void *x, const void *wg, const float *bias,
                    float *logits_out, int32_t *topk_idx, float *topk_w, const StepWs &w,
                    cudaStream_t s) {
    cudaError_t e = moe::launch_router_topk(x, wg, bias, logits_out, topk_idx, topk_w, c->T, c->D,
                                            c->E, c->k, c->score, c->renorm,
                                            c->n_group > 1 ? c->n_group : 0, c->topk_group,
                                            c->dtype == MOE_BF16,
                                            w.router_part, w.router_floats, &w.status->flags, s);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_route_topk");
}

moe_status do_permute(const moe_config *c, const void *x, const int32_t *topk_idx, int32_t *tpe,
                      int32_t *seg, int32_t *row_of, int32_t *tor, void *x_perm, const StepWs &w,
                      cudaStream_t s, float *x_scale = nullptr, float *zero_out = nullptr) {
    cudaError_t e = moe::launch_permute(x, topk_idx, tpe, seg, row_of, tor, x_perm, c->T, c->D, c->E,
                                        c->k, c->e_first, c->E_local, c->layout, c->align_m,
                                        c->capacity, rows_alloc_of(c), elem_bytes(c), w.scratch,
                                        &w.status->flags, s, x_scale, zero_out);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_permute");
}

moe_status do_grouped(const moe_config *c, const void *x_perm, const int32_t *seg,
                      const int32_t *tpe, const void *w1, const void *w3, const void *w2, void *h,
                      void *y_perm, const StepWs &w, cudaStream_t s) {
    cudaError_t e;
    if (c->dtype == MOE_BF16) {
        // Two tcgen05 implementations: one CTA per 128x256 tile, or CTA pairs
        // on 256x256 tiles (cta_group::2, with an M=128 pair tile for an
        // expert's last <= 128 rows).  Measured on GB300 (grouped SwiGLU call,
        // single vs pair): fine-grained 0.364 vs 0.359 ms, DeepSeek-V3-shaped
        // 5.24 vs 4.87 ms, Zipf-skewed 3.19 vs 3.11 ms; decode (about four
        // rows per expert) 3.20 vs 3.28 ms.  MOE_GROUPED_KERNEL=single|pair|pair2
        // overrides the choice.
        const int64_t avg_rows =
            c->E_local ? (int64_t)c->T * (c->k < c->E_local ? c->k : c->E_local) / c->E_local : 0;
        bool single = avg_rows < 64;
        const char *sel = getenv("MOE_GROUPED_KERNEL");
        if (sel && strcmp(sel, "single") == 0) single = true;
        if (sel && strcmp(sel, "pair") == 0) single = false;
        // "pair2": the pair kernel as two launches (GEMM1, then GEMM2)
        const bool two_launches = sel && strcmp(sel, "pair2") == 0;
        if (two_launches) single = false;
        bool launched = false;
        e = cudaSuccess;
        if (!single)
            e = moe::launch_grouped_swiglu_bf16_pair(x_perm, seg, tpe, w1, w3, w2, h, y_perm, c->D,
                                                     c->H_local, c->e_first, c->E_local,
                                                     rows_alloc_of(c),
                                                     two_launches ? nullptr : w.grouped,
                                                     &w.status->flags, s, &launched);
        if (e == cudaSuccess && !launched)
            e = moe::launch_grouped_swiglu_bf16(x_perm, seg, tpe, w1, w3, w2, h, y_perm, c->D,
                                                c->H_local, c->e_first, c->E_local,
                                                rows_alloc_of(c), &w.status->flags, s);
    }
    else
        e = moe::launch_grouped_swiglu_f32((const float *)x_perm, seg, tpe, (const float *)w1,
                                           (const float *)w3, (const float *)w2, (float *)h,
                                           (float *)y_perm, c->D, c->H_local, c->e_first,
                                           c->E_local, rows_alloc_of(c), &w.status->flags, s);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_grouped_swiglu");
}

// What the FP8 path supports: bf16 activations, D in whole 16-byte rows of
// e4m3 codes and k <= 32 (one lane per slot in the quantising dispatch).
moe_status fp8_supported(const moe_config *c) {
    if (c->dtype != MOE_BF16) return arg_fail("FP8 path: bf16 activations only", MOE_ERR_UNSUPPORTED);
    if (c->D % 16) return arg_fail("FP8 path: D must be a multiple of 16", MOE_ERR_UNSUPPORTED);
    if (c->k > 32) return arg_fail("FP8 path: k <= 32", MOE_ERR_UNSUPPORTED);
    return MOE_OK;
}

moe_status do_grouped_fp8(const moe_config *c, const void *x_perm_q, const float *x_scale,
                          const int32_t *seg, const int32_t *tpe, const void *w1_q,
                          const float *w1_scale, const void *w3_q, const float *w3_scale,
                          const void *w2, void *h, void *y_perm, const StepWs &w, cudaStream_t s) {
    const char *sel = getenv("MOE_GROUPED_KERNEL");
    const bool two_launches = sel && strcmp(sel, "pair2") == 0;
    bool launched = false;
    const cudaError_t e = moe::launch_grouped_swiglu_fp8_pair(
        (const uint8_t *)x_perm_q, x_scale, seg, tpe, (const uint8_t *)w1_q, w1_scale,
        (const uint8_t *)w3_q, w3_scale, w2, h, y_perm, c->D, c->H_local, c->e_first, c->E_local,
        rows_alloc_of(c), two_launches ? nullptr : w.grouped, &w.status->flags, s, &launched);
    if (e != cudaSuccess) return cuda_fail(e, "moe_grouped_swiglu_fp8");
    if (!launched)
        return arg_fail("moe_grouped_swiglu_fp8: too many local experts for the pair kernel",
                        MOE_ERR_UNSUPPORTED);
    return MOE_OK;
}

moe_status do_combine(const moe_config *c, const void *y_perm, const int32_t *row_of,
                      const float *topk_w, void *out, const StepWs &w, cudaStream_t s) {
    cudaError_t e = moe::launch_combine(y_perm, row_of, topk_w, out, c->T, c->D, c->k,
                                        rows_alloc_of(c), c->dtype == MOE_BF16, &w.status->flags, s);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_unpermute_combine");
}

}  // namespace

namespace moe {
void set_last_error(const char *msg) { snprintf(g_last_error, sizeof g_last_error, "%s", msg); }

static std::atomic<uint64_t> g_launches{0};
void count_launch(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }
}  // namespace moe

// ---------------------------------------------------------------------
// exported ABI
// ---------------------------------------------------------------------
MOE_EXPORT const char *moe_status_string(int32_t status) {
    switch (status) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_CAPACITY: return "MOE_ERR_CAPACITY";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
    case MOE_ERR_BAD_ROUTING: return "MOE_ERR_BAD_ROUTING";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    default: return "MOE_ERR_UNKNOWN";
    }
}

MOE_EXPORT const char *moe_last_error_string(void) { return g_last_error; }

MOE_EXPORT int32_t moe_abi_version(void) { return kAbiVersion; }

MOE_EXPORT uint64_t moe_kernel_launches(void) { return moe::g_launches.load(std::memory_order_relaxed); }

MOE_EXPORT moe_status moe_validate_config(const moe_config *cfg) { return validate(cfg); }

MOE_EXPORT int64_t moe_rows_alloc(const moe_config *cfg) {
    return validate(cfg) == MOE_OK ? rows_alloc_of(cfg) : -1;
}

MOE_EXPORT int64_t moe_workspace_size(const moe_config *cfg) {
    return validate(cfg) == MOE_OK ? step_ws_bytes(cfg) : -1;
}

MOE_EXPORT int64_t moe_layer_workspace_size(const moe_config *cfg) {
    return validate(cfg) == MOE_OK ? layer_ws_layout(cfg, nullptr, nullptr) : -1;
}

// The host-buffer form: the layer workspace, then x staging, then out staging.
static int64_t act_bytes(const moe_config *c) {
    return (int64_t)c->T * c->D * elem_bytes(c);
}

MOE_EXPORT int64_t moe_layer_host_workspace_size(const moe_config *cfg) {
    if (validate(cfg) != MOE_OK) return -1;
    return layer_ws_layout(cfg, nullptr, nullptr) + 2 * align_up(act_bytes(cfg));
}

MOE_EXPORT moe_status moe_route_topk(const moe_config *cfg, const void *x, const void *wg,
                                     const float *bias, float *logits_out, int32_t *topk_idx,
                                     float *topk_w, void *ws, size_t ws_bytes,
                                     moe_stream_t stream) {
    moe_status st = validate(cfg);
    if (st != MOE_OK) return st;
    StepWs w;
    if ((st = carve_step(cfg, ws, ws_bytes, &w)) != MOE_OK) return st;
    if (cfg->T == 0) return MOE_OK;
    if (!x || !wg || !topk_idx || !topk_w) return arg_fail("moe_route_topk: NULL tensor");
    const uintptr_t a = cfg->dtype == MOE_BF16 ? 16 : (uintptr_t)elem_bytes(cfg);
    if (!aligned(x, a) || !aligned(wg, a) || !aligned(topk_idx, 4) || !aligned(topk_w, 4) ||
        (bias && !aligned(bias, 4)) || (logits_out && !aligned(logits_out, 4)))
        return arg_fail("moe_route_topk: misaligned tensor");
    return do_route(cfg, x, wg, bias, logits_out, topk_idx, topk_w, w, (cudaStream_t)stream);
}

MOE_EXPORT moe_status moe_permute(const moe_config *cfg, const void *x, const int32_t *topk_idx,
                                  int32_t *tokens_per_expert, int32_t *seg_offsets,
                                  int32_t *row_of, int32_t *token_of_row, void *x_perm, void *ws,
                                  size_t ws_bytes, moe_stream_t stream) {
    moe_status st = validate(cfg);
    if (st != MOE_OK) return st;
    StepWs w;
    if ((st = carve_step(cfg, ws, ws_bytes, &w)) != MOE_OK) return st;
    if (!tokens_per_expert || !seg_offsets) return arg_fail("moe_permute: NULL tensor");
    if (cfg->T > 0 && (!topk_idx || !row_of || !need16(x)))
        return arg_fail("moe_permute: NULL or misaligned tensor");
    if (rows_alloc_of(cfg) > 0 && (!token_of_row || !need16(x_perm)))
        return arg_fail("moe_permute: NULL or misaligned tensor");
    return do_permute(cfg, x, topk_idx, tokens_per_expert, seg_offsets, row_of, token_of_row,
                      x_perm, w, (cudaStream_t)stream);
}

MOE_EXPORT moe_status moe_grouped_swiglu(const moe_config *cfg, const void *x_perm,
                                         const int32_t *seg_offsets,
                                         const int32_t *tokens_per_expert, const void *w1,
                                         const void *w3, const void *w2, void *h, void *y_perm,
                                         void *ws, size_t ws_bytes, moe_stream_t stream) {
    moe_status st = validate(cfg);
    if (st != MOE_OK) return st;
    StepWs w;
    if ((st = carve_step(cfg, ws, ws_bytes, &w)) != MOE_OK) return st;
    if (cfg->E_local == 0 || rows_alloc_of(cfg) == 0) return MOE_OK;
    if (!seg_offsets || !tokens_per_expert) return arg_fail("moe_grouped_swiglu: NULL offsets");
    if (!need16(x_perm) || !need16(w1) || !need16(w3) || !need16(w2) || !need16(h) ||
        !need16(y_perm))
        return arg_fail("moe_grouped_swiglu: NULL or misaligned tensor");
    return do_grouped(cfg, x_perm, seg_offsets, tokens_per_expert, w1, w3, w2, h, y_perm, w,
                      (cudaStream_t)stream);
}

MOE_EXPORT moe_status moe_unpermute_combine(const moe_config *cfg, const void *y_perm,
                                            const int32_t *row_of, const float *topk_w,
                                            void *out, void *ws, size_t ws_bytes,
                                            moe_stream_t stream) {
    moe_status st = validate(cfg);
    if (st != MOE_OK) return st;
    StepWs w;
    if ((st = carve_step(cfg, ws, ws_bytes, &w)) != MOE_OK) return st;
    if (cfg->T == 0) return MOE_OK;
    if (!row_of || !topk_w || !need16(out)) return arg_fail("moe_unpermute_combine: NULL tensor");
    if (rows_alloc_of(cfg) > 0 && !need16(y_perm))
        return arg_fail("moe_unpermute_combine: NULL or misaligned y_perm");
    return do_combine(cfg, y_perm, row_of, topk_w, out, w, (cudaStream_t)stream);
}

MOE_EXPORT moe_status moe_layer_forward(const moe_config *cfg, const void *x, const void *wg,
                                        const float *bias, const void *w1, const void *w3,
                                        const void *w2, void *out, void *ws, size_t ws_bytes,
                                        moe_stream_t stream) {
    moe_status st = validate(cfg);
    if (st != MOE_OK) return st;
    if (!ws) return arg_fail("workspace is NULL", MOE_ERR_WORKSPACE);
    if (!aligned(ws, kAlign)) return arg_fail("workspace must be 256-byte aligned", MOE_ERR_WORKSPACE);
    if ((int64_t)ws_bytes < layer_ws_layout(cfg, nullptr, nullptr))
        return arg_fail("workspace too small for moe_layer_forward", MOE_ERR_WORKSPACE);
    if (cfg->T == 0) return MOE_OK;
    if (!need16(x) || !need16(wg) || !need16(out) || (bias && !aligned(bias, 4)))
        return arg_fail("moe_layer_forward: NULL or misaligned tensor");
    if (cfg->E_local > 0 && (!need16(w1) || !need16(w3) || !need16(w2)))
        return arg_fail("moe_layer_forward: NULL or misaligned expert weights");
    LayerWs L;
    carve_step(cfg, ws, ws_bytes, &L.step);
    layer_ws_layout(cfg, static_cast<char *>(ws), &L);
    cudaStream_t s = (cudaStream_t)stream;
    if ((st = do_route(cfg, x, wg, bias, nullptr, L.topk_idx, L.topk_w, L.step, s)) != MOE_OK)
        return st;
    if ((st = do_permute(cfg, x, L.topk_idx, L.tpe, L.seg_off, L.row_of, L.token_of_row, L.x_perm,
                         L.step, s)) != MOE_OK)
        return st;
    if (cfg->E_local > 0 && rows_alloc_of(cfg) > 0 &&
        (st = do_grouped(cfg, L.x_perm, L.seg_off, L.tpe, w1, w3, w2, L.h, L.y_perm, L.step, s)) !=
            MOE_OK)
        return st;
    return do_combine(cfg, L.y_perm, L.row_of, L.topk_w, out, L.step, s);
}

MOE_EXPORT moe_status moe_layer_forward_host(const moe_config *cfg, const void *x_host,
                                             const void *wg, const float *bias, const void *w1,
                                             const void *w3, const void *w2, void *out_host,
                                             void *ws, size_t ws_bytes, moe_stream_t stream) {
    moe_status st = validate(cfg);
    if (st != MOE_OK) return st;
    if (!ws) return arg_fail("workspace is NULL", MOE_ERR_WORKSPACE);
    if (!aligned(ws, kAlign)) return arg_fail("workspace must be 256-byte aligned", MOE_ERR_WORKSPACE);
    const int64_t lws = layer_ws_layout(cfg, nullptr, nullptr);
    if ((int64_t)ws_bytes < lws + 2 * align_up(act_bytes(cfg)))
        return arg_fail("workspace too small for moe_layer_forward_host", MOE_ERR_WORKSPACE);
    if (cfg->T == 0) return MOE_OK;
    if (!x_host || !out_host) return arg_fail("moe_layer_forward_host: NULL host buffer");
    char *base = static_cast<char *>(ws);
    void *x_dev = base + lws;
    void *out_dev = base + lws + align_up(act_bytes(cfg));
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaMemcpyAsync(x_dev, x_host, (size_t)act_bytes(cfg), cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "moe_layer_forward_host: copy in");
    // A page-locked out_host mapped into the device's address space takes the
    // combine's stores directly: the write-back over the host link then runs
    // under the combine's reads of y_perm instead of after them.  Otherwise
    // the output is staged on the device and copied back.
    void *out_target = out_dev;
    bool direct = false;
    const char *dsel = getenv("MOE_HOST_DIRECT");
    cudaPointerAttributes pa{};
    if (!(dsel && strcmp(dsel, "0") == 0)) {
        if (cudaPointerGetAttributes(&pa, out_host) == cudaSuccess && pa.type == cudaMemoryTypeHost &&
            pa.devicePointer && aligned(pa.devicePointer, 16)) {
            out_target = pa.devicePointer;
            direct = true;
        } else {
            cudaGetLastError();
        }
    }
    if ((st = moe_layer_forward(cfg, x_dev, wg, bias, w1, w3, w2, out_target, ws, (size_t)lws,
                                stream)) != MOE_OK)
        return st;
    if (direct) return MOE_OK;
    e = cudaMemcpyAsync(out_host, out_dev, (size_t)act_bytes(cfg), cudaMemcpyDeviceToHost, s);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_layer_forward_host: copy out");
}

// ---------------------------------------------------------------------
// Host-buffer pipeline: workspace = layer workspace | x slot 0 | x slot 1 |
// out slot 0 | out slot 1.  Per call (slot = call number mod 2):
//   h2d stream:     wait x_free[slot]; copy x_host -> x slot; record x_ready
//   compute stream: wait x_ready; route, permute; record x_free; grouped;
//                   wait out_free[slot]; combine -> out slot; record out_ready
//   d2h stream:     wait out_ready; copy out slot -> out_host; record out_free
// A fresh event counts as complete, so the first use of a slot waits on
// nothing.
// ---------------------------------------------------------------------
struct moe_host_pipeline {
    moe_config cfg;
    char *ws;
    size_t ws_bytes;
    int64_t lws, slot_bytes;
    cudaStream_t h2d, d2h, last_compute;
    cudaEvent_t x_ready[2], x_free[2], out_ready[2], out_free[2];
    unsigned long long calls;
    unsigned long long pending;  // calls submitted since the last sync
};

static int64_t pipeline_ws_bytes(const moe_config *cfg) {
    return layer_ws_layout(cfg, nullptr, nullptr) + 4 * align_up(act_bytes(cfg));
}

MOE_EXPORT int64_t moe_host_pipeline_workspace_size(const moe_config *cfg) {
    return validate(cfg) == MOE_OK ? pipeline_ws_bytes(cfg) : -1;
}

static void pipeline_free(moe_host_pipeline *p) {
    if (!p) return;
    if (p->h2d) cudaStreamSynchronize(p->h2d);
    if (p->d2h) cudaStreamSynchronize(p->d2h);
    for (int i = 0; i < 2; ++i) {
        cudaEvent_t *evs[4] = {&p->x_ready[i], &p->x_free[i], &p->out_ready[i], &p->out_free[i]};
        for (cudaEvent_t *ev : evs)
            if (*ev) cudaEventDestroy(*ev);
    }
    if (p->h2d) cudaStreamDestroy(p->h2d);
    if (p->d2h) cudaStreamDestroy(p->d2h);
    delete p;
}

MOE_EXPORT moe_status moe_host_pipeline_create(const moe_config *cfg, void *ws, size_t ws_bytes,
                                               moe_host_pipeline **out) {
    if (!out) return arg_fail("moe_host_pipeline_create: out is NULL");
    *out = nullptr;
    moe_status st = validate(cfg);
    if (st != MOE_OK) return st;
    if (!ws) return arg_fail("workspace is NULL", MOE_ERR_WORKSPACE);
    if (!aligned(ws, kAlign)) return arg_fail("workspace must be 256-byte aligned", MOE_ERR_WORKSPACE);
    if ((int64_t)ws_bytes < pipeline_ws_bytes(cfg))
        return arg_fail("workspace too small for moe_host_pipeline", MOE_ERR_WORKSPACE);
    moe_host_pipeline *p = new moe_host_pipeline{};
    p->cfg = *cfg;
    p->ws = static_cast<char *>(ws);
    p->ws_bytes = ws_bytes;
    p->lws = layer_ws_layout(cfg, nullptr, nullptr);
    p->slot_bytes = align_up(act_bytes(cfg));
    cudaError_t e = cudaStreamCreateWithFlags(&p->h2d, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->d2h, cudaStreamNonBlocking);
    for (int i = 0; i < 2 && e == cudaSuccess; ++i) {
        cudaEvent_t *evs[4] = {&p->x_ready[i], &p->x_free[i], &p->out_ready[i], &p->out_free[i]};
        for (cudaEvent_t *ev : evs)
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
    }
    if (e != cudaSuccess) {
        pipeline_free(p);
        return cuda_fail(e, "moe_host_pipeline_create");
    }
    *out = p;
    return MOE_OK;
}

MOE_EXPORT moe_status moe_host_pipeline_submit(moe_host_pipeline *p, const void *x_host,
                                               const void *wg, const float *bias, const void *w1,
                                               const void *w3, const void *w2, void *out_host,
                                               moe_stream_t stream) {
    if (!p) return arg_fail("moe_host_pipeline_submit: pipeline is NULL");
    const moe_config *cfg = &p->cfg;
    if (cfg->T == 0) return MOE_OK;
    if (!x_host || !out_host) return arg_fail("moe_host_pipeline_submit: NULL host buffer");
    if (!need16(wg) || (bias && !aligned(bias, 4)))
        return arg_fail("moe_host_pipeline_submit: NULL or misaligned router weights");
    if (cfg->E_local > 0 && (!need16(w1) || !need16(w3) || !need16(w2)))
        return arg_fail("moe_host_pipeline_submit: NULL or misaligned expert weights");
    if (p->pending > 0 && (cudaStream_t)stream != p->last_compute)
        return arg_fail("moe_host_pipeline_submit: calls between two syncs must share one stream");
    const int slot = (int)(p->calls & 1);
    void *x_dev = p->ws + p->lws + slot * p->slot_bytes;
    void *out_dev = p->ws + p->lws + (2 + slot) * p->slot_bytes;
    const size_t n = (size_t)act_bytes(cfg);
    cudaStream_t s = (cudaStream_t)stream;
    LayerWs L;
    carve_step(cfg, p->ws, (size_t)p->lws, &L.step);
    layer_ws_layout(cfg, p->ws, &L);
    cudaError_t e;
    if ((e = cudaStreamWaitEvent(p->h2d, p->x_free[slot], 0)) != cudaSuccess ||
        (e = cudaMemcpyAsync(x_dev, x_host, n, cudaMemcpyHostToDevice, p->h2d)) != cudaSuccess ||
        (e = cudaEventRecord(p->x_ready[slot], p->h2d)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(s, p->x_ready[slot], 0)) != cudaSuccess)
        return cuda_fail(e, "moe_host_pipeline_submit: copy in");
    moe_status st;
    if ((st = do_route(cfg, x_dev, wg, bias, nullptr, L.topk_idx, L.topk_w, L.step, s)) != MOE_OK)
        return st;
    if ((st = do_permute(cfg, x_dev, L.topk_idx, L.tpe, L.seg_off, L.row_of, L.token_of_row,
                         L.x_perm, L.step, s)) != MOE_OK)
        return st;
    if ((e = cudaEventRecord(p->x_free[slot], s)) != cudaSuccess)
        return cuda_fail(e, "moe_host_pipeline_submit: event");
    if (cfg->E_local > 0 && rows_alloc_of(cfg) > 0 &&
        (st = do_grouped(cfg, L.x_perm, L.seg_off, L.tpe, w1, w3, w2, L.h, L.y_perm, L.step, s)) !=
            MOE_OK)
        return st;
    if ((e = cudaStreamWaitEvent(s, p->out_free[slot], 0)) != cudaSuccess)
        return cuda_fail(e, "moe_host_pipeline_submit: event");
    if ((st = do_combine(cfg, L.y_perm, L.row_of, L.topk_w, out_dev, L.step, s)) != MOE_OK)
        return st;
    if ((e = cudaEventRecord(p->out_ready[slot], s)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(p->d2h, p->out_ready[slot], 0)) != cudaSuccess ||
        (e = cudaMemcpyAsync(out_host, out_dev, n, cudaMemcpyDeviceToHost, p->d2h)) != cudaSuccess ||
        (e = cudaEventRecord(p->out_free[slot], p->d2h)) != cudaSuccess)
        return cuda_fail(e, "moe_host_pipeline_submit: copy out");
    p->last_compute = s;
    ++p->calls;
    ++p->pending;
    return MOE_OK;
}

MOE_EXPORT moe_status moe_host_pipeline_sync(moe_host_pipeline *p) {
    if (!p) return arg_fail("moe_host_pipeline_sync: pipeline is NULL");
    cudaError_t e = cudaStreamSynchronize(p->h2d);
    if (e == cudaSuccess) e = cudaStreamSynchronize(p->d2h);
    if (e != cudaSuccess) return cuda_fail(e, "moe_host_pipeline_sync");
    p->pending = 0;
    return moe_get_device_status(p->ws, p->ws_bytes, (moe_stream_t)p->last_compute);
}

MOE_EXPORT void moe_host_pipeline_destroy(moe_host_pipeline *p) { pipeline_free(p); }

MOE_EXPORT int64_t moe_layer_train_workspace_size(const moe_config *cfg) {
    if (validate(cfg) != MOE_OK || train_supported(cfg) != MOE_OK) return -1;
    return train_ws_layout(cfg, nullptr, nullptr);
}

MOE_EXPORT moe_status moe_layer_forward_train(const moe_config *cfg, const void *x, const void *wg,
                                              const float *bias, const void *w1, const void *w3,
                                              const void *w2, void *out, void *ws, size_t ws_bytes,
                                              moe_stream_t stream) {
    moe_status st = validate(cfg);
    if (st != MOE_OK) return st;
    if ((st = train_supported(cfg)) != MOE_OK) return st;
    if (!ws) return arg_fail("workspace is NULL", MOE_ERR_WORKSPACE);
    if (!aligned(ws, kAlign)) return arg_fail("workspace must be 256-byte aligned", MOE_ERR_WORKSPACE);
    if ((int64_t)ws_bytes < train_ws_layout(cfg, nullptr, nullptr))
        return arg_fail("workspace too small for moe_layer_forward_train", MOE_ERR_WORKSPACE);
    if (cfg->T == 0) return MOE_OK;
    if (!need16(x) || !need16(wg) || !need16(out) || (bias && !aligned(bias, 4)) || !need16(w1) ||
        !need16(w3) || !need16(w2))
        return arg_fail("moe_layer_forward_train: NULL or misaligned tensor");
    LayerWs L;
    TrainWs W;
    carve_step(cfg, ws, ws_bytes, &L.step);
    layer_ws_layout(cfg, static_cast<char *>(ws), &L);
    train_ws_layout(cfg, static_cast<char *>(ws), &W);
    cudaStream_t s = (cudaStream_t)stream;
    if ((st = do_route(cfg, x, wg, bias, W.logits, L.topk_idx, L.topk_w, L.step, s)) != MOE_OK)
        return st;
    if ((st = do_permute(cfg, x, L.topk_idx, L.tpe, L.seg_off, L.row_of, L.token_of_row, L.x_perm,
                         L.step, s)) != MOE_OK)
        return st;
    if (rows_alloc_of(cfg) > 0) {
        bool launched = false;
        const char *sel = getenv("MOE_GROUPED_KERNEL");  // "pair2": two launches, as in do_grouped
        const bool two_launches = sel && strcmp(sel, "pair2") == 0;
        cudaError_t e = moe::launch_grouped_swiglu_bf16_pair(
            L.x_perm, L.seg_off, L.tpe, w1, w3, w2, L.h, L.y_perm, cfg->D, cfg->H_local,
            cfg->e_first, cfg->E_local, rows_alloc_of(cfg), two_launches ? nullptr : L.step.grouped,
            &L.step.status->flags, s, &launched, W.gu);
        if (e != cudaSuccess) return cuda_fail(e, "moe_layer_forward_train: grouped SwiGLU");
        if (!launched)
            return arg_fail("moe_layer_forward_train: the CTA-pair kernel cannot run here",
                            MOE_ERR_UNSUPPORTED);
    }
    return do_combine(cfg, L.y_perm, L.row_of, L.topk_w, out, L.step, s);
}

MOE_EXPORT moe_status moe_layer_backward_ex(const moe_config *cfg, const void *x, const void *wg,
                                            const void *w1, const void *w3, const void *w2,
                                            const void *dout, void *dx, float *dwg, float *dbias,
                                            void *dw1, void *dw3, void *dw2, int32_t wgrad_dtype,
                                            void *ws, size_t ws_bytes, moe_stream_t stream) {
    if (wgrad_dtype != MOE_F32 && wgrad_dtype != MOE_BF16)
        return arg_fail("moe_layer_backward_ex: wgrad_dtype must be MOE_F32 or MOE_BF16");
    moe_status st = validate(cfg);
    if (st != MOE_OK) return st;
    if ((st = train_supported(cfg)) != MOE_OK) return st;
    if (!ws) return arg_fail("workspace is NULL", MOE_ERR_WORKSPACE);
    if (!aligned(ws, kAlign)) return arg_fail("workspace must be 256-byte aligned", MOE_ERR_WORKSPACE);
    if ((int64_t)ws_bytes < train_ws_layout(cfg, nullptr, nullptr))
        return arg_fail("workspace too small for moe_layer_backward", MOE_ERR_WORKSPACE);
    if (cfg->T == 0) {
        // no token: dx has no rows, and every parameter gradient is zero
        if (!need16(dwg) || !need16(dw1) || !need16(dw3) || !need16(dw2) ||
            (dbias && !aligned(dbias, 4)))
            return arg_fail("moe_layer_backward: NULL or misaligned tensor");
        cudaStream_t s = (cudaStream_t)stream;
        const size_t wb = wgrad_dtype == MOE_BF16 ? 2 : 4;
        const size_t ehd = (size_t)cfg->E * cfg->H_local * cfg->D;
        cudaError_t e = cudaMemsetAsync(dwg, 0, (size_t)cfg->E * cfg->D * sizeof(float), s);
        if (e == cudaSuccess && dbias) e = cudaMemsetAsync(dbias, 0, cfg->E * sizeof(float), s);
        if (e == cudaSuccess) e = cudaMemsetAsync(dw1, 0, ehd * wb, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(dw3, 0, ehd * wb, s);
        if (e == cudaSuccess) e = cudaMemsetAsync(dw2, 0, ehd * wb, s);
        return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_layer_backward: zero gradients");
    }
    if (!need16(x) || !need16(wg) || !need16(w1) || !need16(w3) || !need16(w2) || !need16(dout) ||
        !need16(dx) || !need16(dwg) || !need16(dw1) || !need16(dw3) || !need16(dw2) ||
        (dbias && !aligned(dbias, 4)))
        return arg_fail("moe_layer_backward: NULL or misaligned tensor");
    LayerWs L;
    TrainWs W;
    carve_step(cfg, ws, ws_bytes, &L.step);
    layer_ws_layout(cfg, static_cast<char *>(ws), &L);
    train_ws_layout(cfg, static_cast<char *>(ws), &W);
    cudaStream_t s = (cudaStream_t)stream;
    const int64_t rows = rows_alloc_of(cfg);
    int *flags = &L.step.status->flags;
    cudaError_t e = moe::launch_combine_bwd(dout, L.y_perm, L.row_of, L.topk_w, W.gy,
                                            W.dw, cfg->T, cfg->D, cfg->k, rows, 1, flags, s);
    if (e != cudaSuccess) return cuda_fail(e, "moe_layer_backward: combine backward");
    if (rows > 0) {
        e = moe::launch_grouped_swiglu_bwd(L.x_perm, L.h, W.gu, W.gy, L.seg_off, L.tpe,
                                           L.token_of_row, w1, w3, w2, W.dgu, W.dxp, dw1, dw3, dw2,
                                           cfg->D, cfg->H_local, cfg->e_first, cfg->E_local, rows,
                                           flags, s, wgrad_dtype == MOE_BF16);
        if (e != cudaSuccess) return cuda_fail(e, "moe_layer_backward: grouped SwiGLU backward");
    }
    // the contiguous layout drops no slot: the router's weight gradient can
    // follow the expert segments
    const moe::RouterSegments segs{L.seg_off, L.tpe, L.token_of_row};
    e = moe::launch_router_bwd(x, wg, W.logits, L.topk_idx, L.topk_w, W.dw, W.dl, W.dxr, dwg, dbias,
                               W.rsplit, cfg->T, cfg->D, cfg->E, cfg->k, cfg->score, cfg->renorm, 1,
                               s, cfg->layout == MOE_LAYOUT_CONTIGUOUS ? &segs : nullptr);
    if (e != cudaSuccess) return cuda_fail(e, "moe_layer_backward: router backward");
    // the router's part of dx: a GEMM where dl is dense, else folded in here
    const bool dense = moe::router_dl_dense(cfg->score, cfg->renorm);
    e = moe::launch_dispatch_bwd(W.dxp, L.row_of, dense ? W.dxr : nullptr, L.topk_idx, W.dl, wg,
                                 cfg->E, dx, cfg->T, cfg->D, cfg->k, rows, 1, s);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_layer_backward: dispatch backward");
}

MOE_EXPORT moe_status moe_quantize_rows_fp8(const void *src, int64_t rows, int32_t cols,
                                           uint8_t *dst, float *scale, moe_stream_t stream) {
    if (rows < 0 || cols <= 0 || cols % 16) return arg_fail("moe_quantize_rows_fp8: bad shape");
    if (rows == 0) return MOE_OK;
    if (!need16(src) || !need16(dst) || !scale || !aligned(scale, 4))
        return arg_fail("moe_quantize_rows_fp8: NULL or misaligned tensor");
    const cudaError_t e = moe::launch_quantize_rows_e4m3(src, rows, cols, nullptr, 1, dst, scale,
                                                         (cudaStream_t)stream);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_quantize_rows_fp8");
}

MOE_EXPORT moe_status moe_permute_fp8(const moe_config *cfg, const void *x,
                                      const int32_t *topk_idx, int32_t *tokens_per_expert,
                                      int32_t *seg_offsets, int32_t *row_of,
                                      int32_t *token_of_row, uint8_t *x_perm_q, float *x_scale,
                                      void *ws, size_t ws_bytes, moe_stream_t stream) {
    moe_status st = validate(cfg);
    if (st != MOE_OK) return st;
    if ((st = fp8_supported(cfg)) != MOE_OK) return st;
    StepWs w;
    if ((st = carve_step(cfg, ws, ws_bytes, &w)) != MOE_OK) return st;
    if (!tokens_per_expert || !seg_offsets) return arg_fail("moe_permute_fp8: NULL tensor");
    if (cfg->T > 0 && (!topk_idx || !row_of || !need16(x)))
        return arg_fail("moe_permute_fp8: NULL or misaligned tensor");
    if (rows_alloc_of(cfg) > 0 &&
        (!token_of_row || !need16(x_perm_q) || !x_scale || !aligned(x_scale, 4)))
        return arg_fail("moe_permute_fp8: NULL or misaligned tensor");
    return do_permute(cfg, x, topk_idx, tokens_per_expert, seg_offsets, row_of, token_of_row,
                      x_perm_q, w, (cudaStream_t)stream, x_scale);
}

MOE_EXPORT moe_status moe_grouped_swiglu_fp8(const moe_config *cfg, const uint8_t *x_perm_q,
                                             const float *x_scale, const int32_t *seg_offsets,
                                             const int32_t *tokens_per_expert,
                                             const uint8_t *w1_q, const float *w1_scale,
                                             const uint8_t *w3_q, const float *w3_scale,
                                             const void *w2, void *h, void *y_perm, void *ws,
                                             size_t ws_bytes, moe_stream_t stream) {
    moe_status st = validate(cfg);
    if (st != MOE_OK) return st;
    if ((st = fp8_supported(cfg)) != MOE_OK) return st;
    StepWs w;
    if ((st = carve_step(cfg, ws, ws_bytes, &w)) != MOE_OK) return st;
    if (cfg->E_local == 0 || rows_alloc_of(cfg) == 0) return MOE_OK;
    if (!seg_offsets || !tokens_per_expert) return arg_fail("moe_grouped_swiglu_fp8: NULL offsets");
    if (!need16(x_perm_q) || !need16(w1_q) || !need16(w3_q) || !need16(w2) || !need16(h) ||
        !need16(y_perm) || !x_scale || !w1_scale || !w3_scale || !aligned(x_scale, 4) ||
        !aligned(w1_scale, 4) || !aligned(w3_scale, 4))
        return arg_fail("moe_grouped_swiglu_fp8: NULL or misaligned tensor");
    return do_grouped_fp8(cfg, x_perm_q, x_scale, seg_offsets, tokens_per_expert, w1_q, w1_scale,
                          w3_q, w3_scale, w2, h, y_perm, w, (cudaStream_t)stream);
}

MOE_EXPORT moe_status moe_layer_forward_fp8(const moe_config *cfg, const void *x, const void *wg,
                                            const float *bias, const uint8_t *w1_q,
                                            const float *w1_scale, const uint8_t *w3_q,
                                            const float *w3_scale, const void *w2, void *out,
                                            void *ws, size_t ws_bytes, moe_stream_t stream) {
    moe_status st = validate(cfg);
    if (st != MOE_OK) return st;
    if ((st = fp8_supported(cfg)) != MOE_OK) return st;
    if (!ws) return arg_fail("workspace is NULL", MOE_ERR_WORKSPACE);
    if (!aligned(ws, kAlign)) return arg_fail("workspace must be 256-byte aligned", MOE_ERR_WORKSPACE);
    if ((int64_t)ws_bytes < layer_ws_layout(cfg, nullptr, nullptr))
        return arg_fail("workspace too small for moe_layer_forward_fp8", MOE_ERR_WORKSPACE);
    if (cfg->T == 0) return MOE_OK;
    if (!need16(x) || !need16(wg) || !need16(out) || (bias && !aligned(bias, 4)))
        return arg_fail("moe_layer_forward_fp8: NULL or misaligned tensor");
    if (cfg->E_local > 0 &&
        (!need16(w1_q) || !need16(w3_q) || !need16(w2) || !w1_scale || !w3_scale ||
         !aligned(w1_scale, 4) || !aligned(w3_scale, 4)))
        return arg_fail("moe_layer_forward_fp8: NULL or misaligned expert weights");
    LayerWs L;
    carve_step(cfg, ws, ws_bytes, &L.step);
    layer_ws_layout(cfg, static_cast<char *>(ws), &L);
    cudaStream_t s = (cudaStream_t)stream;
    if ((st = do_route(cfg, x, wg, bias, nullptr, L.topk_idx, L.topk_w, L.step, s)) != MOE_OK)
        return st;
    if ((st = do_permute(cfg, x, L.topk_idx, L.tpe, L.seg_off, L.row_of, L.token_of_row, L.x_perm,
                         L.step, s, L.x_scale)) != MOE_OK)
        return st;
    if (cfg->E_local > 0 && rows_alloc_of(cfg) > 0 &&
        (st = do_grouped_fp8(cfg, L.x_perm, L.x_scale, L.seg_off, L.tpe, w1_q, w1_scale, w3_q,
                             w3_scale, w2, L.h, L.y_perm, L.step, s)) != MOE_OK)
        return st;
    return do_combine(cfg, L.y_perm, L.row_of, L.topk_w, out, L.step, s);
}

MOE_EXPORT moe_status moe_layer_forward_fused(const moe_config *cfg, const void *x, const void *wg,
                                              const float *bias, const void *w1, const void *w3,
                                              const void *w2, void *out, void *ws,
                                              size_t ws_bytes, moe_stream_t stream) {
    moe_status st = validate(cfg);
    if (st != MOE_OK) return st;
    if (cfg->dtype != MOE_BF16)
        return arg_fail("moe_layer_forward_fused: bf16 only", MOE_ERR_UNSUPPORTED);
    if (cfg->D % 4) return arg_fail("moe_layer_forward_fused: D % 4 != 0", MOE_ERR_UNSUPPORTED);
    // the fp32 accumulator [T, D] lives in the y_perm region (sized to hold it)
    if (cfg->E_local == 0)
        return moe_layer_forward(cfg, x, wg, bias, w1, w3, w2, out, ws, ws_bytes, stream);
    if (!ws) return arg_fail("workspace is NULL", MOE_ERR_WORKSPACE);
    if (!aligned(ws, kAlign)) return arg_fail("workspace must be 256-byte aligned", MOE_ERR_WORKSPACE);
    if ((int64_t)ws_bytes < layer_ws_layout(cfg, nullptr, nullptr))
        return arg_fail("workspace too small for moe_layer_forward_fused", MOE_ERR_WORKSPACE);
    if (cfg->T == 0) return MOE_OK;
    if (!need16(x) || !need16(wg) || !need16(out) || (bias && !aligned(bias, 4)))
        return arg_fail("moe_layer_forward_fused: NULL or misaligned tensor");
    if (!need16(w1) || !need16(w3) || !need16(w2))
        return arg_fail("moe_layer_forward_fused: NULL or misaligned expert weights");
    LayerWs L;
    carve_step(cfg, ws, ws_bytes, &L.step);
    layer_ws_layout(cfg, static_cast<char *>(ws), &L);
    cudaStream_t s = (cudaStream_t)stream;
    float *comb = static_cast<float *>(L.y_perm);
    if ((st = do_route(cfg, x, wg, bias, nullptr, L.topk_idx, L.topk_w, L.step, s)) != MOE_OK)
        return st;
    if ((st = do_permute(cfg, x, L.topk_idx, L.tpe, L.seg_off, L.row_of, L.token_of_row, L.x_perm,
                         L.step, s, nullptr, comb)) != MOE_OK)
        return st;
    const moe::FusedCombine fc{comb, L.token_of_row, L.row_of, L.topk_w, cfg->k};
    const char *sel = getenv("MOE_GROUPED_KERNEL");
    const bool two_launches = sel && strcmp(sel, "pair2") == 0;
    bool launched = false;
    cudaError_t e = moe::launch_grouped_swiglu_bf16_pair(
        L.x_perm, L.seg_off, L.tpe, w1, w3, w2, L.h, L.y_perm, cfg->D, cfg->H_local, cfg->e_first,
        cfg->E_local, rows_alloc_of(cfg), two_launches ? nullptr : L.step.grouped,
        &L.step.status->flags, s, &launched, nullptr, &fc);
    if (e != cudaSuccess) return cuda_fail(e, "moe_layer_forward_fused: grouped SwiGLU");
    if (!launched)
        return arg_fail("moe_layer_forward_fused: too many local experts for the pair kernel",
                        MOE_ERR_UNSUPPORTED);
    e = moe::launch_comb_to_bf16(comb, out, (int64_t)cfg->T * cfg->D, s);
    return e == cudaSuccess ? MOE_OK : cuda_fail(e, "moe_layer_forward_fused: output");
}

moe_status do_grouped_gather(const moe_config *c, const void *x, const int32_t *tor,
                              const int32_t *seg, const int32_t *tpe, const void *w1,
                              const void *w3, const void *w2, void *h, void *y_perm,
                              const StepWs &w, cudaStream_t s) {
    const char *sel = getenv("MOE_GROUPED_KERNEL");
    const bool two_launches = sel && strcmp(sel, "pair2") == 0;
    bool launched = false;
    const moe::GatherA ga{x, tor, c->T};
    const cudaError_t e = moe::launch_grouped_swiglu_bf16_pair(
        nullptr, seg, tpe, w1, w3, w2, h, y_perm, c->D, c->H_local, c->e_first, c->E_local,
        rows_alloc_of(c), two_launches ? nullptr : w.grouped, &w.status->flags, s, &launched,
        nullptr, nullptr, &ga);
    if (e != cudaSuccess) return cuda_fail(e, "moe_grouped_swiglu_gather");
    if (!launched)
        return arg_fail("moe_grouped_swiglu_gather: too many local experts for the pair kernel",
                        MOE_ERR_UNSUPPORTED);
    return MOE_OK;
}

MOE_EXPORT moe_status moe_permute_index(const moe_config *cfg, const int32_t *topk_idx,
                                        int32_t *tokens_per_expert, int32_t *seg_offsets,
                                        int32_t *row_of, int32_t *token_of_row, void *ws,
                                        size_t ws_bytes, moe_stream_t stream) {
    moe_status st = validate(cfg);
    if (st != MOE_OK) return st;
    StepWs w;
    if ((st = carve_step(cfg, ws, ws_bytes, &w)) != MOE_OK) return st;
    if (!tokens_per_expert || !seg_offsets) return arg_fail("moe_permute_index: NULL tensor");
    if (cfg->T > 0 && (!topk_idx || !row_of)) return arg_fail("moe_permute_index: NULL tensor");
    if (rows_alloc_of(cfg) > 0 && !token_of_row)
        return arg_fail("moe_permute_index: NULL token_of_row");
    return do_permute(cfg, nullptr, topk_idx, tokens_per_expert, seg_offsets, row_of,
                      token_of_row, nullptr, w, (cudaStream_t)stream);
}

MOE_EXPORT moe_status moe_grouped_swiglu_gather(const moe_config *cfg, const void *x,
                                                const int32_t *token_of_row,
                                                const int32_t *seg_offsets,
                                                const int32_t *tokens_per_expert, const void *w1,
                                                const void *w3, const void *w2, void *h,
                                                void *y_perm, void *ws, size_t ws_bytes,
                                                moe_stream_t stream) {
    moe_status st = validate(cfg);
    if (st != MOE_OK) return st;
    if (cfg->dtype != MOE_BF16)
        return arg_fail("moe_grouped_swiglu_gather: bf16 only", MOE_ERR_UNSUPPORTED);
    StepWs w;
    if ((st = carve_step(cfg, ws, ws_bytes, &w)) != MOE_OK) return st;
    if (cfg->E_local == 0 || rows_alloc_of(cfg) == 0) return MOE_OK;
    if (!seg_offsets || !tokens_per_expert || !token_of_row)
        return arg_fail("moe_grouped_swiglu_gather: NULL offsets or token_of_row");
    if (!need16(x) || !need16(w1) || !need16(w3) || !need16(w2) || !need16(h) || !need16(y_perm))
        return arg_fail("moe_grouped_swiglu_gather: NULL or misaligned tensor");
    return do_grouped_gather(cfg, x, token_of_row, seg_offsets, tokens_per_expert, w1, w3, w2, h,
                             y_perm, w, (cudaStream_t)stream);
}

MOE_EXPORT moe_status moe_layer_forward_gather(const moe_config *cfg, const void *x,
                                               const void *wg, const float *bias, const void *w1,
                                               const void *w3, const void *w2, void *out,
                                               void *ws, size_t ws_bytes, moe_stream_t stream) {
    moe_status st = validate(cfg);
    if (st != MOE_OK) return st;
    if (cfg->dtype != MOE_BF16)
        return arg_fail("moe_layer_forward_gather: bf16 only", MOE_ERR_UNSUPPORTED);
    if (!ws) return arg_fail("workspace is NULL", MOE_ERR_WORKSPACE);
    if (!aligned(ws, kAlign)) return arg_fail("workspace must be 256-byte aligned", MOE_ERR_WORKSPACE);
    if ((int64_t)ws_bytes < layer_ws_layout(cfg, nullptr, nullptr))
        return arg_fail("workspace too small for moe_layer_forward_gather", MOE_ERR_WORKSPACE);
    if (cfg->T == 0) return MOE_OK;
    if (!need16(x) || !need16(wg) || !need16(out) || (bias && !aligned(bias, 4)))
        return arg_fail("moe_layer_forward_gather: NULL or misaligned tensor");
    if (cfg->E_local > 0 && (!need16(w1) || !need16(w3) || !need16(w2)))
        return arg_fail("moe_layer_forward_gather: NULL or misaligned expert weights");
    LayerWs L;
    carve_step(cfg, ws, ws_bytes, &L.step);
    layer_ws_layout(cfg, static_cast<char *>(ws), &L);
    cudaStream_t s = (cudaStream_t)stream;
    if ((st = do_route(cfg, x, wg, bias, nullptr, L.topk_idx, L.topk_w, L.step, s)) != MOE_OK)
        return st;
    if ((st = do_permute(cfg, nullptr, L.topk_idx, L.tpe, L.seg_off, L.row_of, L.token_of_row,
                         nullptr, L.step, s)) != MOE_OK)
        return st;
    if (cfg->E_local > 0 && rows_alloc_of(cfg) > 0 &&
        (st = do_grouped_gather(cfg, x, L.token_of_row, L.seg_off, L.tpe, w1, w3, w2, L.h,
                                L.y_perm, L.step, s)) != MOE_OK)
        return st;
    return do_combine(cfg, L.y_perm, L.row_of, L.topk_w, out, L.step, s);
}

MOE_EXPORT moe_status moe_layer_backward(const moe_config *cfg, const void *x, const void *wg,
                                         const void *w1, const void *w3, const void *w2,
                                         const void *dout, void *dx, float *dwg, float *dbias,
                                         float *dw1, float *dw3, float *dw2, void *ws,
                                         size_t ws_bytes, moe_stream_t stream) {
    return moe_layer_backward_ex(cfg, x, wg, w1, w3, w2, dout, dx, dwg, dbias, dw1, dw3, dw2,
                                 MOE_F32, ws, ws_bytes, stream);
}

MOE_EXPORT moe_status moe_get_device_status(const void *ws, size_t ws_bytes, moe_stream_t stream) {
    if (!ws || ws_bytes < sizeof(moe::StatusBlock) || !aligned(ws, kAlign))
        return arg_fail("moe_get_device_status: bad workspace", MOE_ERR_WORKSPACE);
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "moe_get_device_status: sync");
    int host[2] = {0, 0};
    e = cudaMemcpy(host, ws, sizeof host, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "moe_get_device_status: read");
    if (host[0] != 0) {
        e = cudaMemset(const_cast<void *>(ws), 0, sizeof host);
        if (e != cudaSuccess) return cuda_fail(e, "moe_get_device_status: clear");
    }
    if (host[0] & moe::FLAG_TIMEOUT) {
        snprintf(g_last_error, sizeof g_last_error, "bounded device wait ran out (CTA %d)", host[1] - 1);
        return MOE_ERR_TIMEOUT;
    }
    if (host[0] & moe::FLAG_LAUNCH) {
        snprintf(g_last_error, sizeof g_last_error,
                 "a kernel was launched without the thread-block cluster it needs; no work done");
        return MOE_ERR_CUDA;
    }
    if (host[0] & moe::FLAG_RANGE) {
        snprintf(g_last_error, sizeof g_last_error,
                 "an expert output is beyond the fp16 range of y_perm (|y| >= 65520)");
        return MOE_ERR_UNSUPPORTED;
    }
    if (host[0] & moe::FLAG_CAPACITY) return MOE_ERR_CAPACITY;
    if (host[0] & moe::FLAG_BAD_ROUTING) return MOE_ERR_BAD_ROUTING;
    return MOE_OK;
}
