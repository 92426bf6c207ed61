// moe_permute_noalloc: the dispatch permute without a caller workspace.
//
// Who this is for: code that must not allocate device memory at the point
// where it dispatches tokens -- for example a serving loop that runs inside
// a memory pool it does not own, a plugin that a host framework calls with
// only its input and output tensors, or a real-time path where cudaMalloc's
// implicit device synchronisation is not acceptable.  Such callers cannot
// provide the scratch that moe_permute takes through `ws`, so this entry
// point keeps that scratch in a fixed device array that is part of the
// loaded library and exists from module load until the process exits, on
// every GPU that loads the library.
//
// The scratch holds the per-block expert counts and per-block row bases of
// the counting sort (2 * ceil(T / 256) * E int32, plus per-warp masks for
// small count matrices) after a 64-int head whose first word is the count
// kernel's completion ticket.  The ticket must start at zero, which a
// __device__ array does at module load, and every call leaves it at zero;
// everything else is written before it is read.  The array keeps whatever
// the last call left in it.  All calls share it, so two calls whose kernels
// overlap on the GPU (different streams, or different host threads without
// ordering) race on it and produce wrong permutations; issue them in order
// on one stream, or use moe_permute with separate workspaces instead.
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <stdio.h>

#include <mutex>

#include "../../include/moe.h"
#include "launch.h"

#define MOE_EXPORT extern "C" __attribute__((visibility("default")))

namespace {

// Fixed scratch: the 64-int head and 1 MiB of int32.  Holds 2 * ceil(T / 256)
// * E entries, so for example T = 16384 tokens with E <= 2048 experts, or
// T = 131072 tokens with E <= 256 experts.
constexpr size_t kNoAllocScratchInts = 64 + (1u << 20) / sizeof(int);
static __device__ __align__(256) int g_noalloc_scratch[kNoAllocScratchInts];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
int *g_scratch_addr[kMaxDevices] = {nullptr};
CUcontext g_scratch_ctx[kMaxDevices] = {nullptr};

void fail(const char *msg) { moe::set_last_error(msg); }

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);

// The context current on the calling thread (null if the driver entry point
// is unavailable).  Taken through the runtime's driver entry-point query, so
// the library does not link the driver library itself.
CUcontext current_context() {
    static CtxGetCurrentFn fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(ptr);
    }
    CUcontext c = nullptr;
    if (fn && fn(&c) != CUDA_SUCCESS) c = nullptr;
    return c;
}

// Device address of g_noalloc_scratch on the current device, looked up once
// per device (with that device current) and again whenever the device's
// current context is not the one the address was taken in (the module, and
// with it the array, is loaded anew into a context created after
// cudaDeviceReset).  In host code the name g_noalloc_scratch is only a
// host-side stand-in, never a device address.
cudaError_t scratch_address(int **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    const CUcontext ctx = current_context();
    if (!g_scratch_addr[dev] || !ctx || g_scratch_ctx[dev] != ctx) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // makes the device's context current
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = static_cast<int *>(p);
        g_scratch_ctx[dev] = current_context();
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

bool aligned16(const void *p) { return p && (reinterpret_cast<uintptr_t>(p) % 16) == 0; }

}  // namespace

MOE_EXPORT moe_status moe_permute_noalloc(const moe_config *cfg, const void *x,
                                          const int32_t *topk_idx, int32_t *tokens_per_expert,
                                          int32_t *seg_offsets, int32_t *row_of,
                                          int32_t *token_of_row, void *x_perm,
                                          int32_t *device_flags, moe_stream_t stream) {
    moe_status st = moe_validate_config(cfg);
    if (st != MOE_OK) return st;
    const int64_t need = moe::permute_scratch_ints(cfg->T, cfg->E);
    if (need > (int64_t)kNoAllocScratchInts) {
        char msg[200];
        snprintf(msg, sizeof msg,
                 "moe_permute_noalloc: the counting sort needs %lld ints, more than the fixed "
                 "scratch of %lld ints; use moe_permute with a workspace",
                 (long long)need, (long long)kNoAllocScratchInts);
        fail(msg);
        return MOE_ERR_UNSUPPORTED;
    }
    const int64_t rows = moe_rows_alloc(cfg);
    if (!tokens_per_expert || !seg_offsets ||
        (cfg->T > 0 && (!topk_idx || !row_of || !aligned16(x))) ||
        (rows > 0 && (!token_of_row || !aligned16(x_perm)))) {
        fail("moe_permute_noalloc: NULL or misaligned tensor");
        return MOE_ERR_INVALID_ARG;
    }
    int *scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) {
        char msg[200];
        snprintf(msg, sizeof msg, "moe_permute_noalloc: set-up: %s", cudaGetErrorString(e));
        fail(msg);
        return MOE_ERR_CUDA;
    }
    const int elem = cfg->dtype == MOE_BF16 ? 2 : 4;
    e = moe::launch_permute(x, topk_idx, tokens_per_expert, seg_offsets, row_of, token_of_row,
                            x_perm, cfg->T, cfg->D, cfg->E, cfg->k, cfg->e_first, cfg->E_local,
                            cfg->layout, cfg->align_m, cfg->capacity, rows, elem, scratch,
                            device_flags, (cudaStream_t)stream);
    if (e != cudaSuccess) {
        char msg[200];
        snprintf(msg, sizeof msg, "moe_permute_noalloc: %s", cudaGetErrorString(e));
        fail(msg);
        return MOE_ERR_CUDA;
    }
    return MOE_OK;
}
