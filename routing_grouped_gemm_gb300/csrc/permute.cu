// Dispatch permute and weighted combine.
//
// Page "Expert Parallelism (EP)" (llm-infra-atlas):
//   section 1 -- preprocess computes tokens_per_expert; permute-1 sorts the
//     tokens by expert; combine post-process is the unpermute that reduces
//     the top-k weighted expert outputs back into the original order;
//   section 2 -- the layout contract: each expert's rows are contiguous and
//     every segment is aligned to the grouped GEMM's M tile;
//   section 5 -- permute (gather) and unpermute (scatter-add) are each
//     other's transpose.
//
// The permutation is a stable counting sort (rows of an expert are in
// ascending token order), built without order-dependent atomics so that it
// is bit-identical run to run:
//   count : per block of 256 tokens, per warp of 32 tokens, a bitmask per
//           expert of which lanes route to it; block counts per expert
//   index : recomputes the masks; rank of (t, e) = rows of e in earlier
//           blocks + earlier warps + popc(mask & lanes below); for small
//           count matrices each block also derives the totals and padded
//           segment offsets itself (no separate scan launch), otherwise
//   scan  : one CTA computes tokens_per_expert, the padded segment offsets,
//           each block's first row per local expert and the padding rows
//   copy  : one warp per token reads x[t] once and writes its k copies
//
// For count matrices up to CS_MAX_CELLS the same counting sort runs in two
// launches instead of three:
//   count+scan : each block stores its per-warp masks with the rows of
//                earlier warps of the block; the last block to finish
//                (a self-resetting ticket, no waiting) derives the totals,
//                the padded offsets and each block's first row per expert
//   index+copy : one warp per token ranks its k slots from those tables,
//                copies x[t] to the rows it found and writes a share of the
//                padding entries of token_of_row
#include <algorithm>

#include "common.cuh"
#include "e4m3_row.cuh"
#include "launch.h"

namespace moe {
namespace {

constexpr int PB_TOKENS = 256;  // tokens per count/index block (8 warps x 32)
constexpr int PB_WARPS = PB_TOKENS / 32;

// Slot (t, j) takes part in the layout when its expert id is in [0, E) and
// no earlier slot of the same token names the same expert.
__device__ __forceinline__ bool slot_active(const int *__restrict__ row, int j, int E) {
    const int e = row[j];
    if (e < 0 || e >= E) return false;
    for (int q = 0; q < j; ++q)
        if (row[q] == e) return false;
    return true;
}

__device__ __forceinline__ void build_masks(const int *__restrict__ topk_idx, int T, int k, int E,
                                            uint32_t *s_mask, int *status) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t *m = s_mask + warp * E;
    for (int e = lane; e < E; e += 32) m[e] = 0u;
    __syncwarp();
    const int t = blockIdx.x * PB_TOKENS + warp * 32 + lane;
    if (t < T) {
        const int *row = topk_idx + (size_t)t * k;
        bool bad = false;
        for (int j = 0; j < k; ++j) {
            if (slot_active(row, j, E)) atomicOr(&m[row[j]], 1u << lane);
            else bad = true;
        }
        if (bad) raise_flag(status, FLAG_BAD_ROUTING);
    }
}

__global__ void __launch_bounds__(PB_TOKENS)
permute_count_kernel(const int *__restrict__ topk_idx, int T, int k, int E, int *__restrict__ blk_cnt,
                     int *status) {
    griddep_launch_dependents();  // the next kernel may be scheduled now
    griddep_wait();               // every input of this kernel is complete
    extern __shared__ uint32_t s_mask[];  // [PB_WARPS][E]
    build_masks(topk_idx, T, k, E, s_mask, status);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += PB_TOKENS) {
        int c = 0;
#pragma unroll
        for (int w = 0; w < PB_WARPS; ++w) c += __popc(s_mask[w * E + e]);
        blk_cnt[(size_t)blockIdx.x * E + e] = c;
    }
}

constexpr int SCAN_THREADS = 1024;

// Sum of one expert's counts over the blocks; loads are issued 8 at a time
// so the chain of L2 round trips is nblk / 8 long, not nblk.
__device__ __forceinline__ int sum_blocks(const int *__restrict__ blk_cnt, int nblk, int E, int e) {
    int run = 0, b = 0;
    for (; b + 8 <= nblk; b += 8) {
        int c[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) c[u] = blk_cnt[(size_t)(b + u) * E + e];
#pragma unroll
        for (int u = 0; u < 8; ++u) run += c[u];
    }
    for (; b < nblk; ++b) run += blk_cnt[(size_t)b * E + e];
    return run;
}

__global__ void __launch_bounds__(SCAN_THREADS)
permute_scan_kernel(const int *__restrict__ blk_cnt, int nblk, int E, int e_first, int E_local,
                    int layout, int align_m, int capacity, long long rows_alloc,
                    int *__restrict__ tokens_per_expert, int *__restrict__ seg_offsets,
                    int *__restrict__ blk_base, int *__restrict__ token_of_row, int *status) {
    griddep_launch_dependents();  // the next kernel may be scheduled now
    griddep_wait();               // every input of this kernel is complete
    extern __shared__ int s_int[];
    int *s_cnt = s_int;              // [E]
    int *s_off = s_cnt + E;          // [E_local + 1]  (inclusive scan, shifted)
    const int tid = threadIdx.x;

    for (int e = tid; e < E; e += SCAN_THREADS) {
        const int total = sum_blocks(blk_cnt, nblk, E, e);
        tokens_per_expert[e] = total;
        s_cnt[e] = total;
    }
    __syncthreads();

    // padded segment sizes -> inclusive scan (E_local <= 1024, one per thread)
    if (tid < E_local) {
        const int c = s_cnt[e_first + tid];
        int size;
        if (layout == 1) {
            size = capacity;
            if (c > capacity) raise_flag(status, FLAG_CAPACITY);
        } else {
            size = (c + align_m - 1) / align_m * align_m;
        }
        s_off[tid + 1] = size;
    }
    if (tid == 0) s_off[0] = 0;
    __syncthreads();
    for (int o = 1; o < E_local; o <<= 1) {
        int v = 0;
        if (tid < E_local && tid + 1 > o) v = s_off[tid + 1 - o];
        __syncthreads();
        if (tid < E_local && tid + 1 > o) s_off[tid + 1] += v;
        __syncthreads();
    }
    for (int i = tid; i <= E_local; i += SCAN_THREADS) seg_offsets[i] = s_off[i];

    // local experts: absolute first row of each block's run; padding rows -> -1
    for (int i = tid; i < E_local; i += SCAN_THREADS) {
        const int e = e_first + i;
        const int base = s_off[i];
        int run = base, b = 0;
        for (; b + 8 <= nblk; b += 8) {
            int c[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) c[u] = blk_cnt[(size_t)(b + u) * E + e];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                blk_base[(size_t)(b + u) * E + e] = run;
                run += c[u];
            }
        }
        for (; b < nblk; ++b) {
            blk_base[(size_t)b * E + e] = run;
            run += blk_cnt[(size_t)b * E + e];
        }
        const int used = min(s_cnt[e], s_off[i + 1] - base);
        for (int r = base + used; r < s_off[i + 1]; ++r) token_of_row[r] = -1;
    }
    for (long long r = (long long)s_off[E_local] + tid; r < rows_alloc; r += SCAN_THREADS)
        token_of_row[r] = -1;
}

__global__ void __launch_bounds__(PB_TOKENS)
permute_index_kernel(const int *__restrict__ topk_idx, int T, int k, int E, int e_first,
                     int E_local, const int *__restrict__ blk_base,
                     const int *__restrict__ seg_offsets, int *__restrict__ row_of,
                     int *__restrict__ token_of_row, int *status) {
    griddep_launch_dependents();  // the next kernel may be scheduled now
    griddep_wait();               // every input of this kernel is complete
    extern __shared__ uint32_t s_mask[];  // [PB_WARPS][E]
    build_masks(topk_idx, T, k, E, s_mask, nullptr);
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * PB_TOKENS + warp * 32 + lane;
    if (t >= T) return;
    const int *row = topk_idx + (size_t)t * k;
    const uint32_t below = lanemask_lt();
    for (int j = 0; j < k; ++j) {
        int r = -1;
        if (slot_active(row, j, E)) {
            const int e = row[j];
            const int i = e - e_first;
            if (i >= 0 && i < E_local) {
                int prior = __popc(s_mask[warp * E + e] & below);
                for (int w = 0; w < warp; ++w) prior += __popc(s_mask[w * E + e]);
                const int cand = blk_base[(size_t)blockIdx.x * E + e] + prior;
                if (cand < seg_offsets[i + 1]) {
                    r = cand;
                    token_of_row[cand] = t;
                } else {
                    raise_flag(status, FLAG_CAPACITY);
                }
            }
        }
        row_of[(size_t)t * k + j] = r;
    }
}

// Index kernel with the scan folded in, for small count matrices: every
// block re-derives the per-expert totals, the padded segment offsets and its
// own first row per expert from blk_cnt [nblk][E] (a few KB), so no
// separate single-CTA scan launch sits between count and index.  Block b
// also writes the padding entries of token_of_row for local experts
// i = b, b + nblk, ... and its share of the rows after the last segment;
// block 0 writes tokens_per_expert and seg_offsets.
constexpr int FUSED_MAX_CELLS = 16384;  // nblk * E handled by the fused kernel

__global__ void __launch_bounds__(PB_TOKENS)
permute_index_scan_kernel(const int *__restrict__ topk_idx, int T, int k, int E, int e_first,
                          int E_local, int layout, int align_m, int capacity, long long rows_alloc,
                          const int *__restrict__ blk_cnt, int nblk,
                          int *__restrict__ tokens_per_expert, int *__restrict__ seg_offsets,
                          int *__restrict__ row_of, int *__restrict__ token_of_row, int *status) {
    griddep_launch_dependents();  // the next kernel may be scheduled now
    griddep_wait();               // every input of this kernel is complete
    extern __shared__ uint32_t s_dyn[];
    uint32_t *s_mask = s_dyn;                                       // [PB_WARPS][E]
    int *s_tot = reinterpret_cast<int *>(s_mask + PB_WARPS * E);    // [E]  totals
    int *s_pre = s_tot + E;                                         // [E]  rows in earlier blocks
    int *s_off = s_pre + E;                                         // [E_local + 1] padded offsets
    __shared__ int s_warp_sum[PB_TOKENS / 32];
    const int tid = threadIdx.x;
    const int b = blockIdx.x;

    build_masks(topk_idx, T, k, E, s_mask, nullptr);
    // totals and this block's prefix, per expert
    for (int e = tid; e < E; e += PB_TOKENS) {
        int tot = 0, pre = 0, bb = 0;
        for (; bb + 8 <= nblk; bb += 8) {  // 8 independent loads in flight
            int c[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) c[u] = blk_cnt[(size_t)(bb + u) * E + e];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                tot += c[u];
                pre += (bb + u) < b ? c[u] : 0;
            }
        }
        for (; bb < nblk; ++bb) {
            const int c = blk_cnt[(size_t)bb * E + e];
            tot += c;
            pre += bb < b ? c : 0;
        }
        s_tot[e] = tot;
        s_pre[e] = pre;
    }
    __syncthreads();
    // padded sizes of the local segments -> exclusive scan (thread chunks)
    const int per = (E_local + PB_TOKENS - 1) / PB_TOKENS;
    const int lo = tid * per, hi = min(E_local, lo + per);
    int run = 0;
    for (int i = lo; i < hi; ++i) {
        const int c = s_tot[e_first + i];
        const int size = layout == 1 ? capacity : (c + align_m - 1) / align_m * align_m;
        s_off[i] = size;  // temporarily the size
        run += size;
    }
    const int warp = tid >> 5, lane = tid & 31;
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) s_warp_sum[warp] = incl;
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; ++w) base += s_warp_sum[w];
    int acc = base + incl - run;
    for (int i = lo; i < hi; ++i) {
        const int size = s_off[i];
        s_off[i] = acc;
        acc += size;
    }
    if (tid == PB_TOKENS - 1) s_off[E_local] = acc;
    __syncthreads();

    if (b == 0) {
        for (int e = tid; e < E; e += PB_TOKENS) tokens_per_expert[e] = s_tot[e];
        for (int i = tid; i <= E_local; i += PB_TOKENS) seg_offsets[i] = s_off[i];
        if (layout == 1)
            for (int i = tid; i < E_local; i += PB_TOKENS)
                if (s_tot[e_first + i] > capacity) raise_flag(status, FLAG_CAPACITY);
    }
    // padding rows of this block's share of the local experts
    for (int i = b; i < E_local; i += nblk) {
        const int used = min(s_tot[e_first + i], s_off[i + 1] - s_off[i]);
        for (int r = s_off[i] + used + tid; r < s_off[i + 1]; r += PB_TOKENS) token_of_row[r] = -1;
    }
    // rows after the last segment, split over the blocks
    for (long long r = (long long)s_off[E_local] + (long long)b * PB_TOKENS + tid; r < rows_alloc;
         r += (long long)nblk * PB_TOKENS)
        token_of_row[r] = -1;

    const int t = b * PB_TOKENS + warp * 32 + lane;
    if (t >= T) return;
    const int *row = topk_idx + (size_t)t * k;
    const uint32_t below = lanemask_lt();
    for (int j = 0; j < k; ++j) {
        int r = -1;
        if (slot_active(row, j, E)) {
            const int e = row[j];
            const int i = e - e_first;
            if (i >= 0 && i < E_local) {
                int prior = __popc(s_mask[warp * E + e] & below);
                for (int w = 0; w < warp; ++w) prior += __popc(s_mask[w * E + e]);
                const int cand = s_off[i] + s_pre[e] + prior;
                if (cand < s_off[i + 1]) {
                    r = cand;
                    token_of_row[cand] = t;
                } else {
                    raise_flag(status, FLAG_CAPACITY);
                }
            }
        }
        row_of[(size_t)t * k + j] = r;
    }
}

// ---------------------------------------------------------------------
// two-launch form: count+scan, then index+copy
// ---------------------------------------------------------------------
constexpr int CS_MAX_CELLS = 8192;  // nblk * E staged in the last block's shared memory

// Each block: masks of its 8 warps per expert -> wmeta[(8b + w) E + e] =
// (mask, rows of e in warps 0..w-1 of the block) and blk_cnt[b E + e].  With
// kScan = false that is all (small count matrices: every index+copy block
// derives the offsets from blk_cnt).  Otherwise the
// last block to finish stages blk_cnt in shared memory and writes
// tokens_per_expert, seg_offsets, blk_base[b E_local + i] (the absolute
// first row of block b in local expert i), the padding entries of
// token_of_row and the masked-capacity flag.
template <bool kScan>
__global__ void __launch_bounds__(PB_TOKENS)
permute_count_scan_kernel(const int *__restrict__ topk_idx, int T, int k, int E, int e_first,
                          int E_local, int layout, int align_m, int capacity, long long rows_alloc,
                          int *__restrict__ blk_cnt, int2 *__restrict__ wmeta,
                          int *__restrict__ blk_base, unsigned *__restrict__ ticket,
                          int *__restrict__ tokens_per_expert, int *__restrict__ seg_offsets,
                          int *__restrict__ token_of_row, int *status) {
    griddep_launch_dependents();  // the next kernel may be scheduled now
    griddep_wait();               // every input of this kernel is complete
    extern __shared__ uint32_t s_dyn[];
    uint32_t *s_mask = s_dyn;  // [PB_WARPS][E]
    __shared__ int s_last;
    __shared__ int s_warp_sum[PB_WARPS];
    const int tid = threadIdx.x, b = blockIdx.x, nblk = gridDim.x;

    build_masks(topk_idx, T, k, E, s_mask, status);
    __syncthreads();
    for (int e = tid; e < E; e += PB_TOKENS) {
        int run = 0;
#pragma unroll
        for (int w = 0; w < PB_WARPS; ++w) {
            const uint32_t m = s_mask[w * E + e];
            wmeta[((size_t)b * PB_WARPS + w) * E + e] = make_int2((int)m, run);
            run += __popc(m);
        }
        blk_cnt[(size_t)b * E + e] = run;
    }
    if (!kScan) return;  // the index+copy blocks derive the offsets themselves
    // the block's counts (ordered before thread 0 by the barrier) are
    // released with its ticket; the last block acquires all of them
    __syncthreads();
    if (tid == 0) {
        fence_acq_rel_gpu();
        const bool last = atomicInc(ticket, (unsigned)(nblk - 1)) == (unsigned)(nblk - 1);
        if (last) fence_acq_rel_gpu();
        s_last = last;
    }
    __syncthreads();
    if (!s_last) return;

    int *s_cnt = reinterpret_cast<int *>(s_mask + PB_WARPS * E);  // [nblk][E]
    int *s_tot = s_cnt + (size_t)nblk * E;                           // [E]
    int *s_off = s_tot + E;                                          // [E_local + 1]
    for (int c = tid; c < nblk * E; c += PB_TOKENS) s_cnt[c] = __ldcg(blk_cnt + c);
    __syncthreads();
    for (int e = tid; e < E; e += PB_TOKENS) {
        int tot = 0;
        for (int bb = 0; bb < nblk; ++bb) tot += s_cnt[bb * E + e];
        s_tot[e] = tot;
        tokens_per_expert[e] = tot;
    }
    __syncthreads();
    // padded sizes of the local segments -> exclusive scan (thread chunks)
    const int per = (E_local + PB_TOKENS - 1) / PB_TOKENS;
    const int lo = tid * per, hi = min(E_local, lo + per);
    int run = 0;
    for (int i = lo; i < hi; ++i) {
        const int c = s_tot[e_first + i];
        int size;
        if (layout == 1) {
            size = capacity;
            if (c > capacity) raise_flag(status, FLAG_CAPACITY);
        } else {
            size = (c + align_m - 1) / align_m * align_m;
        }
        s_off[i] = size;  // temporarily the size
        run += size;
    }
    const int warp = tid >> 5, lane = tid & 31;
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) s_warp_sum[warp] = incl;
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; ++w) base += s_warp_sum[w];
    int acc = base + incl - run;
    for (int i = lo; i < hi; ++i) {
        const int size = s_off[i];
        s_off[i] = acc;
        acc += size;
    }
    if (tid == PB_TOKENS - 1) s_off[E_local] = acc;
    __syncthreads();
    for (int i = tid; i <= E_local; i += PB_TOKENS) seg_offsets[i] = s_off[i];
    for (int i = tid; i < E_local; i += PB_TOKENS) {
        const int e = e_first + i;
        int row = s_off[i];
        for (int bb = 0; bb < nblk; ++bb) {
            blk_base[(size_t)bb * E_local + i] = row;
            row += s_cnt[bb * E + e];
        }
    }
    // the padding entries of token_of_row are written by the index+copy
    // kernel, spread over its warps
}

// One warp per token (x_perm NULL: the layout arrays only, no row copy).
// Lane j < k ranks slot j: the slot is active when its
// expert id is in [0, E) and no earlier slot of the token names it; a local
// expert i gets row blk_base[b][i] + (rows of the expert in earlier warps of
// the block) + popc(mask & lanes below), or -1 past the segment's end (the
// masked layout's capacity, flagged by the count kernel).  Then x[t] is read
// once in 16-byte vectors and written to every row found -- or, for the FP8
// dispatch (kFp8), quantised to e4m3 once with one scale per row and the
// codes and scale written to every row found.  Warp t also writes -1 into
// token_of_row for the padding rows of local segments i = t, t + T, ... and
// for its 32-row share of the rows after the last segment.
constexpr int IC_UNROLL = 8;

// Offsets of the small count matrices (kDerive): every block stages the
// per-expert totals and its count block's prefix from blk_cnt [nblk][E],
// scans the padded local segment sizes into seg_offsets in shared memory
// (block 0 also writes tokens_per_expert, seg_offsets and the capacity
// flag), so no block of the count kernel has to wait for the others.
constexpr int DERIVE_MAX_CELLS = 2048;  // nblk * E read by every block

__device__ __forceinline__ void derive_offsets(const int *__restrict__ blk_cnt, int nblk, int b,
                                               int E, int e_first, int E_local, int layout,
                                               int align_m, int capacity, int *s_tot, int *s_pre,
                                               int *s_off, int *s_wsum,
                                               int *__restrict__ tokens_per_expert,
                                               int *__restrict__ seg_offsets, int *status) {
    const int tid = threadIdx.x;
    for (int e = tid; e < E; e += blockDim.x) {
        int tot = 0, pre = 0;
        for (int bb = 0; bb < nblk; ++bb) {
            const int c = __ldcg(blk_cnt + (size_t)bb * E + e);
            tot += c;
            pre += bb < b ? c : 0;
        }
        s_tot[e] = tot;
        s_pre[e] = pre;
    }
    __syncthreads();
    const int nt = blockDim.x;
    const int per = (E_local + nt - 1) / nt;
    const int lo = tid * per, hi = min(E_local, lo + per);
    int run = 0;
    for (int i = lo; i < hi; ++i) {
        const int c = s_tot[e_first + i];
        const int size = layout == 1 ? capacity : (c + align_m - 1) / align_m * align_m;
        s_off[i] = size;  // temporarily the size
        run += size;
    }
    const int warp = tid >> 5, lane = tid & 31;
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) s_wsum[warp] = incl;
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; ++w) base += s_wsum[w];
    int acc = base + incl - run;
    for (int i = lo; i < hi; ++i) {
        const int size = s_off[i];
        s_off[i] = acc;
        acc += size;
    }
    if (tid == nt - 1) s_off[E_local] = acc;
    __syncthreads();
    if (blockIdx.x == 0) {
        for (int e = tid; e < E; e += nt) tokens_per_expert[e] = s_tot[e];
        for (int i = tid; i <= E_local; i += nt) seg_offsets[i] = s_off[i];
        if (layout == 1)
            for (int i = tid; i < E_local; i += nt)
                if (s_tot[e_first + i] > capacity) raise_flag(status, FLAG_CAPACITY);
    }
}

// Tokens (warps) per block of the index+copy kernel.  16: half as many
// blocks derive the offsets from the count matrix as with 8, two blocks per
// SM in one wave.  Fine-grained permute call 25.8-26.5 against 26.5-26.9 us in
// the step (three repeats), 28.0 against 29.4 us alone with a cold L2;
// 32 tokens per block: 26.8-27.6 us.
#ifndef MOE_IC_WARPS
#define MOE_IC_WARPS 16
#endif
constexpr int IC_WARPS = MOE_IC_WARPS;
static_assert(PB_TOKENS % IC_WARPS == 0, "a block's tokens lie in one count block");
template <bool kFp8, bool kDerive>
__global__ void __launch_bounds__(32 * IC_WARPS)
permute_index_copy_kernel(const uint4 *__restrict__ x, const int *__restrict__ topk_idx,
                          const int2 *__restrict__ wmeta, const int *__restrict__ blk_base,
                          const int *__restrict__ seg_offsets_in, int *__restrict__ row_of,
                          int *__restrict__ token_of_row, uint4 *__restrict__ x_perm, int T, int k,
                          int E, int e_first, int E_local, int vpr, float4 *__restrict__ zero_out,
                          int zvpr, const int *__restrict__ tokens_per_expert_in,
                          long long rows_alloc, int cols, float *__restrict__ x_scale,
                          const int *__restrict__ blk_cnt, int nblk, int layout, int align_m,
                          int capacity, int *__restrict__ tpe_out, int *__restrict__ seg_out,
                          int *status) {
    griddep_launch_dependents();  // the next kernel may be scheduled now
    griddep_wait();               // every input of this kernel is complete
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    // offsets: derived here (kDerive; the whole block takes part before any
    // warp leaves), or written by the count kernel's last block
    extern __shared__ int s_dv[];
    const int *seg_offsets = seg_offsets_in;
    const int *tokens_per_expert = tokens_per_expert_in;
    int *s_pre = nullptr;
    if (kDerive) {
        int *s_tot = s_dv;
        s_pre = s_tot + E;
        int *s_off = s_pre + E;
        int *s_wsum = s_off + E_local + 1;
        derive_offsets(blk_cnt, nblk, (blockIdx.x * (blockDim.x >> 5)) / PB_TOKENS, E, e_first,
                       E_local, layout, align_m, capacity, s_tot, s_pre, s_off, s_wsum, tpe_out,
                       seg_out, status);
        seg_offsets = s_off;
        tokens_per_expert = s_tot;
    }
    if (t >= T) return;
    const int e = lane < k ? topk_idx[(size_t)t * k + lane] : -1;
    const uint4 *src = x + (size_t)t * vpr;
    uint4 buf[IC_UNROLL];
    if (!kFp8 && x_perm) {
#pragma unroll
        for (int u = 0; u < IC_UNROLL; ++u) {  // the first chunk of x[t] is in flight meanwhile
            const int v = u * 32 + lane;
            if (v < vpr) buf[u] = __ldcs(src + v);
        }
    }
    bool act = lane < k && e >= 0 && e < E;
    for (int q = 0; q < k; ++q) {
        const int o = __shfl_sync(0xffffffffu, e, q);
        if (q < lane && o == e) act = false;
    }
    const int i = e - e_first;
    int my_row = -1;
    if (act && i >= 0 && i < E_local) {
        const int2 m = wmeta[(size_t)(t >> 5) * E + e];
        const int first = kDerive ? seg_offsets[i] + s_pre[e]
                                  : blk_base[(size_t)(t / PB_TOKENS) * E_local + i];
        const int cand = first + m.y + __popc((uint32_t)m.x & ((1u << (t & 31)) - 1u));
        if (cand < seg_offsets[i + 1]) {
            my_row = cand;
            token_of_row[cand] = t;
        }
    }
    if (lane < k) row_of[(size_t)t * k + lane] = my_row;
    for (int s = t; s < E_local; s += T) {
        const int lo = seg_offsets[s], hi = seg_offsets[s + 1];
        const int used = min(tokens_per_expert[e_first + s], hi - lo);
        for (int r = lo + used + lane; r < hi; r += 32) token_of_row[r] = -1;
    }
    for (long long r = (long long)seg_offsets[E_local] + (long long)t * 32 + lane; r < rows_alloc;
         r += (long long)T * 32)
        token_of_row[r] = -1;
    if (kFp8) {
        quantize_row_e4m3_warp(src, cols, my_row, k, reinterpret_cast<uint8_t *>(x_perm), x_scale,
                               lane);
        return;
    }
    if (zero_out) {  // the fused combine's accumulator row of this token starts at zero
        float4 *z = zero_out + (size_t)t * zvpr;
        for (int v = lane; v < zvpr; v += 32) z[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (!x_perm) return;  // the layout only (GEMM1 gathers the rows from x itself)
    for (int v0 = 0;;) {
        for (int j = 0; j < k; ++j) {
            const int r = __shfl_sync(0xffffffffu, my_row, j);
            if (r < 0) continue;
            uint4 *dst = x_perm + (size_t)r * vpr;
#pragma unroll
            for (int u = 0; u < IC_UNROLL; ++u) {
                const int v = v0 + u * 32 + lane;
                if (v < vpr) dst[v] = buf[u];
            }
        }
        v0 += 32 * IC_UNROLL;
        if (v0 >= vpr) break;
#pragma unroll
        for (int u = 0; u < IC_UNROLL; ++u) {
            const int v = v0 + u * 32 + lane;
            if (v < vpr) buf[u] = __ldcs(src + v);
        }
    }
}

// One warp per token: read x[t] once in 16-byte vectors, write k copies.
constexpr int CP_UNROLL = 4;

__global__ void __launch_bounds__(256)
permute_copy_kernel(const uint4 *__restrict__ x, const int *__restrict__ row_of,
                    uint4 *__restrict__ x_perm, int T, int k, int vpr,
                    float4 *__restrict__ zero_out, int zvpr) {
    griddep_launch_dependents();  // the next kernel may be scheduled now
    griddep_wait();               // every input of this kernel is complete
    const int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (t >= T) return;
    if (zero_out) {  // the fused combine's accumulator row of this token starts at zero
        float4 *z = zero_out + (size_t)t * zvpr;
        for (int v = lane; v < zvpr; v += 32) z[v] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const int my_row = lane < k ? row_of[(size_t)t * k + lane] : -1;
    const uint4 *src = x + (size_t)t * vpr;
    for (int v0 = 0; v0 < vpr; v0 += 32 * CP_UNROLL) {
        uint4 buf[CP_UNROLL];
#pragma unroll
        for (int u = 0; u < CP_UNROLL; ++u) {
            const int v = v0 + u * 32 + lane;
            if (v < vpr) buf[u] = __ldcs(src + v);  // x[t] is read once here
        }
        for (int j = 0; j < k; ++j) {
            const int r = __shfl_sync(0xffffffffu, my_row, j);
            if (r < 0) continue;
            uint4 *dst = x_perm + (size_t)r * vpr;
#pragma unroll
            for (int u = 0; u < CP_UNROLL; ++u) {
                const int v = v0 + u * 32 + lane;
                if (v < vpr) dst[v] = buf[u];
            }
        }
    }
}

// ---------------------------------------------------------------------
// combine: out[t] = sum_j w[t,j] * y_perm[row_of[t,j]]  (fp32, slot order)
// ---------------------------------------------------------------------
constexpr int CB_SLOTS = 8;  // slots whose loads are issued together
// y_perm is read once: its loads are evict-first (ld.global.cs), which
// measured 39 against 45 us with the default policy on the fine-grained step.

#ifndef MOE_COMBINE_PARTS
#define MOE_COMBINE_PARTS 1
#endif
constexpr int CB_PARTS = MOE_COMBINE_PARTS;  // warps per token (1: 45 us, 2: 52 us, 4: 51 us
                                              // on the fine-grained step, fp32 y_perm)
// 32-vector chunks of the row whose loads one warp issues together
#ifndef MOE_COMBINE_CHUNKS
#define MOE_COMBINE_CHUNKS 1
#endif
constexpr int CB_CHUNKS = MOE_COMBINE_CHUNKS;

// Blocks per SM the register budget is capped for.  4 (64 registers, no
// spills): 512 blocks of 8 warps fit in one wave of 152 SMs, where the
// uncapped kernel (84 registers, 3 blocks per SM) ran a second, nearly empty
// wave.  Fine-grained combine 23.1 against 28.2 us in the step (three
// repeats), 27.0 against 30.5 us alone with a cold L2; DeepSeek-V3-shaped
// 175.8 against 190.6 us.  2 blocks per SM, two 32-vector chunks per load
// batch, and two or four warps per token were slower or equal.
#ifndef MOE_COMBINE_MINB
#define MOE_COMBINE_MINB 4
#endif
#ifndef MOE_COMBINE_WPB
#define MOE_COMBINE_WPB 8
#endif
constexpr int CB_WPB = MOE_COMBINE_WPB;  // warps per block

// y_perm is fp16 for bf16 layers (out bf16) and fp32 for fp32 layers.  The
// loop over 16-byte output vectors is uniform across the warp (the shuffles
// inside need every lane), with per-lane predicates for the row tail.
template <bool BF16>
__global__ void __launch_bounds__(32 * CB_WPB, MOE_COMBINE_MINB)
combine_kernel(const void *__restrict__ y, const int *__restrict__ row_of,
               const float *__restrict__ topk_w, void *__restrict__ out, int T, int k, int D,
               long long rows_alloc, int *status) {
    griddep_launch_dependents();  // the next kernel may be scheduled now
    griddep_wait();               // every input of this kernel is complete
    // One warp per (token, part): a token's row is split into CB_PARTS parts
    // of whole 32-vector chunks, so the grid has CB_PARTS x T warps.
    constexpr int EPV = BF16 ? 8 : 4;      // output (and y) elements per 16-byte vector
    const int vpr = D / EPV;               // 16-byte vectors per output row and per y row
    const int nchunk = (vpr + 31) / 32;
    const int lane = threadIdx.x & 31;
    const long long wid = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int t = (int)(wid / CB_PARTS);
    const int part = (int)(wid - (long long)t * CB_PARTS);
    if (t >= T) return;
    const uint4 *yv = static_cast<const uint4 *>(y);
    int my_row = -1;
    float my_w = 0.f;
    if (lane < k) {
        my_row = row_of[(size_t)t * k + lane];
        my_w = topk_w[(size_t)t * k + lane];
        if (my_row < -1 || (long long)my_row >= rows_alloc) {
            if (part == 0) raise_flag(status, FLAG_BAD_ROUTING);
            my_row = -1;
        }
    }
    const int c_lo = part * nchunk / CB_PARTS, c_hi = (part + 1) * nchunk / CB_PARTS;
    for (int c = c_lo; c < c_hi; c += CB_CHUNKS) {
        int v[CB_CHUNKS];
        bool act[CB_CHUNKS];
        float acc[CB_CHUNKS][EPV];
#pragma unroll
        for (int q = 0; q < CB_CHUNKS; ++q) {
            v[q] = (c + q) * 32 + lane;
            act[q] = c + q < c_hi && v[q] < vpr;
#pragma unroll
            for (int i = 0; i < EPV; ++i) acc[q][i] = 0.f;
        }
        for (int j0 = 0; j0 < k; j0 += CB_SLOTS) {
            uint4 val[CB_SLOTS][CB_CHUNKS];
            float wj[CB_SLOTS];
            int rj[CB_SLOTS];
#pragma unroll
            for (int u = 0; u < CB_SLOTS; ++u) {
                const int j = j0 + u;
                rj[u] = __shfl_sync(0xffffffffu, my_row, j & 31);
                wj[u] = __shfl_sync(0xffffffffu, my_w, j & 31);
                if (j >= k) rj[u] = -1;
#pragma unroll
                for (int q = 0; q < CB_CHUNKS; ++q)
                    if (act[q] && rj[u] >= 0) val[u][q] = __ldcs(yv + (size_t)rj[u] * vpr + v[q]);
            }
#pragma unroll
            for (int u = 0; u < CB_SLOTS; ++u) {
#pragma unroll
                for (int q = 0; q < CB_CHUNKS; ++q) {
                    if (!act[q] || rj[u] < 0) continue;
                    float f[EPV];
                    if constexpr (BF16) {
                        const __half2 *h2 = reinterpret_cast<const __half2 *>(&val[u][q]);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float2 p2 = __half22float2(h2[i]);
                            f[2 * i] = p2.x;
                            f[2 * i + 1] = p2.y;
                        }
                    } else {
                        f[0] = __uint_as_float(val[u][q].x);
                        f[1] = __uint_as_float(val[u][q].y);
                        f[2] = __uint_as_float(val[u][q].z);
                        f[3] = __uint_as_float(val[u][q].w);
                    }
#pragma unroll
                    for (int i = 0; i < EPV; ++i) acc[q][i] = fmaf(wj[u], f[i], acc[q][i]);
                }
            }
        }
#pragma unroll
        for (int q = 0; q < CB_CHUNKS; ++q) {
            if (!act[q]) continue;
            uint4 o;
            if (BF16) {
                __nv_bfloat162 *hh = reinterpret_cast<__nv_bfloat162 *>(&o);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    hh[i] = __floats2bfloat162_rn(acc[q][2 * i], acc[q][2 * i + 1]);
            } else {
                o = make_uint4(__float_as_uint(acc[q][0]), __float_as_uint(acc[q][1]),
                               __float_as_uint(acc[q][2]), __float_as_uint(acc[q][3]));
            }
            reinterpret_cast<uint4 *>(out)[(size_t)t * vpr + v[q]] = o;
        }
    }
}


}  // namespace

// Scratch: [0, 64) the count+scan kernel's ticket (zero between calls),
// then blk_cnt [nblk][E], blk_base [nblk][E], and for the two-launch form
// (nblk E <= CS_MAX_CELLS) wmeta [8 nblk][E] of int2.
constexpr int64_t SCR_HEAD = 64;

int64_t permute_scratch_ints(int T, int E) {
    const int64_t cells = (T + PB_TOKENS - 1) / PB_TOKENS * (int64_t)E;
    return SCR_HEAD + 2 * cells + (cells <= CS_MAX_CELLS ? 2 * PB_WARPS * cells : 0);
}

cudaError_t launch_permute(const void *x, const int *topk_idx, int *tokens_per_expert,
                           int *seg_offsets, int *row_of, int *token_of_row, void *x_perm,
                           int T, int D, int E, int k, int e_first, int E_local, int layout,
                           int align_m, int capacity, int64_t rows_alloc, int elem_bytes,
                           int *scratch, int *status, cudaStream_t stream, float *x_scale,
                           float *zero_out) {
    const int nblk = (T + PB_TOKENS - 1) / PB_TOKENS;
    unsigned *ticket = reinterpret_cast<unsigned *>(scratch);
    int *blk_cnt = scratch + SCR_HEAD;
    int *blk_base = blk_cnt + (size_t)nblk * E;
    int2 *wmeta = reinterpret_cast<int2 *>(blk_base + (size_t)nblk * E);
    const size_t mask_smem = sizeof(uint32_t) * PB_WARPS * (size_t)E;
    cudaError_t err;
    if (x_scale && (D % 8 || k > 32)) return cudaErrorInvalidValue;  // before any launch
    if (nblk > 0 && (int64_t)nblk * E <= CS_MAX_CELLS) {
        // small count matrices: the copy blocks derive the offsets themselves
        const bool derive = (int64_t)nblk * E <= DERIVE_MAX_CELLS;
        const size_t smem =
            mask_smem + (derive ? 0 : sizeof(int) * ((size_t)nblk * E + E + E_local + 1));
        const void *ck = derive ? (const void *)permute_count_scan_kernel<false>
                                : (const void *)permute_count_scan_kernel<true>;
        err = ensure_smem(ck, smem);
        if (err != cudaSuccess) return err;
        if ((err = launch_pdl(derive ? permute_count_scan_kernel<false>
                                     : permute_count_scan_kernel<true>,
                              dim3(nblk), dim3(PB_TOKENS), smem, stream,
                              topk_idx, T, k, E, e_first, E_local, layout, align_m, capacity,
                              (long long)rows_alloc, blk_cnt, wmeta, blk_base, ticket,
                              tokens_per_expert, seg_offsets, token_of_row, status)) != cudaSuccess)
            return err;
        count_launch();
        const int warps_per_block = IC_WARPS;
        const int blocks = (T + warps_per_block - 1) / warps_per_block;
        const size_t csmem =
            derive ? sizeof(int) * (2 * (size_t)E + E_local + 1 + warps_per_block) : 0;
        auto copy_kernel = x_scale ? (derive ? permute_index_copy_kernel<true, true>
                                             : permute_index_copy_kernel<true, false>)
                                   : (derive ? permute_index_copy_kernel<false, true>
                                             : permute_index_copy_kernel<false, false>);
        if (csmem > 0 && (err = ensure_smem((const void *)copy_kernel, csmem)) != cudaSuccess)
            return err;
        if ((err = launch_pdl(copy_kernel, dim3(blocks), dim3(32 * warps_per_block), csmem, stream,
                              (const uint4 *)x, topk_idx, (const int2 *)wmeta,
                              (const int *)blk_base, (const int *)seg_offsets, row_of, token_of_row,
                              (uint4 *)x_perm, T, k, E, e_first, E_local, D * elem_bytes / 16,
                              (float4 *)zero_out, D / 4, (const int *)tokens_per_expert,
                              (long long)rows_alloc, D, x_scale, (const int *)blk_cnt, nblk,
                              layout, align_m, capacity, tokens_per_expert, seg_offsets,
                              status)) != cudaSuccess)
            return err;
        count_launch();
        return cudaGetLastError();
    }
    if (nblk > 0) {
        err = ensure_smem((const void *)permute_count_kernel, mask_smem);
        if (err != cudaSuccess) return err;
        if ((err = launch_pdl(permute_count_kernel, dim3(nblk), dim3(PB_TOKENS), mask_smem, stream,
                              topk_idx, T, k, E, blk_cnt, status)) != cudaSuccess)
            return err;
        count_launch();
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    if (nblk > 0 && (int64_t)nblk * E <= FUSED_MAX_CELLS) {
        const size_t smem = mask_smem + sizeof(int) * (2 * (size_t)E + E_local + 1);
        err = ensure_smem((const void *)permute_index_scan_kernel, smem);
        if (err != cudaSuccess) return err;
        if ((err = launch_pdl(permute_index_scan_kernel, dim3(nblk), dim3(PB_TOKENS), smem, stream,
                              topk_idx, T, k, E, e_first, E_local, layout, align_m, capacity,
                              rows_alloc, blk_cnt, nblk, tokens_per_expert, seg_offsets, row_of,
                              token_of_row, status)) != cudaSuccess)
            return err;
        count_launch();
        if ((err = cudaGetLastError()) != cudaSuccess) return err;
    } else {
    const size_t scan_smem = sizeof(int) * ((size_t)E + E_local + 1);
    if ((err = launch_pdl(permute_scan_kernel, dim3(1), dim3(SCAN_THREADS), scan_smem, stream,
                          blk_cnt, nblk, E, e_first, E_local, layout, align_m, capacity, rows_alloc,
                          tokens_per_expert, seg_offsets, blk_base, token_of_row, status)) !=
        cudaSuccess)
        return err;
    count_launch();
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    if (nblk == 0) return cudaSuccess;
    err = ensure_smem((const void *)permute_index_kernel, mask_smem);
    if (err != cudaSuccess) return err;
    if ((err = launch_pdl(permute_index_kernel, dim3(nblk), dim3(PB_TOKENS), mask_smem, stream,
                          topk_idx, T, k, E, e_first, E_local, blk_base, seg_offsets, row_of,
                          token_of_row, status)) != cudaSuccess)
        return err;
    count_launch();
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    }
    if (x_scale)  // FP8 dispatch: the copy quantises each token row once
        return launch_quantize_rows_e4m3(x, T, D, row_of, k, (uint8_t *)x_perm, x_scale, stream);
    if (!x_perm) return cudaSuccess;  // the layout only
    const int vpr = D * elem_bytes / 16;
    const int warps_per_block = 8;
    const int blocks = (T + warps_per_block - 1) / warps_per_block;
    if ((err = launch_pdl(permute_copy_kernel, dim3(blocks), dim3(32 * warps_per_block), 0, stream,
                          (const uint4 *)x, row_of, (uint4 *)x_perm, T, k, vpr,
                          (float4 *)zero_out, D / 4)) != cudaSuccess)
        return err;
    count_launch();
    return cudaGetLastError();
}

namespace {
// out[i] = bf16(comb[i]), four elements per thread step.
__global__ void __launch_bounds__(256)
comb_to_bf16_kernel(const float4 *__restrict__ comb, uint2 *__restrict__ out, long long n4) {
    griddep_launch_dependents();  // the next kernel may be scheduled now
    griddep_wait();               // every input of this kernel is complete
    const long long stride = (long long)gridDim.x * blockDim.x;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) {
        const float4 v = __ldcs(comb + i);
        __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
        __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
        uint2 o;
        o.x = *reinterpret_cast<uint32_t *>(&lo);
        o.y = *reinterpret_cast<uint32_t *>(&hi);
        out[i] = o;
    }
}
}  // namespace

cudaError_t launch_comb_to_bf16(const float *comb, void *out, int64_t n, cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    if (n % 4) return cudaErrorInvalidValue;
    const long long n4 = n / 4;
    const unsigned blocks = (unsigned)std::min<long long>((n4 + 255) / 256, 8 * 152);
    const cudaError_t e = launch_pdl(comb_to_bf16_kernel, dim3(blocks), dim3(256), 0, stream,
                                     (const float4 *)comb, (uint2 *)out, n4);
    if (e == cudaSuccess) count_launch();
    return e;
}

cudaError_t launch_combine(const void *y_perm, const int *row_of, const float *topk_w, void *out,
                           int T, int D, int k, int64_t rows_alloc, int is_bf16, int *status,
                           cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const int warps_per_block = CB_WPB;
    const long long warps = (long long)T * CB_PARTS;
    const int blocks = (int)((warps + warps_per_block - 1) / warps_per_block);
    const cudaError_t err =
        is_bf16 ? launch_pdl(combine_kernel<true>, dim3(blocks), dim3(32 * warps_per_block), 0, stream,
                             y_perm, row_of, topk_w, out, T, k, D, (long long)rows_alloc, status)
                : launch_pdl(combine_kernel<false>, dim3(blocks), dim3(32 * warps_per_block), 0, stream,
                             y_perm, row_of, topk_w, out, T, k, D, (long long)rows_alloc, status);
    if (err != cudaSuccess) return err;
    count_launch();
    return cudaSuccess;
}

}  // namespace moe
