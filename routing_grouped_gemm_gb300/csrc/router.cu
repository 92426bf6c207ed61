// Router: gating logits, top-k selection and routing weights.
//
// Page "Expert Parallelism (EP)" (llm-infra-atlas), section 1: the router
// computes logits = x . W_g^T ([T, E]) and then "top-k + score_func" gives
// the routing probabilities and the routing map.
//
// Two implementations of the same contract:
//   * bf16 with E <= 256: the logits are a dense contraction, so they run on
//     the tensor cores (tcgen05, TMA-fed, fp32 accumulation in TMEM), split
//     along D so that every SM takes part; a second kernel adds the fp32
//     partials in a fixed split order (deterministic), adds the bias and
//     selects the top-k with one warp per token;
//   * otherwise (fp32, where TF32 would miss the 1e-4 accuracy, or E > 256):
//     one fused SIMT kernel -- a CTA accumulates 32 tokens' logits for all E
//     in fp32 FFMA, keeps them in shared memory, and one warp per token
//     selects the top-k.
#include <cuda.h>

#include <stdlib.h>
#include <string.h>

#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

constexpr int RT_TOKENS = 32;   // tokens per CTA
constexpr int RT_ECHUNK = 128;  // experts per logits pass
constexpr int RT_BK = 32;       // reduction slice
constexpr int RT_THREADS = 256;
constexpr int SX_LD = RT_TOKENS + 1;  // padded strides keep the transposing
constexpr int SW_LD = RT_ECHUNK + 1;  // shared-memory stores conflict-free
static_assert(RT_TOKENS * RT_BK % RT_THREADS == 0 && RT_ECHUNK * RT_BK % RT_THREADS == 0,
              "each thread stages whole shares of the x and W_g slices");

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
    return __bfloat162float(v);
}

// Top-k of one token's E keys (in shared memory) by one warp: k rounds of a
// warp-wide arg-max in selection order (larger key first, equal keys by
// lower expert index, NaN after every number, -0 equal to +0), then the
// routing weights: softmax over all E (or sigmoid) of the chosen keys,
// divided by their sum when renormalising.  Lane i owns experts i, i+32, ...
// (E <= 1024); the winner of round j is kept by lane j, which computes and
// writes slot j.
//
// Group-limited routing (n_group > 1; page "Expert Parallelism (EP)",
// section 3): first each of the n_group groups of E/n_group consecutive
// experts is scored by the fp32 sum of its m = k/topk_group largest keys
// (added in selection order), the topk_group best groups are kept (ties to
// the lower group, NaN last), and the k rounds only consider their experts.

// The selection order as one unsigned 64-bit number, larger = chosen first.
// High word: the key's binary32 bits mapped order-preservingly onto unsigned
// integers (negative values bit-inverted, the sign bit set on the others),
// with -0 folded onto +0 and NaN mapped to 0, below every number.  Low word:
// ~e, so that of two equal keys the lower expert index is larger.  0 means
// "no candidate": a real candidate's low word ~e is nonzero.
__device__ __forceinline__ uint64_t sel_key(float v, int e) {
    uint32_t b = __float_as_uint(v);
    b = b == 0x80000000u ? 0u : b;
    uint32_t u = (b & 0x80000000u) ? ~b : (b | 0x80000000u);
    u = v != v ? 0u : u;
    return ((uint64_t)u << 32) | (uint64_t)(~(uint32_t)e);
}

// Warp-wide maximum of the lanes' selection keys (two redux.sync steps: the
// high words, then the low words of the lanes that hold the largest high
// word); every lane gets the result.
__device__ __forceinline__ uint64_t warp_max_key(uint64_t x) {
    const uint32_t hi = (uint32_t)(x >> 32);
    const uint32_t mhi = __reduce_max_sync(0xffffffffu, hi);
    const uint32_t mlo = __reduce_max_sync(0xffffffffu, hi == mhi ? (uint32_t)x : 0u);
    return ((uint64_t)mhi << 32) | mlo;
}

__device__ __forceinline__ int key_expert(uint64_t x) { return x ? (int)~(uint32_t)x : -1; }

// KC: selection keys cached in registers per lane (E <= 32 KC); the keys are
// formed once, and each round is a masked maximum over the cache plus the
// warp-wide maximum.
template <int KC>
__device__ __forceinline__ void warp_topk_cached(const float *l, int E, int k, int score,
                                                 int renorm, int n_group, int topk_group, int t,
                                                 int *__restrict__ topk_idx,
                                                 float *__restrict__ topk_w, int *status,
                                                 int lane) {
    uint64_t key[KC];  // key[q]: expert lane + 32 q, 0 when absent
    bool any_nan = false;
#pragma unroll
    for (int q = 0; q < KC; ++q) {
        const int e = lane + 32 * q;
        const float v = e < E ? l[e] : 0.f;
        any_nan |= v != v;
        key[q] = e < E ? sel_key(v, e) : 0ull;
    }
    if (__any_sync(0xffffffffu, any_nan) && lane == 0) raise_flag(status, FLAG_BAD_ROUTING);

    const bool grouped = n_group > 1;
    uint32_t avail = 0xffffffffu;  // bit q: expert lane + 32 q may still be chosen
    if (grouped) {
        const int gsz = E / n_group;
        const int m = k / topk_group;
        float my_score = 0.f;  // lane g: score of group g
        for (int g = 0; g < n_group; ++g) {
            const int e0 = g * gsz;
            uint32_t in = 0;  // bit q: expert lane + 32 q is in group g
#pragma unroll
            for (int q = 0; q < KC; ++q) {
                const int e = lane + 32 * q;
                if (e >= e0 && e < e0 + gsz) in |= 1u << q;
            }
            float sum = 0.f;
            for (int i = 0; i < m; ++i) {
                uint64_t best = 0;
#pragma unroll
                for (int q = 0; q < KC; ++q) {
                    const uint64_t c = ((in >> q) & 1u) ? key[q] : 0ull;
                    best = c > best ? c : best;
                }
                const int be = key_expert(warp_max_key(best));
                if (be >= 0 && (be & 31) == lane) in &= ~(1u << (be >> 5));
                sum += be >= 0 ? l[be] : 0.f;
            }
            if (lane == g) my_score = sum;
        }
        uint32_t allowed = 0;  // bit g: group g may be chosen
        for (int r = 0; r < topk_group; ++r) {
            const uint64_t c =
                (lane < n_group && !(allowed & (1u << lane))) ? sel_key(my_score, lane) : 0ull;
            const int bg = key_expert(warp_max_key(c));
            if (bg >= 0) allowed |= 1u << bg;
        }
        avail = 0;
#pragma unroll
        for (int q = 0; q < KC; ++q) {
            const int e = lane + 32 * q;
            if (e < E && ((allowed >> (e / gsz)) & 1u)) avail |= 1u << q;
        }
    }

    int my_e = -1;  // slot `lane`'s expert and key (lanes < k)
    float my_v = 0.f, top = 0.f;
    for (int j = 0; j < k; ++j) {
        uint64_t best = 0;
#pragma unroll
        for (int q = 0; q < KC; ++q) {
            const uint64_t c = ((avail >> q) & 1u) ? key[q] : 0ull;
            best = c > best ? c : best;
        }
        const int be = key_expert(warp_max_key(best));
        const float bv = be >= 0 ? l[be] : 0.f;
        if (be >= 0 && (be & 31) == lane) avail &= ~(1u << (be >> 5));
        if (lane == j) { my_e = be; my_v = bv; }
        if (j == 0) top = bv;  // the largest chosen key (unless NaN)
    }
    if (grouped && score == 0 && !renorm) {
        // softmax over all E: shift by the largest key of all, which may lie
        // in a group that was not chosen
        uint64_t best = 0;
#pragma unroll
        for (int q = 0; q < KC; ++q) best = key[q] > best ? key[q] : best;
        const int be = key_expert(warp_max_key(best));
        top = be >= 0 ? l[be] : 0.f;
    }

    float p = 0.f;
    if (lane < k) p = (score == 0) ? expf(my_v - top) : 1.f / (1.f + expf(-my_v));
    float div = 1.f;
    if (renorm) {
        float sum = p;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        div = sum;
    } else if (score == 0) {
        float sum = 0.f;
        for (int e = lane; e < E; e += 32) sum += expf(l[e] - top);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        div = sum;
    }
    if (lane < k) {
        topk_idx[(size_t)t * k + lane] = my_e;
        topk_w[(size_t)t * k + lane] = p / div;
    }
}

// EMAX: the largest E the calling kernel handles (256 or 1024).
template <int EMAX>
__device__ void warp_topk_weights(const float *l, int E, int k, int score, int renorm,
                                  int n_group, int topk_group, int t,
                                  int *__restrict__ topk_idx, float *__restrict__ topk_w,
                                  int *status, int lane) {
    if (E <= 64)
        warp_topk_cached<2>(l, E, k, score, renorm, n_group, topk_group, t, topk_idx, topk_w,
                            status, lane);
    else if (EMAX <= 256 || E <= 256)
        warp_topk_cached<8>(l, E, k, score, renorm, n_group, topk_group, t, topk_idx, topk_w,
                            status, lane);
    else
        warp_topk_cached<32>(l, E, k, score, renorm, n_group, topk_group, t, topk_idx, topk_w,
                             status, lane);
}

template <typename T>
__global__ void __launch_bounds__(RT_THREADS)
router_topk_kernel(const T *__restrict__ x, const T *__restrict__ wg, const float *__restrict__ bias,
                   float *__restrict__ logits_out, int *__restrict__ topk_idx,
                   float *__restrict__ topk_w, int Tn, int D, int E, int k, int score, int renorm,
                   int n_group, int topk_group, int *status) {
    griddep_launch_dependents();  // the next kernel may be scheduled now
    griddep_wait();               // every input of this kernel is complete
    extern __shared__ float smem[];
    float *s_logit = smem;                              // [RT_TOKENS][E]
    float *s_x = s_logit + RT_TOKENS * E;               // [RT_BK][SX_LD]
    float *s_w = s_x + RT_BK * SX_LD;                   // [RT_BK][SW_LD]

    const int tid = threadIdx.x;
    const int t0 = blockIdx.x * RT_TOKENS;
    const int ty = tid / 32;   // token group: tokens ty*4 .. ty*4+3
    const int tx = tid % 32;   // experts tx + 32*i, i < 4

    for (int e0 = 0; e0 < E; e0 += RT_ECHUNK) {
        float acc[4][4];
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
            for (int b = 0; b < 4; ++b) acc[a][b] = 0.f;

        // the next D slice is loaded into registers while this one is
        // multiplied out of shared memory
        constexpr int XPER = RT_TOKENS * RT_BK / RT_THREADS, WPER = RT_ECHUNK * RT_BK / RT_THREADS;
        float rx[XPER], rw[WPER];
        auto load_slices = [&](int d0) {
#pragma unroll
            for (int q = 0; q < XPER; ++q) {  // x slice: 32 tokens x 32 d
                const int i = tid + q * RT_THREADS;
                const int tt = i / RT_BK, dd = i % RT_BK;
                const int t = t0 + tt, d = d0 + dd;
                rx[q] = (t < Tn && d < D) ? to_f32(x[(size_t)t * D + d]) : 0.f;
            }
#pragma unroll
            for (int q = 0; q < WPER; ++q) {  // W_g slice: 128 experts x 32 d
                const int i = tid + q * RT_THREADS;
                const int ee = i / RT_BK, dd = i % RT_BK;
                const int e = e0 + ee, d = d0 + dd;
                rw[q] = (e < E && d < D) ? to_f32(wg[(size_t)e * D + d]) : 0.f;
            }
        };
        load_slices(0);
        for (int d0 = 0; d0 < D; d0 += RT_BK) {
            // both slices stored transposed: [d][token] and [d][expert]
#pragma unroll
            for (int q = 0; q < XPER; ++q) {
                const int i = tid + q * RT_THREADS;
                s_x[(i % RT_BK) * SX_LD + i / RT_BK] = rx[q];
            }
#pragma unroll
            for (int q = 0; q < WPER; ++q) {
                const int i = tid + q * RT_THREADS;
                s_w[(i % RT_BK) * SW_LD + i / RT_BK] = rw[q];
            }
            __syncthreads();
            if (d0 + RT_BK < D) load_slices(d0 + RT_BK);
#pragma unroll 8
            for (int dd = 0; dd < RT_BK; ++dd) {
                float xv[4], wv[4];
#pragma unroll
                for (int a = 0; a < 4; ++a) xv[a] = s_x[dd * SX_LD + ty * 4 + a];
#pragma unroll
                for (int b = 0; b < 4; ++b) wv[b] = s_w[dd * SW_LD + tx + 32 * b];
#pragma unroll
                for (int a = 0; a < 4; ++a)
#pragma unroll
                    for (int b = 0; b < 4; ++b) acc[a][b] = fmaf(xv[a], wv[b], acc[a][b]);
            }
            __syncthreads();
        }
#pragma unroll
        for (int a = 0; a < 4; ++a) {
            const int tt = ty * 4 + a, t = t0 + tt;
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int e = e0 + tx + 32 * b;
                if (e < E) {
                    float v = acc[a][b];
                    if (bias) v += bias[e];
                    s_logit[tt * E + e] = v;
                    if (logits_out && t < Tn) logits_out[(size_t)t * E + e] = v;
                }
            }
        }
    }
    __syncthreads();

    // top-k: one warp per token, lanes own experts lane, lane+32, ...
    const int warp = tid / 32, lane = tid % 32;
    for (int tt = warp; tt < RT_TOKENS; tt += RT_THREADS / 32) {
        const int t = t0 + tt;
        if (t >= Tn) break;
        warp_topk_weights<1024>(s_logit + tt * E, E, k, score, renorm, n_group, topk_group, t,
                                topk_idx, topk_w, status, lane);
    }
}


// ---------------------------------------------------------------------
// tensor-core logits: part[s][e][t] = sum over D-slice s of x[t,:] wg[e,:]
// ---------------------------------------------------------------------
constexpr int RC_BM = 128, RC_BK = 64, RC_STAGES = 4, RC_THREADS = 192;
constexpr int RC_NBARS = 2 * RC_STAGES + 2;  // full, empty, done (+1 spare)
// The cluster form runs extra warps that only join the reduction and top-k.
#ifndef MOE_ROUTER_CL_WARPS
#define MOE_ROUTER_CL_WARPS 16
#endif
constexpr int RC_CL_THREADS = 32 * MOE_ROUTER_CL_WARPS;
static_assert(MOE_ROUTER_CL_WARPS >= 6, "warps 0-5 hold the pipeline roles");
constexpr int RC_A_BYTES = RC_BM * RC_BK * 2;  // 16 KB

struct RouterTcParams {
    int T, E, n_pad, nk, kps;
    float *part;  // [splits][E][T] (two-kernel form)
    int *status;
    // one-kernel (cluster) form: the top-k arguments
    const float *bias;
    float *logits_out;
    int *topk_idx;
    float *topk_w;
    int k, score, renorm, splits;
    int n_group, topk_group;
};

__host__ __device__ inline int rc_stage_bytes(int n_pad) { return RC_A_BYTES + n_pad * RC_BK * 2; }

inline size_t rc_smem_bytes(int n_pad) {
    return 1024 + (size_t)RC_STAGES * rc_stage_bytes(n_pad) + RC_NBARS * sizeof(uint64_t) + 16;
}

__host__ __device__ inline uint32_t rc_tmem_cols(int n_pad) {
    uint32_t c = 32;
    while (c < (uint32_t)n_pad) c <<= 1;
    return c;
}

// kCluster = false: the CTA writes its fp32 partial to part[split][e][t] and a
// second kernel reduces.  kCluster = true: the `splits` CTAs of one m-tile
// form a cluster; each stages its partial in its own shared memory (the
// operand ring, free once the MMAs are done), and after a cluster barrier
// CTA r sums the partials of its share of the 128 tokens from all CTAs
// through distributed shared memory, in split order, then selects the top-k.
template <bool kCluster>
__global__ void __launch_bounds__(kCluster ? RC_CL_THREADS : RC_THREADS)
router_logits_tc_kernel(const __grid_constant__ CUtensorMap tmX,
                        const __grid_constant__ CUtensorMap tmW, const RouterTcParams p) {
    griddep_launch_dependents();  // the next kernel may be scheduled now
    griddep_wait();               // every input of this kernel is complete
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *ring = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
    const int stage_bytes = rc_stage_bytes(p.n_pad);
    uint64_t *bars = reinterpret_cast<uint64_t *>(ring + RC_STAGES * stage_bytes);
    uint64_t *full = bars;                 // [RC_STAGES]
    uint64_t *empty = bars + RC_STAGES;    // [RC_STAGES]
    uint64_t *done = bars + 2 * RC_STAGES; // accumulator complete
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + RC_NBARS);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.x * RC_BM;
    const int split = kCluster ? (int)cluster_ctarank() : (int)blockIdx.y;
    const int kb0 = split * p.kps;
    const int kb1 = min(p.nk, kb0 + p.kps);
    const uint32_t ncols = rc_tmem_cols(p.n_pad);

    if (warp == 0 && lane == 0) {
        for (int s = 0; s < RC_STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(done, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
        prefetch_tmap(&tmX);
        prefetch_tmap(&tmW);
    } else if (warp == 1) {
        tmem_alloc(tmem_slot, ncols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            int s = 0;
            uint32_t ph = 0;
            int last_parity[RC_STAGES];
            for (int q = 0; q < RC_STAGES; ++q) last_parity[q] = -1;
            bool ok = true;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!mbar_wait_bounded(&empty[s], ph ^ 1u, abort_flag)) { ok = false; break; }
                mbar_arrive_expect_tx(&full[s], (uint32_t)stage_bytes);
                uint8_t *sa = ring + s * stage_bytes;
                tma_load_2d(sa, &tmX, &full[s], kb * RC_BK, m0);
                tma_load_2d(sa + RC_A_BYTES, &tmW, &full[s], kb * RC_BK, 0);
                last_parity[s] = (int)ph;
                if (++s == RC_STAGES) { s = 0; ph ^= 1u; }
            }
            if (!ok) {
                volatile int local_abort = 0;
                for (int q = 0; q < RC_STAGES; ++q)
                    if (last_parity[q] >= 0)
                        mbar_wait_bounded(&full[q], (uint32_t)last_parity[q], &local_abort);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = idesc_bf16_f32(RC_BM, p.n_pad);
            int s = 0;
            uint32_t ph = 0;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!mbar_wait_bounded(&full[s], ph, abort_flag)) break;
                tc_fence_after();
                const uint32_t a_addr = smem_u32(ring + s * stage_bytes);
                const uint32_t b_addr = a_addr + RC_A_BYTES;
#pragma unroll
                for (int kk = 0; kk < RC_BK / 16; ++kk)
                    tc_mma_f16(tmem_base, sdesc_kmajor_sw128(a_addr + kk * 32),
                               sdesc_kmajor_sw128(b_addr + kk * 32), idesc,
                               (kb > kb0 || kk > 0) ? 1u : 0u);
                tc_commit(&empty[s]);
                if (++s == RC_STAGES) { s = 0; ph ^= 1u; }
            }
            tc_commit(done);  // arrives once every MMA above has completed
            // every MMA issued here completes before TMEM is freed, even if
            // the epilogue gave up waiting
            volatile int local_abort = 0;
            mbar_wait_bounded(done, 0u, &local_abort);
        }
    } else if (warp < 6) {
        const int q = warp & 3;
        const bool got = mbar_wait_bounded(done, 0u, abort_flag);
        if (__all_sync(0xffffffffu, got) && !*abort_flag) {
            tc_fence_after();
            if (kCluster) {
                // this CTA's partial into its own shared memory, [token][e]
                // with an odd row stride (conflict-free for these writes and
                // for the peers' row reads)
                float *sp = reinterpret_cast<float *>(ring);
                const int ld = p.n_pad + 1;
                const int tl = q * 32 + lane;
                for (int c0 = 0; c0 < p.n_pad; c0 += 32) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)c0, v);
                    tc_wait_ld();
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (c0 + i < p.n_pad) sp[tl * ld + c0 + i] = __uint_as_float(v[i]);
                }
            } else {
            // partials are token-minor, part[split][e][t]: for each expert
            // column the warp's 32 lanes (32 consecutive tokens) write one
            // contiguous 128-byte line
            const int t = m0 + q * 32 + lane;
            float *pcol = p.part + (size_t)split * p.E * p.T + t;
            for (int c0 = 0; c0 < p.n_pad; c0 += 32) {
                uint32_t v[32];
                tmem_ld_32x32b_x32(tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)c0, v);
                tc_wait_ld();
                if (t < p.T) {
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (c0 + i < p.E) pcol[(size_t)(c0 + i) * p.T] = __uint_as_float(v[i]);
                }
            }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) {
        raise_flag(p.status, FLAG_TIMEOUT);
        atomicCAS(p.status + 1, 0, 1 + blockIdx.x);
        // loads issued for stages the MMA warp never consumed land first
        settle_inflight_copies();
    }
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, ncols);
    }
    if (kCluster) {
        cluster_sync();  // every CTA's partial is in its shared memory
        const int S = p.splits;
        const int per = (RC_BM + S - 1) / S;
        const int tl0 = split * per, tl1 = min(RC_BM, tl0 + per);
        const int ld = p.n_pad + 1;
        const uint32_t sp_local = smem_u32(ring);
        // per-warp key row after the partial buffer
        float *key = reinterpret_cast<float *>(ring) + (size_t)RC_BM * ld + warp * p.E;
        const int nwarps = (int)(blockDim.x >> 5);
        for (int tl = tl0 + warp; tl < tl1; tl += nwarps) {
            const int t = m0 + tl;
            if (t >= p.T) break;
            for (int e0 = lane; e0 < p.E; e0 += 64) {
                // the loads of two expert columns and all splits in flight
                // together, then each sum in split order
                float part[2][kRouterMaxSplits];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int e = e0 + 32 * u;
                    const uint32_t off = (uint32_t)((tl * ld + e) * sizeof(float));
#pragma unroll
                    for (int sidx = 0; sidx < kRouterMaxSplits; ++sidx)
                        if (sidx < S && e < p.E)
                            part[u][sidx] = ld_shared_cluster_f32(mapa_shared(sp_local + off, (uint32_t)sidx));
                }
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int e = e0 + 32 * u;
                    if (e >= p.E) break;
                    float v = 0.f;
#pragma unroll
                    for (int sidx = 0; sidx < kRouterMaxSplits; ++sidx)
                        if (sidx < S) v += part[u][sidx];
                    if (p.bias) v += p.bias[e];
                    key[e] = v;
                    if (p.logits_out) p.logits_out[(size_t)t * p.E + e] = v;
                }
            }
            __syncwarp();
            warp_topk_weights<kRouterTcMaxE>(key, p.E, p.k, p.score, p.renorm, p.n_group,
                                             p.topk_group, t, p.topk_idx, p.topk_w, p.status,
                                             lane);
            __syncwarp();
        }
        cluster_sync();  // the peers are done reading this CTA's partial
    }
}

// Sum of the split partials (fixed split order), bias, then the warp top-k.
// A block owns 32 tokens: lanes read the token-minor partials coalesced and
// build the 32 x E keys in shared memory, then each of the 32 warps selects
// the top-k of one token.
constexpr int RR_THREADS = 1024;
constexpr int RR_TOKENS = 32;

__global__ void __launch_bounds__(RR_THREADS)
router_reduce_topk_kernel(const float *__restrict__ part, int splits, const float *__restrict__ bias,
                          float *__restrict__ logits_out, int *__restrict__ topk_idx,
                          float *__restrict__ topk_w, int Tn, int E, int k, int score, int renorm,
                          int n_group, int topk_group, int *status) {
    griddep_launch_dependents();  // the next kernel may be scheduled now
    griddep_wait();               // every input of this kernel is complete
    extern __shared__ float s_key[];  // [RR_TOKENS][E + 1]
    const int ld = E + 1;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t0 = blockIdx.x * RR_TOKENS;
    const int t = t0 + lane;
    for (int e = warp; e < E; e += RR_THREADS / 32) {
        float v = 0.f;
        if (t < Tn) {
            for (int s = 0; s < splits; ++s) v += part[((size_t)s * E + e) * Tn + t];
            if (bias) v += bias[e];
        }
        s_key[lane * ld + e] = v;
    }
    __syncthreads();
    for (int tt = warp; tt < RR_TOKENS; tt += RR_THREADS / 32) {
        const int tok = t0 + tt;
        if (tok >= Tn) break;
        const float *l = s_key + tt * ld;
        if (logits_out)
            for (int e = lane; e < E; e += 32) logits_out[(size_t)tok * E + e] = l[e];
        warp_topk_weights<kRouterTcMaxE>(l, E, k, score, renorm, n_group, topk_group, tok,
                                         topk_idx, topk_w, status, lane);
    }
}

}  // namespace

int64_t router_scratch_floats(int T, int E, int is_bf16) {
    if (!is_bf16 || E > kRouterTcMaxE) return 0;
    return (int64_t)kRouterMaxSplits * T * E;
}

namespace {

cudaError_t launch_router_tc(const void *x, const void *wg, const float *bias, float *logits_out,
                             int *topk_idx, float *topk_w, int T, int D, int E, int k, int score,
                             int renorm, int n_group, int topk_group, float *part, int *status,
                             cudaStream_t stream) {
    const int n_pad = (E + 15) / 16 * 16;
    CUtensorMap tm_x, tm_w;
    if (!make_tmap_2d(&tm_x, x, D, T, RC_BM) || !make_tmap_2d(&tm_w, wg, D, E, n_pad))
        return cudaErrorInvalidValue;
    const int nsm = sm_count();
    if (nsm <= 0) return cudaErrorNoDevice;
    const int m_tiles = (T + RC_BM - 1) / RC_BM;
    const int nk = (D + RC_BK - 1) / RC_BK;
    // about one CTA per SM (measured on GB300: T=4096, E=64 best at 4 splits
    // of 32 m-tiles; T=8192, E=256 at 2 splits of 64 m-tiles)
    int splits = std::max(1, std::min({kRouterMaxSplits, nk, nsm / m_tiles}));
    const int kps = (nk + splits - 1) / splits;
    splits = (nk + kps - 1) / kps;  // no empty split
    RouterTcParams p{T, E, n_pad, nk, kps, part, status};
    const size_t smem = rc_smem_bytes(n_pad);
    cudaError_t err;
    {
        // one launch: clusters of `splits` CTAs reduce through shared memory.
        // The partials and the key rows reuse the operand ring.
        const size_t need = sizeof(float) * ((size_t)RC_BM * (n_pad + 1) + (RC_CL_THREADS / 32) * (size_t)E);
        const char *sel = getenv("MOE_ROUTER_KERNEL");
        const bool two = sel && strcmp(sel, "split") == 0;
        if (!two && need <= (size_t)RC_STAGES * rc_stage_bytes(n_pad)) {
            p.bias = bias;
            p.logits_out = logits_out;
            p.topk_idx = topk_idx;
            p.topk_w = topk_w;
            p.k = k;
            p.score = score;
            p.renorm = renorm;
            p.splits = splits;
            p.n_group = n_group;
            p.topk_group = topk_group;
            err = ensure_smem((const void *)router_logits_tc_kernel<true>, smem);
            if (err != cudaSuccess) return err;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(m_tiles, splits);
            cfg.blockDim = dim3(RC_CL_THREADS);
            cfg.dynamicSmemBytes = smem;
            cfg.stream = stream;
            cudaLaunchAttribute attr[2];
            attr[0].id = cudaLaunchAttributeClusterDimension;
            attr[0].val.clusterDim.x = 1;
            attr[0].val.clusterDim.y = splits;
            attr[0].val.clusterDim.z = 1;
            attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[1].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = MOE_PDL ? 2 : 1;
            err = cudaLaunchKernelEx(&cfg, router_logits_tc_kernel<true>, tm_x, tm_w, p);
            if (err == cudaSuccess) {
                count_launch();
                return cudaSuccess;
            }
            cudaGetLastError();  // cluster refused: the two-kernel form below
        }
    }
    err = ensure_smem((const void *)router_logits_tc_kernel<false>, smem);
    if (err != cudaSuccess) return err;
    if ((err = launch_pdl(router_logits_tc_kernel<false>, dim3(m_tiles, splits), dim3(RC_THREADS), smem,
                          stream, tm_x, tm_w, p)) != cudaSuccess)
        return err;
    count_launch();
    if ((err = cudaGetLastError()) != cudaSuccess) return err;
    const size_t rsmem = sizeof(float) * RR_TOKENS * (size_t)(E + 1);
    if ((err = launch_pdl(router_reduce_topk_kernel, dim3((T + RR_TOKENS - 1) / RR_TOKENS),
                          dim3(RR_THREADS), rsmem, stream, part, splits, bias, logits_out, topk_idx,
                          topk_w, T, E, k, score, renorm, n_group, topk_group, status)) != cudaSuccess)
        return err;
    count_launch();
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_router_topk(const void *x, const void *wg, const float *bias, float *logits_out,
                               int *topk_idx, float *topk_w, int T, int D, int E, int k,
                               int score, int renorm, int n_group, int topk_group, int is_bf16,
                               float *scratch, int64_t scratch_floats, int *status,
                               cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    if (is_bf16 && E <= kRouterTcMaxE && scratch &&
        scratch_floats >= router_scratch_floats(T, E, is_bf16))
        return launch_router_tc(x, wg, bias, logits_out, topk_idx, topk_w, T, D, E, k, score,
                                renorm, n_group, topk_group, scratch, status, stream);
    const size_t smem = sizeof(float) * ((size_t)RT_TOKENS * E + RT_BK * SX_LD + RT_BK * SW_LD);
    const dim3 grid((T + RT_TOKENS - 1) / RT_TOKENS);
    cudaError_t err;
    if (is_bf16) {
        auto kern = router_topk_kernel<__nv_bfloat16>;
        err = ensure_smem((const void *)kern, smem);
        if (err != cudaSuccess) return err;
        if ((err = launch_pdl(kern, grid, dim3(RT_THREADS), smem, stream, (const __nv_bfloat16 *)x,
                              (const __nv_bfloat16 *)wg, bias, logits_out, topk_idx, topk_w, T, D, E,
                              k, score, renorm, n_group, topk_group, status)) != cudaSuccess)
            return err;
    } else {
        auto kern = router_topk_kernel<float>;
        err = ensure_smem((const void *)kern, smem);
        if (err != cudaSuccess) return err;
        if ((err = launch_pdl(kern, grid, dim3(RT_THREADS), smem, stream, (const float *)x,
                              (const float *)wg, bias, logits_out, topk_idx, topk_w, T, D, E, k, score,
                              renorm, n_group, topk_group, status)) != cudaSuccess)
            return err;
    }
    count_launch();
    return cudaGetLastError();
}

}  // namespace moe
