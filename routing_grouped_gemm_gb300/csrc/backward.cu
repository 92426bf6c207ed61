// Backward of the data movement and of the router.
//
// Page "Expert Parallelism (EP)" (llm-infra-atlas), section 5: the backward
// runs the forward in mirror -- the combine's backward is a dispatch (each
// slot's row receives the token's output gradient times the slot weight) and
// the dispatch's backward is a combine (a token's input gradient sums its k
// rows) -- and section 1's router (top-k + score function) is differentiated
// through the score function; the selection itself carries no gradient.
//
// All sums run in a fixed order (slots in slot order, tokens in token
// order), so every result is bit-identical run to run.
#include <algorithm>

#include <type_traits>

#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

// Slots handled together: their loads are issued before any of them is
// used, so a warp keeps BW_SLOTS row reads in flight.
constexpr int BW_SLOTS = 8;
#ifndef MOE_DB_SLOTS
#define MOE_DB_SLOTS 4
#endif
constexpr int DB_SLOTS = MOE_DB_SLOTS;  // the dispatch backward also holds wg rows: fewer registers

__device__ __forceinline__ void load4(const void *p, size_t i, bool bf16, float (&g)[4]) {
    if (bf16) {
        const uint2 v = *reinterpret_cast<const uint2 *>(static_cast<const __nv_bfloat16 *>(p) + i);
        const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&v);
        g[0] = __low2float(h2[0]);
        g[1] = __high2float(h2[0]);
        g[2] = __low2float(h2[1]);
        g[3] = __high2float(h2[1]);
    } else {
        const float4 v = *reinterpret_cast<const float4 *>(static_cast<const float *>(p) + i);
        g[0] = v.x; g[1] = v.y; g[2] = v.z; g[3] = v.w;
    }
}

// One warp per token.  gy[row] = bf16(w_j * dout[t]) for each slot j whose
// row is in the buffer; dw[t, j] = <dout[t], y_perm[row]> (y_perm fp16, the
// products and sums fp32: each lane sums its columns in order, then the
// lanes' sums are added in a fixed butterfly order), 0 for a slot without row.
// Blocks per SM the register budget is capped for: 8 (64 registers, no
// spills) puts one block per 4 tokens of the fine-grained batch (1024 blocks)
// in a single wave of 152 SMs; uncapped (134 registers) 3 blocks per SM fit.
// Fine-grained: 35.4 against 49.4 us under ncu, backward 1.102-1.105 against
// 1.118-1.119 ms.  16-byte row vectors per lane (MOE_COMBINE_BWD_VEC=8) were
// no faster (37.3 us; 34.7 us capped at 6 blocks, backward 1.106 ms).
#ifndef MOE_COMBINE_BWD_MINB
#define MOE_COMBINE_BWD_MINB 8
#endif
// elements of a row per lane per step (4: 8-byte fp16 loads, 8: 16-byte)
#ifndef MOE_COMBINE_BWD_VEC
#define MOE_COMBINE_BWD_VEC 4
#endif
constexpr int CBW_VEC = MOE_COMBINE_BWD_VEC;
static_assert(CBW_VEC == 4 || CBW_VEC == 8, "4 or 8 elements per lane");
using CbwVec = std::conditional_t<CBW_VEC == 8, uint4, uint2>;
template <bool BF16>
__global__ void __launch_bounds__(128, MOE_COMBINE_BWD_MINB)
combine_bwd_kernel(const void *__restrict__ dout, const __half *__restrict__ y_perm,
                   const int *__restrict__ row_of, const float *__restrict__ topk_w,
                   __nv_bfloat16 *__restrict__ gy, float *__restrict__ dw, int T, int k, int D,
                   long long rows_alloc, int *status) {
    griddep_launch_dependents();  // the next kernel may be scheduled now
    griddep_wait();               // every input of this kernel is complete
    const int t = (int)(((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= T) return;
    int my_r = -1;
    float my_w = 0.f;
    if (lane < k) {
        my_r = row_of[(size_t)t * k + lane];
        my_w = topk_w[(size_t)t * k + lane];
        if (my_r < -1 || (long long)my_r >= rows_alloc) {
            raise_flag(status, FLAG_BAD_ROUTING);
            my_r = -1;
        }
    }
    for (int j0 = 0; j0 < k; j0 += BW_SLOTS) {
        int r[BW_SLOTS];
        float w[BW_SLOTS], dot[BW_SLOTS];
#pragma unroll
        for (int u = 0; u < BW_SLOTS; ++u) {
            const int j = j0 + u;
            r[u] = __shfl_sync(0xffffffffu, my_r, j & 31);
            w[u] = __shfl_sync(0xffffffffu, my_w, j & 31);
            if (j >= k) r[u] = -1;
            dot[u] = 0.f;
        }
        for (int d0 = lane * CBW_VEC; d0 < D; d0 += 32 * CBW_VEC) {
            float g[CBW_VEC];
            {
                float g4[4];
#pragma unroll
                for (int q = 0; q < CBW_VEC / 4; ++q) {
                    load4(dout, (size_t)t * D + d0 + 4 * q, BF16, g4);
#pragma unroll
                    for (int i = 0; i < 4; ++i) g[4 * q + i] = g4[i];
                }
            }
            CbwVec y[BW_SLOTS];
#pragma unroll
            for (int u = 0; u < BW_SLOTS; ++u)
                if (r[u] >= 0)
                    y[u] = __ldcs(reinterpret_cast<const CbwVec *>(y_perm + (size_t)r[u] * D + d0));
#pragma unroll
            for (int u = 0; u < BW_SLOTS; ++u) {
                if (r[u] < 0) continue;
                const __half2 *yh = reinterpret_cast<const __half2 *>(&y[u]);
                uint32_t ow[CBW_VEC / 2];
#pragma unroll
                for (int i = 0; i < CBW_VEC / 2; ++i) {
                    const float2 f = __half22float2(yh[i]);
                    dot[u] = fmaf(g[2 * i], f.x, dot[u]);
                    dot[u] = fmaf(g[2 * i + 1], f.y, dot[u]);
                    __nv_bfloat162 b = __floats2bfloat162_rn(w[u] * g[2 * i], w[u] * g[2 * i + 1]);
                    ow[i] = *reinterpret_cast<uint32_t *>(&b);
                }
                if constexpr (CBW_VEC == 8)
                    *reinterpret_cast<uint4 *>(gy + (size_t)r[u] * D + d0) = make_uint4(ow[0], ow[1], ow[2], ow[3]);
                else
                    *reinterpret_cast<uint2 *>(gy + (size_t)r[u] * D + d0) = make_uint2(ow[0], ow[1]);
            }
        }
#pragma unroll
        for (int u = 0; u < BW_SLOTS; ++u) {
            float v = dot[u];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0 && j0 + u < k) dw[(size_t)t * k + j0 + u] = v;
        }
    }
}

// One warp per token: dx[t] = sum_j dxp[row_of[t, j]] + r[t], fp32 in slot
// order, rounded once to the output type; r[t] = add[t] when add, else (wg
// given) sum_j dl[t, e_j] wg[e_j] in slot order.
template <bool BF16>
__global__ void __launch_bounds__(128)
dispatch_bwd_kernel(const float *__restrict__ dxp, const int *__restrict__ row_of,
                    const float *__restrict__ add, const int *__restrict__ topk_idx,
                    const float *__restrict__ dl, const void *__restrict__ wg, int E,
                    void *__restrict__ dx, int T, int k, int D, long long rows_alloc) {
    griddep_launch_dependents();  // the next kernel may be scheduled now
    griddep_wait();               // every input of this kernel is complete
    const int t = (int)(((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= T) return;
    // lane j < k holds slot j: its row, its expert and dl at that expert
    int my_r = -1, my_e = -1;
    float my_g = 0.f;
    if (lane < k) {
        my_r = row_of[(size_t)t * k + lane];
        if (my_r < 0 || (long long)my_r >= rows_alloc) my_r = -1;
        if (!add && wg) {
            my_e = topk_idx[(size_t)t * k + lane];
            if (my_e < 0 || my_e >= E) my_e = -1;
            else my_g = dl[(size_t)t * E + my_e];
        }
    }
    for (int d0 = lane * 4; d0 < D; d0 += 128) {
        float a[4] = {0.f, 0.f, 0.f, 0.f};
        for (int j0 = 0; j0 < k; j0 += DB_SLOTS) {
            int r[DB_SLOTS];
            float4 v[DB_SLOTS];
#pragma unroll
            for (int u = 0; u < DB_SLOTS; ++u) {
                r[u] = __shfl_sync(0xffffffffu, my_r, (j0 + u) & 31);
                if (j0 + u >= k) r[u] = -1;
                if (r[u] >= 0)
                    v[u] = __ldcs(reinterpret_cast<const float4 *>(dxp + (size_t)r[u] * D + d0));
            }
#pragma unroll
            for (int u = 0; u < DB_SLOTS; ++u) {
                if (r[u] < 0) continue;
                a[0] += v[u].x; a[1] += v[u].y; a[2] += v[u].z; a[3] += v[u].w;
            }
        }
        if (add) {
            const float4 v = *reinterpret_cast<const float4 *>(add + (size_t)t * D + d0);
            a[0] += v.x; a[1] += v.y; a[2] += v.z; a[3] += v.w;
        } else if (wg) {
            for (int j0 = 0; j0 < k; j0 += DB_SLOTS) {
                int e[DB_SLOTS];
                float g[DB_SLOTS], w[DB_SLOTS][4];
#pragma unroll
                for (int u = 0; u < DB_SLOTS; ++u) {
                    e[u] = __shfl_sync(0xffffffffu, my_e, (j0 + u) & 31);
                    g[u] = __shfl_sync(0xffffffffu, my_g, (j0 + u) & 31);
                    if (j0 + u >= k) e[u] = -1;
                    if (e[u] >= 0) load4(wg, (size_t)e[u] * D + d0, BF16, w[u]);
                }
#pragma unroll
                for (int u = 0; u < DB_SLOTS; ++u) {
                    if (e[u] < 0) continue;
#pragma unroll
                    for (int i = 0; i < 4; ++i) a[i] = fmaf(g[u], w[u][i], a[i]);
                }
            }
        }
        if (BF16) {
            __nv_bfloat162 lo = __floats2bfloat162_rn(a[0], a[1]);
            __nv_bfloat162 hi = __floats2bfloat162_rn(a[2], a[3]);
            uint2 o;
            o.x = *reinterpret_cast<uint32_t *>(&lo);
            o.y = *reinterpret_cast<uint32_t *>(&hi);
            *reinterpret_cast<uint2 *>(static_cast<__nv_bfloat16 *>(dx) + (size_t)t * D + d0) = o;
        } else {
            *reinterpret_cast<float4 *>(static_cast<float *>(dx) + (size_t)t * D + d0) =
                make_float4(a[0], a[1], a[2], a[3]);
        }
    }
}

// One warp per token: dl[t, :] from dw[t, :] through the score function of
// the forward's selection (logits are the forward's fp32 keys l = x.wg^T + b):
//   softmax:          dl_e = p_e (G_e - sum_j dw_j p_{S_j})   (G_e = dw_j at e = S_j)
//   softmax, renorm:  dl_{S_j} = w_j (dw_j - sum_i dw_i w_i)
//   sigmoid:          dl_{S_j} = dw_j s_j (1 - s_j)
//   sigmoid, renorm:  dl_{S_j} = (dw_j - sum_i dw_i w_i) / sum_i s_{S_i} * s_j (1 - s_j)
// with p the softmax over all E, s the sigmoid, w the forward's weights.
__global__ void __launch_bounds__(256)
router_dl_kernel(const float *__restrict__ logits, const int *__restrict__ topk_idx,
                 const float *__restrict__ topk_w, const float *__restrict__ dw,
                 float *__restrict__ dl, int T, int E, int k, int score, int renorm,
                 int *__restrict__ ctr, int n_ctr) {
    griddep_launch_dependents();  // the next kernel may be scheduled now
    griddep_wait();               // every input of this kernel is complete
    // the split-K counters of the router GEMM that follows start at zero
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i < n_ctr; i += blockDim.x) ctr[i] = 0;
    const int t = (int)(((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= T) return;
    const float *l = logits + (size_t)t * E;
    float *o = dl + (size_t)t * E;
    // slot sums in slot order (every lane computes the same values)
    float dot = 0.f, sp = 0.f, ssum = 0.f, mx = -INFINITY, z = 0.f;
    if (score == 0 && !renorm) {
        for (int e = 0; e < E; ++e) mx = fmaxf(mx, l[e]);
        for (int e = 0; e < E; ++e) z += expf(l[e] - mx);
    }
    for (int j = 0; j < k; ++j) {
        const int e = topk_idx[(size_t)t * k + j];
        const float dwj = dw[(size_t)t * k + j];
        dot += dwj * topk_w[(size_t)t * k + j];
        if (score == 0 && !renorm) sp += dwj * (expf(l[e] - mx) / z);
        if (score != 0 && renorm) ssum += 1.f / (1.f + expf(-l[e]));
    }
    if (score == 0 && !renorm) {
        for (int e = lane; e < E; e += 32) o[e] = -(expf(l[e] - mx) / z) * sp;
    } else {
        for (int e = lane; e < E; e += 32) o[e] = 0.f;
    }
    __syncwarp();
    if (lane == 0) {
        for (int j = 0; j < k; ++j) {
            const int e = topk_idx[(size_t)t * k + j];
            if (e < 0 || e >= E) continue;
            const float dwj = dw[(size_t)t * k + j];
            const float wj = topk_w[(size_t)t * k + j];
            if (score == 0 && !renorm) {
                o[e] += (expf(l[e] - mx) / z) * dwj;
            } else if (score == 0) {
                o[e] = wj * (dwj - dot);
            } else {
                const float s = 1.f / (1.f + expf(-l[e]));
                o[e] = renorm ? (dwj - dot) / ssum * s * (1.f - s) : dwj * s * (1.f - s);
            }
        }
    }
}

// Split-K SIMT GEMM for the router's two products (fp32 FMAs; the router's
// gradients stay in fp32):
//   C(m, n) = sum_k A(m, k) B(k, n),
// A(m, k) = a[m * a_m + k * a_k] fp32 (a_m == 1 or a_k == 1), B(k, n) =
// b[k * ldb + n] (bf16 or fp32), C row-major [M, N].  With colsum, the
// blocks of the first N tile also form colsum[m] = sum_k A(m, k).  Split z
// of S sums k in [z kc, (z+1) kc) in ascending order; with S > 1 each split
// writes its partial tile to part (cpart for the column sums) and the last
// split of a tile to finish (a per-tile counter in ctr, zero on entry and
// left zero) adds the S partials in split order, so the result does not
// depend on which split finishes last.  64 x 128 tiles, 4 x 8 outputs per
// thread, the next K slice loaded into registers while the current one is
// multiplied; N a multiple of 4.
constexpr int RG_BM = 64, RG_BN = 128, RG_BK = 32, RG_PAD = 4;
template <bool BBF16>
__global__ void __launch_bounds__(256)
router_gemm_kernel(const float *__restrict__ a, long long a_m, long long a_k,
                   const void *__restrict__ b, long long ldb, float *__restrict__ c,
                   float *__restrict__ colsum, float *__restrict__ part, float *__restrict__ cpart,
                   int *__restrict__ ctr, int M, int N, int K, int kc, int S) {
    griddep_launch_dependents();  // the next kernel may be scheduled now
    griddep_wait();               // every input of this kernel is complete
    __shared__ __align__(16) float As[RG_BK][RG_BM + RG_PAD];
    __shared__ __align__(16) float Bs[RG_BK][RG_BN];
    __shared__ int s_last;
    const int tid = threadIdx.x, tx = tid & 15, ty = tid >> 4;
    const int m0 = blockIdx.y * RG_BM, n0 = blockIdx.x * RG_BN, z = blockIdx.z;
    const int kb = z * kc, ke = min(K, kb + kc);
    const bool do_sum = colsum != nullptr && blockIdx.x == 0 && tid < RG_BM;
    const bool a_mcont = a_m == 1;
    float ra[8];
    float4 rb[4];
    auto gload = [&](int k0) {
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = tid + 256 * u;
            const int kk = a_mcont ? i / RG_BM : i % RG_BK;
            const int mm = a_mcont ? i % RG_BM : i / RG_BK;
            const int m = m0 + mm, k = k0 + kk;
            ra[u] = (m < M && k < ke) ? a[(long long)m * a_m + (long long)k * a_k] : 0.f;
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = tid + 256 * u;
            const int kk = i / (RG_BN / 4), n = n0 + (i % (RG_BN / 4)) * 4, k = k0 + kk;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (n < N && k < ke) {
                if (BBF16) {
                    const uint2 q = *reinterpret_cast<const uint2 *>(
                        static_cast<const __nv_bfloat16 *>(b) + (long long)k * ldb + n);
                    const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&q);
                    v = make_float4(__low2float(h2[0]), __high2float(h2[0]), __low2float(h2[1]),
                                    __high2float(h2[1]));
                } else {
                    v = *reinterpret_cast<const float4 *>(static_cast<const float *>(b) +
                                                          (long long)k * ldb + n);
                }
            }
            rb[u] = v;
        }
    };
    float acc[4][8] = {};
    float cs = 0.f;
    if (kb < ke) gload(kb);
    for (int k0 = kb; k0 < ke; k0 += RG_BK) {
        __syncthreads();  // the previous slice's products are done with smem
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = tid + 256 * u;
            As[a_mcont ? i / RG_BM : i % RG_BK][a_mcont ? i % RG_BM : i / RG_BK] = ra[u];
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = tid + 256 * u;
            *reinterpret_cast<float4 *>(&Bs[i / (RG_BN / 4)][(i % (RG_BN / 4)) * 4]) = rb[u];
        }
        __syncthreads();
        if (k0 + RG_BK < ke) gload(k0 + RG_BK);  // in flight during the products below
        if (do_sum)
            for (int kk = 0; kk < RG_BK; ++kk) cs += As[kk][tid];
#pragma unroll 8
        for (int kk = 0; kk < RG_BK; ++kk) {
            const float4 av = *reinterpret_cast<const float4 *>(&As[kk][ty * 4]);
            const float4 b0 = *reinterpret_cast<const float4 *>(&Bs[kk][tx * 4]);
            const float4 b1 = *reinterpret_cast<const float4 *>(&Bs[kk][RG_BN / 2 + tx * 4]);
            const float ar[4] = {av.x, av.y, av.z, av.w};
            const float br[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(ar[i], br[j], acc[i][j]);
        }
    }
    float *dst = S > 1 ? part + (size_t)z * M * N : c;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty * 4 + i;
        if (m >= M) continue;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int n = n0 + h * (RG_BN / 2) + tx * 4;
            if (n < N)
                *reinterpret_cast<float4 *>(dst + (size_t)m * N + n) =
                    make_float4(acc[i][h * 4], acc[i][h * 4 + 1], acc[i][h * 4 + 2], acc[i][h * 4 + 3]);
        }
    }
    if (do_sum && m0 + tid < M) (S > 1 ? cpart + (size_t)z * M : colsum)[m0 + tid] = cs;
    if (S == 1) return;
    // the last split of this tile adds the partials in split order
    __threadfence();
    __syncthreads();
    const int tile = blockIdx.y * gridDim.x + blockIdx.x;
    if (tid == 0) s_last = atomicAdd(&ctr[tile], 1) == S - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int m = m0 + ty * 4 + i;
        if (m >= M) continue;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int n = n0 + h * (RG_BN / 2) + tx * 4;
            if (n >= N) continue;
            float4 sum = __ldcg(reinterpret_cast<const float4 *>(part + (size_t)m * N + n));
            for (int zz = 1; zz < S; ++zz) {
                const float4 v =
                    __ldcg(reinterpret_cast<const float4 *>(part + ((size_t)zz * M + m) * N + n));
                sum.x += v.x; sum.y += v.y; sum.z += v.z; sum.w += v.w;
            }
            *reinterpret_cast<float4 *>(c + (size_t)m * N + n) = sum;
        }
    }
    if (do_sum && m0 + tid < M) {
        float sum = __ldcg(cpart + m0 + tid);
        for (int zz = 1; zz < S; ++zz) sum += __ldcg(cpart + (size_t)zz * M + m0 + tid);
        colsum[m0 + tid] = sum;
    }
    if (tid == 0) ctr[tile] = 0;  // ready for the next call
}

// dwg and dbias from the expert-contiguous layout, where dl is zero off each
// token's selected experts and every selected (token, expert) has a row:
//   dwg[e, :] = sum_{rows r of e} dl[t_r, e] x[t_r, :],  dbias[e] = sum_r dl[t_r, e]
// Block (c, e) walks the segment in chunks of RS_CHUNK rows: the block first
// stages each row's token and dl value in shared memory, then its warps take
// the chunk's rows round-robin, each lane 8 columns of the 256-column chunk c
// (one 16-byte load of x's row, which the L2 holds).  The warps' partial
// sums are added in warp order, so the result is deterministic.
// 16 warps (24 rows of a 384-row segment each, four loads in flight per
// warp): fine-grained backward 1.085-1.088 ms against 1.095-1.096 ms with 8
// and 1.090 ms with 32.
#ifndef MOE_RS_WARPS
#define MOE_RS_WARPS 16
#endif
constexpr int RS_COLS = 256, RS_WARPS = MOE_RS_WARPS, RS_CHUNK = 512;
template <bool BF16>
__global__ void __launch_bounds__(32 * RS_WARPS)
router_wgrad_seg_kernel(const void *__restrict__ x, const float *__restrict__ dl,
                        const int *__restrict__ seg_off, const int *__restrict__ tpe,
                        const int *__restrict__ token_of_row, int T, int D, int E,
                        float *__restrict__ dwg, float *__restrict__ dbias) {
    griddep_launch_dependents();  // the next kernel may be scheduled now
    griddep_wait();               // every input of this kernel is complete
    __shared__ float part[RS_WARPS][RS_COLS + 1];
    __shared__ float bpart[RS_WARPS];
    __shared__ int s_tok[RS_CHUNK];
    __shared__ float s_g[RS_CHUNK];
    const int e = blockIdx.y, c0 = blockIdx.x * RS_COLS;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = seg_off[e], n = min(tpe[e], seg_off[e + 1] - seg_off[e]);
    const int col = c0 + lane * 8;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float bsum = 0.f;
    for (int base = 0; base < n; base += RS_CHUNK) {
        const int m = min(RS_CHUNK, n - base);
        __syncthreads();  // the previous chunk's entries are consumed
        for (int i = threadIdx.x; i < m; i += blockDim.x) {
            const int t = token_of_row[b + base + i];
            const bool ok = t >= 0 && t < T;
            s_tok[i] = ok ? t : -1;
            s_g[i] = ok ? dl[(size_t)t * E + e] : 0.f;
        }
        __syncthreads();
#pragma unroll 4
        for (int i = warp; i < m; i += RS_WARPS) {
            const int t = s_tok[i];
            if (t < 0) continue;
            const float g = s_g[i];
            bsum += g;
            if (col < D) {
                float v[8];
                if (BF16) {
                    const uint4 q = *reinterpret_cast<const uint4 *>(
                        static_cast<const __nv_bfloat16 *>(x) + (size_t)t * D + col);
                    const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&q);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        v[2 * u] = __low2float(h2[u]);
                        v[2 * u + 1] = __high2float(h2[u]);
                    }
                } else {
                    const float4 a = *reinterpret_cast<const float4 *>(
                        static_cast<const float *>(x) + (size_t)t * D + col);
                    const float4 a2 = *reinterpret_cast<const float4 *>(
                        static_cast<const float *>(x) + (size_t)t * D + col + 4);
                    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
                    v[4] = a2.x; v[5] = a2.y; v[6] = a2.z; v[7] = a2.w;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) acc[u] = fmaf(g, v[u], acc[u]);
            }
        }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) part[warp][lane * 8 + u] = acc[u];
    if (lane == 0) bpart[warp] = bsum;
    __syncthreads();
    for (int cc = threadIdx.x; cc < RS_COLS; cc += blockDim.x) {
        if (c0 + cc >= D) continue;
        float sum = part[0][cc];
        for (int w = 1; w < RS_WARPS; ++w) sum += part[w][cc];
        dwg[(size_t)e * D + c0 + cc] = sum;
    }
    if (dbias && blockIdx.x == 0 && threadIdx.x == 0) {
        float sum = bpart[0];
        for (int w = 1; w < RS_WARPS; ++w) sum += bpart[w];
        dbias[e] = sum;
    }
}

// Splits of dwg's K (= T): enough (tile, split) blocks for two waves of the
// 152 SMs, at least 256 tokens per split, at most 16 splits.
struct RouterSplit {
    int S, kc;
};
RouterSplit router_split(int T, int D, int E) {
    const long long tiles = (long long)((E + RG_BM - 1) / RG_BM) * ((D + RG_BN - 1) / RG_BN);
    long long S = std::max(1LL, (304 + tiles - 1) / tiles);
    S = std::min<long long>({S, 16, std::max(1, T / 256)});
    int kc = (int)(((T + S - 1) / S + RG_BK - 1) / RG_BK * RG_BK);
    if (kc == 0) kc = RG_BK;
    return {(int)((T + kc - 1) / kc), kc};
}

template <bool BBF16>
cudaError_t router_gemm(const float *a, long long a_m, long long a_k, const void *b, long long ldb,
                        float *c, float *colsum, float *part, float *cpart, int *ctr, int M, int N,
                        int K, int S, int kc, cudaStream_t stream) {
    if (M == 0 || N == 0) return cudaSuccess;
    const dim3 grid((N + RG_BN - 1) / RG_BN, (M + RG_BM - 1) / RG_BM, S);
    const cudaError_t e = launch_pdl(router_gemm_kernel<BBF16>, grid, dim3(256), 0, stream, a, a_m,
                                     a_k, b, ldb, c, colsum, part, cpart, ctr, M, N, K, kc, S);
    if (e == cudaSuccess) count_launch();
    return e;
}

}  // namespace

cudaError_t launch_combine_bwd(const void *dout, const void *y_perm, const int *row_of,
                               const float *topk_w, void *gy, float *dw, int T, int D, int k,
                               int64_t rows_alloc, int is_bf16, int *status, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const dim3 grid((unsigned)((T + 3) / 4));  // 4 warps (tokens) per block
    const cudaError_t e =
        is_bf16 ? launch_pdl(combine_bwd_kernel<true>, grid, dim3(128), 0, stream, dout,
                             (const __half *)y_perm, row_of, topk_w, (__nv_bfloat16 *)gy, dw, T, k, D, (long long)rows_alloc,
                             status)
                : launch_pdl(combine_bwd_kernel<false>, grid, dim3(128), 0, stream, dout,
                             (const __half *)y_perm, row_of, topk_w, (__nv_bfloat16 *)gy, dw, T, k, D, (long long)rows_alloc,
                             status);
    if (e == cudaSuccess) count_launch();
    return e;
}

cudaError_t launch_dispatch_bwd(const float *dxp, const int *row_of, const float *add,
                                const int *topk_idx, const float *dl, const void *wg, int E,
                                void *dx, int T, int D, int k, int64_t rows_alloc, int is_bf16,
                                cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    if (k > 32) return cudaErrorInvalidValue;  // one lane per slot
    const dim3 grid((unsigned)((T + 3) / 4));  // 4 warps (tokens) per block
    const cudaError_t e =
        is_bf16 ? launch_pdl(dispatch_bwd_kernel<true>, grid, dim3(128), 0, stream, dxp, row_of, add,
                             topk_idx, dl, wg, E, dx, T, k, D, (long long)rows_alloc)
                : launch_pdl(dispatch_bwd_kernel<false>, grid, dim3(128), 0, stream, dxp, row_of,
                             add, topk_idx, dl, wg, E, dx, T, k, D, (long long)rows_alloc);
    if (e == cudaSuccess) count_launch();
    return e;
}

// Router backward scratch (S > 1): partial tiles [S, E, D], partial column
// sums [S, E], then one counter per output tile (ints).
int64_t router_bwd_scratch_floats(int T, int D, int E) {
    const RouterSplit sp = router_split(T, D, E);
    const int64_t tiles = (int64_t)((E + RG_BM - 1) / RG_BM) * ((D + RG_BN - 1) / RG_BN);
    return sp.S > 1 ? (int64_t)sp.S * E * D + (int64_t)sp.S * E + tiles : 0;
}

cudaError_t launch_router_bwd(const void *x, const void *wg, const float *logits,
                              const int *topk_idx, const float *topk_w, const float *dw, float *dl,
                              float *dx_router, float *dwg, float *dbias, float *scratch, int T,
                              int D, int E, int k, int score, int renorm, int is_bf16,
                              cudaStream_t stream, const RouterSegments *segs) {
    if (T == 0) return cudaSuccess;
    if (D % 4) return cudaErrorInvalidValue;
    const RouterSplit sp = router_split(T, D, E);
    const int tiles = ((E + RG_BM - 1) / RG_BM) * ((D + RG_BN - 1) / RG_BN);
    float *part = sp.S > 1 ? scratch : nullptr;
    float *cpart = sp.S > 1 ? scratch + (size_t)sp.S * E * D : nullptr;
    int *ctr = sp.S > 1 ? reinterpret_cast<int *>(cpart + (size_t)sp.S * E) : nullptr;
    cudaError_t e = launch_pdl(router_dl_kernel, dim3((unsigned)((T + 7) / 8)), dim3(256), 0, stream,
                               logits, topk_idx, topk_w, dw, dl, T, E, k, score, renorm, ctr,
                               ctr ? tiles : 0);
    if (e != cudaSuccess) return e;
    count_launch();
    if (segs && !router_dl_dense(score, renorm) && D % 8 == 0) {
        // dl is zero off the selected experts: sum x rows over each expert's segment
        const dim3 grid((unsigned)((D + RS_COLS - 1) / RS_COLS), (unsigned)E);
        e = is_bf16 ? launch_pdl(router_wgrad_seg_kernel<true>, grid, dim3(32 * RS_WARPS), 0,
                                 stream, x, (const float *)dl, segs->seg_off, segs->tpe,
                                 segs->token_of_row, T, D, E, dwg, dbias)
                    : launch_pdl(router_wgrad_seg_kernel<false>, grid, dim3(32 * RS_WARPS), 0,
                                 stream, x, (const float *)dl, segs->seg_off, segs->tpe,
                                 segs->token_of_row, T, D, E, dwg, dbias);
        if (e == cudaSuccess) count_launch();
        return e;
    }
    // dwg [E, D] = dl^T x  (K = T, split), dbias = the column sums of dl
    e = is_bf16 ? router_gemm<true>(dl, 1, E, x, D, dwg, dbias, part, cpart, ctr, E, D, T, sp.S,
                                    sp.kc, stream)
                : router_gemm<false>(dl, 1, E, x, D, dwg, dbias, part, cpart, ctr, E, D, T, sp.S,
                                     sp.kc, stream);
    if (e != cudaSuccess) return e;
    // dx_router [T, D] = dl wg  (K = E), only where dl is dense
    if (!router_dl_dense(score, renorm)) return cudaSuccess;
    return is_bf16 ? router_gemm<true>(dl, E, 1, wg, D, dx_router, nullptr, nullptr, nullptr,
                                       nullptr, T, D, E, 1, E, stream)
                   : router_gemm<false>(dl, E, 1, wg, D, dx_router, nullptr, nullptr, nullptr,
                                        nullptr, T, D, E, 1, E, stream);
}

}  // namespace moe
