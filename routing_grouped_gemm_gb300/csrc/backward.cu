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

#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

// One warp per token.  gy[row] = bf16(w_j * dout[t]) for each slot j whose
// row is in the buffer; dw[t, j] = <dout[t], y_perm[row]> (fp32, lanes'
// partial sums added in a fixed butterfly order), 0 for a slot without row.
template <bool BF16>
__global__ void __launch_bounds__(256)
combine_bwd_kernel(const void *__restrict__ dout, const float *__restrict__ y_perm,
                   const int *__restrict__ row_of, const float *__restrict__ topk_w,
                   __nv_bfloat16 *__restrict__ gy, float *__restrict__ dw, int T, int k, int D,
                   long long rows_alloc, int *status) {
    griddep_launch_dependents();  // the next kernel may be scheduled now
    griddep_wait();               // every input of this kernel is complete
    const int t = (int)(((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= T) return;
    for (int j = 0; j < k; ++j) {
        int r = row_of[(size_t)t * k + j];
        if (r < -1 || (long long)r >= rows_alloc) {
            if (lane == 0) raise_flag(status, FLAG_BAD_ROUTING);
            r = -1;
        }
        const float w = topk_w[(size_t)t * k + j];
        float dot = 0.f;
        if (r >= 0) {
            for (int d0 = lane * 4; d0 < D; d0 += 128) {
                float g[4];
                if (BF16) {
                    const uint2 v = *reinterpret_cast<const uint2 *>(
                        static_cast<const __nv_bfloat16 *>(dout) + (size_t)t * D + d0);
                    const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&v);
                    g[0] = __low2float(h2[0]);
                    g[1] = __high2float(h2[0]);
                    g[2] = __low2float(h2[1]);
                    g[3] = __high2float(h2[1]);
                } else {
                    const float4 v = *reinterpret_cast<const float4 *>(
                        static_cast<const float *>(dout) + (size_t)t * D + d0);
                    g[0] = v.x; g[1] = v.y; g[2] = v.z; g[3] = v.w;
                }
                const float4 y = *reinterpret_cast<const float4 *>(y_perm + (size_t)r * D + d0);
                dot = fmaf(g[0], y.x, dot);
                dot = fmaf(g[1], y.y, dot);
                dot = fmaf(g[2], y.z, dot);
                dot = fmaf(g[3], y.w, dot);
                __nv_bfloat162 lo = __floats2bfloat162_rn(w * g[0], w * g[1]);
                __nv_bfloat162 hi = __floats2bfloat162_rn(w * g[2], w * g[3]);
                uint2 o;
                o.x = *reinterpret_cast<uint32_t *>(&lo);
                o.y = *reinterpret_cast<uint32_t *>(&hi);
                *reinterpret_cast<uint2 *>(gy + (size_t)r * D + d0) = o;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        if (lane == 0) dw[(size_t)t * k + j] = dot;
    }
}

// One warp per token: dx[t] = sum_j dxp[row_of[t, j]] (+ add[t]), fp32 in
// slot order, rounded once to the output type.
template <bool BF16>
__global__ void __launch_bounds__(256)
dispatch_bwd_kernel(const float *__restrict__ dxp, const int *__restrict__ row_of,
                    const float *__restrict__ add, void *__restrict__ dx, int T, int k, int D,
                    long long rows_alloc) {
    griddep_launch_dependents();  // the next kernel may be scheduled now
    griddep_wait();               // every input of this kernel is complete
    const int t = (int)(((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= T) return;
    for (int d0 = lane * 4; d0 < D; d0 += 128) {
        float a[4] = {0.f, 0.f, 0.f, 0.f};
        for (int j = 0; j < k; ++j) {
            const int r = row_of[(size_t)t * k + j];
            if (r < 0 || (long long)r >= rows_alloc) continue;
            const float4 v = __ldcs(reinterpret_cast<const float4 *>(dxp + (size_t)r * D + d0));
            a[0] += v.x; a[1] += v.y; a[2] += v.z; a[3] += v.w;
        }
        if (add) {
            const float4 v = *reinterpret_cast<const float4 *>(add + (size_t)t * D + d0);
            a[0] += v.x; a[1] += v.y; a[2] += v.z; a[3] += v.w;
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
                 float *__restrict__ dl, int T, int E, int k, int score, int renorm) {
    griddep_launch_dependents();  // the next kernel may be scheduled now
    griddep_wait();               // every input of this kernel is complete
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

// C[m, n] = sum_k A(m, k) B(k, n) (+ C when accumulate), fp32, k ascending:
// A(m, k) = a[m * a_m + k * a_k], B(k, n) = b[k * b_k + n * b_n]; a, b fp32
// (ABF16 / BBF16: bf16).  64 x 64 tiles, 4 x 4 per thread.
constexpr int SG_T = 64, SG_K = 16;
template <bool ABF16, bool BBF16>
__global__ void __launch_bounds__(256)
simt_gemm_kernel(const void *__restrict__ a, long long a_m, long long a_k,
                 const void *__restrict__ b, long long b_k, long long b_n, float *__restrict__ c,
                 int M, int N, int K, int accumulate) {
    griddep_launch_dependents();  // the next kernel may be scheduled now
    griddep_wait();               // every input of this kernel is complete
    __shared__ float sa[SG_K][SG_T + 1], sb[SG_K][SG_T + 1];
    const int m0 = blockIdx.y * SG_T, n0 = blockIdx.x * SG_T;
    const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
    float acc[4][4] = {};
    auto ld = [](const void *p, long long i, bool bf) -> float {
        return bf ? __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[i])
                  : static_cast<const float *>(p)[i];
    };
    for (int k0 = 0; k0 < K; k0 += SG_K) {
        for (int i = threadIdx.x; i < SG_K * SG_T; i += blockDim.x) {
            const int kk = i / SG_T, mm = i % SG_T;
            const int m = m0 + mm, n = n0 + mm, k = k0 + kk;
            sa[kk][mm] = (m < M && k < K) ? ld(a, (long long)m * a_m + (long long)k * a_k, ABF16) : 0.f;
            sb[kk][mm] = (n < N && k < K) ? ld(b, (long long)k * b_k + (long long)n * b_n, BBF16) : 0.f;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < SG_K; ++kk) {
            float av[4], bv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                av[i] = sa[kk][ty * 4 + i];
                bv[i] = sb[kk][tx * 4 + i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int m = m0 + ty * 4 + i, n = n0 + tx * 4 + j;
            if (m < M && n < N) {
                float *p = c + (size_t)m * N + n;
                *p = accumulate ? *p + acc[i][j] : acc[i][j];
            }
        }
}

// dbias[e] = sum_t dl[t, e], tokens in order.
__global__ void __launch_bounds__(256)
column_sum_kernel(const float *__restrict__ dl, float *__restrict__ out, int T, int E) {
    griddep_launch_dependents();  // the next kernel may be scheduled now
    griddep_wait();               // every input of this kernel is complete
    const int e = blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= E) return;
    float s = 0.f;
    for (int t = 0; t < T; ++t) s += dl[(size_t)t * E + e];
    out[e] = s;
}

template <bool ABF16, bool BBF16>
cudaError_t simt_gemm(const void *a, long long a_m, long long a_k, const void *b, long long b_k,
                      long long b_n, float *c, int M, int N, int K, cudaStream_t stream) {
    if (M == 0 || N == 0) return cudaSuccess;
    const dim3 grid((N + SG_T - 1) / SG_T, (M + SG_T - 1) / SG_T);
    const cudaError_t e = launch_pdl(simt_gemm_kernel<ABF16, BBF16>, grid, dim3(256), 0, stream, a,
                                     a_m, a_k, b, b_k, b_n, c, M, N, K, 0);
    if (e == cudaSuccess) count_launch();
    return e;
}

}  // namespace

cudaError_t launch_combine_bwd(const void *dout, const float *y_perm, const int *row_of,
                               const float *topk_w, void *gy, float *dw, int T, int D, int k,
                               int64_t rows_alloc, int is_bf16, int *status, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const dim3 grid((unsigned)((T + 7) / 8));
    const cudaError_t e =
        is_bf16 ? launch_pdl(combine_bwd_kernel<true>, grid, dim3(256), 0, stream, dout, y_perm,
                             row_of, topk_w, (__nv_bfloat16 *)gy, dw, T, k, D, (long long)rows_alloc,
                             status)
                : launch_pdl(combine_bwd_kernel<false>, grid, dim3(256), 0, stream, dout, y_perm,
                             row_of, topk_w, (__nv_bfloat16 *)gy, dw, T, k, D, (long long)rows_alloc,
                             status);
    if (e == cudaSuccess) count_launch();
    return e;
}

cudaError_t launch_dispatch_bwd(const float *dxp, const int *row_of, const float *add, void *dx,
                                int T, int D, int k, int64_t rows_alloc, int is_bf16,
                                cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const dim3 grid((unsigned)((T + 7) / 8));
    const cudaError_t e =
        is_bf16 ? launch_pdl(dispatch_bwd_kernel<true>, grid, dim3(256), 0, stream, dxp, row_of, add,
                             dx, T, k, D, (long long)rows_alloc)
                : launch_pdl(dispatch_bwd_kernel<false>, grid, dim3(256), 0, stream, dxp, row_of,
                             add, dx, T, k, D, (long long)rows_alloc);
    if (e == cudaSuccess) count_launch();
    return e;
}

cudaError_t launch_router_bwd(const void *x, const void *wg, const float *logits,
                              const int *topk_idx, const float *topk_w, const float *dw, float *dl,
                              float *dx_router, float *dwg, float *dbias, int T, int D, int E,
                              int k, int score, int renorm, int is_bf16, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    cudaError_t e = launch_pdl(router_dl_kernel, dim3((unsigned)((T + 7) / 8)), dim3(256), 0, stream,
                               logits, topk_idx, topk_w, dw, dl, T, E, k, score, renorm);
    if (e != cudaSuccess) return e;
    count_launch();
    if (dbias) {
        if ((e = launch_pdl(column_sum_kernel, dim3((unsigned)((E + 255) / 256)), dim3(256), 0,
                            stream, (const float *)dl, dbias, T, E)) != cudaSuccess)
            return e;
        count_launch();
    }
    // dwg [E, D] = dl^T x  (K = T);  dx_router [T, D] = dl wg  (K = E)
    if (is_bf16) {
        if ((e = simt_gemm<false, true>(dl, 1, E, x, D, 1, dwg, E, D, T, stream)) != cudaSuccess) return e;
        return simt_gemm<false, true>(dl, E, 1, wg, D, 1, dx_router, T, D, E, stream);
    }
    if ((e = simt_gemm<false, false>(dl, 1, E, x, D, 1, dwg, E, D, T, stream)) != cudaSuccess) return e;
    return simt_gemm<false, false>(dl, E, 1, wg, D, 1, dx_router, T, D, E, stream);
}

}  // namespace moe
