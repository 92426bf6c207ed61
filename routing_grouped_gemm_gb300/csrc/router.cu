// Router: gating logits, top-k selection and routing weights, fused.
//
// Page "Expert Parallelism (EP)" (llm-infra-atlas), section 1: the router
// computes logits = x . W_g^T ([T, E]) and then "top-k + score_func" gives
// the routing probabilities and the routing map.  One CTA owns 32 tokens:
// it accumulates their logits for all E experts in fp32 (SIMT FFMA over
// shared-memory tiles), keeps them in shared memory, and one warp per token
// then selects the top-k by warp-wide arg-max rounds and computes weights.
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

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
    return __bfloat162float(v);
}

template <typename T>
__global__ void __launch_bounds__(RT_THREADS)
router_topk_kernel(const T *__restrict__ x, const T *__restrict__ wg, const float *__restrict__ bias,
                   float *__restrict__ logits_out, int *__restrict__ topk_idx,
                   float *__restrict__ topk_w, int Tn, int D, int E, int k, int score, int renorm,
                   int *status) {
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

        for (int d0 = 0; d0 < D; d0 += RT_BK) {
            // x slice: 32 tokens x 32 d, stored transposed [d][token]
            for (int i = tid; i < RT_TOKENS * RT_BK; i += RT_THREADS) {
                const int tt = i / RT_BK, dd = i % RT_BK;
                const int t = t0 + tt, d = d0 + dd;
                s_x[dd * SX_LD + tt] = (t < Tn && d < D) ? to_f32(x[(size_t)t * D + d]) : 0.f;
            }
            // W_g slice: 128 experts x 32 d, stored transposed [d][expert]
            for (int i = tid; i < RT_ECHUNK * RT_BK; i += RT_THREADS) {
                const int ee = i / RT_BK, dd = i % RT_BK;
                const int e = e0 + ee, d = d0 + dd;
                s_w[dd * SW_LD + ee] = (e < E && d < D) ? to_f32(wg[(size_t)e * D + d]) : 0.f;
            }
            __syncthreads();
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
        const float *l = s_logit + tt * E;
        bool any_nan = false;
        for (int e = lane; e < E; e += 32) any_nan |= (l[e] != l[e]);
        if (__any_sync(0xffffffffu, any_nan) && lane == 0) raise_flag(status, FLAG_BAD_ROUTING);

        // experts already chosen by this lane: bit q stands for expert lane + 32 q
        uint32_t taken = 0;
        int sel_e[32];
        float sel_v[32];
        for (int j = 0; j < k; ++j) {
            float bv = 0.f;
            int be = -1;
            for (int q = 0, e = lane; e < E; ++q, e += 32) {
                if (taken & (1u << q)) continue;
                if (be < 0 || key_before(l[e], e, bv, be)) { bv = l[e]; be = e; }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oe = __shfl_xor_sync(0xffffffffu, be, o);
                if (oe >= 0 && (be < 0 || key_before(ov, oe, bv, be))) { bv = ov; be = oe; }
            }
            if (be >= 0 && (be & 31) == lane) taken |= 1u << (be >> 5);
            sel_e[j] = be;
            sel_v[j] = bv;
        }

        // scores of the chosen experts
        float m = sel_v[0];  // the largest key (unless NaN)
        float denom = 1.f;
        if (score == 0 && !renorm) {
            float s = 0.f;
            for (int e = lane; e < E; e += 32) s += expf(l[e] - m);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
            denom = s;
        }
        if (lane == 0) {
            float p[32];
            float psum = 0.f;
            for (int j = 0; j < k; ++j) {
                p[j] = (score == 0) ? expf(sel_v[j] - m) : 1.f / (1.f + expf(-sel_v[j]));
                psum += p[j];
            }
            const float div = renorm ? psum : (score == 0 ? denom : 1.f);
            for (int j = 0; j < k; ++j) {
                topk_idx[(size_t)t * k + j] = sel_e[j];
                topk_w[(size_t)t * k + j] = p[j] / div;
            }
        }
    }
}

}  // namespace

cudaError_t launch_router_topk(const void *x, const void *wg, const float *bias, float *logits_out,
                               int *topk_idx, float *topk_w, int T, int D, int E, int k,
                               int score, int renorm, int is_bf16, int *status,
                               cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const size_t smem = sizeof(float) * ((size_t)RT_TOKENS * E + RT_BK * SX_LD + RT_BK * SW_LD);
    const dim3 grid((T + RT_TOKENS - 1) / RT_TOKENS);
    cudaError_t err;
    if (is_bf16) {
        auto kern = router_topk_kernel<__nv_bfloat16>;
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        kern<<<grid, RT_THREADS, smem, stream>>>((const __nv_bfloat16 *)x, (const __nv_bfloat16 *)wg,
                                                 bias, logits_out, topk_idx, topk_w, T, D, E, k,
                                                 score, renorm, status);
    } else {
        auto kern = router_topk_kernel<float>;
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (err != cudaSuccess) return err;
        kern<<<grid, RT_THREADS, smem, stream>>>((const float *)x, (const float *)wg, bias,
                                                 logits_out, topk_idx, topk_w, T, D, E, k, score,
                                                 renorm, status);
    }
    return cudaGetLastError();
}

}  // namespace moe
