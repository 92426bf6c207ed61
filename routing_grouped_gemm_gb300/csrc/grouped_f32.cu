// fp32 m-grouped SwiGLU expert FFN on CUDA cores (FFMA).
//
// Page "Expert Parallelism (EP)" (llm-infra-atlas), section 1 (routed
// experts: grouped fc1 -> act -> fc2 over the permuted rows) and section 2
// (one m-grouped kernel over same-shaped GEMMs whose M differs, a tile
// scheduler spanning the groups).  Weight shapes from "Expert Tensor
// Parallel design", section 4.3: w1/w3 [E, H, D], w2 [E, D, H].
//
// The fp32 workload asks for 1e-4 relative accuracy, which TF32 tensor
// cores would not meet, so this path stays in fp32 FFMA.  Each CTA computes
// one 64 x 64 output tile of one expert; the tile table (per-expert m-tiles
// over the valid rows of each segment) is rebuilt by each CTA from the
// segment offsets in device memory, so no host synchronisation is needed.
#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

constexpr int F_BM = 64, F_BN = 64, F_BK = 32, F_THREADS = 256;
constexpr int F_PER = F_BM * F_BK / F_THREADS;  // tile elements each thread stages per k-step
constexpr int F_LD = F_BM + 4;
constexpr int F_MAX_EXPERTS = 1024;

template <int MODE>  // 1: h = SiLU(A w1^T) * (A w3^T); 2: y = A w2^T
__global__ void __launch_bounds__(F_THREADS)
grouped_f32_kernel(const float *__restrict__ A, int K, const float *__restrict__ Bg,
                   const float *__restrict__ Bu, int N, float *__restrict__ out,
                   const int *__restrict__ seg_off, const int *__restrict__ tpe, int e_first,
                   int E_local, long long rows_alloc, int n_tiles, int *status) {
    griddep_launch_dependents();  // the next kernel may be scheduled now
    griddep_wait();               // every input of this kernel is complete
    __shared__ int s_base[F_MAX_EXPERTS], s_valid[F_MAX_EXPERTS], s_mtoff[F_MAX_EXPERTS + 1];
    __shared__ float As[F_BK][F_LD], Bgs[F_BK][F_LD], Bus[F_BK][F_LD];

    const int tid = threadIdx.x;
    if (tid < 32)
        build_tile_table(tid, E_local, e_first, (int)rows_alloc, F_BM, seg_off, tpe, s_base,
                         s_valid, s_mtoff, blockIdx.x == 0 ? status : nullptr);
    __syncthreads();
    const int total = s_mtoff[E_local] * n_tiles;
    const int tile = blockIdx.x;
    if (tile >= total) return;
    const int mt = tile / n_tiles, nt = tile % n_tiles;
    const int i = tile_expert(s_mtoff, E_local, mt);
    const int lm = mt - s_mtoff[i];
    const int row0 = s_base[i] + lm * F_BM;
    const int nvalid = min(F_BM, s_valid[i] - lm * F_BM);
    const int n0 = nt * F_BN;
    const size_t bstride = (size_t)N * K;  // per-expert weight stride
    const float *Bg_e = Bg + (size_t)i * bstride;
    const float *Bu_e = (MODE == 1) ? Bu + (size_t)i * bstride : nullptr;

    const int ty = tid / 16, tx = tid % 16;
    float accg[4][4], accu[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int b = 0; b < 4; ++b) accg[a][b] = accu[a][b] = 0.f;

    // the next k-step's tiles are loaded into registers while this one is
    // multiplied out of shared memory
    float ra[F_PER], rg[F_PER], ru[F_PER];
    auto load_tiles = [&](int k0) {
#pragma unroll
        for (int q = 0; q < F_PER; ++q) {
            const int e = tid + q * F_THREADS;
            const int r = e / F_BK, kk = e % F_BK;
            ra[q] = (r < nvalid && k0 + kk < K) ? A[(size_t)(row0 + r) * K + k0 + kk] : 0.f;
            const int n = n0 + r;
            const bool okb = n < N && k0 + kk < K;
            rg[q] = okb ? Bg_e[(size_t)n * K + k0 + kk] : 0.f;
            if (MODE == 1) ru[q] = okb ? Bu_e[(size_t)n * K + k0 + kk] : 0.f;
        }
    };
    load_tiles(0);
    for (int k0 = 0; k0 < K; k0 += F_BK) {
#pragma unroll
        for (int q = 0; q < F_PER; ++q) {
            const int e = tid + q * F_THREADS;
            const int r = e / F_BK, kk = e % F_BK;
            As[kk][r] = ra[q];
            Bgs[kk][r] = rg[q];
            if (MODE == 1) Bus[kk][r] = ru[q];
        }
        __syncthreads();
        if (k0 + F_BK < K) load_tiles(k0 + F_BK);
#pragma unroll
        for (int kk = 0; kk < F_BK; ++kk) {
            float av[4], gv[4], uv[4];
#pragma unroll
            for (int a = 0; a < 4; ++a) av[a] = As[kk][ty + 16 * a];
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                gv[b] = Bgs[kk][tx + 16 * b];
                if (MODE == 1) uv[b] = Bus[kk][tx + 16 * b];
            }
#pragma unroll
            for (int a = 0; a < 4; ++a)
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    accg[a][b] = fmaf(av[a], gv[b], accg[a][b]);
                    if (MODE == 1) accu[a][b] = fmaf(av[a], uv[b], accu[a][b]);
                }
        }
        __syncthreads();
    }
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        const int r = ty + 16 * a;
        if (r >= nvalid) continue;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int c = n0 + tx + 16 * b;
            if (c >= N) continue;
            float v = accg[a][b];
            if (MODE == 1) v = v / (1.f + expf(-v)) * accu[a][b];
            out[(size_t)(row0 + r) * N + c] = v;
        }
    }
}

}  // namespace

cudaError_t launch_grouped_swiglu_f32(const float *x_perm, const int *seg_offsets,
                                      const int *tokens_per_expert, const float *w1,
                                      const float *w3, const float *w2, float *h, float *y_perm,
                                      int D, int H_local, int e_first, int E_local,
                                      int64_t rows_alloc, int *status, cudaStream_t stream) {
    if (E_local == 0 || rows_alloc == 0) return cudaSuccess;
    const long long mt_bound = (rows_alloc + F_BM - 1) / F_BM + E_local;
    const int nt1 = (H_local + F_BN - 1) / F_BN;
    const int nt2 = (D + F_BN - 1) / F_BN;
    cudaError_t err = launch_pdl(grouped_f32_kernel<1>, dim3((unsigned)(mt_bound * nt1)),
                                 dim3(F_THREADS), 0, stream, x_perm, D, w1, w3, H_local, h,
                                 seg_offsets, tokens_per_expert, e_first, E_local, rows_alloc,
                                 nt1, status);
    if (err != cudaSuccess) return err;
    count_launch();
    err = launch_pdl(grouped_f32_kernel<2>, dim3((unsigned)(mt_bound * nt2)), dim3(F_THREADS), 0,
                     stream, h, H_local, w2, nullptr, D, y_perm, seg_offsets, tokens_per_expert,
                     e_first, E_local, rows_alloc, nt2, nullptr);
    if (err != cudaSuccess) return err;
    count_launch();
    return cudaSuccess;
}

}  // namespace moe
