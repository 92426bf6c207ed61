// FP8 e4m3 dispatch: row-wise quantisation of bf16 rows.
//
// Page "Expert Parallelism (EP)" (llm-infra-atlas), its FP8 dispatch (the
// dispatched activations travel as e4m3 values with scales into an FP8
// grouped GEMM).  The scale granularity is not on the page; the reading
// taken is one binary32 scale per row:
//   amax = max_c |x[r, c]|,  s[r] = amax / 448 (1 when amax is 0),
//   q[r, c] = e4m3(x[r, c] / s[r])   (nearest, ties to even, saturating),
// with both divisions correctly rounded binary32 operations, so that the
// codes are a deterministic function of the bf16 input.  Per-row scales
// factor out of a GEMM's K sum: the grouped GEMM applies s_x[row] * s_w[col]
// to its fp32 accumulator in the epilogue.
//
// One warp per row: a first pass finds amax (16-byte loads), the second
// forms the codes (the row comes back from L1) and writes them to every
// destination row -- the k dispatched rows of a token (row_of), or the row
// itself.
#include <cuda_fp8.h>

#include "common.cuh"
#include "launch.h"

namespace moe {
namespace {

__device__ __forceinline__ void unpack8(const uint4 v, float (&f)[8]) {
    const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __low2float(h2[i]);
        f[2 * i + 1] = __high2float(h2[i]);
    }
}

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
    return (lo & 0xFFFFu) | (hi << 16);
}

// rows x cols bf16 (cols % 8 == 0) -> codes and one scale per row.  With
// row_of ([rows, k]) the codes of row t go to rows row_of[t, j] of dst (and
// the scale to scale[row_of[t, j]]), skipping -1; without it to row t.
__global__ void __launch_bounds__(256)
quantize_rows_e4m3_kernel(const uint4 *__restrict__ src, long long rows, int cols,
                          const int *__restrict__ row_of, int k, uint8_t *__restrict__ dst,
                          float *__restrict__ scale) {
    griddep_launch_dependents();  // the next kernel may be scheduled now
    griddep_wait();               // every input of this kernel is complete
    const long long t = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (t >= rows) return;
    const int nv = cols / 8;
    const uint4 *x = src + (size_t)t * nv;
    int my_row = -1;
    if (row_of) {
        if (lane < k) my_row = row_of[(size_t)t * k + lane];
    } else if (lane == 0) {
        my_row = (int)t;
    }
    const int n_dst = row_of ? k : 1;
    float amax = 0.f;
    for (int v = lane; v < nv; v += 32) {
        float f[8];
        unpack8(x[v], f);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float a = fabsf(f[i]);
            amax = a > amax ? a : amax;  // NaN never replaces the running max
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float b = __shfl_xor_sync(0xffffffffu, amax, o);
        amax = b > amax ? b : amax;
    }
    const float s = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
    for (int v = lane; v < nv; v += 32) {
        float f[8];
        unpack8(__ldcs(x + v), f);  // last read of this row
        uint2 q;
        q.x = e4m3x4(__fdiv_rn(f[0], s), __fdiv_rn(f[1], s), __fdiv_rn(f[2], s), __fdiv_rn(f[3], s));
        q.y = e4m3x4(__fdiv_rn(f[4], s), __fdiv_rn(f[5], s), __fdiv_rn(f[6], s), __fdiv_rn(f[7], s));
        for (int j = 0; j < n_dst; ++j) {
            const int r = __shfl_sync(0xffffffffu, my_row, j);
            if (r < 0) continue;
            reinterpret_cast<uint2 *>(dst + (size_t)r * cols)[v] = q;
        }
    }
    if (lane < n_dst && my_row >= 0) scale[my_row] = s;
}

}  // namespace

cudaError_t launch_quantize_rows_e4m3(const void *src, int64_t rows, int cols, const int *row_of,
                                      int k, uint8_t *dst, float *scale, cudaStream_t stream) {
    if (rows == 0) return cudaSuccess;
    if (cols % 8 || k > 32) return cudaErrorInvalidValue;
    const unsigned blocks = (unsigned)((rows + 7) / 8);
    const cudaError_t e = launch_pdl(quantize_rows_e4m3_kernel, dim3(blocks), dim3(256), 0, stream,
                                     (const uint4 *)src, (long long)rows, cols, row_of, k, dst,
                                     scale);
    if (e == cudaSuccess) count_launch();
    return e;
}

}  // namespace moe
