// FP8 e4m3 dispatch: row-wise quantisation of bf16 rows (the arithmetic is
// in e4m3_row.cuh).  Per-row scales factor out of a GEMM's K sum: the
// grouped GEMM applies s_x[row] * s_w[col] to its fp32 accumulator in the
// epilogue.
//
// One warp per row, writing to every destination row -- the k dispatched
// rows of a token (row_of), or the row itself.
#include "common.cuh"
#include "e4m3_row.cuh"
#include "launch.h"

namespace moe {
namespace {

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
    int my_row = -1;
    if (row_of) {
        if (lane < k) my_row = row_of[(size_t)t * k + lane];
    } else if (lane == 0) {
        my_row = (int)t;
    }
    quantize_row_e4m3_warp(src + (size_t)t * (cols / 8), cols, my_row, row_of ? k : 1, dst, scale,
                           lane);
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
