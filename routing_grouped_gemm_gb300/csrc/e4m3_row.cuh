// Row-wise e4m3 quantisation of one bf16 row by one warp, shared by the
// standalone quantiser and the quantising dispatch.
//
// Page "Expert Parallelism (EP)" (llm-infra-atlas), its FP8 dispatch (the
// dispatched activations travel as e4m3 values with scales into an FP8
// grouped GEMM).  The scale granularity is not on the page; the reading
// taken is one binary32 scale per row:
//   amax = max_c |x[r, c]|,  s[r] = amax / 448 (1 when amax is 0),
//   q[r, c] = e4m3(x[r, c] / s[r])   (nearest, ties to even, saturating),
// with both divisions correctly rounded binary32 operations, so that the
// codes are a deterministic function of the bf16 input.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace moe {

__device__ __forceinline__ void unpack8_bf16(const uint4 v, float (&f)[8]) {
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

// x: the row's nv = cols / 8 16-byte vectors.  Lane j < n_dst holds in
// my_row the destination row of copy j (-1: none); the codes go to rows
// my_row of dst ([*, cols] bytes) and the scale to scale[my_row].  A first
// pass finds amax, the second forms the codes (the row comes back from L1).
__device__ __forceinline__ void quantize_row_e4m3_warp(const uint4 *__restrict__ x, int cols,
                                                       int my_row, int n_dst,
                                                       uint8_t *__restrict__ dst,
                                                       float *__restrict__ scale, int lane) {
    const int nv = cols / 8;
    float amax = 0.f;
    for (int v = lane; v < nv; v += 32) {
        float f[8];
        unpack8_bf16(x[v], f);
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
        unpack8_bf16(__ldcs(x + v), f);  // last read of this row
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

}  // namespace moe
