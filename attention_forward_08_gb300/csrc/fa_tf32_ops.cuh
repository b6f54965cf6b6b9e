// fa_tf32_ops.cuh -- the HBM-bound preparation kernels of the fp32 (TF32)
// paths: round a [B, H, rows, D] view to tf32 in a contiguous copy, and write
// a tf32-rounded transpose [B, H, D, row_len] (rows innermost, zero-padded to
// row_len).  The tensor core reads fp32 operands as tf32 and drops their low
// 13 mantissa bits, so rounding (to nearest) first keeps the products
// accurate; and a tf32 MMA takes its B operand K-major only, so products whose
// reduction runs over rows read the transpose.  Used by the forward's pre-pass
// (fa_tf32_prep.cu) and the fp32 backward (fa_bwd_tf32.cu).
#pragma once

#include <cuda_runtime.h>

#include "fa_ptx.cuh"

namespace fa {

namespace {

// Rounds a strided [B, H, rows, D] fp32 view into a contiguous copy: one
// thread per 4 consecutive elements of the destination (16-byte accesses; the
// source strides are multiples of 4 elements, checked by the caller).
__global__ void __launch_bounds__(256) tf32_round_rows_kernel(const float* __restrict__ src, long long sb,
                                                              long long sh, long long sr, float* __restrict__ dst,
                                                              int H, int rows, int D, long long n4) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (long long)gridDim.x * blockDim.x) {
    const long long e = i * 4;
    const int d = (int)(e % D);
    const long long rr = e / D;
    const int r = (int)(rr % rows);
    const long long bh = rr / rows;
    const int h = (int)(bh % H);
    const long long b = bh / H;
    const float4 v = __ldg(reinterpret_cast<const float4*>(src + b * sb + h * sh + r * sr + d));
    float4 o;
    o.x = __uint_as_float(to_tf32(v.x));
    o.y = __uint_as_float(to_tf32(v.y));
    o.z = __uint_as_float(to_tf32(v.z));
    o.w = __uint_as_float(to_tf32(v.w));
    reinterpret_cast<float4*>(dst)[i] = o;
  }
}

// V [B, H, kL, D] (strided) -> tf32-rounded V^T [B, H, D, vt_row]: 32 x 32
// tiles through shared memory (reads along D, writes along keys, both
// coalesced).  Block (32, 8); grid (vt_row / 32 rounded up, D / 32, up to
// 65535), the z blocks striding over the BH = B * H (batch, head) pairs.
__global__ void __launch_bounds__(256) tf32_transpose_v_kernel(const float* __restrict__ v, long long sb,
                                                               long long sh, long long sr, float* __restrict__ vt,
                                                               int H, long long BH, int kL, int D,
                                                               long long vt_row) {
  __shared__ float tile[32][33];
  const int k0 = blockIdx.x * 32, d0 = blockIdx.y * 32;
  for (long long bh = blockIdx.z; bh < BH; bh += gridDim.z) {
    const long long b = bh / H, h = bh % H;
    const float* src = v + b * sb + h * sh;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int key = k0 + threadIdx.y + 8 * i;
      const float x = key < kL ? __ldg(src + (long long)key * sr + d0 + threadIdx.x) : 0.0f;
      tile[threadIdx.y + 8 * i][threadIdx.x] = __uint_as_float(to_tf32(x));
    }
    __syncthreads();
    float* dst = vt + bh * D * vt_row;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int d = d0 + threadIdx.y + 8 * i;
      const int key = k0 + threadIdx.x;
      if (key < vt_row) dst[(long long)d * vt_row + key] = tile[threadIdx.x][threadIdx.y + 8 * i];
    }
    __syncthreads();  // the tile is refilled for the next (b, h)
  }
}

}  // namespace

}  // namespace fa
