// fa_tf32_prep.cu -- the pre-pass of the fp32 (TF32) forward and the three
// kernel plans it feeds.
//
// The tensor core reads fp32 operands as tf32 and ignores their low 13
// mantissa bits, so Q, K and V are rounded to tf32 (round to nearest) before
// the products; and a tf32 MMA takes its B operand K-major only, so O += P V
// needs V transposed (keys innermost).  Without a workspace the forward
// kernel does both in shared memory with helper warps for every tile it
// loads.  With one, this pass does them once in HBM:
//   qr = tf32(Q)    contiguous [B, H_q, qL, D]
//   kr = tf32(K)    contiguous [B, H_kv, kL, D]
//   vt = tf32(V)^T  [B, H_kv, D, vt_row], vt_row = kL rounded up to a multiple
//                   of 4 (16-byte rows for TMA), the pad columns zero
// and the forward kernel then streams them by TMA like the 16-bit plans.
// HBM-bound: each input is read once and each output written once.
#include <cuda_runtime.h>

#include <algorithm>

#include "fa_launch.cuh"

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
// coalesced).  Block (32, 8); grid (vt_row / 32 rounded up, D / 32, B * H).
__global__ void __launch_bounds__(256) tf32_transpose_v_kernel(const float* __restrict__ v, long long sb,
                                                               long long sh, long long sr, float* __restrict__ vt,
                                                               int H, int kL, int D, long long vt_row) {
  __shared__ float tile[32][33];
  const int k0 = blockIdx.x * 32, d0 = blockIdx.y * 32;
  const long long bh = blockIdx.z;
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
}

int check_launch(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("%s launch failed: %s", what, cudaGetErrorString(e));
    return 4;
  }
  return 0;
}

}  // namespace

int launch_tf32_prep(const LaunchArgs& a, float* qr, float* kr, float* vt) {
  const int grid_cap = (a.num_sms > 0 ? a.num_sms : 1) * 8;
  auto blocks_for = [&](long long n4) { return (unsigned)std::min<long long>((n4 + 255) / 256, grid_cap); };
  const long long nq4 = (long long)a.B * a.Hq * a.qL * a.D / 4, nk4 = (long long)a.B * a.Hkv * a.kL * a.D / 4;
  tf32_round_rows_kernel<<<blocks_for(nq4), 256, 0, a.stream>>>(static_cast<const float*>(a.q), a.qs[0], a.qs[1],
                                                                 a.qs[2], qr, a.Hq, a.qL, a.D, nq4);
  if (int rc = check_launch("tf32 rounding of Q")) return rc;
  tf32_round_rows_kernel<<<blocks_for(nk4), 256, 0, a.stream>>>(static_cast<const float*>(a.k), a.ks[0], a.ks[1],
                                                                 a.ks[2], kr, a.Hkv, a.kL, a.D, nk4);
  if (int rc = check_launch("tf32 rounding of K")) return rc;
  const dim3 grid((unsigned)((a.vt_row + 31) / 32), (unsigned)(a.D / 32), (unsigned)(a.B * a.Hkv));
  tf32_transpose_v_kernel<<<grid, dim3(32, 8), 0, a.stream>>>(static_cast<const float*>(a.v), a.vs[0], a.vs[1],
                                                              a.vs[2], vt, a.Hkv, a.kL, a.D, a.vt_row);
  return check_launch("tf32 transpose of V");
}

int launch_pre_f32_d64(const LaunchArgs& a) { return launch_fa_fwd<CfgF32PreD64>(a); }
int launch_pre_f32_d128(const LaunchArgs& a) { return launch_fa_fwd<CfgF32PreD128>(a); }
int launch_pre_f32_d256(const LaunchArgs& a) { return launch_fa_fwd<CfgF32PreD256>(a); }

}  // namespace fa
