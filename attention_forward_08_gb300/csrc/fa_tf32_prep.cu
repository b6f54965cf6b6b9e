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
#include "fa_tf32_ops.cuh"

namespace fa {

namespace {

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
  const long long BH = (long long)a.B * a.Hkv;
  const dim3 grid((unsigned)((a.vt_row + 31) / 32), (unsigned)(a.D / 32), (unsigned)std::min<long long>(BH, 65535));
  tf32_transpose_v_kernel<<<grid, dim3(32, 8), 0, a.stream>>>(static_cast<const float*>(a.v), a.vs[0], a.vs[1],
                                                              a.vs[2], vt, a.Hkv, BH, a.kL, a.D, a.vt_row);
  return check_launch("tf32 transpose of V");
}

int launch_pre_f32_d64(const LaunchArgs& a) { return launch_fa_fwd<CfgF32PreD64>(a); }
int launch_pre_f32_d128(const LaunchArgs& a) { return launch_fa_fwd<CfgF32PreD128>(a); }
int launch_pre_f32_d256(const LaunchArgs& a) { return launch_fa_fwd<CfgF32PreD256>(a); }

}  // namespace fa
