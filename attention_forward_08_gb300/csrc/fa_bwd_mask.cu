// fa_bwd_mask.cu -- backward plans with the forward's bool mask (with or
// without dropout, window and offset).
#include "fa_bwd_impl.cuh"

namespace fa {

int launch_bwd_mask(const BwdLaunchArgs& a) {
  using namespace bwd_impl;
  if (a.dropout_p != 0.0f) {
    if (a.f16) return a.D == 64 ? launch_bwd_d<64, true, true, true, 1>(a) : launch_bwd_d<128, true, true, true, 1>(a);
    return a.D == 64 ? launch_bwd_d<64, false, true, true, 1>(a) : launch_bwd_d<128, false, true, true, 1>(a);
  }
  if (a.f16) return a.D == 64 ? launch_bwd_d<64, true, true, false, 1>(a) : launch_bwd_d<128, true, true, false, 1>(a);
  return a.D == 64 ? launch_bwd_d<64, false, true, false, 1>(a) : launch_bwd_d<128, false, true, false, 1>(a);
}

}  // namespace fa
