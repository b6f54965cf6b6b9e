// fa_bwd_mask_add.cu -- backward plans with the forward's additive mask (with
// or without dropout, window and offset).
#include "fa_bwd_impl.cuh"

namespace fa {

int launch_bwd_mask_add(const BwdLaunchArgs& a) {
  using namespace bwd_impl;
  if (a.dropout_p != 0.0f) {
    if (a.f16) return a.D == 64 ? launch_bwd_d<64, true, true, true, 2>(a) : launch_bwd_d<128, true, true, true, 2>(a);
    return a.D == 64 ? launch_bwd_d<64, false, true, true, 2>(a) : launch_bwd_d<128, false, true, true, 2>(a);
  }
  if (a.f16) return a.D == 64 ? launch_bwd_d<64, true, true, false, 2>(a) : launch_bwd_d<128, true, true, false, 2>(a);
  return a.D == 64 ? launch_bwd_d<64, false, true, false, 2>(a) : launch_bwd_d<128, false, true, false, 2>(a);
}

}  // namespace fa
