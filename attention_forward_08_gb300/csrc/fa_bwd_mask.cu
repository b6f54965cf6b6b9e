// fa_bwd_mask.cu -- backward plans with the forward's bool or additive mask
// (with or without dropout, window and offset).
#include "fa_bwd_impl.cuh"

namespace fa {

int launch_bwd_mask(const BwdLaunchArgs& a) {
  using namespace bwd_impl;
  if (a.dropout_p != 0.0f) {
    if (a.f16)
      return a.D == 64 ? launch_bwd_d<64, true, true, true, true>(a) : launch_bwd_d<128, true, true, true, true>(a);
    return a.D == 64 ? launch_bwd_d<64, false, true, true, true>(a) : launch_bwd_d<128, false, true, true, true>(a);
  }
  if (a.f16)
    return a.D == 64 ? launch_bwd_d<64, true, true, false, true>(a) : launch_bwd_d<128, true, true, false, true>(a);
  return a.D == 64 ? launch_bwd_d<64, false, true, false, true>(a) : launch_bwd_d<128, false, true, false, true>(a);
}

}  // namespace fa
