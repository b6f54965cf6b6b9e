// fa_bwd_drop.cu -- backward plans with the forward's dropout (and the other features).
#include "fa_bwd_impl.cuh"

namespace fa {

int launch_bwd_drop(const BwdLaunchArgs& a) {
  using namespace bwd_impl;
  if (a.f16) return a.D == 64 ? launch_bwd_d<64, true, true, true>(a) : launch_bwd_d<128, true, true, true>(a);
  return a.D == 64 ? launch_bwd_d<64, false, true, true>(a) : launch_bwd_d<128, false, true, true>(a);
}

}  // namespace fa
