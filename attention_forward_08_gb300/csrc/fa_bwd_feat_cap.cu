// fa_bwd_feat_cap.cu -- backward plans with a softcap (and sliding window /
// causal offset).
#include "fa_bwd_impl.cuh"

namespace fa {

int launch_bwd_feat_cap(const BwdLaunchArgs& a) {
  using namespace bwd_impl;
  if (a.f16)
    return a.D == 64 ? launch_bwd_d<64, true, true, false, 0, true>(a) : launch_bwd_d<128, true, true, false, 0, true>(a);
  return a.D == 64 ? launch_bwd_d<64, false, true, false, 0, true>(a) : launch_bwd_d<128, false, true, false, 0, true>(a);
}

}  // namespace fa
