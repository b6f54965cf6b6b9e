// fa_bwd_feat.cu -- backward plans with sliding window / causal offset and no
// softcap (the softcap plans: fa_bwd_feat_cap.cu).
#include "fa_bwd_impl.cuh"

namespace fa {

int launch_bwd_feat_cap(const BwdLaunchArgs& a);  // fa_bwd_feat_cap.cu

int launch_bwd_feat(const BwdLaunchArgs& a) {
  using namespace bwd_impl;
  if (a.softcap != 0.0f) return launch_bwd_feat_cap(a);
  if (a.f16) return a.D == 64 ? launch_bwd_d<64, true, true>(a) : launch_bwd_d<128, true, true>(a);
  return a.D == 64 ? launch_bwd_d<64, false, true>(a) : launch_bwd_d<128, false, true>(a);
}

}  // namespace fa
