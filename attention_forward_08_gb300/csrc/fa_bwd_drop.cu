// fa_bwd_drop.cu -- backward plans with the forward's dropout (and window /
// offset) and no softcap (dropout with a softcap: fa_bwd_drop_cap.cu).
#include "fa_bwd_impl.cuh"

namespace fa {

int launch_bwd_drop_cap(const BwdLaunchArgs& a);  // fa_bwd_drop_cap.cu

int launch_bwd_drop(const BwdLaunchArgs& a) {
  using namespace bwd_impl;
  if (a.softcap != 0.0f) return launch_bwd_drop_cap(a);
  if (a.f16) return a.D == 64 ? launch_bwd_d<64, true, true, true>(a) : launch_bwd_d<128, true, true, true>(a);
  return a.D == 64 ? launch_bwd_d<64, false, true, true>(a) : launch_bwd_d<128, false, true, true>(a);
}

}  // namespace fa
