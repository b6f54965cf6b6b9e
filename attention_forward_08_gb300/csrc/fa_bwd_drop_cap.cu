// fa_bwd_drop_cap.cu -- backward plans with the forward's dropout and a
// softcap (and window / offset).
#include "fa_bwd_impl.cuh"

namespace fa {

int launch_bwd_drop_cap(const BwdLaunchArgs& a) {
  using namespace bwd_impl;
  if (a.f16)
    return a.D == 64 ? launch_bwd_d<64, true, true, true, 0, true>(a) : launch_bwd_d<128, true, true, true, 0, true>(a);
  return a.D == 64 ? launch_bwd_d<64, false, true, true, 0, true>(a) : launch_bwd_d<128, false, true, true, 0, true>(a);
}

}  // namespace fa
