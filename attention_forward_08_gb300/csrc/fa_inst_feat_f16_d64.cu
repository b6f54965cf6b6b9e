// The f16 D=64 forward plan with sliding window, softcap and query offset
// compiled in (its own translation unit, built in parallel with the rest).
#include "fa_launch.cuh"

namespace fa {
int launch_feat_f16_d64(const LaunchArgs& a) { return launch_fa_fwd<WithFeat<CfgF16D64>>(a); }
}  // namespace fa
