// The f32 D=256 forward plan with sliding window, softcap and query offset
// compiled in, and the same plan with dropout as well (their own translation
// unit, built in parallel with the rest).
#include "fa_launch.cuh"

namespace fa {
int launch_feat_f32_d256(const LaunchArgs& a) { return launch_fa_fwd<WithFeat<CfgF32D256>>(a); }
int launch_drop_f32_d256(const LaunchArgs& a) { return launch_fa_fwd<WithDrop<CfgF32D256>>(a); }
}  // namespace fa
