// The f16 D=64 forward plan with sliding window, softcap and query offset
// compiled in, and the same plan with dropout as well (their own translation
// unit, built in parallel with the rest).
#include "fa_launch.cuh"

namespace fa {
int launch_feat_f16_d64(const LaunchArgs& a) { return launch_fa_fwd<WithFeat<CfgF16D64>>(a); }
int launch_drop_f16_d64(const LaunchArgs& a) { return launch_fa_fwd<WithDrop<CfgF16D64>>(a); }
}  // namespace fa
