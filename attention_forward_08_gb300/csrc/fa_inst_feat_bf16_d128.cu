// The bf16 D=128 forward plan with sliding window, softcap and query offset
// compiled in, and the same plan with dropout as well (their own translation
// unit, built in parallel with the rest).
#include "fa_launch.cuh"

namespace fa {
int launch_feat_bf16_d128(const LaunchArgs& a) { return launch_fa_fwd<WithFeat<CfgBf16D128>>(a); }
int launch_drop_bf16_d128(const LaunchArgs& a) { return launch_fa_fwd<WithDrop<CfgBf16D128>>(a); }
}  // namespace fa
