// The one-Q-tile bf16 D=128 forward plan for small grids (its own translation
// unit, built in parallel with the rest).
#include "fa_launch.cuh"

namespace fa {
int launch_q1_bf16_d128(const LaunchArgs& a) { return launch_fa_fwd<CfgBf16D128Q1>(a); }
}  // namespace fa
