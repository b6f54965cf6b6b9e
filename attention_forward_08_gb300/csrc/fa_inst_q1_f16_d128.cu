// The one-Q-tile f16 D=128 forward plan for small grids (its own translation
// unit, built in parallel with the rest).
#include "fa_launch.cuh"

namespace fa {
int launch_q1_f16_d128(const LaunchArgs& a) { return launch_fa_fwd<CfgF16D128Q1>(a); }
}  // namespace fa
