// The one-Q-tile bf16 D=64 forward plan for small grids (its own translation
// unit, built in parallel with the rest).
#include "fa_launch.cuh"

namespace fa {
int launch_q1_bf16_d64(const LaunchArgs& a) { return launch_fa_fwd<CfgBf16D64Q1>(a); }
}  // namespace fa
