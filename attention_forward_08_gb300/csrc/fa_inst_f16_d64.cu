// One instantiation of the forward kernel and its launcher (compiled on its
// own so the variants build in parallel).
#include "fa_launch.cuh"

namespace fa {
int launch_f16_d64(const LaunchArgs& a) { return launch_fa_fwd<CfgF16D64>(a); }
}  // namespace fa
