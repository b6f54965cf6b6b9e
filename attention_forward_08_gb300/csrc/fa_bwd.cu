// fa_bwd.cu -- the backward pass's dispatcher (launch_bwd) and the plain
// plans at head dims 64 and 128: bf16 or fp16 I/O, no window, offset,
// softcap, dropout or mask.  The other plans live in fa_bwd_feat.cu,
// fa_bwd_drop.cu, fa_bwd_mask.cu (bool mask), fa_bwd_mask_add.cu (additive
// mask), fa_bwd256.cu (head dim 256) and fa_bwd_tf32.cu (fp32 I/O): separate
// translation units, compiled in parallel.
#include "fa_bwd_impl.cuh"

namespace fa {

int launch_bwd_feat(const BwdLaunchArgs& a);  // fa_bwd_feat.cu
int launch_bwd_drop(const BwdLaunchArgs& a);  // fa_bwd_drop.cu
int launch_bwd_mask(const BwdLaunchArgs& a);      // fa_bwd_mask.cu
int launch_bwd_mask_add(const BwdLaunchArgs& a);  // fa_bwd_mask_add.cu
int launch_bwd256(const BwdLaunchArgs& a);    // fa_bwd256.cu
int launch_bwd_tf32(const BwdLaunchArgs& a);  // fa_bwd_tf32.cu

int launch_bwd(const BwdLaunchArgs& a) {
  using namespace bwd_impl;
  if (a.f32) return launch_bwd_tf32(a);     // plain plans only (the validator refuses the rest)
  if (a.D == 256) return launch_bwd256(a);  // plain plans only (the validator refuses the rest)
  if (a.mask_kind == 1) return launch_bwd_mask(a);
  if (a.mask_kind == 2) return launch_bwd_mask_add(a);
  if (a.dropout_p != 0.0f) return launch_bwd_drop(a);
  if (a.window != 0 || a.q_offset != 0 || a.softcap != 0.0f) return launch_bwd_feat(a);
  if (a.f16) return a.D == 64 ? launch_bwd_d<64, true, false>(a) : launch_bwd_d<128, true, false>(a);
  return a.D == 64 ? launch_bwd_d<64, false, false>(a) : launch_bwd_d<128, false, false>(a);
}

}  // namespace fa
