"""GB300 (sm_103a) FlashAttention-2: the forward pass (O and the natural-log
logsumexp L) and its gradients (dQ, dK, dV).

The computation runs in ``libfa_gb300.so`` (hand-written CUDA: TMA, tcgen05,
TMEM); this package only builds it (``_build``) and binds its C ABI (``fa``).
"""
from .fa import (FA_DTYPE_BF16, FA_DTYPE_F16, FA_DTYPE_F32, FA_MASK_ADDITIVE, FA_MASK_BOOL, FA_MASK_NONE, FaBwdArgs,
                 FaError, FaFwdArgs, attach_workspace, attention, attention_bwd, fa_bwd, fa_bwd_ex,
                 fa_bwd_ex_workspace_bytes, fa_bwd_full, fa_bwd_full_workspace_bytes, fa_bwd_workspace_bytes, fa_fwd,
                 fa_fwd_ex, fa_fwd_workspace_bytes, fa_last_error, fa_set_max_ctas, fa_set_q_tiles, fa_set_kv_splits,
                 fa_set_timeout_cycles, fa_sync_status, fa_version, load_library, make_args)

__all__ = ["attach_workspace", "attention", "attention_bwd", "fa_bwd", "fa_bwd_ex", "fa_bwd_ex_workspace_bytes",
           "fa_bwd_full", "fa_bwd_full_workspace_bytes", "fa_bwd_workspace_bytes", "fa_fwd", "fa_fwd_ex",
           "fa_fwd_workspace_bytes", "fa_last_error", "fa_sync_status", "fa_set_timeout_cycles",
           "fa_set_max_ctas", "fa_set_q_tiles", "fa_set_kv_splits", "fa_version", "load_library", "make_args", "FaFwdArgs", "FaBwdArgs",
           "FaError", "FA_DTYPE_BF16", "FA_DTYPE_F16", "FA_DTYPE_F32", "FA_MASK_NONE", "FA_MASK_BOOL",
           "FA_MASK_ADDITIVE"]
