"""Failure containment on the GPU without a fault: with a one-cycle wait bound
the kernel's bounded waits run out, every role unwinds (in-flight copies and
MMAs are drained, TMEM is freed), the host reads FA_ERR_DEVICE_TIMEOUT from
the status word, and the context stays usable for a correct run."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import compare, fp32_scale, oracle_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("bf16", 256), ("f32", 128)])
def test_wait_bound_reports_timeout_then_recovers(dtype, D):
    import attention_forward_08_gb300 as fa
    w = W.small_case(f"timeout_{dtype}_{D}", 1, 4, 2, 640, 640, D, dtype, causal=True, seed=21)
    q, k, v = W.make_qkv(w)
    dev = "cuda:0"
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    assert fa.fa_sync_status(None) == fa.fa.FA_OK
    try:
        fa.fa_set_timeout_cycles(1)
        fa.attention(qd, kd, vd, scale=w.sm_scale, causal=True)
        rc = fa.fa_sync_status(None)
    finally:
        fa.fa_set_timeout_cycles(0)
    assert rc == fa.fa.FA_ERR_DEVICE_TIMEOUT, fa.fa_last_error()
    assert fa.fa_sync_status(None) == fa.fa.FA_OK   # the status word was cleared
    o, lse = fa.attention(qd, kd, vd, scale=w.sm_scale, causal=True)
    assert fa.fa_sync_status(None) == fa.fa.FA_OK
    qo, ko, vo, _ = oracle_inputs(q, k, v, None)
    o_r, l_r = oracle.attention(qo, ko, vo, fp32_scale(w), causal=True)
    compare(w, o.double().cpu().numpy(), lse.double().cpu().numpy(), o_r, l_r, what=w.name)
