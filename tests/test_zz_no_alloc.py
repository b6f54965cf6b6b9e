"""fa_bwd_noalloc (the backward with its D scratch in a built-in device array)
against fa_bwd with a caller workspace.

Named to be collected last.  The GPU test makes two calls in a row on
different problems (and repeats the first) and requires results bitwise
equal to fa_bwd's: the same kernels run, only the scratch differs.  The host
test checks that an over-size problem is refused before any CUDA call.
"""
import pytest
import torch

import workloads as W


@pytest.fixture(scope="module")
def fa():
    from attention_forward_08_gb300 import _build
    _build.build()
    import attention_forward_08_gb300 as fa
    fa.load_library()
    return fa


def test_noalloc_rejects_oversize(fa):
    P = 0x10000
    rc = fa.fa.fa_bwd_noalloc(P, P, P, P, P, P, P, P, P, 4, 64, 8, 16384, 16384, 128, 0.088, 1,
                              fa.FA_DTYPE_BF16, None)
    assert rc == fa.fa.FA_ERR_UNSUPPORTED
    assert "built-in scratch" in fa.fa_last_error()


def _noalloc(fa, B, H_q, qL, dq=0x10000):
    P = 0x10000
    return fa.fa.fa_bwd_noalloc(P, P, P, P, P, P, dq, P, P, B, H_q, 1, qL, 128, 128, 0.088, 1,
                                fa.FA_DTYPE_BF16, None)


def test_noalloc_limit_edge(fa):
    """Exactly 2^21 query rows fit the built-in scratch: the call passes the size guard and reaches the
    ordinary argument checks (a NULL dq is then the error); one row more is refused."""
    rc = _noalloc(fa, 1, 2, 1 << 20, dq=None)
    assert rc == fa.fa.FA_ERR_INVALID_ARGUMENT
    assert "built-in scratch" not in fa.fa_last_error() and "non-NULL" in fa.fa_last_error()
    assert _noalloc(fa, 1, 1, (1 << 21) + 1) == fa.fa.FA_ERR_UNSUPPORTED
    assert "built-in scratch" in fa.fa_last_error()
    assert _noalloc(fa, 3, 1, 699051) == fa.fa.FA_ERR_UNSUPPORTED        # 3 * 699051 = 2^21 + 1


def test_noalloc_row_count_does_not_wrap(fa):
    """B * H_q * qL = 2^63 would wrap a 64-bit product negative; the guard compares one factor at a time."""
    assert _noalloc(fa, 1 << 21, 1 << 21, 1 << 21) == fa.fa.FA_ERR_UNSUPPORTED
    assert _noalloc(fa, 2**31 - 1, 2**31 - 1, 2**31 - 1) == fa.fa.FA_ERR_UNSUPPORTED


def _problem(w):
    q, k, v = W.make_qkv(w)
    do = W.make_dout(w)
    dev = "cuda:0"
    return [t.to(dev) for t in (q, k, v, do)]


@pytest.mark.gpu
def test_noalloc_matches_workspace_entry_point(fa):
    import attention_forward_08_gb300 as pkg
    cases = [W.small_case("noalloc_a", 1, 4, 2, 384, 384, 128, "bf16", causal=True, seed=51),
             W.small_case("noalloc_b", 2, 2, 1, 200, 330, 64, "bf16", seed=52)]
    runs = cases + [cases[0]]
    for w in runs:
        q, k, v, do = _problem(w)
        o, lse = pkg.attention(q, k, v, scale=w.sm_scale, causal=w.causal)
        ref = pkg.attention_bwd(q, k, v, o, do, lse, scale=w.sm_scale, causal=w.causal)
        got = [torch.empty_like(t) for t in (q, k, v)]
        stream = torch.cuda.current_stream().cuda_stream
        rc = fa.fa.fa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                                  lse.data_ptr(), got[0].data_ptr(), got[1].data_ptr(), got[2].data_ptr(),
                                  w.B, w.H_q, w.H_kv, w.qL, w.kL, w.D, w.sm_scale, int(w.causal),
                                  fa.FA_DTYPE_BF16, stream)
        assert rc == 0, fa.fa_last_error()
        assert fa.fa_sync_status(None) == 0, fa.fa_last_error()
        for name, a, b in zip(("dq", "dk", "dv"), got, ref):
            assert torch.equal(a, b), f"{w.name}: {name} differs from fa_bwd's"
