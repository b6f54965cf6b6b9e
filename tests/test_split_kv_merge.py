"""Split-KV's merge rule, checked on the oracle (CPU).

Attention over all keys equals the merge of attention over disjoint key
ranges: O = sum_s w_s O_s / sum_s w_s with w_s = exp(L_s - max_s L_s) and
L = max_s L_s + log sum_s w_s, where O_s and L_s are the normalised output
and logsumexp over range s (FlashAttention-2, Section 3.1: the online softmax
rescales partial results by exactly these factors).  This is the rule the
library's split-KV combine pass applies to its per-range partials.  A causal
row that sees no key of a range has L_s = -inf there and weight 0; a row that
sees no key at all keeps O = 0, L = -inf.
"""
import numpy as np
import pytest

import oracle


def _merge(parts):
    L = np.stack([l for _, l in parts])
    O = np.stack([o for o, _ in parts])
    m = np.max(L, axis=0)
    seen = np.isfinite(m)
    w = np.where(seen, np.exp(L - np.where(seen, m, 0.0)), 0.0)
    sw = w.sum(axis=0)
    o = np.where(seen[..., None], (w[..., None] * O).sum(axis=0) / np.where(seen, sw, 1.0)[..., None], 0.0)
    l = np.where(seen, m + np.log(np.where(seen, sw, 1.0)), -np.inf)
    return o, l


@pytest.mark.parametrize("causal,q_offset", [(False, 0), (True, 0), (True, -40)], ids=["full", "causal", "causal_offset"])
@pytest.mark.parametrize("cuts", [(0, 300), (0, 128, 256, 300), (0, 1, 97, 250, 300)], ids=["one", "blocks", "ragged"])
def test_split_kv_merge_equals_full_attention(causal, q_offset, cuts):
    rng = np.random.default_rng(11)
    B, Hq, Hkv, qL, kL, D = 1, 4, 2, 37, 300, 16
    q = rng.standard_normal((B, Hq, qL, D)) * 2.0
    k = rng.standard_normal((B, Hkv, kL, D))
    v = rng.standard_normal((B, Hkv, kL, D))
    scale = D ** -0.5
    o_all, l_all = oracle.attention(q, k, v, scale, causal=causal, q_offset=q_offset)
    # Range [a, b): its keys j' = j - a, so row i sees key j' when a + j' <= i + q_offset.
    parts = [oracle.attention(q, k[:, :, a:b], v[:, :, a:b], scale, causal=causal, q_offset=q_offset - a)
             for a, b in zip(cuts[:-1], cuts[1:])]
    o, l = _merge(parts)
    assert np.array_equal(np.isfinite(l), np.isfinite(l_all))
    np.testing.assert_allclose(o, o_all, rtol=0, atol=1e-12)
    fin = np.isfinite(l_all)
    np.testing.assert_allclose(l[fin], l_all[fin], rtol=0, atol=1e-12)
    if causal and q_offset < 0:
        assert not np.all(fin)  # rows before the first visible key: O = 0, L = -inf on both sides
        assert np.all(o[~fin] == 0.0)


def test_split_kv_merge_catches_a_wrong_weight():
    """The pin fails when the merge drops the max shift from one range's weight
    (a plausible slip): the check above is not vacuous."""
    rng = np.random.default_rng(12)
    q = rng.standard_normal((1, 1, 5, 8)) * 3.0
    k = rng.standard_normal((1, 1, 40, 8))
    v = rng.standard_normal((1, 1, 40, 8))
    o_all, _ = oracle.attention(q, k, v, 0.5)
    parts = [oracle.attention(q, k[:, :, a:b], v[:, :, a:b], 0.5) for a, b in ((0, 17), (17, 40))]
    (o0, l0), (o1, l1) = parts
    w0, w1 = np.exp(l0), np.exp(l1 - np.maximum(l0, l1))  # range 0 unshifted: wrong
    o_bad = (w0[..., None] * o0 + w1[..., None] * o1) / (w0 + w1)[..., None]
    assert not np.allclose(o_bad, o_all, rtol=0, atol=1e-9)


def test_workspace_bytes_without_a_device():
    """Split-KV depends on the device's SM count: with no device,
    fa_fwd_workspace_bytes asks for no scratch for a 16-bit call (and sets no
    error)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present: the split plan may apply")
    from attention_forward_08_gb300 import _build
    _build.build()
    import attention_forward_08_gb300 as fa
    fa.load_library()
    from test_abi import _fwd_args
    a = _fwd_args(fa, fa.FA_DTYPE_BF16, 1, 8, 8, 256, 65536, 128)  # few long query tiles
    assert fa.fa_fwd_workspace_bytes(a) == 0
    assert fa.fa_last_error() == ""
