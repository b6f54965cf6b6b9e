"""GPU parity: the CUDA library against the fp64 oracle on the same seeded inputs.

Reduced sizes are compared element by element (several Q and KV tiles,
ragged tails, every head dim, dtype, mask kind, causal, GQA, the
token-major output, sliding windows, softcaps and query offsets); the
full-size workloads are compared on sampled rows computed one by one by the
oracle, in the launch configuration the benchmark times.  Tolerances (inputs
N(0,1)): bf16 max|dO| <= 2e-2 and max|dL| <= 1e-2; fp32 via TF32 max|dO| <=
2e-3 and max|dL| <= 1e-3; fp16 a quarter of the bf16 bounds.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from gpu_helpers import oracle_features, compare, fp32_scale, gpu_run, oracle_inputs, sample_rows

pytestmark = pytest.mark.gpu

W = workloads
S = W.small_case

SMALL = [
    S("bf16_d128_plain", 1, 2, 2, 384, 384, 128, "bf16"),
    S("bf16_d128_causal_gqa", 1, 4, 2, 512, 512, 128, "bf16", causal=True),
    S("bf16_d128_causal_ragged", 2, 2, 1, 333, 333, 128, "bf16", causal=True),
    # 16-bit O token-major ([qL, H * D]): the two-tile plans store O through a tensor map with
    # the caller's strides (head stride D, row stride H * D), rows past qL clipped
    S("bf16_d128_tokenmajor_causal_ragged", 1, 3, 3, 300, 300, 128, "bf16", causal=True, layout="dit"),
    S("f16_d64_tokenmajor_gqa", 1, 4, 2, 260, 260, 64, "f16", layout="dit"),
    S("bf16_d64_causal_ragged", 2, 2, 2, 300, 300, 64, "bf16", causal=True),
    S("bf16_d64_plain_long_kv", 1, 2, 2, 200, 700, 64, "bf16"),
    S("bf16_d256_additive_ragged", 1, 2, 2, 200, 200, 256, "bf16", mask_kind=W.MASK_ADDITIVE),
    S("bf16_d256_bool_ragged", 1, 2, 2, 200, 200, 256, "bf16", mask_kind=W.MASK_BOOL),
    S("bf16_d256_causal", 1, 2, 1, 260, 260, 256, "bf16", causal=True),
    S("bf16_d128_bool_causal", 1, 2, 2, 300, 300, 128, "bf16", causal=True, mask_kind=W.MASK_BOOL),
    S("bf16_d64_additive_causal", 1, 2, 2, 257, 257, 64, "bf16", causal=True, mask_kind=W.MASK_ADDITIVE),
    S("f32_d64_plain", 1, 2, 2, 128, 128, 64, "f32"),
    S("f32_d64_causal_ragged", 1, 3, 3, 290, 290, 64, "f32", causal=True),
    S("f32_d128_tokenmajor", 1, 3, 3, 300, 300, 128, "f32", layout="dit"),
    S("f32_d128_causal_gqa", 1, 4, 1, 260, 260, 128, "f32", causal=True),
    S("f32_d256_plain", 1, 2, 2, 150, 150, 256, "f32"),
    S("f32_d256_additive", 1, 2, 2, 100, 170, 256, "f32", mask_kind=W.MASK_ADDITIVE),
    S("bf16_d128_q_longer_than_k_causal", 1, 2, 2, 400, 150, 128, "bf16", causal=True),
    S("bf16_d128_tiny", 1, 1, 1, 1, 1, 128, "bf16"),
    S("bf16_d64_tiny_ragged", 1, 1, 1, 5, 3, 64, "bf16", causal=True),
    S("f32_d64_tiny", 1, 1, 1, 3, 7, 64, "f32"),
    S("bf16_d128_gqa8", 1, 8, 1, 256, 256, 128, "bf16", causal=True),
    S("f16_d128_causal_gqa", 1, 4, 2, 512, 512, 128, "f16", causal=True),
    S("f16_d64_additive_causal_ragged", 1, 2, 2, 257, 257, 64, "f16", causal=True, mask_kind=W.MASK_ADDITIVE),
    S("f16_d256_bool_ragged", 1, 2, 2, 200, 200, 256, "f16", mask_kind=W.MASK_BOOL),
    S("f16_d256_additive_tma_mask", 1, 2, 2, 256, 256, 256, "f16", mask_kind=W.MASK_ADDITIVE),
]


def _run_small(w, scale=None, mask=None, qkv=None, tol_mult=1.0, tol_mult_l=None, tf32_relative=False,
               workspace=None):
    if qkv is None:
        q, k, v, m = W.make_inputs(w)
    else:
        (q, k, v), m = qkv, mask
    o_g, l_g, _ = gpu_run(w, q, k, v, m, scale=scale, workspace=workspace)
    qo, ko, vo, mo = oracle_inputs(q, k, v, m)
    o_r, l_r = oracle.attention(qo, ko, vo, fp32_scale(w, scale), causal=w.causal, mask=mo,
                                mask_kind=w.mask_kind if m is not None else 0, **oracle_features(w))
    if tf32_relative and w.dtype == "f32":
        # TF32 score errors are relative to the scores; L tracks the largest score.
        big = float(np.max(np.abs(l_r[np.isfinite(l_r)]))) / 8.0
        tol_mult = tol_mult_l = max(1.0, big)
    return compare(w, o_g, l_g, o_r, l_r, what=w.name, tol_mult=tol_mult, tol_mult_l=tol_mult_l)


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_small_elementwise(w):
    _run_small(w)


# bf16 / fp16 at D <= 128 run with two Q tiles per CTA, or one when two-tile
# units cannot fill the GPU (every small case above): force each plan.
TWO_PLANS = [w for w in SMALL if w.dtype in ("bf16", "f16") and w.D <= 128]


@pytest.mark.parametrize("q_tiles", [1, 2])
@pytest.mark.parametrize("w", TWO_PLANS, ids=lambda w: w.name)
def test_small_both_tile_plans(w, q_tiles):
    import attention_forward_08_gb300 as fa
    fa.fa_set_q_tiles(q_tiles)
    try:
        _run_small(w)
    finally:
        fa.fa_set_q_tiles(0)


# fp32 I/O has two plans once kL >= 1024: the tf32 pre-pass (Q, K rounded and V
# rounded and transposed in a workspace, then a TMA-only kernel) and the
# in-kernel helper warps (no workspace).  Both against the oracle: ragged kL
# (V^T rows padded to 4 keys), GQA, causal, each head dim, an additive mask.
FP32_PLANS = [
    S("f32pre_d128_ragged_kl", 1, 2, 2, 300, 1030, 128, "f32", seed=91),
    S("f32pre_d64_causal_gqa", 1, 4, 2, 1030, 1030, 64, "f32", causal=True, seed=92),
    S("f32pre_d256_additive", 1, 2, 2, 260, 1024, 256, "f32", mask_kind=W.MASK_ADDITIVE, seed=93),
    S("f32pre_d128_b2_causal_qlonger", 2, 2, 1, 1300, 1100, 128, "f32", causal=True, seed=94),
]


@pytest.mark.parametrize("workspace", [None, False], ids=["prepass", "helpers"])
@pytest.mark.parametrize("w", FP32_PLANS, ids=lambda w: w.name)
def test_fp32_both_plans(w, workspace):
    import attention_forward_08_gb300 as fa
    q, k, v, m = W.make_inputs(w)
    qd = q.cuda()
    args = fa.make_args(qd, k.cuda(), v.cuda(), torch.empty_like(qd), torch.empty((w.B, w.H_q, w.qL), device="cuda"),
                        scale=w.sm_scale, causal=w.causal)
    assert fa.fa_fwd_workspace_bytes(args) > 0  # the pre-pass plan applies to these shapes
    _run_small(w, qkv=(q, k, v), mask=m, workspace=workspace)


# Split-KV (the one-Q-tile 16-bit plans without features): each query tile's
# key blocks cut into ranges, one work unit each, the partial O and L merged
# by a second launch.  Forced counts that leave ranges empty (early causal
# tiles, kL past the causal limit) or exceed the key blocks, and the automatic
# count on decoding-like shapes (few query tiles, long kL); both head dims and
# 16-bit types, ragged qL and kL, GQA, bool and additive masks.
SPLIT_KV = [
    (S("splitkv_bf16_d128_gqa", 1, 4, 1, 130, 3000, 128, "bf16", seed=101), 5),
    (S("splitkv_f16_d64_auto", 2, 2, 2, 64, 5000, 64, "f16", seed=102), 0),
    (S("splitkv_bf16_d128_causal", 1, 2, 1, 1000, 1000, 128, "bf16", causal=True, seed=103), 3),
    (S("splitkv_bf16_d64_beyond_blocks", 1, 2, 2, 100, 300, 64, "bf16", seed=104), 64),
    (S("splitkv_f16_d128_causal_kl_longer", 1, 4, 2, 200, 2500, 128, "f16", causal=True, seed=105), 4),
    (S("splitkv_bf16_d128_bool_mask", 1, 2, 2, 130, 2000, 128, "bf16", mask_kind=W.MASK_BOOL, seed=106), 0),
    (S("splitkv_f16_d64_additive_ragged", 1, 2, 1, 300, 1801, 64, "f16", mask_kind=W.MASK_ADDITIVE, seed=107), 5),
]


@pytest.mark.parametrize("w,splits", SPLIT_KV, ids=[w.name for w, _ in SPLIT_KV])
def test_split_kv(w, splits):
    import attention_forward_08_gb300 as fa
    fa.fa_set_kv_splits(splits)
    try:
        q, k, v, m = W.make_inputs(w)
        qd = q.cuda()
        md = None if m is None else m.cuda()
        args = fa.make_args(qd, k.cuda(), v.cuda(), torch.empty_like(qd),
                            torch.empty((w.B, w.H_q, w.qL), device="cuda"), scale=w.sm_scale, causal=w.causal,
                            mask=md, mask_kind=None if md is None else w.mask_kind)
        assert fa.fa_fwd_workspace_bytes(args) > 0  # the split plan applies
        _run_small(w, qkv=(q, k, v), mask=m)
    finally:
        fa.fa_set_kv_splits(0)


# Sliding window, softcap and query offset on every kernel plan (two Q tiles,
# one Q tile, TF32, masks).  Softcaps of 1.5-4 against N(0,1) inputs with a
# raised scale make the cap bend most scores.
FEATURES = [
    S("swa_bf16_d128", 1, 4, 2, 700, 700, 128, "bf16", causal=True, window=200, seed=61),
    S("swa_bf16_d64_offset", 2, 2, 1, 300, 350, 64, "bf16", causal=True, window=130, q_offset=50, seed=62),
    S("swa_bf16_d256", 1, 2, 2, 600, 600, 256, "bf16", causal=True, window=300, seed=63),
    S("swa_f32_d128", 1, 2, 2, 500, 500, 128, "f32", causal=True, window=256, seed=64),
    S("swa_noncausal_f32_d64", 1, 2, 2, 300, 420, 64, "f32", window=100, seed=65),
    S("swa_f16_d128_window1", 1, 2, 2, 260, 260, 128, "f16", causal=True, window=1, seed=66),
    S("softcap_bf16_d128", 1, 4, 2, 384, 384, 128, "bf16", causal=True, softcap=3.0, scale=0.3, seed=67),
    S("softcap_bf16_d256_additive", 1, 2, 2, 256, 256, 256, "bf16", mask_kind=W.MASK_ADDITIVE, softcap=2.0,
      scale=0.2, seed=68),
    S("softcap_f32_d128", 1, 2, 2, 300, 300, 128, "f32", softcap=4.0, seed=69),
    S("softcap_f32_d64_causal", 1, 3, 3, 290, 290, 64, "f32", causal=True, softcap=1.5, scale=0.4, seed=70),
    S("prefill_f16_d128", 1, 2, 2, 200, 900, 128, "f16", causal=True, q_offset=700, seed=71),
    S("neg_offset_bf16_d128", 1, 2, 2, 300, 300, 128, "bf16", causal=True, q_offset=-50, seed=72),
    S("all_bf16_d64_bool", 1, 2, 1, 257, 400, 64, "bf16", causal=True, mask_kind=W.MASK_BOOL, window=150,
      softcap=2.5, q_offset=143, seed=73),
    S("swa_offset_bf16_d256_gqa", 1, 4, 1, 333, 500, 256, "bf16", causal=True, window=170, q_offset=167, seed=74),
]


# Dropout (kL a multiple of 4): keep decisions must agree exactly with the
# oracle's generator, so O compares at the usual bounds; p = 1 gives O = 0.
DROPOUT = [
    S("drop_bf16_d128_causal_gqa", 1, 4, 2, 384, 384, 128, "bf16", causal=True, dropout_p=0.1, dropout_seed=7,
      dropout_offset=3, seed=81),
    S("drop_bf16_d64_plain", 2, 2, 2, 256, 320, 64, "bf16", dropout_p=0.5, dropout_seed=2 ** 40 + 11, seed=82),
    S("drop_bf16_d256_additive", 1, 2, 2, 256, 256, 256, "bf16", mask_kind=W.MASK_ADDITIVE, dropout_p=0.25,
      dropout_seed=5, dropout_offset=2 ** 34, seed=83),
    S("drop_f32_d128", 1, 2, 2, 300, 300, 128, "f32", dropout_p=0.2, dropout_seed=9, seed=84),
    S("drop_f16_d64_window_causal", 1, 2, 1, 260, 260, 64, "f16", causal=True, window=100, dropout_p=0.3,
      dropout_seed=13, dropout_offset=77, seed=85),
    S("drop_all_bf16_d128", 1, 2, 2, 200, 200, 128, "bf16", causal=True, dropout_p=1.0, dropout_seed=1, seed=86),
    S("drop_f16_d256_bool", 1, 2, 2, 200, 200, 256, "f16", mask_kind=W.MASK_BOOL, dropout_p=0.4, dropout_seed=21,
      seed=87),
    S("drop_bf16_d128_softcap_offset", 1, 4, 2, 192, 320, 128, "bf16", causal=True, q_offset=128, softcap=15.0,
      dropout_p=0.15, dropout_seed=3, seed=88),
]


@pytest.mark.parametrize("w", DROPOUT, ids=lambda w: w.name)
def test_dropout(w):
    _run_small(w)


@pytest.mark.parametrize("w", FEATURES, ids=lambda w: w.name)
def test_window_softcap_offset(w):
    """fp32 cases with a raised scale take the TF32 rule of test_unusual_scales: raw scores of
    standard deviation |scale|*sqrt(D) carry proportionally larger product errors into the cap."""
    sd = abs(w.sm_scale) * w.D ** 0.5
    if w.dtype == "f32" and sd > 1.0:
        _run_small(w, tol_mult=sd, tol_mult_l=4.0 * sd)
    else:
        _run_small(w, tf32_relative=True)


@pytest.mark.parametrize("scale", [0.0, -0.3, 2.5])
@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("bf16", 256), ("f32", 64), ("f32", 128)])
def test_unusual_scales(scale, dtype, D):
    """scale = 0 (uniform weights), a negative scale, and a large one (the running max moves often).

    The stated fp32 tolerances hold for the standard scale 1/sqrt(D).  With TF32 products the
    score error is relative to the score (Q and K carry 10 mantissa bits), and scores have
    standard deviation |scale|*sqrt(D): the O bound is scaled by max(1, |scale|*sqrt(D)) and the
    L bound (L follows the largest scores, about 4 standard deviations) by max(1, 4*|scale|*sqrt(D)).
    bf16 products are exact in fp32 and keep the stated bounds.
    """
    sd = abs(scale) * D ** 0.5
    mult, mult_l = (max(1.0, sd), max(1.0, 4.0 * sd)) if dtype == "f32" else (1.0, 1.0)
    _run_small(S(f"{dtype}_d{D}_scale", 1, 2, 2, 200, 300, D, dtype, causal=True), scale=scale, tol_mult=mult,
               tol_mult_l=mult_l)


@pytest.mark.parametrize("scale", [1e-39, 1e-6])
@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("f16", 64), ("f16", 256), ("bf16", 256)])
def test_extreme_scale_additive_mask(scale, dtype, D):
    """An additive mask of 0 and +-1e4 entries with a subnormal scale (1e-39: 1 / scale is not a
    finite fp32) and a tiny normal one (1e-6: mask / scale = 1e10).  The mask decides the weights:
    each row averages V over its keys of the largest mask value.  Mask values are not divided by
    the scale where that could overflow, so no 0 * inf or inf - inf reaches the softmax."""
    w = S(f"{dtype}_d{D}_tiny_scale_mask", 1, 2, 2, 200, 260, D, dtype, mask_kind=W.MASK_ADDITIVE, seed=98)
    q, k, v = W.make_qkv(w)
    g = torch.Generator().manual_seed(99)
    u = torch.rand(1, 2, 200, 260, generator=g)
    m = torch.zeros(1, 2, 200, 260)
    m[u < 0.08] = 1e4
    m[(u >= 0.08) & (u < 0.2)] = -1e4
    _run_small(w, scale=scale, mask=m.to(w.torch_dtype), qkv=(q, k, v))


@pytest.mark.parametrize("dtype,D", [("bf16", 64), ("bf16", 128), ("bf16", 256), ("f32", 128)])
def test_rising_scores_rescale_every_block(dtype, D):
    """Keys drift along q so each KV block's max exceeds the last by ~12 (base 2): the running
    max moves, O is rescaled, and P is recomputed in every block.  Scores grow to ~100; for fp32
    every input sits on a 1/8 grid (exact in TF32), so the score products are exact and the
    standard bounds apply."""
    w = S(f"{dtype}_d{D}_ramp", 1, 2, 2, 256, 640, D, dtype)
    q, k, v = W.make_qkv(w)
    qf, kf, vf = q.float(), k.float(), v.float()
    if dtype == "f32":
        qf, kf, vf = [(t * 8).round().clamp(-64, 64) / 8 for t in (qf, kf, vf)]
    direction = qf.mean(dim=2, keepdim=True)                       # [1,2,1,D]
    direction = direction / direction.norm(dim=-1, keepdim=True)
    qn = (qf * direction).sum(-1).mean().item()                     # typical q . direction
    step = 12.0 / (w.sm_scale * max(qn, 1.0) * 1.4426950408889634)  # score rise per 128 keys
    ramp = (torch.arange(640, dtype=torch.float32) / 128.0 * step).view(1, 1, 640, 1)
    k2 = kf + ramp * direction
    if dtype == "f32":
        k2 = (k2 * 8).round() / 8
    _run_small(w, mask=None, qkv=(qf.to(q.dtype), k2.to(q.dtype), vf.to(q.dtype)))


def test_fully_masked_rows():
    """Rows whose bool mask keeps nothing: O = 0 and L = -inf; other rows unaffected."""
    w = S("bf16_d128_bool_empty_rows", 1, 2, 2, 256, 256, 128, "bf16", mask_kind=W.MASK_BOOL)
    q, k, v = W.make_qkv(w)
    g = torch.Generator().manual_seed(5)
    m = (torch.rand(1, 2, 256, 256, generator=g) < 0.5).to(torch.uint8)
    m[0, 0, 7] = 0
    m[0, 1, 130:140] = 0
    _run_small(w, mask=m, qkv=(q, k, v))


def test_broadcast_mask_strides():
    """An additive mask broadcast over batch and heads through zero strides."""
    w = S("bf16_d64_bcast_mask", 2, 2, 2, 200, 200, 64, "bf16", mask_kind=W.MASK_ADDITIVE)
    q, k, v = W.make_qkv(w)
    g = torch.Generator().manual_seed(9)
    base = torch.randn(1, 1, 200, 200, generator=g).to(torch.bfloat16)
    import attention_forward_08_gb300 as fa
    dev = "cuda:0"
    o, lse = fa.attention(q.to(dev), k.to(dev), v.to(dev), scale=w.sm_scale,
                          mask=base.to(dev).expand(2, 2, 200, 200), mask_kind=2)
    assert fa.fa_sync_status(None) == 0
    qo, ko, vo, _ = oracle_inputs(q, k, v, None)
    o_r, l_r = oracle.attention(qo, ko, vo, fp32_scale(w), mask=np.broadcast_to(base.double().numpy(),
                                                                                 (2, 2, 200, 200)), mask_kind=2)
    compare(w, o.double().cpu().numpy(), lse.double().cpu().numpy(), o_r, l_r, what=w.name)


def test_repeat_is_deterministic():
    """Two launches on identical inputs give bit-identical O and L."""
    w = S("bf16_d128_repeat", 1, 4, 2, 300, 300, 128, "bf16", causal=True)
    q, k, v, m = W.make_inputs(w)
    o1, l1, _ = gpu_run(w, q, k, v, m)
    o2, l2, _ = gpu_run(w, q, k, v, m)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


# Full-size workloads whose fp64 oracle finishes in seconds (at most ~2e10 multiply-adds) are
# compared on every row; the larger ones on sampled rows.
def _oracle_cheap(w):
    return 2.0 * w.B * w.H_q * w.qL * w.kL * w.D <= 2e10


@pytest.mark.parametrize("name", list(W.WORKLOADS), ids=list(W.WORKLOADS))
def test_full_workload_sampled_rows(name):
    """Full-size workloads: every output finite where it should be, and every row (cheap workloads:
    C1, C2 and both D = 256 masked workloads, whose last Q tile holds 80 rows) or sampled rows vs
    the oracle."""
    w = W.WORKLOADS[name]
    q, k, v, m = W.make_inputs(w)
    o_g, l_g, _ = gpu_run(w, q, k, v, m)
    # properties over every row
    assert np.all(np.isfinite(o_g)), "non-finite O"
    assert np.all(np.isfinite(l_g)), "every row of these workloads has an allowed key"
    if _oracle_cheap(w):
        qo, ko, vo, mo = oracle_inputs(q, k, v, m)
        o_r, l_r = oracle.attention(qo, ko, vo, fp32_scale(w), causal=w.causal, mask=mo,
                                    mask_kind=w.mask_kind, **oracle_features(w))
        compare(w, o_g, l_g, o_r, l_r, what=name + " (every row)")
        return
    rows = sample_rows(w, n_per_head=3 if w.qL * w.kL > 4e6 else 8)
    qo, ko, vo, mo = oracle_inputs(q, k, v, m)
    o_r, l_r = oracle.attention(qo, ko, vo, fp32_scale(w), causal=w.causal, mask=mo,
                                mask_kind=w.mask_kind, rows=rows, **oracle_features(w))
    D = w.D
    compare(w, o_g.reshape(-1, D)[rows], l_g.reshape(-1)[rows], o_r, l_r, what=name)


# Long sequences: 256 key blocks per unit, row and position arithmetic past
# 2^31 (the dropout case's positions ((b H_q + h) qL + i) kL + j reach 2^32,
# on top of a 2^33 counter offset), and the fp32 pre-pass at size.
LONG = [
    S("long_bf16_causal_gqa_l32768_d128", 1, 4, 2, 32768, 32768, 128, "bf16", causal=True, seed=95),
    S("long_bf16_dropout_l32768_d64", 1, 4, 1, 32768, 32768, 64, "bf16", causal=True, dropout_p=0.2,
      dropout_seed=77, dropout_offset=2 ** 33, seed=96),
    S("long_f32_prepass_l16384_d128", 1, 2, 2, 16384, 16384, 128, "f32", seed=97),
]


@pytest.mark.parametrize("w", LONG, ids=lambda w: w.name)
def test_long_sequence_sampled_rows(w):
    q, k, v, m = W.make_inputs(w)
    o_g, l_g, _ = gpu_run(w, q, k, v, m)
    assert np.all(np.isfinite(o_g)) and np.all(np.isfinite(l_g))
    rows = sample_rows(w, n_per_head=4)
    qo, ko, vo, mo = oracle_inputs(q, k, v, m)
    o_r, l_r = oracle.attention(qo, ko, vo, fp32_scale(w), causal=w.causal, mask=mo, mask_kind=w.mask_kind,
                                rows=rows, **oracle_features(w))
    compare(w, o_g.reshape(-1, w.D)[rows], l_g.reshape(-1)[rows], o_r, l_r, what=w.name)


PERSISTENT = [
    S("bf16_d128_causal_gqa_units", 2, 4, 2, 520, 520, 128, "bf16", causal=True),
    S("bf16_d64_plain_units", 1, 3, 3, 300, 500, 64, "bf16"),
    S("bf16_d256_bool_units", 1, 3, 3, 300, 300, 256, "bf16", mask_kind=W.MASK_BOOL),
    S("f32_d64_causal_units", 1, 3, 1, 300, 300, 64, "f32", causal=True),
    S("f32_d128_tokenmajor_units", 1, 3, 3, 260, 260, 128, "f32", layout="dit"),
    S("f32_d256_additive_units", 1, 2, 2, 170, 200, 256, "f32", mask_kind=W.MASK_ADDITIVE),
    # two heads of one K/V head per unit (sliding window / dropout with an even GQA group)
    S("swa_bf16_d64_gqa4_head_pairs_units", 2, 8, 2, 520, 520, 64, "bf16", causal=True, window=150, seed=77),
    S("drop_f16_d128_gqa2_head_pairs_units", 1, 4, 2, 300, 300, 128, "f16", causal=True, dropout_p=0.2,
      dropout_seed=4, seed=78),
]


@pytest.mark.parametrize("max_ctas", [1, 3])
@pytest.mark.parametrize("w", PERSISTENT, ids=lambda w: w.name)
@pytest.mark.parametrize("q_tiles", [0, 1])
def test_persistent_many_units_per_cta(w, max_ctas, q_tiles):
    """The kernel is persistent: with the CTA count capped, each CTA walks many work units
    (down to one CTA doing all of them), carrying its barrier phases from unit to unit; with
    the one-Q-tile plan forced as well where it exists."""
    import attention_forward_08_gb300 as fa
    fa.fa_set_max_ctas(max_ctas)
    fa.fa_set_q_tiles(q_tiles)
    try:
        _run_small(w)
    finally:
        fa.fa_set_max_ctas(0)
        fa.fa_set_q_tiles(0)


# One Q tile per CTA (bf16 / fp16 at D = 256, and at D <= 128 for small grids) runs two softmax
# warpgroups, each on 64 of a block's 128 keys: every D = 256 case with the grid capped (one and
# three CTAs walking every unit), plus a causal GQA case with more units than SMs.
D256 = [w for w in SMALL if w.D == 256 and w.dtype != "f32"] + [
    S("bf16_d256_causal_gqa_units", 2, 4, 2, 700, 700, 256, "bf16", causal=True, seed=111),
    S("f16_d256_additive_q_longer", 1, 2, 1, 520, 300, 256, "f16", mask_kind=W.MASK_ADDITIVE, seed=112),
]


@pytest.mark.parametrize("max_ctas", [0, 1, 3])
@pytest.mark.parametrize("w", D256, ids=lambda w: w.name)
def test_d256_split_rows(w, max_ctas):
    import attention_forward_08_gb300 as fa
    fa.fa_set_max_ctas(max_ctas)
    try:
        _run_small(w)
    finally:
        fa.fa_set_max_ctas(0)
