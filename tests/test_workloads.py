"""The seeded input generators (CPU): reproducible, shaped and distributed as stated."""
import math

import torch

import workloads as W


def test_seeded_and_reproducible():
    w = W.small_case("t", 1, 2, 1, 33, 47, 64, "bf16", mask_kind=W.MASK_ADDITIVE, seed=3)
    a = W.make_inputs(w)
    b = W.make_inputs(w)
    for x, y in zip(a, b):
        assert torch.equal(x, y)
    q, k, v, m = a
    assert q.shape == (1, 2, 33, 64) and k.shape == (1, 1, 47, 64) and v.shape == k.shape
    assert q.dtype == torch.bfloat16 and m.dtype == torch.bfloat16


def test_qkv_are_standard_normal():
    w = W.small_case("t", 1, 4, 4, 512, 512, 128, "f32", seed=1)
    q, k, v = W.make_qkv(w)
    for t in (q, k, v):
        assert abs(t.mean().item()) < 0.02 and abs(t.std().item() - 1.0) < 0.02


def test_additive_mask_recipe():
    w = W.small_case("t", 1, 2, 2, 300, 300, 64, "bf16", mask_kind=W.MASK_ADDITIVE, seed=5)
    m = W.make_mask(w)
    frac = torch.isinf(m).float().mean().item()
    assert 0.08 < frac < 0.12
    assert torch.isfinite(m.diagonal(dim1=-2, dim2=-1)).all()
    assert (torch.isinf(m) <= (m < 0)).all()   # only -inf, never +inf


def test_bool_mask_recipe():
    w = W.small_case("t", 1, 2, 2, 300, 300, 64, "bf16", mask_kind=W.MASK_BOOL, seed=5)
    m = W.make_mask(w)
    assert m.dtype == torch.uint8
    keep = m.float().mean().item()
    assert 0.88 < keep < 0.92
    assert (m.diagonal(dim1=-2, dim2=-1) == 1).all()
    assert (m.sum(-1) > 0).all()


def test_named_workloads_match_their_definitions():
    ws = W.WORKLOADS
    c3 = ws[W.BENCH_WORKLOAD]
    assert (c3.B, c3.H_q, c3.H_kv, c3.qL, c3.kL, c3.D, c3.dtype, c3.causal) == (2, 32, 8, 4096, 4096, 128,
                                                                                 "bf16", True)
    assert c3.sm_scale == 1 / math.sqrt(128)
    assert abs(c3.flops() - 274.877906944e9) < 1e3
    dit = ws["fp32_dit_h24_l4608_d128_tokenmajor"]
    assert dit.layout == "dit" and dit.dtype == "f32" and not dit.causal
    assert ws["bf16_additive_mask_h8_l2000_d256"].mask_kind == W.MASK_ADDITIVE
    assert ws["bf16_bool_mask_h8_l2000_d256"].mask_kind == W.MASK_BOOL
    assert ws["fp32_b1_h2_l128_d64"].sm_scale == 0.125
