"""Backward parity on the GPU: dQ, dK, dV from the C ABI against the fp64
gradient oracle, element by element.

The GPU backward consumes what the GPU forward produced (O in bf16, L in
fp32), as a training step would.  Tolerance (bf16 I/O): every gradient
element within 2e-2 of the oracle's, measured relative to the largest
|oracle| entry of that tensor, and cosine similarity >= 0.999.  The bound
follows the arithmetic: P and dS are rounded to bf16 (relative error <= 2^-9
each) before the dV, dK and dQ products, the inputs and the stored results
are bf16, and accumulation is fp32; the resulting error is a few 2^-9 of the
tensor's scale, well inside 2e-2.  fp16 I/O (P and dS rounded to fp16,
relative error <= 2^-11) gets a quarter of that bound, 5e-3, as the forward's
fp16 tolerance does; so does fp32 I/O, whose products run on the TF32 tensor cores (inputs, P and dS
rounded to tf32, relative error <= 2^-11 each; accumulation and outputs fp32).  With dropout the backward regenerates the forward's
keep decisions from the same seed and offset; the oracle takes its
multipliers from the forward oracle's generator, so a backward that drew
other bits than the forward fails the comparison.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from gpu_helpers import fp32_scale

pytestmark = pytest.mark.gpu

S = W.small_case
CASES = [
    S("bwd_d128_plain", 1, 2, 2, 256, 256, 128, "bf16", seed=31),
    S("bwd_d128_causal_gqa", 1, 4, 2, 384, 384, 128, "bf16", causal=True, seed=32),
    S("bwd_d64_causal_ragged", 2, 2, 1, 200, 200, 64, "bf16", causal=True, seed=33),
    S("bwd_d128_causal_q_longer", 1, 2, 2, 300, 170, 128, "bf16", causal=True, seed=34),
    S("bwd_d128_causal_k_longer", 1, 2, 1, 150, 420, 128, "bf16", causal=True, seed=35),
    S("bwd_d64_plain_long_kv", 1, 2, 2, 130, 600, 64, "bf16", seed=36),
    S("bwd_d64_tiny", 1, 1, 1, 5, 3, 64, "bf16", causal=True, seed=37),
    S("bwd_d128_gqa8", 1, 8, 1, 256, 256, 128, "bf16", causal=True, seed=38),
    S("bwd_f16_d128_causal_gqa", 1, 4, 2, 384, 384, 128, "f16", causal=True, seed=41),
    S("bwd_f16_d64_ragged", 2, 2, 1, 200, 200, 64, "f16", causal=True, seed=42),
    S("bwd_f16_d128_plain_long_kv", 1, 2, 2, 130, 600, 128, "f16", seed=43),
    # head dim 256 (causal or full attention): two CTAs per 128-key tile, 64-query steps; 64-key dQ blocks
    S("bwd_d256_plain", 1, 2, 2, 256, 256, 256, "bf16", seed=44),
    S("bwd_d256_causal_gqa", 1, 4, 2, 384, 384, 256, "bf16", causal=True, seed=45),
    S("bwd_d256_causal_ragged", 2, 2, 1, 200, 200, 256, "bf16", causal=True, seed=46),
    S("bwd_d256_causal_q_longer", 1, 2, 2, 300, 170, 256, "bf16", causal=True, seed=47),
    S("bwd_d256_causal_k_longer", 1, 2, 1, 150, 420, 256, "bf16", causal=True, seed=48),
    S("bwd_d256_plain_long_kv", 1, 2, 2, 130, 600, 256, "bf16", seed=49),
    S("bwd_d256_tiny", 1, 1, 1, 5, 3, 256, "bf16", causal=True, seed=50),
    S("bwd_f16_d256_causal_gqa", 1, 4, 2, 384, 384, 256, "f16", causal=True, seed=58),
    S("bwd_f16_d256_plain_ragged", 1, 2, 1, 250, 333, 256, "f16", seed=59),
    # fp32 I/O on the TF32 tensor cores (fa_bwd_full): separate dV, dK and dQ kernels
    S("bwd_f32_d64_plain", 1, 2, 2, 128, 128, 64, "f32", seed=81),
    S("bwd_f32_d64_causal_ragged", 2, 2, 1, 200, 200, 64, "f32", causal=True, seed=82),
    S("bwd_f32_d128_causal_gqa", 1, 4, 2, 384, 384, 128, "f32", causal=True, seed=83),
    S("bwd_f32_d128_plain_long_kv", 1, 2, 2, 130, 600, 128, "f32", seed=84),
    S("bwd_f32_d128_causal_k_longer", 1, 2, 1, 150, 420, 128, "f32", causal=True, seed=85),
    S("bwd_f32_d128_causal_q_longer", 1, 2, 2, 300, 170, 128, "f32", causal=True, seed=86),
    S("bwd_f32_d64_tiny", 1, 1, 1, 5, 3, 64, "f32", causal=True, seed=87),
    S("bwd_f32_d64_gqa8_noncausal", 1, 8, 1, 256, 333, 64, "f32", seed=88),
    # sliding window / causal diagonal offset (fa_bwd_ex)
    S("bwd_swa_d128_causal_gqa", 1, 4, 2, 640, 640, 128, "bf16", causal=True, window=200, seed=51),
    S("bwd_offset_d64_bottom_right", 1, 2, 1, 300, 560, 64, "bf16", causal=True, q_offset=260, seed=52),
    S("bwd_swa_offset_f16_d128", 2, 2, 2, 384, 500, 128, "f16", causal=True, window=150, q_offset=116, seed=53),
    S("bwd_window_noncausal_d64", 1, 2, 2, 256, 400, 64, "bf16", window=100, seed=54),
    S("bwd_negative_offset_d128", 1, 2, 2, 300, 300, 128, "bf16", causal=True, q_offset=-150, seed=55),
    # softcap (fa_bwd_ex): scale raised so the cap bends most scores
    S("bwd_softcap_d128_causal_gqa", 1, 4, 2, 384, 384, 128, "bf16", causal=True, softcap=2.0, seed=56),
    S("bwd_softcap_window_f16_d64", 1, 2, 1, 300, 420, 64, "f16", causal=True, window=120, q_offset=120,
      softcap=3.0, seed=57),
    # dropout (fa_bwd_ex): the forward's seed and offset; kL a multiple of 4
    S("bwd_dropout_d128_causal_gqa", 1, 4, 2, 384, 384, 128, "bf16", causal=True, dropout_p=0.1,
      dropout_seed=2024, seed=61),
    S("bwd_dropout_f16_d64_ragged", 2, 2, 1, 200, 200, 64, "f16", causal=True, dropout_p=0.3,
      dropout_seed=77, dropout_offset=12345, seed=62),
    S("bwd_dropout_d64_noncausal_long_kv", 1, 2, 2, 130, 600, 64, "bf16", dropout_p=0.5, dropout_seed=5,
      seed=63),
    S("bwd_dropout_softcap_window_d128", 1, 2, 1, 300, 420, 128, "bf16", causal=True, window=120, q_offset=120,
      softcap=3.0, dropout_p=0.2, dropout_seed=9, seed=64),
    S("bwd_dropout_offset_past_2p32_d128", 1, 2, 2, 256, 256, 128, "bf16", causal=True, dropout_p=0.15,
      dropout_seed=(1 << 40) + 3, dropout_offset=(1 << 33) + 5, seed=65),
]
SOFTCAP_SCALE = 0.35  # scale * |q.k| ~ 0.35 * sqrt(D) * N(0, 1): several times the cap

REL_TOL = {"bf16": 2e-2, "f16": 5e-3, "f32": 5e-3}
COS_MIN = 0.999


def _run(w):
    import attention_forward_08_gb300 as fa
    q, k, v = W.make_qkv(w)
    do = W.make_dout(w)
    dev = "cuda:0"
    qd, kd, vd, dod = q.to(dev), k.to(dev), v.to(dev), do.to(dev)
    scale = SOFTCAP_SCALE if w.softcap else w.sm_scale
    drop = dict(dropout_p=w.dropout_p, dropout_seed=w.dropout_seed, dropout_offset=w.dropout_offset)
    o, lse = fa.attention(qd, kd, vd, scale=scale, causal=w.causal, window=w.window, q_offset=w.q_offset,
                          softcap=w.softcap, **drop)
    dq, dk, dv = fa.attention_bwd(qd, kd, vd, o, dod, lse, scale=scale, causal=w.causal, window=w.window,
                                  q_offset=w.q_offset, softcap=w.softcap, **drop)
    assert fa.fa_sync_status(None) == fa.fa.FA_OK, fa.fa_last_error()
    return (q, k, v, do), (dq, dk, dv)


def _compare(name, got, ref, rel_tol=REL_TOL["bf16"]):
    got = got.double().cpu().numpy()
    assert np.all(np.isfinite(got)), f"{name}: non-finite gradient"
    scale = max(np.abs(ref).max(), 1e-30)
    err = np.abs(got - ref).max() / scale
    a, b = got.ravel(), ref.ravel()
    cos = float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b) + 1e-300))
    print(f"{name}: max|d| / max|ref| = {err:.3e}, cos = {cos:.7f}")
    assert err <= rel_tol, f"{name}: max|d| / max|ref| = {err:.3e} > {rel_tol} (cos {cos:.6f})"
    assert cos >= COS_MIN, f"{name}: cosine {cos:.6f} < {COS_MIN}"
    return err, cos


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_bwd_elementwise(w):
    (q, k, v, do), (dq, dk, dv) = _run(w)
    rq, rk, rv = oracle.attention_bwd(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                                      do.double().numpy(),
                                      fp32_scale(w, SOFTCAP_SCALE if w.softcap else None), causal=w.causal,
                                      window=w.window, q_offset=w.q_offset, softcap=float(np.float32(w.softcap)),
                                      dropout_p=float(np.float32(w.dropout_p)), seed=w.dropout_seed,
                                      offset=w.dropout_offset)
    tol = REL_TOL[w.dtype]
    _compare(f"{w.name} dQ", dq, rq, tol)
    _compare(f"{w.name} dK", dk, rk, tol)
    _compare(f"{w.name} dV", dv, rv, tol)
    if w.causal and w.kL > w.qL and w.q_offset == 0 and w.window == 0:
        # keys no query reaches get exactly zero gradient
        assert torch.count_nonzero(dk[:, :, w.qL:]).item() == 0
        assert torch.count_nonzero(dv[:, :, w.qL:]).item() == 0


def test_bwd_deterministic():
    w = CASES[1]
    _, a = _run(w)
    _, b = _run(w)
    for x, y in zip(a, b):
        assert torch.equal(x, y), "two identical backward calls differ"


def test_bwd_gqa_sums_group_heads():
    """dK, dV of a GQA problem equal the per-head MHA gradients (K/V repeated) summed over each group."""
    import attention_forward_08_gb300 as fa
    w = S("bwd_gqa_vs_mha", 1, 4, 1, 256, 256, 128, "bf16", causal=True, seed=39)
    (q, k, v, do), (dq, dk, dv) = _run(w)
    dev = "cuda:0"
    kr, vr = k.repeat_interleave(4, dim=1).to(dev), v.repeat_interleave(4, dim=1).to(dev)
    qd, dod = q.to(dev), do.to(dev)
    o, lse = fa.attention(qd, kr, vr, scale=w.sm_scale, causal=True)
    dq2, dk2, dv2 = fa.attention_bwd(qd, kr, vr, o, dod, lse, scale=w.sm_scale, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(dq, dq2)
    for g, g2 in ((dk, dk2), (dv, dv2)):
        s = g2.float().sum(dim=1, keepdim=True)
        err = (g.float() - s).abs().max().item() / max(s.abs().max().item(), 1e-30)
        assert err < 2e-2, err


def test_bwd_dropout_all_dropped_gives_zero_gradients():
    """p = 1 drops every weight: O = 0, so D = 0 and dS = P (0 dP - 0) = 0; all three gradients are exactly 0."""
    w = S("bwd_dropout_p1", 1, 2, 1, 256, 256, 64, "bf16", causal=True, dropout_p=1.0, dropout_seed=3, seed=66)
    _, grads = _run(w)
    for g in grads:
        assert torch.count_nonzero(g).item() == 0


def test_bwd_dropout_seed_changes_gradients():
    """Another seed gives other keep decisions and so other gradients; the same seed repeats them exactly."""
    w = CASES[-1]
    _, a = _run(w)
    _, b = _run(w)
    _, c = _run(w.with_(dropout_seed=w.dropout_seed + 1))
    for x, y, z in zip(a, b, c):
        assert torch.equal(x, y)
        assert not torch.equal(x, z)


# The benchmarked backward at its full size (B2, H_q 32 / H_kv 8, L 4096, D 128, causal): the
# multi-wave grid and the long per-CTA loops (each dK/dV CTA walks 4 heads x up to 32 query
# blocks) are only exercised at this size.
BENCH_BWD = W.WORKLOADS["bf16_gqa_causal_b2_hq32_hkv8_l4096_d128"]
BENCH_BWD_DROPOUT = W.WORKLOADS["bf16_gqa_causal_dropout10_b2_hq32_hkv8_l4096_d128"]


def _gpu_bwd_full(w):
    import attention_forward_08_gb300 as fa
    q, k, v = W.make_qkv(w)
    do = W.make_dout(w)
    dev = "cuda:0"
    qd, kd, vd, dod = q.to(dev), k.to(dev), v.to(dev), do.to(dev)
    drop = dict(dropout_p=w.dropout_p, dropout_seed=w.dropout_seed, dropout_offset=w.dropout_offset)
    o, lse = fa.attention(qd, kd, vd, scale=w.sm_scale, causal=w.causal, **drop)
    dq, dk, dv = fa.attention_bwd(qd, kd, vd, o, dod, lse, scale=w.sm_scale, causal=w.causal, **drop)
    assert fa.fa_sync_status(None) == fa.fa.FA_OK, fa.fa_last_error()
    return (q, k, v, do), (dq.cpu(), dk.cpu(), dv.cpu())


def test_bwd_bench_workload_every_element():
    """Every element of dQ, dK and dV of the benchmarked backward against the gradient oracle
    (all 16 GQA groups, the oracle's threads one group each)."""
    w = BENCH_BWD
    (q, k, v, do), (dq, dk, dv) = _gpu_bwd_full(w)
    rq, rk, rv = oracle.attention_bwd(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                                      do.double().numpy(), fp32_scale(w), causal=True)
    _compare(f"{w.name} dQ", dq, rq)
    _compare(f"{w.name} dK", dk, rk)
    _compare(f"{w.name} dV", dv, rv)


def test_bwd_f32_dit_workload_every_element():
    """fp32 at the size of the fp32 DiT joint-attention forward workload (B1, H 24, L 4608, D 128,
    non-causal): 864 CTAs in each of the dV, dK and dQ kernels, 72 steps per CTA; every element
    against the gradient oracle."""
    w = S("bwd_f32_dit_h24_l4608_d128", 1, 24, 24, 4608, 4608, 128, "f32", seed=89)
    (q, k, v, do), (dq, dk, dv) = _gpu_bwd_full(w)
    rq, rk, rv = oracle.attention_bwd(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                                      do.double().numpy(), fp32_scale(w), causal=False)
    _compare(f"{w.name} dQ", dq, rq, REL_TOL["f32"])
    _compare(f"{w.name} dK", dk, rk, REL_TOL["f32"])
    _compare(f"{w.name} dV", dv, rv, REL_TOL["f32"])


def test_bwd_d256_multi_wave_every_element():
    """Head dim 256 at the size of the D = 256 forward workload (B1, H_q 8, L 2000) with GQA 4:1 and
    causal masking: 256 dK/dV CTAs (two per 128-key tile) and 128 dQ CTAs, each dK/dV CTA walking 4
    heads x up to 32 query steps; every element against the gradient oracle."""
    w = S("bwd_d256_causal_gqa_h8_l2000", 1, 8, 2, 2000, 2000, 256, "bf16", causal=True, seed=67)
    (q, k, v, do), (dq, dk, dv) = _gpu_bwd_full(w)
    rq, rk, rv = oracle.attention_bwd(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                                      do.double().numpy(), fp32_scale(w), causal=True)
    _compare(f"{w.name} dQ", dq, rq)
    _compare(f"{w.name} dK", dk, rk)
    _compare(f"{w.name} dV", dv, rv)


@pytest.mark.parametrize("b,kvh", [(0, 0), (1, 5)])
def test_bwd_bench_dropout_workload_one_group(b, kvh):
    """The benchmarked dropout backward (p 0.1, seed 2024) on one whole GQA group: dQ of its four
    query heads and dK, dV of its K/V head, element by element.  The oracle runs on the group's
    slice, with the generator's multipliers at the full problem's positions
    ((b H_q + h) qL + i) kL + j."""
    w = BENCH_BWD_DROPOUT
    (q, k, v, do), (dq, dk, dv) = _gpu_bwd_full(w)
    g = w.H_q // w.H_kv
    heads = list(range(kvh * g, (kvh + 1) * g))
    keep = np.stack([oracle.dropout_keep(float(np.float32(w.dropout_p)), w.dropout_seed, w.dropout_offset,
                                         ((b * w.H_q + h) * w.qL) * w.kL, w.qL * w.kL).reshape(w.qL, w.kL)
                     for h in heads])[None]
    sl = lambda t: t[b:b + 1, heads].double().numpy()
    rq, rk, rv = oracle.attention_bwd(sl(q), k[b:b + 1, kvh:kvh + 1].double().numpy(),
                                      v[b:b + 1, kvh:kvh + 1].double().numpy(), sl(do), fp32_scale(w),
                                      causal=True, keep=keep)
    del keep
    _compare(f"{w.name} b{b} kvh{kvh} dQ", dq[b:b + 1, heads], rq)
    _compare(f"{w.name} b{b} kvh{kvh} dK", dk[b:b + 1, kvh:kvh + 1], rk)
    _compare(f"{w.name} b{b} kvh{kvh} dV", dv[b:b + 1, kvh:kvh + 1], rv)


def test_bwd_bool_mask_workload_every_element():
    """The benchmarked bool-mask backward (B1, H 8, L 2000, D 128; a tenth of the entries dropped,
    the diagonal kept): the keep-bits pre-pass, 128 dK/dV and 128 dQ CTAs; every element of dQ, dK
    and dV against the gradient oracle."""
    _run_masked(W.WORKLOADS["bf16_bool_mask_h8_l2000_d128"])


def test_bwd_bool_mask_bench_shape_one_group():
    """A bool mask on the benchmarked causal shape (B2, H_q 32, H_kv 8, L 4096, D 128): the bits
    pre-pass skips the tiles above the diagonal and the gradient kernels fetch each step's keep
    words a step ahead, over up to 128 steps per dK/dV CTA.  dQ of one GQA group's four query
    heads and dK, dV of its K/V head, element by element."""
    import attention_forward_08_gb300 as fa
    w = BENCH_BWD.with_(name="bwd_bool_mask_bench_shape", mask_kind=W.MASK_BOOL)
    q, k, v, m = W.make_inputs(w)
    do = W.make_dout(w)
    dev = "cuda:0"
    qd, kd, vd, dod, md = q.to(dev), k.to(dev), v.to(dev), do.to(dev), m.to(dev)
    kw = dict(scale=w.sm_scale, causal=True, mask=md, mask_kind=W.MASK_BOOL)
    o, lse = fa.attention(qd, kd, vd, **kw)
    dq, dk, dv = fa.attention_bwd(qd, kd, vd, o, dod, lse, **kw)
    assert fa.fa_sync_status(None) == fa.fa.FA_OK, fa.fa_last_error()
    dq, dk, dv = dq.cpu(), dk.cpu(), dv.cpu()
    del qd, kd, vd, dod, md, o, lse
    b, kvh = 1, 3
    g = w.H_q // w.H_kv
    heads = list(range(kvh * g, (kvh + 1) * g))
    sl = lambda t: t[b:b + 1, heads].double().numpy()
    rq, rk, rv = oracle.attention_bwd(sl(q), k[b:b + 1, kvh:kvh + 1].double().numpy(),
                                      v[b:b + 1, kvh:kvh + 1].double().numpy(), sl(do), fp32_scale(w),
                                      causal=True, mask=sl(m), mask_kind=W.MASK_BOOL)
    _compare(f"{w.name} b{b} kvh{kvh} dQ", dq[b:b + 1, heads], rq)
    _compare(f"{w.name} b{b} kvh{kvh} dK", dk[b:b + 1, kvh:kvh + 1], rk)
    _compare(f"{w.name} b{b} kvh{kvh} dV", dv[b:b + 1, kvh:kvh + 1], rv)


# The forward's mask in the backward (fa_bwd_full): bool (nonzero keeps) and additive (-inf excludes),
# with causal, GQA, ragged tails, fp16, dropout and a sliding window; mask rows whose byte stride is not a
# multiple of 16 take the element-wise load path.
MASKED = [
    S("bwd_mask_bool_d128_causal_gqa", 1, 4, 2, 384, 384, 128, "bf16", causal=True, mask_kind=W.MASK_BOOL, seed=71),
    S("bwd_mask_add_d64_ragged_unaligned", 2, 2, 1, 200, 333, 64, "bf16", mask_kind=W.MASK_ADDITIVE, seed=72),
    S("bwd_mask_add_f16_d128_causal", 1, 2, 2, 300, 300, 128, "f16", causal=True, mask_kind=W.MASK_ADDITIVE,
      seed=73),
    S("bwd_mask_bool_f16_d64_q_longer", 1, 2, 2, 260, 130, 64, "f16", mask_kind=W.MASK_BOOL, seed=74),
    S("bwd_mask_bool_d64_dropout", 1, 2, 1, 256, 256, 64, "bf16", causal=True, mask_kind=W.MASK_BOOL,
      dropout_p=0.2, dropout_seed=31, seed=75),
    S("bwd_mask_add_d128_window", 1, 2, 2, 300, 300, 128, "bf16", causal=True, mask_kind=W.MASK_ADDITIVE,
      window=100, seed=76),
    S("bwd_mask_add_d128_gqa_long_kv", 1, 4, 1, 130, 520, 128, "bf16", mask_kind=W.MASK_ADDITIVE, seed=77),
    # causal with the diagonal moved right (kL > qL): the mask pre-passes skip the tiles no row of which
    # sees any key, on a 128 (bool) or 64 (additive) grid that the offset does not align with
    S("bwd_mask_bool_causal_offset", 1, 2, 2, 200, 456, 128, "bf16", causal=True, q_offset=200,
      mask_kind=W.MASK_BOOL, seed=80),
    S("bwd_mask_add_d64_causal_offset", 1, 2, 1, 300, 520, 64, "bf16", causal=True, q_offset=220,
      mask_kind=W.MASK_ADDITIVE, seed=81),
    S("bwd_mask_bool_negative_offset", 1, 2, 2, 300, 300, 64, "bf16", causal=True, q_offset=-150,
      mask_kind=W.MASK_BOOL, seed=82),
]


def _run_masked(w, mask=None):
    import attention_forward_08_gb300 as fa
    q, k, v, m = W.make_inputs(w)
    if mask is not None:
        m = mask
    do = W.make_dout(w)
    dev = "cuda:0"
    qd, kd, vd, dod, md = q.to(dev), k.to(dev), v.to(dev), do.to(dev), m.to(dev)
    kw = dict(scale=w.sm_scale, causal=w.causal, window=w.window, q_offset=w.q_offset, dropout_p=w.dropout_p,
              dropout_seed=w.dropout_seed, dropout_offset=w.dropout_offset, mask=md, mask_kind=w.mask_kind)
    o, lse = fa.attention(qd, kd, vd, **kw)
    dq, dk, dv = fa.attention_bwd(qd, kd, vd, o, dod, lse, **kw)
    assert fa.fa_sync_status(None) == fa.fa.FA_OK, fa.fa_last_error()
    rq, rk, rv = oracle.attention_bwd(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                                      do.double().numpy(), fp32_scale(w), causal=w.causal, mask=m.double().numpy(),
                                      mask_kind=w.mask_kind, window=w.window, q_offset=w.q_offset,
                                      dropout_p=float(np.float32(w.dropout_p)), seed=w.dropout_seed,
                                      offset=w.dropout_offset)
    tol = REL_TOL[w.dtype]
    _compare(f"{w.name} dQ", dq, rq, tol)
    _compare(f"{w.name} dK", dk, rk, tol)
    _compare(f"{w.name} dV", dv, rv, tol)
    return (dq, dk, dv), lse


@pytest.mark.parametrize("w", MASKED, ids=lambda w: w.name)
def test_bwd_masked(w):
    _run_masked(w)


def test_bwd_masked_empty_rows_and_keys():
    """Rows whose bool mask keeps no key (L = -inf) get dQ = 0 exactly, and keys no row keeps get dK = dV = 0."""
    w = S("bwd_mask_bool_empty", 1, 2, 2, 256, 256, 128, "bf16", mask_kind=W.MASK_BOOL, seed=78)
    g = torch.Generator().manual_seed(6)
    m = (torch.rand(1, 2, 256, 256, generator=g) < 0.6).to(torch.uint8)
    m[0, 0, 17] = 0
    m[0, 1, 130:140] = 0
    m[0, :, :, 200] = 0
    (dq, dk, dv), lse = _run_masked(w, mask=m)
    assert torch.isneginf(lse[0, 0, 17]) and torch.isneginf(lse[0, 1, 130:140]).all()
    assert torch.count_nonzero(dq[0, 0, 17]).item() == 0 and torch.count_nonzero(dq[0, 1, 130:140]).item() == 0
    assert torch.count_nonzero(dk[0, :, 200]).item() == 0 and torch.count_nonzero(dv[0, :, 200]).item() == 0


def test_bwd_masked_broadcast_strides():
    """An additive mask broadcast over batch and heads through zero strides."""
    w = S("bwd_mask_add_bcast", 2, 2, 2, 200, 264, 64, "bf16", causal=True, mask_kind=W.MASK_ADDITIVE, seed=79)
    g = torch.Generator().manual_seed(8)
    base = torch.randn(1, 1, 200, 264, generator=g).to(torch.bfloat16)
    base[0, 0, torch.rand(200, 264, generator=g) < 0.1] = float("-inf")
    base[0, 0, torch.arange(200), torch.arange(200)] = 0.0
    _run_masked(w, mask=base)  # [1, 1, qL, kL]: the binding expands it with zero strides
