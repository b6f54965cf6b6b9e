"""Seeded synthetic inputs shared by the parity tests, the smoke check and the bench.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  Both the fp64 oracle and the CUDA library consume what
it produces, so it imports neither of them.

Recipe (same for every workload): a CPU ``torch.Generator`` seeded with
``seed`` draws Q, K, V in that order as fp32 N(0, 1), which are then cast to
the workload's I/O dtype.  Masks use their own generator (``mask_seed``):
  additive  -- N(0, 1) cast to the I/O dtype, then Bernoulli(0.1) entries set
               to -inf, with the diagonal left finite so no row is empty;
  bool      -- Bernoulli(0.9) keep, with the diagonal forced to keep.
Backward runs draw the upstream gradient dO as N(0, 1) from seed + 500.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch

MASK_NONE, MASK_BOOL, MASK_ADDITIVE = 0, 1, 2


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H_q: int
    H_kv: int
    qL: int
    kL: int
    D: int
    dtype: str            # "bf16", "f16" or "f32"
    causal: bool = False
    mask_kind: int = MASK_NONE
    layout: str = "bhsd"  # "bhsd", or "dit": O written token-major [seq, H*D]
    seed: int = 1000
    mask_seed: int = 2000
    scale: float = field(default=float("nan"))
    window: int = 0        # > 0: sliding window of keys j > i + q_offset - window
    softcap: float = 0.0   # > 0: scores capped as softcap * tanh(s / softcap)
    q_offset: int = 0      # causal diagonal of row i is key i + q_offset
    dropout_p: float = 0.0  # > 0: weights of O dropped with probability p (counter-based generator)
    dropout_seed: int = 0
    dropout_offset: int = 0

    @property
    def sm_scale(self) -> float:
        return 1.0 / math.sqrt(self.D) if math.isnan(self.scale) else self.scale

    @property
    def torch_dtype(self):
        return {"bf16": torch.bfloat16, "f16": torch.float16}.get(self.dtype, torch.float32)

    def flops(self) -> float:
        """Algorithmic FLOP: 4*B*H_q*qL*kL*D, halved when causal; with a window
        or a query offset, 4*B*H_q*D times the exact number of allowed (i, j) pairs."""
        if self.window == 0 and self.q_offset == 0:
            f = 4.0 * self.B * self.H_q * self.qL * self.kL * self.D
            return f / 2.0 if self.causal else f
        pairs = 0
        for i in range(self.qL):
            hi = min(self.kL - 1, i + self.q_offset) if self.causal else self.kL - 1
            lo = max(0, i + self.q_offset - self.window + 1) if self.window > 0 else 0
            pairs += max(0, hi - lo + 1)
        return 4.0 * self.B * self.H_q * self.D * pairs

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# The five workloads of the pages (FA-2 forward on one GPU).
WORKLOADS = {
    "fp32_b1_h2_l128_d64": Workload("fp32_b1_h2_l128_d64", 1, 2, 2, 128, 128, 64, "f32", seed=1000),
    "bf16_causal_b4_h8_l1024_d64": Workload("bf16_causal_b4_h8_l1024_d64", 4, 8, 8, 1024, 1024, 64,
                                            "bf16", causal=True, seed=1001),
    "bf16_gqa_causal_b2_hq32_hkv8_l4096_d128": Workload(
        "bf16_gqa_causal_b2_hq32_hkv8_l4096_d128", 2, 32, 8, 4096, 4096, 128, "bf16",
        causal=True, seed=1002),
    "fp32_dit_h24_l4608_d128_tokenmajor": Workload(
        "fp32_dit_h24_l4608_d128_tokenmajor", 1, 24, 24, 4608, 4608, 128, "f32",
        layout="dit", seed=1003),
    "bf16_additive_mask_h8_l2000_d256": Workload(
        "bf16_additive_mask_h8_l2000_d256", 1, 8, 8, 2000, 2000, 256, "bf16",
        mask_kind=MASK_ADDITIVE, seed=1004),
    "bf16_bool_mask_h8_l2000_d256": Workload(
        "bf16_bool_mask_h8_l2000_d256", 1, 8, 8, 2000, 2000, 256, "bf16",
        mask_kind=MASK_BOOL, seed=1004),
}

BENCH_WORKLOAD = "bf16_gqa_causal_b2_hq32_hkv8_l4096_d128"

# Beyond the pages' workloads: the bench workload with fp16 I/O, with a
# 1024-key sliding window, with a softcap of 20, and with dropout 0.1 (same seeds);
# two backward shapes.
EXTRA_WORKLOADS = {
    "f16_gqa_causal_b2_hq32_hkv8_l4096_d128": Workload(
        "f16_gqa_causal_b2_hq32_hkv8_l4096_d128", 2, 32, 8, 4096, 4096, 128, "f16", causal=True, seed=1002),
    "bf16_gqa_causal_swa1024_b2_hq32_hkv8_l4096_d128": Workload(
        "bf16_gqa_causal_swa1024_b2_hq32_hkv8_l4096_d128", 2, 32, 8, 4096, 4096, 128, "bf16", causal=True,
        seed=1002, window=1024),
    "bf16_gqa_causal_softcap20_b2_hq32_hkv8_l4096_d128": Workload(
        "bf16_gqa_causal_softcap20_b2_hq32_hkv8_l4096_d128", 2, 32, 8, 4096, 4096, 128, "bf16", causal=True,
        seed=1002, softcap=20.0),
    "bf16_gqa_causal_dropout10_b2_hq32_hkv8_l4096_d128": Workload(
        "bf16_gqa_causal_dropout10_b2_hq32_hkv8_l4096_d128", 2, 32, 8, 4096, 4096, 128, "bf16", causal=True,
        seed=1002, dropout_p=0.1, dropout_seed=2024, dropout_offset=0),
    # The D = 256 shape of the masked workloads without a mask (the head dim the backward
    # takes at 256), and at D = 128 with the bool mask (a masked backward).
    "bf16_h8_l2000_d256": Workload("bf16_h8_l2000_d256", 1, 8, 8, 2000, 2000, 256, "bf16", seed=1004),
    "bf16_bool_mask_h8_l2000_d128": Workload(
        "bf16_bool_mask_h8_l2000_d128", 1, 8, 8, 2000, 2000, 128, "bf16", mask_kind=MASK_BOOL, seed=1004),
}
WORKLOADS.update(EXTRA_WORKLOADS)


def make_qkv(w: Workload):
    """Q [B,H_q,qL,D], K and V [B,H_kv,kL,D] on the CPU in the I/O dtype."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    q = torch.randn(w.B, w.H_q, w.qL, w.D, generator=g, dtype=torch.float32)
    k = torch.randn(w.B, w.H_kv, w.kL, w.D, generator=g, dtype=torch.float32)
    v = torch.randn(w.B, w.H_kv, w.kL, w.D, generator=g, dtype=torch.float32)
    dt = w.torch_dtype
    return q.to(dt), k.to(dt), v.to(dt)


def make_dout(w: Workload):
    """The upstream gradient dO [B,H_q,qL,D] for backward runs: N(0, 1) from seed + 500, I/O dtype."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed + 500)
    return torch.randn(w.B, w.H_q, w.qL, w.D, generator=g, dtype=torch.float32).to(w.torch_dtype)


def make_mask(w: Workload):
    """The workload's mask on the CPU: None, uint8 keep-mask, or additive in the I/O dtype."""
    if w.mask_kind == MASK_NONE:
        return None
    g = torch.Generator(device="cpu")
    g.manual_seed(w.mask_seed)
    shape = (w.B, w.H_q, w.qL, w.kL)
    n = min(w.qL, w.kL)
    idx = torch.arange(n)
    if w.mask_kind == MASK_ADDITIVE:
        vals = torch.randn(*shape, generator=g, dtype=torch.float32).to(w.torch_dtype)
        drop = torch.rand(*shape, generator=g) < 0.1
        drop[..., idx, idx] = False
        vals[drop] = float("-inf")
        return vals
    keep = torch.rand(*shape, generator=g) < 0.9
    keep[..., idx, idx] = True
    return keep.to(torch.uint8)


def make_inputs(w: Workload):
    q, k, v = make_qkv(w)
    return q, k, v, make_mask(w)


def small_case(name, B, H_q, H_kv, qL, kL, D, dtype, causal=False, mask_kind=MASK_NONE,
               layout="bhsd", seed=7, scale=float("nan"), window=0, softcap=0.0, q_offset=0,
               dropout_p=0.0, dropout_seed=0, dropout_offset=0) -> Workload:
    """A reduced-size workload for element-by-element parity runs."""
    return Workload(name, B, H_q, H_kv, qL, kL, D, dtype, causal=causal, mask_kind=mask_kind,
                    layout=layout, seed=seed, mask_seed=seed + 1000, scale=scale, window=window,
                    softcap=softcap, q_offset=q_offset, dropout_p=dropout_p, dropout_seed=dropout_seed,
                    dropout_offset=dropout_offset)
