"""Shared helpers for the GPU parity tests: run the CUDA library and the oracle
on the same seeded inputs and compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import workloads

# Tolerances on N(0,1) inputs, max over every output with a finite oracle L.
# (max |dO|, max |dL|).  bf16 and fp32 (TF32) are the stated bounds; fp16 I/O
# (three more mantissa bits than bf16: O rounding <= 2^-10 for |O| < 4, P
# rounding 2^-11 relative) takes a quarter of the bf16 bounds.
TOL = {"bf16": (2e-2, 1e-2), "f16": (5e-3, 2.5e-3), "f32": (2e-3, 1e-3)}


def gpu_run(w: workloads.Workload, q, k, v, mask, scale=None, workspace=None):
    """Copy the CPU inputs to cuda:0, run the library, return (O, L) as fp64 numpy, O in [B,H,qL,D].
    workspace=False runs without the library's scratch (fp32: the in-kernel tf32 helper plan)."""
    import attention_forward_08_gb300 as fa
    dev = torch.device("cuda:0")
    qd, kd, vd = q.to(dev), k.to(dev), v.to(dev)
    md = mask.to(dev) if mask is not None else None
    B, H, qL, D = q.shape
    if w.layout == "dit":
        o_tok = torch.full((qL, H * D), float("nan"), dtype=q.dtype, device=dev)
        o = o_tok.view(qL, H, D).permute(1, 0, 2).unsqueeze(0)
    else:
        o = torch.full((B, H, qL, D), float("nan"), dtype=q.dtype, device=dev)
    lse = torch.full((B, H, qL), float("nan"), dtype=torch.float32, device=dev)
    fa.attention(qd, kd, vd, scale=w.sm_scale if scale is None else scale, causal=w.causal, mask=md,
                 mask_kind=None if mask is None else w.mask_kind, out=o, lse=lse, window=w.window,
                 q_offset=w.q_offset, softcap=w.softcap, dropout_p=w.dropout_p, dropout_seed=w.dropout_seed,
                 dropout_offset=w.dropout_offset, workspace=workspace)
    rc = fa.fa_sync_status(None)
    assert rc == 0, f"device status {rc}: {fa.fa_last_error()}"
    if w.layout == "dit":
        o_bhsd = o_tok.view(qL, H, D).permute(1, 0, 2).unsqueeze(0)
        return o_bhsd.double().cpu().numpy(), lse.double().cpu().numpy(), o_tok
    return o.double().cpu().numpy(), lse.double().cpu().numpy(), o


def oracle_features(w: workloads.Workload) -> dict:
    """The workload's window / softcap / query offset / dropout as oracle keyword arguments
    (real-valued ones rounded to the fp32 values the GPU receives)."""
    return dict(window=w.window, softcap=float(np.float32(w.softcap)), q_offset=w.q_offset,
                dropout_p=float(np.float32(w.dropout_p)), seed=w.dropout_seed, offset=w.dropout_offset)


def oracle_inputs(q, k, v, mask):
    return (q.double().numpy(), k.double().numpy(), v.double().numpy(),
            None if mask is None else mask.double().numpy())


def fp32_scale(w: workloads.Workload, scale=None) -> float:
    """The scale exactly as the GPU receives it (an fp32 value)."""
    s = w.sm_scale if scale is None else scale
    return float(np.float32(s))


def compare(w, o_gpu, l_gpu, o_ref, l_ref, what="", tol_mult=1.0, tol_mult_l=None):
    tol_o, tol_l = TOL[w.dtype]
    tol_o, tol_l = tol_o * tol_mult, tol_l * (tol_mult if tol_mult_l is None else tol_mult_l)
    fin = np.isfinite(l_ref)
    # rows with no allowed key: O = 0, L = -inf exactly
    assert np.array_equal(np.isneginf(l_gpu), ~fin), f"{what}: -inf rows of L differ"
    if (~fin).any():
        assert np.all(o_gpu[~fin] == 0.0), f"{what}: empty rows must have O = 0"
    assert np.all(np.isfinite(o_gpu)), f"{what}: non-finite O"
    d_o = np.abs(o_gpu[fin] - o_ref[fin]).max() if fin.any() else 0.0
    d_l = np.abs(l_gpu[fin] - l_ref[fin]).max() if fin.any() else 0.0
    a = o_gpu[fin].ravel(); b = o_ref[fin].ravel()
    cos = float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b) + 1e-300)) if a.size else 1.0
    assert d_o <= tol_o, f"{what}: max|dO| = {d_o:.3e} > {tol_o} (cos {cos:.6f})"
    assert d_l <= tol_l, f"{what}: max|dL| = {d_l:.3e} > {tol_l}"
    return d_o, d_l, cos


def sample_rows(w: workloads.Workload, n_per_head: int, seed: int = 0):
    """Flat row indices: first, last and random rows of every (b, h), plus every tile boundary row
    of one head."""
    r = np.random.default_rng(seed)
    rows = []
    for b in range(w.B):
        for h in range(w.H_q):
            base = (b * w.H_q + h) * w.qL
            pick = {0, w.qL - 1, *r.integers(0, w.qL, size=n_per_head).tolist()}
            rows += [base + i for i in sorted(pick)]
    for i in range(127, w.qL, 128):
        rows += [i, min(i + 1, w.qL - 1)]
    return sorted(set(rows))
