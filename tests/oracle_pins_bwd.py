"""Pins for the fp64 gradient oracle: facts fixed by mathematics, not by the oracle.

Each ``pin_*`` takes ``grad`` (a callable with the signature of
``oracle.attention_bwd`` minus ``lib``) and ``fwd`` (``oracle.attention``,
itself pinned by ``oracle_pins``), and raises AssertionError when the
gradients disagree with:
  - central finite differences of the forward oracle's loss sum(O * dO)
    along random directions, with every feature switched on in turn,
  - an independent library routine (torch fp64 CPU autograd through
    scaled_dot_product_attention, K/V repeated per GQA group),
  - closed forms (Q = 0 gives uniform weights, so dV_j sums dO_i / n_i over
    the rows that see key j, each times its dropout multiplier when there is
    dropout; rows of equal V make O independent of Q and K),
  - invariants that hold exactly (shifting every key by the same vector leaves
    every softmax row unchanged, so sum_j dK_j = 0; gradients are linear in dO).
Each planted mistake (dropped scale in dK, sign of the D term, q in place of
dO in dV, wrong heads summed into dK/dV, causal off by one, dQ sign, the
query offset's sign, a window one key too wide, the softcap's derivative
dropped, dropout left out of dV) fails one.
"""
from __future__ import annotations

import numpy as np
import torch

TOL = 1e-9


def _rng(seed):
    return np.random.default_rng(seed)


def _close(a, b, tol=TOL, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    err = np.max(np.abs(a - b) / (1.0 + np.abs(b))) if a.size else 0.0
    assert err <= tol, f"{what}: max rel err {err:.3e} > {tol:.1e}"


def _inputs(r, B, Hq, Hkv, qL, kL, D):
    q = r.standard_normal((B, Hq, qL, D))
    k = r.standard_normal((B, Hkv, kL, D))
    v = r.standard_normal((B, Hkv, kL, D))
    g = r.standard_normal((B, Hq, qL, D))
    return q, k, v, g


CASES = [
    # (B, Hq, Hkv, qL, kL, D, causal, mask_kind)
    (1, 2, 2, 5, 7, 4, False, 0),
    (2, 4, 2, 6, 6, 3, True, 0),
    (1, 3, 1, 4, 9, 5, False, 1),
    (1, 2, 1, 7, 5, 4, True, 2),
]


def _mask(r, kind, B, Hq, qL, kL):
    if kind == 1:
        m = (r.random((B, Hq, qL, kL)) < 0.7).astype(np.uint8)
        m[..., 0] = 1
        return m
    if kind == 2:
        m = r.standard_normal((B, Hq, qL, kL))
        m[r.random((B, Hq, qL, kL)) < 0.2] = -np.inf
        m[..., 0] = 0.0
        return m
    return None


# --------------------------------------------------------------------------- finite differences

def pin_finite_differences(grad, fwd):
    """Directional derivatives of sum(O * dO) by central differences of the forward oracle."""
    r = _rng(101)
    eps = 1e-5
    for (B, Hq, Hkv, qL, kL, D, causal, kind) in CASES:
        q, k, v, g = _inputs(r, B, Hq, Hkv, qL, kL, D)
        m = _mask(r, kind, B, Hq, qL, kL)
        scale = 0.45
        dq, dk, dv = grad(q, k, v, g, scale, causal=causal, mask=m, mask_kind=kind)

        def loss(qq, kk, vv):
            o, _ = fwd(qq, kk, vv, scale, causal=causal, mask=m, mask_kind=kind)
            return float(np.sum(o * g))

        for which, x, dx in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            for _ in range(2):
                e = r.standard_normal(x.shape)
                args_p = [q, k, v]
                args_m = [q, k, v]
                idx = "qkv".index(which)
                args_p[idx] = x + eps * e
                args_m[idx] = x - eps * e
                fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
                an = float(np.sum(dx * e))
                assert abs(fd - an) <= 1e-6 * (1.0 + abs(fd)), \
                    f"d{which} case {(B, Hq, Hkv, qL, kL, D, causal, kind)}: fd {fd:.9f} vs {an:.9f}"


def pin_finite_differences_softcap(grad, fwd):
    """The same directional derivatives with a softcap (the forward oracle's softcap is pinned on its
    own), with scores large enough for the cap to bend them, alone and with a causal window."""
    r = _rng(107)
    eps = 1e-5
    for (B, Hq, Hkv, qL, kL, D, causal, window, cap) in (
            (1, 2, 1, 6, 7, 4, False, 0, 1.5),
            (1, 2, 2, 7, 7, 3, True, 3, 2.5)):
        q, k, v, g = _inputs(r, B, Hq, Hkv, qL, kL, D)
        scale = 1.3
        dq, dk, dv = grad(q, k, v, g, scale, causal=causal, window=window, softcap=cap)

        def loss(qq, kk, vv):
            o, _ = fwd(qq, kk, vv, scale, causal=causal, window=window, softcap=cap)
            return float(np.sum(o * g))

        for which, x, dx in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            for _ in range(2):
                e = r.standard_normal(x.shape)
                args_p, args_m = [q, k, v], [q, k, v]
                idx = "qkv".index(which)
                args_p[idx] = x + eps * e
                args_m[idx] = x - eps * e
                fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
                an = float(np.sum(dx * e))
                assert abs(fd - an) <= 1e-6 * (1.0 + abs(fd)), \
                    f"d{which} softcap {cap}: fd {fd:.9f} vs {an:.9f}"


def pin_finite_differences_dropout(grad, fwd):
    """The same directional derivatives with dropout: the forward oracle's generator fixes the
    multipliers for a given seed, so the loss is smooth in q, k and v."""
    r = _rng(109)
    eps = 1e-5
    for (B, Hq, Hkv, qL, kL, D, causal, p, seed, off) in (
            (1, 2, 1, 6, 8, 4, False, 0.3, 11, 0),
            (2, 2, 2, 5, 8, 3, True, 0.5, 2 ** 40 + 5, 2 ** 32 - 3)):
        q, k, v, g = _inputs(r, B, Hq, Hkv, qL, kL, D)
        scale = 0.45
        dq, dk, dv = grad(q, k, v, g, scale, causal=causal, dropout_p=p, seed=seed, offset=off)

        def loss(qq, kk, vv):
            o, _ = fwd(qq, kk, vv, scale, causal=causal, dropout_p=p, seed=seed, offset=off)
            return float(np.sum(o * g))

        for which, x, dx in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            for _ in range(2):
                e = r.standard_normal(x.shape)
                args_p, args_m = [q, k, v], [q, k, v]
                idx = "qkv".index(which)
                args_p[idx] = x + eps * e
                args_m[idx] = x - eps * e
                fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
                an = float(np.sum(dx * e))
                assert abs(fd - an) <= 1e-6 * (1.0 + abs(fd)), \
                    f"d{which} dropout {p}: fd {fd:.9f} vs {an:.9f}"


def pin_finite_differences_window_offset(grad, fwd):
    """The same directional derivatives with a sliding window and a causal diagonal offset (the
    forward oracle's window / q_offset are pinned on their own), including a non-causal window and
    an offset that leaves some rows without keys."""
    r = _rng(103)
    eps = 1e-5
    for (B, Hq, Hkv, qL, kL, D, causal, window, off) in (
            (1, 2, 1, 6, 9, 4, True, 3, 2),
            (2, 2, 2, 7, 7, 3, True, 4, 0),
            (1, 2, 2, 5, 8, 4, False, 3, 1),
            (1, 2, 1, 6, 6, 3, True, 0, -2)):
        q, k, v, g = _inputs(r, B, Hq, Hkv, qL, kL, D)
        scale = 0.45
        dq, dk, dv = grad(q, k, v, g, scale, causal=causal, window=window, q_offset=off)

        def loss(qq, kk, vv):
            o, _ = fwd(qq, kk, vv, scale, causal=causal, window=window, q_offset=off)
            return float(np.sum(o * g))

        for which, x, dx in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            for _ in range(2):
                e = r.standard_normal(x.shape)
                args_p, args_m = [q, k, v], [q, k, v]
                idx = "qkv".index(which)
                args_p[idx] = x + eps * e
                args_m[idx] = x - eps * e
                fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
                an = float(np.sum(dx * e))
                assert abs(fd - an) <= 1e-6 * (1.0 + abs(fd)), \
                    f"d{which} window {window} offset {off}: fd {fd:.9f} vs {an:.9f}"


# --------------------------------------------------------------------------- library cross-check

def pin_torch_autograd(grad, fwd):
    """torch fp64 CPU autograd through scaled_dot_product_attention (K/V repeated per group)."""
    r = _rng(102)
    for (B, Hq, Hkv, qL, kL, D, causal, kind) in CASES:
        q, k, v, g = _inputs(r, B, Hq, Hkv, qL, kL, D)
        m = _mask(r, kind, B, Hq, qL, kL)
        scale = 0.6
        dq, dk, dv = grad(q, k, v, g, scale, causal=causal, mask=m, mask_kind=kind)
        tq = torch.tensor(q, requires_grad=True)
        tk = torch.tensor(k, requires_grad=True)
        tv = torch.tensor(v, requires_grad=True)
        rep = Hq // Hkv
        bias = torch.zeros((B, Hq, qL, kL), dtype=torch.float64)
        if causal:
            bias = bias.masked_fill(torch.ones(qL, kL, dtype=torch.bool).triu(1), float("-inf"))
        if kind == 1:
            bias = bias.masked_fill(torch.tensor(m == 0), float("-inf"))
        elif kind == 2:
            bias = bias + torch.tensor(m)
        o = torch.nn.functional.scaled_dot_product_attention(
            tq, tk.repeat_interleave(rep, dim=1), tv.repeat_interleave(rep, dim=1), attn_mask=bias, scale=scale)
        (o * torch.tensor(g)).sum().backward()
        _close(dq, tq.grad.numpy(), 1e-10, "dq vs torch")
        _close(dk, tk.grad.numpy(), 1e-10, "dk vs torch")
        _close(dv, tv.grad.numpy(), 1e-10, "dv vs torch")


# --------------------------------------------------------------------------- closed forms

def pin_uniform_weights_dv(grad, fwd):
    """Q = 0: row i weighs its n_i allowed keys equally, so dV_j = sum over heads/rows seeing j of dO_i / n_i."""
    r = _rng(103)
    B, Hq, Hkv, qL, kL, D = 1, 4, 2, 6, 6, 3
    q = np.zeros((B, Hq, qL, D))
    _, k, v, g = _inputs(r, B, Hq, Hkv, qL, kL, D)
    for causal in (False, True):
        _, _, dv = grad(q, k, v, g, 0.8, causal=causal)
        want = np.zeros_like(v)
        rep = Hq // Hkv
        for h in range(Hq):
            for i in range(qL):
                n = (i + 1) if causal else kL
                for j in range(n):
                    want[0, h // rep, j] += g[0, h, i] / n
        _close(dv, want, 1e-12, f"dV closed form causal={causal}")


def pin_uniform_weights_dv_dropout(grad, fwd):
    """Q = 0 with dropout: row i weighs its n_i allowed keys by Z_ij / n_i, so dV_j sums
    Z_ij dO_i / n_i; Z_ij is the forward oracle generator's multiplier at position
    ((b H_q + h) qL + i) kL + j."""
    import oracle
    r = _rng(113)
    B, Hq, Hkv, qL, kL, D = 1, 4, 2, 6, 8, 3
    q = np.zeros((B, Hq, qL, D))
    _, k, v, g = _inputs(r, B, Hq, Hkv, qL, kL, D)
    p, seed, off = 0.4, 77, 5
    z = oracle.dropout_keep(p, seed, off, 0, B * Hq * qL * kL).reshape(B, Hq, qL, kL)
    assert 0 < int(np.sum(z == 0.0)) < z.size  # some weights dropped, some kept
    rep = Hq // Hkv
    for causal in (False, True):
        _, _, dv = grad(q, k, v, g, 0.8, causal=causal, dropout_p=p, seed=seed, offset=off)
        want = np.zeros_like(v)
        for h in range(Hq):
            for i in range(qL):
                n = (i + 1) if causal else kL
                for j in range(n):
                    want[0, h // rep, j] += z[0, h, i, j] * g[0, h, i] / n
        _close(dv, want, 1e-12, f"dV closed form with dropout causal={causal}")


def pin_equal_values_no_qk_gradient(grad, fwd):
    """Every V row equal: O_i = V_0 whatever the weights, so dQ = dK = 0 and dV_j = sum_i P_ij dO_i."""
    r = _rng(104)
    B, Hq, Hkv, qL, kL, D = 1, 2, 1, 5, 8, 4
    q, k, _, g = _inputs(r, B, Hq, Hkv, qL, kL, D)
    v = np.broadcast_to(r.standard_normal((1, 1, 1, D)), (B, Hkv, kL, D)).copy()
    dq, dk, dv = grad(q, k, v, g, 0.7, causal=True)
    assert np.max(np.abs(dq)) < 1e-12 and np.max(np.abs(dk)) < 1e-12, "dQ/dK must vanish when V rows are equal"
    assert np.abs(dv.sum(axis=2) - g.sum(axis=(1, 2))[:, None]).max() < 1e-12, "sum_j dV_j = sum_i dO_i"


# --------------------------------------------------------------------------- invariants

def pin_key_shift_invariance(grad, fwd):
    """Adding one vector to every key shifts each softmax row uniformly: sum_j dK_j = 0."""
    r = _rng(105)
    for (B, Hq, Hkv, qL, kL, D, causal, kind) in CASES:
        q, k, v, g = _inputs(r, B, Hq, Hkv, qL, kL, D)
        m = _mask(r, kind, B, Hq, qL, kL)
        _, dk, _ = grad(q, k, v, g, 0.9, causal=causal, mask=m, mask_kind=kind)
        assert np.abs(dk.sum(axis=2)).max() < 1e-12, "sum over keys of dK must vanish"


def pin_linear_in_dout(grad, fwd):
    """Gradients are linear in dO."""
    r = _rng(106)
    B, Hq, Hkv, qL, kL, D = 1, 2, 2, 4, 6, 3
    q, k, v, g1 = _inputs(r, B, Hq, Hkv, qL, kL, D)
    g2 = r.standard_normal(g1.shape)
    a = grad(q, k, v, g1, 0.5, causal=True)
    b = grad(q, k, v, g2, 0.5, causal=True)
    c = grad(q, k, v, 2.0 * g1 - 3.0 * g2, 0.5, causal=True)
    for x, y, z, n in zip(a, b, c, ("dq", "dk", "dv")):
        _close(z, 2.0 * x - 3.0 * y, 1e-12, f"{n} linear in dO")


ALL_PINS = [
    pin_finite_differences,
    pin_finite_differences_window_offset,
    pin_finite_differences_softcap,
    pin_finite_differences_dropout,
    pin_torch_autograd,
    pin_uniform_weights_dv,
    pin_uniform_weights_dv_dropout,
    pin_equal_values_no_qk_gradient,
    pin_key_shift_invariance,
    pin_linear_in_dout,
]
