"""Pins for the fp64 oracle: facts fixed by mathematics, not by the oracle itself.

Each ``pin_*`` takes ``attn`` (a callable with the signature of
``oracle.attention`` minus ``lib``) and raises AssertionError when the oracle
disagrees with:
  - closed forms (equal scores give the mean of V and L = ln(n) + s; a one-hot
    key gives that key's V row and its score; causal row 0 gives V[0]),
  - a hand-worked example stored under tests/golden/,
  - brute force in 50-digit decimal arithmetic on tiny inputs,
  - an independent library routine (torch's fp64 CPU scaled_dot_product_attention
    and logsumexp),
  - invariants that hold exactly (key permutation, additive-mask shift,
    linearity in V, GQA == MHA with K/V repeated, mask-kind equivalences).
  - for the sliding window, softcap and query offset: decimal brute force,
    window of one key, equal scores in a window, bottom-right causal as the
    suffix of the full causal problem, and a huge cap recovering plain scores.
The pins are chosen so each planted mistake in the oracle (dropped scale,
wrong GQA map, causal off by one, L without the max, transposed product,
scaled mask, flipped bool polarity, missing division by l, softcap not
multiplied back, query-offset sign, window one key too wide) fails one.
"""
from __future__ import annotations

import json
import math
import os
from decimal import Decimal, getcontext

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
TOL = 1e-11


def _rng(seed):
    return np.random.default_rng(seed)


def _close(a, b, tol=TOL, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    fin = np.isfinite(b)
    assert np.array_equal(np.isfinite(a), fin), f"{what}: finiteness differs"
    assert np.array_equal(a[~fin], b[~fin]), f"{what}: non-finite values differ"
    err = np.max(np.abs(a[fin] - b[fin]) / (1.0 + np.abs(b[fin]))) if fin.any() else 0.0
    assert err <= tol, f"{what}: max rel err {err:.3e} > {tol:.1e}"


# --------------------------------------------------------------------------- closed forms

def pin_equal_scores_zero_query(attn):
    """Q = 0: every score is 0, so O is the plain mean of V and L = ln(kL)."""
    r = _rng(1)
    B, Hq, Hkv, qL, kL, D = 2, 4, 2, 6, 9, 5
    q = np.zeros((B, Hq, qL, D))
    k = r.standard_normal((B, Hkv, kL, D))
    v = r.standard_normal((B, Hkv, kL, D))
    o, lse = attn(q, k, v, 0.37)
    group = Hq // Hkv
    for b in range(B):
        for h in range(Hq):
            want = v[b, h // group].mean(axis=0)
            _close(o[b, h], np.broadcast_to(want, (qL, D)), what="O = mean(V)")
    _close(lse, np.full((B, Hq, qL), math.log(kL)), what="L = ln kL")


def pin_equal_scores_identical_keys(attn):
    """All keys equal: s_i is the same for every key, so O = mean(V), L = ln(kL) + s_i."""
    r = _rng(2)
    B, Hq, Hkv, qL, kL, D = 1, 3, 1, 5, 11, 4
    scale = 0.6
    q = r.standard_normal((B, Hq, qL, D))
    k0 = r.standard_normal((B, Hkv, 1, D))
    k = np.repeat(k0, kL, axis=2)
    v = r.standard_normal((B, Hkv, kL, D))
    o, lse = attn(q, k, v, scale)
    for h in range(Hq):
        s = scale * (q[0, h] @ k0[0, 0, 0])
        _close(lse[0, h], math.log(kL) + s, what="L = ln kL + s")
        _close(o[0, h], np.broadcast_to(v[0, 0].mean(axis=0), (qL, D)), what="O = mean(V)")


def pin_equal_scores_causal(attn):
    """Q = 0 with causal masking: O_i = mean(V[0..i]) and L_i = ln(i + 1)."""
    r = _rng(3)
    B, H, L, D = 1, 2, 7, 3
    q = np.zeros((B, H, L, D))
    k = r.standard_normal((B, H, L, D))
    v = r.standard_normal((B, H, L, D))
    o, lse = attn(q, k, v, 0.5, causal=True)
    n = np.arange(1, L + 1, dtype=np.float64)
    for h in range(H):
        _close(o[0, h], np.cumsum(v[0, h], axis=0) / n[:, None], what="causal prefix mean")
        _close(lse[0, h], np.log(n), what="causal L = ln(i+1)")


def _one_hot_targets(r, B, H, qL, kL):
    return r.integers(0, kL, size=(B, H, qL))


def pin_one_hot_bool(attn):
    """A bool mask keeping exactly one key j*: O_i = V[j*], L_i = scale * q_i . k_j*."""
    r = _rng(4)
    B, Hq, Hkv, L, D = 1, 2, 2, 6, 4
    scale = 0.45
    q = r.standard_normal((B, Hq, L, D))
    k = r.standard_normal((B, Hkv, L, D))
    v = r.standard_normal((B, Hkv, L, D))
    tgt = _one_hot_targets(r, B, Hq, L, L)
    mask = np.zeros((B, Hq, L, L), dtype=np.uint8)
    for h in range(Hq):
        for i in range(L):
            mask[0, h, i, tgt[0, h, i]] = 1
    o, lse = attn(q, k, v, scale, mask=mask, mask_kind=1)
    for h in range(Hq):
        for i in range(L):
            j = tgt[0, h, i]
            _close(o[0, h, i], v[0, h, j], what="one-hot O")
            _close(lse[0, h, i], scale * float(q[0, h, i] @ k[0, h, j]), what="one-hot L")


def pin_one_hot_additive(attn):
    """Additive mask: c_i at j*, -inf elsewhere: O_i = V[j*], L_i = scale*q_i.k_j* + c_i."""
    r = _rng(5)
    B, Hq, Hkv, L, D = 1, 2, 1, 5, 3
    scale = 0.3
    q = r.standard_normal((B, Hq, L, D))
    k = r.standard_normal((B, Hkv, L, D))
    v = r.standard_normal((B, Hkv, L, D))
    tgt = _one_hot_targets(r, B, Hq, L, L)
    c = r.standard_normal((B, Hq, L)) * 3.0
    mask = np.full((B, Hq, L, L), -np.inf)
    for h in range(Hq):
        for i in range(L):
            mask[0, h, i, tgt[0, h, i]] = c[0, h, i]
    o, lse = attn(q, k, v, scale, mask=mask, mask_kind=2)
    for h in range(Hq):
        for i in range(L):
            j = tgt[0, h, i]
            _close(o[0, h, i], v[0, 0, j], what="one-hot additive O")
            _close(lse[0, h, i], scale * float(q[0, h, i] @ k[0, 0, j]) + c[0, h, i],
                   what="one-hot additive L")


def pin_causal_row0(attn):
    """Causal row 0 sees only key 0: O_0 = V[0], L_0 = scale * q_0 . k_0."""
    r = _rng(6)
    B, Hq, Hkv, L, D = 2, 2, 1, 8, 6
    scale = 0.7
    q = r.standard_normal((B, Hq, L, D))
    k = r.standard_normal((B, Hkv, L, D))
    v = r.standard_normal((B, Hkv, L, D))
    o, lse = attn(q, k, v, scale, causal=True)
    for b in range(B):
        for h in range(Hq):
            _close(o[b, h, 0], v[b, 0, 0], what="causal row 0 O")
            _close(lse[b, h, 0], scale * float(q[b, h, 0] @ k[b, 0, 0]), what="causal row 0 L")


def pin_fully_masked_row(attn):
    """A row with no allowed key: O = 0 and L = -inf (the empty logsumexp)."""
    r = _rng(7)
    B, H, L, D = 1, 1, 4, 3
    q = r.standard_normal((B, H, L, D))
    k = r.standard_normal((B, H, L, D))
    v = r.standard_normal((B, H, L, D))
    mask = np.ones((B, H, L, L), dtype=np.uint8)
    mask[0, 0, 2, :] = 0
    o, lse = attn(q, k, v, 0.5, mask=mask, mask_kind=1)
    assert np.all(o[0, 0, 2] == 0.0), "masked row O must be 0"
    assert lse[0, 0, 2] == -np.inf, "masked row L must be -inf"
    assert np.all(np.isfinite(lse[0, 0, [0, 1, 3]]))


def pin_large_margin(attn):
    """q = t e0, k_j* = t e0, other keys 0: O -> V[j*] within (kL-1) e^(-scale t^2)."""
    r = _rng(8)
    B, H, qL, kL, D = 1, 1, 3, 10, 4
    t, scale, js = 6.0, 0.5, 7
    q = np.zeros((B, H, qL, D)); q[..., 0] = t
    k = np.zeros((B, H, kL, D)); k[0, 0, js, 0] = t
    v = r.standard_normal((B, H, kL, D))
    o, lse = attn(q, k, v, scale)
    bound = (kL - 1) * math.exp(-scale * t * t) * (np.abs(v).max() * 2)
    assert np.max(np.abs(o[0, 0] - v[0, 0, js])) <= bound
    _close(lse[0, 0], np.full(qL, scale * t * t + math.log1p((kL - 1) * math.exp(-scale * t * t))),
           what="large-margin L")


# --------------------------------------------------------------------------- golden file

def pin_golden_handworked(attn):
    """Hand-derived examples (tests/golden/handworked.json)."""
    with open(os.path.join(GOLDEN, "handworked.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        q = np.array(c["q"], dtype=np.float64)
        k = np.array(c["k"], dtype=np.float64)
        v = np.array(c["v"], dtype=np.float64)
        kw = {}
        if "mask" in c:
            m = np.array([[float(x) for x in row] for row in c["mask"]], dtype=np.float64)
            kw = dict(mask=m[None, None], mask_kind=c["mask_kind"])
        o, lse = attn(q[None, None], k[None, None], v[None, None], c["scale"],
                      causal=c.get("causal", False), **kw)
        want_o = np.array(c["O"], dtype=np.float64)
        want_l = np.array([float(x) for x in c["L"]], dtype=np.float64)
        _close(o[0, 0], want_o, tol=1e-12, what=c["name"] + " O")
        _close(lse[0, 0], want_l, tol=1e-12, what=c["name"] + " L")


# --------------------------------------------------------------------------- brute force

def _decimal_tanh(x):
    """tanh from its exponential definition, in the current Decimal context."""
    e = (2 * x).exp()
    return (e - 1) / (e + 1)


def _decimal_attention(q, k, v, scale, causal, mask, mask_kind, window=0, softcap=0.0, q_offset=0):
    getcontext().prec = 50
    B, Hq, qL, D = q.shape
    Hkv, kL = k.shape[1], k.shape[2]
    group = Hq // Hkv
    O = np.zeros((B, Hq, qL, D))
    L = np.zeros((B, Hq, qL))
    dscale = Decimal(float(scale))
    for b in range(B):
        for h in range(Hq):
            kh = h // group
            for i in range(qL):
                scores = []
                for j in range(kL):
                    dot = sum(Decimal(float(q[b, h, i, d])) * Decimal(float(k[b, kh, j, d]))
                              for d in range(D))
                    s = dscale * dot
                    if softcap > 0:
                        cap = Decimal(float(softcap))
                        s = cap * _decimal_tanh(s / cap)
                    ok = (not causal) or j <= i + q_offset
                    if window > 0:
                        ok = ok and j > i + q_offset - window
                    if mask_kind == 1:
                        ok = ok and mask[b, h, i, j] != 0
                    elif mask_kind == 2:
                        mv = float(mask[b, h, i, j])
                        if mv == -math.inf:
                            ok = False
                        else:
                            s = s + Decimal(mv)
                    if ok:
                        scores.append((j, s))
                if not scores:
                    L[b, h, i] = -math.inf
                    continue
                m = max(s for _, s in scores)
                w = [(j, (s - m).exp()) for j, s in scores]
                l = sum(x for _, x in w)
                for d in range(D):
                    O[b, h, i, d] = float(sum(x * Decimal(float(v[b, kh, j, d])) for j, x in w) / l)
                L[b, h, i] = float(m + l.ln())
    return O, L


def pin_bruteforce_decimal_window_softcap_offset(attn):
    """50-digit decimal brute force with a sliding window, a softcap and a query offset."""
    r = _rng(20)
    B, Hq, Hkv, qL, kL, D = 1, 2, 1, 5, 9, 3
    q = 2.0 * r.standard_normal((B, Hq, qL, D))
    k = 2.0 * r.standard_normal((B, Hkv, kL, D))
    v = r.standard_normal((B, Hkv, kL, D))
    amask = r.standard_normal((B, Hq, qL, kL))
    for causal, window, softcap, q_offset, kind in ((True, 3, 0.0, 0, 0), (True, 2, 0.0, 4, 0), (False, 4, 0.0, 2, 0),
                                                    (False, 0, 1.5, 0, 0), (True, 3, 2.0, 4, 2), (True, 0, 0.0, -2, 0)):
        m = amask if kind == 2 else None
        o, lse = attn(q, k, v, 0.7, causal=causal, mask=m, mask_kind=kind, window=window, softcap=softcap,
                      q_offset=q_offset)
        wo, wl = _decimal_attention(q, k, v, 0.7, causal, m, kind, window, softcap, q_offset)
        what = f"causal={causal} window={window} softcap={softcap} q_offset={q_offset} kind={kind}"
        _close(o, wo, what="decimal O " + what)
        _close(lse, wl, what="decimal L " + what)


def pin_window_of_one_key(attn):
    """Causal with window 1: row i sees only key i + q_offset, so O_i = V[i + q_offset], L_i = its score."""
    r = _rng(21)
    B, Hq, Hkv, qL, kL, D = 1, 2, 2, 6, 9, 4
    q, k, v = r.standard_normal((B, Hq, qL, D)), r.standard_normal((B, Hkv, kL, D)), r.standard_normal((B, Hkv, kL, D))
    for q_offset in (0, 3):
        o, lse = attn(q, k, v, 0.5, causal=True, window=1, q_offset=q_offset)
        for h in range(Hq):
            for i in range(qL):
                j = i + q_offset
                _close(o[0, h, i], v[0, h, j], what=f"window-1 O row {i}")
                _close(lse[0, h, i], 0.5 * float(q[0, h, i] @ k[0, h, j]), what=f"window-1 L row {i}")


def pin_window_equal_scores(attn):
    """Q = 0, causal, window W: O_i = mean of V over keys (i + q_offset - W, i + q_offset], L_i = ln(count)."""
    r = _rng(22)
    B, Hq, Hkv, qL, kL, D = 1, 2, 1, 7, 10, 3
    q = np.zeros((B, Hq, qL, D))
    k, v = r.standard_normal((B, Hkv, kL, D)), r.standard_normal((B, Hkv, kL, D))
    for W, q_offset in ((3, 0), (4, 3), (20, 2)):
        o, lse = attn(q, k, v, 0.9, causal=True, window=W, q_offset=q_offset)
        for i in range(qL):
            hi = min(i + q_offset, kL - 1)
            lo = max(0, i + q_offset - W + 1)
            _close(o[0, 0, i], v[0, 0, lo:hi + 1].mean(axis=0), what=f"window {W} O row {i}")
            _close(lse[0, 0, i], math.log(hi - lo + 1), what=f"window {W} L row {i}")


def pin_q_offset_is_a_suffix(attn):
    """Causal with q_offset = kL - qL (bottom-right) gives the last qL rows of the full causal problem."""
    r = _rng(23)
    B, Hq, Hkv, kL, D, qL = 1, 2, 1, 11, 4, 4
    k, v = r.standard_normal((B, Hkv, kL, D)), r.standard_normal((B, Hkv, kL, D))
    q_full = r.standard_normal((B, Hq, kL, D))
    for window in (0, 5):
        of, lf = attn(q_full, k, v, 0.6, causal=True, window=window)
        o, lse = attn(q_full[:, :, kL - qL:], k, v, 0.6, causal=True, window=window, q_offset=kL - qL)
        _close(o, of[:, :, kL - qL:], 0.0, "suffix O")
        _close(lse, lf[:, :, kL - qL:], 0.0, "suffix L")


def pin_softcap_large_cap(attn):
    """softcap c -> infinity recovers the plain scores: c * tanh(s / c) = s - s^3 / (3 c^2) + ..."""
    r = _rng(24)
    B, Hq, Hkv, qL, kL, D = 1, 2, 2, 5, 8, 4
    q, k, v = r.standard_normal((B, Hq, qL, D)), r.standard_normal((B, Hkv, kL, D)), r.standard_normal((B, Hkv, kL, D))
    o0, l0 = attn(q, k, v, 0.5, causal=True)
    o1, l1 = attn(q, k, v, 0.5, causal=True, softcap=1e6)
    _close(o1, o0, 1e-9, "softcap 1e6 O")
    _close(l1, l0, 1e-9, "softcap 1e6 L")


# --------------------------------------------------------------------------- dropout

def _dropout_inputs(seed):
    r = _rng(seed)
    B, Hq, Hkv, qL, kL, D = 1, 2, 1, 6, 12, 4
    return (r.standard_normal((B, Hq, qL, D)), r.standard_normal((B, Hkv, kL, D)),
            r.standard_normal((B, Hkv, kL, D)))


def pin_dropout_p0_and_p1(attn):
    """p = 0 is the plain forward bit for bit; p = 1 drops every weight (O = 0) and leaves L alone."""
    q, k, v = _dropout_inputs(30)
    o0, l0 = attn(q, k, v, 0.5, causal=True)
    o1, l1 = attn(q, k, v, 0.5, causal=True, dropout_p=0.0, seed=99, offset=5)
    _close(o1, o0, 0.0, "p=0 O")
    _close(l1, l0, 0.0, "p=0 L")
    o2, l2 = attn(q, k, v, 0.5, causal=True, dropout_p=1.0, seed=99, offset=5)
    assert np.all(o2 == 0.0), "p=1 must drop every weight"
    _close(l2, l0, 0.0, "p=1 L")


def pin_dropout_keep_rate(lib=None):
    """The generator keeps a fraction 1 - p of positions (binomial bounds) with multipliers {0, 1/(1-p)}."""
    import oracle
    for p, seed, offset in ((0.2, 7, 0), (0.65, 2 ** 40 + 3, 2 ** 33 - 5)):
        n = 400_000
        keep = oracle.dropout_keep(p, seed, offset, 12345, n, lib=lib)
        assert set(np.unique(keep)) <= {0.0, 1.0 / (1.0 - p)}, "multipliers must be 0 or 1/(1-p)"
        frac = float(np.mean(keep > 0))
        sd = math.sqrt(p * (1 - p) / n)
        assert abs(frac - (1 - p)) < 6 * sd, f"keep rate {frac:.5f} for p={p}"


def _triton_philox_words(seeds, offsets):
    """Philox4x32-10 words from Triton's generator on the CPU (its interpreter), in a child process."""
    import subprocess
    import sys
    try:
        import triton  # noqa: F401
    except ImportError:
        import pytest
        pytest.skip("triton is not installed: no independent Philox at hand")
    script = os.path.join(os.path.dirname(os.path.abspath(__file__)), "philox_triton_words.py")
    req = json.dumps({"seeds": [str(s) for s in seeds], "offsets": [str(o) for o in offsets]})
    res = subprocess.run([sys.executable, script, req], capture_output=True, text=True, timeout=600,
                         env=dict(os.environ, TRITON_INTERPRET="1"))
    assert res.returncode == 0, res.stderr[-2000:]
    return json.loads(res.stdout.strip().splitlines()[-1])


def pin_philox_matches_triton(lib=None):
    """The oracle's Philox4x32-10 block equals Triton's, word for word, and its dropout multipliers are
    the contract's decision on those words: word (position mod 4) of the block at counter
    offset + position / 4 (64-bit, carry into the high word), kept iff (word >> 8) / 2^24 >= p."""
    import oracle
    M64 = (1 << 64) - 1
    seeds = [0, 1, 0x1234567890ABCDEF, M64, 2 ** 40 + 3]
    offsets = [0, 1, 2, 3, 2 ** 31, 2 ** 32 - 1, 2 ** 32, 2 ** 32 + 1, 2 ** 33 - 5, 0xDEADBEEFCAFEF00D, M64 - 1, M64]
    words = _triton_philox_words(seeds, offsets)
    for seed, per_seed in zip(seeds, words):
        for off, ref in zip(offsets, per_seed):
            got = oracle.philox4x32_10([off & 0xFFFFFFFF, off >> 32, 0, 0], (seed & 0xFFFFFFFF, seed >> 32), lib=lib)
            assert [int(x) for x in got] == ref, f"Philox block differs at seed {seed:#x}, counter {off:#x}"
    # the decision chain: position -> counter and word, threshold, multiplier
    for p, seed, offset, first in ((0.3, 0x1234567890ABCDEF, 2 ** 32 - 3, 5), (0.85, 7, M64 - 2, 0)):
        n = 40
        blocks = sorted({(offset + (first + t) // 4) & M64 for t in range(n)})
        bw = dict(zip(blocks, _triton_philox_words([seed], blocks)[0]))
        keep = oracle.dropout_keep(p, seed, offset, first, n, lib=lib)
        for t in range(n):
            pos = first + t
            word = bw[(offset + pos // 4) & M64][pos % 4]
            want = 1.0 / (1.0 - p) if (word >> 8) / 16777216.0 >= p else 0.0
            assert keep[t] == want, f"multiplier at position {pos}: {keep[t]} vs {want}"


def pin_dropout_unbiased(attn):
    """Averaged over many seeds, the dropped-out O converges to the plain O (the 1/(1-p) rescale)."""
    q, k, v = _dropout_inputs(31)
    o0, _ = attn(q, k, v, 0.5, causal=True)
    samples = np.stack([attn(q, k, v, 0.5, causal=True, dropout_p=0.3, seed=1000 + t)[0] for t in range(400)])
    mean, sd = samples.mean(axis=0), samples.std(axis=0) / math.sqrt(len(samples))
    assert np.all(np.abs(mean - o0) <= 6 * sd + 1e-12), "dropout is biased"


def pin_dropout_position_map(attn):
    """O rebuilt from the plain softmax weights and the generator at position ((b H_q + h) qL + i) kL + j."""
    import oracle
    q, k, v = _dropout_inputs(32)
    B, Hq, qL, D = q.shape
    kL = k.shape[2]
    scale, p, seed, offset = 0.5, 0.4, 77, 2 ** 35 + 1
    o, lse = attn(q, k, v, scale, causal=False, dropout_p=p, seed=seed, offset=offset)
    group = Hq // k.shape[1]
    for h in range(Hq):
        sc = scale * q[0, h] @ k[0, h // group].T
        w = np.exp(sc - sc.max(axis=1, keepdims=True))
        w /= w.sum(axis=1, keepdims=True)
        for i in range(qL):
            keep = oracle.dropout_keep(p, seed, offset, ((0 * Hq + h) * qL + i) * kL, kL)
            _close(o[0, h, i], (w[i] * keep) @ v[0, h // group], 1e-12, f"dropout row {h},{i}")


def pin_bruteforce_decimal(attn):
    """50-digit decimal brute force on tiny inputs, every feature switched on in turn."""
    r = _rng(9)
    B, Hq, Hkv, qL, kL, D = 1, 2, 1, 5, 7, 3
    q = r.standard_normal((B, Hq, qL, D))
    k = r.standard_normal((B, Hkv, kL, D))
    v = r.standard_normal((B, Hkv, kL, D))
    bmask = (r.random((B, Hq, qL, kL)) < 0.7).astype(np.uint8)
    bmask[..., 0] = 1
    amask = r.standard_normal((B, Hq, qL, kL))
    amask[r.random((B, Hq, qL, kL)) < 0.2] = -np.inf
    amask[..., 0] = 0.25
    for causal in (False, True):
        for kind, m in ((0, None), (1, bmask), (2, amask)):
            o, lse = attn(q, k, v, 0.55, causal=causal, mask=m, mask_kind=kind)
            wo, wl = _decimal_attention(q, k, v, 0.55, causal, m, kind)
            _close(o, wo, what=f"decimal O causal={causal} kind={kind}")
            _close(lse, wl, what=f"decimal L causal={causal} kind={kind}")


# --------------------------------------------------------------------------- library cross-check

def _float_mask(qL, kL, causal, mask, mask_kind, B, Hq):
    fm = torch.zeros((B, Hq, qL, kL), dtype=torch.float64)
    if causal:
        fm = fm.masked_fill(~torch.ones(qL, kL, dtype=torch.bool).tril(), float("-inf"))
    if mask_kind == 1:
        fm = fm.masked_fill(torch.from_numpy(np.asarray(mask)) == 0, float("-inf"))
    elif mask_kind == 2:
        fm = fm + torch.from_numpy(np.asarray(mask, dtype=np.float64))
    return fm


def pin_torch_sdpa(attn):
    """torch fp64 CPU scaled_dot_product_attention with K/V repeated per GQA group."""
    r = _rng(10)
    B, Hq, Hkv, qL, kL, D = 2, 4, 2, 37, 53, 16
    scale = 0.21
    q = r.standard_normal((B, Hq, qL, D))
    k = r.standard_normal((B, Hkv, kL, D))
    v = r.standard_normal((B, Hkv, kL, D))
    bmask = (r.random((B, Hq, qL, kL)) < 0.8).astype(np.uint8)
    bmask[..., 0] = 1
    amask = r.standard_normal((B, Hq, qL, kL))
    amask[r.random((B, Hq, qL, kL)) < 0.15] = -np.inf
    amask[..., 0] = 0.0
    tq = torch.from_numpy(q)
    tk = torch.from_numpy(k).repeat_interleave(Hq // Hkv, dim=1)
    tv = torch.from_numpy(v).repeat_interleave(Hq // Hkv, dim=1)
    for causal in (False, True):
        for kind, m in ((0, None), (1, bmask), (2, amask)):
            fm = _float_mask(qL, kL, causal, m, kind, B, Hq)
            want_o = torch.nn.functional.scaled_dot_product_attention(
                tq, tk, tv, attn_mask=fm, scale=scale).numpy()
            want_l = torch.logsumexp(torch.matmul(tq, tk.transpose(-1, -2)) * scale + fm, dim=-1).numpy()
            o, lse = attn(q, k, v, scale, causal=causal, mask=m, mask_kind=kind)
            _close(o, want_o, tol=1e-10, what=f"sdpa O causal={causal} kind={kind}")
            _close(lse, want_l, tol=1e-10, what=f"sdpa L causal={causal} kind={kind}")


# --------------------------------------------------------------------------- invariants

def pin_key_permutation(attn):
    """Non-causal: permuting keys (and the mask's key axis with them) changes nothing."""
    r = _rng(11)
    B, H, qL, kL, D = 1, 2, 5, 9, 4
    q = r.standard_normal((B, H, qL, D))
    k = r.standard_normal((B, H, kL, D))
    v = r.standard_normal((B, H, kL, D))
    am = r.standard_normal((B, H, qL, kL))
    perm = r.permutation(kL)
    o1, l1 = attn(q, k, v, 0.4, mask=am, mask_kind=2)
    o2, l2 = attn(q, k[:, :, perm], v[:, :, perm], 0.4, mask=am[..., perm], mask_kind=2)
    _close(o2, o1, what="permuted O")
    _close(l2, l1, what="permuted L")


def pin_additive_shift(attn):
    """Adding c to every additive-mask entry leaves O unchanged and shifts L by c."""
    r = _rng(12)
    B, H, L, D = 1, 2, 6, 4
    q = r.standard_normal((B, H, L, D))
    k = r.standard_normal((B, H, L, D))
    v = r.standard_normal((B, H, L, D))
    am = r.standard_normal((B, H, L, L))
    c = 1.75
    o1, l1 = attn(q, k, v, 0.8, causal=True, mask=am, mask_kind=2)
    o2, l2 = attn(q, k, v, 0.8, causal=True, mask=am + c, mask_kind=2)
    _close(o2, o1, what="shifted O")
    _close(l2, l1 + c, what="shifted L")


def pin_linear_in_v(attn):
    """O is linear in V, and V = 1 gives O = 1."""
    r = _rng(13)
    B, Hq, Hkv, L, D = 1, 4, 2, 7, 5
    q = r.standard_normal((B, Hq, L, D))
    k = r.standard_normal((B, Hkv, L, D))
    v1 = r.standard_normal((B, Hkv, L, D))
    v2 = r.standard_normal((B, Hkv, L, D))
    a, b = 0.7, -1.3
    o1, _ = attn(q, k, v1, 0.5, causal=True)
    o2, _ = attn(q, k, v2, 0.5, causal=True)
    o3, _ = attn(q, k, a * v1 + b * v2, 0.5, causal=True)
    _close(o3, a * o1 + b * o2, tol=1e-10, what="linearity")
    o4, _ = attn(q, k, np.ones_like(v1), 0.5, causal=True)
    _close(o4, np.ones_like(o4), what="V = 1")


def pin_gqa_equals_repeated_mha(attn):
    """GQA with H_kv heads equals MHA on K/V repeated H_q/H_kv times per head."""
    r = _rng(14)
    B, Hq, Hkv, L, D = 2, 6, 2, 5, 3
    q = r.standard_normal((B, Hq, L, D))
    k = r.standard_normal((B, Hkv, L, D))
    v = r.standard_normal((B, Hkv, L, D))
    o1, l1 = attn(q, k, v, 0.6, causal=True)
    o2, l2 = attn(q, np.repeat(k, Hq // Hkv, axis=1), np.repeat(v, Hq // Hkv, axis=1), 0.6, causal=True)
    _close(o1, o2, what="GQA O")
    _close(l1, l2, what="GQA L")


def pin_mask_kind_equivalences(attn):
    """bool all-true = additive all-zero = no mask; bool tril = additive -inf upper = causal."""
    r = _rng(15)
    B, H, L, D = 1, 2, 6, 4
    q = r.standard_normal((B, H, L, D))
    k = r.standard_normal((B, H, L, D))
    v = r.standard_normal((B, H, L, D))
    o0, l0 = attn(q, k, v, 0.5)
    o1, l1 = attn(q, k, v, 0.5, mask=np.ones((B, H, L, L), np.uint8), mask_kind=1)
    o2, l2 = attn(q, k, v, 0.5, mask=np.zeros((B, H, L, L)), mask_kind=2)
    for o, l in ((o1, l1), (o2, l2)):
        _close(o, o0, what="all-keep O"); _close(l, l0, what="all-keep L")
    tril = np.tril(np.ones((L, L), np.uint8))
    oc, lc = attn(q, k, v, 0.5, causal=True)
    ob, lb = attn(q, k, v, 0.5, mask=np.broadcast_to(tril, (B, H, L, L)), mask_kind=1)
    oa, la = attn(q, k, v, 0.5, mask=np.broadcast_to(np.where(tril == 1, 0.0, -np.inf), (B, H, L, L)),
                  mask_kind=2)
    for o, l in ((ob, lb), (oa, la)):
        _close(o, oc, what="tril O"); _close(l, lc, what="tril L")


def pin_rows_subset(attn):
    """The row-subset mode returns exactly the rows of a full run."""
    r = _rng(16)
    B, Hq, Hkv, qL, kL, D = 2, 2, 1, 9, 12, 4
    q = r.standard_normal((B, Hq, qL, D))
    k = r.standard_normal((B, Hkv, kL, D))
    v = r.standard_normal((B, Hkv, kL, D))
    o, lse = attn(q, k, v, 0.5, causal=True)
    rows = [0, 5, 17, 35, 3]
    os_, ls_ = attn(q, k, v, 0.5, causal=True, rows=rows)
    _close(os_, o.reshape(-1, D)[rows], tol=0.0, what="row subset O")
    _close(ls_, lse.reshape(-1)[rows], tol=0.0, what="row subset L")


ALL_PINS = [
    pin_equal_scores_zero_query, pin_equal_scores_identical_keys, pin_equal_scores_causal,
    pin_one_hot_bool, pin_one_hot_additive, pin_causal_row0, pin_fully_masked_row,
    pin_large_margin, pin_golden_handworked, pin_bruteforce_decimal, pin_torch_sdpa,
    pin_key_permutation, pin_additive_shift, pin_linear_in_v, pin_gqa_equals_repeated_mha,
    pin_mask_kind_equivalences, pin_rows_subset, pin_bruteforce_decimal_window_softcap_offset,
    pin_window_of_one_key, pin_window_equal_scores, pin_q_offset_is_a_suffix, pin_softcap_large_cap,
    pin_dropout_p0_and_p1, pin_dropout_unbiased, pin_dropout_position_map,
]
# Pins of the generator alone (no attention callable).
GENERATOR_PINS = [pin_dropout_keep_rate, pin_philox_matches_triton]
