"""fp64 CPU oracle for the attention forward pass -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never does, and this
package imports nothing from the library: the two share no code.

The arithmetic lives in ``attn_oracle.c`` (the forward: plain C, fp64, one
score row at a time, full-row softmax) and ``attn_oracle_bwd.c`` (its
gradients, written out from the chain rule through the softmax).  This module builds it with the host C compiler,
loads it with ctypes and marshals numpy arrays.  See the C file's header for
the definition and the page sections it follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_SRC_BWD = os.path.join(_HERE, "attn_oracle_bwd.c")
_LIB_BWD_PATH = os.path.join(_HERE, "liboracle_bwd.so")
_lib = None
_lib_bwd = None


def _compile(src: str, default_path: str, tag: str, mutant: int, out_path: str | None) -> str:
    if out_path is None:
        out_path = default_path if mutant == 0 else os.path.join(
            tempfile.mkdtemp(prefix="oracle_mut"), f"lib{tag}_m{mutant}.so")
    tmp = out_path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-pthread",
           "-fno-fast-math", f"-DORACLE_MUTANT={int(mutant)}", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out_path)
    return out_path


def build(mutant: int = 0, out_path: str | None = None) -> str:
    """Compile the forward oracle (or a variant with a planted mistake) to a shared object.

    ``mutant`` 0 is the oracle itself; 1..8 each plant one known mistake and
    exist only so the tests can show that the pins catch it.
    """
    return _compile(_SRC, _LIB_PATH, "oracle", mutant, out_path)


def build_bwd(mutant: int = 0, out_path: str | None = None) -> str:
    """Compile the gradient oracle (or a variant with planted mistake 1..10)."""
    return _compile(_SRC_BWD, _LIB_BWD_PATH, "oracle_bwd", mutant, out_path)


def _bind(lib):
    f = lib.oracle_attention_ex
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int] + [ctypes.c_void_p] * 2 + \
        [ctypes.c_longlong] * 6 + [ctypes.c_double, ctypes.c_int, ctypes.c_longlong, ctypes.c_double,
                                   ctypes.c_longlong, ctypes.c_double, ctypes.c_uint64, ctypes.c_uint64,
                                   ctypes.c_void_p, ctypes.c_longlong, ctypes.c_int]
    g = lib.oracle_dropout_keep
    g.restype = ctypes.c_int
    g.argtypes = [ctypes.c_double, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint64, ctypes.c_longlong,
                  ctypes.c_void_p]
    g = lib.oracle_philox4x32_10
    g.restype = ctypes.c_int
    g.argtypes = [ctypes.c_void_p, ctypes.c_uint32, ctypes.c_uint32, ctypes.c_void_p]
    lib.oracle_mutant_id.restype = ctypes.c_int
    return lib


def load(path: str | None = None):
    """Load the oracle shared object (building it first if it is missing or stale)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        if (not os.path.exists(_LIB_PATH)
                or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
            build()
        _lib = _bind(ctypes.CDLL(_LIB_PATH))
    return _lib


def _bind_bwd(lib):
    f = lib.oracle_attention_bwd
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int] + [ctypes.c_void_p] * 4 + \
        [ctypes.c_longlong] * 6 + [ctypes.c_double, ctypes.c_int, ctypes.c_int]
    f = lib.oracle_attention_bwd_ex
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_int] + [ctypes.c_void_p] * 4 + \
        [ctypes.c_longlong] * 6 + [ctypes.c_double, ctypes.c_int, ctypes.c_longlong, ctypes.c_longlong, ctypes.c_double,
                                   ctypes.c_void_p, ctypes.c_int]
    lib.oracle_bwd_mutant_id.restype = ctypes.c_int
    return lib


def load_bwd(path: str | None = None):
    """Load the gradient oracle (building it first if it is missing or stale)."""
    global _lib_bwd
    if path is not None:
        return _bind_bwd(ctypes.CDLL(path))
    if _lib_bwd is None:
        if (not os.path.exists(_LIB_BWD_PATH)
                or os.path.getmtime(_LIB_BWD_PATH) < os.path.getmtime(_SRC_BWD)):
            build_bwd()
        _lib_bwd = _bind_bwd(ctypes.CDLL(_LIB_BWD_PATH))
    return _lib_bwd


def _mask_arg(mask, mask_kind, shape):
    if mask_kind == 1:
        m = np.ascontiguousarray(np.broadcast_to(np.asarray(mask) != 0, shape).astype(np.uint8))
        return m, m.ctypes.data
    if mask_kind == 2:
        m = _f64(np.broadcast_to(np.asarray(mask, dtype=np.float64), shape))
        return m, m.ctypes.data
    if mask_kind != 0:
        raise ValueError("mask_kind must be 0, 1 or 2")
    return None, None


def attention_bwd(q, k, v, dO, scale: float, causal: bool = False, mask=None,
                  mask_kind: int = 0, n_threads: int | None = None, lib=None, window: int = 0, q_offset: int = 0,
                  softcap: float = 0.0, dropout_p: float = 0.0, seed: int = 0, offset: int = 0, keep=None):
    """dQ, dK, dV of sum(O * dO) for O = softmax(scale * q k^T + mask) v, in fp64.

    Shapes and mask conventions as ``attention``; dO has the shape of q.
    window / q_offset / softcap: the forward's sliding window, causal diagonal offset and softcap.
    dropout_p / seed / offset: the forward's dropout; its multipliers come from the forward
    oracle's generator (``dropout_keep``) and enter the gradient oracle as an input.
    keep: instead, the multipliers themselves ([B, H_q, qL, kL] fp64), e.g. those of a slice of
    a larger problem, whose generator positions are not this call's.
    Returns (dQ [B,H_q,qL,D], dK [B,H_kv,kL,D], dV [B,H_kv,kL,D]).
    """
    lib = lib or load_bwd()
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    B, Hq, qL, D = q.shape
    Bk, Hkv, kL, Dk = k.shape
    if (Bk, Dk) != (B, D) or v.shape != k.shape or dO.shape != q.shape:
        raise ValueError("shape mismatch between q, k, v and dO")
    mask_arr, mptr = _mask_arg(mask, mask_kind, (B, Hq, qL, kL))  # held until the call returns
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    if n_threads is None:
        n_threads = os.cpu_count() or 1
    if keep is not None:
        keep = _f64(keep)
        if keep.shape != (B, Hq, qL, kL):
            raise ValueError("keep must be [B, H_q, qL, kL]")
    elif dropout_p > 0.0:
        keep = np.ascontiguousarray(dropout_keep(dropout_p, seed, offset, 0, B * Hq * qL * kL))
    kptr = None if keep is None else keep.ctypes.data
    rc = lib.oracle_attention_bwd_ex(q.ctypes.data, k.ctypes.data, v.ctypes.data, mptr, int(mask_kind),
                                     dO.ctypes.data, dq.ctypes.data, dk.ctypes.data, dv.ctypes.data,
                                     B, Hq, Hkv, qL, kL, D, float(scale), int(bool(causal)), int(window),
                                     int(q_offset), float(softcap), kptr, int(n_threads))
    del keep, mask_arr
    if rc != 0:
        raise ValueError("oracle_attention_bwd rejected its arguments")
    return dq, dk, dv


def _f64(a) -> np.ndarray:
    a = np.asarray(a, dtype=np.float64)
    return np.ascontiguousarray(a)


def attention(q, k, v, scale: float, causal: bool = False, mask=None,
              mask_kind: int = 0, rows=None, n_threads: int | None = None,
              lib=None, window: int = 0, softcap: float = 0.0, q_offset: int = 0,
              dropout_p: float = 0.0, seed: int = 0, offset: int = 0):
    """O and L of softmax(scale * q k^T + mask) v in fp64.

    q: [B, H_q, qL, D]; k, v: [B, H_kv, kL, D] (any real dtype; widened to
    fp64 exactly).  mask: None, or [B, H_q, qL, kL] -- bool/uint8 with
    nonzero = keep (mask_kind 1) or additive real values (mask_kind 2).
    ``scale`` is used as given (pass the fp32-rounded value the GPU sees).
    window > 0 keeps keys j > i + q_offset - window; softcap > 0 maps each
    scaled score s to softcap * tanh(s / softcap) before the mask; q_offset
    shifts the causal diagonal (j <= i + q_offset).  dropout_p > 0 scales each
    weight of O by keep in {0, 1 / (1 - p)} from the counter-based generator
    keyed by seed at counter offset + position / 4; L is unchanged.
    rows: optional iterable of flat row indices (b*H_q + h)*qL + i.
    Returns (O, L): O [B,H_q,qL,D] and L [B,H_q,qL], or [n,D] and [n] for rows.
    """
    lib = lib or load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, Hq, qL, D = q.shape
    Bk, Hkv, kL, Dk = k.shape
    if (Bk, Dk) != (B, D) or v.shape != k.shape:
        raise ValueError("shape mismatch between q, k and v")
    mptr = None
    if mask_kind == 1:
        mask = np.ascontiguousarray(np.broadcast_to(np.asarray(mask) != 0, (B, Hq, qL, kL)).astype(np.uint8))
        mptr = mask.ctypes.data
    elif mask_kind == 2:
        mask = _f64(np.broadcast_to(np.asarray(mask, dtype=np.float64), (B, Hq, qL, kL)))
        mptr = mask.ctypes.data
    elif mask_kind != 0:
        raise ValueError("mask_kind must be 0, 1 or 2")
    if rows is not None:
        rows_arr = np.ascontiguousarray(np.asarray(list(rows), dtype=np.int64))
        n = int(rows_arr.size)
        o = np.empty((n, D), dtype=np.float64)
        lse = np.empty((n,), dtype=np.float64)
        rptr = rows_arr.ctypes.data
    else:
        rows_arr = None
        n = 0
        o = np.empty((B, Hq, qL, D), dtype=np.float64)
        lse = np.empty((B, Hq, qL), dtype=np.float64)
        rptr = None
    if n_threads is None:
        n_threads = os.cpu_count() or 1
    rc = lib.oracle_attention_ex(q.ctypes.data, k.ctypes.data, v.ctypes.data, mptr,
                                 int(mask_kind), o.ctypes.data, lse.ctypes.data,
                                 B, Hq, Hkv, qL, kL, D, float(scale), int(bool(causal)),
                                 int(window), float(softcap), int(q_offset), float(dropout_p), int(seed),
                                 int(offset), rptr, n, int(n_threads))
    if rc != 0:
        raise ValueError("oracle_attention rejected its arguments")
    return o, lse


def philox4x32_10(counter, key, lib=None):
    """The four output words of one Philox4x32-10 block (counter: 4 words, key: 2 words)."""
    lib = lib or load()
    ctr = np.ascontiguousarray(counter, dtype=np.uint32)
    assert ctr.shape == (4,)
    out = np.empty(4, dtype=np.uint32)
    lib.oracle_philox4x32_10(ctr.ctypes.data, int(key[0]) & 0xFFFFFFFF, int(key[1]) & 0xFFFFFFFF, out.ctypes.data)
    return out


def dropout_keep(p: float, seed: int, offset: int, first: int, n: int, lib=None):
    """The generator's multipliers (1 / (1 - p) or 0) of n consecutive positions from `first`."""
    lib = lib or load()
    out = np.empty(n, dtype=np.float64)
    lib.oracle_dropout_keep(float(p), int(seed), int(offset), int(first), int(n), out.ctypes.data)
    return out
