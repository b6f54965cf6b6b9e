"""ctypes binding of the C ABI in ``include/fa.h`` (argument marshalling only).

``fa_fwd``, ``fa_fwd_ex``, ``fa_bwd``, ``fa_bwd_workspace_bytes``,
``fa_last_error``, ``fa_sync_status``, ``fa_set_timeout_cycles``,
``fa_set_max_ctas`` and ``fa_version`` mirror the C entry points one to one
and take raw device pointers (ints).  ``attention`` and ``attention_bwd`` are
convenience wrappers for torch CUDA tensors: they check device, dtype, shape
and strides (the buffer checks of mlx-native "ops/flash_attn_train.rs",
`validate_buffer_size`), allocate outputs (and the backward's workspace) if
none are given and call the C ABI on the current torch stream.  Every step of the computation
runs in the CUDA library; there is no fallback.
"""
from __future__ import annotations

import ctypes
import math
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfa_gb300.so")

FA_DTYPE_F32, FA_DTYPE_BF16, FA_DTYPE_F16 = 0, 1, 2
FA_MASK_NONE, FA_MASK_BOOL, FA_MASK_ADDITIVE = 0, 1, 2
FA_OK, FA_ERR_INVALID_ARGUMENT, FA_ERR_UNSUPPORTED, FA_ERR_MISALIGNED, FA_ERR_CUDA, FA_ERR_DEVICE_TIMEOUT = range(6)
STATUS_NAMES = {0: "FA_OK", 1: "FA_ERR_INVALID_ARGUMENT", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_MISALIGNED",
                4: "FA_ERR_CUDA", 5: "FA_ERR_DEVICE_TIMEOUT"}

EXPORTED = ("fa_fwd", "fa_fwd_ex", "fa_fwd_workspace_bytes", "fa_last_error", "fa_sync_status",
            "fa_set_timeout_cycles", "fa_set_max_ctas", "fa_set_q_tiles", "fa_set_kv_splits", "fa_bwd_workspace_bytes",
            "fa_bwd_ex_workspace_bytes", "fa_bwd", "fa_bwd_ex", "fa_bwd_full", "fa_bwd_full_workspace_bytes",
            "fa_bwd_noalloc", "fa_version")


class FaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status
        self.message = message


class FaFwdArgs(ctypes.Structure):
    """Layout of ``fa_fwd_args`` in include/fa.h."""
    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
        ("o", ctypes.c_void_p), ("lse", ctypes.c_void_p), ("mask", ctypes.c_void_p),
        ("B", ctypes.c_int), ("H_q", ctypes.c_int), ("H_kv", ctypes.c_int),
        ("qL", ctypes.c_int), ("kL", ctypes.c_int), ("D", ctypes.c_int),
        ("scale", ctypes.c_float), ("causal", ctypes.c_int), ("mask_kind", ctypes.c_int),
        ("dtype", ctypes.c_int),
        ("q_strides", ctypes.c_longlong * 3), ("k_strides", ctypes.c_longlong * 3),
        ("v_strides", ctypes.c_longlong * 3), ("o_strides", ctypes.c_longlong * 3),
        ("mask_strides", ctypes.c_longlong * 3),
        ("stream", ctypes.c_void_p),
        ("window", ctypes.c_int), ("q_offset", ctypes.c_int), ("softcap", ctypes.c_float),
        ("dropout_p", ctypes.c_float), ("dropout_seed", ctypes.c_ulonglong), ("dropout_offset", ctypes.c_ulonglong),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_longlong),
    ]


class FaBwdArgs(ctypes.Structure):
    """Layout of ``fa_bwd_args`` in include/fa.h."""
    _fields_ = [
        ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("o", ctypes.c_void_p),
        ("dout", ctypes.c_void_p), ("lse", ctypes.c_void_p),
        ("dq", ctypes.c_void_p), ("dk", ctypes.c_void_p), ("dv", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_longlong),
        ("B", ctypes.c_int), ("H_q", ctypes.c_int), ("H_kv", ctypes.c_int),
        ("qL", ctypes.c_int), ("kL", ctypes.c_int), ("D", ctypes.c_int),
        ("scale", ctypes.c_float), ("causal", ctypes.c_int),
        ("window", ctypes.c_int), ("q_offset", ctypes.c_int), ("softcap", ctypes.c_float),
        ("dropout_p", ctypes.c_float), ("dropout_seed", ctypes.c_ulonglong), ("dropout_offset", ctypes.c_ulonglong),
        ("mask", ctypes.c_void_p), ("mask_kind", ctypes.c_int), ("mask_strides", ctypes.c_longlong * 3),
        ("dtype", ctypes.c_int), ("stream", ctypes.c_void_p),
    ]


_lib = None


def load_library(path: str = LIB_PATH):
    """Load ``libfa_gb300.so``; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build the CUDA library first "
                          f"(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    lib.fa_fwd.restype = ctypes.c_int
    lib.fa_fwd.argtypes = [ctypes.c_void_p] * 4 + [ctypes.c_void_p] + [ctypes.c_int] * 6 + \
        [ctypes.c_float, ctypes.c_int, ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    lib.fa_fwd_ex.restype = ctypes.c_int
    lib.fa_fwd_ex.argtypes = [ctypes.POINTER(FaFwdArgs)]
    lib.fa_fwd_workspace_bytes.restype = ctypes.c_longlong
    lib.fa_fwd_workspace_bytes.argtypes = [ctypes.POINTER(FaFwdArgs)]
    lib.fa_last_error.restype = ctypes.c_char_p
    lib.fa_last_error.argtypes = []
    lib.fa_sync_status.restype = ctypes.c_int
    lib.fa_sync_status.argtypes = [ctypes.c_void_p]
    lib.fa_set_timeout_cycles.restype = None
    lib.fa_set_timeout_cycles.argtypes = [ctypes.c_longlong]
    lib.fa_set_max_ctas.restype = None
    lib.fa_set_max_ctas.argtypes = [ctypes.c_int]
    lib.fa_set_q_tiles.restype = None
    lib.fa_set_q_tiles.argtypes = [ctypes.c_int]
    lib.fa_set_kv_splits.restype = None
    lib.fa_set_kv_splits.argtypes = [ctypes.c_int]
    lib.fa_version.restype = ctypes.c_int
    lib.fa_version.argtypes = []
    lib.fa_bwd_workspace_bytes.restype = ctypes.c_longlong
    lib.fa_bwd_workspace_bytes.argtypes = [ctypes.c_int] * 3
    lib.fa_bwd_ex_workspace_bytes.restype = ctypes.c_longlong
    lib.fa_bwd_ex_workspace_bytes.argtypes = [ctypes.c_int] * 4 + [ctypes.c_float]
    lib.fa_bwd.restype = ctypes.c_int
    lib.fa_bwd.argtypes = [ctypes.c_void_p] * 10 + [ctypes.c_longlong] + [ctypes.c_int] * 6 + \
        [ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    lib.fa_bwd_ex.restype = ctypes.c_int
    lib.fa_bwd_ex.argtypes = [ctypes.c_void_p] * 10 + [ctypes.c_longlong] + [ctypes.c_int] * 6 + \
        [ctypes.c_float] + [ctypes.c_int] * 3 + [ctypes.c_float, ctypes.c_float, ctypes.c_ulonglong,
                                                 ctypes.c_ulonglong, ctypes.c_int, ctypes.c_void_p]
    lib.fa_bwd_full.restype = ctypes.c_int
    lib.fa_bwd_full.argtypes = [ctypes.POINTER(FaBwdArgs)]
    lib.fa_bwd_full_workspace_bytes.restype = ctypes.c_longlong
    lib.fa_bwd_full_workspace_bytes.argtypes = [ctypes.POINTER(FaBwdArgs)]
    lib.fa_bwd_noalloc.restype = ctypes.c_int
    lib.fa_bwd_noalloc.argtypes = [ctypes.c_void_p] * 9 + [ctypes.c_int] * 6 + \
        [ctypes.c_float, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
    _lib = lib
    return lib


def _check(rc: int) -> int:
    if rc != FA_OK:
        raise FaError(rc, fa_last_error())
    return rc


# ----------------------------------------------------------------- raw C entry points

def fa_fwd(q, k, v, o, lse, B, H_q, H_kv, qL, kL, D, scale, causal, mask, mask_kind, dtype, stream):
    """``fa_fwd`` of include/fa.h; pointers are ints (device addresses). Returns the status."""
    return load_library().fa_fwd(q, k, v, o, lse, B, H_q, H_kv, qL, kL, D, float(scale), int(causal),
                                  mask, int(mask_kind), int(dtype), stream)


def fa_fwd_ex(args: FaFwdArgs) -> int:
    return load_library().fa_fwd_ex(ctypes.byref(args))


def fa_fwd_workspace_bytes(args: FaFwdArgs) -> int:
    """``fa_fwd_workspace_bytes`` of include/fa.h: scratch bytes the fastest plan wants (0: none, -1: invalid)."""
    return load_library().fa_fwd_workspace_bytes(ctypes.byref(args))


def fa_last_error() -> str:
    return load_library().fa_last_error().decode(errors="replace")


def fa_sync_status(stream=None) -> int:
    return load_library().fa_sync_status(stream)


def fa_set_timeout_cycles(cycles: int) -> None:
    load_library().fa_set_timeout_cycles(int(cycles))


def fa_set_max_ctas(n: int) -> None:
    load_library().fa_set_max_ctas(int(n))


def fa_set_q_tiles(n: int) -> None:
    load_library().fa_set_q_tiles(int(n))


def fa_set_kv_splits(n: int) -> None:
    """``fa_set_kv_splits`` of include/fa.h: key ranges per query tile for split-KV (0: automatic)."""
    load_library().fa_set_kv_splits(int(n))


def fa_version() -> int:
    return load_library().fa_version()


def fa_bwd_workspace_bytes(B: int, H_q: int, qL: int) -> int:
    return load_library().fa_bwd_workspace_bytes(int(B), int(H_q), int(qL))


def fa_bwd_ex_workspace_bytes(B: int, H_q: int, qL: int, kL: int, dropout_p: float = 0.0) -> int:
    """``fa_bwd_ex_workspace_bytes`` of include/fa.h (adds the keep mask when dropout_p > 0)."""
    return load_library().fa_bwd_ex_workspace_bytes(int(B), int(H_q), int(qL), int(kL), float(dropout_p))


def fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H_q, H_kv, qL, kL, D, scale, causal,
           dtype, stream):
    """``fa_bwd`` of include/fa.h; pointers are ints (device addresses). Returns the status."""
    return load_library().fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, int(workspace_bytes), B, H_q, H_kv,
                                  qL, kL, D, float(scale), int(causal), int(dtype), stream)


def fa_bwd_ex(q, k, v, o, dout, lse, dq, dk, dv, workspace, workspace_bytes, B, H_q, H_kv, qL, kL, D, scale, causal,
              window, q_offset, softcap, dropout_p, dropout_seed, dropout_offset, dtype, stream):
    """``fa_bwd_ex`` of include/fa.h (fa_bwd with a sliding window / causal diagonal offset / softcap /
    the forward's dropout). Returns the status."""
    return load_library().fa_bwd_ex(q, k, v, o, dout, lse, dq, dk, dv, workspace, int(workspace_bytes), B, H_q, H_kv,
                                     qL, kL, D, float(scale), int(causal), int(window), int(q_offset),
                                     float(softcap), float(dropout_p), int(dropout_seed) & (2**64 - 1),
                                     int(dropout_offset) & (2**64 - 1), int(dtype), stream)


def fa_bwd_full(args: FaBwdArgs) -> int:
    """``fa_bwd_full`` of include/fa.h (every backward option in one argument block). Returns the status."""
    return load_library().fa_bwd_full(ctypes.byref(args))


def fa_bwd_full_workspace_bytes(args: FaBwdArgs) -> int:
    """``fa_bwd_full_workspace_bytes`` of include/fa.h (-1: invalid arguments)."""
    return load_library().fa_bwd_full_workspace_bytes(ctypes.byref(args))


def fa_bwd_noalloc(q, k, v, o, dout, lse, dq, dk, dv, B, H_q, H_kv, qL, kL, D, scale, causal, dtype, stream):
    """``fa_bwd_noalloc`` of include/fa.h (built-in scratch, no workspace). Returns the status."""
    return load_library().fa_bwd_noalloc(q, k, v, o, dout, lse, dq, dk, dv, B, H_q, H_kv, qL, kL, D,
                                          float(scale), int(causal), int(dtype), stream)


# ----------------------------------------------------------------- torch convenience layer

def _strides_bhs(t, name):
    if t.dim() != 4:
        raise ValueError(f"{name} must be 4-D [B, H, rows, D] (got {tuple(t.shape)})")
    if t.stride(3) != 1:
        raise ValueError(f"{name} must have unit stride along its last dimension")
    return (t.stride(0), t.stride(1), t.stride(2))


def make_args(q, k, v, o, lse, *, scale=None, causal=False, mask=None, mask_kind=None, stream=None, window=0,
              q_offset=0, softcap=0.0, dropout_p=0.0, dropout_seed=0, dropout_offset=0) -> FaFwdArgs:
    """Fill ``fa_fwd_args`` from torch CUDA tensors (4-D views with unit inner stride).

    q, o: [B, H_q, qL, D]; k, v: [B, H_kv, kL, D]; lse: contiguous [B, H_q, qL]
    fp32; mask: None, bool/uint8 (keep = nonzero) or an additive tensor of
    q's dtype, broadcastable to [B, H_q, qL, kL] through its strides.
    """
    import torch
    B, H_q, qL, D = q.shape
    Bk, H_kv, kL, Dk = k.shape
    if tuple(v.shape) != (Bk, H_kv, kL, Dk) or Bk != B or Dk != D:
        raise ValueError(f"shape mismatch: q {tuple(q.shape)}, k {tuple(k.shape)}, v {tuple(v.shape)}")
    if tuple(o.shape) != (B, H_q, qL, D):
        raise ValueError(f"o must be [B, H_q, qL, D] = {(B, H_q, qL, D)} (got {tuple(o.shape)})")
    if tuple(lse.shape) != (B, H_q, qL) or lse.dtype != torch.float32 or not lse.is_contiguous():
        raise ValueError(f"lse must be a contiguous fp32 [B, H_q, qL] = {(B, H_q, qL)} tensor")
    if q.dtype == torch.bfloat16:
        dtype = FA_DTYPE_BF16
    elif q.dtype == torch.float16:
        dtype = FA_DTYPE_F16
    elif q.dtype == torch.float32:
        dtype = FA_DTYPE_F32
    else:
        raise ValueError(f"q dtype {q.dtype} is not bfloat16, float16 or float32")
    for name, t in (("k", k), ("v", v), ("o", o)):
        if t.dtype != q.dtype:
            raise ValueError(f"{name} dtype {t.dtype} differs from q dtype {q.dtype}")
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("lse", lse)):
        if not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
    a = FaFwdArgs()
    a.q, a.k, a.v, a.o, a.lse = q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr()
    a.B, a.H_q, a.H_kv, a.qL, a.kL, a.D = B, H_q, H_kv, qL, kL, D
    a.scale = float(1.0 / math.sqrt(D) if scale is None else scale)
    a.causal = int(bool(causal))
    a.dtype = dtype
    a.window, a.q_offset, a.softcap = int(window), int(q_offset), float(softcap)
    a.dropout_p, a.dropout_seed, a.dropout_offset = float(dropout_p), int(dropout_seed), int(dropout_offset)
    a.q_strides[:] = _strides_bhs(q, "q")
    a.k_strides[:] = _strides_bhs(k, "k")
    a.v_strides[:] = _strides_bhs(v, "v")
    a.o_strides[:] = _strides_bhs(o, "o")
    if mask is None:
        a.mask, a.mask_kind = None, FA_MASK_NONE
        a.mask_strides[:] = (0, 0, 0)
    else:
        if mask_kind is None:
            mask_kind = FA_MASK_BOOL if mask.dtype in (torch.bool, torch.uint8) else FA_MASK_ADDITIVE
        if mask_kind == FA_MASK_BOOL:
            if mask.dtype == torch.bool:
                mask = mask.view(torch.uint8)
            if mask.dtype != torch.uint8:
                raise ValueError("a bool mask must be torch.bool or torch.uint8")
        elif mask.dtype != q.dtype:
            raise ValueError(f"an additive mask must have q's dtype {q.dtype} (got {mask.dtype})")
        if not mask.is_cuda:
            raise ValueError("mask must be a CUDA tensor")
        mask = mask.expand(B, H_q, qL, kL)
        if mask.stride(3) != 1:
            raise ValueError("mask must have unit stride along the key dimension")
        a.mask, a.mask_kind = mask.data_ptr(), int(mask_kind)
        a.mask_strides[:] = (mask.stride(0), mask.stride(1), mask.stride(2))
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    a.stream = stream
    return a


def attach_workspace(args, device, workspace=None):
    """Give ``args`` the scratch its fastest plan needs (``fa_fwd_workspace_bytes``):
    ``workspace`` if given (a device tensor), else a new one from torch's
    allocator on the current stream; ``workspace=False`` leaves the call
    without.  Returns the tensor or None.  A call on another stream than the
    current one should pass its own workspace and keep it alive until the call
    has run."""
    import torch
    if workspace is False:
        return None
    need = fa_fwd_workspace_bytes(args)
    if need < 0:
        _check(FA_ERR_INVALID_ARGUMENT)
    if need == 0:
        return None
    if workspace is None:
        workspace = torch.empty(need + 256, dtype=torch.uint8, device=device)
    base = workspace.data_ptr()
    start = (base + 255) // 256 * 256
    if workspace.numel() * workspace.element_size() - (start - base) < need:
        raise ValueError(f"workspace holds fewer than the {need} bytes (256-byte aligned) required")
    args.workspace, args.workspace_bytes = start, need
    return workspace


def _keep_until_stream_done(t, stream, device):
    """Tell torch's caching allocator that ``t`` (allocated on the current
    stream) is used by work queued on ``stream`` (a raw cudaStream_t), so its
    memory is not handed out again before that work has run."""
    import torch
    if stream != torch.cuda.current_stream(device).cuda_stream:
        t.record_stream(torch.cuda.ExternalStream(stream, device=device))


def attention(q, k, v, *, scale=None, causal=False, mask=None, mask_kind=None, out=None, lse=None,
              stream=None, window=0, q_offset=0, softcap=0.0, dropout_p=0.0, dropout_seed=0, dropout_offset=0,
              workspace=None):
    """O and L for torch CUDA tensors (see ``make_args``); returns (o, lse).

    workspace: scratch for plans that want one (see ``attach_workspace``):
    None allocates it when needed, False runs without."""
    import torch
    B, H_q, qL, D = q.shape
    if out is None:
        out = torch.empty((B, H_q, qL, D), dtype=q.dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H_q, qL), dtype=torch.float32, device=q.device)
    args = make_args(q, k, v, out, lse, scale=scale, causal=causal, mask=mask, mask_kind=mask_kind,
                     stream=stream, window=window, q_offset=q_offset, softcap=softcap, dropout_p=dropout_p,
                     dropout_seed=dropout_seed, dropout_offset=dropout_offset)
    ws = attach_workspace(args, q.device, workspace)
    if ws is not None and workspace is None and stream is not None:
        _keep_until_stream_done(ws, stream, q.device)
    _check(fa_fwd_ex(args))
    del ws  # torch hands the block out again only to work queued later on the same stream
    return out, lse


def attention_bwd(q, k, v, o, dout, lse, *, scale=None, causal=False, dq=None, dk=None, dv=None, workspace=None,
                  stream=None, window=0, q_offset=0, softcap=0.0, dropout_p=0.0, dropout_seed=0, dropout_offset=0,
                  mask=None, mask_kind=None):
    """dQ, dK, dV for torch CUDA tensors; returns (dq, dk, dv).

    window, q_offset, softcap, dropout_p, dropout_seed, dropout_offset, mask,
    mask_kind: the forward's (``attention``), so that the backward sees the
    same softmax and regenerates the same keep decisions.

    q, o, dout: contiguous bf16, fp16 or fp32 [B, H_q, qL, D]; k, v: the same
    dtype, [B, H_kv, kL, D]; lse: the forward's contiguous fp32 [B, H_q, qL].
    fp32 (TF32 products) takes D 64 or 128 and causal or full attention only.
    mask: None, bool/uint8 (nonzero keeps) or additive in q's dtype,
    broadcastable to [B, H_q, qL, kL] through its strides.
    workspace: optional device tensor of at least ``fa_bwd_full_workspace_bytes``
    bytes, 256-byte aligned (allocated here if None).
    """
    import torch
    B, H_q, qL, D = q.shape
    Bk, H_kv, kL, Dk = k.shape
    if tuple(v.shape) != (Bk, H_kv, kL, Dk) or Bk != B or Dk != D:
        raise ValueError(f"shape mismatch: q {tuple(q.shape)}, k {tuple(k.shape)}, v {tuple(v.shape)}")
    for name, t in (("o", o), ("dout", dout)):
        if tuple(t.shape) != (B, H_q, qL, D):
            raise ValueError(f"{name} must be [B, H_q, qL, D] = {(B, H_q, qL, D)} (got {tuple(t.shape)})")
    if tuple(lse.shape) != (B, H_q, qL) or lse.dtype != torch.float32:
        raise ValueError(f"lse must be fp32 [B, H_q, qL] = {(B, H_q, qL)}")
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout), ("lse", lse)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
        if name != "lse" and t.dtype != q.dtype:
            raise ValueError(f"{name} must have q's dtype {q.dtype}")
    if q.dtype not in (torch.bfloat16, torch.float16, torch.float32):
        raise ValueError("the backward pass supports bfloat16, float16 and float32 I/O")
    if dq is None:
        dq = torch.empty_like(q)
    if dk is None:
        dk = torch.empty_like(k)
    if dv is None:
        dv = torch.empty_like(v)
    # the kernels write every element of dq, dk and dv through raw pointers: a
    # wrong size or layout would be written out of bounds
    for name, t, like in (("dq", dq, q), ("dk", dk, k), ("dv", dv, v)):
        if tuple(t.shape) != tuple(like.shape) or t.dtype != like.dtype:
            raise ValueError(f"{name} must be {like.dtype} {tuple(like.shape)} (got {t.dtype} {tuple(t.shape)})")
        if not t.is_cuda or t.device != q.device or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor on {q.device}")
    a = FaBwdArgs()
    a.q, a.k, a.v, a.o, a.dout, a.lse = (t.data_ptr() for t in (q, k, v, o, dout, lse))
    a.dq, a.dk, a.dv = dq.data_ptr(), dk.data_ptr(), dv.data_ptr()
    a.B, a.H_q, a.H_kv, a.qL, a.kL, a.D = B, H_q, H_kv, qL, kL, D
    a.scale = float(1.0 / math.sqrt(D) if scale is None else scale)
    a.causal = int(bool(causal))
    a.window, a.q_offset, a.softcap = int(window), int(q_offset), float(softcap)
    a.dropout_p = float(dropout_p)
    a.dropout_seed, a.dropout_offset = int(dropout_seed) & (2**64 - 1), int(dropout_offset) & (2**64 - 1)
    a.dtype = {torch.float16: FA_DTYPE_F16, torch.float32: FA_DTYPE_F32}.get(q.dtype, FA_DTYPE_BF16)
    if mask is None:
        a.mask, a.mask_kind = None, FA_MASK_NONE
    else:
        if mask_kind is None:
            mask_kind = FA_MASK_BOOL if mask.dtype in (torch.bool, torch.uint8) else FA_MASK_ADDITIVE
        if mask_kind == FA_MASK_BOOL:
            if mask.dtype == torch.bool:
                mask = mask.view(torch.uint8)
            if mask.dtype != torch.uint8:
                raise ValueError("a bool mask must be torch.bool or torch.uint8")
        elif mask.dtype != q.dtype:
            raise ValueError(f"an additive mask must have q's dtype {q.dtype} (got {mask.dtype})")
        if not mask.is_cuda:
            raise ValueError("mask must be a CUDA tensor")
        mask = mask.expand(B, H_q, qL, kL)
        if mask.stride(3) != 1:
            raise ValueError("mask must have unit stride along the key dimension")
        a.mask, a.mask_kind = mask.data_ptr(), int(mask_kind)
        a.mask_strides[:] = (mask.stride(0), mask.stride(1), mask.stride(2))
    need = fa_bwd_full_workspace_bytes(a)
    if need < 0:
        _check(FA_ERR_INVALID_ARGUMENT)
    own_workspace = workspace is None
    if own_workspace:
        workspace = torch.empty(need + 256, dtype=torch.uint8, device=q.device)
    base = workspace.data_ptr()
    start = (base + 255) // 256 * 256
    if workspace.numel() * workspace.element_size() - (start - base) < need:
        raise ValueError(f"workspace holds fewer than the {need} bytes (256-byte aligned) required")
    a.workspace, a.workspace_bytes = start, need
    if stream is None:
        stream = torch.cuda.current_stream(q.device).cuda_stream
    elif own_workspace:
        _keep_until_stream_done(workspace, stream, q.device)
    a.stream = stream
    _check(fa_bwd_full(a))
    return dq, dk, dv
