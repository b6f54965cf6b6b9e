"""Host-side tests of the C ABI (no GPU needed): the library builds and loads,
exports every entry point include/fa.h declares, its argument struct matches
the header's layout, and validation rejects bad arguments before any CUDA
call, with the documented status codes and a message."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def fa():
    from attention_forward_08_gb300 import _build
    _build.build()
    import attention_forward_08_gb300 as fa
    fa.load_library()
    return fa


def _declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:int|void|long long|const char\*)\s+(fa_\w+)\s*\(", text, re.M)))


def test_header_declares_the_abi():
    assert _declared_functions() == sorted(
        ["fa_fwd", "fa_fwd_ex", "fa_fwd_workspace_bytes", "fa_bwd", "fa_bwd_ex", "fa_bwd_workspace_bytes",
         "fa_bwd_ex_workspace_bytes", "fa_bwd_full", "fa_bwd_full_workspace_bytes", "fa_bwd_noalloc",
         "fa_last_error",
         "fa_sync_status",
         "fa_set_kv_splits", "fa_set_max_ctas", "fa_set_q_tiles", "fa_set_timeout_cycles", "fa_version"])


def test_library_exports_every_declared_symbol(fa):
    lib = fa.load_library()
    for name in _declared_functions():
        assert hasattr(lib, name), f"{name} not exported"
    out = subprocess.run(["nm", "-D", "--defined-only", fa.fa.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (fa_\w+)", out))
    assert set(_declared_functions()) <= exported


@pytest.mark.parametrize("cname,pyname", [("fa_fwd_args", "FaFwdArgs"), ("fa_bwd_args", "FaBwdArgs")])
def test_args_struct_matches_header(tmp_path, cname, pyname):
    """ctypes' argument structs have the same size and field offsets as the C structs."""
    from attention_forward_08_gb300 import fa as binding
    S = getattr(binding, pyname)
    fields = [f for f, _ in S._fields_]
    src = tmp_path / "layout.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "fa.h"\nint main(void){\n'
                   f'  printf("%zu\\n", sizeof({cname}));\n'
                   + "".join(f'  printf("%zu\\n", offsetof({cname}, {f}));\n' for f in fields)
                   + "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", f"-I{ROOT}/include", str(src), "-o", str(exe)], check=True)
    vals = [int(x) for x in subprocess.run([str(exe)], capture_output=True, text=True).stdout.split()]
    assert vals[0] == ctypes.sizeof(S)
    for f, off in zip(fields, vals[1:]):
        assert getattr(S, f).offset == off, f


def test_version(fa):
    assert fa.fa_version() == 111


P = 0x10000  # a 16-byte aligned stand-in address: validation never dereferences it


def _call(fa, **kw):
    a = dict(q=P, k=P, v=P, o=P, lse=P, B=1, H_q=2, H_kv=2, qL=128, kL=128, D=128, scale=0.125, causal=0,
             mask=None, mask_kind=0, dtype=1, stream=None)
    a.update(kw)
    return fa.fa_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H_q"], a["H_kv"], a["qL"], a["kL"],
                     a["D"], a["scale"], a["causal"], a["mask"], a["mask_kind"], a["dtype"], a["stream"])


@pytest.mark.parametrize("kw,status,needle", [
    (dict(q=None), 1, "non-NULL"),
    (dict(lse=None), 1, "non-NULL"),
    (dict(B=0), 1, "> 0"),
    (dict(qL=-5), 1, "> 0"),
    (dict(kL=0), 1, "> 0"),
    (dict(H_q=6, H_kv=4), 1, "divisible"),
    (dict(dtype=7), 1, "dtype"),
    (dict(dtype=3), 1, "dtype"),
    (dict(mask_kind=3, mask=P), 1, "mask_kind"),
    (dict(mask_kind=1, mask=None), 1, "mask must be non-NULL"),
    (dict(mask_kind=0, mask=P), 1, "mask must be non-NULL"),
    (dict(scale=float("nan")), 1, "finite"),
    (dict(scale=float("inf")), 1, "finite"),
    (dict(D=96), 2, "head dim"),
    (dict(D=32), 2, "head dim"),
    (dict(q=P + 8), 3, "16-byte"),
    (dict(o=P + 2), 3, "16-byte"),
    (dict(lse=P + 2), 3, "4-byte"),
])
def test_validation_rejects(fa, kw, status, needle):
    rc = _call(fa, **kw)
    assert rc == status
    assert needle in fa.fa_last_error()


def test_misaligned_strides_rejected(fa):
    """fa_fwd_ex: a row stride that is not a multiple of 16 bytes cannot feed TMA."""
    a = fa.FaFwdArgs()
    a.q = a.k = a.v = a.o = a.lse = P
    a.B, a.H_q, a.H_kv, a.qL, a.kL, a.D = 1, 2, 2, 64, 64, 64
    a.scale, a.dtype = 0.125, 1
    for s in (a.q_strides, a.k_strides, a.v_strides, a.o_strides):
        s[:] = (2 * 64 * 64, 64 * 64, 64)
    a.o_strides[:] = (2 * 64 * 68, 64 * 68, 68 + 1)   # 69 bf16 = 138 bytes per row
    assert fa.fa_fwd_ex(a) == 3
    assert "strides" in fa.fa_last_error()
    a.o_strides[:] = (2 * 64 * 64, 64 * 64, 32)        # rows overlap: stride < D
    assert fa.fa_fwd_ex(a) == 1


def test_dropout_arguments_validated(fa):
    """fa_fwd_ex: dropout_p outside [0, 1] is invalid; dropout with kL not a multiple of 4 is unsupported."""
    a = fa.FaFwdArgs()
    a.q = a.k = a.v = a.o = a.lse = P
    a.B, a.H_q, a.H_kv, a.qL, a.kL, a.D = 1, 2, 2, 64, 64, 64
    a.scale, a.dtype = 0.125, 1
    for t in (a.q_strides, a.k_strides, a.v_strides, a.o_strides):
        t[:] = (2 * 64 * 64, 64 * 64, 64)
    a.dropout_p = 1.5
    assert fa.fa_fwd_ex(a) == 1 and "dropout_p" in fa.fa_last_error()
    a.dropout_p, a.kL = 0.1, 66
    for t in (a.k_strides, a.v_strides):
        t[:] = (2 * 66 * 64, 66 * 64, 64)
    assert fa.fa_fwd_ex(a) == 2 and "multiple of 4" in fa.fa_last_error()


def _fwd_args(fa, dtype, B, H_q, H_kv, qL, kL, D):
    a = fa.FaFwdArgs()
    a.q = a.k = a.v = a.o = a.lse = P
    a.B, a.H_q, a.H_kv, a.qL, a.kL, a.D = B, H_q, H_kv, qL, kL, D
    a.scale, a.dtype = D ** -0.5, dtype
    a.q_strides[:] = a.o_strides[:] = (H_q * qL * D, qL * D, D)
    a.k_strides[:] = a.v_strides[:] = (H_kv * kL * D, kL * D, D)
    return a


def test_forward_workspace_size(fa):
    """fa_fwd_workspace_bytes: the tf32 pre-pass plan (fp32, plain, kL >= 1024) wants rounded Q and K and a
    transposed V with rows padded to 4 keys, each part 256-byte aligned; other calls want nothing."""
    al = lambda n: (n + 255) // 256 * 256
    a = _fwd_args(fa, 0, 2, 4, 2, 300, 1030, 128)
    want = al(2 * 4 * 300 * 128 * 4) + al(2 * 2 * 1030 * 128 * 4) + al(2 * 2 * 128 * 1032 * 4)
    assert fa.fa_fwd_workspace_bytes(a) == want
    assert fa.fa_fwd_workspace_bytes(_fwd_args(fa, 1, 2, 4, 2, 300, 1030, 128)) == 0   # bf16
    assert fa.fa_fwd_workspace_bytes(_fwd_args(fa, 0, 1, 2, 2, 128, 128, 64)) == 0     # short kL
    a.window = 64
    assert fa.fa_fwd_workspace_bytes(a) == 0
    a.window, a.H_q = 0, 3                                                            # 3 % 2 != 0
    assert fa.fa_fwd_workspace_bytes(a) == -1 and "divisible" in fa.fa_last_error()


def test_forward_workspace_validated(fa):
    """fa_fwd_ex: a misaligned workspace, or one smaller than the plan needs, is rejected before any launch."""
    a = _fwd_args(fa, 0, 1, 2, 2, 256, 2048, 64)
    need = fa.fa_fwd_workspace_bytes(a)
    a.workspace, a.workspace_bytes = P + 16, need
    assert fa.fa_fwd_ex(a) == 1 and "256-byte" in fa.fa_last_error()
    a.workspace, a.workspace_bytes = P, need - 256
    assert fa.fa_fwd_ex(a) == 1 and "smaller" in fa.fa_last_error()


def test_no_gpu_is_a_cuda_error(fa):
    """A fully valid call on a machine without a usable GPU reports FA_ERR_CUDA (it never falls back)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rc = _call(fa)
    assert rc == 4
    assert fa.fa_last_error()


def test_error_message_cleared_on_success_path(fa):
    _call(fa, D=96)
    assert fa.fa_last_error()
    _call(fa, q=None)
    assert "non-NULL" in fa.fa_last_error()


def _bwd_call(fa, **kw):
    a = dict(q=P, k=P, v=P, o=P, dout=P, lse=P, dq=P, dk=P, dv=P, ws=P, ws_bytes=1 << 20, B=1, H_q=2, H_kv=2,
             qL=128, kL=128, D=128, scale=0.125, causal=1, dtype=1, stream=None)
    a.update(kw)
    return fa.fa_bwd(a["q"], a["k"], a["v"], a["o"], a["dout"], a["lse"], a["dq"], a["dk"], a["dv"], a["ws"],
                     a["ws_bytes"], a["B"], a["H_q"], a["H_kv"], a["qL"], a["kL"], a["D"], a["scale"], a["causal"],
                     a["dtype"], a["stream"])


def test_bwd_workspace_size(fa):
    assert fa.fa_bwd_workspace_bytes(2, 32, 4096) == 2 * 32 * 4096 * 4
    assert fa.fa_bwd_workspace_bytes(1, 1, 3) == 256
    assert fa.fa_bwd_workspace_bytes(0, 1, 3) == -1


def test_row_counts_never_overflow(fa):
    """Row counts whose product leaves the int64 range are refused, not wrapped: the forward, the
    backward and the workspace size queries compare one factor at a time."""
    big = 1 << 21
    assert _call(fa, B=big, H_q=big, H_kv=big, qL=big, kL=128) == 2
    assert "2^31" in fa.fa_last_error()
    assert _call(fa, B=1, H_q=2, H_kv=2, qL=128, kL=2**31 - 1) == 2
    assert _bwd_call(fa, B=big, H_q=big, H_kv=big, qL=big) == 2
    assert fa.fa_bwd_workspace_bytes(big, big, big) == -1
    assert fa.fa_bwd_ex_workspace_bytes(big, big, big, 128, 0.1) == -1
    assert fa.fa_bwd_workspace_bytes(1, 1, 2**31 - 1) == (4 * (2**31 - 1) + 255) // 256 * 256


def test_bwd_ex_workspace_size(fa):
    # no dropout: the D vector alone; with dropout: plus 16 bytes per row and 128-key block
    assert fa.fa_bwd_ex_workspace_bytes(2, 32, 4096, 4096, 0.0) == fa.fa_bwd_workspace_bytes(2, 32, 4096)
    assert fa.fa_bwd_ex_workspace_bytes(2, 32, 4096, 4096, 0.1) == 2 * 32 * 4096 * 4 + 2 * 32 * 4096 * 32 * 16
    assert fa.fa_bwd_ex_workspace_bytes(1, 1, 3, 200, 1.0) == 256 + 3 * 2 * 16
    assert fa.fa_bwd_ex_workspace_bytes(1, 1, 3, 0, 0.1) == -1
    assert fa.fa_bwd_ex_workspace_bytes(1, 1, 3, 8, 1.5) == -1
    assert fa.fa_bwd_ex_workspace_bytes(0, 1, 3, 8, 0.0) == -1


def test_bwd_ex_rejects_workspace_without_room_for_the_keep_mask(fa):
    # enough for the D vector, not for the keep mask of a dropout call
    need = fa.fa_bwd_ex_workspace_bytes(1, 2, 128, 128, 0.1)
    assert fa.fa_bwd_ex(P, P, P, P, P, P, P, P, P, P, need - 16, 1, 2, 2, 128, 128, 128, 0.125, 1, 0, 0, 0.0, 0.1,
                        7, 0, 1, None) == 1
    assert "workspace" in fa.fa_last_error()


@pytest.mark.parametrize("kw,status,needle", [
    (dict(dout=None), 1, "non-NULL"),
    (dict(ws=None), 1, "non-NULL"),
    (dict(H_q=6, H_kv=4), 1, "divisible"),
    (dict(kL=0), 1, "> 0"),
    (dict(scale=float("nan")), 1, "finite"),
    (dict(dtype=0), 2, "bf16 and fp16"),
    (dict(dtype=5), 1, "dtype"),
    (dict(D=96), 2, "head dim"),
    (dict(D=512), 2, "head dim"),
    (dict(ws_bytes=100), 1, "workspace"),
    (dict(dk=P + 4), 3, "16-byte"),
])
def test_bwd_validation_rejects(fa, kw, status, needle):
    assert _bwd_call(fa, **kw) == status
    assert needle in fa.fa_last_error()


@pytest.mark.parametrize("window,q_offset,softcap,drop_p,kL,status,needle", [
    (-1, 0, 0.0, 0.0, 128, 1, "window"), (0, 1 << 30, 0.0, 0.0, 128, 1, "q_offset"),
    (0, -(1 << 30), 0.0, 0.0, 128, 1, "q_offset"), (0, 0, -1.0, 0.0, 128, 1, "softcap"),
    (0, 0, float("inf"), 0.0, 128, 1, "softcap"), (0, 0, 0.0, -0.1, 128, 1, "dropout_p"),
    (0, 0, 0.0, 1.5, 128, 1, "dropout_p"), (0, 0, 0.0, float("nan"), 128, 1, "dropout_p"),
    (0, 0, 0.0, 0.1, 130, 2, "multiple of 4")])
def test_bwd_ex_validation_rejects(fa, window, q_offset, softcap, drop_p, kL, status, needle):
    assert fa.fa_bwd_ex(P, P, P, P, P, P, P, P, P, P, 1 << 20, 1, 2, 2, 128, kL, 128, 0.125, 1, window, q_offset,
                        softcap, drop_p, 7, 0, 1, None) == status
    assert needle in fa.fa_last_error()


def test_product_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "attention_forward_08_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"\b(import|from)\s+oracle\b", text), f
                assert "attn_oracle" not in text and "liboracle" not in text, f


def test_binding_fails_loudly_without_library(tmp_path):
    from attention_forward_08_gb300 import fa as binding
    with pytest.raises(ImportError):
        saved = binding._lib
        binding._lib = None
        try:
            binding.load_library(str(tmp_path / "missing.so"))
        finally:
            binding._lib = saved


def _bwd_args(fa, **kw):
    a = fa.FaBwdArgs()
    a.q = a.k = a.v = a.o = a.dout = a.lse = a.dq = a.dk = a.dv = P
    a.workspace, a.workspace_bytes = P, 1 << 30
    a.B, a.H_q, a.H_kv, a.qL, a.kL, a.D = 1, 2, 2, 200, 300, 128
    a.scale, a.causal, a.dtype = 0.088, 1, 1
    for k_, v_ in kw.items():
        if k_ == "mask_strides":
            a.mask_strides[:] = v_
        else:
            setattr(a, k_, v_)
    return a


def test_bwd_full_workspace_with_mask(fa):
    """fa_bwd_full_workspace_bytes: the D vector, then (dropout) the keep words, then (additive mask) a key-major
    copy of the mask with whole 128-row query blocks per key, or (bool mask) its keep bits key-major and
    row-major, 16 bytes per row (key) and 128-entry block; each part 256-byte aligned."""
    al = lambda n: (n + 255) // 256 * 256
    base = fa.fa_bwd_ex_workspace_bytes(1, 2, 200, 300, 0.0)
    assert fa.fa.fa_bwd_full_workspace_bytes(_bwd_args(fa)) == base
    a = _bwd_args(fa, mask=P, mask_kind=2, mask_strides=(2 * 200 * 300, 200 * 300, 300))
    assert fa.fa.fa_bwd_full_workspace_bytes(a) == al(base) + al(1 * 2 * 300 * 256 * 2)
    a = _bwd_args(fa, mask=P, mask_kind=1, mask_strides=(0, 0, 300), dropout_p=0.1)
    base = fa.fa_bwd_ex_workspace_bytes(1, 2, 200, 300, 0.1)
    assert fa.fa.fa_bwd_full_workspace_bytes(a) == al(base) + al(1 * 2 * 300 * (256 // 32) * 4) + \
        al(1 * 2 * 200 * (3 * 4) * 4)


def test_bwd_full_workspace_fp32(fa):
    """fp32: the D vector, then tf32-rounded Q, dO, K, V and the transposes Q^T, dO^T [B, H_q, D, qL
    rounded up to 4] and K^T [B, H_kv, D, kL rounded up to 4], each part 256-byte aligned."""
    al = lambda n: (n + 255) // 256 * 256
    a = _bwd_args(fa, dtype=0, qL=201, kL=299, D=64)
    qt, kt = (201 + 3) // 4 * 4, (299 + 3) // 4 * 4
    expect = (al(al(1 * 2 * 201 * 4)) + 2 * al(1 * 2 * 201 * 64 * 4) + 2 * al(1 * 2 * 299 * 64 * 4)
              + 2 * al(1 * 2 * 64 * qt * 4) + al(1 * 2 * 64 * kt * 4))
    assert fa.fa.fa_bwd_full_workspace_bytes(a) == expect
    a.workspace_bytes = expect - 1
    assert fa.fa.fa_bwd_full(a) == 1 and "workspace" in fa.fa_last_error()


def test_bwd_entries_without_full_workspace_refuse_fp32(fa):
    assert _bwd_call(fa, dtype=0) == 2 and "fa_bwd_full" in fa.fa_last_error()
    assert fa.fa.fa_bwd_noalloc(P, P, P, P, P, P, P, P, P, 1, 2, 2, 128, 128, 64, 0.125, 1, 0, None) == 2
    assert "fa_bwd_full" in fa.fa_last_error()


@pytest.mark.parametrize("kw,status,needle", [
    (dict(mask=P, mask_kind=0), 1, "mask must be non-NULL"),
    (dict(mask=None, mask_kind=2), 1, "mask must be non-NULL"),
    (dict(mask=P, mask_kind=3), 1, "mask_kind"),
    (dict(mask=P, mask_kind=1, mask_strides=(0, -1, 300)), 1, "strides"),
    (dict(mask=P, mask_kind=2, softcap=5.0), 2, "softcap"),
    (dict(mask=P, mask_kind=2, workspace=P + 16), 3, "256-byte"),
    (dict(mask=P, mask_kind=2, workspace_bytes=1024), 1, "workspace"),
    # fp32: D 64 or 128, causal or full attention only
    (dict(dtype=0, D=256), 2, "fp32"),
    (dict(dtype=0, window=64), 2, "fp32"),
    (dict(dtype=0, mask=P, mask_kind=1), 2, "fp32"),
    (dict(dtype=0, dropout_p=0.1), 2, "fp32"),
    (dict(dtype=7), 1, "dtype"),
    # head dim 256: causal or full attention only
    (dict(D=256, mask=P, mask_kind=1), 2, "D = 256"),
    (dict(D=256, window=64), 2, "D = 256"),
    (dict(D=256, q_offset=100), 2, "D = 256"),
    (dict(D=256, softcap=5.0), 2, "D = 256"),
    (dict(D=256, dropout_p=0.1), 2, "D = 256"),
])
def test_bwd_full_validation_rejects(fa, kw, status, needle):
    a = _bwd_args(fa, **kw)
    assert fa.fa.fa_bwd_full(a) == status
    assert needle in fa.fa_last_error()
