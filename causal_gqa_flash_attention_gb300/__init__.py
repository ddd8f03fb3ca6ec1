"""Python binding of libneattn (causal GQA + RoPE flash attention for sm_103a).

Argument marshalling only: every function checks dtypes, shapes and devices, then
calls the C ABI declared in include/neattn.h with raw device pointers and the
current torch CUDA stream.  All arithmetic runs in the library's CUDA kernels.  There
is no CPU fallback: if libneattn.so is missing or no sm_103 device is present the
calls raise.

Layouts: q, o, dO, dq are [B, T, Hq, D]; k, v, dk, dv are [B, T, Hkv, D]; lse is
[B, Hq, T] fp32.  bf16 tensors run on bf16 tensor cores, fp32 tensors on TF32.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import synthetic  # noqa: F401  (seeded inputs; no attention arithmetic)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libneattn.so")
_lock = threading.Lock()
_lib = None

NE_OK, NE_ERR_INVALID_ARG, NE_ERR_UNSUPPORTED, NE_ERR_CUDA, NE_ERR_DEVICE_TIMEOUT, NE_ERR_NO_DEVICE = range(6)

# Every symbol include/neattn.h declares (checked by the tests).
EXPORTS = (
    "ne_rope_table", "ne_attn_fwd", "ne_attn_fwd_f32", "ne_attn_bwd_workspace_size", "ne_attn_bwd",
    "ne_attn_bwd_f32", "ne_status_string", "ne_last_error", "ne_get_device_error",
    "ne_set_wait_timeout_ms", "ne_selftest_wait_timeout", "ne_shutdown", "ne_attn_bwd_noalloc",
    "ne_profile_enable", "ne_profile_totals", "ne_attn_decode_workspace_size", "ne_attn_decode",
    "ne_attn_decode_f32", "ne_noalloc_get_device_error", "ne_attn_fwd_varlen", "ne_attn_fwd_varlen_f32",
    "ne_attn_bwd_varlen", "ne_attn_bwd_varlen_f32", "ne_qkv_prologue", "ne_attn_fwd_train",
    "ne_attn_fwd_train_f32", "ne_attn_bwd_train", "ne_attn_bwd_train_f32", "ne_qkv_prologue_workspace_size",
)


class NeError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{msg} [status {status}]")
        self.status = status


def load(path: str | None = None):
    """Load libneattn.so (built by ``_build.build()``).  Raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise ImportError(f"libneattn.so not found at {p}; run __graft_entry__.build() first")
        lib = ctypes.CDLL(p)
        vp, i, d, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_double, ctypes.c_size_t
        lib.ne_rope_table.argtypes = [vp, vp, i, i, d, vp]
        lib.ne_attn_fwd.argtypes = [vp] * 5 + [i] * 5 + [d, vp]
        lib.ne_attn_fwd_f32.argtypes = lib.ne_attn_fwd.argtypes
        lib.ne_attn_bwd_workspace_size.argtypes = [i] * 5
        lib.ne_attn_bwd_workspace_size.restype = sz
        lib.ne_attn_bwd.argtypes = [vp] * 9 + [i] * 5 + [d, vp, sz, vp]
        lib.ne_attn_bwd_f32.argtypes = lib.ne_attn_bwd.argtypes
        lib.ne_status_string.argtypes = [i]
        lib.ne_status_string.restype = ctypes.c_char_p
        lib.ne_last_error.argtypes = []
        lib.ne_last_error.restype = ctypes.c_char_p
        lib.ne_get_device_error.argtypes = [vp]
        lib.ne_set_wait_timeout_ms.argtypes = [ctypes.c_uint32]
        lib.ne_set_wait_timeout_ms.restype = None
        lib.ne_selftest_wait_timeout.argtypes = [ctypes.c_uint32, vp]
        lib.ne_attn_bwd_noalloc.argtypes = [vp] * 9 + [i] * 5 + [d, vp]
        lib.ne_attn_fwd_varlen.argtypes = [vp] * 6 + [i] * 5 + [d, vp]
        lib.ne_attn_fwd_varlen_f32.argtypes = lib.ne_attn_fwd_varlen.argtypes
        lib.ne_attn_bwd_varlen.argtypes = [vp] * 10 + [i] * 5 + [d, vp, sz, vp]
        lib.ne_attn_bwd_varlen_f32.argtypes = lib.ne_attn_bwd_varlen.argtypes
        lib.ne_qkv_prologue.argtypes = [vp] * 6 + [i] * 6 + [d, d, i, vp, sz, vp]
        lib.ne_qkv_prologue_workspace_size.argtypes = [i] * 6
        lib.ne_qkv_prologue_workspace_size.restype = sz
        lib.ne_attn_fwd_train.argtypes = [vp] * 6 + [sz] + [i] * 5 + [d, vp]
        lib.ne_attn_fwd_train_f32.argtypes = lib.ne_attn_fwd_train.argtypes
        lib.ne_attn_bwd_train.argtypes = lib.ne_attn_bwd.argtypes
        lib.ne_attn_bwd_train_f32.argtypes = lib.ne_attn_bwd.argtypes
        lib.ne_noalloc_get_device_error.argtypes = [vp]
        lib.ne_profile_enable.argtypes = [i]
        lib.ne_profile_enable.restype = None
        lib.ne_profile_totals.argtypes = [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int)]
        lib.ne_profile_totals.restype = i
        lib.ne_shutdown.argtypes = []
        lib.ne_shutdown.restype = None
        lib.ne_attn_decode_workspace_size.argtypes = [i] * 5
        lib.ne_attn_decode_workspace_size.restype = sz
        lib.ne_attn_decode.argtypes = [vp] * 6 + [i] * 5 + [d, vp, sz, vp]
        lib.ne_attn_decode_f32.argtypes = lib.ne_attn_decode.argtypes
        for f in ("ne_rope_table", "ne_attn_fwd", "ne_attn_fwd_f32", "ne_attn_bwd", "ne_attn_bwd_f32",
                  "ne_get_device_error", "ne_selftest_wait_timeout", "ne_attn_bwd_noalloc", "ne_attn_decode",
                  "ne_noalloc_get_device_error", "ne_attn_fwd_varlen", "ne_attn_fwd_varlen_f32",
                  "ne_attn_bwd_varlen", "ne_attn_bwd_varlen_f32", "ne_qkv_prologue",
                  "ne_attn_decode_f32"):
            getattr(lib, f).restype = i
        _lib = lib
    return _lib


def _check(status: int):
    if status != NE_OK:
        lib = load()
        raise NeError(status, f"{lib.ne_status_string(status).decode()}: {lib.ne_last_error().decode()}")


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _dims(q, k, v):
    if q.dim() != 4 or k.dim() != 4 or v.dim() != 4:
        raise ValueError("q, k, v must be [B, T, H, D]")
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    if tuple(k.shape) != (B, T, Hkv, D) or tuple(v.shape) != (B, T, Hkv, D):
        raise ValueError(f"k, v must be [B, T, Hkv, D]; got {tuple(k.shape)}, {tuple(v.shape)}")
    for t in (q, k, v):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != q.dtype:
            raise ValueError("q, k, v must be contiguous CUDA tensors of one dtype")
    if q.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("dtype must be bfloat16 or float32")
    return B, T, Hq, Hkv, D


def rope_table(T: int, D: int, theta: float = 10000.0, device="cuda"):
    """cos, sin [T, D/2] fp32 on ``device`` (ne_rope_table)."""
    lib = load()
    c = torch.empty((T, D // 2), dtype=torch.float32, device=device)
    s = torch.empty_like(c)
    _check(lib.ne_rope_table(_ptr(c), _ptr(s), T, D, float(theta), _stream(c)))
    return c, s


def attn_fwd(q, k, v, theta: float = 10000.0, o=None, lse=None):
    """Forward: returns (o [B,T,Hq,D], lse [B,Hq,T] fp32)."""
    lib = load()
    B, T, Hq, Hkv, D = _dims(q, k, v)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, T), dtype=torch.float32, device=q.device)
    fn = lib.ne_attn_fwd if q.dtype == torch.bfloat16 else lib.ne_attn_fwd_f32
    _check(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, T, Hq, Hkv, D, float(theta), _stream(q)))
    return o, lse


def _check_lens(seq_lens, B, device):
    if seq_lens.dtype != torch.int32 or tuple(seq_lens.shape) != (B,) or not seq_lens.is_cuda \
            or not seq_lens.is_contiguous() or seq_lens.device != device:
        raise ValueError("seq_lens must be a contiguous int32 CUDA tensor [B] on the tensors' device")


def attn_fwd_varlen(q, k, v, seq_lens, theta: float = 10000.0, o=None, lse=None):
    """Forward over a padded batch of sequences of lengths seq_lens (int32 [B] on the
    device): returns (o, lse); padding rows get o = 0 and lse = -inf."""
    lib = load()
    B, T, Hq, Hkv, D = _dims(q, k, v)
    _check_lens(seq_lens, B, q.device)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, T), dtype=torch.float32, device=q.device)
    fn = lib.ne_attn_fwd_varlen if q.dtype == torch.bfloat16 else lib.ne_attn_fwd_varlen_f32
    _check(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(seq_lens), _ptr(o), _ptr(lse), B, T, Hq, Hkv, D, float(theta),
              _stream(q)))
    return o, lse


def workspace_size(B, T, Hq, Hkv, D) -> int:
    return int(load().ne_attn_bwd_workspace_size(B, T, Hq, Hkv, D))


def alloc_workspace(B, T, Hq, Hkv, D, device="cuda"):
    n = workspace_size(B, T, Hq, Hkv, D)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def attn_bwd(q, k, v, o, lse, dO, theta: float = 10000.0, workspace=None, dq=None, dk=None, dv=None):
    """Backward: returns (dq, dk, dv) in the input dtype."""
    lib = load()
    B, T, Hq, Hkv, D = _dims(q, k, v)
    for t in (o, dO):
        if tuple(t.shape) != tuple(q.shape) or t.dtype != q.dtype or not t.is_contiguous():
            raise ValueError("o and dO must match q")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, Hq, T) or not lse.is_contiguous():
        raise ValueError("lse must be contiguous fp32 [B, Hq, T]")
    if workspace is None:
        workspace = alloc_workspace(B, T, Hq, Hkv, D, q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    fn = lib.ne_attn_bwd if q.dtype == torch.bfloat16 else lib.ne_attn_bwd_f32
    _check(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk), _ptr(dv),
              B, T, Hq, Hkv, D, float(theta), _ptr(workspace), workspace.numel() * workspace.element_size(),
              _stream(q)))
    return dq, dk, dv


def attn_fwd_train(q, k, v, workspace, theta: float = 10000.0, o=None, lse=None):
    """Training forward: what attn_fwd returns, and (bf16, head_dim 32/64) the backward
    workspace filled for attn_bwd_train of the same layer (see include/neattn.h)."""
    lib = load()
    B, T, Hq, Hkv, D = _dims(q, k, v)
    if o is None:
        o = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, T), dtype=torch.float32, device=q.device)
    fn = lib.ne_attn_fwd_train if q.dtype == torch.bfloat16 else lib.ne_attn_fwd_train_f32
    _check(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(workspace),
              workspace.numel() * workspace.element_size(), B, T, Hq, Hkv, D, float(theta), _stream(q)))
    return o, lse


def attn_bwd_train(q, k, v, o, lse, dO, workspace, theta: float = 10000.0, dq=None, dk=None, dv=None):
    """Backward after attn_fwd_train on the same workspace: returns (dq, dk, dv)."""
    lib = load()
    B, T, Hq, Hkv, D = _dims(q, k, v)
    for t in (o, dO):
        if tuple(t.shape) != tuple(q.shape) or t.dtype != q.dtype or not t.is_contiguous():
            raise ValueError("o and dO must match q")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, Hq, T) or not lse.is_contiguous():
        raise ValueError("lse must be contiguous fp32 [B, Hq, T]")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    fn = lib.ne_attn_bwd_train if q.dtype == torch.bfloat16 else lib.ne_attn_bwd_train_f32
    _check(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(dq), _ptr(dk), _ptr(dv),
              B, T, Hq, Hkv, D, float(theta), _ptr(workspace), workspace.numel() * workspace.element_size(),
              _stream(q)))
    return dq, dk, dv


def attn_bwd_varlen(q, k, v, o, lse, dO, seq_lens, theta: float = 10000.0, workspace=None, dq=None, dk=None,
                    dv=None):
    """Backward over a padded batch (see attn_fwd_varlen): returns (dq, dk, dv); padding
    positions get zero gradients."""
    lib = load()
    B, T, Hq, Hkv, D = _dims(q, k, v)
    _check_lens(seq_lens, B, q.device)
    for t in (o, dO):
        if tuple(t.shape) != tuple(q.shape) or t.dtype != q.dtype or not t.is_contiguous():
            raise ValueError("o and dO must match q")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, Hq, T) or not lse.is_contiguous():
        raise ValueError("lse must be contiguous fp32 [B, Hq, T]")
    if workspace is None:
        workspace = alloc_workspace(B, T, Hq, Hkv, D, q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    fn = lib.ne_attn_bwd_varlen if q.dtype == torch.bfloat16 else lib.ne_attn_bwd_varlen_f32
    _check(fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dO), _ptr(seq_lens), _ptr(dq), _ptr(dk), _ptr(dv),
              B, T, Hq, Hkv, D, float(theta), _ptr(workspace), workspace.numel() * workspace.element_size(),
              _stream(q)))
    return dq, dk, dv


def qkv_prologue(x, gamma, w, Hq: int, Hkv: int, D: int, eps: float = 1e-5, theta: float = 10000.0,
                 rotate: bool = False, q=None, k=None, v=None, workspace=None):
    """RMSNorm (gain gamma) -> projection w [(Hq + 2 Hkv) D, dim] -> q, k, v heads, RoPE
    on q and k when `rotate` (the attention calls take the unrotated form).  x [B, T, dim]
    bf16; returns q [B, T, Hq, D], k and v [B, T, Hkv, D] bf16."""
    lib = load()
    if x.dim() != 3:
        raise ValueError("x must be [B, T, dim]")
    B, T, dim = x.shape
    N = (Hq + 2 * Hkv) * D
    for t in (x, gamma, w):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != torch.bfloat16 or t.device != x.device:
            raise ValueError("x, gamma and w must be contiguous bf16 CUDA tensors on one device")
    if tuple(gamma.shape) != (dim,) or tuple(w.shape) != (N, dim):
        raise ValueError(f"gamma must be [dim] and w [(Hq + 2 Hkv) D, dim] = [{N}, {dim}]")
    q = torch.empty((B, T, Hq, D), dtype=torch.bfloat16, device=x.device) if q is None else q
    k = torch.empty((B, T, Hkv, D), dtype=torch.bfloat16, device=x.device) if k is None else k
    v = torch.empty((B, T, Hkv, D), dtype=torch.bfloat16, device=x.device) if v is None else v
    if workspace is None:
        n = int(lib.ne_qkv_prologue_workspace_size(B, T, dim, Hq, Hkv, D))
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=x.device)
    _check(lib.ne_qkv_prologue(_ptr(x), _ptr(gamma), _ptr(w), _ptr(q), _ptr(k), _ptr(v), B, T, dim, Hq, Hkv, D,
                               float(eps), float(theta), 1 if rotate else 0, _ptr(workspace),
                               workspace.numel() * workspace.element_size(), _stream(x)))
    return q, k, v


def decode_workspace_size(B, T_max, Hq, Hkv, D) -> int:
    return int(load().ne_attn_decode_workspace_size(B, T_max, Hq, Hkv, D))


def attn_decode(q, k_cache, v_cache, seq_lens, theta: float = 10000.0, o=None, lse=None, workspace=None):
    """Decode step: q [B, Hq, D] is the newest token of each sequence (unrotated),
    k_cache / v_cache [B, T_max, Hkv, D] hold positions 0 .. seq_lens[b] - 1 (the newest
    token's key and value included), seq_lens int32 [B] on the device.  Returns
    (o [B, Hq, D], lse [B, Hq] fp32): row seq_lens[b] - 1 of the causal attention."""
    lib = load()
    if q.dim() != 3 or k_cache.dim() != 4 or v_cache.dim() != 4:
        raise ValueError("q must be [B, Hq, D] and the caches [B, T_max, Hkv, D]")
    B, Hq, D = q.shape
    T_max, Hkv = k_cache.shape[1], k_cache.shape[2]
    if tuple(k_cache.shape) != (B, T_max, Hkv, D) or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError(f"caches must be [B, T_max, Hkv, D]; got {tuple(k_cache.shape)}, {tuple(v_cache.shape)}")
    for t in (q, k_cache, v_cache):
        if not t.is_cuda or not t.is_contiguous() or t.dtype != q.dtype:
            raise ValueError("q and the caches must be contiguous CUDA tensors of one dtype")
    if q.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("dtype must be bfloat16 or float32")
    if seq_lens.dtype != torch.int32 or tuple(seq_lens.shape) != (B,) or not seq_lens.is_cuda \
            or not seq_lens.is_contiguous():
        raise ValueError("seq_lens must be a contiguous int32 CUDA tensor [B]")
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device) if lse is None else lse
    need = decode_workspace_size(B, T_max, Hq, Hkv, D)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    fn = lib.ne_attn_decode if q.dtype == torch.bfloat16 else lib.ne_attn_decode_f32
    _check(fn(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(seq_lens), _ptr(o), _ptr(lse), B, T_max, Hq, Hkv, D,
              float(theta), _ptr(workspace), ws_bytes, _stream(q)))
    return o, lse


def get_device_error(device=None) -> int:
    """Synchronise the current stream and return (and clear) the device error status."""
    lib = load()
    s = torch.cuda.current_stream(device).cuda_stream
    return int(lib.ne_get_device_error(ctypes.c_void_p(s)))


def set_wait_timeout_ms(ms: int):
    load().ne_set_wait_timeout_ms(int(ms))


def selftest_wait_timeout(timeout_ms: int = 50):
    lib = load()
    _check(lib.ne_selftest_wait_timeout(int(timeout_ms), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)))


PHASES = ("attn_fwd", "bwd_pre", "attn_bwd", "bwd_post")


def profile_enable(on: bool = True):
    """Diagnostic: record CUDA events around every kernel the calls launch."""
    load().ne_profile_enable(1 if on else 0)


def profile_totals() -> dict:
    """{phase: (total_ms, launches)} since profile_enable(True); synchronises."""
    lib = load()
    ms = (ctypes.c_double * 4)()
    n = (ctypes.c_int * 4)()
    _check(lib.ne_profile_totals(ms, n))
    return {PHASES[i]: (float(ms[i]), int(n[i])) for i in range(4)}


def last_error() -> str:
    return load().ne_last_error().decode()


def shutdown():
    load().ne_shutdown()
