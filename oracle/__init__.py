"""fp64 CPU oracle for causal GQA + RoPE attention (forward and backward).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg may import this module; the product library never does.  It shares
no code with the CUDA path.  The arithmetic lives in ``neattn_ref.cpp`` (plain loops,
OpenMP over heads), built here with the host C++ compiler; this module only
marshals numpy arrays.

Every array is float64.  Layouts: q, o, dO, dq are [B, T, Hq, D]; k, v, dk, dv are
[B, T, Hkv, D]; lse and delta are [B, Hq, T]; probs are [B, Hq, T, T].

Sources (page title, section):
- causal mask j <= i: "Tiny hackable CUDA language model implementation", Core
  Mechanics (causal self-attention bullet);
- grouped-query heads: "NanoEuler: C와 CUDA로 밑바닥부터 구축한 GPT-2 규모의 LLM",
  기술 사양 (GQA bullet) and the model-config table;
- RoPE on queries and keys: same page, 기술 사양 (RoPE bullet);
- the softmax result FlashAttention reaches without the T x T matrix: same page,
  커널 구현;
- backward checked against central finite differences in fp64: same page,
  검증 및 안정성.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "neattn_ref.cpp")
_LIB_PATH = os.path.join(_HERE, "libneattn_ref.so")
_lock = threading.Lock()
_lib = None


def compile_source(src: str, out: str) -> str:
    """Compile one C++ source of the oracle's form into the shared library `out` with
    g++ -O2 -fopenmp (portable flags only)."""
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-fopenmp", "-fPIC", "-shared", src, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle shared library (once; again when the source is newer)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    return compile_source(_SRC, _LIB_PATH)


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            dp = ctypes.POINTER(ctypes.c_double)
            i = ctypes.c_int
            lib.ne_ref_rope_table.argtypes = [dp, dp, i, i, ctypes.c_double]
            lib.ne_ref_rope_apply.argtypes = [dp, dp, i, i, i, i, ctypes.c_double]
            lib.ne_ref_attn_fwd.argtypes = [dp, dp, dp, dp, dp, ctypes.c_void_p, i, i, i, i, i,
                                            ctypes.c_double]
            lib.ne_ref_attn_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, ctypes.c_void_p, i, i, i, i,
                                            i, ctypes.c_double]
            ip = ctypes.POINTER(ctypes.c_int)
            vp = ctypes.c_void_p
            lib.ne_ref_attn_qrows.argtypes = [dp, dp, dp, vp, i, i, ip, i, dp, dp, vp, vp, i, i, i, i, i,
                                              ctypes.c_double]
            lib.ne_ref_attn_krows.argtypes = [dp, dp, dp, dp, i, i, ip, i, dp, dp, i, i, i, i, i,
                                              ctypes.c_double]
            lib.ne_ref_qkv_prologue.argtypes = [dp] * 6 + [i] * 6 + [ctypes.c_double, ctypes.c_double, i]
            for f in (lib.ne_ref_rope_table, lib.ne_ref_rope_apply, lib.ne_ref_attn_fwd,
                      lib.ne_ref_attn_bwd, lib.ne_ref_attn_qrows, lib.ne_ref_attn_krows,
                      lib.ne_ref_num_threads, lib.ne_ref_qkv_prologue):
                f.restype = ctypes.c_int
            lib.ne_ref_num_threads.argtypes = []
            _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def num_threads() -> int:
    """OpenMP threads the oracle uses (OMP_NUM_THREADS, else all host cores)."""
    return int(_load().ne_ref_num_threads())


def rope_table(T: int, D: int, theta: float = 10000.0):
    """cos, sin of t * theta^(-2i/D), each [T, D/2] float64."""
    lib = _load()
    c = np.zeros((T, D // 2), np.float64)
    s = np.zeros((T, D // 2), np.float64)
    if lib.ne_ref_rope_table(_ptr(c), _ptr(s), T, D, float(theta)) != 0:
        raise ValueError("bad rope_table shape")
    return c, s


def rope_apply(x, theta: float = 10000.0) -> np.ndarray:
    """R_t x for x [B, T, H, D] (adjacent-pair rotation)."""
    x = _f64(x)
    B, T, H, D = x.shape
    out = np.zeros_like(x)
    if _load().ne_ref_rope_apply(_ptr(x), _ptr(out), B, T, H, D, float(theta)) != 0:
        raise ValueError("bad rope_apply shape")
    return out


def attn_fwd(q, k, v, theta: float = 10000.0, return_probs: bool = False):
    """O [B,T,Hq,D], LSE [B,Hq,T] (and probs [B,Hq,T,T] if asked)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    if k.shape != (B, T, Hkv, D) or v.shape != k.shape:
        raise ValueError("shape mismatch")
    o = np.zeros_like(q)
    lse = np.zeros((B, Hq, T), np.float64)
    P = np.zeros((B, Hq, T, T), np.float64) if return_probs else None
    rc = _load().ne_ref_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                 P.ctypes.data if P is not None else None,
                                 B, T, Hq, Hkv, D, float(theta))
    if rc != 0:
        raise ValueError("bad attention shape")
    return (o, lse, P) if return_probs else (o, lse)


def attn_bwd(q, k, v, dO, theta: float = 10000.0, return_delta: bool = False):
    """dq [B,T,Hq,D], dk, dv [B,T,Hkv,D] (and delta [B,Hq,T] if asked)."""
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    B, T, Hq, D = q.shape
    Hkv = k.shape[2]
    if k.shape != (B, T, Hkv, D) or v.shape != k.shape or dO.shape != q.shape:
        raise ValueError("shape mismatch")
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    delta = np.zeros((B, Hq, T), np.float64) if return_delta else None
    rc = _load().ne_ref_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dO), _ptr(dq), _ptr(dk), _ptr(dv),
                                 delta.ctypes.data if delta is not None else None,
                                 B, T, Hq, Hkv, D, float(theta))
    if rc != 0:
        raise ValueError("bad attention shape")
    return (dq, dk, dv, delta) if return_delta else (dq, dk, dv)


def _batch(x, b):
    """Batch row b of x (a NumPy array or a CPU tensor of any float dtype) as a
    C-contiguous fp64 array of shape [1, T, H, D]."""
    xb = x[b:b + 1]
    if hasattr(xb, "detach"):          # a tensor: bf16 has no NumPy dtype, widen first
        xb = xb.detach().double().cpu().numpy()
    return np.ascontiguousarray(_f64(xb))


def attn_qrows(q, k, v, dO, b: int, h: int, rows, theta: float = 10000.0):
    """Query rows `rows` of (batch b, query head h), each computed on its own from the
    definitions: O rows [n, D], LSE [n], and with dO also dQ rows [n, D] and Delta [n]
    (None otherwise).  For checks at sizes where the full oracle does not fit."""
    qb, kb, vb = _batch(q, b), _batch(k, b), _batch(v, b)
    _, T, Hq, D = qb.shape
    Hkv = kb.shape[2]
    r = np.ascontiguousarray(np.asarray(rows, np.int32))
    n = r.size
    o = np.zeros((n, D), np.float64)
    lse = np.zeros(n, np.float64)
    dob = _batch(dO, b) if dO is not None else None
    dq = np.zeros((n, D), np.float64) if dO is not None else None
    delta = np.zeros(n, np.float64) if dO is not None else None
    rc = _load().ne_ref_attn_qrows(_ptr(qb), _ptr(kb), _ptr(vb), dob.ctypes.data if dob is not None else None,
                                   0, h, r.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), n, _ptr(o), _ptr(lse),
                                   dq.ctypes.data if dq is not None else None,
                                   delta.ctypes.data if delta is not None else None,
                                   1, T, Hq, Hkv, D, float(theta))
    if rc != 0:
        raise ValueError("bad attn_qrows arguments")
    return o, lse, dq, delta


def attn_krows(q, k, v, dO, b: int, g: int, rows, theta: float = 10000.0):
    """dK and dV rows [n, D] of key rows `rows` of (batch b, kv head g), summed over the
    group's query heads, from the definitions; cheap for rows near the end of the
    sequence (every query row at or after the first requested key is visited)."""
    qb, kb, vb, dob = _batch(q, b), _batch(k, b), _batch(v, b), _batch(dO, b)
    _, T, Hq, D = qb.shape
    Hkv = kb.shape[2]
    r = np.ascontiguousarray(np.asarray(rows, np.int32))
    n = r.size
    dk = np.zeros((n, D), np.float64)
    dv = np.zeros((n, D), np.float64)
    rc = _load().ne_ref_attn_krows(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(dob), 0, g,
                                   r.ctypes.data_as(ctypes.POINTER(ctypes.c_int)), n, _ptr(dk), _ptr(dv),
                                   1, T, Hq, Hkv, D, float(theta))
    if rc != 0:
        raise ValueError("bad attn_krows arguments")
    return dk, dv


def qkv_prologue(x, gamma, w, Hq: int, Hkv: int, D: int, eps: float = 1e-5, theta: float = 10000.0,
                 rotate: bool = True):
    """RMSNorm (gain gamma, no bias) -> one bias-free projection w [(Hq + 2 Hkv) D, dim]
    -> split into q, k, v heads -> RoPE on q and k when `rotate`.  x [B, T, dim];
    returns q [B, T, Hq, D], k and v [B, T, Hkv, D], all float64."""
    x, gamma, w = _f64(x), _f64(gamma), _f64(w)
    B, T, dim = x.shape
    if gamma.shape != (dim,) or w.shape != ((Hq + 2 * Hkv) * D, dim):
        raise ValueError("shape mismatch")
    q = np.zeros((B, T, Hq, D), np.float64)
    k = np.zeros((B, T, Hkv, D), np.float64)
    v = np.zeros((B, T, Hkv, D), np.float64)
    rc = _load().ne_ref_qkv_prologue(_ptr(x), _ptr(gamma), _ptr(w), _ptr(q), _ptr(k), _ptr(v), B, T, dim, Hq,
                                     Hkv, D, float(eps), float(theta), 1 if rotate else 0)
    if rc != 0:
        raise ValueError("bad prologue shape")
    return q, k, v
