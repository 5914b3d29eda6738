"""Test infrastructure only: the fp64 CPU oracle for causal NeoX-rotary attention.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path
(``causal_rope_self_neox_b300``) never does, and shares no code with it.

The arithmetic lives in ``neox_oracle.c`` (plain C, fp64, pthreads); this module
compiles it with gcc when the shared library is missing and wraps it with ctypes.
Every function takes the packed ``qkv[B,S,H,3,D]`` bf16 input as its raw 16-bit
patterns (a ``numpy.uint16`` array), because the oracle widens bf16 to fp64 itself.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "neox_oracle.c")
_LIB = os.path.join(_HERE, "libneox_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``neox_oracle.c`` into ``libneox_oracle.so`` (gcc, -O2, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
                               "-D_POSIX_C_SOURCE=200809L", _SRC, "-o", tmp, "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.neox_oracle_inv_freq.argtypes = [i32, f64, P]
            lib.neox_oracle_inv_freq.restype = None
            lib.neox_oracle_rotate.argtypes = [P, i32, i32, f64, i64, P]
            lib.neox_oracle_rotate.restype = None
            lib.neox_oracle_fwd.argtypes = [P, i32, i32, i32, i32, i32, f64, P, P, i32]
            lib.neox_oracle_fwd.restype = i32
            lib.neox_oracle_fwd_rows.argtypes = [P, i32, i32, i32, i32, i32, f64, P, i64, P, P, i32]
            lib.neox_oracle_fwd_rows.restype = i32
            lib.neox_oracle_probs.argtypes = [P, i32, i32, i32, i32, i32, f64, i32, i32, i32, P]
            lib.neox_oracle_probs.restype = i32
            lib.neox_oracle_decode.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, f64, P, P, i32]
            lib.neox_oracle_decode.restype = i32
            lib.neox_oracle_bwd.argtypes = [P, P, i32, i32, i32, i32, i32, f64, P, i32]
            lib.neox_oracle_bwd.restype = i32
            lib.neox_oracle_qkv_proj.argtypes = [P, P, P, ctypes.c_int64, i32, i32, P, ctypes.c_int64, P, i32]
            lib.neox_oracle_qkv_proj.restype = i32
            lib.neox_oracle_alibi_slopes.argtypes = [i32, P]
            lib.neox_oracle_alibi_slopes.restype = None
            lib.neox_oracle_fwd_alibi.argtypes = [P, i32, i32, i32, i32, P, P, i32]
            lib.neox_oracle_fwd_alibi.restype = i32
            _lib = lib
    return _lib


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1))


def _u16(qkv_bits: np.ndarray, shape) -> np.ndarray:
    a = np.ascontiguousarray(qkv_bits)
    if a.dtype != np.uint16:
        raise TypeError("qkv must be passed as bf16 bit patterns (numpy.uint16)")
    if a.size != int(np.prod(shape)):
        raise ValueError(f"qkv has {a.size} elements, expected {shape}")
    return a


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def inv_freq(rotary_dim: int, base: float) -> np.ndarray:
    """inv_freq[i] = base^(-2i/rotary_dim), i < rotary_dim/2 (fp64)."""
    out = np.zeros(rotary_dim // 2, dtype=np.float64)
    _load().neox_oracle_inv_freq(rotary_dim, float(base), _ptr(out))
    return out


def rotate(x: np.ndarray, pos: int, rotary_dim: int, base: float) -> np.ndarray:
    """Rotate-half rotary embedding of one head vector ``x[D]`` (fp64) at position ``pos``."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    _load().neox_oracle_rotate(_ptr(x), x.shape[0], rotary_dim, float(base), int(pos), _ptr(y))
    return y


def fwd(qkv_bits: np.ndarray, B: int, S: int, H: int, D: int, rotary_dim: int, base: float,
        threads: int | None = None):
    """All rows.  Returns ``(out[B,S,H,D] fp64, lse[B,H,S] fp64)``."""
    q = _u16(qkv_bits, (B, S, H, 3, D))
    out = np.empty((B, S, H, D), dtype=np.float64)
    lse = np.empty((B, H, S), dtype=np.float64)
    rc = _load().neox_oracle_fwd(_ptr(q), B, S, H, D, rotary_dim, float(base), _ptr(out), _ptr(lse),
                                 threads or default_threads())
    if rc != 0:
        raise RuntimeError(f"neox_oracle_fwd failed: {rc}")
    return out, lse


def fwd_rows(qkv_bits: np.ndarray, B: int, S: int, H: int, D: int, rotary_dim: int, base: float,
             rows, threads: int | None = None):
    """Listed rows ``rows[n,3] = (b, h, i)``.  Returns ``(out[n,D], lse[n])`` in fp64."""
    q = _u16(qkv_bits, (B, S, H, 3, D))
    R = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    n = R.shape[0]
    out = np.empty((n, D), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    rc = _load().neox_oracle_fwd_rows(_ptr(q), B, S, H, D, rotary_dim, float(base), _ptr(R), n,
                                      _ptr(out), _ptr(lse), threads or default_threads())
    if rc != 0:
        raise RuntimeError(f"neox_oracle_fwd_rows failed: {rc}")
    return out, lse


def probs(qkv_bits: np.ndarray, B: int, S: int, H: int, D: int, rotary_dim: int, base: float,
          b: int, h: int, i: int) -> np.ndarray:
    """The softmax probability row ``p[0..i]`` of query ``(b, h, i)`` (fp64)."""
    q = _u16(qkv_bits, (B, S, H, 3, D))
    p = np.empty((i + 1,), dtype=np.float64)
    rc = _load().neox_oracle_probs(_ptr(q), B, S, H, D, rotary_dim, float(base), b, h, i, _ptr(p))
    if rc != 0:
        raise RuntimeError(f"neox_oracle_probs failed: {rc}")
    return p


def decode(qkv_new_bits: np.ndarray, k_cache_bits, v_cache_bits, pos, B: int, H: int, Smax: int, D: int,
           rotary_dim: int, base: float = 10000.0, threads: int | None = None):
    """Incremental decode: one new token per sequence against a cache of earlier ones.

    qkv_new_bits: bf16 bits [B,H,3,D] (the new token's packed projections);
    k_cache_bits / v_cache_bits: bf16 bits [B,H,Smax,D], keys NOT rotated (rows p < pos[b]
    are read, the rest ignored; may be None when every pos is 0);
    pos: int [B], the new token's position (= tokens already cached), 0 <= pos < Smax.
    Returns (out fp64 [B,H,D], lse fp64 [B,H]): by definition row pos[b] of the prefill.
    """
    q = _u16(qkv_new_bits, (B, H, 3, D))
    kc = _u16(k_cache_bits, (B, H, Smax, D)) if k_cache_bits is not None else None
    vc = _u16(v_cache_bits, (B, H, Smax, D)) if v_cache_bits is not None else None
    p = np.ascontiguousarray(np.asarray(pos, dtype=np.int32))
    if p.shape != (B,):
        raise ValueError("pos must have shape [B]")
    out = np.zeros((B, H, D), dtype=np.float64)
    lse = np.zeros((B, H), dtype=np.float64)
    rc = _load().neox_oracle_decode(_ptr(q), _ptr(kc) if kc is not None else None,
                                    _ptr(vc) if vc is not None else None, _ptr(p), B, H, Smax, D, rotary_dim,
                                    float(base), _ptr(out), _ptr(lse), threads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle decode failed ({rc})")
    return out, lse


def bwd(qkv_bits: np.ndarray, dout_bits: np.ndarray, B: int, S: int, H: int, D: int, rotary_dim: int,
        base: float = 10000.0, threads: int | None = None) -> np.ndarray:
    """Gradient of sum(dout * out) with respect to the packed qkv, out being the forward.

    qkv_bits: bf16 bits [B,S,H,3,D]; dout_bits: bf16 bits [B,S,H,D].
    Returns dqkv fp64 [B,S,H,3,D] (slot 0 = dq, 1 = dk, 2 = dv), exact in fp64.
    """
    q = _u16(qkv_bits, (B, S, H, 3, D))
    g = _u16(dout_bits, (B, S, H, D))
    dqkv = np.zeros((B, S, H, 3, D), dtype=np.float64)
    rc = _load().neox_oracle_bwd(_ptr(q), _ptr(g), B, S, H, D, rotary_dim, float(base), _ptr(dqkv),
                                 threads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle backward failed ({rc})")
    return dqkv


def qkv_proj(x_bits: np.ndarray, w_bits: np.ndarray, bias_bits=None, rows=None, threads: int | None = None):
    """The fused query_key_value projection in fp64: ``x[M,K] @ w[K,N] + bias[N]`` from the
    bf16 bits (``w`` laid out [hidden, H, 3, D] flattened to [K, N]).  ``rows``: token rows
    to compute (default all).  Returns fp64 ``[n_rows, N]``."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    w = np.ascontiguousarray(w_bits, dtype=np.uint16)
    M, K = x.shape
    K2, N = w.shape
    if K2 != K:
        raise ValueError("x and w disagree on the hidden size")
    b = None if bias_bits is None else np.ascontiguousarray(bias_bits, dtype=np.uint16)
    if b is not None and b.shape != (N,):
        raise ValueError("bias must have N entries")
    R = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1))
    n = M if R is None else R.shape[0]
    out = np.empty((n, N), dtype=np.float64)
    rc = _load().neox_oracle_qkv_proj(_ptr(x), _ptr(w), None if b is None else _ptr(b), M, K, N,
                                      None if R is None else _ptr(R), 0 if R is None else n, _ptr(out),
                                      threads or default_threads())
    if rc != 0:
        raise RuntimeError(f"neox_oracle_qkv_proj failed: {rc}")
    return out


def round_bf16(a: np.ndarray) -> np.ndarray:
    """fp64 -> nearest bf16 (ties to even) -> fp64, through torch's conversion."""
    import torch

    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64)).to(torch.bfloat16).double().numpy()


def qkv_proj_rotated(x_bits: np.ndarray, w_bits: np.ndarray, bias_bits, B: int, S: int, H: int, D: int,
                     rotary_dim: int, base: float = 10000.0, rows=None, threads: int | None = None,
                     bf16_steps: bool = False) -> np.ndarray:
    """The projection followed by the rotary embedding of its query and key slots, in fp64.

    Tokens are ``x`` rows ``t = b*S + s`` (position ``s``).  Each token's projection
    ``qkv_proj`` row is read as ``[H, 3, D]`` (slot 0 = query, 1 = key, 2 = value); the query
    and key vectors of every head are rotated by ``rotate`` at the token's position, the
    value vectors are left as they are.  ``rows``: token rows to compute (default all).
    ``bf16_steps``: round the projection to bf16 before the rotation and the result after
    it, as a model that holds its activations in bf16 does (default: exact throughout).
    Returns fp64 ``[n_rows, H, 3, D]``.
    """
    if x_bits.shape[0] != B * S:
        raise ValueError("x must hold B*S token rows")
    y = qkv_proj(x_bits, w_bits, bias_bits, rows=rows, threads=threads).reshape(-1, H, 3, D)
    if bf16_steps:
        y = round_bf16(y)
    toks = np.arange(B * S, dtype=np.int64) if rows is None else np.asarray(rows, dtype=np.int64).reshape(-1)
    if rotary_dim:
        for n, t in enumerate(toks):
            pos = int(t % S)
            for h in range(H):
                for slot in (0, 1):
                    y[n, h, slot] = rotate(y[n, h, slot], pos, rotary_dim, base)
    return round_bf16(y) if bf16_steps else y


def alibi_slopes(H: int) -> np.ndarray:
    """The ALiBi slope of each of H heads (fp64)."""
    out = np.zeros(H, dtype=np.float64)
    _load().neox_oracle_alibi_slopes(H, _ptr(out))
    return out


def fwd_alibi(qkv_bits: np.ndarray, B: int, S: int, H: int, D: int, threads: int | None = None):
    """Causal attention with the ALiBi bias -m_h (i - j) and no rotation.

    qkv_bits: bf16 bits [B,S,H,3,D].  Returns (out fp64 [B,S,H,D], lse fp64 [B,H,S])."""
    q = _u16(qkv_bits, (B, S, H, 3, D))
    out = np.zeros((B, S, H, D), dtype=np.float64)
    lse = np.zeros((B, H, S), dtype=np.float64)
    rc = _load().neox_oracle_fwd_alibi(_ptr(q), B, S, H, D, _ptr(out), _ptr(lse), threads or default_threads())
    if rc != 0:
        raise ValueError(f"oracle ALiBi forward failed ({rc})")
    return out, lse
