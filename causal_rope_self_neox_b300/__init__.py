"""causal_rope_self_neox_b300 -- B300 (sm_103a) causal NeoX-rotary self-attention forward.

The compute lives in the CUDA library ``libneox_attn.so`` (built in-tree from
``csrc/`` by ``build.py``); this module is argument marshalling over its C ABI
(``include/neox_attn.h``) with the same entry-point names, plus a torch
convenience wrapper that allocates the outputs.  There is no CPU fallback: if the
library is missing or the device is not a B300, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libneox_attn.so")

NEOX_OK = 0
NEOX_ERR_INVALID_ARG = -1
NEOX_ERR_UNSUPPORTED_HEAD_DIM = -2
NEOX_ERR_MISALIGNED = -3
NEOX_ERR_CUDA = -4
NEOX_ERR_DEVICE_TIMEOUT = -5
NEOX_ERR_NO_DEVICE_SUPPORT = -6
NEOX_ERR_TOO_LARGE = -7
NEOX_ERR_DEVICE_BAD_POSITION = -8
NEOX_ERR_DEVICE_RANGE = -9

NEOX_ROTATION_AUTO = 0
NEOX_ROTATION_FUSED = 1
NEOX_ROTATION_PRE = 2

EXPORTS = ("neox_attn_fwd", "neox_attn_fwd_ex", "neox_attn_fwd_alibi", "neox_attn_qkv_proj", "neox_attn_fwd_simple", "neox_attn_get_device_error", "neox_attn_status_string",
           "neox_attn_last_cuda_error", "neox_attn_release", "neox_attn_selftest_wait_timeout",
           "neox_attn_version", "neox_attn_fwd_noalloc", "neox_attn_decode", "neox_attn_bwd")

_lock = threading.Lock()
_lib = None


class NeoxAttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load the CUDA library (raises OSError if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise OSError(f"{path} is missing: build it with `python -m causal_rope_self_neox_b300.build`")
            lib = ctypes.CDLL(path)
            P, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
            fwd_args = [P, i32, i32, i32, i32, i32, f32, P, P, P]
            for name in ("neox_attn_fwd", "neox_attn_fwd_simple", "neox_attn_fwd_noalloc"):
                getattr(lib, name).argtypes = fwd_args
                getattr(lib, name).restype = i32
            lib.neox_attn_fwd_ex.argtypes = [P, i32, i32, i32, i32, i32, f32, P, P, i32, P]
            lib.neox_attn_fwd_ex.restype = i32
            lib.neox_attn_fwd_alibi.argtypes = [P, i32, i32, i32, i32, P, P, P]
            lib.neox_attn_fwd_alibi.restype = i32
            lib.neox_attn_qkv_proj.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32, f32, P, P]
            lib.neox_attn_qkv_proj.restype = i32
            lib.neox_attn_decode.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, f32, P, P, P]
            lib.neox_attn_decode.restype = i32
            lib.neox_attn_bwd.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, f32, P, P]
            lib.neox_attn_bwd.restype = i32
            lib.neox_attn_get_device_error.argtypes = []
            lib.neox_attn_get_device_error.restype = i32
            lib.neox_attn_status_string.argtypes = [i32]
            lib.neox_attn_status_string.restype = ctypes.c_char_p
            lib.neox_attn_last_cuda_error.argtypes = []
            lib.neox_attn_last_cuda_error.restype = i32
            lib.neox_attn_release.argtypes = []
            lib.neox_attn_release.restype = None
            lib.neox_attn_selftest_wait_timeout.argtypes = [i64, P]
            lib.neox_attn_selftest_wait_timeout.restype = i32
            lib.neox_attn_version.argtypes = []
            lib.neox_attn_version.restype = i32
            _lib = lib
    return _lib


# ------------------------------------------------------------- raw C ABI ----

def neox_attn_fwd(qkv_ptr: int, B: int, S: int, H: int, D: int, rotary_dim: int, rotary_base: float,
                  out_ptr: int, lse_ptr: int, stream: int = 0) -> int:
    """Raw call: device pointers and a cudaStream_t handle as integers; returns a status."""
    return load_library().neox_attn_fwd(qkv_ptr, B, S, H, D, rotary_dim, rotary_base, out_ptr, lse_ptr, stream)


def neox_attn_fwd_ex(qkv_ptr: int, B: int, S: int, H: int, D: int, rotary_dim: int, rotary_base: float,
                     out_ptr: int, lse_ptr: int, rotation: int, stream: int = 0) -> int:
    """Raw call with the rotation placement (NEOX_ROTATION_AUTO / _FUSED / _PRE)."""
    return load_library().neox_attn_fwd_ex(qkv_ptr, B, S, H, D, rotary_dim, rotary_base, out_ptr, lse_ptr, rotation,
                                           stream)


def neox_attn_fwd_alibi(qkv_ptr: int, B: int, S: int, H: int, D: int, out_ptr: int, lse_ptr: int,
                        stream: int = 0) -> int:
    """Raw call of the ALiBi forward (no rotation; linear distance bias per head)."""
    return load_library().neox_attn_fwd_alibi(qkv_ptr, B, S, H, D, out_ptr, lse_ptr, stream)


def neox_attn_qkv_proj(x_ptr: int, w_ptr: int, bias_ptr: int, B: int, S: int, hidden: int, H: int, D: int,
                       rotary_dim: int, rotary_base: float, qkv_ptr: int, stream: int = 0) -> int:
    """Raw call of the query_key_value projection (bias_ptr 0 = no bias; rotary_dim > 0
    rotates the query/key slots of the result)."""
    return load_library().neox_attn_qkv_proj(x_ptr, w_ptr, bias_ptr or None, B, S, hidden, H, D, rotary_dim,
                                             rotary_base, qkv_ptr, stream)


def neox_attn_fwd_simple(qkv_ptr: int, B: int, S: int, H: int, D: int, rotary_dim: int, rotary_base: float,
                         out_ptr: int, lse_ptr: int, stream: int = 0) -> int:
    return load_library().neox_attn_fwd_simple(qkv_ptr, B, S, H, D, rotary_dim, rotary_base, out_ptr, lse_ptr,
                                               stream)


def neox_attn_fwd_noalloc(qkv_ptr: int, B: int, S: int, H: int, D: int, rotary_dim: int, rotary_base: float,
                          out_ptr: int, lse_ptr: int, stream: int = 0) -> int:
    """Raw call of the allocation-free variant (fixed 8 MiB cos/sin table inside the
    library, S * rotary_dim/2 <= 1048576): for callers that cannot let the library
    cudaMalloc.  Calls that overlap on the GPU share that table and race."""
    return load_library().neox_attn_fwd_noalloc(qkv_ptr, B, S, H, D, rotary_dim, rotary_base, out_ptr, lse_ptr,
                                                stream)


def neox_attn_decode(qkv_new_ptr: int, k_cache_ptr: int, v_cache_ptr: int, pos_ptr: int, B: int, H: int, Smax: int,
                     D: int, rotary_dim: int, rotary_base: float, out_ptr: int, lse_ptr: int, stream: int = 0) -> int:
    """Raw call of the incremental decode (one new token per sequence against a K/V cache)."""
    return load_library().neox_attn_decode(qkv_new_ptr, k_cache_ptr, v_cache_ptr, pos_ptr, B, H, Smax, D, rotary_dim,
                                           rotary_base, out_ptr, lse_ptr, stream)


def neox_attn_bwd(qkv_ptr: int, out_ptr: int, lse_ptr: int, dout_ptr: int, B: int, S: int, H: int, D: int,
                  rotary_dim: int, rotary_base: float, dqkv_ptr: int, stream: int = 0) -> int:
    """Raw call of the backward (dq, dk, dv of the packed qkv from dout and the forward's out, lse)."""
    return load_library().neox_attn_bwd(qkv_ptr, out_ptr, lse_ptr, dout_ptr, B, S, H, D, rotary_dim, rotary_base,
                                        dqkv_ptr, stream)


def neox_attn_get_device_error() -> int:
    return load_library().neox_attn_get_device_error()


def neox_attn_status_string(status: int) -> str:
    return load_library().neox_attn_status_string(status).decode()


def status_string(status: int) -> str:
    try:
        return neox_attn_status_string(status)
    except OSError:
        return "library not loaded"


def neox_attn_last_cuda_error() -> int:
    return load_library().neox_attn_last_cuda_error()


def neox_attn_release() -> None:
    load_library().neox_attn_release()


def neox_attn_selftest_wait_timeout(timeout_ns: int, stream: int = 0) -> int:
    return load_library().neox_attn_selftest_wait_timeout(timeout_ns, stream)


def neox_attn_version() -> int:
    return load_library().neox_attn_version()


# ----------------------------------------------------- torch convenience ----

def attn_fwd(qkv, rotary_dim: int, rotary_base: float = 10000.0, out=None, lse=None, stream=None,
             kernel: str = "default", rotation: int = NEOX_ROTATION_AUTO):
    """Causal NeoX-rotary attention forward on CUDA tensors.

    ``qkv``: bf16 ``[B, S, H, 3, D]`` contiguous on a CUDA device.  Returns
    ``(out[B,S,H,D] bf16, lse[B,H,S] fp32)``; ``out``/``lse`` may be passed in.
    ``rotation`` places the rotary embedding (NEOX_ROTATION_AUTO / _FUSED / _PRE, see
    ``neox_attn_fwd_ex``); ``kernel="simple"`` runs the plain cross-check kernel.
    torch only allocates memory and supplies the stream; the library computes.
    """
    import torch

    if qkv.dim() != 5 or qkv.shape[3] != 3 or qkv.dtype != torch.bfloat16 or not qkv.is_cuda:
        raise ValueError("qkv must be a CUDA bf16 tensor of shape [B, S, H, 3, D]")
    if not qkv.is_contiguous():
        raise ValueError("qkv must be contiguous")
    B, S, H, _, D = qkv.shape
    if out is None:
        out = torch.empty((B, S, H, D), dtype=torch.bfloat16, device=qkv.device)
    if lse is None:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=qkv.device)
    if stream is None:
        stream = torch.cuda.current_stream(qkv.device)
    with torch.cuda.device(qkv.device):
        if kernel == "default":
            rc = neox_attn_fwd_ex(qkv.data_ptr(), B, S, H, D, rotary_dim, float(rotary_base), out.data_ptr(),
                                  lse.data_ptr(), rotation, stream.cuda_stream)
        else:
            rc = neox_attn_fwd_simple(qkv.data_ptr(), B, S, H, D, rotary_dim, float(rotary_base), out.data_ptr(),
                                      lse.data_ptr(), stream.cuda_stream)
    if rc != NEOX_OK:
        raise NeoxAttnError(rc, "neox_attn_fwd")
    return out, lse


def attn_fwd_alibi(qkv, out=None, lse=None, stream=None):
    """Causal attention with the ALiBi bias (no rotation) on CUDA tensors: ``qkv`` bf16
    ``[B, S, H, 3, D]``.  Returns ``(out[B,S,H,D] bf16, lse[B,H,S] fp32)``."""
    import torch

    if qkv.dim() != 5 or qkv.shape[3] != 3 or qkv.dtype != torch.bfloat16 or not qkv.is_cuda:
        raise ValueError("qkv must be a CUDA bf16 tensor of shape [B, S, H, 3, D]")
    if not qkv.is_contiguous():
        raise ValueError("qkv must be contiguous")
    B, S, H, _, D = qkv.shape
    if out is None:
        out = torch.empty((B, S, H, D), dtype=torch.bfloat16, device=qkv.device)
    if lse is None:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=qkv.device)
    if stream is None:
        stream = torch.cuda.current_stream(qkv.device)
    with torch.cuda.device(qkv.device):
        rc = neox_attn_fwd_alibi(qkv.data_ptr(), B, S, H, D, out.data_ptr(), lse.data_ptr(), stream.cuda_stream)
    if rc != NEOX_OK:
        raise NeoxAttnError(rc, "neox_attn_fwd_alibi")
    return out, lse


def qkv_proj(x, w, bias, B: int, S: int, H: int, D: int, rotary_dim: int = 0, rotary_base: float = 10000.0,
             out=None, stream=None):
    """The query_key_value projection on CUDA tensors: ``x`` bf16 ``[B*S, hidden]`` (or
    ``[B, S, hidden]``), ``w`` bf16 ``[hidden, H, 3, D]`` (or ``[hidden, 3*H*D]``), ``bias``
    bf16 ``[3*H*D]`` or None.  Returns the packed ``qkv[B, S, H, 3, D]`` bf16, its query and
    key slots rotated when ``rotary_dim > 0``."""
    import torch

    for name, t in (("x", x), ("w", w)) + ((("bias", bias),) if bias is not None else ()):
        if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA bf16 tensor")
    hidden = x.shape[-1]
    if x.numel() != B * S * hidden or w.numel() != hidden * 3 * H * D or w.shape[0] != hidden:
        raise ValueError("x must be [B*S, hidden] and w [hidden, H, 3, D]")
    if bias is not None and bias.numel() != 3 * H * D:
        raise ValueError("bias must have 3*H*D entries")
    if out is None:
        out = torch.empty((B, S, H, 3, D), dtype=torch.bfloat16, device=x.device)
    if stream is None:
        stream = torch.cuda.current_stream(x.device)
    with torch.cuda.device(x.device):
        rc = neox_attn_qkv_proj(x.data_ptr(), w.data_ptr(), 0 if bias is None else bias.data_ptr(), B, S, hidden, H,
                                D, rotary_dim, rotary_base, out.data_ptr(), stream.cuda_stream)
    if rc != NEOX_OK:
        raise NeoxAttnError(rc, "neox_attn_qkv_proj")
    return out


def attn_decode(qkv_new, k_cache, v_cache, pos, rotary_dim: int, rotary_base: float = 10000.0, out=None, lse=None,
                stream=None):
    """Incremental decode on CUDA tensors: ``qkv_new`` bf16 ``[B,H,3,D]``, caches bf16
    ``[B,H,Smax,D]`` (keys not rotated; row ``pos[b]`` is overwritten with the new k/v),
    ``pos`` int32 ``[B]`` on the device.  Returns ``(out[B,H,D] bf16, lse[B,H] fp32)``."""
    import torch

    if qkv_new.dim() != 4 or qkv_new.shape[2] != 3 or qkv_new.dtype != torch.bfloat16 or not qkv_new.is_cuda:
        raise ValueError("qkv_new must be a CUDA bf16 tensor of shape [B, H, 3, D]")
    B, H, _, D = qkv_new.shape
    for c in (k_cache, v_cache):
        if c.dim() != 4 or c.shape[0] != B or c.shape[1] != H or c.shape[3] != D or c.dtype != torch.bfloat16 \
                or not c.is_cuda or not c.is_contiguous():
            raise ValueError("caches must be contiguous CUDA bf16 tensors of shape [B, H, Smax, D]")
    if pos.dtype != torch.int32 or pos.shape != (B,) or not pos.is_cuda:
        raise ValueError("pos must be a CUDA int32 tensor of shape [B]")
    if not qkv_new.is_contiguous():
        raise ValueError("qkv_new must be contiguous")
    Smax = k_cache.shape[2]
    if out is None:
        out = torch.empty((B, H, D), dtype=torch.bfloat16, device=qkv_new.device)
    if lse is None:
        lse = torch.empty((B, H), dtype=torch.float32, device=qkv_new.device)
    if stream is None:
        stream = torch.cuda.current_stream(qkv_new.device)
    with torch.cuda.device(qkv_new.device):
        rc = neox_attn_decode(qkv_new.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), pos.data_ptr(), B, H, Smax,
                              D, rotary_dim, float(rotary_base), out.data_ptr(), lse.data_ptr(), stream.cuda_stream)
    if rc != NEOX_OK:
        raise NeoxAttnError(rc, "neox_attn_decode")
    return out, lse


def attn_bwd(qkv, out, lse, dout, rotary_dim: int, rotary_base: float = 10000.0, dqkv=None, stream=None):
    """Backward on CUDA tensors: ``qkv`` bf16 ``[B,S,H,3,D]``, the forward's ``out`` bf16
    ``[B,S,H,D]`` and ``lse`` fp32 ``[B,H,S]``, ``dout`` bf16 ``[B,S,H,D]``.  Returns
    ``dqkv`` bf16 ``[B,S,H,3,D]`` (slot 0 = dq, 1 = dk, 2 = dv)."""
    import torch

    if qkv.dim() != 5 or qkv.shape[3] != 3 or qkv.dtype != torch.bfloat16 or not qkv.is_cuda:
        raise ValueError("qkv must be a CUDA bf16 tensor of shape [B, S, H, 3, D]")
    B, S, H, _, D = qkv.shape
    for t, shape, dt in ((out, (B, S, H, D), torch.bfloat16), (dout, (B, S, H, D), torch.bfloat16),
                         (lse, (B, H, S), torch.float32)):
        if tuple(t.shape) != shape or t.dtype != dt or not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"expected a contiguous CUDA {dt} tensor of shape {list(shape)}")
    if not qkv.is_contiguous():
        raise ValueError("qkv must be contiguous")
    if dqkv is None:
        dqkv = torch.empty_like(qkv)
    if stream is None:
        stream = torch.cuda.current_stream(qkv.device)
    with torch.cuda.device(qkv.device):
        rc = neox_attn_bwd(qkv.data_ptr(), out.data_ptr(), lse.data_ptr(), dout.data_ptr(), B, S, H, D, rotary_dim,
                           float(rotary_base), dqkv.data_ptr(), stream.cuda_stream)
    if rc != NEOX_OK:
        raise NeoxAttnError(rc, "neox_attn_bwd")
    return dqkv


def check_device_error() -> None:
    """Raise if a kernel's bounded wait ran out since the last check (synchronizes first)."""
    import torch

    torch.cuda.synchronize()
    rc = neox_attn_get_device_error()
    if rc != NEOX_OK:
        raise NeoxAttnError(rc, "device")
