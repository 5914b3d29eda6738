"""The C ABI without a GPU: the library loads, exports what the header declares, and
rejects bad arguments before touching CUDA (pointers here are never dereferenced)."""
import ctypes
import os
import re

import pytest
import torch

import causal_rope_self_neox_b300 as na
from causal_rope_self_neox_b300 import build as nb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "neox_attn.h")


@pytest.fixture(scope="module")
def lib():
    nb.build()
    return na.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(neox_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    assert "neox_attn_fwd" in names and "neox_attn_get_device_error" in names
    assert set(names) == set(na.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    assert na.neox_attn_status_string(na.NEOX_OK) == "ok"
    assert "head dim" in na.neox_attn_status_string(na.NEOX_ERR_UNSUPPORTED_HEAD_DIM)
    assert na.neox_attn_status_string(12345) == "unknown status"
    assert na.neox_attn_version() >= 100


A = 0x10000000  # fake, 16-byte aligned device addresses: validation never dereferences them
OUT = 0x20000000
LSE = 0x30000000


@pytest.mark.parametrize("args,status", [
    ((0, 1, 128, 2, 64, 16, 1e4, OUT, LSE), na.NEOX_ERR_INVALID_ARG),          # null qkv
    ((A, 1, 128, 2, 64, 16, 1e4, 0, LSE), na.NEOX_ERR_INVALID_ARG),            # null out
    ((A, 1, 128, 2, 64, 16, 1e4, OUT, 0), na.NEOX_ERR_INVALID_ARG),            # null lse
    ((A, 0, 128, 2, 64, 16, 1e4, OUT, LSE), na.NEOX_ERR_INVALID_ARG),          # B = 0
    ((A, 1, 0, 2, 64, 16, 1e4, OUT, LSE), na.NEOX_ERR_INVALID_ARG),            # S = 0
    ((A, 1, 128, 0, 64, 16, 1e4, OUT, LSE), na.NEOX_ERR_INVALID_ARG),          # H = 0
    ((A, 1, 128, 2, 80, 16, 1e4, OUT, LSE), na.NEOX_ERR_UNSUPPORTED_HEAD_DIM),  # D = 80
    ((A, 1, 128, 2, 256, 16, 1e4, OUT, LSE), na.NEOX_ERR_UNSUPPORTED_HEAD_DIM),
    ((A, 1, 128, 2, 64, 15, 1e4, OUT, LSE), na.NEOX_ERR_INVALID_ARG),          # odd rotary_dim
    ((A, 1, 128, 2, 64, 66, 1e4, OUT, LSE), na.NEOX_ERR_INVALID_ARG),          # rotary_dim > D
    ((A, 1, 128, 2, 64, -2, 1e4, OUT, LSE), na.NEOX_ERR_INVALID_ARG),
    ((A, 1, 128, 2, 64, 16, 0.0, OUT, LSE), na.NEOX_ERR_INVALID_ARG),          # base <= 0
    ((A, 1, 128, 2, 64, 16, float("inf"), OUT, LSE), na.NEOX_ERR_INVALID_ARG),
    ((A, 1, 128, 2, 64, 16, float("nan"), OUT, LSE), na.NEOX_ERR_INVALID_ARG),
    ((A + 8, 1, 128, 2, 64, 16, 1e4, OUT, LSE), na.NEOX_ERR_MISALIGNED),      # qkv not 16-B aligned
    ((A, 1, 128, 2, 64, 16, 1e4, OUT + 2, LSE), na.NEOX_ERR_MISALIGNED),
    ((A, 1, 128, 2, 64, 16, 1e4, OUT, LSE + 2), na.NEOX_ERR_MISALIGNED),
    ((A, 1, 128, 2, 64, 16, 1e4, A + 4096, LSE), na.NEOX_ERR_INVALID_ARG),     # out overlaps qkv
    ((A, 1, 128, 2, 64, 16, 1e4, OUT, A + 64), na.NEOX_ERR_INVALID_ARG),       # lse overlaps qkv
    ((A, 1 << 20, 1 << 20, 64, 128, 16, 1e4, OUT, LSE), na.NEOX_ERR_INVALID_ARG),  # too large
])
@pytest.mark.parametrize("entry", ["neox_attn_fwd", "neox_attn_fwd_simple"])
def test_invalid_arguments_rejected_before_cuda(lib, entry, args, status):
    fn = getattr(na, entry)
    assert fn(*args, stream=0) == status


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU error path")
def test_valid_arguments_without_a_gpu_report_a_cuda_error(lib):
    rc = na.neox_attn_fwd(A, 1, 128, 2, 64, 16, 1e4, OUT, LSE, stream=0)
    assert rc in (na.NEOX_ERR_CUDA, na.NEOX_ERR_NO_DEVICE_SUPPORT)
    assert na.neox_attn_selftest_wait_timeout(1000, 0) in (na.NEOX_ERR_CUDA, na.NEOX_ERR_NO_DEVICE_SUPPORT)
    assert na.neox_attn_selftest_wait_timeout(10, 0) == na.NEOX_ERR_INVALID_ARG


def test_torch_wrapper_rejects_cpu_tensors(lib):
    x = torch.zeros((1, 4, 1, 3, 64), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        na.attn_fwd(x, 16)


# ---- decode: neox_attn_decode(qkv_new, k_cache, v_cache, pos, B, H, Smax, D, r, base, out, lse)
KC = 0x40000000
VC = 0x50000000
POS = 0x60000000


@pytest.mark.parametrize("args,status", [
    ((0, KC, VC, POS, 2, 4, 256, 64, 16, 1e4, OUT, LSE), na.NEOX_ERR_INVALID_ARG),    # null qkv_new
    ((A, 0, VC, POS, 2, 4, 256, 64, 16, 1e4, OUT, LSE), na.NEOX_ERR_INVALID_ARG),     # null k_cache
    ((A, KC, 0, POS, 2, 4, 256, 64, 16, 1e4, OUT, LSE), na.NEOX_ERR_INVALID_ARG),     # null v_cache
    ((A, KC, VC, 0, 2, 4, 256, 64, 16, 1e4, OUT, LSE), na.NEOX_ERR_INVALID_ARG),      # null pos
    ((A, KC, VC, POS, 2, 4, 256, 64, 16, 1e4, 0, LSE), na.NEOX_ERR_INVALID_ARG),      # null out
    ((A, KC, VC, POS, 0, 4, 256, 64, 16, 1e4, OUT, LSE), na.NEOX_ERR_INVALID_ARG),    # B = 0
    ((A, KC, VC, POS, 2, 0, 256, 64, 16, 1e4, OUT, LSE), na.NEOX_ERR_INVALID_ARG),    # H = 0
    ((A, KC, VC, POS, 2, 4, 0, 64, 16, 1e4, OUT, LSE), na.NEOX_ERR_INVALID_ARG),      # Smax = 0
    ((A, KC, VC, POS, 70000, 1, 16, 64, 16, 1e4, OUT, LSE), na.NEOX_ERR_INVALID_ARG),  # B > 65535
    ((A, KC, VC, POS, 2, 4, 256, 80, 16, 1e4, OUT, LSE), na.NEOX_ERR_UNSUPPORTED_HEAD_DIM),
    ((A, KC, VC, POS, 2, 4, 256, 64, 15, 1e4, OUT, LSE), na.NEOX_ERR_INVALID_ARG),    # odd rotary_dim
    ((A, KC, VC, POS, 2, 4, 256, 64, 16, -1.0, OUT, LSE), na.NEOX_ERR_INVALID_ARG),   # base <= 0
    ((A, KC + 8, VC, POS, 2, 4, 256, 64, 16, 1e4, OUT, LSE), na.NEOX_ERR_MISALIGNED),  # k_cache 8-B aligned
    ((A, KC, VC, POS + 2, 2, 4, 256, 64, 16, 1e4, OUT, LSE), na.NEOX_ERR_MISALIGNED),  # pos 2-B aligned
    ((A, KC, KC + 4096, POS, 2, 4, 256, 64, 16, 1e4, OUT, LSE), na.NEOX_ERR_INVALID_ARG),  # caches overlap
    ((A, KC, VC, POS, 2, 4, 256, 64, 16, 1e4, KC + 64, LSE), na.NEOX_ERR_INVALID_ARG),  # out inside k_cache
    ((A, KC, VC, POS, 1 << 10, 1 << 10, 1 << 20, 128, 16, 1e4, OUT, LSE), na.NEOX_ERR_INVALID_ARG),  # too large
])
def test_decode_invalid_arguments_rejected_before_cuda(lib, args, status):
    assert na.neox_attn_decode(*args, stream=0) == status


def test_decode_status_string(lib):
    assert "position" in na.neox_attn_status_string(na.NEOX_ERR_DEVICE_BAD_POSITION)


# ---- backward: neox_attn_bwd(qkv, out, lse, dout, B, S, H, D, r, base, dqkv)
GD = 0x70000000
DQ = 0x80000000


@pytest.mark.parametrize("args,status", [
    ((0, OUT, LSE, GD, 2, 256, 4, 64, 16, 1e4, DQ), na.NEOX_ERR_INVALID_ARG),        # null qkv
    ((A, 0, LSE, GD, 2, 256, 4, 64, 16, 1e4, DQ), na.NEOX_ERR_INVALID_ARG),          # null out
    ((A, OUT, 0, GD, 2, 256, 4, 64, 16, 1e4, DQ), na.NEOX_ERR_INVALID_ARG),          # null lse
    ((A, OUT, LSE, 0, 2, 256, 4, 64, 16, 1e4, DQ), na.NEOX_ERR_INVALID_ARG),         # null dout
    ((A, OUT, LSE, GD, 2, 256, 4, 64, 16, 1e4, 0), na.NEOX_ERR_INVALID_ARG),         # null dqkv
    ((A, OUT, LSE, GD, 0, 256, 4, 64, 16, 1e4, DQ), na.NEOX_ERR_INVALID_ARG),        # B = 0
    ((A, OUT, LSE, GD, 2, 256, 4, 80, 16, 1e4, DQ), na.NEOX_ERR_UNSUPPORTED_HEAD_DIM),
    ((A, OUT, LSE, GD, 2, 256, 4, 64, 15, 1e4, DQ), na.NEOX_ERR_INVALID_ARG),        # odd rotary_dim
    ((A, OUT, LSE, GD, 2, 256, 4, 64, 16, 0.0, DQ), na.NEOX_ERR_INVALID_ARG),        # base <= 0
    ((A, OUT, LSE, GD + 8, 2, 256, 4, 64, 16, 1e4, DQ), na.NEOX_ERR_MISALIGNED),     # dout 8-B aligned
    ((A, OUT, LSE, GD, 2, 256, 4, 64, 16, 1e4, DQ + 4), na.NEOX_ERR_MISALIGNED),     # dqkv 4-B aligned
    ((A, OUT, LSE, GD, 2, 256, 4, 64, 16, 1e4, A + 4096), na.NEOX_ERR_INVALID_ARG),  # dqkv overlaps qkv
    ((A, OUT, LSE, GD, 2, 256, 4, 64, 16, 1e4, GD), na.NEOX_ERR_INVALID_ARG),        # dqkv on dout
])
def test_bwd_invalid_arguments_rejected_before_cuda(lib, args, status):
    assert na.neox_attn_bwd(*args, stream=0) == status


def test_rotation_placement_is_validated_before_any_cuda_call(lib):
    # an unknown placement, and the pre-rotated one where it does not apply (rotary_dim neither
    # a multiple of 16 nor 24, or no rotary dims), are rejected without touching the (fake)
    # device addresses
    s = 0
    assert na.neox_attn_fwd_ex(A, 1, 128, 2, 64, 16, 1e4, OUT, LSE, 3, s) == na.NEOX_ERR_INVALID_ARG
    assert na.neox_attn_fwd_ex(A, 1, 128, 2, 64, 16, 1e4, OUT, LSE, -1, s) == na.NEOX_ERR_INVALID_ARG
    assert na.neox_attn_fwd_ex(A, 1, 128, 2, 96, 40, 1e4, OUT, LSE, na.NEOX_ROTATION_PRE, s) \
        == na.NEOX_ERR_INVALID_ARG
    assert na.neox_attn_fwd_ex(A, 1, 128, 2, 64, 0, 1e4, OUT, LSE, na.NEOX_ROTATION_PRE, s) \
        == na.NEOX_ERR_INVALID_ARG
    # and the usual argument checks still apply first-class
    assert na.neox_attn_fwd_ex(0, 1, 128, 2, 64, 16, 1e4, OUT, LSE, na.NEOX_ROTATION_FUSED, s) \
        == na.NEOX_ERR_INVALID_ARG
