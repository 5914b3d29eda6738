"""The pins must catch plausible mistakes in the oracle.

Each case copies ``oracle/neox_oracle.c`` to a temporary directory, plants one
mistake by text substitution (a flipped sign, a wrong index or denominator, a
dropped term, a swapped operand, an off-by-one position, a mask without the
diagonal), builds that copy with gcc, and checks that the dense brute force or
the two-token worked example or the rotation worked example (all independent of
the oracle) tells it apart.  A shift of every position by the same amount leaves
attention unchanged (only position differences enter the scores), so that one
is caught by the rotation step's own worked example.
Nothing here touches a GPU.
"""
import ctypes
import math
import os
import subprocess

import numpy as np
import pytest

from brute_force import brute_force
from causal_rope_self_neox_b300.workloads import bf16_bits, make_qkv

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "neox_oracle.c")

MUTATIONS = {
    "rotation_sign": ("y[i] = x[i] * c - x[i + h] * s;", "y[i] = x[i] * c + x[i + h] * s;"),
    "rotation_second_sign": ("y[i + h] = x[i + h] * c + x[i] * s;", "y[i + h] = x[i + h] * c - x[i] * s;"),
    "inv_freq_over_D": ("double theta = (double)p * pow(base, -2.0 * (double)i / (double)r);",
                        "double theta = (double)p * pow(base, -2.0 * (double)i / (double)D);"),
    "position_off_by_one": ("double theta = (double)p * pow(", "double theta = (double)(p + 1) * pow("),
    "scale_wrong": ("double scale = 1.0 / sqrt((double)D);", "double scale = 1.0 / (double)D;"),
    "mask_without_diagonal": ("for (int64_t j = 0; j <= i; ++j) {\n    double dot",
                              "for (int64_t j = 0; j < i || j == 0; ++j) {\n    double dot"),
    "lse_drops_max": ("*lse_out = m + log(l);", "*lse_out = log(l);"),
    "keys_from_query_slot": ("const uint16_t* k = J->qkv + qkv_off(b, s, h, 1,", "const uint16_t* k = J->qkv + qkv_off(b, s, h, 0,"),
    "values_from_key_slot": ("const uint16_t* v = J->qkv + qkv_off(b, s, h, 2,", "const uint16_t* v = J->qkv + qkv_off(b, s, h, 1,"),
    "query_unrotated": ("neox_oracle_rotate(qraw, D, J->r, J->base, i, qr);", "neox_oracle_rotate(qraw, D, J->r, J->base, 0, qr);"),
    "no_normalisation": ("double w = scores[j] / l;", "double w = scores[j];"),
}


def build_mutant(tmp_path, name):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"{name}.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-D_POSIX_C_SOURCE=200809L",
                           str(path), "-o", str(so), "-lm", "-lpthread"])
    lib = ctypes.CDLL(str(so))
    P, i32, f64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
    lib.neox_oracle_fwd.argtypes = [P, i32, i32, i32, i32, i32, f64, P, P, i32]
    lib.neox_oracle_fwd.restype = i32
    lib.neox_oracle_rotate.argtypes = [P, i32, i32, f64, ctypes.c_int64, P]
    lib.neox_oracle_rotate.restype = None
    return lib


def run_lib(lib, bits, B, S, H, D, r):
    out = np.empty((B, S, H, D))
    lse = np.empty((B, H, S))
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    rc = lib.neox_oracle_fwd(p(np.ascontiguousarray(bits)), B, S, H, D, r, 1e4, p(out), p(lse), 1)
    assert rc == 0
    return out, lse


def pins_pass(lib) -> bool:
    """The independent checks: dense brute force on a small case, plus the worked example."""
    ok = True
    qkv = make_qkv(1, 40, 2, 16, seed=5)
    out, lse = run_lib(lib, bf16_bits(qkv), 1, 40, 2, 16, 8)
    ref_out, ref_lse = brute_force(qkv.double().numpy(), 8, 1e4)
    with np.errstate(invalid="ignore"):
        ok &= bool(np.allclose(out, ref_out, atol=1e-12, rtol=0) and np.allclose(lse, ref_lse, atol=1e-12, rtol=0))
    # two-token example: k0 = e2, q1 = k1 = e0, v0 = e1, v1 = e3 (D = r = 4)
    x = np.zeros((1, 2, 1, 3, 4), dtype=np.float32)
    x[0, 0, 0, 1, 2] = x[0, 1, 0, 0, 0] = x[0, 1, 0, 1, 0] = x[0, 0, 0, 2, 1] = x[0, 1, 0, 2, 3] = 1.0
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    out, lse = run_lib(lib, bits, 1, 2, 1, 4, 4)
    s10, s11 = math.sin(1.0) / 2, 0.5
    ok &= abs(lse[0, 0, 1] - math.log(math.exp(s10) + math.exp(s11))) < 1e-15
    # the rotation step on its own: e_0 at position 1 (D = r = 8) -> cos(1) e_0 + sin(1) e_4
    e0 = np.zeros(8)
    e0[0] = 1.0
    y = np.empty(8)
    lib.neox_oracle_rotate(e0.ctypes.data_as(ctypes.c_void_p), 8, 8, 1e4, 1, y.ctypes.data_as(ctypes.c_void_p))
    expect = np.zeros(8)
    expect[0], expect[4] = math.cos(1.0), math.sin(1.0)
    ok &= bool(np.allclose(y, expect, atol=1e-15, rtol=0))
    return ok


def test_unmodified_copy_passes(tmp_path):
    src = open(SRC).read()
    path = tmp_path / "same.c"
    path.write_text(src)
    so = tmp_path / "same.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-D_POSIX_C_SOURCE=200809L",
                           str(path), "-o", str(so), "-lm", "-lpthread"])
    lib = ctypes.CDLL(str(so))
    P, i32, f64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
    lib.neox_oracle_fwd.argtypes = [P, i32, i32, i32, i32, i32, f64, P, P, i32]
    lib.neox_oracle_fwd.restype = i32
    lib.neox_oracle_rotate.argtypes = [P, i32, i32, f64, ctypes.c_int64, P]
    lib.neox_oracle_rotate.restype = None
    assert pins_pass(lib)


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(tmp_path, name):
    assert not pins_pass(build_mutant(tmp_path, name)), f"mutation {name} slipped through the pins"
