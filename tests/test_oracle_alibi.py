"""Pins of the ALiBi oracle (causal attention with a linear distance bias, no rotation).

Checked against things that do not share its code: the slope sequence in closed form
(powers of two, and the interleaved extra slopes for a head count that is not one);
a dense numpy statement with a full bias matrix and scipy's logsumexp; the closed form
of a zero query (weights decay geometrically with distance); and planted mistakes in a
copy of the oracle, each of which one of those checks must catch.  Nothing here touches
a GPU.
"""
import ctypes
import os
import subprocess

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

import oracle
from causal_rope_self_neox_b300.workloads import bf16_bits, make_qkv

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "neox_oracle.c")


def test_slopes_closed_forms():
    assert np.array_equal(oracle.alibi_slopes(8), 2.0 ** -np.arange(1, 9))
    assert np.array_equal(oracle.alibi_slopes(1), [2.0 ** -8])
    s64 = oracle.alibi_slopes(64)
    assert np.allclose(s64, 2.0 ** (-np.arange(1, 65) / 8.0), rtol=0, atol=1e-15)
    # 12 heads: the 8 slopes of 8 heads, then slopes 1, 3, 5, 7 of 16 heads (2^-(k/2))
    s12 = oracle.alibi_slopes(12)
    assert np.allclose(s12, np.concatenate([2.0 ** -np.arange(1, 9), 2.0 ** -(np.array([1, 3, 5, 7]) / 2)]),
                       rtol=0, atol=1e-15)


def dense_alibi(qkv_f64, slopes):
    B, S, H, _, D = qkv_f64.shape
    out, lse = np.empty((B, S, H, D)), np.empty((B, H, S))
    dist = np.arange(S)[:, None] - np.arange(S)[None, :]
    for b in range(B):
        for h in range(H):
            q, k, v = qkv_f64[b, :, h, 0], qkv_f64[b, :, h, 1], qkv_f64[b, :, h, 2]
            sc = q @ k.T / np.sqrt(D) - slopes[h] * dist
            sc = np.where(dist >= 0, sc, -np.inf)
            l = logsumexp(sc, axis=1)
            out[b, :, h] = np.exp(sc - l[:, None]) @ v
            lse[b, h] = l
    return out, lse


@pytest.mark.parametrize("B,S,H,D", [(1, 9, 8, 16), (2, 33, 12, 32), (1, 70, 3, 64)])
def test_matches_the_dense_statement(B, S, H, D):
    qkv = make_qkv(B, S, H, D, seed=S + H)
    out, lse = oracle.fwd_alibi(bf16_bits(qkv), B, S, H, D)
    ref_out, ref_lse = dense_alibi(qkv.to(torch.float64).numpy(), oracle.alibi_slopes(H))
    assert np.abs(out - ref_out).max() < 1e-12 and np.abs(lse - ref_lse).max() < 1e-12


def test_zero_query_closed_form():
    # q = 0: scores are -m (i - j), so lse_i = log sum_{t <= i} e^{-m t} and out_i is
    # the e^{-m (i - j)}-weighted mean of v_j
    B, S, H, D = 1, 40, 4, 16
    qkv = make_qkv(B, S, H, D, seed=5)
    qkv[:, :, :, 0, :] = 0
    out, lse = oracle.fwd_alibi(bf16_bits(qkv), B, S, H, D)
    v = qkv[0, :, :, 2].to(torch.float64).numpy()  # [S, H, D]
    for h, m in enumerate(oracle.alibi_slopes(H)):
        for i in (0, 1, 17, S - 1):
            w = np.exp(-m * (i - np.arange(i + 1)))
            assert abs(lse[0, h, i] - np.log((1 - np.exp(-m * (i + 1))) / (1 - np.exp(-m)))) < 1e-12
            assert np.abs(out[0, i, h] - (w[:, None] * v[: i + 1, h]).sum(0) / w.sum()).max() < 1e-12


MUTATIONS = {
    "bias_sign": ("sc[j] = dot * inv_sqrt_d - m_h * (double)(i - j);", "sc[j] = dot * inv_sqrt_d + m_h * (double)(i - j);"),
    "distance_off_by_one": ("sc[j] = dot * inv_sqrt_d - m_h * (double)(i - j);",
                            "sc[j] = dot * inv_sqrt_d - m_h * (double)(i - j + 1);"),
    "slopes_reversed": ("const double m_h = J->slopes[h];", "const double m_h = J->slopes[H - 1 - h];"),
    "extra_slopes_even": ("for (int k = n, e = 1; k < H; ++k, e += 2)", "for (int k = n, e = 2; k < H; ++k, e += 2)"),
}


@pytest.mark.parametrize("name", list(MUTATIONS))
def test_a_planted_mistake_is_caught(tmp_path, name):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"{name}.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-D_POSIX_C_SOURCE=200809L",
                           str(path), "-o", str(so), "-lm", "-lpthread"])
    lib = ctypes.CDLL(str(so))
    P, i32 = ctypes.c_void_p, ctypes.c_int
    lib.neox_oracle_fwd_alibi.argtypes = [P, i32, i32, i32, i32, P, P, i32]
    lib.neox_oracle_fwd_alibi.restype = i32
    B, S, H, D = 1, 24, 12, 16
    qkv = make_qkv(B, S, H, D, seed=8)
    qb = np.ascontiguousarray(bf16_bits(qkv).reshape(-1))
    out, lse = np.zeros((B, S, H, D)), np.zeros((B, H, S))
    assert lib.neox_oracle_fwd_alibi(qb.ctypes.data, B, S, H, D, out.ctypes.data, lse.ctypes.data, 1) == 0
    slopes = 2.0 ** -np.arange(1, 9)
    slopes = np.concatenate([slopes, 2.0 ** -(np.array([1, 3, 5, 7]) / 2)])  # closed form, 12 heads
    ref_out, ref_lse = dense_alibi(qkv.to(torch.float64).numpy(), slopes)
    assert max(np.abs(out - ref_out).max(), np.abs(lse - ref_lse).max()) > 1e-6
