"""Pins of the backward oracle (gradient of sum(dout * out) with respect to qkv).

The backward oracle is checked against things that do not share its derivation:
central finite differences of the dense brute-force forward (tests/brute_force.py:
dense rotation matrices, a full masked score matrix, scipy's logsumexp); torch
autograd through a small fp64 torch forward written here from the definition; for
rotary_dim = 0, torch's own causal scaled_dot_product_attention backward; closed forms
(one token; a constant key set); and planted mistakes in a copy of the oracle, each of
which one of those checks must catch.  Nothing here touches a GPU.
"""
import ctypes
import subprocess
import os

import numpy as np
import pytest
import torch

import oracle
from brute_force import brute_force
from causal_rope_self_neox_b300.workloads import bf16_bits, make_qkv

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle", "neox_oracle.c")


def bf16_inputs(B, S, H, D, seed):
    qkv = make_qkv(B, S, H, D, seed=seed)
    g = torch.Generator().manual_seed(seed + 7)
    dout = torch.randn((B, S, H, D), generator=g).to(torch.bfloat16)
    return qkv, dout


def torch_forward(qkv, r, base=10000.0):
    """fp64 torch statement of the forward: explicit cos/sin per position, causal mask."""
    B, S, H, _, D = qkv.shape
    q, k, v = qkv[..., 0, :], qkv[..., 1, :], qkv[..., 2, :]  # [B,S,H,D]
    h = r // 2
    pos = torch.arange(S, dtype=torch.float64)
    inv = base ** (-2.0 * torch.arange(h, dtype=torch.float64) / r) if h else torch.zeros(0, dtype=torch.float64)
    ang = pos[:, None] * inv[None, :]  # [S, h]
    c, s = torch.cos(ang)[None, :, None, :], torch.sin(ang)[None, :, None, :]

    def rot(x):
        x1, x2, rest = x[..., :h], x[..., h:r], x[..., r:]
        return torch.cat([x1 * c - x2 * s, x2 * c + x1 * s, rest], dim=-1)

    qr, kr = rot(q), rot(k)
    sc = torch.einsum("bihd,bjhd->bhij", qr, kr) / D ** 0.5
    mask = torch.ones(S, S, dtype=torch.bool).tril()
    sc = sc.masked_fill(~mask, float("-inf"))
    p = torch.softmax(sc, dim=-1)
    return torch.einsum("bhij,bjhd->bihd", p, v)


def autograd_grad(qkv_bf16, dout_bf16, r):
    x = qkv_bf16.to(torch.float64).requires_grad_(True)
    out = torch_forward(x, r)
    (out * dout_bf16.to(torch.float64)).sum().backward()
    return x.grad.numpy()


@pytest.mark.parametrize("B,S,H,D,r", [(1, 6, 2, 16, 8), (2, 5, 1, 16, 16), (1, 7, 1, 16, 6), (1, 4, 2, 16, 0)])
def test_matches_finite_differences_of_the_brute_force(B, S, H, D, r):
    qkv, dout = bf16_inputs(B, S, H, D, seed=S * 10 + r)
    got = oracle.bwd(bf16_bits(qkv), bf16_bits(dout), B, S, H, D, r)
    x = qkv.to(torch.float64).numpy()
    g = dout.to(torch.float64).numpy()
    eps = 1e-6
    rng = np.random.default_rng(5)
    idx = [tuple(rng.integers(0, n) for n in x.shape) for _ in range(60)]
    idx += [(0, S - 1, 0, 0, 0), (0, 0, 0, 1, 0), (0, S - 1, 0, 2, D - 1)]
    for i in idx:
        xp, xm = x.copy(), x.copy()
        xp[i] += eps
        xm[i] -= eps
        fd = ((brute_force(xp, r, 10000.0)[0] * g).sum() - (brute_force(xm, r, 10000.0)[0] * g).sum()) / (2 * eps)
        assert abs(fd - got[i]) <= 1e-6 * max(1.0, abs(fd)), (i, fd, got[i])


@pytest.mark.parametrize("B,S,H,D,r", [(1, 33, 2, 64, 16), (2, 20, 3, 96, 24), (1, 17, 1, 128, 128)])
def test_matches_torch_autograd(B, S, H, D, r):
    qkv, dout = bf16_inputs(B, S, H, D, seed=S + D + r)
    got = oracle.bwd(bf16_bits(qkv), bf16_bits(dout), B, S, H, D, r)
    ref = autograd_grad(qkv, dout, r)
    assert np.abs(got - ref).max() <= 1e-10 * max(1.0, np.abs(ref).max())


def test_unrotated_matches_torch_sdpa_backward():
    B, S, H, D = 2, 40, 2, 64
    qkv, dout = bf16_inputs(B, S, H, D, seed=3)
    got = oracle.bwd(bf16_bits(qkv), bf16_bits(dout), B, S, H, D, 0)
    x = qkv.to(torch.float64).permute(0, 2, 3, 1, 4).contiguous().requires_grad_(True)  # [B,H,3,S,D]
    out = torch.nn.functional.scaled_dot_product_attention(x[:, :, 0], x[:, :, 1], x[:, :, 2], is_causal=True)
    (out * dout.to(torch.float64).permute(0, 2, 1, 3)).sum().backward()
    ref = x.grad.permute(0, 3, 1, 2, 4).numpy()  # back to [B,S,H,3,D]
    assert np.abs(got - ref).max() <= 1e-10 * max(1.0, np.abs(ref).max())


def test_single_token_closed_form():
    # one token: out = v_0 whatever q and k are, so dq = dk = 0 and dv = dout
    qkv, dout = bf16_inputs(1, 1, 3, 64, seed=9)
    got = oracle.bwd(bf16_bits(qkv), bf16_bits(dout), 1, 1, 3, 64, 16)
    assert np.all(got[..., 0, :] == 0) and np.all(got[..., 1, :] == 0)
    assert np.array_equal(got[..., 2, :], dout.to(torch.float64).numpy())


def test_identical_keys_give_uniform_weights_and_no_query_gradient():
    # r = 0 and every key equal: the scores of a row are all equal, softmax is uniform
    # whatever the query, so dq = 0 and dv_j = sum_{i >= j} dout_i / (i + 1)
    B, S, H, D = 1, 9, 1, 16
    qkv, dout = bf16_inputs(B, S, H, D, seed=4)
    qkv[:, :, :, 1, :] = qkv[:, :1, :, 1, :]
    got = oracle.bwd(bf16_bits(qkv), bf16_bits(dout), B, S, H, D, 0)
    assert np.abs(got[..., 0, :]).max() < 1e-12
    g = dout.to(torch.float64).numpy()[0, :, 0]
    want = np.stack([sum(g[i] / (i + 1) for i in range(j, S)) for j in range(S)])
    assert np.allclose(got[0, :, 0, 2], want, atol=1e-12)


BWD_MUTATIONS = {
    "delta_dropped": ("const double ds = p[j] * (dp[j] - delta) * inv_sqrt_d;",
                      "const double ds = p[j] * dp[j] * inv_sqrt_d;"),
    "back_rotation_forward": ("neox_oracle_rotate(dQr + s * D, D, J->r, J->base, -s, gq);",
                              "neox_oracle_rotate(dQr + s * D, D, J->r, J->base, s, gq);"),
    "key_not_rotated_back": ("neox_oracle_rotate(dKr + s * D, D, J->r, J->base, -s, gk);",
                             "neox_oracle_rotate(dKr + s * D, D, J->r, J->base, 0, gk);"),
    "dk_from_raw_query": ("dKr[j * D + d] += ds * Qr[i * D + d];", "dKr[j * D + d] += ds * Kr[i * D + d];"),
    "dv_with_wrong_row": ("dV[j * D + d] += p[j] * dO[i * D + d];", "dV[j * D + d] += p[j] * dO[j * D + d];"),
    "probs_unnormalised": ("for (int64_t j = 0; j <= i; ++j) p[j] /= l;", "for (int64_t j = 0; j <= i; ++j) p[j] /= 1.0;"),
}


@pytest.mark.parametrize("name", list(BWD_MUTATIONS))
def test_a_planted_mistake_is_caught(tmp_path, name):
    old, new = BWD_MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / f"{name}.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-D_POSIX_C_SOURCE=200809L",
                           str(path), "-o", str(so), "-lm", "-lpthread"])
    lib = ctypes.CDLL(str(so))
    P, i32, f64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
    lib.neox_oracle_bwd.argtypes = [P, P, i32, i32, i32, i32, i32, f64, P, i32]
    lib.neox_oracle_bwd.restype = i32
    B, S, H, D, r = 1, 9, 2, 32, 16
    qkv, dout = bf16_inputs(B, S, H, D, seed=21)
    qb = np.ascontiguousarray(bf16_bits(qkv).reshape(-1))
    gb = np.ascontiguousarray(bf16_bits(dout).reshape(-1))
    got = np.zeros((B, S, H, 3, D))
    assert lib.neox_oracle_bwd(qb.ctypes.data, gb.ctypes.data, B, S, H, D, r, 10000.0, got.ctypes.data, 1) == 0
    ref = autograd_grad(qkv, dout, r)
    assert np.abs(got - ref).max() > 1e-6
