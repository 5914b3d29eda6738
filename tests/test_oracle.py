"""Pins of the fp64 oracle against things other than itself (no GPU needed).

What each group fixes:
  * rotation worked examples: closed-form values of the rotate-half pairing and
    sign (a GPT-J interleaved pairing or a flipped sign fails them);
  * inv_freq closed forms: base^(-2i/r) at exact decades (a wrong exponent fails);
  * rotation invariants: norm kept, position 0 is the identity, R(a)R(b) = R(a+b),
    and <R(m)q, R(n)k> depends only on n - m;
  * attention with rotary_dim = 0 against torch's CPU scaled_dot_product_attention
    (library routine) in fp64;
  * the dense numpy brute force (tests/brute_force.py) on tiny inputs;
  * closed forms: row 0, Q = 0 (prefix means, lse = ln(i+1)), S = 1, constant V;
  * causality (future tokens cannot change earlier rows) and softmax rows sum to 1;
  * a hand-worked two-token example whose lse depends on the pairing and sign.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from brute_force import brute_force, rotation_matrix
from causal_rope_self_neox_b300.workloads import bf16_bits, make_qkv


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Exact only for values that are representable in bf16 (checked)."""
    x = np.asarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    assert np.all((u & 0xFFFF) == 0), "value not exactly representable in bf16"
    return (u >> 16).astype(np.uint16)


# ---------------------------------------------------------------- rotation ----

def test_rotation_worked_example_pairs_i_with_i_plus_half():
    # D = 8, r = 8 (h = 4), base 10000: inv_freq[0] = 1, so at position p the
    # first pair turns by exactly p radians.  e_0 must land in the (0, h) plane.
    e0 = np.zeros(8); e0[0] = 1.0
    y = oracle.rotate(e0, 1, 8, 10000.0)
    expect = np.zeros(8); expect[0] = math.cos(1.0); expect[4] = math.sin(1.0)
    np.testing.assert_allclose(y, expect, atol=1e-15)
    eh = np.zeros(8); eh[4] = 1.0
    y = oracle.rotate(eh, 1, 8, 10000.0)
    expect = np.zeros(8); expect[0] = -math.sin(1.0); expect[4] = math.cos(1.0)
    np.testing.assert_allclose(y, expect, atol=1e-15)


def test_rotation_second_pair_uses_second_frequency():
    # r = 4, base = 100: inv_freq = [1, 100^(-1/2) = 0.1]; position 10 turns pair 1 by 1 rad.
    e1 = np.zeros(6); e1[1] = 1.0
    y = oracle.rotate(e1, 10, 4, 100.0)
    expect = np.zeros(6); expect[1] = math.cos(1.0); expect[3] = math.sin(1.0)
    np.testing.assert_allclose(y, expect, atol=1e-14)


def test_inv_freq_closed_forms():
    f = oracle.inv_freq(24, 10000.0)  # 10000^(-i/12) = 10^(-i/3)
    assert f.shape == (12,)
    np.testing.assert_allclose(f[[0, 3, 6, 9]], [1.0, 0.1, 0.01, 0.001], rtol=1e-14)
    f = oracle.inv_freq(128, 10000.0)  # 10^(-i/16)
    np.testing.assert_allclose(f[[0, 16, 32, 48]], [1.0, 0.1, 0.01, 0.001], rtol=1e-14)


def test_pass_through_dims_untouched_and_position_zero_identity():
    rng = np.random.default_rng(0)
    x = rng.standard_normal(96)
    y = oracle.rotate(x, 1234, 24, 10000.0)
    np.testing.assert_array_equal(y[24:], x[24:])
    np.testing.assert_array_equal(oracle.rotate(x, 0, 24, 10000.0), x)


@pytest.mark.parametrize("D,r", [(64, 16), (96, 24), (128, 32), (128, 128), (10, 6)])
def test_rotation_norm_and_composition(D, r):
    rng = np.random.default_rng(D + r)
    x = rng.standard_normal(D)
    for p in (1, 7, 2047, 16383):
        y = oracle.rotate(x, p, r, 10000.0)
        assert abs(np.linalg.norm(y) - np.linalg.norm(x)) < 1e-12
    # R(a) R(b) = R(a + b)
    a, b = 123, 4000
    np.testing.assert_allclose(oracle.rotate(oracle.rotate(x, a, r, 10000.0), b, r, 10000.0),
                               oracle.rotate(x, a + b, r, 10000.0), atol=1e-11)


@pytest.mark.parametrize("D,r", [(64, 16), (96, 24), (128, 128)])
def test_relative_position_invariance(D, r):
    rng = np.random.default_rng(7 * D + r)
    q, k = rng.standard_normal(D), rng.standard_normal(D)
    for m, n, t in [(5, 3, 100), (2047, 0, 9000), (16000, 15000, 383), (0, 0, 16383)]:
        s1 = oracle.rotate(q, m, r, 1e4) @ oracle.rotate(k, n, r, 1e4)
        s2 = oracle.rotate(q, m + t, r, 1e4) @ oracle.rotate(k, n + t, r, 1e4)
        assert abs(s1 - s2) < 1e-11 * (1 + abs(s1))


def test_rotation_matches_dense_matrix():
    rng = np.random.default_rng(3)
    for D, r, p in [(64, 16, 77), (96, 24, 2047), (128, 128, 16383), (10, 6, 5)]:
        x = rng.standard_normal(D)
        np.testing.assert_allclose(oracle.rotate(x, p, r, 1e4), rotation_matrix(D, r, 1e4, p) @ x, atol=1e-12)


# --------------------------------------------------------------- attention ----

def _run(qkv_bf16: torch.Tensor, r: int, base: float = 10000.0):
    B, S, H, _, D = qkv_bf16.shape
    return oracle.fwd(bf16_bits(qkv_bf16), B, S, H, D, r, base, threads=2)


@pytest.mark.parametrize("B,S,H,D,r", [(1, 37, 2, 64, 16), (2, 64, 1, 96, 24), (1, 50, 3, 16, 16),
                                       (1, 33, 1, 10, 6), (1, 64, 2, 128, 0)])
def test_matches_dense_brute_force(B, S, H, D, r):
    qkv = make_qkv(B, S, H, D, seed=B * 100 + S + D + r)
    out, lse = _run(qkv, r)
    ref_out, ref_lse = brute_force(qkv.double().numpy(), r, 10000.0)
    np.testing.assert_allclose(out, ref_out, atol=1e-12, rtol=0)
    np.testing.assert_allclose(lse, ref_lse, atol=1e-12, rtol=0)


@pytest.mark.parametrize("D", [64, 96, 128])
def test_no_rotary_equals_library_causal_sdpa(D):
    B, S, H = 2, 70, 3
    qkv = make_qkv(B, S, H, D, seed=D)
    out, lse = _run(qkv, 0)
    x = qkv.double()
    q, k, v = (x[:, :, :, i, :].permute(0, 2, 1, 3) for i in range(3))  # [B,H,S,D]
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True)
    np.testing.assert_allclose(out, ref.permute(0, 2, 1, 3).numpy(), atol=1e-12, rtol=0)
    scores = (q @ k.transpose(-1, -2)) / math.sqrt(D)
    scores = scores.masked_fill(~torch.ones(S, S, dtype=torch.bool).tril(), float("-inf"))
    np.testing.assert_allclose(lse, torch.logsumexp(scores, dim=-1).numpy(), atol=1e-12, rtol=0)


def test_row_zero_closed_form():
    qkv = make_qkv(2, 40, 3, 96, seed=11)
    out, lse = _run(qkv, 24)
    x = qkv.double().numpy()
    # position 0 is unrotated and sees only key 0
    np.testing.assert_array_equal(out[:, 0], x[:, 0, :, 2, :])
    ref_lse = np.einsum("bhd,bhd->bh", x[:, 0, :, 0, :], x[:, 0, :, 1, :]) / math.sqrt(96)
    np.testing.assert_allclose(lse[:, :, 0], ref_lse, atol=1e-14)


def test_zero_query_gives_prefix_mean_and_log_count():
    qkv = make_qkv(1, 50, 2, 64, seed=12)
    qkv[:, :, :, 0, :] = 0
    out, lse = _run(qkv, 16)
    v = qkv.double().numpy()[:, :, :, 2, :]
    cum = np.cumsum(v, axis=1) / np.arange(1, 51)[None, :, None, None]
    np.testing.assert_allclose(out, cum, atol=1e-13)
    np.testing.assert_allclose(lse, np.broadcast_to(np.log(np.arange(1, 51)), lse.shape), atol=1e-14)


def test_single_token_and_constant_values():
    qkv = make_qkv(2, 1, 4, 128, seed=13)
    out, _ = _run(qkv, 128)
    np.testing.assert_array_equal(out[:, 0], qkv.double().numpy()[:, 0, :, 2, :])
    qkv = make_qkv(1, 30, 2, 96, seed=14)
    qkv[:, :, :, 2, :] = qkv[:, :1, :, 2, :]  # every token carries the same value vector
    out, _ = _run(qkv, 24)
    np.testing.assert_allclose(out, np.broadcast_to(qkv.double().numpy()[:, :1, :, 2, :], out.shape), atol=1e-14)


def test_causality_future_tokens_do_not_matter():
    qkv = make_qkv(1, 64, 2, 64, seed=15)
    out, lse = _run(qkv, 16)
    cut = 29
    qkv2 = qkv.clone()
    qkv2[:, cut + 1:] = make_qkv(1, 64 - cut - 1, 2, 64, seed=16)
    out2, lse2 = _run(qkv2, 16)
    np.testing.assert_array_equal(out[:, :cut + 1], out2[:, :cut + 1])
    np.testing.assert_array_equal(lse[:, :, :cut + 1], lse2[:, :, :cut + 1])
    assert not np.array_equal(out[:, cut + 1:], out2[:, cut + 1:])


def test_probability_rows_sum_to_one_and_weight_values():
    qkv = make_qkv(1, 80, 2, 96, seed=17)
    out, lse = _run(qkv, 24)
    v = qkv.double().numpy()[0, :, 1, 2, :]
    for i in (0, 1, 40, 79):
        p = oracle.probs(bf16_bits(qkv), 1, 80, 2, 96, 24, 1e4, 0, 1, i)
        assert p.shape == (i + 1,)
        assert abs(p.sum() - 1.0) < 1e-14 and np.all(p >= 0)
        np.testing.assert_allclose(p @ v[: i + 1], out[0, i, 1], atol=1e-13)


def test_rows_mode_matches_full_mode():
    qkv = make_qkv(2, 90, 3, 64, seed=18)
    out, lse = _run(qkv, 16)
    rows = np.array([[1, 2, 89], [0, 0, 0], [1, 0, 45], [0, 2, 1], [1, 2, 3], [0, 0, 60]])
    o, l = oracle.fwd_rows(bf16_bits(qkv), 2, 90, 3, 64, 16, 1e4, rows, threads=3)
    for k, (b, h, i) in enumerate(rows):
        np.testing.assert_array_equal(o[k], out[b, i, h])
        assert l[k] == lse[b, h, i]


def test_two_token_worked_example_fixes_pairing_and_sign():
    # D = 4, r = 4, base 10000: pair (0,2) turns by p rad, pair (1,3) by p/100 rad.
    # token 0: k0 = e_2;  token 1: q1 = e_0, k1 = e_0.  Values v0 = e_1, v1 = e_3.
    # Rotate-half gives q1' = (cos1, 0, sin1, 0), so s10 = sin(1)/2, s11 = 1/2.
    D = 4
    x = np.zeros((1, 2, 1, 3, D), dtype=np.float32)
    x[0, 0, 0, 1, 2] = 1.0
    x[0, 1, 0, 0, 0] = 1.0
    x[0, 1, 0, 1, 0] = 1.0
    x[0, 0, 0, 2, 1] = 1.0
    x[0, 1, 0, 2, 3] = 1.0
    bits = f32_to_bf16_bits(x)
    out, lse = oracle.fwd(bits, 1, 2, 1, D, 4, 10000.0, threads=1)
    s10, s11 = math.sin(1.0) / 2, 0.5
    assert abs(lse[0, 0, 1] - math.log(math.exp(s10) + math.exp(s11))) < 1e-15
    w0 = math.exp(s10) / (math.exp(s10) + math.exp(s11))
    np.testing.assert_allclose(out[0, 1, 0], [0.0, w0, 0.0, 1 - w0], atol=1e-15)
    # token 0 sees only itself: q0 = 0, so lse = 0 and out = v0
    assert lse[0, 0, 0] == 0.0
    np.testing.assert_array_equal(out[0, 0, 0], [0, 1, 0, 0])


def test_bad_arguments_are_rejected():
    bits = np.zeros(1 * 4 * 1 * 3 * 8, dtype=np.uint16)
    with pytest.raises(RuntimeError):
        oracle.fwd(bits, 1, 4, 1, 8, 3, 1e4)  # odd rotary_dim
    with pytest.raises(RuntimeError):
        oracle.fwd(bits, 1, 4, 1, 8, 10, 1e4)  # rotary_dim > D
    with pytest.raises(RuntimeError):
        oracle.fwd_rows(bits, 1, 4, 1, 8, 8, 1e4, [[0, 0, 4]])  # row out of range
