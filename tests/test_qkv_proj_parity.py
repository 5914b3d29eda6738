"""GPU parity of the query_key_value projection (neox_attn_qkv_proj) against the oracle.

The kernel accumulates in fp32 and rounds each output to bf16 once; with rotary_dim > 0
it rotates the query/key pairs of those bf16 values in fp32 and rounds again.  The oracle
is exact (fp64).  Element-wise bound, for output n of token t with exact value y:

    |gpu - y| <= 2^-8 (|y| + R) + 2^-12 (A + A_partner)

2^-8 |y| covers the last bf16 rounding (half an ulp is at most 2^-8 of the value).  A
rotated element also carries the rounding of its input pair (a, b), rotated: at most
|da cos - db sin| <= sqrt(da^2 + db^2) <= 2^-8 sqrt(a^2 + b^2), and the rotation keeps
a^2 + b^2, so R = sqrt(y^2 + y_partner^2) with y_partner the other element of the
(i, i + r/2) pair (R = 0 for values and dims >= r_dim).  A = sum_k |x_tk w_kn| + |bias_n|
bounds the fp32 accumulation error (K * 2^-24 * A < 2^-12 A for K <= 4096, and the error
grows like sqrt(K) in practice, far below that for K = 6144).
A relative RMS error <= 3e-3 over all checked elements is asserted as well (one bf16
rounding alone gives about 1.7e-3, two about 2.4e-3).
"""
import numpy as np
import pytest
import torch

import oracle
from causal_rope_self_neox_b300.workloads import WORKLOADS, bf16_bits, make_proj_inputs, proj_inputs


def _run(x, w, b, B, S, H, D, r, base=10000.0):
    import causal_rope_self_neox_b300 as na
    xd, wd = x.cuda(), w.cuda()
    bd = None if b is None else b.cuda()
    out = na.qkv_proj(xd, wd, bd, B, S, H, D, r, base)
    torch.cuda.synchronize()
    na.check_device_error()
    return out.float().cpu().numpy().astype(np.float64).reshape(B * S, H, 3, D)


def _bounds(x, w, b, rows, H, D, r):
    """A = sum_k |x w| + |bias| for the listed token rows, shaped [n, H, 3, D]."""
    xa = np.abs(x.double().numpy()[rows])
    A = xa @ np.abs(w.double().numpy())
    if b is not None:
        A = A + np.abs(b.double().numpy())
    return A.reshape(len(rows), H, 3, D)


def _partner(a, r):
    """The (i, i + r/2) partner of every query/key element (0 for values and dims >= r)."""
    p = np.zeros_like(a)
    if r:
        h = r // 2
        p[..., :2, :h] = a[..., :2, h:r]
        p[..., :2, h:r] = a[..., :2, :h]
    return p


def _check(got, ref, A, r):
    R = np.sqrt(ref ** 2 + _partner(ref, r) ** 2) * (_partner(np.ones_like(ref), r) > 0)
    tol = 2.0 ** -8 * (np.abs(ref) + R) + 2.0 ** -12 * (A + _partner(A, r))
    err = np.abs(got - ref)
    assert np.isfinite(got).all()
    worst = np.unravel_index(np.argmax(err - tol), err.shape)
    assert np.all(err <= tol), (worst, got[worst], ref[worst], tol[worst])
    rel_rms = np.sqrt((err ** 2).sum() / (ref ** 2).sum())
    assert rel_rms <= 3e-3, rel_rms


@pytest.mark.gpu
@pytest.mark.parametrize("B,S,hidden,H,D,r,bias", [
    (1, 200, 256, 2, 64, 16, True),     # ragged rows (200 = 128 + 72), N = 384: a half-empty column tile
    (2, 129, 200, 3, 96, 24, True),     # hidden 200: a K step of 8; 9 slots of 96: odd slot count
    (1, 300, 512, 2, 128, 128, False),  # full rotary_dim, no bias
    (1, 96, 96, 2, 96, 0, True),        # no rotation; fewer rows than one tile
    (3, 70, 128, 1, 64, 64, True),      # three sequences: positions restart at every 70 rows
])
def test_projection_matches_oracle_on_every_element(B, S, hidden, H, D, r, bias):
    x, w, b = make_proj_inputs(B, S, hidden, H, D, seed=S + hidden + r, with_bias=bias)
    got = _run(x, w, b, B, S, H, D, r)
    ref = oracle.qkv_proj_rotated(bf16_bits(x), bf16_bits(w), None if b is None else bf16_bits(b), B, S, H, D, r)
    _check(got, ref, _bounds(x, w, b, np.arange(B * S), H, D, r), r)


@pytest.mark.gpu
def test_projection_on_the_neox20b_shape_sampled_rows():
    wl = WORKLOADS["neox20b"]  # hidden 6144 -> 3 x 64 x 96 = 18432, 4096 token rows
    B, S, H, D, r = wl.B, wl.S, wl.H, wl.D, wl.rotary_dim
    x, w, b = proj_inputs(wl)
    got = _run(x, w, b, B, S, H, D, r)
    rng = np.random.default_rng(wl.seed + 7)
    rows = np.unique(np.concatenate([rng.choice(B * S, size=40, replace=False), [0, 1, 127, 128, S - 1, S, B * S - 1]]))
    ref = oracle.qkv_proj_rotated(bf16_bits(x), bf16_bits(w), bf16_bits(b), B, S, H, D, r, rows=rows)
    _check(got[rows], ref, _bounds(x, w, b, rows, H, D, r), r)


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["pythia160m", "pythia1.4b", "long16k"])
def test_projection_on_the_other_workload_shapes_sampled_rows(name):
    # D = 64 (four slots a tile, r = 16), D = 128 (r = 32), and D = 128 with every dim
    # rotated (r = 128: the 16-byte rotation path) at 16384 tokens x hidden 4096
    wl = WORKLOADS[name]
    B, S, H, D, r = wl.B, wl.S, wl.H, wl.D, wl.rotary_dim
    x, w, b = proj_inputs(wl)
    got = _run(x, w, b, B, S, H, D, r)
    rng = np.random.default_rng(wl.seed + 7)
    rows = np.unique(np.concatenate([rng.choice(B * S, size=24, replace=False), [0, S - 1, B * S - 1]]))
    ref = oracle.qkv_proj_rotated(bf16_bits(x), bf16_bits(w), bf16_bits(b), B, S, H, D, r, rows=rows)
    _check(got[rows], ref, _bounds(x, w, b, rows, H, D, r), r)


@pytest.mark.gpu
def test_plain_projection_equals_rotated_one_outside_the_rotary_dims():
    # rotary_dim only touches the first r dims of the query and key slots
    B, S, hidden, H, D, r = 2, 150, 192, 2, 96, 24
    x, w, b = make_proj_inputs(B, S, hidden, H, D, seed=77)
    plain = _run(x, w, b, B, S, H, D, 0)
    rot = _run(x, w, b, B, S, H, D, r)
    assert np.array_equal(plain[..., 2, :], rot[..., 2, :])
    assert np.array_equal(plain[..., :2, r:], rot[..., :2, r:])
    s0 = np.arange(B) * S  # position 0 of each sequence: the rotation is the identity
    assert np.array_equal(plain[s0], rot[s0])


@pytest.mark.gpu
def test_projection_is_deterministic():
    B, S, hidden, H, D, r = 1, 520, 384, 4, 64, 16
    x, w, b = make_proj_inputs(B, S, hidden, H, D, seed=5)
    assert np.array_equal(_run(x, w, b, B, S, H, D, r), _run(x, w, b, B, S, H, D, r))


@pytest.mark.gpu
def test_projection_then_attention_matches_the_oracle_chain():
    # The rotated qkv goes to the attention with rotary_dim 0.  Oracle chain: the projection
    # rounded to bf16, rotated exactly, rounded to bf16 again (the rounding steps the kernel
    # documents), then the exact attention.
    import causal_rope_self_neox_b300 as na
    B, S, hidden, H, D, r = 1, 700, 384, 4, 96, 24
    x, w, b = make_proj_inputs(B, S, hidden, H, D, seed=91)
    qkv = na.qkv_proj(x.cuda(), w.cuda(), b.cuda(), B, S, H, D, r)
    out, lse = na.attn_fwd(qkv, 0)
    torch.cuda.synchronize()
    na.check_device_error()
    ref_qkv = oracle.qkv_proj_rotated(bf16_bits(x), bf16_bits(w), bf16_bits(b), B, S, H, D, r, bf16_steps=True)
    ref_bits = bf16_bits(torch.from_numpy(ref_qkv.reshape(B, S, H, 3, D)).to(torch.bfloat16))
    # the two sides' bf16 qkv differ only where fp32 and fp64 sums round apart
    got_qkv = qkv.float().cpu().numpy().reshape(B * S, H, 3, D)
    assert np.mean(got_qkv != ref_qkv) < 1e-2
    ref_out, ref_lse = oracle.fwd(ref_bits, B, S, H, D, 0, 10000.0)
    e = out.float().cpu().numpy().astype(np.float64) - ref_out
    assert np.abs(e).max() <= 2e-2 and np.sqrt((e ** 2).mean()) <= 3e-3
    assert np.abs(lse.cpu().numpy().astype(np.float64) - ref_lse).max() <= 1e-3


def test_projection_rejects_bad_arguments_before_any_launch():
    import causal_rope_self_neox_b300 as na
    A, W, O = 0x10000000, 0x20000000, 0x80000000
    assert na.neox_attn_qkv_proj(A, W, 0, 1, 128, 100, 1, 64, 16, 1e4, O, 0) == na.NEOX_ERR_INVALID_ARG  # hidden % 8
    assert na.neox_attn_qkv_proj(A, W, 0, 1, 128, 128, 1, 80, 16, 1e4, O, 0) == na.NEOX_ERR_UNSUPPORTED_HEAD_DIM
    assert na.neox_attn_qkv_proj(A, W, 0, 1, 128, 128, 1, 64, 15, 1e4, O, 0) == na.NEOX_ERR_INVALID_ARG
    assert na.neox_attn_qkv_proj(A + 8, W, 0, 1, 128, 128, 1, 64, 16, 1e4, O, 0) == na.NEOX_ERR_MISALIGNED
    assert na.neox_attn_qkv_proj(A, W, 0, 1, 128, 128, 1, 64, 16, 1e4, A + 64, 0) == na.NEOX_ERR_INVALID_ARG
