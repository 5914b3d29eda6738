"""Pins of the decode oracle (one new token against a cache of earlier tokens).

By definition the decode output for a token at position P is row P of the prefill
over the same sequence; the prefill oracle is pinned on its own (test_oracle.py), so
matching it at every tested position pins the decode oracle's rotation offsets, cache
indexing and softmax.  Closed forms cover the single-token case.
"""
import numpy as np
import pytest
import torch

import oracle
from causal_rope_self_neox_b300.workloads import bf16_bits, decode_from_sequence, make_decode_inputs, make_qkv


def _decode_vs_prefill(B, S, H, D, r, pos, seed, Smax=None):
    Smax = Smax or S
    qkv = make_qkv(B, S, H, D, seed)
    new, kc, vc = decode_from_sequence(qkv, pos, Smax)
    out, lse = oracle.decode(bf16_bits(new), bf16_bits(kc), bf16_bits(vc), pos, B, H, Smax, D, r)
    rows = np.array([[b, h, pos[b]] for b in range(B) for h in range(H)], dtype=np.int64)
    ref_out, ref_lse = oracle.fwd_rows(bf16_bits(qkv), B, S, H, D, r, 10000.0, rows)
    return out.reshape(B * H, D), lse.reshape(B * H), ref_out, ref_lse


@pytest.mark.parametrize("B,S,H,D,r,pos", [
    (1, 64, 2, 64, 16, [63]),
    (2, 130, 3, 96, 24, [129, 7]),      # ragged positions across the batch
    (3, 40, 1, 128, 128, [0, 1, 39]),   # full rotary, first and second token
    (1, 33, 2, 64, 0, [32]),            # no rotary dims
    (2, 50, 2, 96, 6, [17, 49]),        # odd rotary chunk (r % 16 != 0)
])
def test_decode_is_the_prefill_row_at_its_position(B, S, H, D, r, pos):
    out, lse, ref_out, ref_lse = _decode_vs_prefill(B, S, H, D, r, pos, seed=B * 100 + S + r)
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_first_token_is_its_own_value_and_plain_dot_product():
    # position 0: one key, weight 1, and the rotation at angle 0 is the identity
    B, H, D, r = 2, 3, 64, 16
    new, kc, vc = make_decode_inputs(B, H, 8, D, seed=5)
    out, lse = oracle.decode(bf16_bits(new), None, None, [0, 0], B, H, 8, D, r)
    q = new[:, :, 0].double().numpy()
    k = new[:, :, 1].double().numpy()
    v = new[:, :, 2].double().numpy()
    np.testing.assert_array_equal(out, v)
    np.testing.assert_allclose(lse, (q * k).sum(-1) / np.sqrt(D), rtol=0, atol=1e-12)


def test_cache_rows_past_the_position_are_not_read():
    B, H, Smax, D, r = 2, 2, 32, 96, 24
    new, kc, vc = make_decode_inputs(B, H, Smax, D, seed=9)
    pos = [10, 31]
    a = oracle.decode(bf16_bits(new), bf16_bits(kc), bf16_bits(vc), pos, B, H, Smax, D, r)
    kc2, vc2 = kc.clone(), vc.clone()
    kc2[0, :, 10:] = 7.0
    vc2[0, :, 10:] = -7.0
    b = oracle.decode(bf16_bits(new), bf16_bits(kc2), bf16_bits(vc2), pos, B, H, Smax, D, r)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


def test_rejects_bad_positions():
    new, kc, vc = make_decode_inputs(1, 1, 4, 64, seed=1)
    with pytest.raises(ValueError):
        oracle.decode(bf16_bits(new), bf16_bits(kc), bf16_bits(vc), [4], 1, 1, 4, 64, 16)
    with pytest.raises(ValueError):
        oracle.decode(bf16_bits(new), None, None, [1], 1, 1, 4, 64, 16)
