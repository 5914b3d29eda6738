"""The two placements of the rotary embedding give the same attention, bit for bit.

NEOX_ROTATION_FUSED rotates Q and K tiles inside the attention kernel (shared memory, hi/lo
split in registers); NEOX_ROTATION_PRE rotates them once in a separate pass that writes
hi and lo of q' and k' to the library's scratch, which the kernel then loads by TMA.  Both
evaluate the same fp32 expressions on the same table entries, so the outputs must be
bit-identical; each placement is also held to the oracle on its own.
"""
import numpy as np
import pytest
import torch

import oracle
from causal_rope_self_neox_b300.workloads import bf16_bits, make_qkv
from test_parity import assert_close

pytestmark = pytest.mark.gpu


def run(qkv_cpu, r, rotation):
    import causal_rope_self_neox_b300 as na
    out, lse = na.attn_fwd(qkv_cpu.cuda(), r, 1e4, rotation=rotation)
    na.check_device_error()
    return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


SHAPES = [
    (1, 130, 2, 64, 16, 1.0),     # ragged, one rotated chunk pair
    (2, 300, 3, 96, 24, 1.0),     # r = 24: the packed cross-term chunk of the side tile
    (1, 200, 2, 128, 24, 1.0),    # r = 24 at D = 128, ragged
    (2, 300, 3, 96, 32, 1.0),     # D = 96, two tiles, ragged
    (1, 640, 2, 96, 96, 1.0),     # every dim rotated at D = 96
    (3, 523, 2, 128, 64, 1.0),    # half rotary, several tiles
    (1, 900, 2, 128, 128, 3.0),   # full rotary, sharpened softmax (the long-context setting)
    (2, 256, 5, 64, 64, 1.0),     # full rotary at D = 64, exactly two tiles
]


@pytest.mark.parametrize("B,S,H,D,r,ks", SHAPES)
def test_fused_and_pre_rotated_are_bit_identical_and_match_the_oracle(B, S, H, D, r, ks):
    import causal_rope_self_neox_b300 as na
    qkv = make_qkv(B, S, H, D, seed=S + 11 * D + r, k_scale=ks)
    f_out, f_lse = run(qkv, r, na.NEOX_ROTATION_FUSED)
    p_out, p_lse = run(qkv, r, na.NEOX_ROTATION_PRE)
    np.testing.assert_array_equal(f_out, p_out)
    np.testing.assert_array_equal(f_lse, p_lse)
    ref_out, ref_lse = oracle.fwd(bf16_bits(qkv), B, S, H, D, r, 1e4)
    assert_close(p_out, p_lse, ref_out, ref_lse, f"B{B} S{S} H{H} D{D} r{r}")


def test_auto_placement_matches_both():
    import causal_rope_self_neox_b300 as na
    qkv = make_qkv(1, 400, 2, 128, seed=77)
    a = run(qkv, 128, na.NEOX_ROTATION_AUTO)
    p = run(qkv, 128, na.NEOX_ROTATION_PRE)
    np.testing.assert_array_equal(a[0], p[0])
    b = run(qkv, 32, na.NEOX_ROTATION_AUTO)
    f = run(qkv, 32, na.NEOX_ROTATION_FUSED)
    np.testing.assert_array_equal(b[0], f[0])


def test_pre_rotated_scratch_survives_a_larger_call_in_between():
    # the rotated copy lives in the library's scratch, grown on demand: a small call after a
    # larger one reuses the grown buffer and still gets its own rows
    import causal_rope_self_neox_b300 as na
    big = make_qkv(2, 1000, 4, 128, seed=5)
    small = make_qkv(1, 200, 2, 64, seed=6)
    run(big, 64, na.NEOX_ROTATION_PRE)
    s_out, s_lse = run(small, 64, na.NEOX_ROTATION_PRE)
    ref_out, ref_lse = oracle.fwd(bf16_bits(small), 1, 200, 2, 64, 64, 1e4)
    assert_close(s_out, s_lse, ref_out, ref_lse, "small after big")
