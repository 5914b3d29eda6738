"""The two placements of the rotary embedding give the same attention.

NEOX_ROTATION_FUSED rotates Q and K tiles inside the attention kernel (shared memory);
NEOX_ROTATION_PRE rotates them once in a separate pass that writes hi and lo of q' and k'
to the library's scratch, which the kernel then loads by TMA.  Both evaluate the same fp32
expressions on the same table entries.  Where both keep the hi/lo split (rotary_dim 64 and
up) the outputs must be bit-identical; at rotary_dim 16, 24 and 32 the in-kernel rotation
rounds the rotated chunks to fp16 instead, so there each placement is held to the oracle
and the two to each other within the tolerances.
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


FP16_CHUNKS = (16, 24, 32)  # rotary_dims whose in-kernel rotation uses fp16 operands


@pytest.mark.parametrize("B,S,H,D,r,ks", SHAPES)
def test_fused_and_pre_rotated_agree_and_match_the_oracle(B, S, H, D, r, ks):
    import causal_rope_self_neox_b300 as na
    qkv = make_qkv(B, S, H, D, seed=S + 11 * D + r, k_scale=ks)
    f_out, f_lse = run(qkv, r, na.NEOX_ROTATION_FUSED)
    p_out, p_lse = run(qkv, r, na.NEOX_ROTATION_PRE)
    ref_out, ref_lse = oracle.fwd(bf16_bits(qkv), B, S, H, D, r, 1e4)
    assert_close(p_out, p_lse, ref_out, ref_lse, f"pre B{B} S{S} H{H} D{D} r{r}")
    if r in FP16_CHUNKS:
        assert_close(f_out, f_lse, ref_out, ref_lse, f"fused B{B} S{S} H{H} D{D} r{r}")
        assert_close(f_out, f_lse, p_out, p_lse, f"fused vs pre B{B} S{S} H{H} D{D} r{r}")
    else:
        np.testing.assert_array_equal(f_out, p_out)
        np.testing.assert_array_equal(f_lse, p_lse)


def test_fp16_operand_range_is_reported_and_the_pass_takes_the_whole_range():
    # A query value in rotated dim 3 at position 5 (pair (3, 15) turned by 0.5 rad): 70000
    # rotates to about 61557 and 33629, inside fp16's 65504, and nothing is reported;
    # 299008 (bf16 of 3e5) rotates to about 262404 and 143352, and the in-kernel rotation
    # reports it.  The pre-rotation pass (hi/lo) takes that input; every row but the
    # altered one against the oracle.
    import causal_rope_self_neox_b300 as na
    B, S, H, D, r = 1, 200, 2, 96, 24
    base = make_qkv(B, S, H, D, seed=31).float()
    inside = base.clone()
    inside[0, 5, 1, 0, 3] = 70000.0
    na.attn_fwd(inside.to(torch.bfloat16).cuda(), r, 1e4, rotation=na.NEOX_ROTATION_FUSED)
    na.check_device_error()
    qkv = base.clone()
    qkv[0, 5, 1, 0, 3] = 3e5
    qkv = qkv.to(torch.bfloat16)
    na.attn_fwd(qkv.cuda(), r, 1e4, rotation=na.NEOX_ROTATION_FUSED)
    with pytest.raises(na.NeoxAttnError) as e:
        na.check_device_error()
    assert e.value.status == na.NEOX_ERR_DEVICE_RANGE
    na.check_device_error()  # the report cleared the error word
    p_out, p_lse = run(qkv, r, na.NEOX_ROTATION_PRE)
    ref_out, ref_lse = oracle.fwd(bf16_bits(qkv), B, S, H, D, r, 1e4)
    keep = np.ones((B, S, H), dtype=bool)
    keep[0, 5, 1] = False
    assert_close(p_out[keep], p_lse.transpose(0, 2, 1)[keep], ref_out[keep], ref_lse.transpose(0, 2, 1)[keep], "pre")


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
