"""GPU parity of the ALiBi forward (neox_attn_fwd_alibi) against the fp64 ALiBi oracle.

ALiBi is the pages' other positional scheme for GPT-NeoX: no rotation, a linear bias
-m_h (i - j) on every score (slopes of the published method, pinned in
tests/test_oracle_alibi.py).  The kernel is the forward kernel with the bias added in
the softmax; tolerances are the forward's (out max abs <= 2e-2, RMS <= 3e-3, lse max abs
<= 1e-3).  Head counts cover powers of two and the extra odd-numbered slopes (H = 12, 5).
"""
import numpy as np
import pytest
import torch

import oracle
from causal_rope_self_neox_b300.workloads import WORKLOADS, bf16_bits, make_qkv
from test_parity import assert_close

pytestmark = pytest.mark.gpu


def run_alibi(qkv_cpu):
    import causal_rope_self_neox_b300 as na
    out, lse = na.attn_fwd_alibi(qkv_cpu.cuda())
    na.check_device_error()
    return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("B,S,H,D", [
    (1, 128, 2, 64),      # one tile
    (2, 200, 3, 96),      # ragged, H not a power of two
    (1, 523, 5, 128),     # several tiles, ragged, extra slopes
    (2, 300, 12, 64),     # the pythia-160M head count (8 + 4 extra slopes)
    (1, 1100, 8, 96),     # many blocks, power of two
])
def test_alibi_matches_the_oracle_on_every_row(B, S, H, D):
    qkv = make_qkv(B, S, H, D, seed=B * S + H * D)
    out, lse = run_alibi(qkv)
    ref_out, ref_lse = oracle.fwd_alibi(bf16_bits(qkv), B, S, H, D)
    assert_close(out, lse, ref_out, ref_lse, f"alibi B{B} S{S} H{H} D{D}")


def test_alibi_on_the_neox20b_shape_every_row():
    w = WORKLOADS["neox20b"]
    qkv = make_qkv(w.B, w.S, w.H, w.D, seed=w.seed)
    out, lse = run_alibi(qkv)
    ref_out, ref_lse = oracle.fwd_alibi(bf16_bits(qkv), w.B, w.S, w.H, w.D)
    assert_close(out, lse, ref_out, ref_lse, "alibi neox20b")


def test_alibi_is_deterministic_and_differs_from_plain_causal():
    import causal_rope_self_neox_b300 as na
    qkv = make_qkv(1, 400, 4, 96, seed=41)
    a1, l1 = run_alibi(qkv)
    a2, l2 = run_alibi(qkv)
    np.testing.assert_array_equal(a1, a2)
    np.testing.assert_array_equal(l1, l2)
    out, lse = na.attn_fwd(qkv.cuda(), 0, 1e4)  # no bias, no rotation
    assert np.abs(out.float().cpu().numpy() - a1).max() > 1e-2
