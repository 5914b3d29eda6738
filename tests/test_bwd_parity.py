"""GPU parity of the backward (neox_attn_bwd) against the fp64 backward oracle, through
the C ABI.  The forward's out and lse come from neox_attn_fwd on the same input.

Tolerances per gradient slot (dq, dk, dv): max abs error <= 1.5e-2 of the slot's
largest reference value, and RMS error <= 8e-3 of the reference's RMS.  They come from
the kernel's rounding points (rotated q', k', the probabilities and ds rounded to bf16
before the tensor cores, outputs rounded to bf16, fp32 everywhere else): restating
those roundings in fp64 on CPU gives at most 6.0e-3 and 3.9e-3 on such shapes, and
tests/test_tolerance_budget.py checks that they stay within half of each bound.
"""
import numpy as np
import pytest
import torch

import oracle
from causal_rope_self_neox_b300.workloads import WORKLOADS, bf16_bits, make_qkv

pytestmark = pytest.mark.gpu

MAX_REL, REL_RMS = 1.5e-2, 8e-3


def make_dout(B, S, H, D, seed):
    g = torch.Generator().manual_seed(seed + 7)
    return torch.randn((B, S, H, D), generator=g).to(torch.bfloat16)


def gpu_bwd(qkv, dout, r):
    import causal_rope_self_neox_b300 as na
    dq = qkv.cuda()
    out, lse = na.attn_fwd(dq, r)
    dqkv = na.attn_bwd(dq, out, lse, dout.cuda(), r)
    na.check_device_error()
    return dqkv.float().cpu().numpy()


def check(got, ref, what):
    assert np.isfinite(got).all(), what
    for slot, name in enumerate(("dq", "dk", "dv")):
        e = got[..., slot, :] - ref[..., slot, :]
        rms_ref = np.sqrt((ref[..., slot, :] ** 2).mean())
        # a slot that is exactly zero by definition (dq, dk of a one-token sequence) has
        # no scale for a relative error: there an absolute bound of 1e-4 applies
        bound = max(MAX_REL * np.abs(ref[..., slot, :]).max(), 1e-4)
        mx, rel = np.abs(e).max(), (np.sqrt((e ** 2).mean()) / rms_ref if rms_ref > 1e-6 else 0.0)
        assert mx <= bound and rel <= REL_RMS, (what, name, mx, bound, rel)


@pytest.mark.parametrize("B,S,H,D,r", [
    (1, 128, 2, 64, 16),
    (2, 300, 3, 64, 16),     # ragged last block, several key blocks
    (1, 256, 2, 96, 24),
    (1, 129, 2, 128, 32),    # one row past a block
    (1, 200, 1, 128, 128),   # every dim rotated
    (2, 64, 2, 96, 0),       # shorter than one block, no rotation
    (1, 1, 2, 64, 16),       # one token: dq = dk = 0, dv = dout
    (1, 384, 1, 96, 6),      # rotary_dim not a multiple of 8
    (1, 1000, 1, 128, 32),
    (1, 700, 2, 96, 24),     # six key blocks, ragged: both query-side buffers cycle (dq' staged in them)
    (1, 300, 2, 128, 40),    # two of four 32-column blocks of q', k' rotated, two read from the input
    (1, 260, 1, 96, 48),     # two of three rotated
    # 150 (key block, head) work items, two more than a 148-SM GPU has CTAs: the first
    # items come from the grid, the rest from the work counter (two query-side buffers,
    # and one at D = 128)
    (1, 1280, 15, 64, 16),
    (1, 1280, 15, 128, 32),
])
def test_bwd_small_shapes(B, S, H, D, r):
    qkv = make_qkv(B, S, H, D, seed=S + D + r)
    dout = make_dout(B, S, H, D, seed=S + D + r)
    got = gpu_bwd(qkv, dout, r)
    ref = oracle.bwd(bf16_bits(qkv), bf16_bits(dout), B, S, H, D, r)
    check(got, ref, f"{B},{S},{H},{D},{r}")


# (b, h) slices per workload: first and last heads, and both sides of each boundary between
# the kernel's L2 head groups (48 MB of Q'/dO per group: 64 heads for neox20b, so the
# groups are the batches; 48 for pythia1.4b, whose 64 heads leave a short second group;
# one group of all 96 heads for pythia160m)
SAMPLED_HEADS = {
    "neox20b": ((0, 0), (0, 37), (0, 63), (1, 0), (1, 63)),
    "pythia1.4b": ((0, 0), (2, 15), (3, 0), (3, 15)),
    "pythia160m": ((0, 0), (4, 7), (7, 11)),
}


@pytest.mark.parametrize("name", sorted(SAMPLED_HEADS))
def test_bwd_workload_sampled_heads(name):
    # the full workload-shaped problem on the GPU, as the benchmark runs it; heads are
    # independent, so a few (b, h) slices are checked against the oracle run on those
    # heads alone
    w = WORKLOADS[name]
    qkv = make_qkv(w.B, w.S, w.H, w.D, w.seed, w.k_scale)
    dout = make_dout(w.B, w.S, w.H, w.D, seed=w.seed)
    got = gpu_bwd(qkv, dout, w.rotary_dim)
    for b, h in SAMPLED_HEADS[name]:
        q1 = qkv[b:b + 1, :, h:h + 1].contiguous()
        g1 = dout[b:b + 1, :, h:h + 1].contiguous()
        ref = oracle.bwd(bf16_bits(q1), bf16_bits(g1), 1, w.S, 1, w.D, w.rotary_dim)
        check(got[b:b + 1, :, h:h + 1], ref, f"{name} b={b} h={h}")


def test_bwd_repeat_calls_dk_dv_bit_identical_dq_within_one_rounding():
    # dk and dv accumulate inside one CTA in a fixed order: bit-identical from call to call.
    # dq' is summed in fp32 by tensor reductions from the CTAs of every key block, in the
    # order they land, so dq may differ by one bf16 rounding of nearly equal fp32 sums
    import causal_rope_self_neox_b300 as na
    B, S, H, D, r = 1, 1100, 3, 96, 24
    qkv = make_qkv(B, S, H, D, seed=31).cuda()
    dout = make_dout(B, S, H, D, seed=31).cuda()
    out, lse = na.attn_fwd(qkv, r)
    g1 = na.attn_bwd(qkv, out, lse, dout, r)
    g2 = na.attn_bwd(qkv, out, lse, dout, r)
    na.check_device_error()
    assert torch.equal(g1[..., 1:, :], g2[..., 1:, :])
    a, b = g1[..., 0, :].float(), g2[..., 0, :].float()
    bound = 2.0 ** -7 * torch.maximum(a.abs(), b.abs()) + 1e-5 * a.abs().max()
    assert bool(((a - b).abs() <= bound).all())
