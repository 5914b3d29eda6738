"""GPU parity of the incremental decode (neox_attn_decode) against the fp64 decode oracle,
through the C ABI, plus the cache-append contract and the device-side position check."""
import numpy as np
import pytest
import torch

import oracle
from causal_rope_self_neox_b300.workloads import (DECODE_WORKLOADS, bf16_bits, decode_from_sequence,
                                                  make_decode_inputs, make_qkv)

pytestmark = pytest.mark.gpu

OUT_MAX, OUT_RMS, LSE_MAX = 2e-2, 3e-3, 1e-3


def run_decode(new, kc, vc, pos, r, base=10000.0):
    import causal_rope_self_neox_b300 as na
    dn, dk, dv = new.cuda(), kc.clone().cuda(), vc.clone().cuda()
    dp = torch.tensor(pos, dtype=torch.int32, device="cuda")
    out, lse = na.attn_decode(dn, dk, dv, dp, r, base)
    na.check_device_error()
    return out.float().cpu().numpy(), lse.cpu().numpy(), dk.cpu(), dv.cpu()


def check(new, kc, vc, pos, r, what=""):
    B, H, _, D = new.shape
    Smax = kc.shape[2]
    out, lse, dk, dv = run_decode(new, kc, vc, pos, r)
    ref_out, ref_lse = oracle.decode(bf16_bits(new), bf16_bits(kc), bf16_bits(vc), pos, B, H, Smax, D, r)
    e = out - ref_out
    omax, orms, lmax = np.abs(e).max(), np.sqrt((e ** 2).mean()), np.abs(lse - ref_lse).max()
    assert np.isfinite(out).all() and np.isfinite(lse).all(), what
    assert omax <= OUT_MAX and orms <= OUT_RMS and lmax <= LSE_MAX, (what, omax, orms, lmax)
    # the new token's raw k / v land in row pos[b]; every other row is untouched
    for b in range(B):
        p = pos[b]
        assert torch.equal(dk[b, :, p].view(torch.int16), new[b, :, 1].view(torch.int16))
        assert torch.equal(dv[b, :, p].view(torch.int16), new[b, :, 2].view(torch.int16))
        mask = torch.ones(Smax, dtype=torch.bool)
        mask[p] = False
        assert torch.equal(dk[b][:, mask].view(torch.int16), kc[b][:, mask].view(torch.int16))
        assert torch.equal(dv[b][:, mask].view(torch.int16), vc[b][:, mask].view(torch.int16))
    return omax, orms, lmax


@pytest.mark.parametrize("B,H,Smax,D,r,pos", [
    (1, 1, 8, 64, 16, [0]),                  # the first token: only itself
    (2, 3, 300, 64, 16, [1, 299]),           # second token; last row of a ragged cache
    (3, 2, 384, 96, 24, [127, 128, 129]),    # tile edges
    (2, 4, 1000, 128, 32, [999, 517]),
    (2, 2, 200, 96, 0, [150, 3]),            # no rotary dims
    (1, 3, 260, 128, 128, [259]),            # full rotary (per-key table path)
    (2, 2, 140, 64, 6, [139, 64]),           # odd rotary chunk
    (2, 2, 700, 96, 96, [600, 699]),         # rotary_dim = D (per-key table path)
])
def test_decode_small_shapes(B, H, Smax, D, r, pos):
    new, kc, vc = make_decode_inputs(B, H, Smax, D, seed=Smax * 3 + D + r)
    check(new, kc, vc, pos, r, f"{B},{H},{Smax},{D},{r},{pos}")


def test_decode_matches_the_prefill_problem_row():
    # a real sequence split into cache + new token: the decode answer is the prefill's row
    B, S, H, D, r = 2, 520, 4, 96, 24
    qkv = make_qkv(B, S, H, D, seed=77)
    pos = [519, 260]
    new, kc, vc = decode_from_sequence(qkv, pos, S)
    out, lse, _, _ = run_decode(new, kc, vc, pos, r)
    rows = np.array([[b, h, pos[b]] for b in range(B) for h in range(H)], dtype=np.int64)
    ref_out, ref_lse = oracle.fwd_rows(bf16_bits(qkv), B, S, H, D, r, 10000.0, rows)
    e = out.reshape(B * H, D) - ref_out
    assert np.abs(e).max() <= OUT_MAX and np.abs(lse.reshape(-1) - ref_lse).max() <= LSE_MAX


@pytest.mark.parametrize("name", list(DECODE_WORKLOADS))
def test_decode_workloads_every_head(name):
    w = DECODE_WORKLOADS[name]
    new, kc, vc = make_decode_inputs(w.B, w.H, w.Smax, w.D, w.seed)
    check(new, kc, vc, [w.pos] * w.B, w.rotary_dim, name)


def test_decode_bad_position_is_reported_and_the_context_survives():
    import causal_rope_self_neox_b300 as na
    B, H, Smax, D = 2, 2, 64, 64
    new, kc, vc = make_decode_inputs(B, H, Smax, D, seed=3)
    dn, dk, dv = new.cuda(), kc.cuda(), vc.cuda()
    dp = torch.tensor([5, Smax], dtype=torch.int32, device="cuda")  # second one out of range
    na.attn_decode(dn, dk, dv, dp, 16)
    torch.cuda.synchronize()
    assert na.neox_attn_get_device_error() == na.NEOX_ERR_DEVICE_BAD_POSITION
    assert na.neox_attn_get_device_error() == na.NEOX_OK
    assert torch.equal(dk[1].cpu().view(torch.int16), kc[1].view(torch.int16))  # nothing written for b = 1
    check(new, kc, vc, [5, 63], 16, "after a bad position")


def test_decode_repeated_calls_are_bit_identical():
    # heads split between several CTAs merge through per-head arrival counters that each
    # call must leave at zero: a second and third call give the same bits
    import causal_rope_self_neox_b300 as na
    B, H, Smax, D = 3, 5, 1200, 96
    new, kc, vc = make_decode_inputs(B, H, Smax, D, seed=11)
    dn, dk, dv = new.cuda(), kc.cuda(), vc.cuda()
    dp = torch.tensor([1199, 640, 5], dtype=torch.int32, device="cuda")
    outs = []
    for _ in range(3):
        out, lse = na.attn_decode(dn, dk, dv, dp, 24)
        outs.append((out.view(torch.int16).cpu(), lse.cpu()))
    na.check_device_error()
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l.view(torch.int32), outs[0][1].view(torch.int32))
    check(new, kc, vc, [1199, 640, 5], 24, "after repeated calls")
