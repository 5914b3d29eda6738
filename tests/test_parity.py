"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances (unit-normal inputs): bf16 output max abs error <= 2e-2 and RMS error
<= 3e-3; lse max abs error <= 1e-3.  Small and medium problems are checked on every
row; the two largest workloads on 256 seeded (b, h, row) triples plus fixed edge rows.
"""
import numpy as np
import pytest
import torch

import oracle
from causal_rope_self_neox_b300.workloads import WORKLOADS, bf16_bits, make_qkv, sample_rows, workload_qkv

pytestmark = pytest.mark.gpu

OUT_MAX, OUT_RMS, LSE_MAX = 2e-2, 3e-3, 1e-3
KERNELS = ["default", "simple"]


def run_gpu(qkv_cpu: torch.Tensor, r: int, base: float = 10000.0, kernel: str = "default"):
    import causal_rope_self_neox_b300 as na
    qkv = qkv_cpu.cuda()
    out, lse = na.attn_fwd(qkv, r, base, kernel=kernel)
    na.check_device_error()
    return out.float().cpu().numpy().astype(np.float64), lse.cpu().numpy().astype(np.float64)


def assert_close(out, lse, ref_out, ref_lse, what=""):
    e = out - ref_out
    omax, orms, lmax = np.abs(e).max(), np.sqrt((e ** 2).mean()), np.abs(lse - ref_lse).max()
    assert np.isfinite(out).all() and np.isfinite(lse).all(), what
    assert omax <= OUT_MAX and orms <= OUT_RMS and lmax <= LSE_MAX, (what, omax, orms, lmax)
    return omax, orms, lmax


def full_check(B, S, H, D, r, seed, k_scale=1.0, kernel="default"):
    qkv = make_qkv(B, S, H, D, seed, k_scale)
    out, lse = run_gpu(qkv, r, kernel=kernel)
    ref_out, ref_lse = oracle.fwd(bf16_bits(qkv), B, S, H, D, r, 1e4)
    return assert_close(out, lse, ref_out, ref_lse, f"B{B} S{S} H{H} D{D} r{r}")


@pytest.mark.parametrize("kernel", KERNELS)
def test_tiny_workload_every_row(kernel):
    w = WORKLOADS["tiny"]
    full_check(w.B, w.S, w.H, w.D, w.rotary_dim, w.seed, kernel=kernel)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("B,S,H,D,r,ks", [
    (1, 1, 2, 64, 16, 1.0),       # single token
    (1, 129, 2, 64, 16, 1.0),     # ragged tail, one extra row
    (2, 200, 3, 96, 24, 1.0),     # D = 96, ragged
    (1, 300, 2, 128, 128, 3.0),   # full rotary, sharpened softmax
    (1, 384, 2, 128, 32, 1.0),    # three tiles exactly
    (2, 257, 1, 64, 0, 1.0),      # no rotary at all
    (1, 170, 2, 64, 6, 1.0),      # r/2 odd (scalar rotation path)
    (1, 640, 2, 96, 96, 1.0),     # five tiles, every dim rotated
    (3, 523, 2, 128, 64, 1.0),    # several tiles, ragged, half rotary
])
def test_small_shapes_every_row(kernel, B, S, H, D, r, ks):
    full_check(B, S, H, D, r, seed=S * 7 + D + r, k_scale=ks, kernel=kernel)


@pytest.mark.parametrize("name", ["pythia160m", "pythia1.4b"])
def test_medium_workloads_every_row(name):
    w = WORKLOADS[name]
    full_check(w.B, w.S, w.H, w.D, w.rotary_dim, w.seed)


@pytest.mark.parametrize("name", ["neox20b", "long16k"])
def test_large_workloads_sampled_rows(name):
    w = WORKLOADS[name]
    qkv = workload_qkv(w)
    out, lse = run_gpu(qkv, w.rotary_dim)
    rows = sample_rows(w)
    ref_out, ref_lse = oracle.fwd_rows(bf16_bits(qkv), w.B, w.S, w.H, w.D, w.rotary_dim, w.rotary_base, rows)
    got_out = out[rows[:, 0], rows[:, 2], rows[:, 1]]
    got_lse = lse[rows[:, 0], rows[:, 1], rows[:, 2]]
    assert_close(got_out, got_lse, ref_out, ref_lse, name)
    assert np.isfinite(out).all() and np.isfinite(lse).all()


@pytest.mark.parametrize("B,S,H,D,r", [
    (4, 300, 40, 64, 16),    # 320 units: CTAs run several, half of them without a second query tile
    (3, 1100, 50, 96, 24),   # 750 units, ragged last block with a second tile of 76 rows
    (2, 650, 48, 128, 32),   # 288 units, last block without a second tile
])
def test_many_units_per_cta_ragged(B, S, H, D, r):
    # more units than SMs, so each persistent CTA walks several units, mixing units with
    # and without a second query tile; every row is checked
    full_check(B, S, H, D, r, seed=B * S + H)


def test_deterministic_and_causal_on_gpu():
    B, S, H, D, r = 1, 600, 2, 96, 24
    qkv = make_qkv(B, S, H, D, seed=5)
    out1, lse1 = run_gpu(qkv, r)
    out2, lse2 = run_gpu(qkv, r)
    np.testing.assert_array_equal(out1, out2)
    np.testing.assert_array_equal(lse1, lse2)
    cut = 300  # rows <= cut must not see tokens > cut, bit for bit
    qkv2 = qkv.clone()
    qkv2[:, cut + 1:] = make_qkv(B, S - cut - 1, H, D, seed=6)
    out3, lse3 = run_gpu(qkv2, r)
    np.testing.assert_array_equal(out1[:, : cut + 1], out3[:, : cut + 1])
    np.testing.assert_array_equal(lse1[:, :, : cut + 1], lse3[:, :, : cut + 1])


def test_kernels_agree():
    qkv = make_qkv(2, 700, 3, 128, seed=9)
    a_out, a_lse = run_gpu(qkv, 32, kernel="default")
    b_out, b_lse = run_gpu(qkv, 32, kernel="simple")
    assert np.abs(a_out - b_out).max() <= 2 * OUT_MAX
    assert np.abs(a_lse - b_lse).max() <= LSE_MAX


def test_wait_timeout_is_reported_not_hung():
    import causal_rope_self_neox_b300 as na
    torch.cuda.synchronize()
    assert na.neox_attn_get_device_error() == na.NEOX_OK
    assert na.neox_attn_selftest_wait_timeout(2_000_000, torch.cuda.current_stream().cuda_stream) == na.NEOX_OK
    torch.cuda.synchronize()
    assert na.neox_attn_get_device_error() == na.NEOX_ERR_DEVICE_TIMEOUT
    assert na.neox_attn_get_device_error() == na.NEOX_OK  # read clears it
    # the context is still usable
    full_check(1, 130, 1, 64, 16, seed=3)


def test_output_buffers_and_rejections_on_device():
    import causal_rope_self_neox_b300 as na
    qkv = make_qkv(1, 64, 1, 64, seed=1).cuda()
    out = torch.full((1, 64, 1, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((1, 1, 64), 7.0, dtype=torch.float32, device="cuda")
    na.attn_fwd(qkv, 16, out=out, lse=lse)
    torch.cuda.synchronize()
    assert not torch.any(out == 7.0) and not torch.any(lse == 7.0)
    s = torch.cuda.current_stream().cuda_stream
    # out overlapping qkv is rejected without launching
    assert na.neox_attn_fwd(qkv.data_ptr(), 1, 64, 1, 64, 16, 1e4, qkv.data_ptr() + 1024, lse.data_ptr(), s) \
        == na.NEOX_ERR_INVALID_ARG
    assert na.neox_attn_fwd(qkv.data_ptr(), 1, 64, 1, 80, 16, 1e4, out.data_ptr(), lse.data_ptr(), s) \
        == na.NEOX_ERR_UNSUPPORTED_HEAD_DIM


def test_head_and_batch_shards_match_the_full_call_bit_for_bit():
    # every (batch, head) is independent: a rank owning a head range (or a batch range)
    # computes exactly what the full call computes for it
    B, S, H, D, r = 2, 520, 4, 96, 24
    qkv = make_qkv(B, S, H, D, seed=31)
    out, lse = run_gpu(qkv, r)
    o1, l1 = run_gpu(qkv[:, :, 1:3].contiguous(), r)
    np.testing.assert_array_equal(o1, out[:, :, 1:3])
    np.testing.assert_array_equal(l1, lse[:, 1:3])
    o2, l2 = run_gpu(qkv[1:].contiguous(), r)
    np.testing.assert_array_equal(o2, out[1:])
    np.testing.assert_array_equal(l2, lse[1:])
