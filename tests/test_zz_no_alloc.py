"""The allocation-free entry point, neox_attn_fwd_noalloc.

It exists for callers that cannot let a library call cudaMalloc: a framework or
server whose own allocator already holds nearly all GPU memory, or a request path
where cudaMalloc/cudaFree (which can synchronize the device) are not allowed.  It keeps
its cos/sin table in one fixed 8 MiB array inside the library instead of allocating
one.  These tests call it through the C ABI: its results must equal the regular entry
point's bit for bit (the same kernel on a table of the same values), on consecutive
calls with different shapes (the shared array keeps the previous call's contents, so each
call must rebuild what it reads), at the array's exact size limit against the oracle,
and a call must leave the device's free memory unchanged.  The file is named to run last.
"""
import numpy as np
import pytest
import torch

import oracle
from causal_rope_self_neox_b300.workloads import bf16_bits, make_qkv

OUT_MAX, OUT_RMS, LSE_MAX = 2e-2, 3e-3, 1e-3


def _regular(qkv, r, base=10000.0):
    import causal_rope_self_neox_b300 as na
    out, lse = na.attn_fwd(qkv, r, base)
    return out, lse


def _noalloc(qkv, r, base=10000.0, out=None, lse=None):
    import causal_rope_self_neox_b300 as na
    B, S, H, _, D = qkv.shape
    if out is None:
        out = torch.full((B, S, H, D), float("nan"), dtype=torch.bfloat16, device=qkv.device)
    if lse is None:
        lse = torch.full((B, H, S), float("nan"), dtype=torch.float32, device=qkv.device)
    rc = na.neox_attn_fwd_noalloc(qkv.data_ptr(), B, S, H, D, r, base, out.data_ptr(), lse.data_ptr(),
                                  torch.cuda.current_stream().cuda_stream)
    assert rc == na.NEOX_OK, na.status_string(rc)
    return out, lse


@pytest.mark.gpu
def test_noalloc_equals_the_regular_entry_point_bit_for_bit_on_consecutive_calls():
    import causal_rope_self_neox_b300 as na
    # growing S with a new rotary_dim, then a smaller S with the same rotary_dim after a
    # larger one: every call must rebuild the rows of the shared table it reads
    for B, S, H, D, r, seed in [(2, 700, 3, 96, 24, 11), (1, 1100, 2, 128, 64, 12), (1, 300, 2, 128, 64, 13)]:
        qkv = make_qkv(B, S, H, D, seed).cuda()
        out, lse = _noalloc(qkv, r)
        ref_out, ref_lse = _regular(qkv, r)
        na.check_device_error()
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse), (S, r)


@pytest.mark.gpu
def test_noalloc_at_the_table_limit_against_the_oracle():
    import causal_rope_self_neox_b300 as na
    # S * rotary_dim / 2 == 1048576: the last table row is the array's last entry
    B, S, H, D, r = 1, 16384, 1, 128, 128
    qkv_cpu = make_qkv(B, S, H, D, seed=21, k_scale=3.0)
    out, lse = _noalloc(qkv_cpu.cuda(), r)
    na.check_device_error()
    rng = np.random.default_rng(22)
    rows_i = np.unique(np.concatenate([rng.choice(S, size=48, replace=False), [0, 1, S // 2, S - 2, S - 1]]))
    rows = np.stack([np.zeros_like(rows_i), np.zeros_like(rows_i), rows_i], axis=1).astype(np.int64)
    ref_out, ref_lse = oracle.fwd_rows(bf16_bits(qkv_cpu), B, S, H, D, r, 1e4, rows)
    got_out = out.float().cpu().numpy().astype(np.float64)[0, rows_i, 0]
    got_lse = lse.cpu().numpy().astype(np.float64)[0, 0, rows_i]
    e = got_out - ref_out
    assert np.isfinite(got_out).all() and np.isfinite(got_lse).all()
    assert np.abs(e).max() <= OUT_MAX and np.sqrt((e ** 2).mean()) <= OUT_RMS
    assert np.abs(got_lse - ref_lse).max() <= LSE_MAX


@pytest.mark.gpu
def test_noalloc_call_leaves_free_device_memory_unchanged():
    import causal_rope_self_neox_b300 as na
    qkv = make_qkv(1, 500, 2, 96, seed=31).cuda()
    out = torch.empty((1, 500, 2, 96), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((1, 2, 500), dtype=torch.float32, device="cuda")
    _noalloc(qkv, 24, out=out, lse=lse)  # loads the library's module on this device
    torch.cuda.synchronize()
    free_before = torch.cuda.mem_get_info()[0]
    # a (rotary_dim, base) pair no earlier call used: the regular entry point would build
    # and cache a new table here; this one must not allocate
    _noalloc(qkv, 48, base=5000.0, out=out, lse=lse)
    torch.cuda.synchronize()
    na.check_device_error()
    assert torch.cuda.mem_get_info()[0] == free_before
    ref_out, ref_lse = _regular(qkv, 48, 5000.0)
    assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)


def test_noalloc_rejects_tables_beyond_its_fixed_size():
    import causal_rope_self_neox_b300 as na
    # validation happens before any CUDA call: the addresses are never dereferenced
    A, OUT, LSE = 0x10000000, 0x80000000, 0xC0000000
    assert na.neox_attn_fwd_noalloc(A, 1, 16385, 1, 128, 128, 1e4, OUT, LSE, 0) == na.NEOX_ERR_TOO_LARGE
    assert "1048576" in na.neox_attn_status_string(na.NEOX_ERR_TOO_LARGE)
    assert na.neox_attn_fwd_noalloc(0, 1, 128, 1, 128, 128, 1e4, OUT, LSE, 0) == na.NEOX_ERR_INVALID_ARG
