"""The allocation-free entry point, neox_attn_fwd_noalloc.

It exists for callers that cannot let a library call cudaMalloc: a framework or
server whose own allocator already holds nearly all GPU memory, or a request path
where cudaMalloc/cudaFree (which can synchronize the device) are not allowed.  It keeps
its cos/sin table in one fixed 8 MiB array inside the library instead of allocating
one.  These tests call it through the C ABI and hold its results to the parity
tolerances against the regular entry point, on two calls in a row with different
shapes (the shared array keeps the previous call's contents, so the second call
must rebuild what it reads).  The file is named to run last.
"""
import numpy as np
import pytest
import torch

import causal_rope_self_neox_b300 as na
from causal_rope_self_neox_b300.workloads import make_qkv

OUT_MAX, OUT_RMS, LSE_MAX = 2e-2, 3e-3, 1e-3


def _regular(qkv, r):
    out, lse = na.attn_fwd(qkv, r, 10000.0)
    return out, lse


def _noalloc(qkv, r):
    B, S, H, _, D = qkv.shape
    out = torch.full((B, S, H, D), float("nan"), dtype=torch.bfloat16, device=qkv.device)
    lse = torch.full((B, H, S), float("nan"), dtype=torch.float32, device=qkv.device)
    rc = na.neox_attn_fwd_noalloc(qkv.data_ptr(), B, S, H, D, r, 10000.0, out.data_ptr(), lse.data_ptr(),
                                  torch.cuda.current_stream().cuda_stream)
    assert rc == na.NEOX_OK, na.status_string(rc)
    return out, lse


@pytest.mark.gpu
def test_noalloc_matches_the_regular_entry_point_on_two_calls_in_a_row():
    for B, S, H, D, r, seed in [(2, 700, 3, 96, 24, 11), (1, 1100, 2, 128, 64, 12)]:
        qkv = make_qkv(B, S, H, D, seed).cuda()
        ref_out, ref_lse = _regular(qkv, r)
        out, lse = _noalloc(qkv, r)
        na.check_device_error()
        e = (out.double() - ref_out.double()).cpu().numpy()
        le = (lse.double() - ref_lse.double()).abs().max().item()
        assert np.isfinite(e).all() and np.isfinite(le)
        assert np.abs(e).max() <= OUT_MAX and np.sqrt((e ** 2).mean()) <= OUT_RMS and le <= LSE_MAX


def test_noalloc_rejects_tables_beyond_its_fixed_size():
    # validation happens before any CUDA call: the addresses are never dereferenced
    A, OUT, LSE = 0x10000000, 0x80000000, 0xC0000000
    assert na.neox_attn_fwd_noalloc(A, 1, 16385, 1, 128, 128, 1e4, OUT, LSE, 0) == na.NEOX_ERR_TOO_LARGE
    assert "1048576" in na.neox_attn_status_string(na.NEOX_ERR_TOO_LARGE)
    assert na.neox_attn_fwd_noalloc(0, 1, 128, 1, 128, 128, 1e4, OUT, LSE, 0) == na.NEOX_ERR_INVALID_ARG
