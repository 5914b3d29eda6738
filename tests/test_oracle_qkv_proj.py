"""Pins for the oracle of the fused query_key_value projection and its rotary step.

"GPT-NeoX on FasterTransformer" guide, section "从 HuggingFace 检查点部署": the weight
attention.query_key_value.weight is stored [hidden_size, num_heads, 3, head_hidden], and
the layer list in "从 EleutherAI 检查点部署" includes the projection's bias.  So token t's
output feature (h, slot, d) is sum_k x[t, k] * w[k, h, slot, d] + bias[h, slot, d], and a
token's outputs, in that order, are the packed [H, 3, D] the attention reads.

The oracle is plain C loops; these pins hold it to things it does not compute itself:
numpy's matmul (a library routine the oracle does not call), a one-hot worked example
of the page's weight layout, the identity weight, and, for the rotated form, the
invariants of a rotation (norms kept, value slots and pass-through dims untouched,
scores that depend only on the position difference).  Planted mistakes in a copy of
the C source must each fail one of them.  Nothing here touches a GPU.
"""
import ctypes
import subprocess

import numpy as np
import pytest
import torch

import oracle
from causal_rope_self_neox_b300.workloads import bf16_bits

SRC = oracle._SRC


def _bf16(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


def _case(M, K, N, seed, with_bias=True):
    x = _bf16((M, K), seed)
    w = _bf16((K, N), seed + 1, scale=K ** -0.5)
    b = _bf16((N,), seed + 2) if with_bias else None
    return x, w, b


def _numpy_ref(x, w, b):
    y = x.double().numpy() @ w.double().numpy()
    return y if b is None else y + b.double().numpy()


def _bits(t):
    return None if t is None else bf16_bits(t)


@pytest.mark.parametrize("M,K,N,with_bias", [(1, 8, 6, True), (37, 96, 3 * 2 * 32, True),
                                             (129, 200, 3 * 1 * 64, False), (64, 1024, 3 * 4 * 16, True)])
def test_projection_equals_numpy_matmul(M, K, N, with_bias):
    x, w, b = _case(M, K, N, seed=M + K, with_bias=with_bias)
    got = oracle.qkv_proj(_bits(x), _bits(w), _bits(b))
    ref = _numpy_ref(x, w, b)
    scale = np.abs(x.double().numpy()) @ np.abs(w.double().numpy()) + 1.0
    assert got.shape == (M, N)
    assert np.all(np.abs(got - ref) <= 1e-13 * scale)


def test_listed_rows_equal_the_full_product():
    x, w, b = _case(50, 64, 96, seed=3)
    full = oracle.qkv_proj(_bits(x), _bits(w), _bits(b))
    rows = [49, 0, 17, 17, 3]
    assert np.array_equal(oracle.qkv_proj(_bits(x), _bits(w), _bits(b), rows=rows), full[rows])


def test_weight_layout_one_hot_worked_example():
    # w[k0, h, slot, d] = 1 + 100h + 10slot + d/100 for one hidden feature k0, zero elsewhere;
    # token t holds (t + 1) at feature k0.  Output (t, h, slot, d) is then (t + 1) * w[k0, h, slot, d]
    # placed at the packed index [h, slot, d] of the token's row.
    K, H, D, M, k0 = 16, 3, 8, 4, 5
    w4 = np.zeros((K, H, 3, D))
    hh, ss, dd = np.meshgrid(np.arange(H), np.arange(3), np.arange(D), indexing="ij")
    w4[k0] = 1 + 100 * hh + 10 * ss + dd / 128.0
    x = np.zeros((M, K))
    x[:, k0] = np.arange(1, M + 1)
    xb = bf16_bits(torch.from_numpy(x).to(torch.bfloat16))
    wb = bf16_bits(torch.from_numpy(w4.reshape(K, H * 3 * D)).to(torch.bfloat16))
    got = oracle.qkv_proj(xb, wb).reshape(M, H, 3, D)
    for t in range(M):
        assert np.array_equal(got[t], (t + 1) * torch.from_numpy(w4[k0]).to(torch.bfloat16).double().numpy())


def test_identity_weight_returns_the_input_plus_bias():
    K = 48
    x = _bf16((7, K), 9)
    eye = torch.eye(K).to(torch.bfloat16)
    b = _bf16((K,), 10)
    got = oracle.qkv_proj(_bits(x), _bits(eye), _bits(b))
    assert np.array_equal(got, x.double().numpy() + b.double().numpy())
    assert np.array_equal(oracle.qkv_proj(_bits(x), _bits(eye)), x.double().numpy())


def test_projection_rejects_bad_arguments():
    x, w, b = _case(4, 8, 6, seed=1)
    with pytest.raises(ValueError):
        oracle.qkv_proj(_bits(x), _bits(w)[:7])
    with pytest.raises(RuntimeError):
        oracle.qkv_proj(_bits(x), _bits(w), rows=[4])


# ---------------------------------------------------------------- rotated form ----
def _rot_case(B, S, H, D, seed, same_token=False):
    K = 64
    x = _bf16((B * S, K), seed)
    if same_token:
        x = x[:1].repeat(B * S, 1)
    w = _bf16((K, H * 3 * D), seed + 1, scale=K ** -0.5)
    b = _bf16((H * 3 * D,), seed + 2)
    return x, w, b


def test_rotated_form_with_no_rotary_dims_is_the_plain_projection():
    B, S, H, D = 2, 9, 2, 32
    x, w, b = _rot_case(B, S, H, D, 4)
    plain = oracle.qkv_proj(_bits(x), _bits(w), _bits(b)).reshape(-1, H, 3, D)
    assert np.array_equal(oracle.qkv_proj_rotated(_bits(x), _bits(w), _bits(b), B, S, H, D, 0), plain)


@pytest.mark.parametrize("r", [8, 24, 32])
def test_rotated_form_keeps_values_pass_through_dims_norms_and_position_zero(r):
    B, S, H, D = 2, 11, 3, 32
    x, w, b = _rot_case(B, S, H, D, 5 + r)
    plain = oracle.qkv_proj(_bits(x), _bits(w), _bits(b)).reshape(B, S, H, 3, D)
    rot = oracle.qkv_proj_rotated(_bits(x), _bits(w), _bits(b), B, S, H, D, r).reshape(B, S, H, 3, D)
    assert np.array_equal(rot[..., 2, :], plain[..., 2, :])         # values untouched
    assert np.array_equal(rot[..., :2, r:], plain[..., :2, r:])     # dims past rotary_dim untouched
    assert np.array_equal(rot[:, 0], plain[:, 0])                   # position 0 is the identity
    h = r // 2
    pair_norm = lambda a: a[..., :h] ** 2 + a[..., h:r] ** 2        # each (i, i + r/2) pair keeps its length
    assert np.allclose(pair_norm(rot[..., :2, :]), pair_norm(plain[..., :2, :]), rtol=1e-12, atol=1e-12)
    assert not np.allclose(rot[:, 1:, :, :2, :r], plain[:, 1:, :, :2, :r])


def test_rotated_form_positions_restart_per_sequence_and_scores_depend_on_offset_only():
    B, S, H, D, r = 2, 12, 1, 32, 32
    x, w, b = _rot_case(B, S, H, D, 6, same_token=True)   # every token identical
    rot = oracle.qkv_proj_rotated(_bits(x), _bits(w), _bits(b), B, S, H, D, r).reshape(B, S, H, 3, D)
    assert np.array_equal(rot[0], rot[1])                  # the second sequence starts again at 0
    q, k = rot[0, :, 0, 0], rot[0, :, 0, 1]
    for t, s in [(5, 3), (9, 2)]:
        for shift in (1, 2):
            assert abs(q[t] @ k[s] - q[t + shift] @ k[s + shift]) <= 1e-10 * (1 + abs(q[t] @ k[s]))
    assert abs(q[5] @ k[3] - q[5] @ k[4]) > 1e-6


def test_rotated_form_rows_equal_the_full_result():
    B, S, H, D, r = 2, 7, 2, 32, 24
    x, w, b = _rot_case(B, S, H, D, 8)
    full = oracle.qkv_proj_rotated(_bits(x), _bits(w), _bits(b), B, S, H, D, r)
    rows = [13, 0, 7, 6]
    assert np.array_equal(oracle.qkv_proj_rotated(_bits(x), _bits(w), _bits(b), B, S, H, D, r, rows=rows), full[rows])


# ------------------------------------------------------------ planted mistakes ----
MUTATIONS = {
    "weight_read_transposed": ("o[n] += a * bf16_to_f64(wk[n]);", "o[n] += a * bf16_to_f64(J->w[(int64_t)n * K + k]);"),
    "bias_dropped": ("o[n] = J->bias ? bf16_to_f64(J->bias[n]) : 0.0;", "o[n] = 0.0;"),
    "bias_first_entry_only": ("o[n] = J->bias ? bf16_to_f64(J->bias[n]) : 0.0;",
                              "o[n] = J->bias ? bf16_to_f64(J->bias[0]) : 0.0;"),
    "output_column_shifted": ("o[n] += a * bf16_to_f64(wk[n]);", "o[n] += a * bf16_to_f64(wk[(n + 1) % N]);"),
    "last_hidden_feature_dropped": ("for (int k = 0; k < K; ++k) {\n      const uint16_t* wk",
                                    "for (int k = 0; k < K - 1; ++k) {\n      const uint16_t* wk"),
    "listed_rows_ignored": ("const int64_t t = J->rows ? J->rows[it] : it;", "const int64_t t = it;"),
}


def _build_mutant(tmp_path, name):
    src = open(SRC).read()
    if name is not None:
        old, new = MUTATIONS[name]
        assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
        src = src.replace(old, new)
    path = tmp_path / "m.c"
    path.write_text(src)
    so = tmp_path / "m.so"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-D_POSIX_C_SOURCE=200809L",
                           str(path), "-o", str(so), "-lm", "-lpthread"])
    lib = ctypes.CDLL(str(so))
    P = ctypes.c_void_p
    lib.neox_oracle_qkv_proj.argtypes = [P, P, P, ctypes.c_int64, ctypes.c_int, ctypes.c_int, P, ctypes.c_int64,
                                         P, ctypes.c_int]
    lib.neox_oracle_qkv_proj.restype = ctypes.c_int
    return lib


def _pins_pass(lib) -> bool:
    p = lambda a: None if a is None else a.ctypes.data_as(ctypes.c_void_p)
    ok = True
    for M, K, N, rows in [(9, 40, 24, None), (12, 16, 18, np.array([11, 2, 5], dtype=np.int64))]:
        x, w, b = _case(M, K, N, seed=K)
        xb, wb, bb = (np.ascontiguousarray(_bits(t)) for t in (x, w, b))
        n = M if rows is None else rows.shape[0]
        out = np.zeros((n, N))
        rc = lib.neox_oracle_qkv_proj(p(xb), p(wb), p(bb), M, K, N, p(rows), 0 if rows is None else n, p(out), 1)
        ref = _numpy_ref(x, w, b)
        ref = ref if rows is None else ref[rows]
        ok &= rc == 0 and bool(np.allclose(out, ref, rtol=0, atol=1e-12))
    return ok


def test_unmodified_projection_copy_passes(tmp_path):
    assert _pins_pass(_build_mutant(tmp_path, None))


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_projection_mistake_is_caught(tmp_path, name):
    assert not _pins_pass(_build_mutant(tmp_path, name))


def test_bf16_steps_round_before_and_after_the_rotation():
    B, S, H, D, r = 1, 9, 2, 32, 16
    x, w, b = _rot_case(B, S, H, D, 12)
    plain = oracle.qkv_proj(_bits(x), _bits(w), _bits(b)).reshape(-1, H, 3, D)
    got = oracle.qkv_proj_rotated(_bits(x), _bits(w), _bits(b), B, S, H, D, r, bf16_steps=True)
    y = torch.from_numpy(plain).to(torch.bfloat16).double().numpy()
    assert np.array_equal(got[..., 2, :], y[..., 2, :])    # values: one rounding, no rotation
    assert np.array_equal(got[0], y[0])                    # position 0: the rotation is the identity
    for t in (3, 8):
        want = oracle.rotate(y[t, 1, 0], t, r, 1e4)
        assert np.array_equal(got[t, 1, 0], torch.from_numpy(want).to(torch.bfloat16).double().numpy())
    # every result is a bf16 value
    assert np.array_equal(got, torch.from_numpy(got).to(torch.bfloat16).double().numpy())
