"""Does the planned GPU arithmetic fit the parity tolerances?  (numpy, no GPU)

The tolerances for unit-normal inputs are: bf16 output max abs error <= 2e-2,
RMS <= 3e-3, lse max abs error <= 1e-3 (against the fp64 oracle).

The kernel multiplies bf16 operands on the tensor cores with fp32 accumulation.
The rotated Q/K dims come out of an fp32 rotation; rounding them to bf16 costs
about 2^-9 relative per element, which on rows with few keys (row 0's lse is a
single score) is too much.  The kernel therefore splits each rotated value into
hi = bf16(y) and lo = bf16(y - hi) and accumulates q_hi.k_hi + q_hi.k_lo +
q_lo.k_hi (the lo.lo term is ~2^-18 relative and dropped).  This test emulates
both schemes around the oracle and shows that only the split one fits.  At rotary_dim 16,
24 and 32 the in-kernel rotation instead rounds the rotated 16-column chunks (dims 0..15,
or 0..31) once to fp16, 11 significant bits to bf16's 8, with no lo products; its
emulation has to fit as well.
"""
import math

import numpy as np
import pytest

import oracle
from causal_rope_self_neox_b300.workloads import bf16_bits, make_qkv

OUT_MAX, OUT_RMS, LSE_MAX = 2e-2, 3e-3, 1e-3


def bf16_round(x):
    """fp32 -> bf16 round-to-nearest-even, returned as fp64."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def f16_round(x):
    """fp32 -> fp16 round-to-nearest-even, returned as fp64."""
    return np.asarray(x, dtype=np.float32).astype(np.float16).astype(np.float64)


def rotate_f32(x, r, base):
    """fp32 rotation with an fp64-built, fp32-stored cos/sin table (the kernel's numerics)."""
    S, D = x.shape
    h = r // 2
    y = x.astype(np.float32).copy()
    if h == 0:
        return y.astype(np.float64)
    inv = base ** (-2.0 * np.arange(h) / r)
    th = np.arange(S)[:, None] * inv[None, :]
    c, s = np.cos(th).astype(np.float32), np.sin(th).astype(np.float32)
    x1, x2 = x[:, :h].astype(np.float32), x[:, h:r].astype(np.float32)
    y[:, :h] = x1 * c - x2 * s
    y[:, h:r] = x2 * c + x1 * s
    return y.astype(np.float64)


def emulate(q, k, v, r, base, rows, split):
    S, D = q.shape
    qr, kr = rotate_f32(q, r, base), rotate_f32(k, r, base)
    qh, kh = bf16_round(qr), bf16_round(kr)
    if split == "f16":  # the first ceil(r/16) 16-column chunks in fp16, the rest exact bf16
        f = 16 * ((r + 15) // 16)
        qh, kh = qr.copy(), kr.copy()
        qh[:, :f], kh[:, :f] = f16_round(qr[:, :f]), f16_round(kr[:, :f])
        split = False
    if split:
        ql, kl = bf16_round(qr - qh), bf16_round(kr - kh)
    c = math.log2(math.e) / math.sqrt(D)
    outs, lses = [], []
    for i in rows:
        s = kh[: i + 1] @ qh[i]
        if split:
            s = s + kl[: i + 1] @ qh[i] + kh[: i + 1] @ ql[i]
        t = (s.astype(np.float32) * np.float32(c)).astype(np.float64)
        m = t.max()
        p = np.exp2(t - m).astype(np.float32).astype(np.float64)
        l = float(np.float32(p.sum()))
        o = (bf16_round(p) @ v[: i + 1]).astype(np.float32).astype(np.float64)
        outs.append(bf16_round(o / l))
        lses.append((m + math.log2(l)) * math.log(2.0))
    return np.array(outs), np.array(lses)


def errors(B, S, H, D, r, seed, k_scale, rows_per_head, split):
    qkv = make_qkv(B, S, H, D, seed=seed, k_scale=k_scale)
    x = qkv.double().numpy()
    rng = np.random.default_rng(seed)
    sel = []
    for b in range(B):
        for h in range(H):
            rows = np.arange(S) if rows_per_head >= S else np.concatenate(
                [[0, 1], np.sort(rng.choice(np.arange(2, S), rows_per_head - 2, replace=False))])
            sel += [(b, h, int(i)) for i in rows]
    ref_o, ref_l = oracle.fwd_rows(bf16_bits(qkv), B, S, H, D, r, 1e4, sel)
    eo, el = [], []
    for b in range(B):
        for h in range(H):
            idx = [k for k, t in enumerate(sel) if t[0] == b and t[1] == h]
            rows = [sel[k][2] for k in idx]
            o, l = emulate(x[b, :, h, 0], x[b, :, h, 1], x[b, :, h, 2], r, 1e4, rows, split)
            eo.append(o - ref_o[idx])
            el.append(l - ref_l[idx])
    eo, el = np.concatenate(eo), np.concatenate(el)
    return np.abs(eo).max(), math.sqrt((eo ** 2).mean()), np.abs(el).max()


CASES = {  # name: (B, S, H, D, r, seed, k_scale, rows_per_head)
    "tiny": (1, 128, 2, 64, 16, 1001, 1.0, 128),
    "d96_r24": (1, 512, 1, 96, 24, 7, 1.0, 48),
    "long_like": (1, 1024, 1, 128, 128, 9, 3.0, 32),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_split_scheme_fits_tolerances(name):
    omax, orms, lmax = errors(*CASES[name], split=True)
    assert omax <= OUT_MAX / 2 and orms <= OUT_RMS / 2 and lmax <= LSE_MAX / 10, (omax, orms, lmax)


@pytest.mark.parametrize("name", ["tiny", "d96_r24", "d128_r32"])
def test_fp16_chunk_scheme_fits_tolerances(name):
    cases = dict(CASES, d128_r32=(1, 512, 1, 128, 32, 11, 1.0, 48))
    omax, orms, lmax = errors(*cases[name], split="f16")
    assert omax <= OUT_MAX / 2 and orms <= OUT_RMS / 2 and lmax <= LSE_MAX / 2, (omax, orms, lmax)


def test_plain_bf16_rotation_breaks_lse_tolerance():
    _, _, lmax = errors(*CASES["tiny"], split=False)
    assert lmax > LSE_MAX, lmax


# ------------------------------------------------------------------- backward ----
# The backward kernel rounds the rotated q', k' to bf16 once (no hi/lo split), rounds the
# probabilities P and ds to bf16 before its MMAs, takes delta from the forward's bf16
# out and the fp32 lse, and writes bf16 gradients; everything else is fp32.  Restating
# those rounding points in fp64 must stay well inside the GPU test's tolerances.
BWD_MAX_REL, BWD_REL_RMS = 1.5e-2, 8e-3  # max abs error / max |ref|; RMS error / RMS ref


def emulate_bwd(qkv, dout, r, base=10000.0):
    """Gradients with the kernel's rounding points, fp64 elsewhere.  qkv, dout: fp64."""
    B, S, H, _, D = qkv.shape
    res = np.zeros((B, S, H, 3, D))
    mask = np.tril(np.ones((S, S), dtype=bool))
    h2 = r // 2
    ang = np.arange(S)[:, None] * (base ** (-2.0 * np.arange(h2) / r))[None, :] if h2 else np.zeros((S, 0))
    c, s = np.cos(ang), np.sin(ang)

    def rot(x, sign):
        y = x.copy()
        y[:, :h2] = x[:, :h2] * c - sign * x[:, h2:r] * s
        y[:, h2:r] = x[:, h2:r] * c + sign * x[:, :h2] * s
        return y

    for b in range(B):
        for h in range(H):
            q, k, v = rot(qkv[b, :, h, 0], 1), rot(qkv[b, :, h, 1], 1), qkv[b, :, h, 2]
            g = dout[b, :, h]
            sc = np.where(mask, q @ k.T / math.sqrt(D), -np.inf)
            mx = sc.max(1, keepdims=True)
            lse = (mx + np.log(np.exp(sc - mx).sum(1, keepdims=True)))[:, 0]
            out = bf16_round(np.exp(sc - lse[:, None]) @ v)
            qb, kb = bf16_round(q), bf16_round(k)
            p = np.where(mask, np.exp(qb @ kb.T / math.sqrt(D) - np.float32(lse)[:, None]), 0.0)
            ds = p * (g @ v.T - (g * out).sum(1)[:, None]) / math.sqrt(D)
            pb, dsb = bf16_round(p), bf16_round(ds)
            res[b, :, h, 0] = bf16_round(rot(dsb @ kb, -1))
            res[b, :, h, 1] = bf16_round(rot(dsb.T @ qb, -1))
            res[b, :, h, 2] = bf16_round(pb.T @ g)
    return res


@pytest.mark.parametrize("B,S,H,D,r", [(1, 300, 2, 64, 16), (1, 256, 2, 96, 24), (1, 200, 1, 128, 128),
                                       (1, 129, 2, 128, 32), (1, 384, 1, 96, 6)])
def test_bwd_rounding_points_fit_tolerances_with_margin(B, S, H, D, r):
    import torch
    qkv = make_qkv(B, S, H, D, seed=S + D + r)
    dout = torch.randn((B, S, H, D), generator=torch.Generator().manual_seed(S + D + r + 7)).to(torch.bfloat16)
    ref = oracle.bwd(bf16_bits(qkv), bf16_bits(dout), B, S, H, D, r)
    got = emulate_bwd(qkv.to(torch.float64).numpy(), dout.to(torch.float64).numpy(), r)
    for slot in range(3):
        e = got[..., slot, :] - ref[..., slot, :]
        rel = np.sqrt((e ** 2).mean()) / np.sqrt((ref[..., slot, :] ** 2).mean())
        mrel = np.abs(e).max() / np.abs(ref[..., slot, :]).max()
        assert mrel <= BWD_MAX_REL / 2 and rel <= BWD_REL_RMS / 2, (slot, mrel, rel)


# ------------------------------------------------------------------- decode ----
# The decode kernel never reads the angle of key 128 t + row from the table directly for
# rotary_dim <= 32: it multiplies the fp32 table entries (cos, sin)(128 t w) and
# (cos, sin)(row w) (angle addition).  The product must stay far below bf16's 2^-9.
@pytest.mark.parametrize("r", [8, 16, 24, 32])
def test_decode_angle_addition_error(r):
    base, h = 10000.0, r // 2
    w = base ** (-2.0 * np.arange(h) / r)
    f32 = lambda x: np.asarray(x, dtype=np.float32).astype(np.float64)
    worst = 0.0
    for t in (0, 1, 7, 15, 63, 127):  # tiles up to position 16383
        for row in (0, 1, 37, 127):
            a, b = 128 * t * w, row * w
            ct, st, cr, sr = f32(np.cos(a)), f32(np.sin(a)), f32(np.cos(b)), f32(np.sin(b))
            c = f32(f32(ct * cr) - f32(st * sr))
            s = f32(f32(st * cr) + f32(ct * sr))
            worst = max(worst, np.abs(c - np.cos(a + b)).max(), np.abs(s - np.sin(a + b)).max())
    assert worst < 1e-6, worst  # 2^-9 = 2.0e-3
