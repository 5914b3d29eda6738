"""Dense numpy restatement of causal rotary attention, for tiny inputs only.

Independent of the oracle's element loops: the rotation is a dense D x D matrix
per position, the scores a full S x S matrix, the mask ``np.tril``, and the row
normaliser ``scipy.special.logsumexp``.  Used to pin the oracle on small cases.
"""
from __future__ import annotations

import numpy as np
from scipy.special import logsumexp


def rotation_matrix(D: int, r: int, base: float, p: int) -> np.ndarray:
    """R(p) with R(p) @ x the rotate-half embedding of x at position p.

    Each pair (i, i + r/2), i < r/2, is a plane rotation by p * base^(-2i/r);
    dims >= r are the identity."""
    R = np.eye(D)
    h = r // 2
    for i in range(h):
        t = p * float(base) ** (-2.0 * i / r)
        c, s = np.cos(t), np.sin(t)
        R[np.ix_([i, i + h], [i, i + h])] = [[c, -s], [s, c]]
    return R


def causal_rope_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, r: int, base: float):
    """q, k, v: [S, D] fp64 of one head.  Returns out[S, D], lse[S], P[S, S]."""
    S, D = q.shape
    Rs = np.stack([rotation_matrix(D, r, base, p) for p in range(S)])  # [S, D, D]
    qr = np.einsum("sij,sj->si", Rs, q)
    kr = np.einsum("sij,sj->si", Rs, k)
    scores = (qr @ kr.T) / np.sqrt(D)
    mask = np.tril(np.ones((S, S), dtype=bool))
    scores = np.where(mask, scores, -np.inf)
    lse = logsumexp(scores, axis=1)
    P = np.exp(scores - lse[:, None])
    return P @ v, lse, P


def qkv_to_heads(qkv_f64: np.ndarray):
    """Split packed [B,S,H,3,D] into per-(b,h) q, k, v arrays of shape [B,H,S,D]."""
    t = np.transpose(qkv_f64, (0, 2, 3, 1, 4))  # [B,H,3,S,D]
    return t[:, :, 0], t[:, :, 1], t[:, :, 2]


def brute_force(qkv_f64: np.ndarray, r: int, base: float):
    """Whole problem.  Returns out[B,S,H,D] and lse[B,H,S]."""
    B, S, H, _, D = qkv_f64.shape
    q, k, v = qkv_to_heads(qkv_f64)
    out = np.empty((B, S, H, D))
    lse = np.empty((B, H, S))
    for b in range(B):
        for h in range(H):
            o, l, _ = causal_rope_attention(q[b, h], k[b, h], v[b, h], r, base)
            out[b, :, h, :] = o
            lse[b, h] = l
    return out, lse
