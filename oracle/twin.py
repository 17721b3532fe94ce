"""Second, independent fp64 implementation of the oracle's definitions (numpy).

TEST INFRASTRUCTURE ONLY (see the package docstring).  It is written
separately from li_oracle.c -- vectorised numpy with library primitives
(einsum, lexsort) instead of loops -- so that the two cross-check each other
on small cases.  Same sources: "LatentIndex: Cross-Layer Sharing with
Layer-Specific Selection for Sparse Attention" (summary page), eqs. (6), (8),
TopK and the "Hierarchical Selection" paragraph.
"""
from __future__ import annotations

import numpy as np


def e4m3_values() -> np.ndarray:
    """All 256 E4M3 ("fn") code values, built by bit fields of the OCP FP8 format."""
    codes = np.arange(256, dtype=np.int64)
    sign = np.where(codes & 0x80, -1.0, 1.0)
    e = (codes >> 3) & 0xF
    m = (codes & 7).astype(np.float64)
    normal = np.ldexp(1.0 + m / 8.0, (e - 7).astype(np.int64))
    sub = np.ldexp(m / 8.0, -6)
    v = sign * np.where(e == 0, sub, normal)
    v[(e == 15) & ((codes & 7) == 7)] = np.nan
    return v


def decode(stored: np.ndarray, scale=None) -> np.ndarray:
    """fp64 values of an array stored as float32 / bf16 bits (uint16) / e4m3 codes (uint8)."""
    a = np.asarray(stored)
    if a.dtype == np.uint8:
        v = e4m3_values()[a]
    elif a.dtype == np.uint16:
        v = (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    else:
        v = a.astype(np.float64)
    if scale is not None:
        v = v * np.asarray(scale, dtype=np.float64)[..., None]
    return v


def absorb(q: np.ndarray, D: np.ndarray) -> np.ndarray:
    """q [..., G, H, d] and D [G, r, d] in fp64 -> q~ [..., G, H, r] (eq. 6)."""
    return np.einsum("grd,...ghd->...ghr", D, q)


def score(c: np.ndarray, qabs: np.ndarray, w: np.ndarray, beta=None, q_pos=None) -> np.ndarray:
    """c [B][L][r], qabs [B][T][G][H][r], w [B][T][G][H] (fp64) -> u [B][T][G][L] (eq. 8)."""
    dots = np.einsum("btghr,blr->btghl", qabs, c)
    if beta is not None:
        dots = dots + np.asarray(beta)[..., None]
    u = np.einsum("btgh,btghl->btgl", w, np.maximum(dots, 0.0))
    if q_pos is not None:
        L = c.shape[1]
        invalid = np.arange(L)[None, :] > np.asarray(q_pos)[:, None]      # [T][L]
        u = np.where(invalid[None, :, None, :], -np.inf, u)
    return u


def topk(scores: np.ndarray, k: int, valid_len=None) -> np.ndarray:
    """Indices of the min(k, V) largest scores per row (ties: lower index first), -1 padded."""
    s = np.asarray(scores, dtype=np.float64)
    L = s.shape[-1]
    flat = s.reshape(-1, L)
    vl = np.full(flat.shape[0], L) if valid_len is None else np.asarray(valid_len).reshape(-1)
    out = np.full((flat.shape[0], k), -1, dtype=np.int32)
    for i, row in enumerate(flat):
        V = int(min(vl[i], L))
        order = np.lexsort((np.arange(V), -row[:V]))
        n = min(k, V)
        out[i, :n] = order[:n]
    return out.reshape(s.shape[:-1] + (k,))


def hs(scores: np.ndarray, m: int, k: int):
    """HS from per-layer rows [B][G][L]: anchor top-m candidates, followers top-k inside them."""
    B, G, L = scores.shape
    cand = np.full((B, m), -1, dtype=np.int32)
    idx = np.full((B, G, k), -1, dtype=np.int32)
    for b in range(B):
        order = np.lexsort((np.arange(L), -scores[b, 0]))
        nc = min(m, L)
        C = order[:nc]
        cand[b, :nc] = C
        idx[b, 0, :min(k, nc)] = C[:min(k, nc)]
        for l in range(1, G):
            sub = np.lexsort((C, -scores[b, l, C]))
            idx[b, l, :min(k, nc)] = C[sub[:min(k, nc)]]
    return cand, idx


def append_latent(x: np.ndarray, P: np.ndarray, rR: int, pos, base: float = 10000.0) -> np.ndarray:
    """Eqs. (1)-(2) of the summary page with complex arithmetic: the RoPE
    branch of P x as rR/2 complex numbers, each multiplied by
    exp(1j * t * base^(-2i/rR)).  x [B][dm], P [r][dm] (fp64 values) -> [B][r]."""
    c = np.einsum("rd,bd->br", np.asarray(P, dtype=np.float64), np.asarray(x, dtype=np.float64))
    t = np.asarray(pos, dtype=np.float64).reshape(-1, 1)
    theta = base ** (-np.arange(0, rR, 2, dtype=np.float64) / rR)
    z = (c[:, 0:rR:2] + 1j * c[:, 1:rR:2]) * np.exp(1j * t * theta)
    out = c.copy()
    out[:, 0:rR:2] = z.real
    out[:, 1:rR:2] = z.imag
    return out
