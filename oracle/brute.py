"""Brute-force numpy statement of bifocal attention, for tiny inputs.

TEST INFRASTRUCTURE ONLY (used to pin the C oracle).  It shares nothing with
``oracle.c``: it starts from RAW (un-rotated) vectors, builds an explicit 2x2
rotation matrix for every pair, rotates the raw query/key of each position by
the position that view assigns -- the exact position p for the local
RoPE-faithful window, the aliased grid position floor(p/g) for the remote
window (researchpod.app summary and transcript: position aliasing onto the
known grid; abstract: local window keeps the original RoPE) -- and takes one
softmax over a materialised score matrix.  The C oracle instead corrects
already-rotated inputs; agreement pins the sign and size of the correction.
"""
from __future__ import annotations

import math

import numpy as np


def smallest_group(s: int, L: int) -> int:
    """Smallest integer g >= 1 such that every grouped position floor(p/g),
    p in [0, s), stays below L.  Checked position by position."""
    g = 1
    while max(p // g for p in range(s)) > L - 1:
        g += 1
    return g


def rot_matrix(angle: float) -> np.ndarray:
    c, s = math.cos(angle), math.sin(angle)
    return np.array([[c, -s], [s, c]])


def rope_raw(x: np.ndarray, pos: int, theta: float) -> np.ndarray:
    """Rotate one raw head vector to position ``pos`` with explicit matrices
    on the pairs (x_d, x_{d+D/2})."""
    D = x.shape[0]
    h = D // 2
    y = np.empty(D)
    for d in range(h):
        th = theta ** (-2.0 * d / D)
        pair = rot_matrix(pos * th) @ np.array([x[d], x[d + h]])
        y[d], y[d + h] = pair
    return y


def bifocal_from_raw(qr, kr, vr, L: int, w: int, theta: float):
    """qr [S,Hq,D], kr/vr [S,Hkv,D] raw vectors (batch of one).
    Returns (out [S,Hq,D], lse [Hq,S], exact-RoPE q [S,Hq,D], k [S,Hkv,D])."""
    S, Hq, D = qr.shape
    Hkv = kr.shape[1]
    grp = Hq // Hkv
    g = smallest_group(S, L)
    tau = 1.0 / math.sqrt(D)
    qx = np.array([[rope_raw(qr[i, h], i, theta) for h in range(Hq)] for i in range(S)])
    kx = np.array([[rope_raw(kr[j, h], j, theta) for h in range(Hkv)] for j in range(S)])
    qa = np.array([[rope_raw(qr[i, h], i // g, theta) for h in range(Hq)] for i in range(S)])
    ka = np.array([[rope_raw(kr[j, h], j // g, theta) for h in range(Hkv)] for j in range(S)])
    out = np.zeros((S, Hq, D))
    lse = np.zeros((Hq, S))
    for h in range(Hq):
        hk = h // grp
        sc = np.full((S, S), -np.inf)
        for i in range(S):
            for j in range(i + 1):
                if i - j < w:
                    sc[i, j] = tau * qx[i, h] @ kx[j, hk]
                else:
                    sc[i, j] = tau * qa[i, h] @ ka[j, hk]
        m = sc.max(axis=1, keepdims=True)
        p = np.exp(sc - m)
        Z = p.sum(axis=1)
        out[:, h, :] = (p @ vr[:, hk, :]) / Z[:, None]
        lse[h] = m[:, 0] + np.log(Z)
    return out, lse, qx, kx


# ---------------------------------------------------------------- variants
PER_QUERY_G, SLIDING, QUERY_SHIFT = 1, 2, 4


def smallest_group_shift(s: int, L: int, w: int):
    """Smallest g >= 1 such that, with the query's aliased position shifted by
    w - floor(w/g), every aliased distance floor(i/g) + shift - floor(j/g),
    0 <= j <= i < s, stays below L; None if no g up to max(s, w) + 1 does.
    Checked pair by pair."""
    for g in range(1, max(s, w) + 2):
        shift = w - w // g
        if max(i // g + shift - j // g for i in range(s) for j in range(i + 1)) <= L - 1:
            return g
    return None


def bifocal_variant_from_raw(qr, kr, vr, L: int, w: int, theta: float, flags: int):
    """Variants of bifocal_from_raw, from raw vectors and explicit rotations:
    PER_QUERY_G -- row i takes g from its own length i + 1; SLIDING -- keys with
    i - j >= w are not attended; QUERY_SHIFT -- the aliased query position is
    floor(i/g) + w - floor(w/g) and g follows the shifted rule.
    Returns (out [S,Hq,D], lse [Hq,S], exact-RoPE q, k), or None when the
    shifted rule has no g for some row."""
    S, Hq, D = qr.shape
    Hkv = kr.shape[1]
    grp = Hq // Hkv
    tau = 1.0 / math.sqrt(D)
    qx = np.array([[rope_raw(qr[i, h], i, theta) for h in range(Hq)] for i in range(S)])
    kx = np.array([[rope_raw(kr[j, h], j, theta) for h in range(Hkv)] for j in range(S)])
    out = np.zeros((S, Hq, D))
    lse = np.zeros((Hq, S))
    for i in range(S):
        s_row = i + 1 if flags & PER_QUERY_G else S
        if flags & QUERY_SHIFT:
            g = smallest_group_shift(s_row, L, w)
            if g is None:
                return None
            shift = w - w // g
        else:
            g, shift = smallest_group(s_row, L), 0
        for h in range(Hq):
            hk = h // grp
            qa = rope_raw(qr[i, h], i // g + shift, theta)
            sc, vals = [], []
            for j in range(i + 1):
                if i - j < w:
                    sc.append(tau * qx[i, h] @ kx[j, hk])
                elif flags & SLIDING:
                    continue
                else:
                    sc.append(tau * qa @ rope_raw(kr[j, hk], j // g, theta))
                vals.append(vr[j, hk])
            sc = np.array(sc)
            m = sc.max()
            p = np.exp(sc - m)
            out[i, h] = (p @ np.array(vals)) / p.sum()
            lse[h, i] = m + math.log(p.sum())
    return out, lse, qx, kx
