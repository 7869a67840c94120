"""Checks that pin the fp64 oracle to facts fixed outside it.

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError on a
mismatch.  They are run against the real oracle (test_oracle_pins.py) and
against deliberately broken copies of it (test_oracle_mutants.py), which
shows that a plausible slip anywhere in the oracle fails at least one pin.

What each pin rests on:
  group rule     brute search over positions + the tiny benchmark's printed
                 g=4 (tests/golden/group_factor.txt)
  rope           complex-number statement z_d * exp(i p theta_d) of RoPE
  brute force    oracle/brute.py: raw vectors rotated to exact or aliased
                 positions with explicit 2x2 matrices (no correction step)
  three-pass     inclusion-exclusion merge == single masked pass
  plain limits   s <= L and w >= s reduce to ordinary causal attention
                 (torch scaled_dot_product_attention, fp64)
  all-remote     w = 1 reduces to causal attention at aliased positions
  closed forms   hand-evaluated tiny cases (constant raw vectors)
"""
from __future__ import annotations

import math
import os

import numpy as np

from oracle import brute

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- helpers
def rope_complex(x: np.ndarray, pos: np.ndarray, theta: float) -> np.ndarray:
    """RoPE as complex multiplication: z_d = x_d + i x_{d+D/2} -> z_d e^{i p theta_d}.
    x [S,H,D], pos [S]."""
    D = x.shape[-1]
    h = D // 2
    th = theta ** (-2.0 * np.arange(h) / D)
    z = x[..., :h] + 1j * x[..., h:]
    z = z * np.exp(1j * pos[:, None, None] * th[None, None, :])
    return np.concatenate([z.real, z.imag], axis=-1)


def causal_sdpa(q, k, v):
    """Ordinary causal softmax attention via torch (fp64 CPU).
    q [S,Hq,D], k/v [S,Hkv,D] -> out [S,Hq,D], lse [Hq,S]."""
    import torch

    Hq, Hkv = q.shape[1], k.shape[1]
    grp = Hq // Hkv
    tq = torch.from_numpy(np.ascontiguousarray(q)).permute(1, 0, 2)
    tk = torch.from_numpy(np.ascontiguousarray(k)).permute(1, 0, 2).repeat_interleave(grp, 0)
    tv = torch.from_numpy(np.ascontiguousarray(v)).permute(1, 0, 2).repeat_interleave(grp, 0)
    out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=True)
    S = q.shape[0]
    scores = (tq @ tk.transpose(1, 2)) / math.sqrt(q.shape[2])
    mask = torch.ones(S, S, dtype=torch.bool).tril()
    lse = torch.logsumexp(scores.masked_fill(~mask, float("-inf")), dim=-1)
    return out.permute(1, 0, 2).numpy(), lse.numpy()


def _close(a, b, tol, what):
    err = float(np.max(np.abs(np.asarray(a) - np.asarray(b)))) if np.size(a) else 0.0
    assert err <= tol, f"{what}: max abs err {err:.3e} > {tol:.1e}"


# ---------------------------------------------------------------- pins
def pin_group_rule(orc):
    for s in range(1, 130):
        for L in range(1, 40):
            g = orc.group_factor(s, L)
            assert g == brute.smallest_group(s, L), (s, L, g)
            assert g == max(1, -(-s // L)), (s, L, g)
    with open(os.path.join(GOLDEN, "group_factor.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            s, L, g = map(int, line.split())
            assert orc.group_factor(s, L) == g, (s, L, g)
    for p in range(0, 50):
        for g in range(1, 7):
            assert orc.grouped_position(p, g) == p // g


def pin_rope(orc):
    r = _rng(11)
    for D, theta in ((2, 10000.0), (8, 10000.0), (16, 1.0e6), (64, 500.0)):
        x = r.standard_normal((2, 9, 3, D))
        for pos0 in (0, 5, 70001):
            got = orc.rope(x, pos0, theta)
            pos = pos0 + np.arange(9)
            want = np.stack([rope_complex(x[b], pos, theta) for b in range(2)])
            _close(got, want, 1e-9, f"rope D={D} pos0={pos0}")
        _close(orc.rope(x, 0, theta)[:, :1], x[:, :1], 0.0, "rope at position 0")


def pin_brute(orc, sizes=range(1, 11), D=4, theta=10.0, seed=3):
    """Every (L, w) on tiny sequences against oracle/brute.py (raw vectors)."""
    r = _rng(seed)
    for S in sizes:
        qr = r.standard_normal((S, 4, D))
        kr = r.standard_normal((S, 2, D))
        vr = r.standard_normal((S, 2, D))
        for L in range(1, S + 2):
            for w in range(1, S + 2):
                out_b, lse_b, qx, kx = brute.bifocal_from_raw(qr, kr, vr, L, w, theta)
                out, lse = orc.bifocal_prefill(qx[None], kx[None], vr[None], L, w, theta)
                _close(out[0], out_b, 1e-12, f"brute out S={S} L={L} w={w}")
                _close(lse[0], lse_b, 1e-12, f"brute lse S={S} L={L} w={w}")


def pin_three_pass(orc):
    r = _rng(5)
    S, D = 150, 16
    q = r.standard_normal((2, S, 4, D))
    k = r.standard_normal((2, S, 2, D))
    v = r.standard_normal((2, S, 2, D))
    for L, w in ((37, 1), (37, 5), (37, 64), (20, 149), (20, 200), (150, 10), (7, 33)):
        o1, l1 = orc.bifocal_prefill(q, k, v, L, w, 1.0e4)
        o3, l3 = orc.bifocal_rows_3pass(q, k, v, np.arange(S), S, L, w, 1.0e4)
        _close(o1, o3, 1e-12, f"3-pass out L={L} w={w}")
        _close(l1, l3, 1e-11, f"3-pass lse L={L} w={w}")


def pin_plain_limits(orc):
    """Base model recovered exactly: s <= L (g = 1) or w >= s gives causal RoPE attention."""
    r = _rng(7)
    S, D = 96, 32
    qr = r.standard_normal((S, 4, D))
    kr = r.standard_normal((S, 2, D))
    v = r.standard_normal((S, 2, D))
    pos = np.arange(S)
    q = rope_complex(qr, pos, 1.0e4)
    k = rope_complex(kr, pos, 1.0e4)
    out_ref, lse_ref = causal_sdpa(q, k, v)
    for L, w in ((S, 3), (S + 50, 1), (4, S), (4, S + 7), (1, 10 ** 6)):
        out, lse = orc.bifocal_prefill(q[None], k[None], v[None], L, w, 1.0e4)
        _close(out[0], out_ref, 1e-12, f"plain out L={L} w={w}")
        _close(lse[0], lse_ref, 1e-12, f"plain lse L={L} w={w}")


def pin_all_remote(orc):
    """w = 1: only the diagonal is local, and there exact and aliased scores
    coincide, so the result is causal attention at positions floor(p/g)."""
    r = _rng(9)
    S, D = 80, 16
    qr = r.standard_normal((S, 2, D))
    kr = r.standard_normal((S, 1, D))
    v = r.standard_normal((S, 1, D))
    pos = np.arange(S)
    q = rope_complex(qr, pos, 1.0e4)
    k = rope_complex(kr, pos, 1.0e4)
    for L in (3, 9, 40):
        g = -(-S // L)
        out_ref, lse_ref = causal_sdpa(rope_complex(qr, pos // g, 1.0e4),
                                       rope_complex(kr, pos // g, 1.0e4), v)
        out, lse = orc.bifocal_prefill(q[None], k[None], v[None], L, 1, 1.0e4)
        _close(out[0], out_ref, 1e-12, f"all-remote out L={L}")
        _close(lse[0], lse_ref, 1e-12, f"all-remote lse L={L}")


def pin_closed_forms(orc):
    """Constant raw vectors q~ = k~ = (1, 0), D = 2 (theta_0 = 1 for any theta).
    Exact scores are tau*cos(i-j); aliased scores are tau*cos(floor(i/g)-floor(j/g))."""
    tau = 1.0 / math.sqrt(2.0)
    S = 6
    pos = np.arange(S, dtype=np.float64)
    q = np.stack([np.cos(pos), np.sin(pos)], axis=-1)[None, :, None, :]
    k = q.copy()
    v = np.stack([pos, -2.0 * pos], axis=-1)[None, :, None, :]
    # (1) S=6, L=2 -> g=3, w=1: aliased positions 0,0,0,1,1,1; everything is remote
    #     except the diagonal (score tau).  Row i: scores tau*cos(G(i)-G(j)).
    out, lse = orc.bifocal_prefill(q, k, v, 2, 1, 1.0e4)
    for i in range(S):
        sc = [tau * math.cos(i // 3 - j // 3) for j in range(i + 1)]
        Z = sum(math.exp(s) for s in sc)
        o0 = sum(math.exp(s) * j for j, s in enumerate(sc)) / Z
        assert abs(out[0, i, 0, 0] - o0) < 1e-13 and abs(out[0, i, 0, 1] + 2 * o0) < 1e-13, i
        assert abs(lse[0, 0, i] - math.log(Z)) < 1e-13, i
    # rows 0..2 see only aliased position 0: uniform weights, out = i/2, lse = tau + ln(i+1)
    for i in range(3):
        assert abs(out[0, i, 0, 0] - i / 2.0) < 1e-13
        assert abs(lse[0, 0, i] - (tau + math.log(i + 1))) < 1e-13
    # (2) same inputs, L=6 -> g=1: plain RoPE, scores tau*cos(i-j)
    out, lse = orc.bifocal_prefill(q, k, v, 6, 1, 1.0e4)
    for i in range(S):
        sc = [tau * math.cos(i - j) for j in range(i + 1)]
        Z = sum(math.exp(s) for s in sc)
        assert abs(lse[0, 0, i] - math.log(Z)) < 1e-13, i
    # (3) S=6, L=3 -> g=2, w=2: keys i and i-1 exact, older keys aliased (G = 0,0,1,1,2,2).
    out, lse = orc.bifocal_prefill(q, k, v, 3, 2, 1.0e4)
    i = 5
    sc = [tau * math.cos(2 - 0), tau * math.cos(2 - 0), tau * math.cos(2 - 1),
          tau * math.cos(2 - 1), tau * math.cos(1.0), tau]
    Z = sum(math.exp(s) for s in sc)
    assert abs(lse[0, 0, i] - math.log(Z)) < 1e-13
    o0 = sum(math.exp(s) * j for j, s in enumerate(sc)) / Z
    assert abs(out[0, i, 0, 0] - o0) < 1e-13


def pin_decode_row(orc):
    """Decode of one token at position n-1 over an n-key cache equals row n-1
    of the length-n prefill (the cache keeps exact positions)."""
    r = _rng(13)
    n, D = 70, 8
    q = r.standard_normal((1, n, 4, D))
    k = r.standard_normal((1, n, 2, D))
    v = r.standard_normal((1, n, 2, D))
    for L, w in ((9, 4), (70, 4), (5, 100)):
        o_p, l_p = orc.bifocal_prefill(q, k, v, L, w, 1.0e4)
        o_d, l_d = orc.bifocal_decode(q[:, n - 1:], k, v, L, w, 1.0e4)
        _close(o_d[0, 0], o_p[0, n - 1], 0.0, "decode out")
        _close(l_d[0, :, 0], l_p[0, :, n - 1], 0.0, "decode lse")


ALL_PINS = [pin_group_rule, pin_rope, pin_brute, pin_three_pass, pin_plain_limits,
            pin_all_remote, pin_closed_forms, pin_decode_row]
