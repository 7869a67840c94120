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
  variants       per-query g, sliding window and query shift: brute force from
                 raw vectors, per-query rows == decodes at their own length,
                 sliding == band-masked SDPA, the shifted g rule's hand-checked
                 golden rows (tests/golden/group_factor_shift.txt), a closed form
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


# ---------------------------------------------------------------- variants
PQ, SW, SH = 1, 2, 4  # per-query g, sliding window, query shift


def pin_variant_group_rule(orc):
    """Shifted g rule: the hand-checked golden rows, and a pair-by-pair search."""
    with open(os.path.join(GOLDEN, "group_factor_shift.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            s, L, w, g = map(int, line.split())
            assert orc.group_factor_shift(s, L, w) == g, (s, L, w, g)
    for s in range(1, 40):
        for L in range(1, 14):
            for w in range(1, 16):
                want = brute.smallest_group_shift(s, L, w)
                assert orc.group_factor_shift(s, L, w) == (-1 if want is None else want), (s, L, w)


def pin_variant_brute(orc, sizes=range(1, 9), D=4, theta=10.0, seed=23):
    """Every (L, w) and flag combination on tiny sequences against the raw-vector
    statement in oracle/brute.py (explicit rotations to aliased positions)."""
    r = _rng(seed)
    for S in sizes:
        qr = r.standard_normal((S, 2, D))
        kr = r.standard_normal((S, 1, D))
        vr = r.standard_normal((S, 1, D))
        for flags in (PQ, SW, SH, PQ | SH):
            for L in range(1, S + 2):
                for w in range(1, S + 2):
                    ref = brute.bifocal_variant_from_raw(qr, kr, vr, L, w, theta, flags)
                    if ref is None:  # no g for the shifted rule: the oracle refuses too
                        try:
                            orc.bifocal_prefill_ex(ref_q(qr, theta), ref_q(kr, theta), vr[None], L, w,
                                                   theta, flags)
                        except ValueError:
                            continue
                        raise AssertionError(f"variant {flags}: accepted S={S} L={L} w={w}")
                    out_b, lse_b, qx, kx = ref
                    out, lse = orc.bifocal_prefill_ex(qx[None], kx[None], vr[None], L, w, theta, flags)
                    _close(out[0], out_b, 1e-12, f"variant {flags} out S={S} L={L} w={w}")
                    _close(lse[0], lse_b, 1e-12, f"variant {flags} lse S={S} L={L} w={w}")


def ref_q(xr, theta):
    """Exact-RoPE copy of raw vectors [S,H,D] at positions 0..S-1, batch of one."""
    return rope_complex(xr, np.arange(xr.shape[0]), theta)[None]


def pin_variant_flags_off(orc):
    """No flag: the variant entry point is the single masked pass, bit for bit."""
    r = _rng(29)
    S, D = 90, 8
    q, k, v = (r.standard_normal((2, S, h, D)) for h in (4, 2, 2))
    for L, w in ((7, 3), (90, 5), (11, 40)):
        o0, l0 = orc.bifocal_prefill(q, k, v, L, w, 1.0e4)
        o1, l1 = orc.bifocal_prefill_ex(q, k, v, L, w, 1.0e4, 0)
        _close(o1, o0, 0.0, "flags 0 out")
        _close(l1, l0, 0.0, "flags 0 lse")


def pin_per_query_rows_are_decodes(orc):
    """Per-query g: row i is the decode of the token at i over keys 0..i, whose
    current length is i + 1 -- and the last row is the ordinary prefill's."""
    r = _rng(31)
    S, D = 60, 8
    q, k, v = (r.standard_normal((1, S, h, D)) for h in (4, 2, 2))
    for L, w in ((7, 3), (13, 1), (60, 4)):
        o, l = orc.bifocal_prefill_ex(q, k, v, L, w, 1.0e4, PQ)
        for i in range(S):
            od, ld = orc.bifocal_decode(q[:, i:i + 1], k[:, :i + 1], v[:, :i + 1], L, w, 1.0e4)
            _close(o[0, i], od[0, 0], 1e-13, f"per-query row {i} out L={L} w={w}")
            _close(l[0, :, i], ld[0, :, 0], 1e-13, f"per-query row {i} lse L={L} w={w}")
        o_p, l_p = orc.bifocal_prefill(q, k, v, L, w, 1.0e4)
        _close(o[0, S - 1], o_p[0, S - 1], 1e-13, "per-query last row")


def pin_sliding_is_banded_attention(orc):
    """Sliding window: causal attention restricted to 0 <= i - j < w (torch
    SDPA with an explicit band mask, fp64); w >= S is plain causal attention."""
    import torch

    r = _rng(37)
    S, D = 70, 16
    q, k, v = (r.standard_normal((S, h, D)) for h in (4, 2, 2))
    i = torch.arange(S)[:, None]
    j = torch.arange(S)[None, :]
    tq = torch.from_numpy(q).permute(1, 0, 2)
    tk = torch.from_numpy(k).permute(1, 0, 2).repeat_interleave(2, 0)
    tv = torch.from_numpy(v).permute(1, 0, 2).repeat_interleave(2, 0)
    for L, w in ((5, 1), (5, 9), (80, 9), (5, 70)):
        band = (j <= i) & (i - j < w)
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=band)
        sc = (tq @ tk.transpose(1, 2)) / math.sqrt(D)
        ref_l = torch.logsumexp(sc.masked_fill(~band, float("-inf")), dim=-1)
        out, lse = orc.bifocal_prefill_ex(q[None], k[None], v[None], L, w, 1.0e4, SW)
        _close(out[0], ref.permute(1, 0, 2).numpy(), 1e-12, f"sliding out w={w}")
        _close(lse[0], ref_l.numpy(), 1e-12, f"sliding lse w={w}")


def pin_shift_closed_form(orc):
    """Query shift with constant raw vectors q~ = k~ = (1, 0), D = 2: an aliased
    score is tau*cos(floor(i/g) + w - floor(w/g) - floor(j/g)).  S = 8, L = 6,
    w = 2: g = 2 (g = 1: 7 + 0 > 5; g = 2: 3 + 1 = 4 <= 5), shift 1."""
    tau = 1.0 / math.sqrt(2.0)
    S, L, w = 8, 6, 2
    pos = np.arange(S, dtype=np.float64)
    q = np.stack([np.cos(pos), np.sin(pos)], axis=-1)[None, :, None, :]
    v = np.stack([pos, pos * pos], axis=-1)[None, :, None, :]
    out, lse = orc.bifocal_prefill_ex(q, q.copy(), v, L, w, 1.0e4, SH)
    for i in range(S):
        sc = [tau * math.cos(i - j) if i - j < w else tau * math.cos(i // 2 + 1 - j // 2)
              for j in range(i + 1)]
        Z = sum(math.exp(x) for x in sc)
        assert abs(lse[0, 0, i] - math.log(Z)) < 1e-13, i
        o0 = sum(math.exp(x) * j for j, x in enumerate(sc)) / Z
        assert abs(out[0, i, 0, 0] - o0) < 1e-13, i
    # at distance exactly w from an even row the aliased distance is w too:
    # the shifted view is continuous with the exact one at the window edge
    assert all((i // 2 + 1 - (i - w) // 2) == w for i in range(w, S, 2))


ALL_PINS = [pin_group_rule, pin_rope, pin_brute, pin_three_pass, pin_plain_limits,
            pin_all_remote, pin_closed_forms, pin_decode_row, pin_variant_group_rule,
            pin_variant_brute, pin_variant_flags_off, pin_per_query_rows_are_decodes,
            pin_sliding_is_banded_attention, pin_shift_closed_form]
