"""Schedule / length robustness sweep: B=4, Hq=32, Hkv=8, D=128, theta=1e6,
S in {4096, 16384, 32768, 65536, 131072} x L in {4096, 32768} x
w in {1024, 2048, 4096, 8192}: 40 prefill cases run in full on the GPU.

Every case is checked against the fp64 oracle, element by element, on rows
of every batch entry: the rows at the edges of every rule (window, group,
pretrained window, tiles) and, for each batch entry, one seeded row of every
eighth 128-row query tile -- the eight (L, w) cases of one S take the eight
residues, so together they check one row of every query tile of every batch
entry.  Every case with S <= L (g = 1) must equal, bit for bit, the same kernel
with bifocal off -- the base model recovered exactly at short inputs (Jet-Long
abstract).  Inputs are drawn once per S (seed 4 + index of S) and shared by
that S's eight (L, w) cases.
"""
import numpy as np
import pytest

import helpers

pytestmark = pytest.mark.gpu

SWEEP_S = (4096, 16384, 32768, 65536, 131072)
SWEEP_L = (4096, 32768)
SWEEP_W = (1024, 2048, 4096, 8192)
B, HQ, HKV, D, THETA = 4, 32, 8, 128, 1e6

_data = {}


def _inputs(S, dev):
    """(q, k, v) on the device and their bf16 bit patterns on the host."""
    if S not in _data:
        from zero_shot_rope_02_b300 import inputs

        _data.clear()  # keep one S resident at a time
        seed = 4 + SWEEP_S.index(S)
        qb = inputs.normal_bf16_bits((B, S, HQ, D), seed, 0)
        kb = inputs.normal_bf16_bits((B, S, HKV, D), seed, 1)
        vb = inputs.normal_bf16_bits((B, S, HKV, D), seed, 2)
        tq, tk, tv = (inputs.to_torch_bf16(x).to(dev) for x in (qb, kb, vb))
        _data[S] = (tq, tk, tv, qb, kb, vb)
    return _data[S]


@pytest.mark.parametrize("w", SWEEP_W)
@pytest.mark.parametrize("L", SWEEP_L)
@pytest.mark.parametrize("S", SWEEP_S)
def test_sweep_case(jl, orc, dev, S, L, w):
    import torch

    from zero_shot_rope_02_b300 import inputs

    tq, tk, tv, qb, kb, vb = _inputs(S, dev)
    out, lse = jl.jl_bifocal_prefill(tq, tk, tv, L, w, THETA)
    assert jl.jl_debug_status() == 0
    g = orc.group_factor(S, L)
    if S <= L:
        assert g == 1
        out_p, lse_p = jl.jl_bifocal_prefill(tq, tk, tv, S, w, THETA)  # bifocal off
        assert torch.equal(out, out_p) and torch.equal(lse, lse_p), "s <= L must be plain RoPE"
    edges = helpers.sample_rows(S, L, w, g, n_random=0)
    case = SWEEP_L.index(L) * len(SWEEP_W) + SWEEP_W.index(w)  # 0..7 within this S
    n_tiles = -(-S // 128)
    rng = np.random.default_rng(S + L + w)
    for b in range(B):
        tiles = np.arange(case, n_tiles, len(SWEEP_L) * len(SWEEP_W))
        picks = tiles * 128 + rng.integers(0, 128, size=len(tiles))
        rows = np.unique(np.concatenate([edges, picks[picks < S]]))
        kf = inputs.bf16_bits_to_f64(kb[b:b + 1])
        vf = inputs.bf16_bits_to_f64(vb[b:b + 1])
        qf = inputs.bf16_bits_to_f64(qb[b:b + 1, rows])
        ref_o, ref_l = orc.bifocal_rows(qf, kf, vf, rows, S, L, w, THETA)
        got_o = helpers.bf16_to_f64(out[b:b + 1, rows])
        got_l = lse[b:b + 1, :, rows].cpu().numpy().astype(np.float64)
        helpers.compare(got_o, got_l, ref_o, ref_l, f"sweep S={S} L={L} w={w} b={b}")
