"""Prefill of a chunk over an existing cache (jl_bifocal_prefill_chunk), the
capacity guard of every cache-reading call, and the RoPE-fused cache write
that fills the cache (jl_rope_cache_write), against the fp64 oracle.

A chunk is S_new queries at positions n_past..n_past+S_new-1 over the keys at
0..n_past+S_new-1, with s = n_past + S_new setting g: the rows a full prefill
of length s gives those positions (ResearchPod transcript on the prefill
phase, run in pieces).  The oracle scores exactly that (its row entry takes
the query positions and s).  Cache rows past the valid keys are filled with
NaN: the kernels must never read them (a 0 * NaN in P.V would show).
"""
import numpy as np
import pytest

import helpers

pytestmark = pytest.mark.gpu


def _caches(B, n_cap, Hkv, D, n_valid, seed):
    """Seeded caches [B, n_cap, Hkv, D]; rows >= n_valid hold NaN."""
    import torch

    k_t, k_f = helpers.bf16_pair((B, n_cap, Hkv, D), seed, 1)
    v_t, v_f = helpers.bf16_pair((B, n_cap, Hkv, D), seed, 2)
    k_t[:, n_valid:] = float("nan")
    v_t[:, n_valid:] = float("nan")
    return k_t, v_t, k_f[:, :n_valid], v_f[:, :n_valid]


@pytest.mark.parametrize("B,Hq,Hkv,S_new,n_past,n_cap,D,L,w", [
    (1, 4, 2, 300, 500, 900, 128, 200, 150),   # chunk not on a tile boundary, g = 4
    (2, 2, 1, 256, 256, 600, 64, 100, 64),     # on a tile boundary, g = 6
    (1, 2, 1, 1, 777, 800, 128, 300, 128),     # one new token (the decode position)
    (1, 4, 4, 200, 0, 300, 128, 128, 64),      # empty cache: a full prefill of 200
    (1, 8, 2, 129, 1000, 1129, 128, 2000, 64), # s <= L: plain RoPE
    (1, 2, 2, 640, 70, 710, 64, 100, 1),       # w = 1: all but the diagonal remote
])
def test_chunk_parity(jl, orc, dev, B, Hq, Hkv, S_new, n_past, n_cap, D, L, w):
    theta = 1e6
    s = n_past + S_new
    q_t, q_f = helpers.bf16_pair((B, S_new, Hq, D), 9, 0)
    k_t, v_t, k_f, v_f = _caches(B, n_cap, Hkv, D, s, 9)
    out, lse = jl.jl_bifocal_prefill_chunk(q_t.to(dev), k_t.to(dev), v_t.to(dev), n_past, L, w, theta)
    assert jl.jl_debug_status() == 0
    ref_o, ref_l = orc.bifocal_rows(q_f, k_f, v_f, n_past + np.arange(S_new), s, L, w, theta)
    helpers.compare(helpers.bf16_to_f64(out), lse.cpu().numpy(), ref_o, ref_l,
                    f"chunk n_past={n_past} S_new={S_new} L={L} w={w}")


def test_chunks_on_tile_boundaries_equal_the_full_prefill_bitwise(jl, dev):
    """Chunks that start on a 128-row boundary visit the same key tiles in the
    same order as the full prefill's query tiles: identical bits."""
    import torch

    B, Hq, Hkv, S, D, L, w = 1, 4, 2, 1000, 128, 300, 256
    q_t, _ = helpers.bf16_pair((B, S, Hq, D), 10, 0)
    k_t, _ = helpers.bf16_pair((B, S, Hkv, D), 10, 1)
    v_t, _ = helpers.bf16_pair((B, S, Hkv, D), 10, 2)
    q, k, v = q_t.to(dev), k_t.to(dev), v_t.to(dev)
    out_f, lse_f = jl.jl_bifocal_prefill(q, k, v, L, w, 1e6)
    for a, b in ((0, 384), (384, 768), (768, 1000)):
        # the cache holds all S rows; a chunk ending at b sees keys < b only,
        # so compare against a full prefill of length b for its own g
        out_b, lse_b = jl.jl_bifocal_prefill(q[:, :b].contiguous(), k[:, :b].contiguous(),
                                             v[:, :b].contiguous(), L, w, 1e6)
        out_c, lse_c = jl.jl_bifocal_prefill_chunk(q[:, a:b].contiguous(), k, v, a, L, w, 1e6)
        assert torch.equal(out_c, out_b[:, a:b]) and torch.equal(lse_c, lse_b[:, :, a:b]), (a, b)
    assert jl.jl_debug_status() == 0
    # the last chunk ends at S: it equals the full prefill's rows too
    assert torch.equal(out_c, out_f[:, 768:]) and torch.equal(lse_c, lse_f[:, :, 768:])


def test_decode_never_reads_past_n(jl, orc, dev):
    """Cache capacity past n filled with NaN: decode stays finite and equal to
    the run whose spare capacity holds ordinary values."""
    import torch

    B, Hq, Hkv, n, n_cap, D, L, w = 1, 32, 8, 3000, 3100, 128, 1000, 256
    q_t, q_f = helpers.bf16_pair((B, Hq, D), 12, 3)
    k_t, v_t, k_f, v_f = _caches(B, n_cap, Hkv, D, n, 12)
    out, lse = jl.jl_bifocal_decode(q_t.to(dev), k_t.to(dev), v_t.to(dev), n, L, w, 1e6)
    assert jl.jl_debug_status() == 0
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    k2, v2 = k_t.clone(), v_t.clone()
    k2[:, n:] = 0.5
    v2[:, n:] = -2.0
    out2, lse2 = jl.jl_bifocal_decode(q_t.to(dev), k2.to(dev), v2.to(dev), n, L, w, 1e6)
    assert torch.equal(out, out2) and torch.equal(lse, lse2)
    ref_o, ref_l = orc.bifocal_decode(q_f[:, None], k_f, v_f, L, w, 1e6)
    helpers.compare(helpers.bf16_to_f64(out), lse.cpu().numpy(), ref_o[:, 0], ref_l[:, :, 0],
                    "decode with NaN past n")


def test_chunk_benchmark_shape_sampled(jl, orc, dev):
    """The 8K chunk that completes the 128K Qwen3-8B-shaped context (g = 4),
    sampled rows against the oracle."""
    from zero_shot_rope_02_b300 import inputs

    B, Hq, Hkv, D, L, w = 1, 32, 8, 128, 32768, 4096
    S_new, n_past = 8192, 131072 - 8192
    s = n_past + S_new
    qb = inputs.normal_bf16_bits((B, S_new, Hq, D), 13, 0)
    k_t, k_f = helpers.bf16_pair((B, s, Hkv, D), 13, 1)
    v_t, v_f = helpers.bf16_pair((B, s, Hkv, D), 13, 2)
    out, lse = jl.jl_bifocal_prefill_chunk(inputs.to_torch_bf16(qb).to(dev), k_t.to(dev), v_t.to(dev),
                                           n_past, L, w, 1e6)
    assert jl.jl_debug_status() == 0
    rows = np.array(sorted({0, 1, 127, 128, 4095, 4096, S_new - 129, S_new - 1} |
                           set(np.random.default_rng(13).integers(0, S_new, 8).tolist())))
    q_rows = inputs.bf16_bits_to_f64(qb[:, rows])
    ref_o, ref_l = orc.bifocal_rows(q_rows, k_f, v_f, n_past + rows, s, L, w, 1e6)
    helpers.compare(helpers.bf16_to_f64(out[:, rows]), lse[:, :, rows].cpu().numpy(), ref_o, ref_l,
                    "chunk 8K over 120K (sampled rows)")


@pytest.mark.parametrize("B,S_new,H,D,n_past,n_cap", [(2, 300, 8, 128, 777, 1200), (1, 65, 4, 64, 0, 65)])
def test_rope_cache_write(jl, orc, dev, B, S_new, H, D, n_past, n_cap):
    """RoPE fused into the cache write: the written keys are jl_rope_apply's
    bits, the values are copied, no other cache row is touched, and the keys
    match the oracle's RoPE within one bf16 rounding."""
    import torch

    theta = 1e6
    k_t, k_f = helpers.bf16_pair((B, S_new, H, D), 14, 1)
    v_t, _ = helpers.bf16_pair((B, S_new, H, D), 14, 2)
    k, v = k_t.to(dev), v_t.to(dev)
    kc = torch.full((B, n_cap, H, D), float("nan"), dtype=torch.bfloat16, device=dev)
    vc = torch.full_like(kc, float("nan"))
    jl.jl_rope_cache_write(k, v, kc, vc, n_past, theta)
    rows = slice(n_past, n_past + S_new)
    assert torch.equal(kc[:, rows], jl.jl_rope_apply(k.clone(), n_past, theta))
    assert torch.equal(vc[:, rows], v)
    for c in (kc, vc):
        assert torch.isnan(c[:, :n_past].float()).all() and torch.isnan(c[:, n_past + S_new:].float()).all()
    got = helpers.bf16_to_f64(kc[:, rows])
    ref = orc.rope(k_f, n_past, theta)
    # one rounding to bf16 of an fp32 result: within 2^-8 relative (+ fp32 slack)
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-5 * np.abs(k_f).max())
