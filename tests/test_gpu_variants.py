"""The method's optional forms (jl_bifocal_prefill_ex / jl_bifocal_decode_ex)
against the fp64 oracle's variant entry point, element by element:

  per-query g   query i takes g from its own length i + 1 (the factor follows
                the current length, abstract); prefill runs one launch per
                range of rows that share g
  sliding       a sliding-window layer of a hybrid model: keys with i - j >= w
                are not attended, nothing is aliased (seventnews.com,
                "Generalization to hybrid attention architectures")
  query shift   Self-Extend-style grouping: the aliased query position is
                floor(i/g) + w - floor(w/g), g from the shifted rule
                (ResearchPod summary: Self-Extend baseline)
"""
import numpy as np
import pytest

import helpers

pytestmark = pytest.mark.gpu

PQ, SW, SH = 1, 2, 4


def _prefill_variant(jl, orc, dev, B, Hq, Hkv, S_new, n_past, D, L, w, flags, seed, theta=1e6, rows=None):
    from zero_shot_rope_02_b300 import inputs

    s = n_past + S_new
    qb = inputs.normal_bf16_bits((B, S_new, Hq, D), seed, 0)
    k_t, k_f = helpers.bf16_pair((B, s, Hkv, D), seed, 1)
    v_t, v_f = helpers.bf16_pair((B, s, Hkv, D), seed, 2)
    out, lse = jl.jl_bifocal_prefill_ex(inputs.to_torch_bf16(qb).to(dev), k_t.to(dev), v_t.to(dev), n_past,
                                        L, w, theta, flags)
    assert jl.jl_debug_status() == 0
    if rows is None:
        rows = np.arange(S_new)
    q_f = inputs.bf16_bits_to_f64(qb[:, rows])
    ref_o, ref_l = orc.bifocal_rows_ex(q_f, k_f, v_f, n_past + rows, s, L, w, theta, flags)
    helpers.compare(helpers.bf16_to_f64(out[:, rows]), lse[:, :, rows].cpu().numpy(), ref_o, ref_l,
                    f"variant {flags} S_new={S_new} n_past={n_past} L={L} w={w}")
    return out, lse


@pytest.mark.parametrize("B,Hq,Hkv,S_new,n_past,D,L,w", [
    (1, 4, 2, 700, 0, 128, 200, 150),    # g = 1..4, L not a multiple of the 128-row tile
    (1, 2, 1, 1000, 0, 64, 256, 64),     # ranges on tile boundaries
    (2, 4, 4, 300, 0, 128, 37, 1),       # nine ranges, everything but the diagonal remote
    (1, 8, 2, 300, 500, 128, 200, 100),  # a chunk over a cache: ranges from position 500
    (1, 4, 2, 900, 0, 128, 1000, 64),    # every row below L: plain RoPE
])
def test_prefill_per_query_g(jl, orc, dev, B, Hq, Hkv, S_new, n_past, D, L, w):
    _prefill_variant(jl, orc, dev, B, Hq, Hkv, S_new, n_past, D, L, w, PQ, seed=41)


@pytest.mark.parametrize("B,Hq,Hkv,S_new,n_past,D,L,w", [
    (1, 4, 2, 700, 0, 128, 200, 150),
    (1, 2, 1, 1000, 0, 64, 50, 64),
    (2, 4, 2, 600, 0, 128, 100, 1),      # only the diagonal
    (1, 2, 2, 900, 0, 128, 100, 300),    # window across several tiles, ragged end
    (1, 4, 2, 300, 700, 128, 100, 200),  # a chunk over a cache
])
def test_prefill_sliding(jl, orc, dev, B, Hq, Hkv, S_new, n_past, D, L, w):
    _prefill_variant(jl, orc, dev, B, Hq, Hkv, S_new, n_past, D, L, w, SW, seed=43)


@pytest.mark.parametrize("B,Hq,Hkv,S_new,n_past,D,L,w,theta", [
    (1, 4, 2, 700, 0, 128, 200, 150, 1e6),
    (1, 1, 1, 2048, 0, 64, 512, 128, 1e4),  # the tiny configuration's shape: g = 6 shifted
    (1, 2, 1, 1000, 0, 64, 300, 64, 1e6),
    (1, 2, 2, 640, 0, 64, 100, 1, 1e6),     # w = 1: the shift is 1 - floor(1/g) = 1
    (1, 8, 2, 300, 500, 128, 200, 100, 1e6),
])
def test_prefill_query_shift(jl, orc, dev, B, Hq, Hkv, S_new, n_past, D, L, w, theta):
    g = jl.jl_group_factor_ex(n_past + S_new, L, w, SH)
    assert g == orc.group_factor_shift(n_past + S_new, L, w)
    _prefill_variant(jl, orc, dev, B, Hq, Hkv, S_new, n_past, D, L, w, SH, seed=47, theta=theta)


def test_variants_reduce_to_the_plain_kernel_bitwise(jl, dev):
    """Sliding with w >= S, a shift with S <= L and per-query g with S <= L
    all visit exactly the tiles of the bifocal-off run: identical bits."""
    import torch

    q_t, _ = helpers.bf16_pair((1, 900, 4, 128), 49, 0)
    k_t, _ = helpers.bf16_pair((1, 900, 2, 128), 49, 1)
    v_t, _ = helpers.bf16_pair((1, 900, 2, 128), 49, 2)
    q, k, v = q_t.to(dev), k_t.to(dev), v_t.to(dev)
    o0, l0 = jl.jl_bifocal_prefill(q, k, v, 900, 64, 1e6)
    for L, w, flags in ((100, 900, SW), (100, 5000, SW), (900, 64, SH), (1000, 64, PQ)):
        o1, l1 = jl.jl_bifocal_prefill_ex(q, k, v, 0, L, w, 1e6, flags)
        assert torch.equal(o0, o1) and torch.equal(l0, l1), (L, w, flags)
    assert jl.jl_debug_status() == 0


@pytest.mark.parametrize("B,Hq,Hkv,n,n_cap,D,L,w,flags", [
    (1, 32, 8, 5000, 5000, 128, 700, 300, SW),
    (2, 8, 2, 200, 260, 64, 50, 300, SW),       # n <= w: every key, capacity > n
    (3, 16, 8, 1000, 1024, 128, 100, 64, SW),
    (1, 32, 8, 5000, 5000, 128, 700, 300, SH),
    (2, 8, 2, 777, 800, 64, 300, 100, SH),
    (1, 32, 8, 5000, 5000, 128, 700, 300, PQ),
])
def test_decode_variants(jl, orc, dev, B, Hq, Hkv, n, n_cap, D, L, w, flags):
    q_t, q_f = helpers.bf16_pair((B, Hq, D), 51, 3)
    k_t, k_f = helpers.bf16_pair((B, n_cap, Hkv, D), 51, 4)
    v_t, v_f = helpers.bf16_pair((B, n_cap, Hkv, D), 51, 5)
    out, lse = jl.jl_bifocal_decode_ex(q_t.to(dev), k_t.to(dev), v_t.to(dev), n, L, w, 1e6, flags)
    assert jl.jl_debug_status() == 0
    ref_o, ref_l = orc.bifocal_rows_ex(q_f[:, None], k_f[:, :n], v_f[:, :n], [n - 1], n, L, w, 1e6, flags)
    helpers.compare(helpers.bf16_to_f64(out), lse.cpu().numpy(), ref_o[:, 0], ref_l[:, :, 0],
                    f"decode variant {flags} n={n} L={L} w={w}")


def test_decode_per_query_g_is_the_plain_decode_bitwise(jl, dev):
    import torch

    q_t, _ = helpers.bf16_pair((1, 32, 128), 53, 3)
    k_t, _ = helpers.bf16_pair((1, 9000, 8, 128), 53, 4)
    v_t, _ = helpers.bf16_pair((1, 9000, 8, 128), 53, 5)
    q, k, v = q_t.to(dev), k_t.to(dev), v_t.to(dev)
    o0, l0 = jl.jl_bifocal_decode(q, k, v, 9000, 2000, 512, 1e6)
    o1, l1 = jl.jl_bifocal_decode_ex(q, k, v, 9000, 2000, 512, 1e6, PQ)
    assert torch.equal(o0, o1) and torch.equal(l0, l1)


@pytest.mark.parametrize("flags", [PQ, SW, SH], ids=["per-query-g", "sliding", "query-shift"])
def test_variants_at_128k_sampled(jl, orc, dev, flags):
    """The Qwen3-8B-shaped 128K layer (B=1, Hq=32, Hkv=8, D=128, L=32768,
    w=4096) under each variant, run in full and checked on one seeded row of
    every 1024-row block plus the rows at the rule edges."""
    S, L, w = 131072, 32768, 4096
    g = max(1, jl.jl_group_factor_ex(S, L, w, flags))
    rng = np.random.default_rng(55 + flags)
    rows = set(int(r) for r in helpers.sample_rows(S, L, w, g, n_random=0))
    rows.update(int(1024 * b + rng.integers(0, 1024)) for b in range(S // 1024))
    rows.update((L - 1, L, 2 * L - 1, 2 * L, 3 * L - 1, 3 * L))  # per-query g changes here
    rows = np.array(sorted(r for r in rows if 0 <= r < S))
    _prefill_variant(jl, orc, dev, 1, 32, 8, S, 0, 128, L, w, flags, seed=2, rows=rows)
