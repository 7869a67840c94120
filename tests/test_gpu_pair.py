"""The two prefill tile kernels against the fp64 oracle and against each
other's selection rules.  The two-SM kernel (a cluster of two CTAs per query
tile of four heads, tcgen05 MMAs of M = 256 across both SMs, each CTA
correcting half of every K tile) is forced with JL_PREFILL_CTA_PAIR on the
shapes it applies to (D = 128, Hq / Hkv a multiple of 4); elsewhere that flag
must leave the result bit for bit as without it.  The one-CTA kernel is
forced with JL_PREFILL_ONE_CTA where the default would pick the two-SM one."""
import numpy as np
import pytest

import helpers

pytestmark = pytest.mark.gpu

PAIR = 8
ONE = 16
PQ, SW, SH = 1, 2, 4


def _case(jl, orc, dev, B, Hq, Hkv, S_new, n_past, L, w, flags, seed, rows=None, D=128, kernel=PAIR):
    from zero_shot_rope_02_b300 import inputs

    s = n_past + S_new
    qb = inputs.normal_bf16_bits((B, S_new, Hq, D), seed, 0)
    k_t, k_f = helpers.bf16_pair((B, s, Hkv, D), seed, 1)
    v_t, v_f = helpers.bf16_pair((B, s, Hkv, D), seed, 2)
    out, lse = jl.jl_bifocal_prefill_ex(inputs.to_torch_bf16(qb).to(dev), k_t.to(dev), v_t.to(dev), n_past, L, w,
                                        1e6, flags | kernel)
    assert jl.jl_debug_status() == 0
    if rows is None:
        rows = np.arange(S_new)
    ref_o, ref_l = orc.bifocal_rows_ex(inputs.bf16_bits_to_f64(qb[:, rows]), k_f, v_f, n_past + rows, s, L, w, 1e6,
                                       flags)
    helpers.compare(helpers.bf16_to_f64(out[:, rows]), lse[:, :, rows].cpu().numpy(), ref_o, ref_l,
                    f"pair kernel S_new={S_new} n_past={n_past} L={L} w={w} flags={flags}")


@pytest.mark.parametrize("B,Hq,Hkv,S_new,n_past,L,w,flags", [
    (1, 4, 1, 1000, 0, 300, 256, 0),     # grp = 4, g = 4
    (2, 8, 2, 700, 0, 200, 150, 0),      # two batch entries, ragged, band tiles
    (1, 8, 1, 1300, 0, 7, 129, 0),       # grp = 8 (two clusters per tile), g = 186
    (1, 4, 1, 640, 0, 100, 1, 0),        # w = 1: all but the diagonal remote
    (1, 8, 2, 900, 0, 1000, 64, 0),      # S <= L: plain
    (1, 4, 1, 300, 700, 100, 200, 0),    # a chunk over a cache
    (1, 4, 1, 700, 0, 200, 150, PQ),     # per-query g
    (1, 4, 1, 700, 0, 200, 150, SW),     # sliding window
    (1, 4, 1, 700, 0, 200, 150, SH),     # query shift
])
def test_pair_kernel_parity(jl, orc, dev, B, Hq, Hkv, S_new, n_past, L, w, flags):
    _case(jl, orc, dev, B, Hq, Hkv, S_new, n_past, L, w, flags, seed=61)


def test_pair_kernel_at_128k_sampled(jl, orc, dev):
    """The Qwen3-8B-shaped 128K layer: one seeded row of every 1024, plus the
    rule edges."""
    S, L, w = 131072, 32768, 4096
    rng = np.random.default_rng(63)
    rows = set(int(r) for r in helpers.sample_rows(S, L, w, 4, n_random=0))
    rows.update(int(1024 * b + rng.integers(0, 1024)) for b in range(S // 1024))
    _case(jl, orc, dev, 1, 32, 8, S, 0, L, w, 0, seed=2, rows=np.array(sorted(rows)))


def test_pair_flag_is_ignored_where_it_does_not_apply(jl, dev):
    """D = 64, or two heads per kv head: the one-CTA kernel runs either way."""
    import torch

    for (Hq, Hkv, D) in ((4, 1, 64), (4, 2, 128)):
        q_t, _ = helpers.bf16_pair((1, 700, Hq, D), 65, 0)
        k_t, _ = helpers.bf16_pair((1, 700, Hkv, D), 65, 1)
        v_t, _ = helpers.bf16_pair((1, 700, Hkv, D), 65, 2)
        q, k, v = q_t.to(dev), k_t.to(dev), v_t.to(dev)
        o0, l0 = jl.jl_bifocal_prefill_ex(q, k, v, 0, 200, 150, 1e6, 0)
        o1, l1 = jl.jl_bifocal_prefill_ex(q, k, v, 0, 200, 150, 1e6, PAIR)
        assert torch.equal(o0, o1) and torch.equal(l0, l1), (Hq, Hkv, D)


@pytest.mark.parametrize("B,Hq,Hkv,S_new,n_past,L,w,flags", [
    (1, 4, 1, 1000, 0, 300, 256, 0),     # grp = 4, g = 4
    (2, 8, 2, 700, 0, 200, 150, 0),      # ragged, band tiles
    (1, 4, 1, 300, 700, 100, 200, 0),    # a chunk over a cache
    (1, 4, 1, 700, 0, 200, 150, PQ),     # per-query g
    (1, 4, 1, 700, 0, 200, 150, SH),     # query shift
])
def test_one_cta_kernel_parity_where_the_pair_is_default(jl, orc, dev, B, Hq, Hkv, S_new, n_past, L, w, flags):
    _case(jl, orc, dev, B, Hq, Hkv, S_new, n_past, L, w, flags, seed=67, kernel=ONE)


def test_one_cta_kernel_at_128k_sampled(jl, orc, dev):
    """The Qwen3-8B-shaped 128K layer on the one-CTA kernel: one seeded row of
    every 1024, plus the rule edges."""
    S, L, w = 131072, 32768, 4096
    rng = np.random.default_rng(69)
    rows = set(int(r) for r in helpers.sample_rows(S, L, w, 4, n_random=0))
    rows.update(int(1024 * b + rng.integers(0, 1024)) for b in range(S // 1024))
    _case(jl, orc, dev, 1, 32, 8, S, 0, L, w, 0, seed=2, rows=np.array(sorted(rows)), kernel=ONE)


def test_default_kernel_choice(jl, dev):
    """Four heads per kv head at D = 128: with remote keys the default is the
    two-SM kernel, bit for bit; all exact (g = 1) it is the one-CTA kernel."""
    import torch

    q_t, _ = helpers.bf16_pair((1, 900, 8, 128), 71, 0)
    k_t, _ = helpers.bf16_pair((1, 900, 2, 128), 71, 1)
    v_t, _ = helpers.bf16_pair((1, 900, 2, 128), 71, 2)
    q, k, v = q_t.to(dev), k_t.to(dev), v_t.to(dev)
    for L, forced in ((200, PAIR), (1000, ONE)):
        o0, l0 = jl.jl_bifocal_prefill_ex(q, k, v, 0, L, 150, 1e6, 0)
        o1, l1 = jl.jl_bifocal_prefill_ex(q, k, v, 0, L, 150, 1e6, forced)
        assert torch.equal(o0, o1) and torch.equal(l0, l1), (L, forced)
    assert jl.jl_debug_status() == 0
