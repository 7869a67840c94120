"""Batched decode over a paged cache with one length per sequence
(jl_bifocal_decode_paged), against the fp64 oracle.  The kernel splits the
batch's keys over its CTAs in proportion to the sequences' lengths, reading
the lengths on the device.

Every sequence b has its own length n_b and so its own g = g(n_b, L) (the
group factor follows the current length: ResearchPod summary, "every
length"); the oracle decodes each sequence alone over its keys gathered from
the pool.  Pages are shuffled in the pool, unused pages and the tail of each
sequence's last page hold NaN, and table entries past a sequence's last page
hold ids outside the pool: none of them may reach a result.
"""
import numpy as np
import pytest

import helpers

pytestmark = pytest.mark.gpu


def _paged_case(jl, orc, dev, lens, Hq, Hkv, D, page_size, L, w, seed, spare_pages=5):
    import torch

    B = len(lens)
    pages_per = [-(-n // page_size) for n in lens]
    max_pages = max(pages_per) + 2
    num_pages = sum(pages_per) + spare_pages
    rng = np.random.default_rng(seed)
    perm = rng.permutation(num_pages)
    q_t, q_f = helpers.bf16_pair((B, Hq, D), seed, 3)
    kp_t, kp_f = helpers.bf16_pair((num_pages, page_size, Hkv, D), seed, 4)
    vp_t, vp_f = helpers.bf16_pair((num_pages, page_size, Hkv, D), seed, 5)
    table = np.full((B, max_pages), num_pages + 7, dtype=np.int32)  # outside the pool
    used = np.zeros(num_pages, dtype=bool)
    nxt = 0
    for b, n in enumerate(lens):
        for p in range(pages_per[b]):
            table[b, p] = perm[nxt]
            used[perm[nxt]] = True
            nxt += 1
        last = table[b, pages_per[b] - 1]
        tail = n - (pages_per[b] - 1) * page_size
        kp_t[last, tail:] = float("nan")
        vp_t[last, tail:] = float("nan")
    kp_t[~torch.from_numpy(used)] = float("nan")
    vp_t[~torch.from_numpy(used)] = float("nan")
    out, lse = jl.jl_bifocal_decode_paged(
        q_t.to(dev), kp_t.to(dev), vp_t.to(dev), torch.from_numpy(table).to(dev),
        torch.tensor(lens, dtype=torch.int32, device=dev), max(lens), L, w, 1e6)
    assert jl.jl_debug_status() == 0
    out_g, lse_g = helpers.bf16_to_f64(out), lse.cpu().numpy()
    for b, n in enumerate(lens):
        idx = table[b, :pages_per[b]]
        k_b = kp_f[idx].reshape(-1, Hkv, D)[:n][None]
        v_b = vp_f[idx].reshape(-1, Hkv, D)[:n][None]
        ref_o, ref_l = orc.bifocal_decode(q_f[b:b + 1, None], k_b, v_b, L, w, 1e6)
        helpers.compare(out_g[b:b + 1], lse_g[b:b + 1], ref_o[:, 0], ref_l[:, :, 0],
                        f"paged decode b={b} n={n} g={orc.group_factor(n, L)}")


@pytest.mark.parametrize("lens,Hq,Hkv,D,page_size,L,w", [
    ((1, 1000, 5000), 32, 8, 128, 64, 700, 256),     # g = 1, 2, 8 in one batch
    ((3000, 64, 4097, 130), 16, 8, 128, 128, 1000, 64),  # page 128, g = 3, 1, 5, 1
    ((777, 2048), 8, 4, 64, 64, 300, 100),            # D = 64, grp = 2, g = 3, 7
    ((9000,), 32, 8, 128, 64, 9000, 4096),            # n <= L: plain RoPE
    # twelve sequences: the device shares the CTAs out in proportion to length
    ((5, 77, 300, 4097, 12000, 64, 1, 2000, 700, 9000, 128, 33), 32, 8, 128, 64, 1000, 256),
])
def test_paged_decode_parity(jl, orc, dev, lens, Hq, Hkv, D, page_size, L, w):
    _paged_case(jl, orc, dev, list(lens), Hq, Hkv, D, page_size, L, w, seed=21)


def test_paged_decode_clamps_a_length_past_the_plan(jl, dev):
    """A seq_lens entry beyond max_n is clamped on the device and reported as
    JL_ERR_GUARD; the call reads nothing past the table."""
    import torch

    B, Hq, Hkv, D, P = 2, 8, 2, 128, 64
    q = torch.zeros((B, Hq, D), dtype=torch.bfloat16, device=dev)
    pages = torch.zeros((4, P, Hkv, D), dtype=torch.bfloat16, device=dev)
    table = torch.tensor([[0, 1], [2, 3]], dtype=torch.int32, device=dev)
    lens = torch.tensor([100, 100000], dtype=torch.int32, device=dev)  # 100000 > max_n = 128
    out, lse = jl.jl_bifocal_decode_paged(q, pages, pages, table, lens, 128, 64, 32, 1e6)
    assert jl.jl_debug_status() == jl.JL_ERR_GUARD
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    assert jl.jl_debug_status() == 0  # the query cleared it


def test_paged_decode_reports_a_page_id_outside_the_pool(jl, dev):
    """A block-table entry that a sequence uses but that names no page of the
    pool reads zeros (never faults) and is reported as JL_ERR_GUARD."""
    import torch

    B, Hq, Hkv, D, P = 1, 8, 2, 128, 64
    q = torch.ones((B, Hq, D), dtype=torch.bfloat16, device=dev)
    pages = torch.ones((4, P, Hkv, D), dtype=torch.bfloat16, device=dev)
    table = torch.tensor([[0, 9]], dtype=torch.int32, device=dev)  # page 9 of a 4-page pool
    lens = torch.tensor([100], dtype=torch.int32, device=dev)       # uses both table entries
    jl.jl_bifocal_decode_paged(q, pages, pages, table, lens, 128, 64, 32, 1e6)
    assert jl.jl_debug_status() == jl.JL_ERR_GUARD
    assert jl.jl_debug_status() == 0
    table_ok = torch.tensor([[0, 3]], dtype=torch.int32, device=dev)
    jl.jl_bifocal_decode_paged(q, pages, pages, table_ok, lens, 128, 64, 32, 1e6)
    assert jl.jl_debug_status() == 0
