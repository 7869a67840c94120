"""CUDA path against the fp64 oracle, element by element, through the C ABI.

Small cases are checked in full; the benchmark-sized configurations are run
in full on the GPU and checked on sampled rows the oracle computes one by one,
plus invariants that hold at any size (bifocal-off equality, determinism).
"""
import numpy as np
import pytest

import helpers

pytestmark = pytest.mark.gpu


def _cuda(t, dev):
    return t.to(dev)


def _prefill_case(jl, orc, dev, B, Hq, Hkv, S, D, L, w, theta, seed, rows=None):
    from zero_shot_rope_02_b300 import inputs

    qb = inputs.normal_bf16_bits((B, S, Hq, D), seed, 0)
    k_t, k_f = helpers.bf16_pair((B, S, Hkv, D), seed, 1)
    v_t, v_f = helpers.bf16_pair((B, S, Hkv, D), seed, 2)
    out, lse = jl.jl_bifocal_prefill(_cuda(inputs.to_torch_bf16(qb), dev), _cuda(k_t, dev),
                                     _cuda(v_t, dev), L, w, theta)
    assert jl.jl_debug_status() == 0
    if rows is None:
        out_g = helpers.bf16_to_f64(out)
        lse_g = lse.cpu().numpy().astype(np.float64)
        ref_o, ref_l = orc.bifocal_prefill(inputs.bf16_bits_to_f64(qb), k_f, v_f, L, w, theta)
        return helpers.compare(out_g, lse_g, ref_o, ref_l, f"prefill S={S} L={L} w={w}")
    out_g = helpers.bf16_to_f64(out[:, rows])
    lse_g = lse[:, :, rows].cpu().numpy().astype(np.float64)
    del out, lse
    q_rows = inputs.bf16_bits_to_f64(qb[:, rows])
    ref_o, ref_l = orc.bifocal_rows(q_rows, k_f, v_f, rows, S, L, w, theta)
    return helpers.compare(out_g, lse_g, ref_o, ref_l, f"prefill S={S} L={L} w={w} (sampled rows)")


# ------------------------------------------------------------------ integer rules
@pytest.mark.parametrize("S,L", [(2048, 512), (131072, 32768), (100, 7), (5, 5), (65536, 4096)])
def test_grouped_positions_bitexact(jl, orc, dev, S, L):
    got = jl.jl_debug_grouped_positions(S, L).cpu().numpy()
    g = orc.group_factor(S, L)
    probe = np.unique(np.concatenate([np.arange(min(S, 300)), np.arange(max(0, S - 300), S),
                                      np.random.default_rng(1).integers(0, S, 500)]))
    want = np.array([orc.grouped_position(int(p), g) for p in probe])
    assert np.array_equal(got[probe], want)
    assert np.array_equal(got, np.arange(S) // g)
    assert got.max() <= L - 1  # every aliased position inside the pretrained window


def _classes_by_definition(S, L, w):
    """Brute force over every (query, key) pair of every 128x128 tile."""
    g = max(1, -(-S // L))
    nt = -(-S // 128)
    out = np.zeros((nt, nt), dtype=np.int8)
    i = np.arange(S)[:, None]
    j = np.arange(S)[None, :]
    causal = j <= i
    local = (i - j) < w
    for a in range(nt):
        for b in range(nt):
            sl = (slice(128 * a, 128 * a + 128), slice(128 * b, 128 * b + 128))
            c = causal[sl]
            if not c.any():
                out[a, b] = 0
            elif g == 1:
                out[a, b] = 1
            else:
                loc = local[sl][c]
                out[a, b] = 1 if loc.all() else (2 if not loc.any() else 3)
    return out


@pytest.mark.parametrize("S,L,w", [(2048, 512, 128), (700, 200, 150), (1000, 300, 1), (513, 600, 5),
                                   (1500, 100, 2000), (900, 250, 64)])
def test_tile_classes_match_definition(jl, dev, S, L, w):
    got = jl.jl_debug_tile_classes(S, L, w).cpu().numpy()
    assert np.array_equal(got, _classes_by_definition(S, L, w))


def test_bounded_wait_gives_up_and_reports(jl, dev):
    """A wait whose phase never completes gives up after its limit, sets
    JL_ERR_TIMEOUT in the status word, and leaves the context usable."""
    import torch

    assert jl.jl_debug_status() == 0
    assert jl.jl_debug_wait_timeout(1_000_000) == 1
    assert jl.jl_debug_status() == jl.JL_ERR_TIMEOUT
    assert jl.jl_debug_status() == 0  # read-and-clear
    x = torch.ones(1024, device=dev)
    assert float(x.sum().item()) == 1024.0


# ------------------------------------------------------------------ rope
@pytest.mark.parametrize("D,pos0,theta", [(128, 0, 1e6), (128, 123457, 1e6), (64, 70000, 1e4),
                                          (16, 5, 500.0), (6, 3, 1e4)])
def test_rope_parity(jl, orc, dev, D, pos0, theta):
    x_t, x_f = helpers.bf16_pair((2, 37, 3, D), 9, 0)
    x = _cuda(x_t, dev)
    jl.jl_rope_apply(x, pos0, theta)
    got = helpers.bf16_to_f64(x)
    ref = orc.rope(x_f, pos0, theta)
    # one rounding to bf16 of an fp32 result: within 2^-8 relative (+ fp32 slack)
    err = np.abs(got - ref)
    assert np.all(err <= np.abs(ref) * 2.0 ** -8 + 1e-5 * np.abs(x_f).max()), float(err.max())
    if pos0 == 0:
        assert np.array_equal(got[:, 0], x_f[:, 0])  # position 0 is the identity, bitwise


# ------------------------------------------------------------------ decode
def _decode_case(jl, orc, dev, B, Hq, Hkv, n, n_cap, D, L, w, theta, seed, ws=None):
    q_t, q_f = helpers.bf16_pair((B, Hq, D), seed, 3)
    k_t, k_f = helpers.bf16_pair((B, n_cap, Hkv, D), seed, 4)
    v_t, v_f = helpers.bf16_pair((B, n_cap, Hkv, D), seed, 5)
    out, lse = jl.jl_bifocal_decode(_cuda(q_t, dev), _cuda(k_t, dev), _cuda(v_t, dev), n, L, w, theta,
                                    workspace=ws)
    assert jl.jl_debug_status() == 0
    ref_o, ref_l = orc.bifocal_decode(q_f[:, None], k_f[:, :n], v_f[:, :n], L, w, theta)
    return helpers.compare(helpers.bf16_to_f64(out), lse.cpu().numpy(), ref_o[:, 0], ref_l[:, :, 0],
                           f"decode n={n} L={L} w={w}")


@pytest.mark.parametrize("B,Hq,Hkv,n,n_cap,D,L,w", [
    (1, 4, 4, 1, 1, 128, 4, 1),         # a single key
    (2, 8, 2, 7, 9, 64, 3, 2),          # capacity > n, g = 3
    (1, 32, 8, 130, 130, 128, 16, 17),  # g = 9, ragged split
    (3, 16, 8, 1000, 1024, 128, 100, 64),
    (1, 8, 1, 5000, 5000, 64, 700, 300),  # grp = 8
    (1, 32, 8, 3000, 3000, 128, 4096, 8),  # n <= L: plain RoPE
    (1, 32, 8, 3000, 3000, 128, 32, 5000),  # w >= n: plain RoPE
])
def test_decode_parity_small(jl, orc, dev, B, Hq, Hkv, n, n_cap, D, L, w):
    _decode_case(jl, orc, dev, B, Hq, Hkv, n, n_cap, D, L, w, 1e6, seed=3)


@pytest.mark.parametrize("B,Hq,Hkv,n,n_cap,L,w", [
    (1, 8, 8, 256, 256, 64, 100),          # the shortest cache on the tensor cores; grp 1, g = 4
    (1, 16, 2, 257, 300, 64, 128),         # grp 8, one key past a tile, edge inside tile 1
    (1, 16, 2, 257, 300, 64, 129),         # edge on a tile boundary: no crossed tile
    (1, 4, 1, 700, 700, 100, 1),           # w = 1: only the last key exact, g = 7
    (2, 32, 8, 1500, 1600, 400, 300),      # B = 2, g = 4, edge inside a middle tile
    (1, 8, 2, 5000, 5000, 1000, 37),       # grp 4, g = 5 (not a divisor of 16), many splits
    (1, 4, 2, 20000, 20000, 3000, 2500),   # grp 2, g = 7, splits of several tiles
    (1, 32, 8, 40000, 40000, 32768, 4096),  # g = 2
    (4, 32, 8, 9000, 9000, 4096, 1024),    # B = 4: four splits per (batch, kv head)
    (20, 16, 8, 600, 600, 128, 200),       # 160 (batch, kv head) pairs: one split each
])
def test_decode_tensor_core_path(jl, orc, dev, B, Hq, Hkv, n, n_cap, L, w):
    """Head dimension 128 and n >= 256 take the tcgen05 kernel: tile classes
    (remote, crossed by the window edge, exact), group sizes, split counts."""
    _decode_case(jl, orc, dev, B, Hq, Hkv, n, n_cap, 128, L, w, 1e6, seed=11)


def test_decode_tensor_core_rescales(jl, orc, dev):
    """The tensor-core decode's running offset under scores that jump by
    hundreds of log2 units from tile to tile inside one split (keys doubled
    every 256 positions from 1000 on, queries x 2^3; six tiles per split):
    O must be rescaled in TMEM between its P.V steps.  L >= n: every tile
    exact, bf16 operands (as the prefill's jumping-scores test)."""
    import torch

    B, Hq, Hkv, n, D, L, w = 4, 8, 8, 3000, 128, 4096, 256
    q_t, q_f = helpers.bf16_pair((B, Hq, D), 17, 3, scale=8.0)
    k_t, k_f = helpers.bf16_pair((B, n, Hkv, D), 17, 4)
    v_t, v_f = helpers.bf16_pair((B, n, Hkv, D), 17, 5, scale=0.25)
    for j in range(1000, n, 256):
        k_t[:, j:] *= 2.0
        k_f[:, j:] *= 2.0
    out, lse = jl.jl_bifocal_decode(_cuda(q_t, dev), _cuda(k_t, dev), _cuda(v_t, dev), n, L, w, 1e6)
    assert jl.jl_debug_status() == 0
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    ref_o, ref_l = orc.bifocal_decode(q_f[:, None], k_f, v_f, L, w, 1e6)
    assert float(np.max(ref_l)) > 500.0  # the jumps are really there
    helpers.compare(helpers.bf16_to_f64(out), lse.cpu().numpy(), ref_o[:, 0], ref_l[:, :, 0],
                    "decode with jumping scores")


@pytest.mark.parametrize("n", [8192, 32768, 131072])
def test_decode_parity_benchmark_sizes(jl, orc, dev, n):
    """Single-batch decode, Hq=32, Hkv=8, D=128, L=32768, w=4096, theta=1e6 (g = 1, 1, 4)."""
    _decode_case(jl, orc, dev, 1, 32, 8, n, n, 128, 32768, 4096, 1e6, seed=3)


def test_decode_workspace_reuse(jl, orc, dev):
    """Calls that share a workspace: counters come back to zero after each call."""
    import torch

    nbytes = jl.jl_bifocal_decode_workspace_size(1, 32, 8, 20000, 128)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
    for n in (20000, 9000, 20000):
        _decode_case(jl, orc, dev, 1, 32, 8, n, 20000, 128, 4096, 1024, 1e6, seed=3, ws=ws)
    hdr = ws[:256].view(torch.int32)[:8]
    assert int(hdr.abs().sum()) == 0


# ------------------------------------------------------------------ prefill
def test_prefill_tiny_config(jl, orc, dev):
    """B=1, H=1, D=64, S=2048, L=512 (g=4), w=128, theta=1e4, seed 0: every row."""
    _prefill_case(jl, orc, dev, 1, 1, 1, 2048, 64, 512, 128, 1e4, seed=0)


@pytest.mark.parametrize("B,Hq,Hkv,S,D,L,w", [
    (1, 1, 1, 1, 128, 1, 1),          # one token
    (1, 2, 1, 127, 128, 30, 20),      # one ragged tile
    (2, 4, 2, 700, 128, 200, 150),    # ragged, several band tiles, g = 4
    (1, 2, 2, 640, 64, 100, 1),       # w = 1: everything but the diagonal is remote
    (1, 4, 1, 1000, 128, 300, 256),   # grp = 4, g = 4
    (1, 2, 1, 900, 128, 1000, 64),    # S <= L: plain
    (1, 2, 1, 900, 64, 50, 5000),     # w >= S: plain
    (1, 1, 1, 1300, 128, 7, 129),     # g = 186 (not a divisor of 128)
])
def test_prefill_parity_small(jl, orc, dev, B, Hq, Hkv, S, D, L, w):
    _prefill_case(jl, orc, dev, B, Hq, Hkv, S, D, L, w, 1e6, seed=5)


def test_prefill_bifocal_off_is_bitwise_plain(jl, orc, dev):
    """With L >= S (g = 1) the kernel takes the plain path: results do not
    depend on L or w at all (base model recovered exactly)."""
    import torch

    q_t, q_f = helpers.bf16_pair((1, 1000, 4, 128), 6, 0)
    k_t, k_f = helpers.bf16_pair((1, 1000, 2, 128), 6, 1)
    v_t, v_f = helpers.bf16_pair((1, 1000, 2, 128), 6, 2)
    q, k, v = (_cuda(t, dev) for t in (q_t, k_t, v_t))
    o1, l1 = jl.jl_bifocal_prefill(q, k, v, 1000, 64, 1e6)
    o2, l2 = jl.jl_bifocal_prefill(q, k, v, 5000, 3, 1e6)
    o3, l3 = jl.jl_bifocal_prefill(q, k, v, 300, 5000, 1e6)  # w >= S
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(o1, o3) and torch.equal(l1, l3)
    ref_o, ref_l = orc.bifocal_prefill(q_f, k_f, v_f, 1000, 64, 1e6)
    helpers.compare(helpers.bf16_to_f64(o1), l1.cpu().numpy(), ref_o, ref_l, "plain")


def test_prefill_deterministic(jl, dev):
    import torch

    q_t, _ = helpers.bf16_pair((1, 1500, 4, 128), 7, 0)
    k_t, _ = helpers.bf16_pair((1, 1500, 2, 128), 7, 1)
    v_t, _ = helpers.bf16_pair((1, 1500, 2, 128), 7, 2)
    q, k, v = (_cuda(t, dev) for t in (q_t, k_t, v_t))
    o1, l1 = jl.jl_bifocal_prefill(q, k, v, 400, 300, 1e6)
    o2, l2 = jl.jl_bifocal_prefill(q, k, v, 400, 300, 1e6)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_decode_matches_last_prefill_row(jl, dev):
    """Decode at position n-1 over the prefill's own k/v equals prefill row n-1."""
    n = 3000
    q_t, _ = helpers.bf16_pair((1, n, 32, 128), 8, 0)
    k_t, _ = helpers.bf16_pair((1, n, 8, 128), 8, 1)
    v_t, _ = helpers.bf16_pair((1, n, 8, 128), 8, 2)
    q, k, v = (_cuda(t, dev) for t in (q_t, k_t, v_t))
    o_p, l_p = jl.jl_bifocal_prefill(q, k, v, 500, 700, 1e6)
    o_d, l_d = jl.jl_bifocal_decode(q[:, n - 1].contiguous(), k, v, n, 500, 700, 1e6)
    d = (o_p[:, n - 1].float() - o_d.float()).abs().max().item()
    assert d <= 1e-2
    assert ((l_p[:, :, n - 1] - l_d).abs() / l_d.abs()).max().item() <= 1e-4


@pytest.mark.parametrize("name,B,Hq,Hkv,S,L,w,seed", [
    ("qwen3-1.7b 64K", 1, 16, 8, 65536, 32768, 4096, 1),
    ("qwen3-8b 128K", 1, 32, 8, 131072, 32768, 4096, 2),
])
def test_prefill_benchmark_configs_sampled(jl, orc, dev, name, B, Hq, Hkv, S, L, w, seed):
    """Run in full; checked on the rule-edge rows and on one seeded row of
    every 128-row query tile (512 / 1024 tiles), every head."""
    g = orc.group_factor(S, L)
    rng = np.random.default_rng(seed)
    per_tile = np.arange(0, S, 128) + rng.integers(0, 128, size=S // 128)
    rows = np.unique(np.concatenate([helpers.sample_rows(S, L, w, g, n_random=0), per_tile]))
    _prefill_case(jl, orc, dev, B, Hq, Hkv, S, 128, L, w, 1e6, seed=seed, rows=rows)


def test_prefill_scores_jumping_by_thousands(jl, orc, dev):
    """Later keys (x 2^6) and all queries (x 2^3) scaled so that a row's maximum
    jumps by hundreds to thousands of log2 units between tiles: the running
    offset must follow without P overflowing (exact power-of-two rescales).
    Run with L >= S (every tile exact, bf16 operands): at scores this large
    the fp16 rounding of corrected operands alone would move a score by about
    one unit, which is outside that path's stated operand range."""
    import torch

    B, Hq, Hkv, S, D, L, w = 1, 2, 1, 700, 128, 1000, 150
    q_t, q_f = helpers.bf16_pair((B, S, Hq, D), 15, 0, scale=8.0)
    k_t, k_f = helpers.bf16_pair((B, S, Hkv, D), 15, 1)
    # v x 2^-2: one key takes nearly all the weight here, so the bf16 rounding
    # of P and of out lands on |out| undivided; small v keeps that inside 1e-2
    v_t, v_f = helpers.bf16_pair((B, S, Hkv, D), 15, 2, scale=0.25)
    k_t[:, 300:] *= 64.0
    k_f[:, 300:] *= 64.0
    out, lse = jl.jl_bifocal_prefill(_cuda(q_t, dev), _cuda(k_t, dev), _cuda(v_t, dev), L, w, 1e6)
    assert jl.jl_debug_status() == 0
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    ref_o, ref_l = orc.bifocal_prefill(q_f, k_f, v_f, L, w, 1e6)
    assert float(np.max(ref_l)) > 500.0  # the jump is really there
    helpers.compare(helpers.bf16_to_f64(out), lse.cpu().numpy(), ref_o, ref_l, "scores jumping")
