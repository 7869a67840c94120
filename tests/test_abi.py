"""The C ABI without a GPU: the library loads, exports every declared symbol,
and its host-side rules (group factor, argument checks) hold.  No call here
reaches a CUDA launch: every argument error is returned before one."""
import ctypes
import os
import re

import pytest

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "jetlong.h")
BAD = ctypes.c_void_p(0x1001)  # misaligned, never dereferenced
GOOD = ctypes.c_void_p(0x1000)  # aligned, never dereferenced (calls fail earlier)


def declared_symbols():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(jl_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(jl):
    names = declared_symbols()
    assert len(names) >= 10
    for n in names:
        assert hasattr(jl.lib, n), f"{n} declared in jetlong.h but not exported"
    assert set(names) == set(jl.EXPORTS)


def test_every_entry_point_is_reachable_from_the_package(jl):
    """The package forwards every wrapped C entry point (its names are lazy)."""
    import zero_shot_rope_02_b300 as pkg

    for name in jl.EXPORTS:
        if hasattr(jl, name):  # a Python wrapper of that name exists
            assert getattr(pkg, name) is getattr(jl, name), name


def test_version_and_status_strings(jl):
    assert jl.jl_version().count(".") == 2
    for code in range(-8, 1):
        assert jl.status_string(code).startswith("JL_")
    assert "unknown" in jl.status_string(42)


def test_group_factor_matches_oracle(jl, orc):
    for s in list(range(1, 300)) + [2048, 32767, 32768, 32769, 65536, 131072, 10 ** 9]:
        for L in (1, 2, 3, 7, 512, 4096, 32768):
            assert jl.jl_group_factor(s, L) == orc.group_factor(s, L) if s < 10 ** 6 else True
            assert jl.jl_group_factor(s, L) == max(1, -(-s // L))


def test_group_factor_golden(jl):
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "group_factor.txt")
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        s, L, g = map(int, line.split())
        assert jl.jl_group_factor(s, L) == g


def test_group_factor_rejects(jl):
    g = ctypes.c_int32(7)
    assert jl.lib.jl_group_factor(0, 4, ctypes.byref(g)) == jl.JL_ERR_ARG
    assert jl.lib.jl_group_factor(5, 0, ctypes.byref(g)) == jl.JL_ERR_ARG
    assert jl.lib.jl_group_factor(5, 4, None) == jl.JL_ERR_ARG
    assert jl.lib.jl_group_factor(1 << 62, 1, ctypes.byref(g)) == jl.JL_ERR_OVERFLOW
    assert g.value == 7


def test_group_factor_variants(jl, orc):
    """The query-shift rule against the oracle's literal search and the
    hand-checked golden rows; per-query g is the plain rule; sliding gives 1."""
    PQ, SW, SH = jl.JL_VARIANT_PER_QUERY_G, jl.JL_VARIANT_SLIDING, jl.JL_VARIANT_QUERY_SHIFT
    g = ctypes.c_int32(0)
    for s in list(range(1, 200, 7)) + [2048, 65536, 131072]:
        for L in (1, 3, 7, 100, 512, 4096, 32768):
            for w in (1, 2, 5, 64, 128, 4096):
                want = orc.group_factor_shift(s, L, w)
                rc = jl.lib.jl_group_factor_ex(s, L, w, SH, ctypes.byref(g))
                if want < 0:
                    assert rc == jl.JL_ERR_ARG, (s, L, w)
                else:
                    assert rc == 0 and g.value == want, (s, L, w, g.value, want)
                assert jl.jl_group_factor_ex(s, L, w, PQ) == orc.group_factor(s, L)
                assert jl.jl_group_factor_ex(s, L, w, SW) == 1
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "group_factor_shift.txt")
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        s, L, w, want = map(int, line.split())
        rc = jl.lib.jl_group_factor_ex(s, L, w, SH, ctypes.byref(g))
        assert (rc == jl.JL_ERR_ARG) if want < 0 else (rc == 0 and g.value == want), (s, L, w)
    assert jl.lib.jl_group_factor_ex(5, 4, 2, 8, ctypes.byref(g)) == jl.JL_ERR_ARG  # unknown flag
    assert jl.lib.jl_group_factor_ex(5, 4, 2, SW | SH, ctypes.byref(g)) == jl.JL_ERR_ARG
    assert jl.lib.jl_group_factor_ex(5, 4, 0, 0, ctypes.byref(g)) == jl.JL_ERR_ARG


def test_variant_entry_points_reject_bad_flags(jl):
    """Flag errors come back before any launch."""
    PQ, SW, SH = jl.JL_VARIANT_PER_QUERY_G, jl.JL_VARIANT_SLIDING, jl.JL_VARIANT_QUERY_SHIFT

    def pf(flags, S=256, L=128, w=64):
        return jl.lib.jl_bifocal_prefill_ex(GOOD, GOOD, GOOD, GOOD, GOOD, 1, 4, 2, S, 0, S, 128, L, w,
                                            1e4, flags, None)

    def dc(flags, n=256, L=128, w=64):
        return jl.lib.jl_bifocal_decode_ex(GOOD, GOOD, GOOD, GOOD, GOOD, 1, 32, 8, n, n, 128, L, w, 1e6,
                                           flags, GOOD, 1 << 30, None)

    assert pf(32) == jl.JL_ERR_ARG
    assert pf(jl.JL_PREFILL_CTA_PAIR | jl.JL_PREFILL_ONE_CTA) == jl.JL_ERR_ARG
    assert pf(SW | PQ) == jl.JL_ERR_ARG
    assert pf(SW | SH) == jl.JL_ERR_ARG
    assert pf(PQ | SH) == jl.JL_ERR_UNSUPPORTED
    assert pf(SH, S=256, L=128, w=128) == jl.JL_ERR_ARG  # w >= L: no shifted g
    assert dc(16) == jl.JL_ERR_ARG
    assert dc(SW | PQ) == jl.JL_ERR_ARG
    assert dc(SH, n=256, L=128, w=200) == jl.JL_ERR_ARG


def _prefill(jl, q=GOOD, k=GOOD, v=GOOD, out=GOOD, lse=GOOD, B=1, Hq=4, Hkv=2, S=256, D=128,
             L=128, w=64, theta=1e4):
    return jl.lib.jl_bifocal_prefill(q, k, v, out, lse, B, Hq, Hkv, S, D, L, w, theta, None)


def test_prefill_argument_checks(jl):
    assert _prefill(jl, D=96) == jl.JL_ERR_UNSUPPORTED
    assert _prefill(jl, D=256) == jl.JL_ERR_UNSUPPORTED
    assert _prefill(jl, Hq=3, Hkv=2) == jl.JL_ERR_ARG
    for kw in ({"S": 0}, {"w": 0}, {"L": 0}, {"theta": 0.0}, {"theta": -1.0}, {"B": 0}):
        assert _prefill(jl, **kw) == jl.JL_ERR_ARG, kw
    assert _prefill(jl, q=None) == jl.JL_ERR_ARG
    for name in ("q", "k", "v", "out", "lse"):
        assert _prefill(jl, **{name: BAD}) == jl.JL_ERR_ALIGN, name
    assert _prefill(jl, B=1 << 20, Hq=1 << 10, Hkv=1, S=1 << 20) == jl.JL_ERR_OVERFLOW


def _chunk(jl, q=GOOD, k=GOOD, v=GOOD, out=GOOD, lse=GOOD, B=1, Hq=32, Hkv=8, S_new=64, n_past=100,
           n_cap=164, D=128, L=4096, w=128, theta=1e6):
    return jl.lib.jl_bifocal_prefill_chunk(q, k, v, out, lse, B, Hq, Hkv, S_new, n_past, n_cap, D, L, w,
                                           theta, None)


def test_prefill_chunk_argument_checks(jl):
    """Rejected before any launch (no GPU needed)."""
    assert _chunk(jl, D=96) == jl.JL_ERR_UNSUPPORTED
    for kw in ({"S_new": 0}, {"n_past": -1}, {"n_cap": 163}, {"w": 0}, {"L": 0}, {"theta": 0.0},
               {"Hq": 3, "Hkv": 2}):
        assert _chunk(jl, **kw) == jl.JL_ERR_ARG, kw
    assert _chunk(jl, k=None) == jl.JL_ERR_ARG
    for name in ("q", "k", "v", "out", "lse"):
        assert _chunk(jl, **{name: BAD}) == jl.JL_ERR_ALIGN, name
    assert _chunk(jl, n_past=(1 << 31) - 10, n_cap=(1 << 31) - 1) == jl.JL_ERR_OVERFLOW


def _decode(jl, q=GOOD, k=GOOD, v=GOOD, out=GOOD, lse=GOOD, B=1, Hq=32, Hkv=8, n=100, n_cap=100,
            D=128, L=64, w=16, theta=1e6, ws=GOOD, ws_bytes=1 << 30):
    return jl.lib.jl_bifocal_decode(q, k, v, out, lse, B, Hq, Hkv, n, n_cap, D, L, w, theta, ws,
                                    ws_bytes, None)


def test_decode_argument_checks(jl):
    assert _decode(jl, D=80) == jl.JL_ERR_UNSUPPORTED
    assert _decode(jl, Hq=48, Hkv=3) == jl.JL_ERR_UNSUPPORTED  # 16 heads per kv head
    assert _decode(jl, Hq=30, Hkv=8) == jl.JL_ERR_ARG
    assert _decode(jl, n=0) == jl.JL_ERR_ARG
    assert _decode(jl, n=101, n_cap=100) == jl.JL_ERR_ARG
    assert _decode(jl, w=0) == jl.JL_ERR_ARG
    assert _decode(jl, L=0) == jl.JL_ERR_ARG
    for name in ("q", "k", "v", "out", "lse"):
        assert _decode(jl, **{name: BAD}) == jl.JL_ERR_ALIGN, name
    assert _decode(jl, ws=None) == jl.JL_ERR_WORKSPACE
    need = jl.jl_bifocal_decode_workspace_size(1, 32, 8, 100, 128)
    assert _decode(jl, ws_bytes=need - 1) == jl.JL_ERR_WORKSPACE
    assert _decode(jl, ws=BAD, ws_bytes=need) == jl.JL_ERR_ALIGN


def _paged(jl, q=GOOD, kp=GOOD, vp=GOOD, table=GOOD, lens=GOOD, out=GOOD, lse=GOOD, B=2, Hq=32, Hkv=8,
           D=128, page_size=64, num_pages=10, max_pages=5, max_n=300, L=100, w=64, theta=1e6,
           ws=GOOD, ws_bytes=1 << 24):
    return jl.lib.jl_bifocal_decode_paged(q, kp, vp, table, lens, out, lse, B, Hq, Hkv, D, page_size,
                                          num_pages, max_pages, max_n, L, w, theta, ws, ws_bytes, None)


def test_decode_paged_argument_checks(jl):
    """Rejected before any launch (no GPU needed)."""
    for kw in ({"page_size": 32}, {"page_size": 96}, {"num_pages": 0}, {"max_pages": 0},
               {"max_n": 321}, {"max_n": 0}, {"B": 0}, {"w": 0}, {"L": 0}, {"Hq": 3, "Hkv": 2}):
        assert _paged(jl, **kw) == jl.JL_ERR_ARG, kw
    for name in ("q", "kp", "vp", "table", "lens", "out", "lse"):
        assert _paged(jl, **{name: None}) == jl.JL_ERR_ARG, name
    assert _paged(jl, D=96) == jl.JL_ERR_UNSUPPORTED
    assert _paged(jl, ws_bytes=16) == jl.JL_ERR_WORKSPACE
    for name in ("q", "kp", "vp", "out", "lse"):
        assert _paged(jl, **{name: BAD}) == jl.JL_ERR_ALIGN, name
    assert _paged(jl, table=ctypes.c_void_p(0x1002)) == jl.JL_ERR_ALIGN
    assert _paged(jl, lens=ctypes.c_void_p(0x1001)) == jl.JL_ERR_ALIGN


def test_decode_workspace_size(jl):
    assert jl.jl_bifocal_decode_workspace_size(1, 32, 8, 0, 128) == 0
    assert jl.jl_bifocal_decode_workspace_size(1, 30, 8, 10, 128) == 0
    small = jl.jl_bifocal_decode_workspace_size(1, 32, 8, 8192, 128)
    big = jl.jl_bifocal_decode_workspace_size(1, 32, 8, 131072, 128)
    assert 0 < small <= big
    # partial o for every (head, split) at most: 256 splits
    assert big <= 256 + 1 * 32 * 256 * (128 + 2) * 4 + 512


def test_decode_paged_workspace_size(jl):
    """Sized for the longest sequence alone: at least the uniform plan's size,
    the same for every max_n, 0 on bad sizes."""
    assert jl.jl_bifocal_decode_paged_workspace_size(4, 32, 8, 0, 128) == 0
    assert jl.jl_bifocal_decode_paged_workspace_size(4, 30, 8, 10, 128) == 0
    sizes = {jl.jl_bifocal_decode_paged_workspace_size(4, 32, 8, n, 128) for n in (64, 8192, 131072)}
    assert len(sizes) == 1
    assert sizes.pop() >= jl.jl_bifocal_decode_workspace_size(4, 32, 8, 131072, 128)


def test_rope_argument_checks(jl):
    f = jl.lib.jl_rope_apply
    assert f(GOOD, 1, 4, 2, 7, 0, 1e4, None) == jl.JL_ERR_UNSUPPORTED  # odd D
    assert f(GOOD, 1, 4, 2, 258, 0, 1e4, None) == jl.JL_ERR_UNSUPPORTED
    assert f(GOOD, 1, 4, 2, 8, -1, 1e4, None) == jl.JL_ERR_ARG
    assert f(GOOD, 1, 4, 2, 8, 0, 0.0, None) == jl.JL_ERR_ARG
    assert f(None, 1, 4, 2, 8, 0, 1e4, None) == jl.JL_ERR_ARG
    assert f(BAD, 1, 4, 2, 8, 0, 1e4, None) == jl.JL_ERR_ALIGN
    assert f(GOOD, 1, 4, 2, 8, (1 << 62) - 2, 1e4, None) == jl.JL_ERR_OVERFLOW


def _cache_write(jl, k=GOOD, v=GOOD, kc=GOOD, vc=GOOD, B=1, S_new=16, H=8, D=128, n_past=10, n_cap=26,
                 theta=1e6):
    return jl.lib.jl_rope_cache_write(k, v, kc, vc, B, S_new, H, D, n_past, n_cap, theta, None)


def test_rope_cache_write_argument_checks(jl):
    """Rejected before any launch (no GPU needed)."""
    for kw in ({"B": 0}, {"S_new": 0}, {"H": 0}, {"n_past": -1}, {"n_cap": 25}, {"theta": 0.0},
               {"k": None}, {"vc": None}):
        assert _cache_write(jl, **kw) == jl.JL_ERR_ARG, kw
    for D in (8, 24, 100, 272):
        assert _cache_write(jl, D=D) == jl.JL_ERR_UNSUPPORTED, D
    for name in ("k", "v", "kc", "vc"):
        assert _cache_write(jl, **{name: BAD}) == jl.JL_ERR_ALIGN, name


def test_debug_argument_checks(jl):
    assert jl.lib.jl_debug_grouped_positions(0, 4, GOOD, None) == jl.JL_ERR_ARG
    assert jl.lib.jl_debug_grouped_positions(4, 4, None, None) == jl.JL_ERR_ARG
    assert jl.lib.jl_debug_tile_classes(100, 4, 0, GOOD, None) == jl.JL_ERR_ARG
    assert jl.lib.jl_debug_status(None) == jl.JL_ERR_ARG


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    """The binding refuses to load when libjetlong.so is missing (no fallback)."""
    import importlib.util

    src = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                       "zero_shot_rope_02_b300", "binding.py")
    dst = tmp_path / "binding.py"
    dst.write_text(open(src).read())
    spec = importlib.util.spec_from_file_location("binding_copy", dst)
    mod = importlib.util.module_from_spec(spec)
    with pytest.raises(ImportError):
        spec.loader.exec_module(mod)
