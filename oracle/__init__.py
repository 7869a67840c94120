"""fp64 CPU oracle for Dynamic Bifocal RoPE attention.

TEST INFRASTRUCTURE ONLY.  Imported by the tests, by the smoke check and by
the benchmark's CPU-baseline leg, never by the product library.  The heavy
lifting is the plain C in ``oracle.c`` (OpenMP over query rows); this module
compiles it with gcc, loads it with ctypes and converts numpy arrays.

What it computes is stated in the header of ``oracle.c``: the single masked
pass (each key scored once with the view its distance selects) and, as an
independent second statement, the three-pass inclusion-exclusion merge that
the Jet-Long abstract and the researchpod.app summary describe.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")


def compile_oracle(src: str, out: str) -> str:
    """gcc -O2 -fopenmp: ``src`` (C file) -> shared library ``out``."""
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` next to it."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(SOURCE):
        compile_oracle(SOURCE, _LIB)
    return _LIB


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


class Oracle:
    """ctypes view of one build of ``oracle.c``."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        i64, dbl, p = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
        lib.oracle_group_factor.restype = i64
        lib.oracle_group_factor.argtypes = [i64, i64]
        lib.oracle_grouped_position.restype = i64
        lib.oracle_grouped_position.argtypes = [i64, i64]
        lib.oracle_rope.restype = None
        lib.oracle_rope.argtypes = [p, p, i64, i64, i64, i64, i64, dbl]
        sig = [p, p, p, i64, i64, i64, i64, i64, i64, p, i64, i64, i64, dbl, p, p]
        for name in ("oracle_bifocal_rows", "oracle_bifocal_rows_3pass"):
            fn = getattr(lib, name)
            fn.restype = ctypes.c_int
            fn.argtypes = sig
        lib.oracle_bifocal_rows_ex.restype = ctypes.c_int
        lib.oracle_bifocal_rows_ex.argtypes = sig[:14] + [i64] + sig[14:]
        lib.oracle_group_factor_shift.restype = i64
        lib.oracle_group_factor_shift.argtypes = [i64, i64, i64]
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_num_threads.argtypes = []
        self.lib = lib
        self.path = lib_path

    def group_factor(self, s: int, L: int) -> int:
        """Smallest integer g >= 1 with floor((s-1)/g) <= L-1 (literal search)."""
        return int(self.lib.oracle_group_factor(int(s), int(L)))

    def grouped_position(self, p: int, g: int) -> int:
        """Aliased position floor(p/g)."""
        return int(self.lib.oracle_grouped_position(int(p), int(g)))

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def rope(self, x, pos0: int, theta: float) -> np.ndarray:
        """Exact RoPE of x [B,S,H,D] at positions pos0+s, fp64."""
        x = _f64(x)
        B, S, H, D = x.shape
        out = np.empty_like(x)
        self.lib.oracle_rope(_ptr(x), _ptr(out), B, S, H, D, int(pos0), float(theta))
        return out

    def _attn(self, fn_name, q, k, v, qpos, s_len, L, w, theta):
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, Sq, Hq, D = q.shape
        Bk, Sk, Hkv, Dk = k.shape
        assert Bk == B and Dk == D and v.shape == k.shape
        qpos = np.ascontiguousarray(np.asarray(qpos, dtype=np.int64))
        assert qpos.shape == (Sq,)
        out = np.empty((B, Sq, Hq, D), dtype=np.float64)
        lse = np.empty((B, Hq, Sq), dtype=np.float64)
        rc = getattr(self.lib, fn_name)(_ptr(q), _ptr(k), _ptr(v), B, Sq, Hq, Hkv, Sk, D,
                                        _ptr(qpos), int(s_len), int(L), int(w), float(theta),
                                        _ptr(out), _ptr(lse))
        if rc != 0:
            raise ValueError(f"{fn_name}: invalid arguments")
        return out, lse

    def bifocal_rows(self, q, k, v, qpos, s_len, L, w, theta):
        """Single masked pass.  q [B,Sq,Hq,D] at positions qpos, k/v [B,Sk,Hkv,D]
        at positions 0..Sk-1.  Returns (out [B,Sq,Hq,D], lse [B,Hq,Sq]) in fp64."""
        return self._attn("oracle_bifocal_rows", q, k, v, qpos, s_len, L, w, theta)

    def bifocal_rows_3pass(self, q, k, v, qpos, s_len, L, w, theta):
        """Three passes merged by inclusion-exclusion; same contract as bifocal_rows."""
        return self._attn("oracle_bifocal_rows_3pass", q, k, v, qpos, s_len, L, w, theta)

    def group_factor_shift(self, s: int, L: int, w: int) -> int:
        """Smallest g with floor((s-1)/g) + w - floor(w/g) <= L-1 (query-shift
        variant; literal search), -1 if none."""
        return int(self.lib.oracle_group_factor_shift(int(s), int(L), int(w)))

    def bifocal_rows_ex(self, q, k, v, qpos, s_len, L, w, theta, flags):
        """bifocal_rows with variant flags (PER_QUERY_G | SLIDING | QUERY_SHIFT)."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, Sq, Hq, D = q.shape
        Bk, Sk, Hkv, Dk = k.shape
        assert Bk == B and Dk == D and v.shape == k.shape
        qpos = np.ascontiguousarray(np.asarray(qpos, dtype=np.int64))
        assert qpos.shape == (Sq,)
        out = np.empty((B, Sq, Hq, D), dtype=np.float64)
        lse = np.empty((B, Hq, Sq), dtype=np.float64)
        rc = self.lib.oracle_bifocal_rows_ex(_ptr(q), _ptr(k), _ptr(v), B, Sq, Hq, Hkv, Sk, D, _ptr(qpos),
                                             int(s_len), int(L), int(w), float(theta), int(flags),
                                             _ptr(out), _ptr(lse))
        if rc != 0:
            raise ValueError("oracle_bifocal_rows_ex: invalid arguments")
        return out, lse

    def bifocal_prefill_ex(self, q, k, v, L, w, theta, flags):
        """Full causal prefill with variant flags."""
        S = q.shape[1]
        return self.bifocal_rows_ex(q, k, v, np.arange(S), S, L, w, theta, flags)

    def bifocal_prefill(self, q, k, v, L, w, theta):
        """Full causal prefill: every row of q [B,S,Hq,D], s = S."""
        S = q.shape[1]
        return self.bifocal_rows(q, k, v, np.arange(S), S, L, w, theta)

    def bifocal_decode(self, q, k_cache, v_cache, L, w, theta):
        """One query token q [B,1,Hq,D] at position n-1 over a cache of n keys."""
        n = k_cache.shape[1]
        return self.bifocal_rows(q, k_cache, v_cache, np.array([n - 1]), n, L, w, theta)


# Variant flags of bifocal_rows_ex (values shared with oracle.c's ORACLE_* macros).
PER_QUERY_G = 1
SLIDING = 2
QUERY_SHIFT = 4

_default = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = Oracle(build())
    return _default


def group_factor(s, L):
    return default().group_factor(s, L)


def grouped_position(p, g):
    return default().grouped_position(p, g)


def num_threads():
    return default().num_threads()


def rope(x, pos0, theta):
    return default().rope(x, pos0, theta)


def bifocal_rows(q, k, v, qpos, s_len, L, w, theta):
    return default().bifocal_rows(q, k, v, qpos, s_len, L, w, theta)


def bifocal_rows_3pass(q, k, v, qpos, s_len, L, w, theta):
    return default().bifocal_rows_3pass(q, k, v, qpos, s_len, L, w, theta)


def bifocal_prefill(q, k, v, L, w, theta):
    return default().bifocal_prefill(q, k, v, L, w, theta)


def bifocal_decode(q, k_cache, v_cache, L, w, theta):
    return default().bifocal_decode(q, k_cache, v_cache, L, w, theta)
