"""Seeded synthetic inputs, shared by the tests, the smoke check and the bench.

This module holds no attention or RoPE arithmetic: it only draws numbers.
Element e of tensor ``tensor_id`` under ``seed`` is a standard normal made
from two counter-based uniforms (SplitMix64 finaliser, Steele/Lea/Flood
"Fast splittable pseudorandom number generators", 2014) by the Box-Muller
transform in fp64, then rounded to fp32 and to bf16 (round to nearest even).
Both the oracle and the GPU therefore see bit-identical values.

Tensor ids used across the repo: q=0, k=1, v=2 (prefill) and 3, 4, 5 (decode
q, k_cache, v_cache).
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, tensor_id: int) -> np.uint64:
    with np.errstate(over="ignore"):
        k = np.array([(seed & 0xFFFFFFFF) << 32 | (tensor_id & 0xFFFFFFFF)], dtype=np.uint64)
        return _mix(k * _GOLDEN + _GOLDEN)[0]


def _uniform(bits: np.ndarray) -> np.ndarray:
    # 53 random bits -> (0, 1), never 0
    return ((bits >> np.uint64(11)).astype(np.float64) + 0.5) * (1.0 / 9007199254740992.0)


def _normal_chunk(key: np.uint64, start: int, count: int) -> np.ndarray:
    with np.errstate(over="ignore"):
        e = np.arange(start, start + count, dtype=np.uint64)
        c0 = key + (np.uint64(2) * e + np.uint64(1)) * _GOLDEN
        c1 = key + (np.uint64(2) * e + np.uint64(2)) * _GOLDEN
        u1 = _uniform(_mix(c0))
        u2 = _uniform(_mix(c1))
    return np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)


def fp32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    with np.errstate(over="ignore"):
        r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp64."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def normal_bf16_bits(shape, seed: int, tensor_id: int, chunk: int = 1 << 22) -> np.ndarray:
    """Seeded N(0,1) tensor of ``shape`` as bf16 bit patterns (uint16)."""
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16)
    key = _key(seed, tensor_id)

    def work(start):
        cnt = min(chunk, n - start)
        out[start:start + cnt] = fp32_to_bf16_bits(_normal_chunk(key, start, cnt).astype(np.float32))

    starts = list(range(0, n, chunk))
    if len(starts) <= 1:
        for s in starts:
            work(s)
    else:
        with ThreadPoolExecutor(max_workers=min(len(starts), os.cpu_count() or 1)) as ex:
            list(ex.map(work, starts))
    return out.reshape(shape)


def normal_f64(shape, seed: int, tensor_id: int) -> np.ndarray:
    """Seeded N(0,1) fp64 tensor (not rounded), for oracle-only pins."""
    n = int(np.prod(shape))
    return _normal_chunk(_key(seed, tensor_id), 0, n).reshape(shape)


def to_torch_bf16(bits: np.ndarray):
    """View uint16 bf16 bit patterns as a CPU torch.bfloat16 tensor (no copy)."""
    import torch

    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
