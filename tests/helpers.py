"""Shared test helpers: seeded inputs on both sides and the parity metrics.

Inputs come from ``zero_shot_rope_02_b300.inputs`` (counter-based generator,
no attention arithmetic), so the CUDA path and the oracle see the same bf16
bits; the oracle receives them widened exactly to fp64.
"""
from __future__ import annotations

import numpy as np

from zero_shot_rope_02_b300 import inputs

# Tolerances the parity tests hold the GPU path to (bf16 outputs, fp32 lse).
OUT_MAX_ABS = 1e-2
OUT_MEAN_ABS = 1e-3
LSE_REL = 1e-4


def bf16_pair(shape, seed, tensor_id, scale=1.0):
    """(torch bf16 CPU tensor, exact fp64 numpy copy) of a seeded N(0, scale^2)
    tensor; ``scale`` must be a power of two so the scaling is exact."""
    bits = inputs.normal_bf16_bits(shape, seed, tensor_id)
    f64 = inputs.bf16_bits_to_f64(bits)
    t = inputs.to_torch_bf16(bits)
    if scale != 1.0:
        assert float(scale).hex().startswith(("0x1.0000000000000p", "0x1p")), "scale must be 2^k"
        t = t * scale
        f64 = f64 * scale
    return t, f64


def bf16_to_f64(t) -> np.ndarray:
    """Exact widening of a (CPU or CUDA) torch bf16 tensor to fp64 numpy."""
    import torch

    return t.detach().to("cpu").to(torch.float64).numpy()


def compare(out_gpu, lse_gpu, out_ref, lse_ref, what=""):
    """Assert the parity bar: bf16 out max|d| <= 1e-2 and mean|d| <= 1e-3,
    fp32 lse relative error <= 1e-4, taken against max(|lse|, 1) so rows whose
    log-sum-exp crosses zero are held to 1e-4 absolutely.  Returns the
    measured errors."""
    d = np.abs(np.asarray(out_gpu, dtype=np.float64) - out_ref)
    mean = float(d.mean())
    mx = float(d.max())
    lse_gpu = np.asarray(lse_gpu, dtype=np.float64)
    dl = np.abs(lse_gpu - lse_ref)
    rel = float(np.max(dl / np.maximum(np.abs(lse_ref), 1.0)))
    assert np.all(np.isfinite(out_gpu)), f"{what}: non-finite output"
    assert mx <= OUT_MAX_ABS, f"{what}: out max abs err {mx:.3e}"
    assert mean <= OUT_MEAN_ABS, f"{what}: out mean abs err {mean:.3e}"
    assert rel <= LSE_REL, f"{what}: lse rel err {rel:.3e}"
    return mx, mean, rel


def sample_rows(S, L, w, g, n_random=64, seed=0):
    """Query rows checked at full size: the edges of every rule the method
    has (window, group, pretrained window, tiles) plus seeded random rows."""
    rows = {0, 1, 127, 128, S // 2, S - 1, S - 2}
    for r in (g - 1, g, g + 1, 2 * g - 1, 2 * g, w - 1, w, w + 1, L - 1, L, L + 1, S - 129, S - 128):
        rows.add(r)
    rng = np.random.default_rng(seed)
    rows.update(int(x) for x in rng.integers(0, S, n_random))
    return np.array(sorted(r for r in rows if 0 <= r < S), dtype=np.int64)
