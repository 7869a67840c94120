"""jl_bifocal_decode_noalloc: decode for callers that cannot allocate device
memory (it runs on a fixed scratch array inside the library instead of a
caller workspace).  Called through the C ABI and held to the same tolerance
as the other parity tests against the workspace entry point, on two calls in
a row -- the second call finds the scratch holding the first call's data.

This file is named to be collected last, so that a run stopping at the first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest

import helpers

pytestmark = pytest.mark.gpu


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(jl, q, k, v, out, lse, n, L, w, theta):
    import torch

    B, Hq, D = q.shape
    _, n_cap, Hkv, _ = k.shape
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return jl.lib.jl_bifocal_decode_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq,
                                            Hkv, n, n_cap, D, L, w, theta, stream)


@pytest.mark.parametrize("B,Hq,Hkv,n,n_cap,D,L,w", [
    (1, 32, 8, 20000, 20000, 128, 4096, 1024),    # g = 5: remote keys corrected
    (1, 32, 8, 131072, 131072, 128, 32768, 4096),  # the benchmark decode at 128K
    (2, 8, 2, 3000, 3100, 64, 4096, 64),           # g = 1, capacity > n
])
def test_noalloc_matches_workspace_decode_twice(jl, dev, B, Hq, Hkv, n, n_cap, D, L, w):
    import torch

    theta = 1e6
    q, _ = helpers.bf16_pair((B, Hq, D), 11, 3)
    k, _ = helpers.bf16_pair((B, n_cap, Hkv, D), 11, 4)
    v, _ = helpers.bf16_pair((B, n_cap, Hkv, D), 11, 5)
    q, k, v = q.to(dev), k.to(dev), v.to(dev)
    ref_out, ref_lse = jl.jl_bifocal_decode(q, k, v, n, L, w, theta)
    torch.cuda.synchronize()
    ref_o = helpers.bf16_to_f64(ref_out)
    ref_l = ref_lse.cpu().numpy().astype(np.float64)
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        lse = torch.full((B, Hq), float("nan"), dtype=torch.float32, device=dev)
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info(dev)[0]
        rc = _noalloc(jl, q, k, v, out, lse, n, L, w, theta)
        assert rc == 0, jl.status_string(rc)
        torch.cuda.synchronize()
        if call == 1:
            # the first call may load the library's module onto the device and
            # look up the scratch address; after that a call takes no device memory
            assert torch.cuda.mem_get_info(dev)[0] == free_before
        helpers.compare(helpers.bf16_to_f64(out), lse.cpu().numpy(), ref_o, ref_l,
                        f"no-alloc decode call {call} n={n}")
    assert jl.jl_debug_status() == 0


def test_noalloc_rejects_shapes_beyond_its_scratch(jl, dev):
    """Split partials above the fixed scratch size are refused before any launch."""
    import torch

    B, Hq, Hkv, n, D = 64, 512, 64, 131072, 128  # 4096 (batch, kv head) units
    assert jl.jl_bifocal_decode_workspace_size(B, Hq, Hkv, n, D) > (8 << 20)
    q = torch.zeros((B, Hq, D), dtype=torch.bfloat16, device=dev)
    kv = torch.zeros((B, 16, Hkv, D), dtype=torch.bfloat16, device=dev)  # never read
    out = torch.empty_like(q)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = jl.lib.jl_bifocal_decode_noalloc(_ptr(q), _ptr(kv), _ptr(kv), _ptr(out), _ptr(lse), B, Hq,
                                          Hkv, n, n, D, 32768, 4096, 1e6, stream)
    assert rc == jl.JL_ERR_WORKSPACE


def test_noalloc_rejects_unsupported_and_misaligned_arguments(jl, dev):
    """Argument errors the workspace entry point reports (an unsupported GQA
    group size, a misaligned cache pointer) are reported by this one too; the
    checks run before the scratch is cleared."""
    import torch

    B, Hq, Hkv, n, D = 1, 12, 4, 1000, 128  # Hq / Hkv = 3: no kernel for that group size
    q = torch.zeros((B, Hq, D), dtype=torch.bfloat16, device=dev)
    kv = torch.zeros((B, n, Hkv, D), dtype=torch.bfloat16, device=dev)
    out = torch.empty_like(q)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = jl.lib.jl_bifocal_decode_noalloc(_ptr(q), _ptr(kv), _ptr(kv), _ptr(out), _ptr(lse), B, Hq,
                                          Hkv, n, n, D, 512, 64, 1e6, stream)
    assert rc == jl.JL_ERR_UNSUPPORTED
    mis = ctypes.c_void_p(kv.data_ptr() + 2)
    rc = jl.lib.jl_bifocal_decode_noalloc(_ptr(q), mis, _ptr(kv), _ptr(out), _ptr(lse), B, 8, 4, n, n,
                                          D, 512, 64, 1e6, stream)
    assert rc == jl.JL_ERR_ALIGN
