"""Thin ctypes binding of ``libjetlong.so`` (argument marshalling only).

Every function keeps the name of the C entry point it wraps (declared in
``include/jetlong.h``) and takes torch tensors that already live on the GPU;
it checks dtype / shape / device, passes raw pointers and the current CUDA
stream, and raises ``JetLongError`` on a non-zero status.  No computation
happens here: every step of the path runs in the library's kernels.  If the
library is missing, importing this module fails loudly -- there is no
fallback.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libjetlong.so")

JL_OK = 0
JL_ERR_ARG = -1
JL_ERR_ALIGN = -2
JL_ERR_UNSUPPORTED = -3
JL_ERR_OVERFLOW = -4
JL_ERR_CUDA = -5
JL_ERR_TIMEOUT = -6
JL_ERR_WORKSPACE = -7
JL_ERR_GUARD = -8

# Every symbol include/jetlong.h declares.
EXPORTS = (
    "jl_status_string", "jl_version", "jl_group_factor", "jl_rope_apply", "jl_bifocal_prefill",
    "jl_bifocal_decode_workspace_size", "jl_bifocal_decode", "jl_debug_grouped_positions",
    "jl_debug_tile_classes", "jl_debug_status", "jl_bifocal_decode_noalloc",
    "jl_debug_wait_timeout", "jl_bifocal_prefill_chunk", "jl_bifocal_decode_paged",
    "jl_bifocal_decode_paged_workspace_size", "jl_rope_cache_write", "jl_group_factor_ex",
    "jl_bifocal_prefill_ex", "jl_bifocal_decode_ex",
)

# Variant flags of the _ex entry points (include/jetlong.h).
JL_VARIANT_PER_QUERY_G = 1
JL_VARIANT_SLIDING = 2
JL_VARIANT_QUERY_SHIFT = 4
# jl_bifocal_prefill_ex kernel choice: force the two-SM (cta_group::2) tile
# kernel where it applies, or force the one-CTA kernel (default: automatic)
JL_PREFILL_CTA_PAIR = 8
JL_PREFILL_ONE_CTA = 16


class JetLongError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {status_string(status)} ({status})")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libjetlong.so not built at {LIB_PATH}; run "
                          "`python -m zero_shot_rope_02_b300.build`")
    lib = ctypes.CDLL(LIB_PATH)
    i32, i64, dbl, p, sz = ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_size_t
    sig = {
        "jl_status_string": (ctypes.c_char_p, [i32]),
        "jl_version": (ctypes.c_char_p, []),
        "jl_group_factor": (i32, [i64, i64, ctypes.POINTER(ctypes.c_int32)]),
        "jl_group_factor_ex": (i32, [i64, i64, i64, ctypes.c_uint, ctypes.POINTER(ctypes.c_int32)]),
        "jl_rope_apply": (i32, [p, i32, i32, i32, i32, i64, dbl, p]),
        "jl_rope_cache_write": (i32, [p, p, p, p, i32, i32, i32, i32, i32, i32, dbl, p]),
        "jl_bifocal_prefill": (i32, [p, p, p, p, p, i32, i32, i32, i32, i32, i32, i32, dbl, p]),
        "jl_bifocal_prefill_chunk": (i32, [p, p, p, p, p, i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                           dbl, p]),
        "jl_bifocal_prefill_ex": (i32, [p, p, p, p, p, i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                        dbl, ctypes.c_uint, p]),
        "jl_bifocal_decode_ex": (i32, [p, p, p, p, p, i32, i32, i32, i32, i32, i32, i32, i32, dbl,
                                       ctypes.c_uint, p, sz, p]),
        "jl_bifocal_decode_workspace_size": (sz, [i32, i32, i32, i32, i32]),
        "jl_bifocal_decode": (i32, [p, p, p, p, p, i32, i32, i32, i32, i32, i32, i32, i32, dbl,
                                    p, sz, p]),
        "jl_bifocal_decode_noalloc": (i32, [p, p, p, p, p, i32, i32, i32, i32, i32, i32, i32, i32,
                                            dbl, p]),
        "jl_bifocal_decode_paged_workspace_size": (sz, [i32, i32, i32, i32, i32]),
        "jl_bifocal_decode_paged": (i32, [p, p, p, p, p, p, p, i32, i32, i32, i32, i32, i32, i32, i32,
                                          i32, i32, dbl, p, sz, p]),
        "jl_debug_grouped_positions": (i32, [i64, i64, p, p]),
        "jl_debug_tile_classes": (i32, [i32, i32, i32, p, p]),
        "jl_debug_status": (i32, [ctypes.POINTER(ctypes.c_int)]),
        "jl_debug_wait_timeout": (i32, [i64, p, p]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


def status_string(status: int) -> str:
    return lib.jl_status_string(int(status)).decode()


def jl_version() -> str:
    return lib.jl_version().decode()


def _check(fn: str, rc: int):
    if rc != JL_OK:
        raise JetLongError(fn, rc)


def _stream(stream=None):
    import torch

    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(t.data_ptr())


def _need(t, dtype, name):
    import torch

    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def jl_group_factor(s: int, L_pre: int) -> int:
    """g(s, L_pre) = max(1, ceil(s / L_pre)) from the library (host only)."""
    g = ctypes.c_int32(0)
    _check("jl_group_factor", lib.jl_group_factor(int(s), int(L_pre), ctypes.byref(g)))
    return int(g.value)


def jl_group_factor_ex(s: int, L_pre: int, w: int, flags: int) -> int:
    """Group factor under variant flags (the query-shift rule with
    JL_VARIANT_QUERY_SHIFT) from the library (host only)."""
    g = ctypes.c_int32(0)
    _check("jl_group_factor_ex", lib.jl_group_factor_ex(int(s), int(L_pre), int(w), int(flags),
                                                        ctypes.byref(g)))
    return int(g.value)


def jl_rope_apply(x, pos0: int, theta: float, stream=None):
    """Exact RoPE in place on bf16 x [B, S, H, D] at positions pos0 + s."""
    import torch

    _need(x, torch.bfloat16, "x")
    B, S, H, D = x.shape
    _check("jl_rope_apply", lib.jl_rope_apply(_ptr(x), B, S, H, D, int(pos0), float(theta),
                                              _stream(stream)))
    return x


def jl_rope_cache_write(k_raw, v, k_cache, v_cache, n_past: int, theta: float, stream=None):
    """RoPE fused into the cache write: k_raw / v [B,S_new,H,D] (k before RoPE)
    into cache rows n_past.. of k_cache / v_cache [B,n_cap,H,D], k rotated."""
    import torch

    for t, nm in ((k_raw, "k_raw"), (v, "v"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, nm)
    B, S_new, H, D = k_raw.shape
    n_cap = k_cache.shape[1]
    if v.shape != k_raw.shape or v_cache.shape != k_cache.shape or k_cache.shape[0] != B or \
            k_cache.shape[2:] != (H, D):
        raise ValueError("k_raw / v [B,S_new,H,D] and caches [B,n_cap,H,D]")
    _check("jl_rope_cache_write",
           lib.jl_rope_cache_write(_ptr(k_raw), _ptr(v), _ptr(k_cache), _ptr(v_cache), B, S_new, H, D,
                                   int(n_past), n_cap, float(theta), _stream(stream)))
    return k_cache, v_cache


def jl_bifocal_prefill(q, k, v, L_pre: int, w: int, theta: float, out=None, lse=None,
                       stream=None):
    """Bifocal causal GQA prefill.  q [B,S,Hq,D], k/v [B,S,Hkv,D] bf16 (exact RoPE).
    Returns (out bf16 [B,S,Hq,D], lse fp32 [B,Hq,S])."""
    import torch

    for t, nm in ((q, "q"), (k, "k"), (v, "v")):
        _need(t, torch.bfloat16, nm)
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    if k.shape != (B, S, Hkv, D) or v.shape != k.shape:
        raise ValueError("k and v must be [B, S, Hkv, D] matching q")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, S), dtype=torch.float32, device=q.device)
    _need(out, torch.bfloat16, "out")
    _need(lse, torch.float32, "lse")
    _check("jl_bifocal_prefill",
           lib.jl_bifocal_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, Hq, Hkv, S, D,
                                  int(L_pre), int(w), float(theta), _stream(stream)))
    return out, lse


def jl_bifocal_prefill_chunk(q, k_cache, v_cache, n_past: int, L_pre: int, w: int, theta: float,
                             out=None, lse=None, stream=None):
    """Bifocal prefill of S_new tokens at positions n_past..n_past+S_new-1 over
    the cache.  q [B,S_new,Hq,D]; caches [B,n_cap,Hkv,D] bf16 (exact RoPE),
    rows 0..n_past+S_new-1 valid.  Returns (out bf16 [B,S_new,Hq,D],
    lse fp32 [B,Hq,S_new])."""
    import torch

    for t, nm in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, nm)
    B, S_new, Hq, D = q.shape
    _, n_cap, Hkv, Dk = k_cache.shape
    if Dk != D or v_cache.shape != k_cache.shape or k_cache.shape[0] != B:
        raise ValueError("caches must be [B, n_cap, Hkv, D] matching q")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, S_new), dtype=torch.float32, device=q.device)
    _need(out, torch.bfloat16, "out")
    _need(lse, torch.float32, "lse")
    _check("jl_bifocal_prefill_chunk",
           lib.jl_bifocal_prefill_chunk(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(lse), B,
                                        Hq, Hkv, S_new, int(n_past), n_cap, D, int(L_pre), int(w),
                                        float(theta), _stream(stream)))
    return out, lse


def jl_bifocal_prefill_ex(q, k_cache, v_cache, n_past: int, L_pre: int, w: int, theta: float, flags: int,
                          out=None, lse=None, stream=None):
    """Bifocal prefill with variant flags (JL_VARIANT_*) of S_new tokens at
    positions n_past.. over the cache.  q [B,S_new,Hq,D]; caches [B,n_cap,Hkv,D]
    bf16 (exact RoPE), rows 0..n_past+S_new-1 valid.  Returns (out, lse)."""
    import torch

    for t, nm in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, nm)
    B, S_new, Hq, D = q.shape
    _, n_cap, Hkv, Dk = k_cache.shape
    if Dk != D or v_cache.shape != k_cache.shape or k_cache.shape[0] != B:
        raise ValueError("caches must be [B, n_cap, Hkv, D] matching q")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq, S_new), dtype=torch.float32, device=q.device)
    _need(out, torch.bfloat16, "out")
    _need(lse, torch.float32, "lse")
    _check("jl_bifocal_prefill_ex",
           lib.jl_bifocal_prefill_ex(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(lse), B, Hq, Hkv,
                                     S_new, int(n_past), n_cap, D, int(L_pre), int(w), float(theta),
                                     int(flags), _stream(stream)))
    return out, lse


def jl_bifocal_decode_ex(q, k_cache, v_cache, n: int, L_pre: int, w: int, theta: float, flags: int,
                         workspace=None, out=None, lse=None, stream=None):
    """jl_bifocal_decode with variant flags (JL_VARIANT_*).  Same arguments and
    workspace as jl_bifocal_decode.  Returns (out bf16 [B,Hq,D], lse fp32 [B,Hq])."""
    import torch

    for t, nm in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, nm)
    B, Hq, D = q.shape
    _, n_cap, Hkv, Dk = k_cache.shape
    if Dk != D or v_cache.shape != k_cache.shape or k_cache.shape[0] != B:
        raise ValueError("caches must be [B, n_cap, Hkv, D] matching q")
    if workspace is None:
        nbytes = jl_bifocal_decode_workspace_size(B, Hq, Hkv, n, D)
        workspace = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    _need(out, torch.bfloat16, "out")
    _need(lse, torch.float32, "lse")
    _check("jl_bifocal_decode_ex",
           lib.jl_bifocal_decode_ex(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(lse), B, Hq, Hkv,
                                    int(n), n_cap, D, int(L_pre), int(w), float(theta), int(flags),
                                    _ptr(workspace), workspace.numel() * workspace.element_size(),
                                    _stream(stream)))
    return out, lse


def jl_bifocal_decode_paged_workspace_size(B: int, Hq: int, Hkv: int, max_n: int, D: int) -> int:
    return int(lib.jl_bifocal_decode_paged_workspace_size(B, Hq, Hkv, max_n, D))


def jl_bifocal_decode_workspace_size(B: int, Hq: int, Hkv: int, n: int, D: int) -> int:
    return int(lib.jl_bifocal_decode_workspace_size(B, Hq, Hkv, n, D))


def jl_bifocal_decode(q, k_cache, v_cache, n: int, L_pre: int, w: int, theta: float,
                      workspace=None, out=None, lse=None, stream=None):
    """Bifocal decode of one token at position n-1.  q [B,Hq,D]; caches
    [B,n_cap,Hkv,D] bf16 (exact RoPE), rows 0..n-1 valid.  ``workspace`` is a
    uint8 CUDA tensor of at least jl_bifocal_decode_workspace_size() bytes whose
    counters start at zero (torch.zeros); allocated here if None.
    Returns (out bf16 [B,Hq,D], lse fp32 [B,Hq])."""
    import torch

    for t, nm in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, nm)
    B, Hq, D = q.shape
    _, n_cap, Hkv, Dk = k_cache.shape
    if Dk != D or v_cache.shape != k_cache.shape or k_cache.shape[0] != B:
        raise ValueError("caches must be [B, n_cap, Hkv, D] matching q")
    if workspace is None:
        nbytes = jl_bifocal_decode_workspace_size(B, Hq, Hkv, n, D)
        workspace = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    _need(out, torch.bfloat16, "out")
    _need(lse, torch.float32, "lse")
    _check("jl_bifocal_decode",
           lib.jl_bifocal_decode(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(lse), B, Hq,
                                 Hkv, int(n), n_cap, D, int(L_pre), int(w), float(theta),
                                 _ptr(workspace), workspace.numel() * workspace.element_size(),
                                 _stream(stream)))
    return out, lse


def jl_bifocal_decode_paged(q, k_pages, v_pages, block_table, seq_lens, max_n: int, L_pre: int, w: int,
                            theta: float, workspace=None, out=None, lse=None, stream=None):
    """Bifocal decode of B sequences of their own lengths over a paged cache.
    q [B,Hq,D]; pages [num_pages,page_size,Hkv,D] bf16 (exact RoPE);
    block_table int32 [B,max_pages] and seq_lens int32 [B] on the device;
    max_n >= every length.  ``workspace`` as for jl_bifocal_decode (sized for
    max_n).  Returns (out bf16 [B,Hq,D], lse fp32 [B,Hq])."""
    import torch

    for t, nm in ((q, "q"), (k_pages, "k_pages"), (v_pages, "v_pages")):
        _need(t, torch.bfloat16, nm)
    _need(block_table, torch.int32, "block_table")
    _need(seq_lens, torch.int32, "seq_lens")
    B, Hq, D = q.shape
    num_pages, page_size, Hkv, Dk = k_pages.shape
    max_pages = block_table.shape[1]
    if Dk != D or v_pages.shape != k_pages.shape or block_table.shape[0] != B or seq_lens.shape != (B,):
        raise ValueError("pages [P, page_size, Hkv, D], block_table [B, max_pages], seq_lens [B]")
    if workspace is None:
        nbytes = jl_bifocal_decode_paged_workspace_size(B, Hq, Hkv, max_n, D)
        workspace = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    _need(out, torch.bfloat16, "out")
    _need(lse, torch.float32, "lse")
    _check("jl_bifocal_decode_paged",
           lib.jl_bifocal_decode_paged(_ptr(q), _ptr(k_pages), _ptr(v_pages), _ptr(block_table),
                                       _ptr(seq_lens), _ptr(out), _ptr(lse), B, Hq, Hkv, D, page_size,
                                       num_pages, max_pages, int(max_n), int(L_pre), int(w), float(theta),
                                       _ptr(workspace), workspace.numel() * workspace.element_size(),
                                       _stream(stream)))
    return out, lse


def jl_bifocal_decode_noalloc(q, k_cache, v_cache, n: int, L_pre: int, w: int, theta: float,
                              out=None, lse=None, stream=None):
    """jl_bifocal_decode with the library's fixed device scratch instead of a
    workspace (for callers that cannot allocate device memory).  Calls whose
    executions overlap on the GPU share that scratch and race."""
    import torch

    for t, nm in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _need(t, torch.bfloat16, nm)
    B, Hq, D = q.shape
    _, n_cap, Hkv, Dk = k_cache.shape
    if Dk != D or v_cache.shape != k_cache.shape or k_cache.shape[0] != B:
        raise ValueError("caches must be [B, n_cap, Hkv, D] matching q")
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, Hq), dtype=torch.float32, device=q.device)
    _need(out, torch.bfloat16, "out")
    _need(lse, torch.float32, "lse")
    _check("jl_bifocal_decode_noalloc",
           lib.jl_bifocal_decode_noalloc(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(lse), B,
                                         Hq, Hkv, int(n), n_cap, D, int(L_pre), int(w), float(theta),
                                         _stream(stream)))
    return out, lse


def jl_debug_grouped_positions(S: int, L_pre: int, stream=None):
    import torch

    out = torch.empty(S, dtype=torch.int32, device="cuda")
    _check("jl_debug_grouped_positions",
           lib.jl_debug_grouped_positions(int(S), int(L_pre), _ptr(out), _stream(stream)))
    return out


def jl_debug_tile_classes(S: int, L_pre: int, w: int, stream=None):
    import torch

    nt = (S + 127) // 128
    out = torch.empty((nt, nt), dtype=torch.int8, device="cuda")
    _check("jl_debug_tile_classes",
           lib.jl_debug_tile_classes(int(S), int(L_pre), int(w), _ptr(out), _stream(stream)))
    return out


def jl_debug_wait_timeout(limit_ns: int, stream=None) -> int:
    """Run the bounded-wait failure probe; returns 1 if the wait gave up."""
    import torch

    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    _check("jl_debug_wait_timeout", lib.jl_debug_wait_timeout(int(limit_ns), _ptr(flag), _stream(stream)))
    return int(flag.item())


def jl_debug_status() -> int:
    """Read and clear the device status word (synchronises the device)."""
    st = ctypes.c_int(0)
    _check("jl_debug_status", lib.jl_debug_status(ctypes.byref(st)))
    return int(st.value)
