"""ctypes binding of libtiled_attn.so (include/attn.h), with the same entry-point names.

Only argument marshalling happens here: torch tensors are passed as raw device pointers and
the current CUDA stream. Every step of the computation runs in the library's kernels. There is
no fallback: if the library is missing, every call raises.
"""
from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_lib", "libtiled_attn.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "attn.h")

ATTN_MASK_NONE = 0
ATTN_MASK_CAUSAL = 1
ATTN_MASK_SLIDING = 2
ATTN_MASK_DOCUMENT = 3
ATTN_MASK_PAGED_DECODE = 4
ATTN_MASK_DECODE = 5
ATTN_MASK_SLIDING_BIDIR = 6
ATTN_MASK_DOCUMENT_BIDIR = 7
ATTN_MASK_PREFIX_LM = 8
ATTN_MASK_PAGED_PREFILL = 9

ATTN_OK = 0
ATTN_ERR_INVALID = -1
ATTN_ERR_UNSUPPORTED = -2
ATTN_ERR_CUDA = -3
ATTN_ERR_TIMEOUT = -4
ATTN_ERR_BOUNDS = -5
ATTN_ERR_WORKSPACE = -6
ATTN_ERR_SEQLENS = -7

_lib = None

_p = ctypes.c_void_p
_i = ctypes.c_int
_SIGS = {
    "attn_fwd": (_i, [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, ctypes.c_float, _i, _i, _p, _p, _i,
                      _i, _p, ctypes.c_size_t, _p]),
    "attn_fwd_paged_prefill": (_i, [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, ctypes.c_float, _p,
                                    _p, _p, _i, _i, _i, _p]),
    "attn_quantize_fp8": (_i, [_p, _p, _p, _i, _i, _i, _p]),
    "attn_fwd_fp8": (_i, [_p, _p, _p, _p, _p, _p, _p, _i, _i, _i, _i, _i, ctypes.c_float, _i, _i,
                          _p]),
    "attn_workspace_bytes": (ctypes.c_size_t, [_i, _i, _i, _i, _i, _i, _i]),
    "attn_gather_pages": (_i, [_p, _p, _p, _i, _i, _i, _i, _i, _i, _p]),
    "attn_get_status": (_i, [_p]),
    "attn_last_error": (ctypes.c_char_p, []),
    "attn_release": (None, []),
    "attn_version": (_i, []),
    "attn_plan_kv_range": (_i, [_i, _i, _i, _i, _i, _i, _i, _i, ctypes.POINTER(_i),
                                ctypes.POINTER(_i)]),
    "attn_plan_tile_kind": (_i, [_i, _i, _i, _i, _i, _i, _i, _i, _i]),
    "attn_plan_units": (_i, [_i, _i, _i, _i, _p, _p, _i]),
    "attn_selftest_wait_timeout": (_i, [ctypes.c_ulonglong, _p]),
    "attn_paged_decode_noalloc": (_i, [_p, _p, _p, _p, _p, _i, _i, _i, _i, _i, ctypes.c_float,
                                       _p, _p, _i, _i, _p]),
    "attn_bench_ex2": (_i, [_p, _i, _i, _p]),
    "attn_noalloc_scratch_bytes": (ctypes.c_size_t, []),
    "attn_cached_device_state": (_i, [_i]),
}


class AttnError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"attn error {code}: {msg}")
        self.code = code


def lib():
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m tiled_attention_gb300.build` (needs nvcc)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def declared_functions():
    """Function names declared in include/attn.h."""
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z_0-9]+)\s*\(", text)))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def last_error() -> str:
    return lib().attn_last_error().decode()


def check(code: int) -> int:
    if code != ATTN_OK:
        raise AttnError(code, last_error())
    return code


def attn_fwd(q, k, v, o, lse, B, Hq, Hkv, N, d, scale, mask_kind, window=0, cu_seqlens=None,
             block_table=None, page_size=0, num_pages=0, workspace=None, stream=None) -> int:
    """Call attn_fwd with torch tensors (device memory); returns the ABI code."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return lib().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, N, d,
                          ctypes.c_float(scale), mask_kind, window, _ptr(cu_seqlens),
                          _ptr(block_table), page_size, num_pages, _ptr(workspace), ws_bytes,
                          _stream(stream))


def attn_fwd_paged_prefill(q, k, v, o, lse, B, Hq, Hkv, total_q, d, scale, cu_seqlens_q,
                           seqlens_k, block_table, max_pages, page_size, num_pages,
                           stream=None) -> int:
    """Chunked prefill over a paged KV cache (torch tensors in device memory)."""
    return lib().attn_fwd_paged_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq,
                                        Hkv, total_q, d, ctypes.c_float(scale),
                                        _ptr(cu_seqlens_q), _ptr(seqlens_k), _ptr(block_table),
                                        max_pages, page_size, num_pages, _stream(stream))


def attn_quantize_fp8(x, x8, scales, planes, N, d, stream=None) -> int:
    """E4M3 block quantization of a bf16 tensor [planes, N, d] (torch tensors on the device)."""
    return lib().attn_quantize_fp8(_ptr(x), _ptr(x8), _ptr(scales), planes, N, d,
                                   _stream(stream))


def attn_fwd_fp8(q8, k8, v, o, lse, q_scales, k_scales, B, Hq, Hkv, N, d, scale, mask_kind,
                 window=0, stream=None) -> int:
    """Attention with E4M3 Q / K and per-128-row-tile scales (torch tensors on the device)."""
    return lib().attn_fwd_fp8(_ptr(q8), _ptr(k8), _ptr(v), _ptr(o), _ptr(lse), _ptr(q_scales),
                              _ptr(k_scales), B, Hq, Hkv, N, d, ctypes.c_float(scale),
                              mask_kind, window, _stream(stream))


def attn_paged_decode_noalloc(q, k, v, o, lse, B, Hq, Hkv, N, d, scale, cu_seqlens, block_table,
                              page_size, num_pages, stream=None) -> int:
    """Paged decode without a workspace argument (the library's fixed scratch is used)."""
    return lib().attn_paged_decode_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq,
                                           Hkv, N, d, ctypes.c_float(scale), _ptr(cu_seqlens),
                                           _ptr(block_table), page_size, num_pages,
                                           _stream(stream))


def attn_workspace_bytes(B, Hq, Hkv, N, d, mask_kind, page_size=0) -> int:
    return lib().attn_workspace_bytes(B, Hq, Hkv, N, d, mask_kind, page_size)


def attn_gather_pages(pool, dst, block_table, B, max_pages, Hkv, page_size, d, num_pages,
                      stream=None) -> int:
    return lib().attn_gather_pages(_ptr(pool), _ptr(dst), _ptr(block_table), B, max_pages, Hkv,
                                   page_size, d, num_pages, _stream(stream))


def attn_selftest_wait_timeout(timeout_ns: int, stream=None) -> int:
    return lib().attn_selftest_wait_timeout(timeout_ns, _stream(stream))


def attn_bench_ex2(out, blocks: int, iters: int, stream=None) -> int:
    """Exp2 throughput probe; `out` is a float32 device tensor of blocks * 256 elements."""
    return lib().attn_bench_ex2(_ptr(out), blocks, iters, _stream(stream))


def attn_get_status(stream=None) -> int:
    return lib().attn_get_status(_stream(stream))


def attn_release() -> None:
    lib().attn_release()


def attn_cached_device_state(device: int) -> int:
    """Bit 0: the status word's address is cached for `device`; bit 1: the allocation-free
    decode's scratch address is."""
    return lib().attn_cached_device_state(device)


def attn_noalloc_scratch_bytes() -> int:
    return lib().attn_noalloc_scratch_bytes()


def attn_version() -> int:
    return lib().attn_version()


def attn_plan_kv_range(mask_kind, window, r0, bm, row_end, k_org, k_end, bn):
    lo, hi = _i(), _i()
    rc = lib().attn_plan_kv_range(mask_kind, window, r0, bm, row_end, k_org, k_end, bn,
                                  ctypes.byref(lo), ctypes.byref(hi))
    if rc != ATTN_OK:
        raise AttnError(rc, "attn_plan_kv_range")
    return lo.value, hi.value


def attn_plan_tile_kind(mask_kind, window, r0, bm, row_end, k_org, k_end, bn, t) -> int:
    return lib().attn_plan_tile_kind(mask_kind, window, r0, bm, row_end, k_org, k_end, bn, t)


def attn_plan_units(mask_kind, B, Hq, N, cu_seqlens=None, seqlens_k=None):
    """Prefill work list in launch order: list of (batch-or-segment, head, pair) tuples.
    For ATTN_MASK_PAGED_PREFILL pass the chunk starts and the context lengths."""
    import numpy as np
    if seqlens_k is not None:
        cu_seqlens = np.concatenate([np.asarray(cu_seqlens), np.asarray(seqlens_k)])
    cu = None if cu_seqlens is None else np.ascontiguousarray(cu_seqlens, dtype=np.int32)
    cu_p = None if cu is None else cu.ctypes.data
    n = lib().attn_plan_units(mask_kind, B, Hq, N, cu_p, None, 0)
    if n < 0:
        raise AttnError(n, "attn_plan_units")
    out = np.zeros((max(n, 1), 3), dtype=np.int32)
    lib().attn_plan_units(mask_kind, B, Hq, N, cu_p, out.ctypes.data, n)
    return [tuple(int(x) for x in r) for r in out[:n]]
