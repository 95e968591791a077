"""fp64 CPU oracle for the attention forward pass (Python marshalling around attn_oracle.c).

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the benchmark's CPU-baseline
leg are the only callers. The CUDA library never imports, links or runs anything here, and
this package imports nothing from the CUDA library; the two meet only in the seeded inputs.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB_DIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIB_DIR, "libattn_oracle.so")
_libs = {}


def compile_source(src: str, out: str) -> str:
    """Compile an oracle C source with gcc (OpenMP, strict IEEE fp64: no fast-math)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                           "-ffp-contract=off", "-o", tmp, src, "-lm"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile attn_oracle.c into oracle/_lib (skipped when the library is up to date)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    return compile_source(_SRC, _LIB)


def _load(path: str = None):
    path = path or build()
    if path not in _libs:
        lib = ctypes.CDLL(path)
        p = ctypes.c_void_p
        i = ctypes.c_int
        i64 = ctypes.c_int64
        lib.oracle_attn.argtypes = [p, p, p, i, i, i, i, i, ctypes.c_float, i, i, p, p, p, i,
                                    i, p, i64, p, p, p, i64, i]
        lib.oracle_attn.restype = i
        lib.oracle_attn_qk_f64.argtypes = lib.oracle_attn.argtypes
        lib.oracle_attn_qk_f64.restype = i
        lib.oracle_max_threads.argtypes = [i]
        lib.oracle_max_threads.restype = i
        _libs[path] = lib
    return _libs[path]


def _ptr(a):
    return None if a is None else a.ctypes.data


def max_threads(threads: int = 0) -> int:
    return _load().oracle_max_threads(threads)


def attention(w, rows=None, probs: bool = False, threads: int = 0, lib_path: str = None):
    """Run the oracle on a ``tiled_attention_gb300.inputs.Workload``-shaped problem. A
    workload carrying FP8 Q / K (``q8``, ``k8``, ``q_scales``, ``k_scales``) is computed on
    their dequantized values.

    rows: optional int64 array of flattened output-row indices (output order of O / LSE);
    default all rows. Returns (o [nrows, d] float64, lse [nrows] float64[, probs]).
    lib_path: another build of an oracle source (the mutation tests use this).
    """
    lib = _load(lib_path)
    fp8 = getattr(w, "q8", None) is not None
    if fp8:
        # FP8 Q / K: the dequantized blocks (code value x block scale), exact in float64.
        from . import fp8 as _fp8
        q = np.ascontiguousarray(_fp8.dequantize(w.q8.reshape(-1, w.q8.shape[-2], w.d),
                                                 w.q_scales.reshape(-1, w.q_scales.shape[-1])))
        k = np.ascontiguousarray(_fp8.dequantize(w.k8.reshape(-1, w.k8.shape[-2], w.d),
                                                 w.k_scales.reshape(-1, w.k_scales.shape[-1])))
        entry = lib.oracle_attn_qk_f64
    else:
        q = np.ascontiguousarray(w.q, dtype=np.uint16)
        k = np.ascontiguousarray(w.k, dtype=np.uint16)
        entry = lib.oracle_attn
    v = np.ascontiguousarray(w.v, dtype=np.uint16)
    cu = None if w.cu_seqlens is None else np.ascontiguousarray(w.cu_seqlens, dtype=np.int32)
    tab = None if w.block_table is None else np.ascontiguousarray(w.block_table, dtype=np.int32)
    lk = getattr(w, "seqlens_k", None)
    lk = None if lk is None else np.ascontiguousarray(lk, dtype=np.int32)
    max_pages = 0 if tab is None else tab.shape[1]
    total = int(np.prod(w.lse_shape))
    if rows is None:
        n = total
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
        n = rows_arr.size
    o = np.zeros((n, w.d), dtype=np.float64)
    lse = np.zeros(n, dtype=np.float64)
    if w.mask_kind in (4, 5):
        nk = int(np.diff(cu).max(initial=0))
    elif lk is not None:
        nk = max(w.N, int(lk.max(initial=0)))
    else:
        nk = w.N
    pr = np.zeros((n, max(nk, 1)), dtype=np.float64) if probs else None
    rc = entry(_ptr(q), _ptr(k), _ptr(v), w.B, w.Hq, w.Hkv, w.N, w.d,
                         ctypes.c_float(w.scale), w.mask_kind, w.window, _ptr(cu), _ptr(lk),
                         _ptr(tab), max_pages, w.page_size, _ptr(rows_arr), n, _ptr(o), _ptr(lse),
                         _ptr(pr), pr.shape[1] if probs else 0, threads)
    if rc != 0:
        raise ValueError(f"oracle_attn rejected the problem (code {rc})")
    return (o, lse, pr) if probs else (o, lse)
