"""Seeded synthetic workloads for the attention forward pass.

This module holds no attention arithmetic. It only draws random numbers, rounds the draws
to bf16 bytes, draws document segment lengths and lays out a paged KV cache. The CUDA path
and the CPU oracle both consume exactly the arrays produced here, so the two never share
anything else.

Recipe (the same for every workload):
  * generator: ``numpy.random.default_rng(seed)``; draw order is lengths, then Q, K, V,
    then the page permutation;
  * values: fp32 N(0, 1), rounded to nearest-even into bf16 and kept as raw uint16 bits;
  * scale: the fp32 value of 1/sqrt(d).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

# Mask-kind codes of the C ABI (``include/attn.h``).
MASK_NONE = 0
MASK_CAUSAL = 1
MASK_SLIDING = 2
MASK_DOCUMENT = 3
MASK_PAGED_DECODE = 4
MASK_DECODE = 5
MASK_SLIDING_BIDIR = 6
MASK_DOCUMENT_BIDIR = 7
MASK_PREFIX_LM = 8
# Chunked prefill over a paged cache: served by attn_fwd_paged_prefill, not attn_fwd.
MASK_PAGED_PREFILL = 9
DECODE_KINDS = (MASK_PAGED_DECODE, MASK_DECODE)
DOCUMENT_KINDS = (MASK_DOCUMENT, MASK_DOCUMENT_BIDIR)
PACKED_KINDS = (MASK_DOCUMENT, MASK_DOCUMENT_BIDIR, MASK_PAGED_PREFILL)

PAGE_SIZE = 64
# Poison written into unused page slots and spare pages: finite, and large enough that any
# leak of a masked or out-of-range key into a result is far outside the parity tolerance.
POISON_K = 30.0
POISON_V = 1000.0


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 values to nearest-even bf16; return the 16-bit patterns (uint16)."""
    src = np.ascontiguousarray(x, dtype=np.float32).reshape(-1).view(np.uint32)
    out = np.empty(src.shape, dtype=np.uint16)
    step = 1 << 22
    u = np.empty(min(step, src.size), dtype=np.uint32)
    lsb = np.empty_like(u)
    for s0 in range(0, src.size, step):
        n = min(step, src.size - s0)
        # uint32 arithmetic cannot overflow for finite inputs (largest finite 0xFF7FFFFF)
        np.right_shift(src[s0:s0 + n], 16, out=lsb[:n])
        lsb[:n] &= 1
        np.add(src[s0:s0 + n], np.uint32(0x7FFF), out=u[:n])
        u[:n] += lsb[:n]
        u[:n] >>= 16
        out[s0:s0 + n] = u[:n]
    return out.reshape(np.shape(x))


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 exactly."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    """i.i.d. N(0,1) fp32 draws rounded to bf16 bits."""
    return f32_to_bf16_bits(rng.standard_normal(size=shape, dtype=np.float32))


def default_scale(d: int) -> float:
    """fp32 value of 1/sqrt(d), the scale every workload passes."""
    return float(np.float32(1.0 / math.sqrt(d)))


@dataclasses.dataclass
class Workload:
    """One attention forward problem in the layouts of the C ABI.

    Dense kinds: q, o ``[B,Hq,N,d]``; k, v ``[B,Hkv,N,d]``; lse ``[B,Hq,N]``.
    DOCUMENT, DOCUMENT_BIDIR: B is the segment count and tensors are packed ``[1,H,T,d]``
    with T = N.
    SLIDING and SLIDING_BIDIR take the window, PREFIX_LM the prefix length, in ``window``.
    PAGED_DECODE: q, o ``[B,Hq,1,d]``; k, v pools ``[num_pages,Hkv,64,d]``;
    lse ``[B,Hq]``; N is the longest context.
    DECODE: q, o ``[B,Hq,1,d]``; k, v dense caches ``[B,Hkv,N,d]``; lse ``[B,Hq]``.
    PAGED_PREFILL: B sequences; query chunks packed ``[1,Hq,N,d]`` with chunk starts in
    cu_seqlens; k, v pools ``[num_pages,Hkv,page,d]``; seqlens_k holds each sequence's context
    length (its chunk included); lse ``[1,Hq,N]``.
    """

    name: str
    mask_kind: int
    B: int
    Hq: int
    Hkv: int
    N: int
    d: int
    scale: float
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    window: int = 0
    cu_seqlens: Optional[np.ndarray] = None
    block_table: Optional[np.ndarray] = None
    page_size: int = 0
    seqlens_k: Optional[np.ndarray] = None
    # FP8 Q / K (E4M3 codes in the q / k layouts) and their per-128-row block scales
    # [planes, ceil(N/128)]; when set, q8 / k8 replace q / k as the attention inputs.
    q8: Optional[np.ndarray] = None
    k8: Optional[np.ndarray] = None
    q_scales: Optional[np.ndarray] = None
    k_scales: Optional[np.ndarray] = None

    @property
    def out_shape(self):
        if self.mask_kind in DECODE_KINDS:
            return (self.B, self.Hq, 1, self.d)
        if self.mask_kind in PACKED_KINDS:
            return (1, self.Hq, self.N, self.d)
        return (self.B, self.Hq, self.N, self.d)

    @property
    def lse_shape(self):
        return self.out_shape[:-1] if self.mask_kind not in DECODE_KINDS else (self.B, self.Hq)

    def valid_pairs_per_head(self) -> np.ndarray:
        """Number of visible (query, key) pairs for each batch entry / segment / sequence."""
        if self.mask_kind == MASK_NONE:
            return np.full(self.B, self.N * self.N, dtype=np.int64)
        if self.mask_kind == MASK_CAUSAL:
            return np.full(self.B, self.N * (self.N + 1) // 2, dtype=np.int64)
        if self.mask_kind == MASK_SLIDING:
            w, n = self.window, self.N
            full = min(w, n)
            # rows i < w see i+1 keys, rows i >= w see w keys
            cnt = full * (full + 1) // 2 + max(0, n - w) * w
            return np.full(self.B, cnt, dtype=np.int64)
        if self.mask_kind == MASK_SLIDING_BIDIR:
            i = np.arange(self.N, dtype=np.int64)
            cnt = (np.minimum(i + self.window, self.N - 1) - np.maximum(i - self.window, 0) + 1)
            return np.full(self.B, int(cnt.sum()), dtype=np.int64)
        if self.mask_kind == MASK_PREFIX_LM:
            i = np.arange(self.N, dtype=np.int64)
            cnt = np.minimum(np.maximum(i + 1, self.window), self.N)
            return np.full(self.B, int(cnt.sum()), dtype=np.int64)
        lens = np.diff(self.cu_seqlens.astype(np.int64))
        if self.mask_kind == MASK_DOCUMENT:
            return lens * (lens + 1) // 2
        if self.mask_kind == MASK_DOCUMENT_BIDIR:
            return lens * lens
        if self.mask_kind == MASK_PAGED_PREFILL:
            lk = self.seqlens_k.astype(np.int64)
            # chunk row t sees lk - lq + t + 1 keys
            return lens * (lk - lens) + lens * (lens + 1) // 2
        return lens  # decode: one query row sees all L_b keys

    def flops(self) -> float:
        """Algorithmic FLOPs 4 * Hq * d * (visible pairs), summed over batch/segments."""
        return 4.0 * self.Hq * self.d * float(self.valid_pairs_per_head().sum())

    def kv_bytes_valid(self) -> int:
        """Decode: K+V bytes of the valid tokens (what an ideal kernel reads)."""
        lens = (self.seqlens_k.astype(np.int64) if self.seqlens_k is not None
                else np.diff(self.cu_seqlens.astype(np.int64)))
        return int(lens.sum()) * self.Hkv * self.d * 2 * 2


def dense_workload(seed: int, B: int, Hq: int, Hkv: int, N: int, d: int,
                   mask_kind: int = MASK_NONE, window: int = 0, name: str = "") -> Workload:
    rng = np.random.default_rng(seed)
    q = normal_bf16(rng, (B, Hq, N, d))
    k = normal_bf16(rng, (B, Hkv, N, d))
    v = normal_bf16(rng, (B, Hkv, N, d))
    return Workload(name or f"dense_m{mask_kind}", mask_kind, B, Hq, Hkv, N, d,
                    default_scale(d), q, k, v, window=window)


def draw_segments(rng: np.random.Generator, total: int, lo: int, hi: int) -> np.ndarray:
    """Segment lengths uniform in [lo, hi], drawn until they cover ``total``; the last one is
    cut to fit (so it may be shorter than ``lo``). Returns cu_seqlens (int32, [S+1])."""
    lens = []
    acc = 0
    while acc < total:
        ln = int(rng.integers(lo, hi + 1))
        ln = min(ln, total - acc)
        lens.append(ln)
        acc += ln
    return np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)


def document_workload(seed: int, T: int, H: int, d: int, lo: int = 256, hi: int = 4096,
                      cu_seqlens: Optional[np.ndarray] = None, Hkv: Optional[int] = None,
                      name: str = "", mask_kind: int = MASK_DOCUMENT) -> Workload:
    rng = np.random.default_rng(seed)
    cu = draw_segments(rng, T, lo, hi) if cu_seqlens is None else np.asarray(cu_seqlens, np.int32)
    hkv = H if Hkv is None else Hkv
    q = normal_bf16(rng, (1, H, T, d))
    k = normal_bf16(rng, (1, hkv, T, d))
    v = normal_bf16(rng, (1, hkv, T, d))
    return Workload(name or "document", mask_kind, len(cu) - 1, H, hkv, T, d,
                    default_scale(d), q, k, v, cu_seqlens=cu)


def paged_decode_workload(seed: int, B: int, Lmin: int, Lmax: int, Hq: int, Hkv: int, d: int,
                          page_size: int = PAGE_SIZE, spare_pages: int = 64,
                          context_lens: Optional[np.ndarray] = None, shuffle: bool = True,
                          name: str = "") -> Workload:
    """Paged KV decode problem: one query token per sequence, KV in a permuted page pool.

    Logical page p of sequence b (pages numbered in order of b, then p) lives at physical page
    perm[index]; the pool has ``spare_pages`` extra pages. Slots past each sequence's end and
    the spare pages hold poison. Block-table padding is -1.
    """
    rng = np.random.default_rng(seed)
    if context_lens is None:
        lens = rng.integers(Lmin, Lmax + 1, size=B).astype(np.int64)
    else:
        lens = np.asarray(context_lens, dtype=np.int64)
    q = normal_bf16(rng, (B, Hq, 1, d))
    tot = int(lens.sum())
    k_all = normal_bf16(rng, (Hkv, tot, d)) if tot else np.zeros((Hkv, 0, d), np.uint16)
    v_all = normal_bf16(rng, (Hkv, tot, d)) if tot else np.zeros((Hkv, 0, d), np.uint16)
    pages_per_seq = (lens + page_size - 1) // page_size
    used = int(pages_per_seq.sum())
    num_pages = used + spare_pages
    perm = rng.permutation(num_pages) if shuffle else np.arange(num_pages)
    pk = f32_to_bf16_bits(np.float32(POISON_K))
    pv = f32_to_bf16_bits(np.float32(POISON_V))
    k_pool = np.full((num_pages, Hkv, page_size, d), pk, dtype=np.uint16)
    v_pool = np.full((num_pages, Hkv, page_size, d), pv, dtype=np.uint16)
    max_pages = int(pages_per_seq.max()) if B else 0
    table = np.full((B, max(max_pages, 1)), -1, dtype=np.int32)
    idx = 0
    tok_phys = np.empty(tot, dtype=np.int64)
    tok_slot = np.empty(tot, dtype=np.int64)
    tok0 = 0
    for b in range(B):
        np_b = int(pages_per_seq[b])
        table[b, :np_b] = perm[idx: idx + np_b]
        idx += np_b
        t = np.arange(int(lens[b]))
        tok_phys[tok0: tok0 + len(t)] = table[b, t // page_size]
        tok_slot[tok0: tok0 + len(t)] = t % page_size
        tok0 += int(lens[b])
    # token-major copy: pool[phys, :, slot, :] = seq_kv[:, token, :]
    k_pool[tok_phys, :, tok_slot, :] = k_all.transpose(1, 0, 2)
    v_pool[tok_phys, :, tok_slot, :] = v_all.transpose(1, 0, 2)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N = int(lens.max()) if B else 0
    return Workload(name or "paged_decode", MASK_PAGED_DECODE, B, Hq, Hkv, N, d,
                    default_scale(d), q, k_pool, v_pool, cu_seqlens=cu, block_table=table,
                    page_size=page_size)


def _paged_pool(rng, lens, Hkv, d, page_size, spare_pages, shuffle):
    """Token-major K / V for the given context lengths laid out in a permuted page pool.
    Returns (k_pool, v_pool, block_table). Draws K, V, then the permutation."""
    B = len(lens)
    tot = int(lens.sum())
    k_all = normal_bf16(rng, (Hkv, tot, d)) if tot else np.zeros((Hkv, 0, d), np.uint16)
    v_all = normal_bf16(rng, (Hkv, tot, d)) if tot else np.zeros((Hkv, 0, d), np.uint16)
    pages_per_seq = (lens + page_size - 1) // page_size
    used = int(pages_per_seq.sum())
    num_pages = used + spare_pages
    perm = rng.permutation(num_pages) if shuffle else np.arange(num_pages)
    pk = f32_to_bf16_bits(np.float32(POISON_K))
    pv = f32_to_bf16_bits(np.float32(POISON_V))
    k_pool = np.full((num_pages, Hkv, page_size, d), pk, dtype=np.uint16)
    v_pool = np.full((num_pages, Hkv, page_size, d), pv, dtype=np.uint16)
    max_pages = int(pages_per_seq.max()) if B else 0
    table = np.full((B, max(max_pages, 1)), -1, dtype=np.int32)
    idx = 0
    tok_phys = np.empty(tot, dtype=np.int64)
    tok_slot = np.empty(tot, dtype=np.int64)
    tok0 = 0
    for b in range(B):
        np_b = int(pages_per_seq[b])
        table[b, :np_b] = perm[idx: idx + np_b]
        idx += np_b
        t = np.arange(int(lens[b]))
        tok_phys[tok0: tok0 + len(t)] = table[b, t // page_size]
        tok_slot[tok0: tok0 + len(t)] = t % page_size
        tok0 += int(lens[b])
    k_pool[tok_phys, :, tok_slot, :] = k_all.transpose(1, 0, 2)
    v_pool[tok_phys, :, tok_slot, :] = v_all.transpose(1, 0, 2)
    return k_pool, v_pool, table


def paged_prefill_workload(seed: int, B: int, Lk_min: int, Lk_max: int, Lq_min: int,
                           Lq_max: int, Hq: int, Hkv: int, d: int, page_size: int = 16,
                           spare_pages: int = 64, context_lens=None, chunk_lens=None,
                           shuffle: bool = True, name: str = "") -> Workload:
    """Chunked prefill over a paged cache: sequence b's context of Lk_b tokens (uniform in
    [Lk_min, Lk_max]) sits in a permuted page pool, and its last Lq_b tokens (uniform in
    [Lq_min, min(Lq_max, Lk_b)]) are the new query chunk. Draw order: context lengths, chunk
    lengths, Q (packed chunks), K, V, page permutation. Pool slots past each context and the
    spare pages hold poison; block-table padding is -1."""
    rng = np.random.default_rng(seed)
    if context_lens is None:
        lk = rng.integers(Lk_min, Lk_max + 1, size=B).astype(np.int64)
    else:
        lk = np.asarray(context_lens, dtype=np.int64)
    if chunk_lens is None:
        lq = np.array([rng.integers(min(Lq_min, L), min(Lq_max, L) + 1) for L in lk],
                      dtype=np.int64)
    else:
        lq = np.asarray(chunk_lens, dtype=np.int64)
    assert np.all(lq <= lk) and np.all(lq >= 0)
    T = int(lq.sum())
    q = normal_bf16(rng, (1, Hq, T, d))
    k_pool, v_pool, table = _paged_pool(rng, lk, Hkv, d, page_size, spare_pages, shuffle)
    cu = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    return Workload(name or "paged_prefill", MASK_PAGED_PREFILL, B, Hq, Hkv, T, d,
                    default_scale(d), q, k_pool, v_pool, cu_seqlens=cu, block_table=table,
                    page_size=page_size, seqlens_k=lk.astype(np.int32))


def dense_decode_workload(seed: int, B: int, Lmin: int, Lmax: int, Hq: int, Hkv: int, d: int,
                          N: Optional[int] = None, context_lens: Optional[np.ndarray] = None,
                          name: str = "") -> Workload:
    """Decode problem on a dense per-sequence cache ``[B,Hkv,N,d]`` (N >= every length).

    Draws lengths, q and the token-major K / V exactly as ``paged_decode_workload`` does with
    the same arguments, so both describe the same attention problem; only the placement of
    the keys differs. Slots past each sequence's end hold poison.
    """
    rng = np.random.default_rng(seed)
    if context_lens is None:
        lens = rng.integers(Lmin, Lmax + 1, size=B).astype(np.int64)
    else:
        lens = np.asarray(context_lens, dtype=np.int64)
    q = normal_bf16(rng, (B, Hq, 1, d))
    tot = int(lens.sum())
    k_all = normal_bf16(rng, (Hkv, tot, d)) if tot else np.zeros((Hkv, 0, d), np.uint16)
    v_all = normal_bf16(rng, (Hkv, tot, d)) if tot else np.zeros((Hkv, 0, d), np.uint16)
    if N is None:
        N = int(lens.max()) if B else 0
    k = np.full((B, Hkv, N, d), f32_to_bf16_bits(np.float32(POISON_K)), dtype=np.uint16)
    v = np.full((B, Hkv, N, d), f32_to_bf16_bits(np.float32(POISON_V)), dtype=np.uint16)
    tok0 = 0
    for b in range(B):
        L = int(lens[b])
        k[b, :, :L, :] = k_all[:, tok0: tok0 + L, :]
        v[b, :, :L, :] = v_all[:, tok0: tok0 + L, :]
        tok0 += L
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return Workload(name or "dense_decode", MASK_DECODE, B, Hq, Hkv, N, d, default_scale(d),
                    q, k, v, cu_seqlens=cu)


# The five workloads the path is specified on, plus the causal shape the headline
# throughput is quoted on (the sliding-window shape without the window).
def config(k) -> Workload:
    if k == 1:
        return dense_workload(1001, 1, 1, 1, 256, 64, MASK_NONE, name="dense B1 H1 N256 d64")
    if k == 2:
        return dense_workload(1002, 4, 16, 16, 2048, 128, MASK_CAUSAL,
                              name="causal B4 H16 N2048 d128")
    if k == 3:
        return dense_workload(1003, 2, 32, 8, 8192, 128, MASK_SLIDING, window=4096,
                              name="sliding W4096 B2 Hq32 Hkv8 N8192 d128")
    if k == "3c":
        return dense_workload(1003, 2, 32, 8, 8192, 128, MASK_CAUSAL,
                              name="causal B2 Hq32 Hkv8 N8192 d128")
    if k == 4:
        return document_workload(1004, 16384, 16, 64, 256, 4096,
                                 name="document T16384 H16 d64 seg U[256,4096]")
    if k == 5:
        return paged_decode_workload(1005, 32, 1024, 16384, 32, 8, 128, name=(
            "paged decode B32 L U[1024,16384] Hq32 Hkv8 d128 page64"))
    # The mask variants on the same shapes: a two-sided window with as many keys per query as
    # the causal window above, a prefix of half the sequence, and the 16384-token document
    # packing's segments without the causal constraint.
    if k == "3b":
        return dense_workload(1003, 2, 32, 8, 8192, 128, MASK_SLIDING_BIDIR, window=2048,
                              name="two-sided window W2048 B2 Hq32 Hkv8 N8192 d128")
    if k == "3p":
        return dense_workload(1003, 2, 32, 8, 8192, 128, MASK_PREFIX_LM, window=4096,
                              name="prefix-LM P4096 B2 Hq32 Hkv8 N8192 d128")
    # Chunked prefill over a paged cache: 16 sequences with contexts U[2048,16384] whose last
    # U[256,2048] tokens are the new chunk, vLLM-sized pages of 16 tokens (and 64).
    if k in ("6", "6p64"):
        ps = 16 if k == "6" else 64
        return paged_prefill_workload(1006, 16, 2048, 16384, 256, 2048, 32, 8, 128,
                                      page_size=ps, name=(
                                          "chunked prefill B16 Lk U[2048,16384] Lq U[256,2048] "
                                          f"Hq32 Hkv8 d128 page{ps}"))
    # Small batches of the paged decode: one 16K-token sequence, and four sequences of 1K-16K.
    if k == "5b1":
        return paged_decode_workload(1051, 1, 16384, 16384, 32, 8, 128, name=(
            "paged decode B1 L16384 Hq32 Hkv8 d128 page64"))
    if k == "5b4":
        return paged_decode_workload(1054, 4, 1024, 16384, 32, 8, 128, name=(
            "paged decode B4 L U[1024,16384] Hq32 Hkv8 d128 page64"))
    if k == "5p16":
        return paged_decode_workload(1005, 32, 1024, 16384, 32, 8, 128, page_size=16, name=(
            "paged decode B32 L U[1024,16384] Hq32 Hkv8 d128 page16"))
    # The headline causal shape at head dim 64 (long sequences: the d = 64 kernel's steady state).
    if k == "3c64":
        return dense_workload(1003, 2, 32, 8, 8192, 64, MASK_CAUSAL,
                              name="causal B2 Hq32 Hkv8 N8192 d64")
    if k == "4b":
        return document_workload(1004, 16384, 16, 64, 256, 4096, mask_kind=MASK_DOCUMENT_BIDIR,
                                 name="non-causal document T16384 H16 d64 seg U[256,4096]")
    raise KeyError(k)
