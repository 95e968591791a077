"""Pins for the fp64 oracle: facts fixed by the mathematics, not by the oracle itself.

Every pin takes ``attn(w, rows=None, probs=False)`` so the same checks run against the real
oracle and against deliberately broken builds of it (tests/test_oracle_mutants.py).
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

from tiled_attention_gb300 import inputs as I

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")

KINDS = ["none", "causal", "sliding", "document", "paged", "decode", "sliding_bidir",
         "document_bidir", "prefix_lm", "paged_prefill"]


def widen(bits):
    return I.bf16_bits_to_f32(bits).astype(np.float64)


def bf16(x):
    return I.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def tiny(kind: str, seed: int = 7, window: int = 5):
    """Small problems with ragged sizes, GQA and several batch entries. ``window`` is the
    window of both sliding kinds and the prefix length of PREFIX_LM (default 9 there)."""
    if kind == "none":
        return I.dense_workload(seed, 2, 4, 2, 37, 16, I.MASK_NONE)
    if kind == "causal":
        return I.dense_workload(seed, 2, 4, 2, 37, 16, I.MASK_CAUSAL)
    if kind == "sliding":
        return I.dense_workload(seed, 2, 4, 2, 37, 16, I.MASK_SLIDING, window=window)
    if kind == "document":
        return I.document_workload(seed, 37, 4, 16, cu_seqlens=[0, 5, 6, 20, 37], Hkv=2)
    if kind == "paged":
        return I.paged_decode_workload(seed, 3, 0, 0, 4, 2, 16, page_size=8, spare_pages=3,
                                       context_lens=[1, 63, 130])
    if kind == "decode":
        return I.dense_decode_workload(seed, 3, 0, 0, 4, 2, 16, N=137, context_lens=[1, 63, 130])
    if kind == "sliding_bidir":
        return I.dense_workload(seed, 2, 4, 2, 37, 16, I.MASK_SLIDING_BIDIR, window=window)
    if kind == "document_bidir":
        return I.document_workload(seed, 37, 4, 16, cu_seqlens=[0, 5, 6, 20, 37], Hkv=2,
                                   mask_kind=I.MASK_DOCUMENT_BIDIR)
    if kind == "prefix_lm":
        return I.dense_workload(seed, 2, 4, 2, 37, 16, I.MASK_PREFIX_LM,
                                window=9 if window == 5 else window)
    if kind == "paged_prefill":
        return I.paged_prefill_workload(seed, 4, 0, 0, 0, 0, 4, 2, 16, page_size=8,
                                        spare_pages=3, context_lens=[1, 40, 130, 9],
                                        chunk_lens=[1, 17, 33, 9])
    raise KeyError(kind)


# ---- an independent dense view of each problem, built with torch library routines ----

def dense_problems(w):
    """Yield (row_index_array, q [R,d], k [L,d], v [L,d], mask [R,L] bool) per (batch, head),
    with the mask written as whole-matrix torch operations (tril / triu / segment ids)."""
    qf, kf, vf = widen(w.q), widen(w.k), widen(w.v)
    group = w.Hq // w.Hkv
    if w.mask_kind in (I.MASK_NONE, I.MASK_CAUSAL, I.MASK_SLIDING, I.MASK_SLIDING_BIDIR,
                       I.MASK_PREFIX_LM):
        N = w.N
        ones = torch.ones(N, N, dtype=torch.bool)
        if w.mask_kind == I.MASK_NONE:
            mask = ones
        elif w.mask_kind == I.MASK_CAUSAL:
            mask = torch.tril(ones)
        elif w.mask_kind == I.MASK_SLIDING:
            mask = torch.tril(ones) & torch.triu(ones, diagonal=-(w.window - 1))
        elif w.mask_kind == I.MASK_SLIDING_BIDIR:
            mask = torch.tril(ones, diagonal=w.window) & torch.triu(ones, diagonal=-w.window)
        else:  # prefix-LM: the lower triangle plus the first P columns
            prefix = torch.zeros(N, N, dtype=torch.bool)
            prefix[:, :w.window] = True
            mask = torch.tril(ones) | prefix
        for b in range(w.B):
            for h in range(w.Hq):
                rows = (b * w.Hq + h) * N + np.arange(N)
                yield rows, qf[b, h], kf[b, h // group], vf[b, h // group], mask.numpy()
    elif w.mask_kind in I.DOCUMENT_KINDS:
        T = w.N
        seg = torch.bucketize(torch.arange(T), torch.as_tensor(w.cu_seqlens[1:]), right=True)
        mask = seg[:, None] == seg[None, :]
        if w.mask_kind == I.MASK_DOCUMENT:
            mask = mask & torch.tril(torch.ones(T, T, dtype=torch.bool))
        for h in range(w.Hq):
            rows = h * T + np.arange(T)
            yield rows, qf[0, h], kf[0, h // group], vf[0, h // group], mask.numpy()
    elif w.mask_kind == I.MASK_PAGED_PREFILL:
        P = w.page_size
        for b in range(w.B):
            a, e = int(w.cu_seqlens[b]), int(w.cu_seqlens[b + 1])
            Lq, Lk = e - a, int(w.seqlens_k[b])
            pages = [int(w.block_table[b, p]) for p in range((Lk + P - 1) // P)]
            mask = torch.tril(torch.ones(Lq, Lk, dtype=torch.bool), diagonal=Lk - Lq).numpy()
            for h in range(w.Hq):
                g = h // group
                kk = np.concatenate([kf[p, g] for p in pages], axis=0)[:Lk]
                vv = np.concatenate([vf[p, g] for p in pages], axis=0)[:Lk]
                yield h * w.N + np.arange(a, e), qf[0, h, a:e], kk, vv, mask
    elif w.mask_kind == I.MASK_DECODE:
        for b in range(w.B):
            L = int(w.cu_seqlens[b + 1] - w.cu_seqlens[b])
            for h in range(w.Hq):
                g = h // group
                yield (np.array([b * w.Hq + h]), qf[b, h], kf[b, g, :L], vf[b, g, :L],
                       np.ones((1, L), dtype=bool))
    else:
        P = w.page_size
        for b in range(w.B):
            L = int(w.cu_seqlens[b + 1] - w.cu_seqlens[b])
            pages = [int(w.block_table[b, p]) for p in range((L + P - 1) // P)]
            for h in range(w.Hq):
                g = h // group
                kk = np.concatenate([kf[p, g] for p in pages], axis=0)[:L] if L else np.zeros((0, w.d))
                vv = np.concatenate([vf[p, g] for p in pages], axis=0)[:L] if L else np.zeros((0, w.d))
                yield (np.array([b * w.Hq + h]), qf[b, h], kk, vv, np.ones((1, L), dtype=bool))


def brute_force(w):
    """softmax(scale * Q K^T with masked entries -inf) @ V and logsumexp, torch fp64."""
    n = int(np.prod(w.lse_shape))
    O = np.zeros((n, w.d))
    L = np.zeros(n)
    s = float(np.float32(w.scale))
    for rows, q, k, v, mask in dense_problems(w):
        z = s * (torch.as_tensor(q) @ torch.as_tensor(k).T)
        z = z.masked_fill(~torch.as_tensor(mask), float("-inf"))
        O[rows] = (torch.softmax(z, dim=-1) @ torch.as_tensor(v)).numpy()
        L[rows] = torch.logsumexp(z, dim=-1).numpy()
    return O, L


def visible_lists(w):
    out = {}
    for rows, q, k, v, mask in dense_problems(w):
        for t, r in enumerate(rows):
            out[int(r)] = (np.nonzero(mask[t])[0], v, k, q[t])
    return out


# ---------------------------------- pins ----------------------------------

def pin_brute_force(attn, kind):
    w = tiny(kind)
    o, lse = attn(w)
    bo, bl = brute_force(w)
    np.testing.assert_allclose(o, bo, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, bl, rtol=0, atol=1e-12)


def pin_q_zero_mean(attn, kind):
    """Q = 0: every visible score is 0, so O is the plain mean of the visible V rows and
    LSE = ln |V(i)|."""
    w = tiny(kind)
    w.q[...] = 0
    o, lse = attn(w)
    for r, (vis, v, _, _) in visible_lists(w).items():
        np.testing.assert_allclose(o[r], v[vis].mean(axis=0), rtol=0, atol=1e-13)
        assert abs(lse[r] - math.log(len(vis))) < 1e-13


def pin_dominant_logit(attn, kind):
    """One key scoring 256 above every other visible key selects its V row."""
    base = tiny(kind)
    vis = visible_lists(base)
    for r in sorted(vis)[:: max(1, len(vis) // 9)]:
        w = tiny(kind)
        idx, _, _, _ = vis[r]
        jstar = int(idx[len(idx) // 2])
        _set_dominant(w, r, jstar)
        o, _ = attn(w, rows=np.array([r]))
        vrow = visible_lists(w)[r][1][jstar]
        np.testing.assert_allclose(o[0], vrow, rtol=0, atol=1e-12)


def _set_dominant(w, r, jstar):
    """Query row r and key j* get component 0 equal to 32; every other key of that head gets
    component 0 equal to 0 and the query's other components are 0. Then z(r, j*) = 1024*s and
    every other visible score is 0."""
    group = w.Hq // w.Hkv
    if w.mask_kind == I.MASK_PAGED_DECODE:
        b, h = divmod(r, w.Hq)
        g = h // group
        w.q[b, h, 0, :] = 0
        w.q[b, h, 0, 0] = bf16(32.0)
        w.k[:, g, :, 0] = 0
        P = w.page_size
        w.k[w.block_table[b, jstar // P], g, jstar % P, 0] = bf16(32.0)
        return
    if w.mask_kind == I.MASK_PAGED_PREFILL:
        h, i = divmod(r, w.N)
        b = int(np.searchsorted(w.cu_seqlens, i, side="right")) - 1
        g = h // group
        w.q[0, h, i, :] = 0
        w.q[0, h, i, 0] = bf16(32.0)
        w.k[:, g, :, 0] = 0
        P = w.page_size
        w.k[w.block_table[b, jstar // P], g, jstar % P, 0] = bf16(32.0)
        return
    if w.mask_kind == I.MASK_DECODE:
        b, h = divmod(r, w.Hq)
        g = h // group
        w.q[b, h, 0, :] = 0
        w.q[b, h, 0, 0] = bf16(32.0)
        w.k[b, g, :, 0] = 0
        w.k[b, g, jstar, 0] = bf16(32.0)
        return
    if w.mask_kind in I.DOCUMENT_KINDS:
        h, i = divmod(r, w.N)
        b = 0
    else:
        b, rem = divmod(r, w.Hq * w.N)
        h, i = divmod(rem, w.N)
    g = h // group
    w.q[b, h, i, :] = 0
    w.q[b, h, i, 0] = bf16(32.0)
    w.k[b, g, :, 0] = 0
    w.k[b, g, jstar, 0] = bf16(32.0)


def pin_probabilities(attn, kind):
    """Each softmax row is non-negative, sums to 1 and is zero off the visible set."""
    w = tiny(kind)
    _, _, p = attn(w, probs=True)
    for r, (vis, _, _, _) in visible_lists(w).items():
        row = p[r]
        assert np.all(row >= 0)
        assert abs(row.sum() - 1.0) < 1e-13
        off = np.ones(row.size, dtype=bool)
        off[vis] = False
        assert np.all(row[off] == 0)


def pin_single_key_rows(attn, kind):
    """A row that sees exactly one key returns that key's V row exactly and LSE = its score."""
    if kind == "sliding":
        w = tiny(kind, window=1)
    elif kind == "sliding_bidir":
        w = tiny(kind, window=0)
    elif kind == "prefix_lm":
        w = tiny(kind, window=1)
    elif kind == "none":
        w = I.dense_workload(5, 2, 4, 2, 1, 16, I.MASK_NONE)
    else:
        w = tiny(kind)
    o, lse = attn(w)
    s = float(np.float32(w.scale))
    seen = 0
    for r, (vis, v, k, q) in visible_lists(w).items():
        if len(vis) != 1:
            continue
        j = int(vis[0])
        assert np.array_equal(o[r], v[j])
        assert abs(lse[r] - s * float(np.dot(q, k[j]))) < 1e-12
        seen += 1
    assert seen > 0


def pin_constant_values(attn, kind):
    """V identically c gives O = c for every row."""
    w = tiny(kind)
    c = 0.3671875
    w.v[...] = bf16(c)
    o, _ = attn(w)
    np.testing.assert_allclose(o, c, rtol=0, atol=1e-14)


def pin_logit_shift(attn, kind):
    """Adding the same constant to every score of a row changes LSE by that constant and
    leaves O unchanged (done through a component that is 1 in every key)."""
    w0 = tiny(kind)
    if kind == "paged":
        w0.k[:, :, :, 0] = bf16(1.0)
        w0.q[:, :, :, 0] = 0
    else:
        w0.k[..., 0] = bf16(1.0)
        w0.q[..., 0] = 0
    w1 = tiny(kind)
    w1.k[...] = w0.k
    w1.q[...] = w0.q
    w1.q[..., 0] = bf16(5.0)
    o0, l0 = attn(w0)
    o1, l1 = attn(w1)
    s = float(np.float32(w0.scale))
    np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-12)
    # Every row of these cases sees at least one key, so both LSEs are finite.
    assert np.isfinite(l0).all() and np.isfinite(l1).all()
    np.testing.assert_allclose(l1 - l0, 5.0 * s, rtol=0, atol=1e-12)


def pin_key_permutation(attn):
    """Without a mask, reordering keys and values together changes nothing."""
    w = tiny("none")
    perm = np.random.default_rng(3).permutation(w.N)
    wp = tiny("none")
    wp.k[...] = w.k[:, :, perm]
    wp.v[...] = w.v[:, :, perm]
    o0, l0 = attn(w)
    o1, l1 = attn(wp)
    np.testing.assert_allclose(o1, o0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1, l0, rtol=0, atol=1e-12)


def pin_window_covering_equals_causal(attn):
    c = tiny("causal")
    for W in (c.N, c.N + 1, 10 * c.N):
        s = tiny("sliding", window=W)
        assert np.array_equal(attn(s)[0], attn(c)[0])
        assert np.array_equal(attn(s)[1], attn(c)[1])
    s = tiny("sliding", window=c.N - 1)
    assert not np.array_equal(attn(s)[0], attn(c)[0])


def pin_single_segment_equals_causal(attn):
    c = I.dense_workload(11, 1, 4, 2, 37, 16, I.MASK_CAUSAL)
    d = I.document_workload(11, 37, 4, 16, cu_seqlens=[0, 37], Hkv=2)
    d.q[...], d.k[...], d.v[...] = c.q, c.k, c.v
    assert np.array_equal(attn(d)[0], attn(c)[0])
    assert np.array_equal(attn(d)[1], attn(c)[1])


def pin_gqa_equals_repeated_mha(attn, kind):
    w = tiny(kind)
    group = w.Hq // w.Hkv
    if kind == "paged":
        m = I.paged_decode_workload(7, 3, 0, 0, 4, 4, 16, page_size=8, spare_pages=3,
                                    context_lens=[1, 63, 130])
        m.block_table = w.block_table.copy()
    elif kind == "decode":
        m = I.dense_decode_workload(7, 3, 0, 0, 4, 4, 16, N=137, context_lens=[1, 63, 130])
    elif kind == "paged_prefill":
        m = I.paged_prefill_workload(7, 4, 0, 0, 0, 0, 4, 4, 16, page_size=8, spare_pages=3,
                                     context_lens=[1, 40, 130, 9], chunk_lens=[1, 17, 33, 9])
        m.block_table = w.block_table.copy()
    elif kind in ("document", "document_bidir"):
        m = I.document_workload(7, 37, 4, 16, cu_seqlens=[0, 5, 6, 20, 37], Hkv=4,
                                mask_kind=w.mask_kind)
    else:
        m = I.dense_workload(7, 2, 4, 4, 37, 16, w.mask_kind, window=w.window)
    m.q[...] = w.q
    m.k[...] = np.repeat(w.k, group, axis=1)
    m.v[...] = np.repeat(w.v, group, axis=1)
    assert np.array_equal(attn(m)[0], attn(w)[0])
    assert np.array_equal(attn(m)[1], attn(w)[1])


def pin_bidir_window_limits(attn):
    """A two-sided window that covers every key is no mask at all; one that covers none but
    the query (W = 0) returns each row's own V row; and the two-sided window W is the union
    of the causal window W + 1 and its mirror image (checked on the probabilities: the row
    of query i is non-zero exactly at keys i - W .. i + W)."""
    n = tiny("none")
    for W in (n.N - 1, n.N, 10 * n.N):
        s = tiny("sliding_bidir", window=W)
        assert np.array_equal(attn(s)[0], attn(n)[0])
        assert np.array_equal(attn(s)[1], attn(n)[1])
    s = tiny("sliding_bidir", window=n.N - 2)
    assert not np.array_equal(attn(s)[0], attn(n)[0])
    w0 = tiny("sliding_bidir", window=0)
    o, _ = attn(w0)
    vv = widen(w0.v)
    group = w0.Hq // w0.Hkv
    for b in range(w0.B):
        for h in range(w0.Hq):
            rows = (b * w0.Hq + h) * w0.N + np.arange(w0.N)
            assert np.array_equal(o[rows], vv[b, h // group])
    w = tiny("sliding_bidir", window=3)
    _, _, p = attn(w, probs=True)
    for r in range(p.shape[0]):
        i = r % w.N
        nz = np.nonzero(p[r])[0]
        assert list(nz) == list(range(max(0, i - 3), min(w.N, i + 4)))


def pin_prefix_limits(attn):
    """A prefix of 0 or 1 tokens is the causal mask; a prefix covering the sequence is no
    mask; with Q = 0 every visible score is 0, so row i's LSE is the log of its visible key
    count, max(i + 1, P)."""
    c = tiny("causal")
    n = tiny("none")
    for P in (0, 1):
        s = tiny("prefix_lm", window=P)
        assert np.array_equal(attn(s)[0], attn(c)[0])
        assert np.array_equal(attn(s)[1], attn(c)[1])
    for P in (n.N, n.N + 5):
        s = tiny("prefix_lm", window=P)
        assert np.array_equal(attn(s)[0], attn(n)[0])
        assert np.array_equal(attn(s)[1], attn(n)[1])
    w = tiny("prefix_lm", window=9)
    w.q[...] = 0
    o, lse = attn(w)
    for r in range(o.shape[0]):
        i = r % w.N
        assert abs(lse[r] - math.log(max(i + 1, 9))) < 1e-13


def pin_document_bidir_segments(attn):
    """Non-causal document attention equals unmasked attention run on each segment alone,
    and a single segment is no mask at all."""
    w = tiny("document_bidir")
    o, lse = attn(w)
    cu = w.cu_seqlens
    for s in range(len(cu) - 1):
        a, e = int(cu[s]), int(cu[s + 1])
        L = e - a
        d = I.dense_workload(0, 1, w.Hq, w.Hkv, L, w.d, I.MASK_NONE)
        d.q[0], d.k[0], d.v[0] = w.q[0, :, a:e], w.k[0, :, a:e], w.v[0, :, a:e]
        od, ld = attn(d)
        rows = (np.arange(w.Hq)[:, None] * w.N + np.arange(a, e)[None, :]).reshape(-1)
        assert np.array_equal(od, o[rows])
        assert np.array_equal(ld, lse[rows])
    n = I.dense_workload(11, 1, 4, 2, 37, 16, I.MASK_NONE)
    d = I.document_workload(11, 37, 4, 16, cu_seqlens=[0, 37], Hkv=2,
                            mask_kind=I.MASK_DOCUMENT_BIDIR)
    d.q[...], d.k[...], d.v[...] = n.q, n.k, n.v
    assert np.array_equal(attn(d)[0], attn(n)[0])
    assert np.array_equal(attn(d)[1], attn(n)[1])


def pin_paged_prefill_whole_context_equals_document(attn):
    """A chunk that is the whole context is causal attention over that sequence: the same as
    the causal document mask over the gathered tokens, bit for bit."""
    lens = [1, 40, 130, 9]
    w = I.paged_prefill_workload(17, 4, 0, 0, 0, 0, 4, 2, 16, page_size=8, spare_pages=3,
                                 context_lens=lens, chunk_lens=lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    d = I.document_workload(0, int(cu[-1]), 4, 16, cu_seqlens=cu, Hkv=2)
    d.q[...] = w.q
    P = w.page_size
    for b, L in enumerate(lens):
        pages = [int(w.block_table[b, p]) for p in range((L + P - 1) // P)]
        d.k[0, :, cu[b]:cu[b + 1]] = np.concatenate([w.k[p] for p in pages], axis=1)[:, :L]
        d.v[0, :, cu[b]:cu[b + 1]] = np.concatenate([w.v[p] for p in pages], axis=1)[:, :L]
    assert np.array_equal(attn(w)[0], attn(d)[0])
    assert np.array_equal(attn(w)[1], attn(d)[1])


def pin_paged_prefill_last_row_equals_decode(attn):
    """The last row of each chunk sees the whole context: it is the paged decode of that
    sequence with the same pool and block table, bit for bit."""
    w = tiny("paged_prefill")
    o, lse = attn(w)
    dec = I.paged_decode_workload(0, w.B, 0, 0, w.Hq, w.Hkv, w.d, page_size=w.page_size,
                                  spare_pages=3, context_lens=w.seqlens_k)
    dec.k, dec.v, dec.block_table = w.k, w.v, w.block_table
    for b in range(w.B):
        dec.q[b, :, 0] = w.q[0, :, w.cu_seqlens[b + 1] - 1]
    od, ld = attn(dec)
    for b in range(w.B):
        rows = np.arange(w.Hq) * w.N + (w.cu_seqlens[b + 1] - 1)
        assert np.array_equal(od[b * w.Hq:(b + 1) * w.Hq], o[rows])
        assert np.array_equal(ld[b * w.Hq:(b + 1) * w.Hq], lse[rows])


def pin_paged_prefill_page_size_invariant(attn):
    """The same tokens in pools of 8- and 16-token pages (different permutations) give the
    same results bit for bit."""
    kw = dict(context_lens=[1, 40, 130, 9], chunk_lens=[1, 17, 33, 9], spare_pages=3)
    a = I.paged_prefill_workload(19, 4, 0, 0, 0, 0, 4, 2, 16, page_size=8, **kw)
    b = I.paged_prefill_workload(19, 4, 0, 0, 0, 0, 4, 2, 16, page_size=16, **kw)
    assert np.array_equal(attn(a)[0], attn(b)[0])
    assert np.array_equal(attn(a)[1], attn(b)[1])


def pin_paged_equals_dense_last_row(attn):
    """Decode of sequence b equals the last row of causal attention over its L_b tokens laid
    out contiguously (the query is the last token and sees the whole context)."""
    w = tiny("paged")
    o, lse = attn(w)
    P = w.page_size
    for b in range(w.B):
        L = int(w.cu_seqlens[b + 1] - w.cu_seqlens[b])
        pages = [int(w.block_table[b, p]) for p in range((L + P - 1) // P)]
        dk = np.concatenate([w.k[p] for p in pages], axis=1)[:, :L]
        dv = np.concatenate([w.v[p] for p in pages], axis=1)[:, :L]
        dn = I.dense_workload(0, 1, w.Hq, w.Hkv, L, w.d, I.MASK_CAUSAL)
        dn.k[0], dn.v[0] = dk, dv
        dn.q[0, :, L - 1] = w.q[b, :, 0]
        rows = np.arange(w.Hq) * L + (L - 1)
        od, ld = attn(dn, rows=rows)
        assert np.array_equal(od, o[b * w.Hq:(b + 1) * w.Hq])
        assert np.array_equal(ld, lse[b * w.Hq:(b + 1) * w.Hq])


def pin_online_recurrence(attn, kind):
    """The running-max / running-sum update over key tiles (m_new = max(m, tile max),
    rescale by exp(m - m_new), l = alpha*l + sum p, acc = alpha*acc + p v; divide by l at
    the end) gives the same function as the two-pass oracle, for any tile width."""
    w = tiny(kind)
    o, lse = attn(w)
    s = float(np.float32(w.scale))
    for tile in (1, 3, 16, 64):
        for rows, q, k, v, mask in dense_problems(w):
            z = s * (q @ k.T)
            z = np.where(mask, z, -np.inf)
            R = z.shape[0]
            m = np.full(R, -np.inf)
            l = np.zeros(R)
            acc = np.zeros((R, w.d))
            for j0 in range(0, z.shape[1], tile):
                st = z[:, j0:j0 + tile]
                m_new = np.maximum(m, st.max(axis=1))
                safe = np.where(np.isinf(m_new), 0.0, m_new)
                alpha = np.exp(m - safe)
                p = np.exp(st - safe[:, None])
                l = alpha * l + p.sum(axis=1)
                acc = alpha[:, None] * acc + p @ v[j0:j0 + tile]
                m = m_new
            np.testing.assert_allclose(acc / l[:, None], o[rows], rtol=0, atol=1e-12)
            np.testing.assert_allclose(m + np.log(l), lse[rows], rtol=0, atol=1e-12)


def pin_dense_decode_equals_paged(attn):
    """A dense-cache decode and a paged decode drawn with the same arguments hold the same
    keys in different places, so they give the same results bit for bit (each sums its keys
    in key order)."""
    for lens in ([1, 63, 130], [64, 65, 7, 300]):
        d = I.dense_decode_workload(13, len(lens), 0, 0, 8, 2, 16, context_lens=lens)
        pg = I.paged_decode_workload(13, len(lens), 0, 0, 8, 2, 16, page_size=8,
                                     spare_pages=5, context_lens=lens)
        od, ld = attn(d)
        op, lp = attn(pg)
        assert np.array_equal(od, op)
        assert np.array_equal(ld, lp)


def pin_closed_form_golden(attn):
    g = json.load(open(os.path.join(GOLDEN, "closed_form_2x2.json")))
    inp = g["inputs"]
    kinds = {"none": I.MASK_NONE, "causal": I.MASK_CAUSAL, "sliding": I.MASK_SLIDING}
    for case in g["cases"]:
        w = I.dense_workload(0, 1, 1, 1, 2, 2, kinds[case["mask"]], window=case["window"])
        w.scale = inp["scale"]
        w.q[0, 0] = bf16(inp["q"])
        w.k[0, 0] = bf16(inp["k"])
        w.v[0, 0] = bf16(inp["v"])
        o, lse = attn(w)
        np.testing.assert_allclose(o, np.array(case["o"]), rtol=0, atol=1e-15)
        np.testing.assert_allclose(lse, np.array(case["lse"]), rtol=0, atol=1e-15)


def all_pins():
    """(name, callable(attn)) for every pin, each kind where it applies."""
    pins = []
    for kind in KINDS:
        for f in (pin_brute_force, pin_q_zero_mean, pin_dominant_logit, pin_probabilities,
                  pin_single_key_rows, pin_constant_values, pin_logit_shift,
                  pin_gqa_equals_repeated_mha, pin_online_recurrence):
            pins.append((f"{f.__name__}[{kind}]", (lambda f, kind: lambda a: f(a, kind))(f, kind)))
    for f in (pin_key_permutation, pin_window_covering_equals_causal,
              pin_single_segment_equals_causal, pin_paged_equals_dense_last_row,
              pin_dense_decode_equals_paged, pin_bidir_window_limits, pin_prefix_limits,
              pin_document_bidir_segments, pin_paged_prefill_whole_context_equals_document,
              pin_paged_prefill_last_row_equals_decode, pin_paged_prefill_page_size_invariant,
              pin_closed_form_golden):
        pins.append((f.__name__, f))
    return pins
