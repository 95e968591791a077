"""C-ABI library checks that need no GPU: it builds for sm_103a, loads, exports every symbol
include/attn.h declares, rejects bad arguments before touching CUDA, and its tile scheduler is
exact (checked exhaustively against the mask definitions on small tiles)."""
import ctypes
import itertools

import numpy as np
import pytest

from tiled_attention_gb300 import attn, build

NONE, CAUSAL, SLIDING, DOCUMENT = 0, 1, 2, 3
SLIDING_BIDIR, DOCUMENT_BIDIR, PREFIX_LM = 6, 7, 8


@pytest.fixture(scope="module", autouse=True)
def library():
    build.build()
    return attn.lib()


def test_exports_every_declared_symbol():
    names = attn.declared_functions()
    assert len(names) >= 10
    L = attn.lib()
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(attn._SIGS), "binding and header disagree"


def test_version():
    assert attn.attn_version() == 1


def _call(**kw):
    a = dict(q=None, k=None, v=None, o=None, lse=None, B=1, Hq=1, Hkv=1, N=128, d=128,
             scale=0.125, mask_kind=CAUSAL, window=0, cu_seqlens=None, block_table=None,
             page_size=0, num_pages=0, workspace=None, stream=0)
    a.update(kw)
    return attn.attn_fwd(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(mask_kind=9), attn.ATTN_ERR_INVALID),
    (dict(mask_kind=-1), attn.ATTN_ERR_INVALID),
    (dict(mask_kind=SLIDING_BIDIR, window=-1), attn.ATTN_ERR_INVALID),
    (dict(mask_kind=PREFIX_LM, window=-3), attn.ATTN_ERR_INVALID),
    (dict(mask_kind=DOCUMENT_BIDIR), attn.ATTN_ERR_INVALID),  # no cu_seqlens
    (dict(Hq=6, Hkv=4), attn.ATTN_ERR_INVALID),
    (dict(d=96), attn.ATTN_ERR_UNSUPPORTED),
    (dict(d=256), attn.ATTN_ERR_UNSUPPORTED),
    (dict(scale=float("nan")), attn.ATTN_ERR_INVALID),
    (dict(scale=-1.0), attn.ATTN_ERR_UNSUPPORTED),
    (dict(mask_kind=SLIDING, window=0), attn.ATTN_ERR_INVALID),
    (dict(mask_kind=DOCUMENT), attn.ATTN_ERR_INVALID),
    (dict(mask_kind=attn.ATTN_MASK_DECODE), attn.ATTN_ERR_INVALID),  # no cu_seqlens
    (dict(B=-1), attn.ATTN_ERR_INVALID),
    (dict(Hkv=0), attn.ATTN_ERR_INVALID),
])
def test_invalid_arguments_are_rejected_without_cuda(kw, code):
    assert _call(**kw) == code
    assert attn.last_error()


def test_empty_problem_is_a_no_op():
    assert _call(B=0) == attn.ATTN_OK
    assert _call(N=0) == attn.ATTN_OK


def test_null_tensors_rejected():
    assert _call() == attn.ATTN_ERR_INVALID


class _FakeDevicePtr:
    """Stands in for a device tensor in calls that must fail validation before any CUDA
    call: non-null and 16-byte aligned, never dereferenced."""

    def __init__(self, addr=1 << 20):
        self.addr = addr

    def data_ptr(self):
        return self.addr


def test_decode_validation_before_cuda():
    t = _FakeDevicePtr()
    base = dict(q=t, k=t, v=t, o=t, lse=t, cu_seqlens=t, N=256)
    # more than 16 query heads per kv head: larger than one MMA tile of heads
    assert _call(mask_kind=attn.ATTN_MASK_DECODE, Hq=17, Hkv=1, **base) == attn.ATTN_ERR_UNSUPPORTED
    # three query heads per kv head are served (here the missing workspace is reported)
    assert _call(mask_kind=attn.ATTN_MASK_DECODE, Hq=3, Hkv=1, **base) == attn.ATTN_ERR_WORKSPACE
    # workspace missing
    assert (_call(mask_kind=attn.ATTN_MASK_DECODE, Hq=4, Hkv=1, **base)
            == attn.ATTN_ERR_WORKSPACE)
    # paged decode still needs its block table
    assert (_call(mask_kind=attn.ATTN_MASK_PAGED_DECODE, Hq=4, Hkv=1, page_size=64,
                  num_pages=4, **base) == attn.ATTN_ERR_INVALID)


def _paged_prefill(**kw):
    t = _FakeDevicePtr()
    a = dict(q=t, k=t, v=t, o=t, lse=t, B=2, Hq=4, Hkv=2, total_q=300, d=128, scale=0.125,
             cu_seqlens_q=t, seqlens_k=t, block_table=t, max_pages=8, page_size=16,
             num_pages=40, stream=0)
    a.update(kw)
    return attn.attn_fwd_paged_prefill(**a)


@pytest.mark.parametrize("kw,code", [
    (dict(page_size=48), attn.ATTN_ERR_UNSUPPORTED),
    (dict(page_size=8), attn.ATTN_ERR_UNSUPPORTED),
    (dict(d=96), attn.ATTN_ERR_UNSUPPORTED),
    (dict(Hq=3), attn.ATTN_ERR_INVALID),
    (dict(scale=-0.5), attn.ATTN_ERR_UNSUPPORTED),
    (dict(block_table=None), attn.ATTN_ERR_INVALID),
    (dict(seqlens_k=None), attn.ATTN_ERR_INVALID),
    (dict(max_pages=0), attn.ATTN_ERR_INVALID),
    (dict(num_pages=0), attn.ATTN_ERR_INVALID),
    (dict(num_pages=2**30, Hkv=4, Hq=4), attn.ATTN_ERR_UNSUPPORTED),
    (dict(q=_FakeDevicePtr(1 << 20 | 8)), attn.ATTN_ERR_INVALID),  # misaligned
])
def test_paged_prefill_validation_before_cuda(kw, code):
    assert _paged_prefill(**kw) == code
    assert attn.last_error()


def test_paged_prefill_empty_is_a_no_op():
    assert _paged_prefill(B=0) == attn.ATTN_OK
    assert _paged_prefill(total_q=0) == attn.ATTN_OK


def test_attn_fwd_rejects_paged_prefill_kind():
    assert _call(mask_kind=attn.ATTN_MASK_PAGED_PREFILL) == attn.ATTN_ERR_INVALID


def test_paged_decode_page_sizes():
    t = _FakeDevicePtr()
    base = dict(q=t, k=t, v=t, o=t, lse=t, cu_seqlens=t, block_table=t, N=256, Hq=4, Hkv=1,
                num_pages=8, mask_kind=attn.ATTN_MASK_PAGED_DECODE)
    for ps in (8, 48, 256):
        assert _call(page_size=ps, **base) == attn.ATTN_ERR_UNSUPPORTED
    for ps in (16, 32, 64, 128):  # valid sizes get as far as the missing workspace
        assert _call(page_size=ps, **base) == attn.ATTN_ERR_WORKSPACE
    # the split-KV scratch does not depend on the page size
    sizes = {attn.attn_workspace_bytes(32, 32, 8, 16384, 128, 4, ps) for ps in (16, 32, 64, 128)}
    assert len(sizes) == 1


def test_fp8_validation_before_cuda():
    t = _FakeDevicePtr()
    base = dict(q8=t, k8=t, v=t, o=t, lse=t, q_scales=t, k_scales=t, B=1, Hq=4, Hkv=2, N=256,
                d=128, scale=0.1, mask_kind=CAUSAL, window=0, stream=0)

    def call(**kw):
        a = dict(base)
        a.update(kw)
        return attn.attn_fwd_fp8(**a)
    assert call(d=64) == attn.ATTN_ERR_UNSUPPORTED
    assert call(mask_kind=DOCUMENT) == attn.ATTN_ERR_UNSUPPORTED
    assert call(mask_kind=attn.ATTN_MASK_PAGED_DECODE) == attn.ATTN_ERR_UNSUPPORTED
    assert call(mask_kind=42) == attn.ATTN_ERR_INVALID
    assert call(q_scales=None) == attn.ATTN_ERR_INVALID
    assert call(mask_kind=SLIDING, window=0) == attn.ATTN_ERR_INVALID
    assert call(Hq=3) == attn.ATTN_ERR_INVALID
    assert call(B=0) == attn.ATTN_OK
    assert attn.attn_quantize_fp8(t, t, t, 4, 100, 96, 0) == attn.ATTN_ERR_UNSUPPORTED
    assert attn.attn_quantize_fp8(t, t, t, 70000, 100, 128, 0) == attn.ATTN_ERR_UNSUPPORTED
    assert attn.attn_quantize_fp8(None, t, t, 4, 100, 128, 0) == attn.ATTN_ERR_INVALID
    assert attn.attn_quantize_fp8(t, t, t, 0, 100, 128, 0) == attn.ATTN_OK


def test_workspace_bytes():
    assert attn.attn_workspace_bytes(4, 16, 16, 2048, 128, CAUSAL, 0) == 0
    n = attn.attn_workspace_bytes(32, 32, 8, 16384, 128, 4, 64)
    # 256 (sequence, kv head) groups, at least one per SM: splits of 32 stages of 64 tokens,
    # 8 splits of a 16384-token context. Partial O for 8 splits x 4 heads x 128 columns per
    # group, plus stats and tickets.
    assert 32 * 8 * 8 * 4 * 128 * 4 <= n < 32 * 8 * 8 * 4 * 130 * 4 + 4096
    # fewer groups than SMs: 1 sequence x 8 kv heads, splits of 16 stages (16 splits)
    m = attn.attn_workspace_bytes(1, 32, 8, 16384, 128, 4, 64)
    assert 8 * 16 * 4 * 128 * 4 <= m < 8 * 16 * 4 * 130 * 4 + 4096
    # the dense-cache decode splits the same way and ignores page_size
    assert attn.attn_workspace_bytes(32, 32, 8, 16384, 128, attn.ATTN_MASK_DECODE, 0) == n


# ---------------------------------------------------------------- tile scheduler

def visible(mask, W, k_org, k_end, i, j):
    """Key j visible to query row i (keys and rows share one index space)."""
    if j < k_org or j >= k_end:
        return False
    if mask in (NONE, DOCUMENT_BIDIR):
        return True
    if mask == CAUSAL or mask == DOCUMENT:
        return j <= i
    if mask == SLIDING_BIDIR:
        return i - W <= j <= i + W
    if mask == PREFIX_LM:
        return j <= i or j < W
    return i - W < j <= i


def check_schedule(mask, W, r0, bm, row_end, k_org, k_end, bn):
    lo, hi = attn.attn_plan_kv_range(mask, W, r0, bm, row_end, k_org, k_end, bn)
    rows = range(r0, min(r0 + bm, row_end))
    ntiles = (k_end - k_org + bn - 1) // bn + 2
    nonempty = []
    for t in range(-1, ntiles):
        keys = range(k_org + t * bn, k_org + (t + 1) * bn)
        vis = [[visible(mask, W, k_org, k_end, i, j) for j in keys] for i in rows]
        anyv = any(any(r) for r in vis)
        allv = len(rows) > 0 and all(all(r) for r in vis)
        if t >= 0:
            kind = attn.attn_plan_tile_kind(mask, W, r0, bm, row_end, k_org, k_end, bn, t)
            want = 0 if not anyv else (1 if allv else 2)
            assert kind == want, (mask, W, r0, bm, row_end, k_org, k_end, bn, t, kind, want)
        if anyv:
            nonempty.append(t)
    if nonempty:
        assert (lo, hi) == (min(nonempty), max(nonempty) + 1)
        assert nonempty == list(range(lo, hi)), "visible tiles must be contiguous"
    else:
        assert hi <= lo


@pytest.mark.parametrize("bm,bn", [(4, 4), (4, 8), (8, 4), (3, 5)])
def test_schedule_dense_exhaustive(bm, bn):
    for N in range(1, 23):
        for r0 in range(0, N, bm):
            check_schedule(NONE, 0, r0, bm, N, 0, N, bn)
            check_schedule(CAUSAL, 0, r0, bm, N, 0, N, bn)
            for W in (1, 2, 3, 4, 5, 7, 8, 9, N, N + 3):
                check_schedule(SLIDING, W, r0, bm, N, 0, N, bn)
            for W in (0, 1, 2, 3, 4, 5, 8, 9, N, N + 3, 2**31 - 1):
                check_schedule(SLIDING_BIDIR, W, r0, bm, N, 0, N, bn)
            for P in (0, 1, 2, 3, 4, 5, 8, 9, N - 1, N, N + 3):
                check_schedule(PREFIX_LM, max(P, 0), r0, bm, N, 0, N, bn)


@pytest.mark.parametrize("bm,bn", [(4, 4), (4, 8), (8, 4)])
def test_schedule_document_exhaustive(bm, bn):
    cu = [0, 1, 3, 8, 9, 17, 30]
    for s in range(len(cu) - 1):
        for r0 in range(cu[s], cu[s + 1], bm):
            check_schedule(DOCUMENT, 0, r0, bm, cu[s + 1], cu[s], cu[s + 1], bn)
            check_schedule(DOCUMENT_BIDIR, 0, r0, bm, cu[s + 1], cu[s], cu[s + 1], bn)


def test_schedule_kernel_tile_sizes():
    """128 x 128 tiles (the kernels' sizes) on ragged sizes, spot-checked per tile."""
    for N in (1, 127, 128, 129, 300):
        for r0 in range(0, N, 128):
            check_schedule(CAUSAL, 0, r0, 128, N, 0, N, 128)
            check_schedule(NONE, 0, r0, 128, N, 0, N, 128)
            for W in (1, 127, 128, 129, 200):
                check_schedule(SLIDING, W, r0, 128, N, 0, N, 128)
                check_schedule(SLIDING_BIDIR, W, r0, 128, N, 0, N, 128)
                check_schedule(PREFIX_LM, W, r0, 128, N, 0, N, 128)


def test_plan_rejects_decode_kinds_and_bad_windows():
    for kind in (attn.ATTN_MASK_PAGED_DECODE, attn.ATTN_MASK_DECODE, 9):
        with pytest.raises(attn.AttnError):
            attn.attn_plan_kv_range(kind, 1, 0, 128, 256, 0, 256, 128)
        assert attn.attn_plan_tile_kind(kind, 1, 0, 128, 256, 0, 256, 128, 0) < 0
    with pytest.raises(attn.AttnError):
        attn.attn_plan_kv_range(SLIDING_BIDIR, -1, 0, 128, 256, 0, 256, 128)


def test_schedule_bidir_and_prefix_shapes():
    """Two-sided window 2048 at N=8192 with 128-wide tiles: 33 key tiles away from the ends,
    two of them boundary tiles; prefix 4096: the first 16 query tiles read the 32 prefix
    tiles, all full except the diagonal ones past the prefix."""
    for r in range(64):
        lo, hi = attn.attn_plan_kv_range(SLIDING_BIDIR, 2048, 128 * r, 128, 8192, 0, 8192, 128)
        kinds = [attn.attn_plan_tile_kind(SLIDING_BIDIR, 2048, 128 * r, 128, 8192, 0, 8192,
                                          128, t) for t in range(lo, hi)]
        if 16 <= r < 48:
            assert (lo, hi) == (r - 16, r + 17)
        assert kinds.count(2) <= 2 and 0 not in kinds
    for r in range(64):
        lo, hi = attn.attn_plan_kv_range(PREFIX_LM, 4096, 128 * r, 128, 8192, 0, 8192, 128)
        assert (lo, hi) == (0, max(32, r + 1))
        kinds = [attn.attn_plan_tile_kind(PREFIX_LM, 4096, 128 * r, 128, 8192, 0, 8192, 128, t)
                 for t in range(lo, hi)]
        assert kinds == ([1] * 32 if r < 32 else [1] * r + [2])


def test_schedule_skips_masked_tiles():
    """Causal N=2048: 8 query-tile pairs; tile row r sees r+1 key tiles, one boundary."""
    total = 0
    for r in range(16):
        lo, hi = attn.attn_plan_kv_range(CAUSAL, 0, 128 * r, 128, 2048, 0, 2048, 128)
        assert (lo, hi) == (0, r + 1)
        kinds = [attn.attn_plan_tile_kind(CAUSAL, 0, 128 * r, 128, 2048, 0, 2048, 128, t)
                 for t in range(16)]
        assert kinds == [1] * r + [2] + [0] * (15 - r)
        total += hi - lo
    assert total == 136
    # Sliding window 4096 at N=8192: at most 33 key tiles, at most 2 boundary tiles.
    for r in range(64):
        lo, hi = attn.attn_plan_kv_range(SLIDING, 4096, 128 * r, 128, 8192, 0, 8192, 128)
        kinds = [attn.attn_plan_tile_kind(SLIDING, 4096, 128 * r, 128, 8192, 0, 8192, 128, t)
                 for t in range(lo, hi)]
        assert hi - lo <= 33 and kinds.count(2) <= 2 and 0 not in kinds


@pytest.mark.parametrize("kind", [NONE, CAUSAL, SLIDING_BIDIR, PREFIX_LM])
def test_units_dense_order_and_cover(kind):
    B, Hq, N = 2, 3, 700
    u = attn.attn_plan_units(kind, B, Hq, N)
    npairs = (N + 255) // 256
    assert len(u) == B * Hq * npairs
    assert sorted(u) == sorted(itertools.product(range(B), range(Hq), range(npairs)))
    levels = [t for _, _, t in u]
    assert levels == sorted(levels, reverse=True)


def test_units_paged_prefill_order_and_cover():
    """Chunk units: every (sequence, head, pair of the chunk) once, ordered by pair index plus
    the pairs of context before the chunk, descending."""
    lq = np.array([1, 300, 0, 2048, 700])
    lk = np.array([5000, 300, 10, 2100, 16384])
    cu = np.concatenate([[0], np.cumsum(lq)]).astype(np.int32)
    Hq = 2
    u = attn.attn_plan_units(attn.ATTN_MASK_PAGED_PREFILL, len(lq), Hq, int(cu[-1]), cu, lk)
    want = [(s, h, t) for s in range(len(lq)) for h in range(Hq)
            for t in range((int(lq[s]) + 255) // 256)]
    assert sorted(u) == sorted(want)
    levels = [t + (int(lk[s]) - int(lq[s])) // 256 for s, _, t in u]
    assert levels == sorted(levels, reverse=True)
    bad = np.array([0, 5, 10], dtype=np.int32)  # second chunk longer than its context
    with pytest.raises(attn.AttnError):
        attn.attn_plan_units(attn.ATTN_MASK_PAGED_PREFILL, 2, 1, 10, bad, np.array([5, 4]))


def test_units_document_order_and_cover():
    cu = np.array([0, 5, 600, 601, 1400, 1400, 1700], dtype=np.int32)
    Hq = 2
    u = attn.attn_plan_units(DOCUMENT, len(cu) - 1, Hq, int(cu[-1]), cu)
    want = [(s, h, t) for s in range(len(cu) - 1) for h in range(Hq)
            for t in range((int(cu[s + 1] - cu[s]) + 255) // 256)]
    assert sorted(u) == sorted(want)
    levels = [t for _, _, t in u]
    assert levels == sorted(levels, reverse=True)
    # within a level: segments ascending, then heads
    for t in set(levels):
        same = [(s, h) for s, h, tt in u if tt == t]
        assert same == sorted(same)


def test_units_document_bidir_sorted_by_cost():
    """Non-causal segments: every unit once, in decreasing cost (key tiles of its two query
    tiles, from the scheduler's own ranges); equal costs by segment, pair, then head."""
    cu = np.array([0, 5, 600, 601, 1400, 1400, 1700, 2000, 2129], dtype=np.int32)
    Hq = 2
    u = attn.attn_plan_units(DOCUMENT_BIDIR, len(cu) - 1, Hq, int(cu[-1]), cu)
    want = [(s, h, t) for s in range(len(cu) - 1) for h in range(Hq)
            for t in range((int(cu[s + 1] - cu[s]) + 255) // 256)]
    assert sorted(u) == sorted(want)

    def cost(s, t):
        k0, k1 = int(cu[s]), int(cu[s + 1])
        c = 0
        for i in range(2):
            r0 = k0 + 256 * t + 128 * i
            if r0 < k1:
                lo, hi = attn.attn_plan_kv_range(DOCUMENT_BIDIR, 0, r0, 128, k1, k0, k1, 128)
                c += hi - lo
        return c

    keys = [(-cost(s, t), s, t, h) for s, h, t in u]
    assert keys == sorted(keys)
    # the 129-row segment: one pair of one tile plus a one-row tile, cost 2 + 2 = 4;
    # the 300-row segment's last pair has one tile of three: cost 3
    assert cost(7, 0) == 4 and cost(5, 1) == 3


@pytest.mark.parametrize("blocks,iters", [(0, 10), (-1, 10), (70000, 10), (4, 0), (4, 1 << 21)])
def test_bench_ex2_rejects_bad_arguments(blocks, iters):
    """Argument checks run before any launch, so they need no GPU."""
    fake = ctypes.c_void_p(256)  # never dereferenced: the call fails before launching
    assert attn.lib().attn_bench_ex2(fake, blocks, iters, None) == attn.ATTN_ERR_INVALID
    assert attn.lib().attn_bench_ex2(None, 4, 10, None) == attn.ATTN_ERR_INVALID
