"""CUDA path against the fp64 oracle, element by element, through the C ABI.

Tolerances: max |O - O_ref| <= 1e-2 (bf16 inputs and output, fp32 accumulation) and
max |LSE - LSE_ref| <= 1e-3 on the five specified workloads. The ragged sweeps include rows
that see only one or two keys, where |O| can reach ~3 and bf16 arithmetic alone exceeds a flat
1e-2: the stored O is rounded to bf16 (error <= 2^-9 |O|) and P enters the P.V product as
bf16 (error <= 2^-9 max|v|). Those sweeps use |O - O_ref| <= 1e-2 + 2^-8 |O_ref|, which covers
both terms for |v| <= 5. Outputs are pre-filled with NaN so a row the kernels never write fails
loudly.
"""
import numpy as np
import pytest
import torch

import oracle
from tiled_attention_gb300 import attn
from tiled_attention_gb300 import inputs as I
from tiled_attention_gb300.runner import DeviceProblem, bf16_tensor

pytestmark = pytest.mark.gpu

O_TOL = 1e-2
LSE_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def cuda_library():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from tiled_attention_gb300 import build
    build.build()
    attn.lib()
    torch.cuda.synchronize()
    assert attn.attn_get_status() == 0


def run(w, stream=None):
    dp = DeviceProblem(w)
    rc = dp.run(stream)
    assert rc == 0, attn.last_error()
    torch.cuda.synchronize()
    status = attn.attn_get_status()
    assert status == 0, f"device status {status}"
    return dp


def compare(w, dp, rows=None, strict=True):
    o, lse = dp.outputs()
    ro, rl = oracle.attention(w, rows=rows)
    if rows is not None:
        o, lse = o[rows], lse[rows]
    assert np.isfinite(o).all() and np.isfinite(lse).all(), "unwritten or non-finite outputs"
    eo = np.abs(o - ro)
    el = np.abs(lse - rl)
    tol = O_TOL if strict else O_TOL + 2.0 ** -8 * np.abs(ro)
    worst = np.unravel_index(np.argmax(eo - tol), eo.shape)
    msg = (f"{w.name}: max|dO|={eo.max():.3e}, worst vs bound at row {worst[0]} "
           f"(|O|={abs(ro[worst]):.3f}, dO={eo[worst]:.3e}), max|dLSE|={el.max():.3e}")
    assert np.all(eo <= tol) and el.max() <= LSE_TOL, msg
    return eo.max(), el.max()


# ------------------------------------------------------------------ the five workloads

def test_dense_b1_h1_n256_d64():
    w = I.config(1)
    compare(w, run(w))


def test_causal_b4_h16_n2048_d128():
    w = I.config(2)
    compare(w, run(w))


def test_sliding_w4096_b2_hq32_hkv8_n8192_d128():
    """Every one of the 524,288 output rows against the oracle."""
    w = I.config(3)
    compare(w, run(w))


def test_document_t16384_h16_d64():
    w = I.config(4)
    compare(w, run(w))


@pytest.mark.parametrize("cfg", ["5b1", "5b4"])
def test_small_batch_paged_decode(cfg):
    """One and four sequences: few (sequence, kv head) groups, so each context is split over
    many CTAs and merged; every output row against the oracle, and a second launch on the same
    inputs gives the same bits (the merge runs in a fixed split order)."""
    w = I.config(cfg)
    dp = run(w)
    compare(w, dp)
    o1, l1 = dp.o.view(torch.int16).clone(), dp.lse.clone()
    dp.o.fill_(float("nan"))
    assert dp.run() == 0, attn.last_error()
    torch.cuda.synchronize()
    assert attn.attn_get_status() == 0
    assert torch.equal(dp.o.view(torch.int16), o1) and torch.equal(dp.lse, l1)


def test_paged_decode_b32_hq32_hkv8_d128_page64():
    w = I.config(5)
    compare(w, run(w))


def test_headline_causal_n8192():
    """The causal B2 Hq32 Hkv8 N8192 d128 shape the throughput is quoted on, in the launch
    configuration the benchmark times: every one of the 524,288 output rows."""
    w = I.config("3c")
    compare(w, run(w))


# ------------------------------------------------------------------ ragged sweeps

@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N", [1, 17, 127, 128, 129, 255, 256, 257, 300, 640])
@pytest.mark.parametrize("mask", [I.MASK_NONE, I.MASK_CAUSAL])
def test_dense_ragged(d, N, mask):
    w = I.dense_workload(100 + N, 2, 4, 2, N, d, mask)
    compare(w, run(w), strict=False)


@pytest.mark.parametrize("mask,window", [(I.MASK_NONE, 0), (I.MASK_CAUSAL, 0),
                                         (I.MASK_SLIDING, 95), (I.MASK_SLIDING, 97),
                                         (I.MASK_SLIDING, 192), (I.MASK_SLIDING_BIDIR, 96),
                                         (I.MASK_PREFIX_LM, 97)])
@pytest.mark.parametrize("N", [95, 96, 97, 191, 193, 287, 289, 385, 577])
def test_d64_key_tile_edges(mask, window, N):
    """d = 64 runs on 96-key tiles against 128-row query tiles: lengths, windows and prefixes
    on either side of multiples of 96 put the diagonal and the window edges at every offset
    inside a key tile, and key tiles across the query tiles' boundaries."""
    w = I.dense_workload(700 + N + window, 2, 4, 2, N, 64, mask, window=window)
    compare(w, run(w), strict=False)


@pytest.mark.parametrize("lens", [[96, 95, 97], [192, 1, 288, 96], [383, 385, 96, 97, 191]])
@pytest.mark.parametrize("mask", [I.MASK_DOCUMENT, I.MASK_DOCUMENT_BIDIR])
def test_d64_document_key_tile_edges(mask, lens):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    w = I.document_workload(800 + len(lens), int(cu[-1]), 4, 64, cu_seqlens=cu, Hkv=1,
                            mask_kind=mask)
    compare(w, run(w), strict=False)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("W", [1, 2, 127, 128, 129, 300, 1000])
def test_sliding_ragged(d, W):
    w = I.dense_workload(200 + W, 1, 4, 1, 777, d, I.MASK_SLIDING, window=W)
    compare(w, run(w), strict=False)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("lens", [[1], [2, 1, 127], [129, 256, 1, 300], [600, 5, 257, 128, 384]])
def test_document_ragged(d, lens):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    w = I.document_workload(300 + len(lens), int(cu[-1]), 4, d, cu_seqlens=cu, Hkv=2)
    compare(w, run(w), strict=False)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("W", [0, 1, 2, 127, 128, 129, 300, 1000])
def test_sliding_bidir_ragged(d, W):
    w = I.dense_workload(600 + W, 1, 4, 2, 777, d, I.MASK_SLIDING_BIDIR, window=W)
    compare(w, run(w), strict=False)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("P", [0, 1, 100, 128, 129, 500, 777, 1000])
def test_prefix_lm_ragged(d, P):
    w = I.dense_workload(700 + P, 1, 4, 2, 777, d, I.MASK_PREFIX_LM, window=P)
    compare(w, run(w), strict=False)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("lens", [[1], [2, 1, 127], [129, 256, 1, 300], [600, 5, 257, 128, 384]])
def test_document_bidir_ragged(d, lens):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    w = I.document_workload(800 + len(lens), int(cu[-1]), 4, d, cu_seqlens=cu, Hkv=2,
                            mask_kind=I.MASK_DOCUMENT_BIDIR)
    compare(w, run(w), strict=False)


@pytest.mark.parametrize("cfg", ["3b", "3p"])
def test_mask_variant_workloads_sampled(cfg):
    """The two-sided window and prefix-LM workloads at full size, in the launch configuration
    the benchmark suite times, on sampled rows (both sequence ends, the window and prefix
    edges, and random rows)."""
    w = I.config(cfg)
    dp = run(w)
    rng = np.random.default_rng(8)
    n = int(np.prod(w.lse_shape))
    heads = np.arange(w.B * w.Hq) * w.N
    rows = np.unique(np.concatenate([rng.integers(0, n, 2000), heads, heads + w.N - 1,
                                     heads + w.window - 1, heads + w.window,
                                     heads + w.N - 1 - w.window]))
    compare(w, dp, rows=rows)


def test_document_bidir_workload():
    w = I.config("4b")
    compare(w, run(w))


def test_bidir_window_covering_equals_none_bit_exact():
    """A two-sided window reaching every key makes every key tile full, so the kernel does
    exactly what the unmasked kernel does."""
    a = I.dense_workload(31, 1, 4, 2, 600, 128, I.MASK_NONE)
    b = I.dense_workload(31, 1, 4, 2, 600, 128, I.MASK_SLIDING_BIDIR, window=600)
    ra, rb = run(a), run(b)
    assert torch.equal(ra.o.view(torch.int16), rb.o.view(torch.int16))
    assert torch.equal(ra.lse, rb.lse)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("group", [1, 2, 3, 4, 5, 6, 8, 12, 16])
def test_paged_ragged(d, group):
    lens = [1, 63, 64, 65, 1000, 1025, 2048, 3000]
    w = I.paged_decode_workload(400 + group, len(lens), 0, 0, 2 * group, 2, d,
                                context_lens=lens)
    compare(w, run(w), strict=False)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("group", [1, 3, 4, 6, 11, 16])
def test_dense_decode_ragged(d, group):
    """Decode on dense per-sequence caches; the cache is longer than every context and its
    tail holds poison, so reading past L_b would show."""
    lens = [1, 63, 64, 65, 1000, 1025, 2048, 3000]
    w = I.dense_decode_workload(500 + group, len(lens), 0, 0, 2 * group, 2, d, N=3100,
                                context_lens=lens)
    compare(w, run(w), strict=False)


@pytest.mark.parametrize("page_size", [16, 32, 128])
@pytest.mark.parametrize("d", [64, 128])
def test_paged_decode_page_sizes(d, page_size):
    lens = [1, 15, 16, 17, 63, 64, 65, 127, 128, 129, 1000, 3000]
    w = I.paged_decode_workload(450 + page_size, len(lens), 0, 0, 8, 2, d,
                                page_size=page_size, context_lens=lens)
    compare(w, run(w), strict=False)


def test_paged_decode_page_size_invariant_bit_exact():
    """The same tokens in pools of 16-, 32-, 64- and 128-token pages fill the decode's
    64-token stages identically, so the results agree bit for bit."""
    lens = [1, 100, 2000, 777]
    outs = []
    for ps in (16, 32, 64, 128):
        w = I.paged_decode_workload(46, len(lens), 0, 0, 16, 4, 128, page_size=ps,
                                    context_lens=lens)
        dp = run(w)
        outs.append((dp.o.view(torch.int16).clone(), dp.lse.clone()))
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])


# ------------------------------------------------------------------ chunked prefill, paged KV

@pytest.mark.parametrize("page_size", [16, 32, 64, 128])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("group", [1, 4])
def test_paged_prefill_ragged(d, page_size, group):
    """Contexts and chunks of ragged lengths (chunk = whole context, single tokens, chunks
    crossing tile and page edges); pool tails and spare pages hold poison."""
    lk = [1, 40, 300, 1000, 2100, 129, 777]
    lq = [1, 40, 129, 1, 700, 128, 300]
    w = I.paged_prefill_workload(900 + page_size + group, len(lk), 0, 0, 0, 0, 2 * group, 2, d,
                                 page_size=page_size, context_lens=lk, chunk_lens=lq)
    compare(w, run(w), strict=False)


def test_paged_prefill_whole_context_equals_document_bit_exact():
    """A chunk that is the whole context runs the same tiles and masks as the causal document
    kernel on the gathered tokens."""
    lens = [300, 129, 700, 1]
    w = I.paged_prefill_workload(47, len(lens), 0, 0, 0, 0, 8, 2, 128, page_size=16,
                                 context_lens=lens, chunk_lens=lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    dw = I.document_workload(0, int(cu[-1]), 8, 128, cu_seqlens=cu, Hkv=2)
    dw.q[...] = w.q
    for b, L in enumerate(lens):
        pages = [int(w.block_table[b, p]) for p in range((L + 15) // 16)]
        dw.k[0, :, cu[b]:cu[b + 1]] = np.concatenate([w.k[p] for p in pages], axis=1)[:, :L]
        dw.v[0, :, cu[b]:cu[b + 1]] = np.concatenate([w.v[p] for p in pages], axis=1)[:, :L]
    a, b = run(w), run(dw)
    assert torch.equal(a.o.view(torch.int16), b.o.view(torch.int16))
    assert torch.equal(a.lse, b.lse)


def test_paged_prefill_page_size_invariant_bit_exact():
    lk, lq = [1000, 50, 3000], [333, 50, 1]
    outs = []
    for ps in (16, 64, 128):
        w = I.paged_prefill_workload(48, 3, 0, 0, 0, 0, 8, 2, 128, page_size=ps,
                                     context_lens=lk, chunk_lens=lq)
        dp = run(w)
        outs.append((dp.o.view(torch.int16).clone(), dp.lse.clone()))
    for o, l in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(l, outs[0][1])


@pytest.mark.parametrize("cfg", ["6", "6p64"])
def test_chunked_prefill_workload_sampled(cfg):
    """Full-size chunked prefill in the launch configuration the benchmark suite times:
    sampled rows (each chunk's first and last rows, and random rows)."""
    w = I.config(cfg)
    dp = run(w)
    rng = np.random.default_rng(9)
    n = int(np.prod(w.lse_shape))
    firsts = w.cu_seqlens[:-1].astype(np.int64)
    lasts = w.cu_seqlens[1:].astype(np.int64) - 1
    heads = np.arange(w.Hq)[:, None] * w.N
    rows = np.unique(np.concatenate([rng.integers(0, n, 1500), (heads + firsts).ravel(),
                                     (heads + lasts).ravel()]))
    compare(w, dp, rows=rows)


def test_paged_prefill_bad_table_entry_reports_bounds():
    w = I.paged_prefill_workload(49, 2, 0, 0, 0, 0, 4, 2, 128, page_size=16,
                                 context_lens=[200, 100], chunk_lens=[50, 100])
    w.block_table[1, 2] = w.k.shape[0] + 7
    dp = DeviceProblem(w)
    assert dp.run() == 0
    torch.cuda.synchronize()
    assert attn.attn_get_status() == attn.ATTN_ERR_BOUNDS
    # sequence 0 is unaffected
    rows = (np.arange(w.Hq)[:, None] * w.N + np.arange(50)[None, :]).ravel()
    compare(w, dp, rows=rows)


def test_paged_prefill_chunk_longer_than_context_reports_status():
    w = I.paged_prefill_workload(50, 2, 0, 0, 0, 0, 4, 2, 64, page_size=16,
                                 context_lens=[64, 100], chunk_lens=[64, 100])
    w.seqlens_k = np.array([64, 90], dtype=np.int32)  # chunk 100 > context 90
    dp = DeviceProblem(w)
    assert dp.run() == 0
    torch.cuda.synchronize()
    assert attn.attn_get_status() == attn.ATTN_ERR_SEQLENS


@pytest.mark.parametrize("group", [1, 3, 4, 12])
def test_dense_decode_empty_context(group):
    w = I.dense_decode_workload(9, 3, 0, 0, 2 * group, 2, 128, N=100, context_lens=[0, 70, 0])
    dp = run(w)
    o, lse = dp.outputs()
    ro, rl = oracle.attention(w)
    assert np.abs(o - ro).max() <= O_TOL
    assert np.array_equal(np.isinf(lse), np.isinf(rl))
    live = np.isfinite(rl)
    assert np.abs(lse[live] - rl[live]).max() <= LSE_TOL


def test_two_stage_paged_equals_fused():
    """Gather the pages into dense caches, then decode on them: the same pages in the same
    order through the same kernel, so the result equals the fused paged decode bit for bit."""
    lens = [1, 64, 65, 300, 1000, 4097]
    w = I.paged_decode_workload(21, len(lens), 0, 0, 16, 4, 128, context_lens=lens)
    fused = run(w)
    max_pages = w.block_table.shape[1]
    L = max_pages * 64
    kd = torch.zeros((w.B, w.Hkv, L, w.d), dtype=torch.bfloat16, device="cuda")
    vd = torch.zeros_like(kd)
    for src, dst in ((fused.k, kd), (fused.v, vd)):
        rc = attn.attn_gather_pages(src, dst, fused.table, w.B, max_pages, w.Hkv, 64, w.d,
                                    fused.num_pages)
        assert rc == 0, attn.last_error()
    o = torch.full(w.out_shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full(w.lse_shape, float("nan"), dtype=torch.float32, device="cuda")
    nbytes = attn.attn_workspace_bytes(w.B, w.Hq, w.Hkv, L, w.d, attn.ATTN_MASK_DECODE, 0)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    rc = attn.attn_fwd(fused.q, kd, vd, o, lse, w.B, w.Hq, w.Hkv, L, w.d, w.scale,
                       attn.ATTN_MASK_DECODE, 0, fused.cu, None, 0, 0, ws)
    assert rc == 0, attn.last_error()
    torch.cuda.synchronize()
    assert attn.attn_get_status() == 0
    assert torch.equal(o.view(torch.int16), fused.o.view(torch.int16))
    assert torch.equal(lse, fused.lse)


def test_dense_decode_length_past_cache_reports_status():
    w = I.dense_decode_workload(23, 2, 0, 0, 4, 1, 64, N=128, context_lens=[100, 128])
    w.cu_seqlens = np.array([0, 100, 229], dtype=np.int32)  # second length 129 > N
    dp = DeviceProblem(w)
    assert dp.run() == 0
    assert attn.attn_get_status() == attn.ATTN_ERR_SEQLENS


@pytest.mark.parametrize("group", [1, 3, 4, 12])
def test_paged_empty_context(group):
    w = I.paged_decode_workload(9, 3, 0, 0, 2 * group, 2, 128, context_lens=[0, 70, 0])
    dp = run(w)
    o, lse = dp.outputs()
    ro, rl = oracle.attention(w)
    assert np.array_equal(o, ro) or np.abs(o - ro).max() <= O_TOL
    assert np.array_equal(np.isinf(lse), np.isinf(rl))
    live = np.isfinite(rl)
    assert np.abs(lse[live] - rl[live]).max() <= LSE_TOL


@pytest.mark.parametrize("fill", ["ones", "random"])
def test_decode_workspace_needs_no_clearing(fill):
    """The split tickets are zeroed on the call's stream before each launch: a workspace holding
    anything (all-ones bytes, random bytes) gives the oracle's results, and so does the next
    call on it."""
    lens = [5000, 70, 16384, 1]
    w = I.paged_decode_workload(23, len(lens), 0, 0, 24, 4, 128, context_lens=lens)
    dp = DeviceProblem(w)
    if fill == "ones":
        dp.workspace.fill_(255)
    else:
        g = torch.Generator(device="cuda").manual_seed(5)
        dp.workspace.copy_(torch.randint(0, 256, dp.workspace.shape, generator=g,
                                         device="cuda", dtype=torch.int32).to(torch.uint8))
    for _ in range(2):
        dp.o.fill_(float("nan"))
        assert dp.run() == 0, attn.last_error()
        torch.cuda.synchronize()
        assert attn.attn_get_status() == 0
        compare(w, dp)


@pytest.mark.parametrize("d,Hq", [(128, 8), (64, 32)])
def test_paged_decode_many_splits(d, Hq):
    """Contexts of ~70K and ~20K tokens split into 69 and 20 splits of 1024 tokens: the last
    split's merge runs its max pass and several batches of 16 splits; every row against the
    oracle (groups of 4 and 16 query heads per kv head)."""
    lens = [70000, 20001]
    w = I.paged_decode_workload(31 + d, len(lens), 0, 0, Hq, 2, d, context_lens=lens)
    compare(w, run(w))


@pytest.mark.parametrize("idx", range(12))
def test_paged_decode_randomized_long(idx):
    """Batch, kv heads, group (1-16), head dim, page size and contexts of up to 40K tokens
    (up to 40 splits per group, several merge batches) drawn from a generator seeded by idx;
    every row against the oracle, and the allocation-free entry point bit-identical to
    attn_fwd whenever its scratch holds the request."""
    rng = np.random.default_rng(9000 + idx)
    B, Hkv, G = int(rng.integers(1, 9)), int(rng.integers(1, 9)), int(rng.integers(1, 17))
    d, page = int(rng.choice([64, 128])), int(rng.choice([16, 32, 64, 128]))
    lens = rng.integers(0, 40001, B)
    w = I.paged_decode_workload(9000 + idx, B, 0, 0, G * Hkv, Hkv, d, page_size=page,
                                context_lens=lens, name=f"decode fuzz {idx}")
    dp = run(w)
    compare(w, dp, strict=False)
    need = attn.attn_workspace_bytes(w.B, w.Hq, w.Hkv, w.N, w.d, w.mask_kind, w.page_size)
    if need <= attn.attn_noalloc_scratch_bytes():
        o = torch.full_like(dp.o, float("nan"))
        lse = torch.full_like(dp.lse, float("nan"))
        rc = attn.attn_paged_decode_noalloc(dp.q, dp.k, dp.v, o, lse, w.B, w.Hq, w.Hkv, w.N,
                                            w.d, w.scale, dp.cu, dp.table, w.page_size,
                                            dp.num_pages, None)
        assert rc == 0, attn.last_error()
        torch.cuda.synchronize()
        assert attn.attn_get_status() == 0
        assert torch.equal(o.view(torch.int16), dp.o.view(torch.int16))
        assert torch.equal(lse, dp.lse)


# ------------------------------------------------------------------ bit-exact properties

def test_gather_pages_bit_exact():
    w = I.paged_decode_workload(11, 5, 0, 0, 4, 2, 128, context_lens=[1, 64, 65, 300, 1000])
    dp = DeviceProblem(w)
    max_pages = w.block_table.shape[1]
    dst = torch.zeros((w.B, w.Hkv, max_pages * 64, w.d), dtype=torch.bfloat16, device="cuda")
    rc = attn.attn_gather_pages(dp.k, dst, dp.table, w.B, max_pages, w.Hkv, 64, w.d,
                                dp.num_pages)
    assert rc == 0, attn.last_error()
    torch.cuda.synchronize()
    assert attn.attn_get_status() == 0
    got = dst.view(torch.int16).cpu().numpy().view(np.uint16)
    want = np.zeros_like(got)
    for b in range(w.B):
        for p in range(max_pages):
            phys = w.block_table[b, p]
            if phys >= 0:
                want[b, :, p * 64:(p + 1) * 64] = w.k[phys]
    assert np.array_equal(got, want)


def test_paged_shuffled_equals_identity_table():
    lens = [100, 2000, 64, 1500]
    a = I.paged_decode_workload(12, 4, 0, 0, 8, 2, 128, context_lens=lens, shuffle=True)
    b = I.paged_decode_workload(12, 4, 0, 0, 8, 2, 128, context_lens=lens, shuffle=False)
    ra, rb = run(a), run(b)
    assert torch.equal(ra.o.view(torch.int16), rb.o.view(torch.int16))
    assert torch.equal(ra.lse, rb.lse)


def test_document_segment_equals_standalone_causal():
    lens = [300, 129, 700]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    w = I.document_workload(13, int(cu[-1]), 4, 128, cu_seqlens=cu, Hkv=2)
    dw = run(w)
    for s, L in enumerate(lens):
        c = I.dense_workload(0, 1, 4, 2, L, 128, I.MASK_CAUSAL)
        c.q[0] = w.q[0, :, cu[s]:cu[s + 1]]
        c.k[0] = w.k[0, :, cu[s]:cu[s + 1]]
        c.v[0] = w.v[0, :, cu[s]:cu[s + 1]]
        dc = run(c)
        assert torch.equal(dw.o[0, :, cu[s]:cu[s + 1]].view(torch.int16),
                           dc.o[0].view(torch.int16)), f"segment {s}"
        assert torch.equal(dw.lse[0, :, cu[s]:cu[s + 1]], dc.lse[0])


@pytest.mark.parametrize("cfg", [2, 4, 5])
def test_deterministic(cfg):
    w = I.config(cfg)
    dp = DeviceProblem(w)
    assert dp.run() == 0
    o1, l1 = dp.o.clone(), dp.lse.clone()
    assert dp.run() == 0
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), dp.o.view(torch.int16))
    assert torch.equal(l1, dp.lse)


# ------------------------------------------------------------------ device-side checks

def test_block_table_out_of_pool_reports_bounds():
    w = I.paged_decode_workload(14, 2, 0, 0, 4, 2, 128, context_lens=[200, 100])
    w.block_table[1, 0] = w.k.shape[0] + 5
    dp = DeviceProblem(w)
    assert dp.run() == 0
    torch.cuda.synchronize()
    assert attn.attn_get_status() == attn.ATTN_ERR_BOUNDS
    assert attn.attn_get_status() == 0  # cleared by the read
    # sequence 0 is unaffected
    o, lse = dp.outputs()
    ro, rl = oracle.attention(w, rows=np.arange(4))
    assert np.abs(o[:4] - ro).max() <= O_TOL


def test_bad_cu_seqlens_reports_status():
    cu = np.array([0, 100, 50, 300], dtype=np.int32)  # not monotone
    w = I.document_workload(15, 300, 2, 64, cu_seqlens=cu)
    dp = DeviceProblem(w)
    assert dp.run() == 0
    torch.cuda.synchronize()
    assert attn.attn_get_status() == attn.ATTN_ERR_SEQLENS


def test_bounded_wait_times_out_and_context_survives():
    """A wait on a barrier nothing arrives on gives up after its limit, records
    ATTN_ERR_TIMEOUT, and the context keeps working (a normal call right after passes)."""
    assert attn.attn_selftest_wait_timeout(20_000_000) == 0  # 20 ms
    torch.cuda.synchronize()
    assert attn.attn_get_status() == attn.ATTN_ERR_TIMEOUT
    assert attn.attn_get_status() == 0
    w = I.config(1)
    compare(w, run(w))


def test_exp2_probe_reaches_the_fixed_point():
    """The exp2 throughput probe runs eight chains x <- 2^(-x) per thread; each converges to
    the fixed point of 2^(-x) = x (0.6411857445...; the map contracts by ln2 * 0.64 = 0.44 per
    round), so every stored value is 8 times it."""
    blocks, iters = 4, 64
    out = torch.full((blocks * 256,), float("nan"), dtype=torch.float32, device="cuda")
    assert attn.attn_bench_ex2(out, blocks, iters) == 0
    torch.cuda.synchronize()
    x = 0.6411857445049859
    assert abs(2.0 ** -x - x) < 1e-12
    assert torch.allclose(out.cpu(), torch.full_like(out.cpu(), 8 * x), rtol=0, atol=2e-5)


def test_side_stream():
    w = I.config(1)
    s = torch.cuda.Stream()
    dp = DeviceProblem(w)
    torch.cuda.synchronize()
    assert dp.run(stream=s) == 0
    s.synchronize()
    compare(w, dp)


# ------------------------------------------------------------------ large and degenerate shapes

def test_long_causal_sequence_sampled():
    """One 32768-token causal sequence: 128 query-tile pairs of up to 256 key tiles each."""
    w = I.dense_workload(1201, 1, 4, 1, 32768, 128, I.MASK_CAUSAL)
    dp = run(w)
    rng = np.random.default_rng(12)
    n = int(np.prod(w.lse_shape))
    heads = np.arange(w.Hq) * w.N
    rows = np.unique(np.concatenate([rng.integers(0, n, 600), heads, heads + w.N - 1,
                                     heads + 16383, heads + 16384]))
    compare(w, dp, rows=rows)


def test_many_units_per_sm():
    """B=32, H=64 at N=512: 4096 work units, many rounds of the persistent grid."""
    w = I.dense_workload(1202, 32, 64, 16, 512, 64, I.MASK_CAUSAL)
    dp = run(w)
    rng = np.random.default_rng(13)
    rows = rng.integers(0, int(np.prod(w.lse_shape)), 3000)
    compare(w, dp, rows=rows)


def test_document_many_tiny_segments():
    """2000 segments of 1-16 tokens: the unit list scans thousands of segments."""
    rng = np.random.default_rng(14)
    lens = rng.integers(1, 17, 2000)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    w = I.document_workload(1203, int(cu[-1]), 4, 64, cu_seqlens=cu, Hkv=2)
    compare(w, run(w), strict=False)


def test_paged_decode_128k_context():
    """A 131072-token context (128 splits of 1024 tokens) next to short ones."""
    lens = [131072, 5, 4000]
    w = I.paged_decode_workload(1204, len(lens), 0, 0, 8, 2, 128, context_lens=lens)
    compare(w, run(w), strict=False)


def test_paged_prefill_empty_chunks():
    """Sequences whose chunk is empty contribute no rows and must not disturb the others."""
    lk = [500, 64, 1000, 7]
    lq = [0, 64, 0, 7]
    w = I.paged_prefill_workload(1205, len(lk), 0, 0, 0, 0, 8, 2, 128, page_size=16,
                                 context_lens=lk, chunk_lens=lq)
    compare(w, run(w), strict=False)


# ------------------------------------------------------------------ randomized shapes

_FUZZ_KINDS = [I.MASK_NONE, I.MASK_CAUSAL, I.MASK_SLIDING, I.MASK_SLIDING_BIDIR, I.MASK_PREFIX_LM,
               I.MASK_DOCUMENT, I.MASK_DOCUMENT_BIDIR, I.MASK_PAGED_DECODE, I.MASK_DECODE,
               I.MASK_PAGED_PREFILL]


def _fuzz_workload(idx):
    """Case idx: its mask kind in turn, the rest drawn from a generator seeded by idx: head dim,
    batch, GQA group (1-4 query heads per kv head for prefill, 1-16 for decode), lengths,
    windows and prefixes past the sequence, empty segments and chunks, page sizes."""
    rng = np.random.default_rng(5000 + idx)
    kind = _FUZZ_KINDS[idx % len(_FUZZ_KINDS)]
    d = int(rng.choice([64, 128]))
    Hkv = int(rng.integers(1, 4))
    decode = kind in (I.MASK_PAGED_DECODE, I.MASK_DECODE)
    Hq = Hkv * int(rng.integers(1, 17) if decode else rng.integers(1, 5))
    seed = 6000 + idx
    if kind in (I.MASK_DOCUMENT, I.MASK_DOCUMENT_BIDIR):
        lens = rng.integers(0, 400, int(rng.integers(1, 7)))
        lens[int(rng.integers(0, len(lens)))] += 1  # at least one row
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
        return I.document_workload(seed, int(cu[-1]), Hq, d, cu_seqlens=cu, Hkv=Hkv,
                                   mask_kind=kind, name=f"fuzz{idx}")
    B = int(rng.integers(1, 5))
    page = int(rng.choice([16, 32, 64, 128]))
    if kind == I.MASK_PAGED_DECODE:
        return I.paged_decode_workload(seed, B, 0, 0, Hq, Hkv, d, page_size=page,
                                       context_lens=rng.integers(1, 3000, B), name=f"fuzz{idx}")
    if kind == I.MASK_DECODE:
        lens = rng.integers(1, 2000, B)
        return I.dense_decode_workload(seed, B, 0, 0, Hq, Hkv, d,
                                       N=int(lens.max() + rng.integers(0, 100)),
                                       context_lens=lens, name=f"fuzz{idx}")
    if kind == I.MASK_PAGED_PREFILL:
        lk = rng.integers(1, 2000, B)
        lq = np.array([int(rng.integers(0, n + 1)) for n in lk])
        lq[int(rng.integers(0, B))] = max(int(lq.max()), 1)
        lq = np.minimum(lq, lk)
        return I.paged_prefill_workload(seed, B, 0, 0, 0, 0, Hq, Hkv, d, page_size=page,
                                        context_lens=lk, chunk_lens=lq, name=f"fuzz{idx}")
    N = int(rng.integers(1, 700))
    window = 0
    if kind == I.MASK_SLIDING:
        window = int(rng.integers(1, N + 130))
    elif kind in (I.MASK_SLIDING_BIDIR, I.MASK_PREFIX_LM):
        window = int(rng.integers(0, N + 130))
    return I.dense_workload(seed, B, Hq, Hkv, N, d, kind, window, name=f"fuzz{idx}")


@pytest.mark.parametrize("idx", range(200))
def test_randomized_shapes(idx):
    w = _fuzz_workload(idx)
    compare(w, run(w), strict=False)


# ------------------------------------------------------------------ CUDA graphs

def test_cuda_graph_capture_and_replay():
    """After one ordinary call (which sets the one-time kernel attributes and caches), every
    entry point enqueues only memsets and kernel launches on the caller's stream, so a causal
    prefill and a paged decode can be captured into one CUDA graph. Replaying it on new
    inputs, written in place into the captured buffers, gives the oracle's results for those
    inputs."""
    wp = I.dense_workload(71, 2, 4, 2, 300, 128, I.MASK_CAUSAL)
    wd = I.paged_decode_workload(72, 3, 100, 2000, 8, 2, 128)
    pp, pd = DeviceProblem(wp), DeviceProblem(wd)
    assert pp.run() == 0 and pd.run() == 0, attn.last_error()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        rc = pp.run() | pd.run()
    assert rc == 0, attn.last_error()
    # new query, key and value values for the prefill, new queries for the decode
    wp2 = I.dense_workload(73, 2, 4, 2, 300, 128, I.MASK_CAUSAL)
    wd2 = I.paged_decode_workload(72, 3, 100, 2000, 8, 2, 128)
    wd2.q = I.dense_workload(74, 3, 8, 2, 1, 128).q
    for dst, src in ((pp.q, wp2.q), (pp.k, wp2.k), (pp.v, wp2.v), (pd.q, wd2.q)):
        dst.copy_(bf16_tensor(src, dst.device).reshape(dst.shape))
    for t in (pp.o, pd.o):
        t.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert attn.attn_get_status() == 0
    compare(wp2, pp, strict=False)
    compare(wd2, pd)
    # A second replay on other queries: the decode's split tickets, left cleared by the first
    # replay, serve the replayed (same) generation again.
    wd3 = I.paged_decode_workload(72, 3, 100, 2000, 8, 2, 128)
    wd3.q = I.dense_workload(75, 3, 8, 2, 1, 128).q
    pd.q.copy_(bf16_tensor(wd3.q, pd.q.device).reshape(pd.q.shape))
    pd.o.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert attn.attn_get_status() == 0
    compare(wd3, pd)
