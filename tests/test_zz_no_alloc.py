"""The allocation-free paged decode entry point against the workspace entry point.

Some callers of this library cannot give it a workspace and cannot let it call cudaMalloc:
code running behind a custom-op interface that hands out no scratch buffer, code inside another
framework's device-memory pool, and serving loops where the device synchronisation that
cudaMalloc / cudaFree imply is not allowed. attn_paged_decode_noalloc serves them from a fixed
16 MiB scratch array inside the library.

Both entry points run the same kernel with the same split of the context and merge the splits
in a fixed order, so their results must agree bit for bit: the GPU tests compare with
torch.equal, on consecutive calls that reuse the array, on a small call right after a large
one (which leaves stale partials behind; the tickets, which this entry point never zeroes,
must be back at zero), at the largest request the array holds,
and after attn_release has made the library look the array's address up again. One case is
also checked against the fp64 oracle. The CPU tests check that invalid arguments report their
own reason and that the size limit falls exactly where attn_workspace_bytes puts it. This file
is collected last on purpose.
"""
import numpy as np
import pytest
import torch

from tiled_attention_gb300 import attn, build
from tiled_attention_gb300 import inputs as I
from tiled_attention_gb300.runner import DeviceProblem

SCRATCH_BYTES = 16 << 20
O_TOL = 1e-2
LSE_TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def library():
    build.build()
    attn.lib()


def _largest_fitting_n(B, Hq, Hkv, d, page_size=64):
    """Largest longest-context N whose split-KV scratch fits the array (found by bisection on
    attn_workspace_bytes, which is nondecreasing in N)."""
    def need(n):
        return attn.attn_workspace_bytes(B, Hq, Hkv, n, d, attn.ATTN_MASK_PAGED_DECODE,
                                         page_size)
    lo, hi = 1, 1 << 26
    assert need(lo) <= SCRATCH_BYTES < need(hi)
    while hi - lo > 1:
        mid = (lo + hi) // 2
        if need(mid) <= SCRATCH_BYTES:
            lo = mid
        else:
            hi = mid
    return lo


# ------------------------------------------------------------------ host side (no GPU needed)

def test_scratch_size_is_declared():
    assert attn.attn_noalloc_scratch_bytes() == SCRATCH_BYTES


def test_request_larger_than_scratch_is_refused():
    # 64 sequences x 16 kv heads x 8 query heads each, 64K-token contexts: far above 16 MiB.
    B, Hkv, Hq, N, d = 64, 16, 128, 65536, 128
    assert attn.attn_workspace_bytes(B, Hq, Hkv, N, d, attn.ATTN_MASK_PAGED_DECODE, 64) > SCRATCH_BYTES
    rc = attn.attn_paged_decode_noalloc(None, None, None, None, None, B, Hq, Hkv, N, d, 0.1,
                                        None, None, 64, 1, 0)
    assert rc == attn.ATTN_ERR_UNSUPPORTED
    assert "scratch" in attn.last_error()


@pytest.mark.parametrize("d,page_size,Hq,Hkv,want,words", [
    (96, 64, 32, 8, attn.ATTN_ERR_UNSUPPORTED, "head dim"),
    (128, 48, 32, 8, attn.ATTN_ERR_UNSUPPORTED, "page_size"),
    (128, 64, 30, 8, attn.ATTN_ERR_INVALID, "Hkv"),
    (128, 64, 136, 8, attn.ATTN_ERR_UNSUPPORTED, "query heads per kv head"),
])
def test_invalid_arguments_report_their_own_reason(d, page_size, Hq, Hkv, want, words):
    """A large N would need far more scratch than the array holds, but an invalid head dim,
    page size or head grouping is what the caller must hear about."""
    rc = attn.attn_paged_decode_noalloc(None, None, None, None, None, 64, Hq, Hkv, 1 << 20, d,
                                        0.1, None, None, page_size, 1, 0)
    assert rc == want, attn.last_error()
    msg = attn.last_error()
    assert words in msg and "scratch" not in msg, msg


def test_limit_falls_where_the_workspace_size_puts_it():
    """The largest N whose attn_workspace_bytes fits is not refused for its size; the next
    64-token stage up is."""
    B, Hq, Hkv, d = 38, 64, 4, 128
    n = _largest_fitting_n(B, Hq, Hkv, d)
    assert attn.attn_workspace_bytes(B, Hq, Hkv, n + 64, d, attn.ATTN_MASK_PAGED_DECODE,
                                     64) > SCRATCH_BYTES
    rc = attn.attn_paged_decode_noalloc(None, None, None, None, None, B, Hq, Hkv, n + 64, d,
                                        0.1, None, None, 64, 1, 0)
    assert rc == attn.ATTN_ERR_UNSUPPORTED and "scratch" in attn.last_error()
    # At n the size check passes; what fails next is the null tensors (or, with no GPU, the
    # device lookup), never the size.
    rc = attn.attn_paged_decode_noalloc(None, None, None, None, None, B, Hq, Hkv, n, d, 0.1,
                                        None, None, 64, 1, 0)
    assert rc != attn.ATTN_ERR_UNSUPPORTED, attn.last_error()
    assert "scratch" not in attn.last_error()


def test_release_forgets_cached_addresses():
    attn.attn_release()
    for dev in (0, 1, 63):
        assert attn.attn_cached_device_state(dev) == 0
    assert attn.attn_cached_device_state(-1) == attn.ATTN_ERR_INVALID
    assert attn.attn_cached_device_state(64) == attn.ATTN_ERR_INVALID


# ------------------------------------------------------------------ on the GPU

def _noalloc(dp, w, stream=None):
    o = torch.full_like(dp.o, float("nan"))
    lse = torch.full_like(dp.lse, float("nan"))
    rc = attn.attn_paged_decode_noalloc(dp.q, dp.k, dp.v, o, lse, w.B, w.Hq, w.Hkv, w.N, w.d,
                                        w.scale, dp.cu, dp.table, w.page_size, dp.num_pages,
                                        stream)
    assert rc == 0, attn.last_error()
    return o, lse


def _workspace_path(w):
    dp = DeviceProblem(w)
    assert dp.run() == 0, attn.last_error()
    return dp


def _assert_bit_identical(w, dp, o, lse):
    torch.cuda.synchronize()
    assert attn.attn_get_status() == 0
    assert torch.equal(o.view(torch.int16), dp.o.view(torch.int16)), \
        f"{w.name}: O differs from the workspace path"
    assert torch.equal(lse, dp.lse), f"{w.name}: LSE differs from the workspace path"


@pytest.mark.gpu
def test_matches_workspace_entry_point_on_consecutive_calls():
    assert torch.cuda.is_available(), "needs a CUDA device"
    cases = [(31, [1, 700, 5000, 64, 4097]), (32, [16384, 333, 2048]), (33, [9000, 1, 65])]
    for seed, lens in cases:
        w = I.paged_decode_workload(seed, len(lens), 0, 0, 32, 8, 128, context_lens=lens,
                                    name=f"noalloc {lens}")
        dp = _workspace_path(w)
        o, lse = _noalloc(dp, w)
        _assert_bit_identical(w, dp, o, lse)


@pytest.mark.gpu
def test_against_the_oracle():
    import oracle
    lens = [1, 63, 64, 65, 3000, 12000]
    w = I.paged_decode_workload(34, len(lens), 0, 0, 24, 4, 128, page_size=16,
                                context_lens=lens, name="noalloc vs oracle")
    dp = DeviceProblem(w)
    o, lse = _noalloc(dp, w)
    torch.cuda.synchronize()
    assert attn.attn_get_status() == 0
    ro, rl = oracle.attention(w)
    go = o.float().reshape(-1, w.d).cpu().numpy().astype(np.float64)
    gl = lse.reshape(-1).cpu().numpy().astype(np.float64)
    assert np.isfinite(go).all() and np.isfinite(gl).all()
    assert np.abs(go - ro).max() <= O_TOL and np.abs(gl - rl).max() <= LSE_TOL


@pytest.mark.gpu
def test_small_call_after_a_large_one():
    """The largest request the array holds fills it with partials and leaves tickets behind;
    a small request that follows, with fewer splits and another grouping, must not see any of
    it. Both agree bit for bit with the workspace path."""
    B, Hq, Hkv, d = 38, 64, 4, 128
    n = _largest_fitting_n(B, Hq, Hkv, d)
    rng = np.random.default_rng(35)
    lens = np.concatenate([[n], rng.integers(1, 3000, B - 1)])
    big = I.paged_decode_workload(35, B, 0, 0, Hq, Hkv, d, context_lens=lens,
                                  name=f"noalloc largest N={n}")
    assert attn.attn_workspace_bytes(B, Hq, Hkv, big.N, d, attn.ATTN_MASK_PAGED_DECODE,
                                     64) <= SCRATCH_BYTES
    dp_big = _workspace_path(big)
    ob, lb = _noalloc(dp_big, big)
    _assert_bit_identical(big, dp_big, ob, lb)
    small = I.paged_decode_workload(36, 3, 0, 0, 6, 2, 64, page_size=32,
                                    context_lens=[5, 2100, 700], name="noalloc small after big")
    dp_small = _workspace_path(small)
    os_, ls = _noalloc(dp_small, small)
    _assert_bit_identical(small, dp_small, os_, ls)
    # and the large one again, now after the small one
    ob2, lb2 = _noalloc(dp_big, big)
    _assert_bit_identical(big, dp_big, ob2, lb2)


@pytest.mark.gpu
def test_release_then_call_again():
    """attn_release forgets the array's cached address; the next call looks it up again and
    gives the same results."""
    lens = [3000, 17, 800]
    w = I.paged_decode_workload(37, len(lens), 0, 0, 16, 4, 128, context_lens=lens,
                                name="noalloc after release")
    dp = _workspace_path(w)
    o1, l1 = _noalloc(dp, w)
    torch.cuda.synchronize()
    assert attn.attn_cached_device_state(torch.cuda.current_device()) & 2
    attn.attn_release()
    assert attn.attn_cached_device_state(torch.cuda.current_device()) == 0
    o2, l2 = _noalloc(dp, w)
    _assert_bit_identical(w, dp, o1, l1)
    _assert_bit_identical(w, dp, o2, l2)
    assert attn.attn_cached_device_state(torch.cuda.current_device()) & 2
