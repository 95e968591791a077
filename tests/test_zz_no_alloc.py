"""The allocation-free paged decode entry point against the workspace entry point.

Some callers of this library cannot give it a workspace and cannot let it call cudaMalloc:
code running behind a custom-op interface that hands out no scratch buffer, code inside another
framework's device-memory pool, and serving loops where the device synchronisation that
cudaMalloc / cudaFree imply is not allowed. attn_paged_decode_noalloc serves them from a fixed
16 MiB scratch array inside the library. These tests check that it returns what attn_fwd with a
caller-provided workspace returns, on consecutive calls that reuse the array, and that a
request larger than the array is refused. This file is collected last on purpose.
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


def test_request_larger_than_scratch_is_refused():
    build.build()
    # 64 sequences x 16 kv heads x 8 query heads each, 64K-token contexts: far above 16 MiB.
    B, Hkv, Hq, N, d = 64, 16, 128, 65536, 128
    assert attn.attn_workspace_bytes(B, Hq, Hkv, N, d, attn.ATTN_MASK_PAGED_DECODE, 64) > SCRATCH_BYTES
    rc = attn.attn_paged_decode_noalloc(None, None, None, None, None, B, Hq, Hkv, N, d, 0.1,
                                        None, None, 64, 1, 0)
    assert rc == attn.ATTN_ERR_UNSUPPORTED
    assert "scratch" in attn.last_error()


@pytest.mark.gpu
def test_matches_workspace_entry_point_on_consecutive_calls():
    assert torch.cuda.is_available(), "needs a CUDA device"
    build.build()
    cases = [(31, [1, 700, 5000, 64, 4097]), (32, [16384, 333, 2048])]
    for seed, lens in cases:
        w = I.paged_decode_workload(seed, len(lens), 0, 0, 32, 8, 128, context_lens=lens)
        ref = DeviceProblem(w)
        assert ref.run() == 0, attn.last_error()
        o = torch.full_like(ref.o, float("nan"))
        lse = torch.full_like(ref.lse, float("nan"))
        rc = attn.attn_paged_decode_noalloc(ref.q, ref.k, ref.v, o, lse, w.B, w.Hq, w.Hkv, w.N,
                                            w.d, w.scale, ref.cu, ref.table, w.page_size,
                                            ref.num_pages)
        assert rc == 0, attn.last_error()
        torch.cuda.synchronize()
        assert attn.attn_get_status() == 0
        eo = (o.float() - ref.o.float()).abs().max().item()
        el = (lse - ref.lse).abs().max().item()
        assert np.isfinite(eo) and eo <= O_TOL, f"{lens}: max|dO| = {eo}"
        assert np.isfinite(el) and el <= LSE_TOL, f"{lens}: max|dLSE| = {el}"
