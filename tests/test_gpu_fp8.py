"""FP8 path against the oracle through the C ABI: the E4M3 block quantizer bit for bit, and
attention with E4M3 Q / K (S = Q K^T on the FP8 tensor cores) against the oracle's attention on
the dequantized blocks, with the bf16 path's tolerances. The FP8 inputs of the parity cases
come from the oracle's quantizer; the quantizer test shows the library's produces the same
bytes."""
import numpy as np
import pytest
import torch

import oracle
from oracle import fp8
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


def gpu_quantize(bits):
    """Quantize bf16 bits [planes, N, d] with the library; returns numpy codes and scales."""
    planes, N, d = bits.shape
    x = bf16_tensor(bits, "cuda")
    x8 = torch.zeros((planes, N, d), dtype=torch.uint8, device="cuda")
    sc = torch.full((planes, (N + 127) // 128), float("nan"), dtype=torch.float32, device="cuda")
    assert attn.attn_quantize_fp8(x, x8, sc, planes, N, d) == 0, attn.last_error()
    torch.cuda.synchronize()
    return x8.cpu().numpy(), sc.cpu().numpy()


@pytest.mark.parametrize("N", [1, 127, 128, 129, 300, 2048])
@pytest.mark.parametrize("d", [64, 128])
def test_quantizer_bit_exact(N, d):
    rng = np.random.default_rng(N + d)
    x = rng.standard_normal((6, N, d)).astype(np.float32) * np.float32(3.0)
    x[1] = 0.0  # a plane of all-zero blocks
    x[2, :min(N, 128)] *= np.float32(1e-3)  # a block of small values (E4M3 subnormals)
    x[3, 0, 0] = -200.0  # a block whose maximum is negative
    bits = I.f32_to_bf16_bits(x)
    codes, scales = gpu_quantize(bits)
    rc, rs = fp8.quantize_blocks(bits)
    assert np.array_equal(scales, rs)
    assert np.array_equal(codes, rc)


def test_quantizer_bit_exact_stress():
    """Many blocks over a wide range of magnitudes, blocks whose scale is a power of two with
    values on E4M3 rounding midpoints, negative zeros, and blocks whose scale is an fp32
    subnormal: codes and scales equal the oracle's quantizer byte for byte."""
    rng = np.random.default_rng(2024)
    planes, N, d = 64, 1024, 128
    x = rng.standard_normal((planes, N, d)).astype(np.float32)
    x *= (10.0 ** rng.uniform(-20, 20, (planes, 1, 1))).astype(np.float32)
    # scale 2^-3 exactly (amax 448 * 2^-3), values on midpoints between E4M3 codes
    mids = np.array([0.5 * (a + b) for a, b in zip(fp8.e4m3_values()[:-1], fp8.e4m3_values()[1:])
                     if 0 < a and b <= 448], dtype=np.float32)
    blk = rng.choice(mids, (128, d)).astype(np.float32) * np.float32(0.125)
    blk *= np.where(rng.random((128, d)) < 0.5, -1, 1).astype(np.float32)
    blk[0, 0] = 448 * 0.125
    x[0, :128] = blk
    x[1, 5, :] = -0.0                                   # negative zeros in a normal block
    x[2, :128] = rng.standard_normal((128, d)).astype(np.float32) * np.float32(1e-38)
    x[3, 128:256] = np.float32(-0.0)                    # a block of negative zeros only
    bits = I.f32_to_bf16_bits(x)
    codes, scales = gpu_quantize(bits)
    rc, rs = fp8.quantize_blocks(bits)
    assert np.array_equal(scales, rs)
    bad = np.argwhere(codes != rc)
    assert bad.size == 0, f"{len(bad)} codes differ, first at {bad[0]}"


def fp8_workload(seed, B, Hq, Hkv, N, mask, window=0):
    w = I.dense_workload(seed, B, Hq, Hkv, N, 128, mask, window=window)
    w.q8, w.q_scales = fp8.quantize_blocks(w.q.reshape(B * Hq, N, 128))
    w.k8, w.k_scales = fp8.quantize_blocks(w.k.reshape(B * Hkv, N, 128))
    w.q8, w.k8 = w.q8.reshape(w.q.shape), w.k8.reshape(w.k.shape)
    w.name = f"fp8 m{mask} N{N}"
    return w


def compare(w, dp, rows=None, strict=True):
    o, lse = dp.outputs()
    ro, rl = oracle.attention(w, rows=rows)
    if rows is not None:
        o, lse = o[rows], lse[rows]
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    eo, el = np.abs(o - ro), np.abs(lse - rl)
    tol = O_TOL if strict else O_TOL + 2.0 ** -8 * np.abs(ro)
    assert np.all(eo <= tol) and el.max() <= LSE_TOL, \
        f"{w.name}: max|dO|={eo.max():.3e} max|dLSE|={el.max():.3e}"


def run(w):
    dp = DeviceProblem(w)
    assert dp.run() == 0, attn.last_error()
    torch.cuda.synchronize()
    assert attn.attn_get_status() == 0
    return dp


@pytest.mark.parametrize("N", [1, 129, 300, 640])
@pytest.mark.parametrize("mask,window", [(I.MASK_NONE, 0), (I.MASK_CAUSAL, 0),
                                         (I.MASK_SLIDING, 300), (I.MASK_SLIDING_BIDIR, 100),
                                         (I.MASK_PREFIX_LM, 200)])
def test_fp8_attention_ragged(mask, window, N):
    w = fp8_workload(1100 + N, 2, 4, 2, N, mask, window)
    compare(w, run(w), strict=False)


_FP8_KINDS = [I.MASK_NONE, I.MASK_CAUSAL, I.MASK_SLIDING, I.MASK_SLIDING_BIDIR, I.MASK_PREFIX_LM]


@pytest.mark.parametrize("idx", range(60))
def test_fp8_randomized_shapes(idx):
    """Case idx: its mask kind in turn; batch, GQA group, length (crossing 128-row tiles) and
    window or prefix (also past the sequence) drawn from a generator seeded by idx."""
    rng = np.random.default_rng(7000 + idx)
    mask = _FP8_KINDS[idx % len(_FP8_KINDS)]
    B = int(rng.integers(1, 4))
    Hkv = int(rng.integers(1, 4))
    Hq = Hkv * int(rng.integers(1, 5))
    N = int(rng.integers(1, 1500))
    window = 0
    if mask == I.MASK_SLIDING:
        window = int(rng.integers(1, N + 130))
    elif mask in (I.MASK_SLIDING_BIDIR, I.MASK_PREFIX_LM):
        window = int(rng.integers(0, N + 130))
    w = fp8_workload(7000 + idx, B, Hq, Hkv, N, mask, window)
    compare(w, run(w), strict=False)


def test_fp8_zero_key_tile():
    """An all-zero key tile has scale 0: its scores are exactly 0 and masked keys stay
    masked (no NaN from 0 * -inf)."""
    w = fp8_workload(77, 1, 4, 2, 300, I.MASK_CAUSAL)
    w.k8[:, :, 128:256] = 0
    w.k_scales[:, 1] = 0
    compare(w, run(w), strict=False)


def test_fp8_headline_shape():
    """Causal B2 Hq32 Hkv8 N8192 with Q / K quantized by the library (checked against the
    oracle's quantizer byte for byte), attention on every output row against the oracle."""
    w = I.config("3c")
    B, Hq, Hkv, N = w.B, w.Hq, w.Hkv, w.N
    q8, qs = gpu_quantize(w.q.reshape(B * Hq, N, 128))
    k8, ks = gpu_quantize(w.k.reshape(B * Hkv, N, 128))
    rq8, rqs = fp8.quantize_blocks(w.q.reshape(B * Hq, N, 128))
    rk8, rks = fp8.quantize_blocks(w.k.reshape(B * Hkv, N, 128))
    assert np.array_equal(q8, rq8) and np.array_equal(qs, rqs)
    assert np.array_equal(k8, rk8) and np.array_equal(ks, rks)
    w.q8, w.k8 = rq8.reshape(w.q.shape), rk8.reshape(w.k.shape)
    w.q_scales, w.k_scales = rqs, rks
    compare(w, run(w))
