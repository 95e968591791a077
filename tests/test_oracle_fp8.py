"""The FP8 (E4M3) block quantizer of the oracle against facts fixed outside it: torch's own
float8_e4m3fn conversion (a library routine) for the value table and the rounding, the bounds
that nearest rounding guarantees, and identities of the attention on dequantized blocks. CPU
only."""
import numpy as np
import pytest
import torch

import oracle
from oracle import fp8
from tiled_attention_gb300 import inputs as I


def torch_e4m3(x32: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x32, np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_value_table_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = fp8.e4m3_values()
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours)) and nan.sum() == 2
    assert np.array_equal(ref[~nan], ours[~nan])
    assert ours[0x7E] == 448.0 and ours[0x08] == 2.0 ** -6 and ours[0x01] == 2.0 ** -9
    assert ours[0x38] == 1.0


def test_rounding_matches_torch():
    rng = np.random.default_rng(0)
    vals = fp8.e4m3_values()[:0x7F]
    mids = ((vals[1:] + vals[:-1]) / 2).astype(np.float32)  # exact ties
    xs = [rng.standard_normal(20000).astype(np.float32) * s for s in (1e-3, 0.05, 1, 30, 150)]
    xs += [mids, -mids, vals.astype(np.float32), np.float32([0.0, -0.0, 448.0, -448.0])]
    x = np.clip(np.concatenate(xs), -448, 448).astype(np.float32)
    assert np.array_equal(fp8.e4m3_round(x), torch_e4m3(x))


def test_ties_go_to_even_codes():
    # 1.0625 lies halfway between 1.0 (mantissa 000) and 1.125 (001): rounds to 1.0;
    # 1.1875 lies halfway between 1.125 (001) and 1.25 (010): rounds to 1.25.
    got = fp8.e4m3_round(np.float32([1.0625, 1.1875, -1.0625]))
    assert list(got) == [0x38, 0x3A, 0xB8]


def test_saturation():
    assert list(fp8.e4m3_round(np.float32([460.0, -1e6]))) == [0x7E, 0xFE]


def test_quantize_blocks_bounds():
    """Each block's largest magnitude lands exactly on +-448; dequantized values are within
    half an E4M3 step of the input; the short last block and an all-zero block behave."""
    rng = np.random.default_rng(1)
    x = rng.standard_normal((3, 300, 128)).astype(np.float32)
    x[:, 5, 7] = 9.0  # a clear maximum in block 0
    x[2, 128:256] = 0.0  # an all-zero block
    bits = I.f32_to_bf16_bits(x)
    xf = I.bf16_bits_to_f32(bits).astype(np.float64)
    codes, scales = fp8.quantize_blocks(bits)
    assert scales.shape == (3, 3) and codes.shape == x.shape
    for pl in range(3):
        for t in range(3):
            blk = xf[pl, 128 * t:128 * (t + 1)]
            amax = np.abs(blk).max()
            assert scales[pl, t] == np.float32(np.float32(amax) / np.float32(448.0))
    assert scales[2, 1] == 0 and not codes[2, 128:256].any()
    assert codes[0, 5, 7] == 0x7E
    deq = fp8.dequantize(codes, scales)
    s_rows = np.repeat(scales.astype(np.float64), 128, axis=1)[:, :300, None]
    y = xf / np.where(s_rows > 0, s_rows, 1)  # the value before rounding, in block units
    # half a step: 2^-4 relative for normals (3 mantissa bits), 2^-10 absolute below 2^-6;
    # plus the fp32 rounding of the division (2^-24 relative)
    bound = np.maximum(np.abs(y) * 2.0 ** -4, 2.0 ** -10) * (1 + 2.0 ** -20)
    err = np.abs(deq / np.where(s_rows > 0, s_rows, 1) - y)
    assert np.all(err <= bound)


def _fp8_problem(seed, N=200, mask=I.MASK_CAUSAL):
    w = I.dense_workload(seed, 2, 4, 2, N, 128, mask)
    w.q8, w.q_scales = fp8.quantize_blocks(w.q.reshape(-1, N, 128))
    w.k8, w.k_scales = fp8.quantize_blocks(w.k.reshape(-1, N, 128))
    w.q8, w.k8 = w.q8.reshape(w.q.shape), w.k8.reshape(w.k.shape)
    return w


def test_unit_scales_equal_the_bf16_oracle():
    """With every scale 1, the FP8 path attends over the E4M3 values themselves, which bf16
    represents exactly: it must equal the bf16 oracle on those values, bit for bit."""
    w = _fp8_problem(3)
    w.q_scales[...] = 1
    w.k_scales[...] = 1
    vals = fp8.e4m3_values()
    b = I.dense_workload(3, 2, 4, 2, 200, 128, I.MASK_CAUSAL)
    b.q = I.f32_to_bf16_bits(vals[w.q8].astype(np.float32))
    b.k = I.f32_to_bf16_bits(vals[w.k8].astype(np.float32))
    b.v = w.v
    o1, l1 = oracle.attention(w)
    o2, l2 = oracle.attention(b)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_doubling_key_scales_doubles_the_logits():
    """Key scales multiply the logits: doubling every key block's scale gives the same result
    as doubling the softmax scale, bit for bit."""
    w = _fp8_problem(4)
    o0, l0 = oracle.attention(w)
    w2 = _fp8_problem(4)
    w2.k_scales = w2.k_scales * np.float32(2)
    w3 = _fp8_problem(4)
    w3.scale = w.scale * 2
    a, b = oracle.attention(w2), oracle.attention(w3)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert not np.array_equal(a[0], o0)


def test_fp8_attention_close_to_bf16_inputs():
    """Quantization error only: the FP8 attention of N(0,1) inputs stays near the bf16
    attention of the unquantized inputs. A sanity bound, not a parity tolerance: E4M3 keeps
    3 mantissa bits, so the logits move by a few percent; rows that see few keys (early causal
    rows) show it most, and the error shrinks as rows average over more keys."""
    w = _fp8_problem(5, N=300)
    b = I.dense_workload(5, 2, 4, 2, 300, 128, I.MASK_CAUSAL)
    o1, l1 = oracle.attention(w)
    o2, l2 = oracle.attention(b)
    eo, el = np.abs(o1 - o2), np.abs(l1 - l2)
    rows = np.arange(eo.shape[0]) % 300
    assert eo.mean() < 0.01 and el.mean() < 0.01
    assert eo.max() < 0.25 and eo[rows >= 100].max() < 0.06


@pytest.mark.parametrize("mask", [I.MASK_NONE, I.MASK_SLIDING_BIDIR])
def test_fp8_oracle_other_masks_run(mask):
    w = _fp8_problem(6, N=150, mask=mask)
    w.window = 20
    o, lse = oracle.attention(w)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
