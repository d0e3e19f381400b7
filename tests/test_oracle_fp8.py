"""Pins of the oracle's fp8 (e4m3) quantization, the arithmetic of the lower-precision
variant (yinghuohong.cn llm.c article, section "脚动完成每一个层前向/反向流传": precision
planned to go from fp32 down to fp16 or lower).  CPU only.

The oracle writes the e4m3 format out from its definition; here it is held against
PyTorch's own float8_e4m3fn conversion (a library routine), the format's closed-form
values, and the invariants of the power-of-two scales."""
import math

import numpy as np
import pytest

from oracle import gpt2_oracle as O
from step_gpt_train_03_b300 import synth


def test_e4m3_table_against_the_format_and_torch():
    import torch
    t = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    for c in range(256):
        a, b = O.E4M3_TABLE[c], t[c]
        assert (np.isnan(a) and np.isnan(b)) or a == b, c
    # closed-form points of the format: 1.0, the largest finite, the smallest normal and
    # subnormal, NaN at S.1111.111
    assert O.e4m3_value(0x38) == 1.0
    assert O.e4m3_value(0x7E) == 448.0 and O.e4m3_value(0xFE) == -448.0
    assert O.e4m3_value(0x08) == 2.0 ** -6
    assert O.e4m3_value(0x01) == 2.0 ** -9
    assert math.isnan(O.e4m3_value(0x7F)) and math.isnan(O.e4m3_value(0xFF))
    # the non-negative codes 0x00..0x7E are increasing (encode relies on it)
    assert np.all(np.diff(O.E4M3_TABLE[:127]) > 0)


def test_e4m3_rounding_against_torch():
    import torch
    rng = np.random.default_rng(0)
    grid = O.E4M3_TABLE[np.isfinite(O.E4M3_TABLE)]
    pos = O.E4M3_TABLE[:127]
    mids = (pos[:-1] + pos[1:]) / 2                       # exact ties: round to even mantissa
    x = np.concatenate([rng.standard_normal(200000) * rng.choice([1e-3, 0.02, 1, 30, 200], 200000),
                        grid, mids, -mids]).astype(np.float32)
    x = x[np.abs(x) <= 448]
    ref = torch.tensor(x).to(torch.float8_e4m3fn)
    assert np.array_equal(O.e4m3_round(x.astype(np.float64)), ref.float().numpy())
    assert np.array_equal(O.e4m3_encode(x.astype(np.float64)), ref.view(torch.uint8).numpy())
    # saturation (torch's conversion is not saturating, so this is pinned by definition)
    assert np.array_equal(O.e4m3_round(np.array([449.0, 1e6, -500.0])), [448.0, 448.0, -448.0])
    # the worst rounding error of a normal-range value is half a spacing: 2^-4 relative
    y = rng.uniform(2.0 ** -6, 448, 100000) * rng.choice([-1, 1], 100000)
    assert np.all(np.abs(O.e4m3_round(y) - y) <= 2.0 ** -4 * np.abs(y) + 1e-300)


def test_power_of_two_scales():
    rng = np.random.default_rng(1)
    amax = np.exp(rng.uniform(-30, 30, 20000))
    for a in np.concatenate([amax, [448.0, 449.0, 0.875, 0.8750001, 2.0 ** -20, 1.0]]):
        k = O.pow2_scale_exponent(a)
        assert a * 2.0 ** k <= 448.0 < a * 2.0 ** (k + 1), a
    assert O.pow2_scale_exponent(0.0) == 0
    assert O.pow2_scale_exponent(448.0) == 0 and O.pow2_scale_exponent(1.0) == 8


def test_row_and_tensor_quantization():
    rng = np.random.default_rng(2)
    y = rng.standard_normal((64, 768)) * np.exp(rng.uniform(-4, 4, (64, 1)))
    deq, codes, ks = O.quantize_rows_e4m3(y)
    # each row's largest magnitude lands in the top binade [224, 448] after scaling
    for r in range(64):
        assert 224.0 <= np.abs(y[r]).max() * 2.0 ** ks[r] <= 448.0
    # decoding the codes and unscaling gives the dequantized values exactly
    assert np.array_equal(O.E4M3_TABLE[codes] * np.exp2(-ks)[:, None], deq)
    # relative error at most 2^-4 where the scaled value is a normal e4m3 number
    scaled = np.abs(y) * np.exp2(ks)[:, None]
    normal = scaled >= 2.0 ** -6
    assert np.all(np.abs(deq - y)[normal] <= 2.0 ** -4 * np.abs(y)[normal])
    # values already on the grid (with amax on the grid's top) pass through unchanged
    g = O.E4M3_TABLE[rng.integers(0, 127, (8, 64))] * rng.choice([-1, 1], (8, 64))
    g[:, 0] = 448.0
    assert np.array_equal(O.quantize_rows_e4m3(g)[0], g)
    w = rng.standard_normal((96, 64)) * 0.02
    wq, wc, k = O.quantize_tensor_e4m3(w)
    assert np.array_equal(O.E4M3_TABLE[wc] * 2.0 ** -k, wq)
    assert O.pow2_scale_exponent(np.abs(w).max()) == k


def test_fp8_model_is_the_plain_model_with_quantized_products():
    """The fp8 oracle differs from the plain one only in the qkv and fc products: with
    the quantization made the identity (both on the grid), the losses agree exactly;
    on the seeded weights the quantization moves the tiny model's initial loss by a
    small amount, and the gradient formulas are the plain model's (straight through)."""
    shape = synth.TINY_HS64
    params = synth.init_params(shape, 0)
    tok, tgt = synth.uniform_tokens(shape.vocab_size, 2, 32, 0)
    plain = O.from_shape(shape)
    plain.load(params)
    q = O.from_shape(shape)
    q.load(params)
    q.fp8 = True
    l0, l1 = plain.forward(tok, tgt), q.forward(tok, tgt)
    assert l0 != l1 and abs(l0 - l1) < 1e-2, (l0, l1)
    q.zero_grad()
    q.backward()
    assert all(np.isfinite(v).all() for v in q.g.values())
    # identity quantization: every product input already an e4m3 value with the scale 1
    x = O.E4M3_TABLE[np.random.default_rng(3).integers(0, 127, (5, 64))]
    x[:, 0] = 448.0
    w = O.E4M3_TABLE[np.random.default_rng(4).integers(0, 127, (7, 64))]
    w[0, 0] = 448.0
    b = np.arange(7.0)
    assert np.array_equal(O.matmul_forward_fp8(x, w, b), O.matmul_forward(x, w, b))
