"""Pins of the block-scaled (MXFP8) quantization oracle (oracle/moe_mx_ref.py)
against things other than itself (CPU only):

* hand-derived blocks (tests/golden/mx_blocks_hand.json);
* the scale exponent by its defining inequality 2^(s + emax) <= amax <
  2^(s + emax + 1), checked by exact comparisons (not through the log2 the
  oracle uses);
* element codes against PyTorch's float8 conversions (library routine) of the
  scaled values that lie in range;
* the correct-rounding bound of every non-saturated element, exact
  reconstruction of values on the scaled grid, block independence, and the
  zero / non-finite blocks.
"""
import json
import os

import numpy as np
import pytest
import torch

from oracle import moe_fp8_ref as q8
from oracle import moe_mx_ref as mx

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
EMAX = {"e4m3": 8, "e5m2": 15}
MBITS = {"e4m3": 3, "e5m2": 2}
BIAS = {"e4m3": 7, "e5m2": 15}
TORCH = {"e4m3": torch.float8_e4m3fn, "e5m2": torch.float8_e5m2}


def _blocks(rng, n, scale_pow):
    """n blocks of 32, each with its own magnitude 2^p, p drawn from scale_pow."""
    p = rng.integers(scale_pow[0], scale_pow[1], size=(n, 1))
    return (rng.standard_normal((n, 32)) * np.ldexp(1.0, p)).astype(np.float32)


def test_golden_blocks():
    g = json.load(open(os.path.join(GOLDEN, "mx_blocks_hand.json")))
    for b in g["blocks"]:
        x = np.zeros((1, 32))
        for i, v in b["x"].items():
            x[0, int(i)] = v
        codes, scales = mx.mx_quantize(x, b["fmt"])
        assert int(scales[0, 0]) == b["scale_code"], b["why"]
        want = np.zeros(32, np.uint8)
        for i, h in b["codes"].items():
            want[int(i)] = int(h, 16)
        assert (codes[0] == want).all(), (b["why"], codes[0])


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_scale_exponent_by_its_inequality(fmt):
    rng = np.random.default_rng(1)
    x = _blocks(rng, 400, (-60, 60))
    _, scales = mx.mx_quantize(x, fmt)
    for r in range(x.shape[0]):
        amax = float(np.abs(x[r].astype(np.float64)).max())
        s = int(scales[r, 0]) - 127
        lo, hi = np.ldexp(1.0, s + EMAX[fmt]), np.ldexp(1.0, s + EMAX[fmt] + 1)
        assert lo <= amax < hi, (r, amax, s)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_elements_match_torch_float8(fmt):
    rng = np.random.default_rng(2)
    x = _blocks(rng, 300, (-20, 20))
    codes, scales = mx.mx_quantize(x, fmt)
    X = mx.e8m0_value(scales)[:, :, None].reshape(-1, 1)
    v = (x.astype(np.float64) / X).astype(np.float32)
    inrange = np.abs(v) <= q8.fp8_max(fmt)
    ref = torch.from_numpy(v).to(TORCH[fmt]).view(torch.uint8).numpy()
    assert inrange.mean() > 0.9
    assert (codes[inrange] == ref[inrange]).all()
    # the rest saturate to the largest finite code, keeping the sign
    big = ~inrange
    if big.any():
        assert (q8.decode(codes[big], fmt) == np.sign(v[big]) * q8.fp8_max(fmt)).all()


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_rounding_bound_and_exact_grid(fmt):
    rng = np.random.default_rng(3)
    x = _blocks(rng, 300, (-30, 30)).astype(np.float64)
    codes, scales = mx.mx_quantize(x, fmt)
    deq = mx.mx_dequantize(codes, scales, fmt)
    X = mx.e8m0_value(scales).reshape(-1, 1)
    v = x / X
    ok = np.abs(v) <= q8.fp8_max(fmt)
    # half an ulp of the element's binade (subnormal binade below 2^(1 - bias))
    e = np.floor(np.log2(np.maximum(np.abs(v), 1e-300)))
    e = np.maximum(e, 1 - BIAS[fmt])
    half_ulp = np.ldexp(0.5, (e - MBITS[fmt]).astype(int)) * X
    assert (np.abs(deq - x)[ok] <= half_ulp[ok] * (1 + 1e-12)).all()
    # values already on the scaled grid come back exactly
    assert (mx.mx_dequantize(codes, scales, fmt) == mx.mx_qdq(deq, fmt)).all()


def test_blocks_are_independent():
    rng = np.random.default_rng(4)
    x = _blocks(rng, 6, (-5, 5)).reshape(2, 96)      # two rows of three blocks
    codes, scales = mx.mx_quantize(x, "e4m3")
    assert scales.shape == (2, 3)
    for r in range(2):
        for b in range(3):
            c1, s1 = mx.mx_quantize(x[r:r + 1, 32 * b:32 * b + 32], "e4m3")
            assert (codes[r, 32 * b:32 * b + 32] == c1[0]).all() and scales[r, b] == s1[0, 0]


def test_zero_and_nonfinite_blocks():
    x = np.zeros((3, 32), np.float32)
    x[1, 7] = np.nan
    x[2, 3] = np.inf
    x[2, 4] = 1.0
    codes, scales = mx.mx_quantize(x, "e4m3")
    assert scales.tolist() == [[0], [255], [255]]
    deq = mx.mx_dequantize(codes, scales, "e4m3")
    assert (deq[0] == 0).all()
    assert np.isnan(deq[1]).all() and np.isnan(deq[2]).all()


def test_scale_exponent_is_clamped():
    # amax far above or below the E8M0 range clamps s to [-127, 127]
    assert mx.scale_exponent(np.ldexp(1.0, 1020), "e4m3") == 127
    assert mx.scale_exponent(np.ldexp(1.0, -1070), "e4m3") == -127
    assert mx.scale_exponent(1.0, "e4m3") == -8 and mx.scale_exponent(1.0, "e5m2") == -15


def _mx_layer_inputs(seed, T=160, d=128, f=128, E=5):
    from moe_synth import bf16_bits, bits_to_f64
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    x = bits_to_f64(bf16_bits(rng.standard_normal((T, d)).astype(np.float32)))
    wi = bits_to_f64(bf16_bits((rng.standard_normal((E, d, 2 * f)) * 0.05).astype(np.float32)))
    wo = bits_to_f64(bf16_bits((rng.standard_normal((E, f, d)) * 0.05).astype(np.float32)))
    dout = bits_to_f64(bf16_bits(rng.standard_normal((T, d)).astype(np.float32)))
    return logits, x, wi, wo, dout


def test_without_quantization_mx_layer_is_bf16_layer(monkeypatch):
    """Identity block quantizers and no bf16 rounding: the MXFP8 layer's forward
    and backward reduce exactly to the bf16 oracle's (every GEMM takes the same
    operands, the weight gradients the same rows)."""
    from oracle import moe_ref
    monkeypatch.setattr(q8, "round_bf16", lambda x: np.asarray(x, np.float64))
    monkeypatch.setattr(mx, "mx_qdq", lambda x, fmt: np.asarray(x, np.float64))
    logits, x, wi, wo, dout = _mx_layer_inputs(3)
    for (k, sfn, ren, align, cap) in [(2, 0, 1, 0, 0), (3, 1, 0, 4, 20)]:
        fm = mx.forward(x, logits, wi, wo, k, sfn, ren, align, cap)
        bm = mx.backward(fm, dout, wi, wo, k)
        fr = moe_ref.forward(x, logits, wi, wo, k, sfn, ren, align, cap)
        br = moe_ref.backward(fr, dout, wi, wo, k)
        np.testing.assert_array_equal(fm["out"], fr["out"])
        for key in ("dx", "d_wi", "d_wo", "d_topk_w"):
            np.testing.assert_array_equal(bm[key], br[key])


def test_group_rows_blocks_stay_in_their_group():
    """The weight gradients' blocks run along each expert's rows from its first
    row: changing another expert's rows leaves a group's values unchanged, and a
    group of one row is quantized alone (its scale from that row only)."""
    rng = np.random.default_rng(4)
    x = rng.standard_normal((70, 32)) * np.ldexp(1.0, rng.integers(-6, 6, size=(70, 1)))
    off = np.array([0, 1, 33, 70])
    a = mx.qdq_group_rows(x, off, q8.E4M3)
    y = x.copy()
    y[1:33] *= 1024.0                       # group 1 much larger
    b = mx.qdq_group_rows(y, off, q8.E4M3)
    assert (a[0] == b[0]).all() and (a[33:] == b[33:]).all()
    # row 0 alone: each column is its own one-element block -> exact up to the format
    np.testing.assert_array_equal(a[0], mx.qdq_along(np.vstack([x[:1], np.zeros((31, 32))]), 0,
                                                     q8.E4M3)[0])


def test_mx_layer_close_to_bf16_layer():
    """Quantization noise only: outputs and gradients within a few percent of
    the unquantized layer, and the noise is there."""
    from oracle import moe_ref
    logits, x, wi, wo, dout = _mx_layer_inputs(5)
    fm = mx.forward(x, logits, wi, wo, 2, 0, 1)
    bm = mx.backward(fm, dout, wi, wo, 2)
    fr = moe_ref.forward(x, logits, wi, wo, 2, 0, 1)
    br = moe_ref.backward(fr, dout, wi, wo, 2)

    def rel(a, b):
        return np.linalg.norm(a - b) / np.linalg.norm(b)
    assert 1e-3 < rel(fm["out"], fr["out"]) < 0.08
    for key in ("dx", "d_wi", "d_wo"):
        assert rel(bm[key], br[key]) < 0.15, key
