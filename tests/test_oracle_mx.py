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
