"""Pins of the FP8 oracle (oracle/moe_fp8_ref.py) against things other than
itself (CPU only):

* hand-decoded codes and rounding cases (tests/golden/fp8_codes_hand.json);
* PyTorch's float8_e4m3fn / float8_e5m2 conversions (library routine) for every
  code and for in-range fp32 values;
* round trips, the half-ulp error bound of current scaling;
* with quantization switched off, the FP8 layer is the bf16 oracle's layer
  (which is pinned on its own) — so every operand sits where the recipe puts it.
"""
import json
import os

import numpy as np
import pytest
import torch

from oracle import moe_fp8_ref as q8
from oracle import moe_ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _val(v):
    return float(v) if not isinstance(v, str) else float(v.replace("inf", "inf"))


def test_golden_codes_and_rounding():
    g = json.load(open(os.path.join(GOLDEN, "fp8_codes_hand.json")))
    for fmt in ("e4m3", "e5m2"):
        for code, want, _ in g[fmt]:
            got = float(q8.decode(int(code, 16), fmt))
            want = float(want)
            if np.isnan(want):
                assert np.isnan(got), (fmt, code)
            else:
                assert got == want and np.signbit(got) == np.signbit(want), (fmt, code, got)
    for fmt, x, code, _ in g["rounding"]:
        assert int(q8.encode(np.float32(x), fmt)) == int(code, 16), (fmt, x)


@pytest.mark.parametrize("fmt,tdt", [("e4m3", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)])
def test_decode_every_code_matches_torch(fmt, tdt):
    codes = np.arange(256, dtype=np.uint8)
    ours = q8.decode(codes, fmt)
    ref = torch.from_numpy(codes).view(tdt).to(torch.float64).numpy()
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert (both_nan | (ours == ref)).all()


@pytest.mark.parametrize("fmt,tdt", [("e4m3", torch.float8_e4m3fn), ("e5m2", torch.float8_e5m2)])
def test_encode_matches_torch_in_range(fmt, tdt):
    rng = np.random.default_rng(7)
    mx = q8.fp8_max(fmt)
    x = np.concatenate([
        rng.uniform(-mx, mx, 20000), rng.standard_normal(20000) * 3,
        rng.standard_normal(20000) * 1e-3, rng.standard_normal(5000) * 1e-6,
        # exact midpoints between neighbouring codes
        (q8.decode(np.arange(0, 123), fmt) + q8.decode(np.arange(1, 124), fmt)) / 2,
    ]).astype(np.float32)
    x = x[np.isfinite(x) & (np.abs(x) <= mx)]
    ours = q8.encode(x, fmt)
    ref = torch.from_numpy(x).to(tdt).view(torch.uint8).numpy()
    mism = ours != ref
    assert not mism.any(), (x[mism][:5], ours[mism][:5], ref[mism][:5])


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_round_trip_and_saturation(fmt):
    codes = np.arange(256, dtype=np.uint8)
    vals = q8.decode(codes, fmt)
    fin = np.isfinite(vals)
    assert (q8.encode(vals[fin].astype(np.float32), fmt) == codes[fin]).all()
    mx = q8.fp8_max(fmt)
    big = np.array([mx * 1.01, mx * 4, np.inf, -np.inf, -mx * 2], np.float32)
    dec = q8.decode(q8.encode(big, fmt), fmt)
    assert (dec == np.array([mx, mx, mx, -mx, -mx])).all()
    assert q8.encode(np.float32(np.nan), fmt) == 0x7F


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_current_scaling_error_bound(fmt):
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((64, 48)) * 5).astype(np.float32)
    deq, codes, s = q8.qdq_tensor(x, fmt)
    amax = np.abs(x).max()
    assert s == np.float32(np.float32(q8.fp8_max(fmt)) / np.float32(amax))
    # the largest element maps onto the largest code
    i = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert abs(float(q8.decode(codes[i], fmt))) == q8.fp8_max(fmt)
    mbits = 3 if fmt == "e4m3" else 2
    bias = 7 if fmt == "e4m3" else 15
    half_ulp_rel = 2.0 ** -(mbits + 1)
    sub_abs = 2.0 ** (1 - bias - mbits - 1) / float(s)   # half the subnormal step, unscaled
    err = np.abs(deq - x)
    assert (err <= half_ulp_rel * np.abs(x) * (1 + 1e-6) + sub_abs).all()
    assert q8.current_scale(0.0, fmt) == 1.0 and q8.current_scale(np.inf, fmt) == 1.0


def _layer_inputs(seed, T=40, d=16, f=24, E=5):
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((T, E)).astype(np.float32)
    x = rng.standard_normal((T, d))
    wi = rng.standard_normal((E, d, 2 * f)) * 0.3
    wo = rng.standard_normal((E, f, d)) * 0.3
    dout = rng.standard_normal((T, d))
    return logits, x, wi, wo, dout


def test_round_bf16_matches_torch():
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.standard_normal(50000) * 10.0 ** rng.uniform(-30, 30, 50000),
                        [0.0, -0.0, 1.0, 3.0e38, -1e-40, np.inf, -np.inf]])
    x32 = x.astype(np.float32)
    want = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    got = q8.round_bf16(x32)
    assert ((got == want) | (np.isnan(got) & np.isnan(want))).all()


def test_without_quantization_fp8_layer_is_bf16_layer(monkeypatch):
    """Identity quantizers and no bf16 rounding: the FP8 forward / backward
    reduce exactly to the bf16 oracle's (same operands in every GEMM, same
    transposes)."""
    monkeypatch.setattr(q8, "round_bf16", lambda x: np.asarray(x, np.float64))
    monkeypatch.setattr(q8, "qdq_tensor", lambda x, fmt: (np.asarray(x, np.float64), None, 1.0))
    monkeypatch.setattr(q8, "qdq_per_expert", lambda w, fmt: (np.asarray(w, np.float64), None,
                                                               np.ones(w.shape[0])))
    logits, x, wi, wo, dout = _layer_inputs(11)
    for (k, sfn, ren, align, cap) in [(2, 0, 1, 0, 0), (3, 1, 0, 4, 20)]:
        f8 = q8.forward(x, logits, wi, wo, k, sfn, ren, align, cap)
        b8 = q8.backward(f8, dout, k)
        fr = moe_ref.forward(x, logits, wi, wo, k, sfn, ren, align, cap)
        br = moe_ref.backward(fr, dout, wi, wo, k)
        np.testing.assert_array_equal(f8["out"], fr["out"])
        for key in ("dx", "d_wi", "d_wo", "d_topk_w"):
            np.testing.assert_array_equal(b8[key], br[key])


def test_fp8_layer_close_to_bf16_layer():
    """Quantization noise only: outputs and gradients within a few percent."""
    logits, x, wi, wo, dout = _layer_inputs(12, T=200, d=64, f=96, E=6)
    f8 = q8.forward(x, logits, wi, wo, 2, 0, 1)
    b8 = q8.backward(f8, dout, 2)
    fr = moe_ref.forward(x, logits, wi, wo, 2, 0, 1)
    br = moe_ref.backward(fr, dout, wi, wo, 2)

    def rel(a, b):
        return np.linalg.norm(a - b) / np.linalg.norm(b)
    assert rel(f8["out"], fr["out"]) < 0.08
    assert rel(b8["dx"], br["dx"]) < 0.15
    assert rel(b8["d_wi"], br["d_wi"]) < 0.15
    assert rel(b8["d_wo"], br["d_wo"]) < 0.15
    # ... and the error is really there (quantization happened)
    assert rel(f8["out"], fr["out"]) > 1e-3


@pytest.mark.parametrize("fmt", [q8.E4M3, q8.E5M2])
def test_encode_lib_is_encode(fmt):
    """The library path of the codes gives encode()'s codes: every fp32 around
    each grid value (ties, both neighbours), subnormals, zeros of both signs,
    values past the largest finite one (saturated), infinities and NaN, and a
    wide random sample."""
    grid, _ = q8._finite_grid(fmt)
    mids = (grid[1:] + grid[:-1]) / 2
    pts = np.concatenate([grid, mids, np.nextafter(mids.astype(np.float32), np.float32(0)),
                          np.nextafter(mids.astype(np.float32), np.float32(1e9)),
                          [q8.fp8_max(fmt) * 1.03, q8.fp8_max(fmt) * 7, 1e30, np.inf]])
    rng = np.random.default_rng(5)
    rnd = rng.standard_normal(200000) * np.exp(rng.uniform(-12, 12, 200000))
    x = np.concatenate([pts, -pts, rnd, [0.0, -0.0, np.nan, -np.inf]]).astype(np.float32)
    assert (q8.encode_lib(x, fmt) == q8.encode(x, fmt)).all()


def test_layer_scales_are_the_layer_scales():
    """The blockwise scale computation for full-size layers gives exactly the
    scales forward() / backward() take from whole tensors (blocks smaller than
    an expert's rows, so that several blocks meet in one amax)."""
    from moe_synth import bits_to_f64, make_inputs, scaled, CONFIGS
    cfg = scaled(CONFIGS["skewed"], T=2048, d=128, f=96, capacity=48)
    inp = make_inputs(cfg, seed=2)
    x, wi, wo, dout = (bits_to_f64(inp[n]) for n in ("x", "wi", "wo", "dout"))
    fw = q8.forward(x, inp["logits"], wi, wo, cfg.k, cfg.score_fn, cfg.renorm, cfg.align,
                    cfg.capacity)
    bw = q8.backward(fw, dout, cfg.k)
    sc = q8.layer_scales(x, inp["logits"], wi, wo, dout, cfg.k, cfg.score_fn, cfg.renorm,
                         cfg.align, cfg.capacity, block_rows=7)
    want = dict(fw["scales"], **bw["scales"])
    for key in ("x", "act", "dy", "dh"):
        assert sc["scales"][key] == want[key], key
    for key in ("wi", "wo"):
        assert (sc["scales"][key] == want[key]).all(), key
    R = fw["layout"]["R"]
    assert (sc["xs_q"] == fw["xs_q"]).all()
    assert (sc["dy_q"] == bw["dy_q"][:R]).all()
