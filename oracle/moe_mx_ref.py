"""Plain NumPy oracle of block-scaled 8-bit quantization (MXFP8), the
block-scaled recipe the pages name for the expert GEMMs.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module;
only the tests do.  It shares no code with the CUDA path (it reuses the 8-bit
encodings of oracle/moe_fp8_ref.py).

The pages name the block-scaled recipes without their arithmetic
(TransformerEngine PR #2912, wi-fusion commit, FP8 note: MXFP8 / NVFP4 keep
one scale per block, so fusing wi_0 and wi_1 leaves them unaffected).  The
reading taken here is the public OCP Microscaling Formats (MX) v1.0
definition:

  * a block is 32 consecutive elements along the contraction axis (the last
    axis of the arrays below);
  * the block's shared scale is the power of two X = 2^s with
        s = floor(log2(amax)) - emax_elem,
    amax = max |x| over the block, emax_elem the exponent of the element
    format's largest normal (8 for E4M3: 448 = 1.75 * 2^8; 15 for E5M2:
    57344 = 1.75 * 2^15), s clamped to the E8M0 range [-127, 127];
  * X is stored as an E8M0 code (unsigned 8-bit exponent, bias 127; 0xFF is
    NaN);
  * each element is the format's code of x / X, rounded to nearest even and
    saturated to the largest finite value (values of x / X in (448, 512) for
    E4M3 saturate, as the definition allows);
  * value = element value * X.

Readings where the definition leaves a choice: a block of zeros takes the
smallest scale (code 0, X = 2^-127); a block holding a NaN or an infinity
takes the NaN scale (0xFF), and every value of that block decodes to NaN.
"""
from __future__ import annotations

import numpy as np

from oracle import moe_fp8_ref as q8

BLOCK = 32
E8M0_BIAS = 127
E8M0_NAN = 0xFF
_EMAX = {q8.E4M3: 8, q8.E5M2: 15}


def scale_exponent(amax: float, fmt: str) -> int:
    """s = floor(log2(amax)) - emax_elem, clamped to [-127, 127]; amax finite,
    >= 0 (0 gives -127).  floor(log2) from the exact binary exponent
    (np.frexp: amax = m 2^e, 0.5 <= m < 1, so floor(log2(amax)) = e - 1)."""
    if amax == 0.0:
        return -E8M0_BIAS
    _, e = np.frexp(np.float64(amax))
    return int(np.clip(int(e) - 1 - _EMAX[fmt], -E8M0_BIAS, E8M0_BIAS))


def mx_quantize(x, fmt: str):
    """x [..., K] (K a multiple of 32), taken in fp32 (bf16 inputs are exact).
    Returns (codes uint8 [..., K], scale codes uint8 [..., K / 32])."""
    x32 = np.asarray(x, dtype=np.float64).astype(np.float32)
    K = x32.shape[-1]
    assert K % BLOCK == 0, "the contraction axis must hold whole blocks of 32"
    blocks = x32.reshape(-1, K // BLOCK, BLOCK).astype(np.float64)
    codes = np.zeros(blocks.shape, np.uint8)
    scales = np.zeros(blocks.shape[:2], np.uint8)
    for r in range(blocks.shape[0]):
        for b in range(blocks.shape[1]):
            v = blocks[r, b]
            if not np.isfinite(v).all():
                scales[r, b] = E8M0_NAN
                continue
            s = scale_exponent(float(np.abs(v).max()), fmt)
            scales[r, b] = s + E8M0_BIAS
            codes[r, b] = q8.encode(v / np.ldexp(1.0, s), fmt)   # exact power-of-two division
    return codes.reshape(x32.shape), scales.reshape(x32.shape[:-1] + (K // BLOCK,))


def e8m0_value(scale_codes) -> np.ndarray:
    """2^(code - 127), NaN for 0xFF."""
    c = np.asarray(scale_codes, dtype=np.int64)
    return np.where(c == E8M0_NAN, np.nan, np.ldexp(1.0, c - E8M0_BIAS))


def mx_dequantize(codes, scale_codes, fmt: str) -> np.ndarray:
    """Element values times their block's scale (float64)."""
    codes = np.asarray(codes)
    K = codes.shape[-1]
    el = q8.decode(codes, fmt).reshape(-1, K // BLOCK, BLOCK)
    sc = e8m0_value(scale_codes).reshape(-1, K // BLOCK, 1)
    return (el * sc).reshape(codes.shape)


def mx_qdq(x, fmt: str) -> np.ndarray:
    """Quantize and dequantize (the values a block-scaled GEMM multiplies)."""
    c, s = mx_quantize(x, fmt)
    return mx_dequantize(c, s, fmt)
