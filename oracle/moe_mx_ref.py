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
from oracle import moe_ref

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
    finite = np.isfinite(blocks).all(axis=-1)
    amax = np.where(finite, np.abs(np.where(np.isfinite(blocks), blocks, 0.0)).max(axis=-1), 0.0)
    # scale_exponent of every block at once: floor(log2 amax) = e - 1 from frexp
    _, e = np.frexp(amax)
    s = np.where(amax == 0.0, -E8M0_BIAS,
                 np.clip(e.astype(np.int64) - 1 - _EMAX[fmt], -E8M0_BIAS, E8M0_BIAS))
    scaled = blocks / np.ldexp(1.0, s)[..., None]          # exact power-of-two division
    codes = np.where(finite[..., None], q8.encode(np.where(finite[..., None], scaled, 0.0), fmt),
                     0).astype(np.uint8)
    scales = np.where(finite, s + E8M0_BIAS, E8M0_NAN).astype(np.uint8)
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


# ----------------------------------------------------------------------------
# the layer with block-scaled GEMM operands
# ----------------------------------------------------------------------------
def qdq_along(x, axis: int, fmt: str) -> np.ndarray:
    """mx_qdq with the blocks of 32 along `axis` (the contraction axis of the
    GEMM the tensor feeds)."""
    x = np.moveaxis(np.asarray(x, dtype=np.float64), axis, -1)
    return np.moveaxis(mx_qdq(x, fmt), -1, axis)


def qdq_group_rows(x, group_offsets, fmt: str) -> np.ndarray:
    """Blocks of 32 along the rows of each expert's group (the contraction of
    the weight-gradient GEMMs), aligned at the group's first row; the last
    block of a group is completed with zeros, never with the next group's
    rows."""
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    for e in range(len(group_offsets) - 1):
        lo, hi = int(group_offsets[e]), int(group_offsets[e + 1])
        if hi == lo:
            continue
        n = (hi - lo + BLOCK - 1) // BLOCK * BLOCK
        g = np.zeros((n, x.shape[1]))
        g[:hi - lo] = x[lo:hi]
        out[lo:hi] = qdq_along(g, 0, fmt)[:hi - lo]
    return out


def forward(x, logits, wi, wo, k, score_fn, renorm, align=0, capacity=0):
    """The layer's forward with MXFP8 GEMM operands: every GEMM multiplies the
    block-scaled E4M3 values of its operands, blocks along the contraction
    (Xs and wi along d_model, Act and wo along d_ff); the stored activations
    are bf16 (Act rounded to bf16 before it is quantized), as in the
    current-scaling oracle (oracle/moe_fp8_ref.py)."""
    E = wi.shape[0]
    topk_idx, topk_w = moe_ref.route_topk(logits, k, score_fn, renorm)
    lay = moe_ref.permute_layout(topk_idx, E, align, capacity)
    off = lay["group_offsets"]
    R = lay["R"]
    xs = moe_ref.permute_rows(x, lay, k)[:R]
    h = moe_ref.gmm(qdq_along(xs, 1, q8.E4M3), qdq_along(wi, 1, q8.E4M3), off)
    act = q8.round_bf16(moe_ref.swiglu(h))
    y = moe_ref.gmm(qdq_along(act, 1, q8.E4M3), qdq_along(wo, 1, q8.E4M3), off)
    out = moe_ref.combine(y, lay["flat_to_sorted"], topk_w)
    return dict(topk_idx=topk_idx, topk_w=topk_w, layout=lay, xs=xs, h=h, act=act, y=y,
                out=out)


def backward(fw: dict, d_out, wi, wo, k):
    """The backward with MXFP8 operands: dY and dH in E5M2 (blocks along
    d_model for dY, along 2 d_ff for dH), the weights re-quantized along the
    dgrad GEMMs' contraction (wo along d_model, wi along 2 d_ff), and the
    weight gradients' operands quantized along the expert's rows (Act, Xs in
    E4M3, dY, dH in E5M2)."""
    lay = fw["layout"]
    off = lay["group_offsets"]
    E = wi.shape[0]
    T = d_out.shape[0]
    R = lay["R"]
    dy, d_topk_w = moe_ref.combine_bwd(d_out, fw["y"], lay["flat_to_sorted"], fw["topk_w"], R)
    dy = q8.round_bf16(dy[:R])
    d_act = moe_ref.gmm(qdq_along(dy, 1, q8.E5M2), qdq_along(wo, 2, q8.E4M3), off,
                        transpose_rhs=True)
    dh = q8.round_bf16(moe_ref.swiglu_bwd(q8.round_bf16(fw["h"]), d_act))
    d_wo = moe_ref.tgmm(qdq_group_rows(fw["act"], off, q8.E4M3),
                        qdq_group_rows(dy, off, q8.E5M2), off, E)
    d_xs = moe_ref.gmm(qdq_along(dh, 1, q8.E5M2), qdq_along(wi, 2, q8.E4M3), off,
                       transpose_rhs=True)
    d_wi = moe_ref.tgmm(qdq_group_rows(fw["xs"], off, q8.E4M3),
                        qdq_group_rows(dh, off, q8.E5M2), off, E)
    dx = moe_ref.dispatch_bwd(d_xs, lay["flat_to_sorted"], T, k)
    return dict(dy=dy, d_topk_w=d_topk_w, dh=dh, d_wo=d_wo, d_xs=d_xs, d_wi=d_wi, dx=dx)
