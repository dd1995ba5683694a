"""Plain NumPy oracle of the FP8 expert layer: 8-bit float encodings, current
tensor scaling, and the layer's forward / backward with FP8 grouped GEMMs.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module;
only the tests and the benchmark's CPU-baseline leg do.  It shares no code with
the CUDA path (it reuses the bf16 oracle's routing, permutation, SwiGLU and
gmm / tgmm definitions from oracle/moe_ref.py).

The recipe is the one the pages configure for the expert GEMMs: MaxText PR
#2319, "[Draft] Integrate TE/JAX GroupedGEMM for MoE", review thread on the
quantizer settings in moe.py: current tensor scaling, forward dtype
float8_e4m3fn, backward dtype float8_e5m2, 2x quantization (a row-wise and a
column-wise copy of each operand).  TransformerEngine PR #2912, the wi-fusion
commit's FP8 note: the fused [wi_0 | wi_1] weight takes one amax per expert
over [H, 2M].

The formats (OCP 8-bit floating point): E4M3FN has 4 exponent bits with bias
7, 3 mantissa bits, no infinities, S.1111.111 is NaN, largest finite 448;
E5M2 has 5 exponent bits with bias 15, 2 mantissa bits, IEEE-style infinities
and NaNs, largest finite 57344.  Both have subnormals.

Readings (the pages name the recipe, not its arithmetic):
  * scale = fp8_max / amax in fp32 (1 when amax is 0 or not finite); the
    quantized code is round-to-nearest-even of fp32(x * scale), saturated to
    the largest finite value; dequantization multiplies by 1 / scale;
  * activations take one scale per tensor (the rows of all groups), weights
    one per expert; gradients dY and dH are quantized to E5M2 per tensor;
  * quantization points: Xs, Act (forward inputs of the two GEMMs), wi, wo
    (per expert), dY and dH (backward inputs); every GEMM accumulates the
    dequantized products exactly (fp64 here, fp32 on the GPU);
  * the quantized activations are the layer's bf16 tensors (the pages train
    in bf16): Act, dY and dH are rounded to bf16 (round-to-nearest-even)
    before their amax and codes are taken, and the SwiGLU backward reads the
    stored bf16 H.
"""
from __future__ import annotations

import numpy as np

from oracle import moe_ref

E4M3 = "e4m3"
E5M2 = "e5m2"
_FMT = {E4M3: dict(ebits=4, mbits=3, bias=7, max=448.0),
        E5M2: dict(ebits=5, mbits=2, bias=15, max=57344.0)}


def round_bf16(x) -> np.ndarray:
    """Round to bf16 (nearest, ties to even) through fp32; returns float64."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    out = u.astype(np.uint32).view(np.float32).astype(np.float64)
    return np.where(np.isnan(f), np.nan, out)


def fp8_max(fmt: str) -> float:
    return _FMT[fmt]["max"]


def decode(codes, fmt: str) -> np.ndarray:
    """Values of 8-bit codes (float64), from the bit fields."""
    f = _FMT[fmt]
    c = np.asarray(codes, dtype=np.int64) & 0xFF
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> f["mbits"]) & ((1 << f["ebits"]) - 1)
    m = c & ((1 << f["mbits"]) - 1)
    frac = m / float(1 << f["mbits"])
    val = np.where(e == 0, frac * 2.0 ** (1 - f["bias"]),
                   (1.0 + frac) * 2.0 ** (e.astype(np.float64) - f["bias"]))
    emax = (1 << f["ebits"]) - 1
    if fmt == E4M3:
        val = np.where((e == emax) & (m == (1 << f["mbits"]) - 1), np.nan, val)
    else:
        val = np.where((e == emax) & (m == 0), np.inf, val)
        val = np.where((e == emax) & (m != 0), np.nan, val)
    return sign * val


def _finite_grid(fmt: str):
    """Non-negative finite values and their codes, ascending."""
    codes = np.arange(128)
    vals = decode(codes, fmt)
    ok = np.isfinite(vals)
    return vals[ok], codes[ok]


def encode(x, fmt: str) -> np.ndarray:
    """Round-to-nearest-even of fp32 values onto the format's grid, saturated
    to the largest finite value (NaN -> the NaN code 0x7F).  Returns uint8."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    grid, gcodes = _finite_grid(fmt)
    a = np.abs(x)
    a_clip = np.minimum(np.nan_to_num(a, nan=0.0, posinf=np.inf), grid[-1])
    hi = np.clip(np.searchsorted(grid, a_clip, side="left"), 0, len(grid) - 1)
    lo = np.clip(hi - 1, 0, len(grid) - 1)
    d_hi = grid[hi] - a_clip
    d_lo = a_clip - grid[lo]
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (gcodes[hi] % 2 == 0))
    code = np.where(pick_hi, gcodes[hi], gcodes[lo])
    code = np.where(a >= grid[-1], gcodes[-1], code)          # saturate (inf included)
    code = code | np.where(np.signbit(x), 0x80, 0)
    code = np.where(np.isnan(x), 0x7F, code)
    return code.astype(np.uint8)


def encode_lib(x, fmt: str) -> np.ndarray:
    """The codes of encode() through PyTorch's float8 conversion (round to
    nearest, ties to even) after saturating to the largest finite value; NaN
    gives the NaN code 0x7F as in encode().  A library step for tensors of
    billions of elements, where encode's per-element search over the value
    grid is too slow; the CPU tests pin it to encode() code for code."""
    import torch
    x32 = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    mx = np.float32(fp8_max(fmt))
    dt = torch.float8_e4m3fn if fmt == E4M3 else torch.float8_e5m2
    codes = torch.from_numpy(np.clip(x32, -mx, mx)).to(dt).view(torch.uint8).numpy()
    return np.where(np.isnan(x32), np.uint8(0x7F), codes).astype(np.uint8)


def current_scale(amax: float, fmt: str) -> np.float32:
    """fp32 scale fp8_max / amax (1 when amax is 0 or not finite)."""
    amax = np.float32(amax)
    if not np.isfinite(amax) or amax <= 0:
        return np.float32(1.0)
    return np.float32(np.float32(fp8_max(fmt)) / amax)


def quantize(x, scale, fmt: str) -> np.ndarray:
    """Codes of fp32(x * scale); x is taken in fp32 (bf16 inputs are exact)."""
    xs = (np.asarray(x, dtype=np.float32) * np.float32(scale)).astype(np.float32)
    return encode(xs, fmt)


def dequantize(codes, scale, fmt: str) -> np.ndarray:
    return decode(codes, fmt) / np.float64(np.float32(scale))


def qdq_tensor(x, fmt: str):
    """Per-tensor current scaling: (dequantized values, codes, scale)."""
    x32 = np.asarray(x, dtype=np.float64).astype(np.float32)
    amax = np.float32(np.abs(x32).max()) if x32.size else np.float32(0)
    s = current_scale(amax, fmt)
    q = quantize(x32, s, fmt)
    return dequantize(q, s, fmt), q, s


def qdq_per_expert(w, fmt: str):
    """One scale per expert (leading axis): (dequantized, codes, scales [E])."""
    w32 = np.asarray(w, dtype=np.float64).astype(np.float32)
    deq = np.empty(w32.shape)
    codes = np.empty(w32.shape, np.uint8)
    scales = np.empty(w32.shape[0], np.float32)
    for e in range(w32.shape[0]):
        deq[e], codes[e], scales[e] = qdq_tensor(w32[e], fmt)
    return deq, codes, scales


def forward(x, logits, wi, wo, k, score_fn, renorm, align=0, capacity=0):
    """FP8 forward: the bf16 oracle's layer with Xs, Act (per tensor) and wi, wo
    (per expert) quantized to E4M3 before their grouped GEMMs."""
    E = wi.shape[0]
    topk_idx, topk_w = moe_ref.route_topk(logits, k, score_fn, renorm)
    lay = moe_ref.permute_layout(topk_idx, E, align, capacity)
    xs = moe_ref.permute_rows(x, lay, k)
    off = lay["group_offsets"]
    R = lay["R"]
    xs_q, _, s_x = qdq_tensor(xs[:R], E4M3)
    wi_q, _, s_wi = qdq_per_expert(wi, E4M3)
    wo_q, _, s_wo = qdq_per_expert(wo, E4M3)
    h = moe_ref.gmm(xs_q, wi_q, off)
    act = round_bf16(moe_ref.swiglu(h))
    act_q, _, s_act = qdq_tensor(act, E4M3)
    y = moe_ref.gmm(act_q, wo_q, off)
    out = moe_ref.combine(y, lay["flat_to_sorted"], topk_w)
    return dict(topk_idx=topk_idx, topk_w=topk_w, layout=lay, xs=xs, xs_q=xs_q, wi_q=wi_q,
                wo_q=wo_q, h=h, act=act, act_q=act_q, y=y, out=out,
                scales=dict(x=s_x, wi=s_wi, wo=s_wo, act=s_act))


def backward(fw: dict, d_out, k):
    """FP8 backward: dY and dH quantized to E5M2 per tensor; the dgrad GEMMs
    take the forward's E4M3 weights, the weight-gradient GEMMs the forward's
    E4M3 activations (the column-wise copies of the 2x quantization)."""
    lay = fw["layout"]
    off = lay["group_offsets"]
    E = fw["wi_q"].shape[0]
    T = d_out.shape[0]
    R = lay["R"]
    dy, d_topk_w = moe_ref.combine_bwd(d_out, fw["y"], lay["flat_to_sorted"], fw["topk_w"], R)
    dy = round_bf16(dy)
    dy_q, _, s_dy = qdq_tensor(dy, E5M2)
    d_act = moe_ref.gmm(dy_q, fw["wo_q"], off, transpose_rhs=True)
    dh = round_bf16(moe_ref.swiglu_bwd(round_bf16(fw["h"]), d_act))
    d_wo = moe_ref.tgmm(fw["act_q"], dy_q, off, E)
    dh_q, _, s_dh = qdq_tensor(dh, E5M2)
    d_xs = moe_ref.gmm(dh_q, fw["wi_q"], off, transpose_rhs=True)
    d_wi = moe_ref.tgmm(fw["xs_q"], dh_q, off, E)
    dx = moe_ref.dispatch_bwd(d_xs, lay["flat_to_sorted"], T, k)
    return dict(dy=dy, dy_q=dy_q, d_topk_w=d_topk_w, d_act=d_act, dh=dh, dh_q=dh_q, d_wo=d_wo,
                d_xs=d_xs, d_wi=d_wi, dx=dx, scales=dict(dy=s_dy, dh=s_dh))


def _qdq_lib(x, scale, fmt):
    """dequantize(quantize(x, scale)) with the codes from encode_lib."""
    xs = (np.asarray(x, dtype=np.float32) * np.float32(scale)).astype(np.float32)
    return dequantize(encode_lib(xs, fmt), scale, fmt)


def layer_scales(x, logits, wi, wo, d_out, k, score_fn, renorm, align=0, capacity=0,
                 block_rows=2048):
    """The scales forward() and backward() take, for a layer too large to keep
    every intermediate: x, Act, dY, dH one each, wi and wo one per expert.

    The same steps as forward / backward (routing, permutation, per-tensor
    amax of the bf16-rounded tensors, per-expert amax of the weights), with
    the grouped GEMMs of Act = SwiGLU(Xs_q wi_q) and dH = SwiGLU'(H, dY_q wo_q^T)
    taken expert by expert over blocks of rows in fp64, keeping only each
    block's amax.  dY = w[t, j] * d_out[t] on the row of every kept assignment
    (TE-2912, review thread on _combine_bwd), zero on padding rows.
    wi, wo: anything that gives expert e's weights as wi[e] (converted to
    float64 one expert at a time) and E as len(wi).
    Returns the routing, the layout, Xs_q and dY_q (dequantized, R rows) and
    the scales (fp32 numbers; wi, wo arrays of E)."""
    E = len(wi)
    T, d = x.shape
    topk_idx, topk_w = moe_ref.route_topk(logits, k, score_fn, renorm)
    lay = moe_ref.permute_layout(topk_idx, E, align, capacity)
    off = lay["group_offsets"]
    R = lay["R"]
    xs = moe_ref.permute_rows(x, lay, k)[:R]
    s_x = current_scale(np.abs(xs.astype(np.float32)).max() if R else 0.0, E4M3)
    xs_q = _qdq_lib(xs, s_x, E4M3)
    s2f = lay["sorted_to_flat"]
    kept = s2f >= 0
    dy = np.zeros((R, d))
    a = s2f[kept]
    dy[kept] = round_bf16(topk_w.reshape(-1)[a][:, None] * d_out[a // k])
    s_dy = current_scale(np.abs(dy.astype(np.float32)).max() if R else 0.0, E5M2)
    dy_q = _qdq_lib(dy, s_dy, E5M2)
    s_wi = np.empty(E, np.float32)
    s_wo = np.empty(E, np.float32)
    amax_act = 0.0
    amax_dh = 0.0
    for e in range(E):
        wi_e = np.asarray(wi[e], dtype=np.float64)
        wo_e = np.asarray(wo[e], dtype=np.float64)
        s_wi[e] = current_scale(np.abs(wi_e.astype(np.float32)).max(), E4M3)
        s_wo[e] = current_scale(np.abs(wo_e.astype(np.float32)).max(), E4M3)
        lo, hi = int(off[e]), int(off[e + 1])
        if hi == lo:
            continue
        wi_q = _qdq_lib(wi_e, s_wi[e], E4M3)
        wo_q = _qdq_lib(wo_e, s_wo[e], E4M3)
        for r0 in range(lo, hi, block_rows):
            r1 = min(hi, r0 + block_rows)
            h = xs_q[r0:r1] @ wi_q
            amax_act = max(amax_act, float(np.abs(round_bf16(moe_ref.swiglu(h))).max()))
            d_act = dy_q[r0:r1] @ wo_q.T
            dh = round_bf16(moe_ref.swiglu_bwd(round_bf16(h), d_act))
            amax_dh = max(amax_dh, float(np.abs(dh).max()))
    return dict(topk_idx=topk_idx, topk_w=topk_w, layout=lay, xs_q=xs_q, dy_q=dy_q,
                scales=dict(x=s_x, act=current_scale(amax_act, E4M3), dy=s_dy,
                            dh=current_scale(amax_dh, E5M2), wi=s_wi, wo=s_wo))
