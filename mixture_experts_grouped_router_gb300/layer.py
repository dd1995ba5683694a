"""The MoE expert layer, forward and backward, as a sequence of C-ABI calls.

This module only allocates device buffers (through PyTorch) and issues the
library calls in order on the current stream; every arithmetic step runs in
libmoe_gb300.so.  The sequence follows the single-VJP MoE block of
TransformerEngine PR #2912 ("[JAX] Add an MoE Block (Layer) that compound
router, permutation, groupedGEMM and communication", sequence diagram),
without the expert-parallel all-to-all:

forward   route_topk -> permute -> gmm(up, SwiGLU epilogue) -> gmm(down) -> combine
backward  unpermute_bwd -> route_topk_bwd (d_logits) -> gmm(dgrad down, SwiGLU-bwd
          epilogue) -> tgmm(dWo) -> gmm(dgrad up) -> tgmm(dWi) -> combine without
          weights (dispatch bwd)

Routing options: group-limited top-k (num_groups > 1: only the topk_group
best expert groups compete), DeepSeek-V3's per-expert selection bias
(``forward(..., expert_bias=...)``: experts are ranked by logit + bias, the
routing weights use the unbiased logits) and, with aux_coeff > 0, the
auxiliary load-balancing loss (forward: b.aux_loss; backward: its logit
gradient is added to b.d_logits).

With fp8=True the four GEMMs run on 8-bit float codes with current tensor
scaling (MaxText PR #2319, "[Draft] Integrate TE/JAX GroupedGEMM for MoE",
review thread on the quantizer settings): Xs, Act, wi, wo in E4M3 (weights
one scale per expert), dY and dH in E5M2, each quantized to a row-wise copy
and a column-wise copy (the latter feeds the weight-gradient GEMMs).

With bias=True the expert FFN carries biases (bi [E, 2f] on [gate | up],
bo [E, d] on the output), added in the GEMM epilogues; their gradients are
per-expert column sums of dH and dY (moe_group_colsum).

With mxfp8=True the four GEMM pairs run block-scaled (MXFP8, TE-2912's
wi-fusion commit names the recipe; the arithmetic is the OCP MX definition):
every operand is quantized with one power-of-two scale per 32 elements along
the contraction of the GEMM it feeds, E4M3 in the forward (Xs, Act, wi, wo),
E5M2 for the gradients (dY, dH); the weights are quantized twice (along each
of their two contractions), the weight gradients read block-scaled
column-wise copies of Xs, Act, dY and dH.

Weight gradients (bf16): by default the weight-gradient GEMMs read the
row-wise tensors as stored (MN-major operands).  With wgrad_colwise both
operands of dWo = Act^T dY and dWi = Xs^T dH are read K-major from
column-wise copies in the padded group layout instead: the SwiGLU forward /
backward epilogues write the copies of Act and dH beside their row-wise
outputs, moe_transpose_act makes those of Xs and dY.  The weight gradients
then run 10% faster, but writing the copies costs more than that on a
power-capped GB300, so it is not the default.

With num_chunks > 1 the up-projection runs as num_chunks K-chunks of d_model
accumulating into an fp32 partial sum in place (MaxText PR #4295, "Overlap
moe comms with collective matmul", Description), SwiGLU fused into the last
chunk; in the backward each chunk's dgrad and tgmm work on their own slice.
"""
from __future__ import annotations

import dataclasses

import torch

from . import _lib as L


@dataclasses.dataclass
class LayerShape:
    T: int
    d: int
    f: int
    E: int
    k: int
    score_fn: int = L.SCORE_SOFTMAX
    renorm: int = 1
    align: int = 0
    capacity: int = 0
    num_chunks: int = 1
    bias: bool = False
    num_groups: int = 0
    topk_group: int = 0
    aux_coeff: float = 0.0
    fp8: bool = False
    wgrad_colwise: bool = False
    mxfp8: bool = False


class MoEBuffers:
    """Device buffers of one layer instance, allocated once and reused every step."""

    def __init__(self, s: LayerShape, device="cuda", dw_dtype=torch.bfloat16):
        self.s = s
        T, d, f, E, k = s.T, s.d, s.f, s.E, s.k
        if s.num_chunks > 1 and d % s.num_chunks != 0:
            # the chunks must tile d_model exactly (MaxText PR #4295, Description:
            # the up-projection is split evenly along d_model)
            raise ValueError("num_chunks=%d does not divide d_model=%d" % (s.num_chunks, d))
        self.rows_cap = L.moe_rows_cap(T, E, k, s.align, s.capacity)
        R = self.rows_cap
        bf, i32, f32 = torch.bfloat16, torch.int32, torch.float32
        dev = device
        self.topk_idx = torch.empty(T, k, dtype=i32, device=dev)
        self.topk_w = torch.empty(T, k, dtype=f32, device=dev)
        self.xs = torch.empty(R, d, dtype=bf, device=dev)
        self.group_sizes = torch.empty(E, dtype=i32, device=dev)
        self.kept_counts = torch.empty(E, dtype=i32, device=dev)
        self.group_offsets = torch.empty(E + 1, dtype=i32, device=dev)
        self.s2f = torch.empty(R, dtype=i32, device=dev)
        self.f2s = torch.empty(T * k, dtype=i32, device=dev)
        self.ws = torch.empty(L.moe_permute_workspace_bytes(T, E), dtype=torch.uint8, device=dev)
        self.h = torch.empty(R, 2 * f, dtype=bf, device=dev)
        self.act = torch.empty(R, f, dtype=bf, device=dev)
        self.y = torch.empty(R, d, dtype=bf, device=dev)
        self.out = torch.empty(T, d, dtype=bf, device=dev)
        self.p = torch.empty(R, 2 * f, dtype=f32, device=dev) if s.num_chunks > 1 else None
        # backward
        self.dy = torch.empty(R, d, dtype=bf, device=dev)
        self.d_topk_w = torch.empty(T, k, dtype=f32, device=dev)
        self.d_logits = torch.empty(T, E, dtype=f32, device=dev)
        self.logits = None
        self.dh = torch.empty(R, 2 * f, dtype=bf, device=dev)
        self.dxs = torch.empty(R, d, dtype=bf, device=dev)
        self.dx = torch.empty(T, d, dtype=bf, device=dev)
        self.dwi = torch.empty(E, d, 2 * f, dtype=dw_dtype, device=dev)
        self.dwo = torch.empty(E, f, d, dtype=dw_dtype, device=dev)
        self.dbi = torch.empty(E, 2 * f, dtype=f32, device=dev) if s.bias else None
        self.dbo = torch.empty(E, d, dtype=f32, device=dev) if s.bias else None
        self.dev_status = torch.zeros(1, dtype=i32, device=dev)
        if s.mxfp8:
            if s.fp8 or s.bias or s.num_chunks > 1:
                raise ValueError("the MXFP8 layer takes neither biases, K-chunks nor fp8")
            if d % 128 or f % 128:
                raise ValueError("MXFP8 needs d_model and d_ff multiples of 128")
            self._alloc_mx(dev)
        self.colwise = s.wgrad_colwise and not s.fp8 and not s.mxfp8
        if self.colwise:
            # column-wise copies (padded group layout) of the weight gradients' operands
            P = L.moe_fp8_padded_rows(R, E)
            self.xs_t = torch.empty(d, P, dtype=bf, device=dev)
            self.act_t = torch.empty(f, P, dtype=bf, device=dev)
            self.dy_t = torch.empty(d, P, dtype=bf, device=dev)
            self.dh_t = torch.empty(2 * f, P, dtype=bf, device=dev)
        if s.fp8:
            if s.bias or s.num_chunks > 1:
                raise ValueError("the FP8 layer takes neither biases nor K-chunks")
            u8 = torch.uint8
            P = L.moe_fp8_padded_rows(R, E)
            self.f8_P = P
            self.xs_q = torch.empty(R, d, dtype=u8, device=dev)
            self.xs_qt = torch.empty(d, P, dtype=u8, device=dev)
            self.act_q = torch.empty(R, f, dtype=u8, device=dev)
            self.act_qt = torch.empty(f, P, dtype=u8, device=dev)
            self.dy_q = torch.empty(R, d, dtype=u8, device=dev)
            self.dy_qt = torch.empty(d, P, dtype=u8, device=dev)
            self.dh_q = torch.empty(R, 2 * f, dtype=u8, device=dev)
            self.dh_qt = torch.empty(2 * f, P, dtype=u8, device=dev)
            self.wi_q = torch.empty(E, d, 2 * f, dtype=u8, device=dev)
            self.wi_qt = torch.empty(E, 2 * f, d, dtype=u8, device=dev)
            self.wo_q = torch.empty(E, f, d, dtype=u8, device=dev)
            self.wo_qt = torch.empty(E, d, f, dtype=u8, device=dev)
            # amax / 1 / scale per quantized tensor: x, act, dy, dh (one each), wi, wo (E each)
            self.f8_amax = torch.empty(4 + 2 * E, dtype=f32, device=dev)
            self.f8_sinv = torch.empty(4 + 2 * E, dtype=f32, device=dev)
        if s.aux_coeff:
            self.aux_counts = torch.empty(E, dtype=i32, device=dev)
            self.aux_probs = torch.empty(E, dtype=f32, device=dev)
            self.aux_loss = torch.empty(1, dtype=f32, device=dev)
            self.aux_ws = torch.empty(L.moe_aux_loss_workspace_bytes(T, E), dtype=torch.uint8,
                                      device=dev)


    def _alloc_mx(self, dev):
        """Codes and scale atoms of every block-scaled operand: each tensor's
        row-wise copy (forward / dgrad GEMMs) and column-wise copy (weight
        gradients; for the weights, the other contraction)."""
        s = self.s
        d, f, E, R = s.d, s.f, s.E, self.rows_cap
        u8 = torch.uint8
        P = L.moe_fp8_padded_rows(R, E)
        self.mx_P = P
        G, PL, SW, TL = L.MX_ROWS_GROUPED, L.MX_ROWS_PLAIN, L.MX_ROWS_SWIGLU, L.MX_ROWS_TILES

        def q(rows, cols, row_map, groups=E):
            return (torch.empty(rows, cols, dtype=u8, device=dev),
                    torch.empty(L.moe_mx_scale_bytes(rows, cols, row_map, groups), dtype=u8,
                                device=dev))
        # A operands (grouped activations, the weight gradients' A copies) and
        # B operands (weights; the weight gradients' B copies) in their tilings
        self.mx = dict(xs=q(R, d, G), act=q(R, f, G), dy=q(R, d, G), dh=q(R, 2 * f, G),
                       xs_t=q(d, P, PL), act_t=q(f, P, PL), dy_t=q(d, P, TL, 1),
                       dh_t=q(2 * f, P, TL, 1),
                       wi_t=q(2 * f, E * d, SW), wi=q(E * d, 2 * f, TL),
                       wo_t=q(d, E * f, TL, 1), wo=q(E * f, d, TL))
        # the experts' weight rows as groups
        self.mx_woff_d = torch.arange(0, E * d + 1, d, dtype=torch.int32, device=dev)
        self.mx_woff_f = torch.arange(0, E * f + 1, f, dtype=torch.int32, device=dev)


def _noop(_name):
    pass


def _mx_both(b, name, x, fmt, qt_map, stream, mark):
    """Row-wise and column-wise block-scaled codes of a permuted activation
    from one read: blocks along its rows' d_model / d_ff, and along each
    expert's rows (qt_map: PLAIN for a weight gradient's A operand, TILES for
    its B operand)."""
    q, sfq = b.mx[name]
    qt, sfqt = b.mx[name + "_t"]
    L.moe_mx_quantize_2x(x, fmt, b.group_offsets, q, sfq, L.MX_ROWS_GROUPED, qt, sfqt, qt_map,
                         qt_cols=b.mx_P, stream=stream)
    mark("mxquant_" + name)


def _forward_mx(b, wi, wo, stream, mark):
    s = b.s
    d, f, E = s.d, s.f, s.E
    e4 = L.FP8_E4M3
    _mx_both(b, "xs", b.xs, e4, L.MX_ROWS_PLAIN, stream, mark)
    # the weights along both contractions from one read each: wi as [E d, 2f]
    # (dgrad-up B, blocks along 2f) and wi^T [2f, E d] (up-projection B, blocks
    # along d, SwiGLU tile order); wo as [E f, d] and wo^T [d, E f]
    L.moe_mx_quantize_2x(wi.view(E * d, 2 * f), e4, b.mx_woff_d, *b.mx["wi"], L.MX_ROWS_TILES,
                         *b.mx["wi_t"], L.MX_ROWS_SWIGLU, qt_cols=E * d, stream=stream)
    L.moe_mx_quantize_2x(wo.view(E * f, d), e4, b.mx_woff_f, *b.mx["wo"], L.MX_ROWS_TILES,
                         *b.mx["wo_t"], L.MX_ROWS_TILES, qt_cols=E * f, stream=stream)
    mark("mxquant_weights")
    qx, sx = b.mx["xs"]
    qw, sw = b.mx["wi_t"]
    L.moe_gmm_mx(qx, sx, e4, qw, sw, 1, e4, b.group_offsets, b.h, L.EPI_SWIGLU_FWD, C2=b.act,
                 dev_status=b.dev_status, stream=stream, E=E, N=2 * f, K=d, ldb=E * d,
                 stride_b=d)
    mark("gmm_up_swiglu")
    _mx_both(b, "act", b.act, e4, L.MX_ROWS_PLAIN, stream, mark)
    qa, sa = b.mx["act"]
    qw, sw = b.mx["wo_t"]
    L.moe_gmm_mx(qa, sa, e4, qw, sw, 1, e4, b.group_offsets, b.y, dev_status=b.dev_status,
                 stream=stream, E=E, N=d, K=f, ldb=E * f, stride_b=f)
    mark("gmm_down")


def _backward_mx(b, stream, mark):
    s = b.s
    d, f, E = s.d, s.f, s.E
    e4, e5 = L.FP8_E4M3, L.FP8_E5M2
    _mx_both(b, "dy", b.dy, e5, L.MX_ROWS_TILES, stream, mark)
    qd, sd = b.mx["dy"]
    qw, sw = b.mx["wo"]
    L.moe_gmm_mx(qd, sd, e5, qw.view(E, f, d), sw, 0, e4, b.group_offsets, b.dh,
                 L.EPI_SWIGLU_BWD, aux=b.h, dev_status=b.dev_status, stream=stream)
    mark("gmm_dgrad_down_swiglu_bwd")
    L.moe_tgmm_mx(*b.mx["act_t"], e4, *b.mx["dy_t"], e5, b.group_offsets, b.rows_cap, b.dwo,
                  dev_status=b.dev_status, stream=stream)
    mark("tgmm_dwo")
    _mx_both(b, "dh", b.dh, e5, L.MX_ROWS_TILES, stream, mark)
    qh, sh = b.mx["dh"]
    qw, sw = b.mx["wi"]
    L.moe_gmm_mx(qh, sh, e5, qw.view(E, d, 2 * f), sw, 0, e4, b.group_offsets, b.dxs,
                 dev_status=b.dev_status, stream=stream)
    mark("gmm_dgrad_up")
    L.moe_tgmm_mx(*b.mx["xs_t"], e4, *b.mx["dh_t"], e5, b.group_offsets, b.rows_cap, b.dwi,
                  dev_status=b.dev_status, stream=stream)
    mark("tgmm_dwi")


def _fp8_slots(b):
    """(amax, 1/scale) views per quantized tensor."""
    E = b.s.E
    a, v = b.f8_amax, b.f8_sinv
    return dict(x=(a[0:1], v[0:1]), act=(a[1:2], v[1:2]), dy=(a[2:3], v[2:3]),
                dh=(a[3:4], v[3:4]), wi=(a[4:4 + E], v[4:4 + E]),
                wo=(a[4 + E:4 + 2 * E], v[4 + E:4 + 2 * E]))


def _quant_act(b, name, x, fmt, q, qt, stream, mark, amax_done=False):
    """amax_done: the GEMM that wrote x already left its amax in the slot."""
    amax, sinv = _fp8_slots(b)[name]
    if not amax_done:
        L.moe_fp8_amax(x, amax, group_offsets=b.group_offsets, E=b.s.E, stream=stream)
    L.moe_fp8_quantize_act(x, b.group_offsets, fmt, amax, q, qt, sinv, stream)
    mark("quant_" + name)


def _forward_fp8(b, x, logits, wi, wo, stream, mark):
    s = b.s
    E = s.E
    sl = _fp8_slots(b)
    _quant_act(b, "x", b.xs, L.FP8_E4M3, b.xs_q, b.xs_qt, stream, mark)
    for name, w, q, qt in (("wi", wi, b.wi_q, b.wi_qt), ("wo", wo, b.wo_q, b.wo_qt)):
        amax, sinv = sl[name]
        L.moe_fp8_amax(w.view(E * w.shape[1], w.shape[2]), amax, groups=E, stream=stream)
        L.moe_fp8_quantize_weights(w, L.FP8_E4M3, amax, q, qt, sinv, stream)
        mark("quant_" + name)
    L.moe_gmm_fp8(b.xs_q, L.FP8_E4M3, sl["x"][1], b.wi_qt, L.FP8_E4M3, sl["wi"][1],
                  b.group_offsets, b.h, L.EPI_SWIGLU_FWD, C2=b.act, dev_status=b.dev_status,
                  stream=stream, amax_out=sl["act"][0])
    mark("gmm_up_swiglu")
    _quant_act(b, "act", b.act, L.FP8_E4M3, b.act_q, b.act_qt, stream, mark, amax_done=True)
    L.moe_gmm_fp8(b.act_q, L.FP8_E4M3, sl["act"][1], b.wo_qt, L.FP8_E4M3, sl["wo"][1],
                  b.group_offsets, b.y, dev_status=b.dev_status, stream=stream)
    mark("gmm_down")


def _backward_fp8(b, stream, mark):
    s = b.s
    sl = _fp8_slots(b)
    _quant_act(b, "dy", b.dy, L.FP8_E5M2, b.dy_q, b.dy_qt, stream, mark)
    L.moe_gmm_fp8(b.dy_q, L.FP8_E5M2, sl["dy"][1], b.wo_q, L.FP8_E4M3, sl["wo"][1],
                  b.group_offsets, b.dh, L.EPI_SWIGLU_BWD, aux=b.h, dev_status=b.dev_status,
                  stream=stream, amax_out=sl["dh"][0])
    mark("gmm_dgrad_down_swiglu_bwd")
    L.moe_tgmm_fp8(b.act_qt, L.FP8_E4M3, sl["act"][1], b.dy_qt, L.FP8_E5M2, sl["dy"][1],
                   b.group_offsets, b.rows_cap, b.dwo, dev_status=b.dev_status, stream=stream)
    mark("tgmm_dwo")
    _quant_act(b, "dh", b.dh, L.FP8_E5M2, b.dh_q, b.dh_qt, stream, mark, amax_done=True)
    L.moe_gmm_fp8(b.dh_q, L.FP8_E5M2, sl["dh"][1], b.wi_q, L.FP8_E4M3, sl["wi"][1],
                  b.group_offsets, b.dxs, dev_status=b.dev_status, stream=stream)
    mark("gmm_dgrad_up")
    L.moe_tgmm_fp8(b.xs_qt, L.FP8_E4M3, sl["x"][1], b.dh_qt, L.FP8_E5M2, sl["dh"][1],
                   b.group_offsets, b.rows_cap, b.dwi, dev_status=b.dev_status, stream=stream)
    mark("tgmm_dwi")


def forward(b: MoEBuffers, x, logits, wi, wo, stream=None, mark=_noop, bi=None, bo=None,
            expert_bias=None):
    """x bf16 [T,d], logits fp32 [T,E], wi bf16 [E,d,2f] ([wi_0 | wi_1]), wo bf16 [E,f,d];
    with a bias layer shape also bi bf16 [E,2f] and bo bf16 [E,d]; expert_bias fp32 [E]
    or None: DeepSeek-V3's selection bias (MaxText PR #2579, "Onboard explicit sharding
    to deepseek": the weights keep the pre-bias logits).

    ``mark(name)`` is called after each library call (the benchmark records a
    CUDA event there)."""
    s = b.s
    if s.bias != (bi is not None and bo is not None):
        raise ValueError("forward: pass bi and bo exactly when the layer shape has bias=True")
    b.logits = logits
    L.moe_route_topk(logits, s.k, s.score_fn, s.renorm, b.topk_idx, b.topk_w, stream,
                     expert_bias=expert_bias, num_groups=s.num_groups,
                     topk_group=s.topk_group)
    mark("route")
    if s.aux_coeff:
        L.moe_aux_loss(logits, b.topk_idx, s.score_fn, s.aux_coeff, b.aux_counts, b.aux_probs,
                       b.aux_loss, b.aux_ws, stream)
        mark("aux_loss")
    L.moe_permute(x, b.topk_idx, s.E, s.align, s.capacity, b.xs, b.group_sizes, b.kept_counts,
                  b.group_offsets, b.s2f, b.f2s, b.ws, b.dev_status, stream)
    mark("permute")
    if s.mxfp8:
        _forward_mx(b, wi, wo, stream, mark)
        L.moe_combine(b.y, b.f2s, b.topk_w, b.out, s.k, stream)
        mark("combine")
        return b.out
    if s.fp8:
        _forward_fp8(b, x, logits, wi, wo, stream, mark)
        L.moe_combine(b.y, b.f2s, b.topk_w, b.out, s.k, stream)
        mark("combine")
        return b.out
    act_t = b.act_t if b.colwise else None
    if s.num_chunks <= 1:
        L.moe_gmm(b.xs, wi, 0, b.group_offsets, b.h, L.EPI_SWIGLU_FWD, C2=b.act,
                  dev_status=b.dev_status, stream=stream, bias=bi, Ct=act_t)
        mark("gmm_up_swiglu")
    else:
        dc = s.d // s.num_chunks
        for c in range(s.num_chunks):
            a_c = b.xs[:, c * dc:(c + 1) * dc]
            w_c = wi[:, c * dc:(c + 1) * dc, :]
            last = c == s.num_chunks - 1
            ps = None if c == 0 else b.p
            if last:
                L.moe_gmm(a_c, w_c, 0, b.group_offsets, b.h, L.EPI_SWIGLU_FWD, partial_sum=ps,
                          C2=b.act, dev_status=b.dev_status, stream=stream, bias=bi, Ct=act_t)
                mark("gmm_up_chunk_swiglu")
            else:
                L.moe_gmm(a_c, w_c, 0, b.group_offsets, b.p, L.EPI_NONE, partial_sum=ps,
                          dev_status=b.dev_status, stream=stream)
                mark("gmm_up_chunk")
    L.moe_gmm(b.act, wo, 0, b.group_offsets, b.y, L.EPI_NONE, dev_status=b.dev_status,
              stream=stream, bias=bo)
    mark("gmm_down")
    L.moe_combine(b.y, b.f2s, b.topk_w, b.out, s.k, stream)
    mark("combine")
    return b.out


def backward(b: MoEBuffers, dout, wi, wo, stream=None, mark=_noop):
    """dout bf16 [T,d] -> (dx, dwi, dwo, d_topk_w) in b's buffers; the router-logit
    gradient lands in b.d_logits, the bias gradients (bias layers) in b.dbi, b.dbo."""
    s = b.s
    L.moe_unpermute_bwd(dout, b.y, b.f2s, b.s2f, b.group_offsets, b.topk_w, b.dy, b.d_topk_w,
                        stream)
    mark("unpermute_bwd")
    L.moe_route_topk_bwd(b.logits, b.topk_idx, b.topk_w, b.d_topk_w, s.score_fn, s.renorm,
                         b.d_logits, stream)
    mark("route_bwd")
    if s.aux_coeff:
        L.moe_aux_loss_bwd(b.logits, b.aux_counts, s.k, s.score_fn, s.aux_coeff, b.d_logits,
                           d_loss=1.0, accumulate=True, stream=stream)
        mark("aux_loss_bwd")
    if s.mxfp8:
        _backward_mx(b, stream, mark)
        L.moe_combine(b.dxs, b.f2s, None, b.dx, s.k, stream)
        mark("dispatch_bwd")
        return b.dx, b.dwi, b.dwo, b.d_topk_w
    if s.fp8:
        _backward_fp8(b, stream, mark)
        L.moe_combine(b.dxs, b.f2s, None, b.dx, s.k, stream)
        mark("dispatch_bwd")
        return b.dx, b.dwi, b.dwo, b.d_topk_w
    # dAct = dY . wo^T, fused with the SwiGLU backward into dH = [dgate | dup]
    L.moe_gmm(b.dy, wo, 1, b.group_offsets, b.dh, L.EPI_SWIGLU_BWD, aux=b.h,
              dev_status=b.dev_status, stream=stream, Ct=b.dh_t if b.colwise else None)
    mark("gmm_dgrad_down_swiglu_bwd")
    if b.colwise:
        L.moe_transpose_act(b.dy, b.group_offsets, b.dy_t, stream)
        mark("transpose_dy")
        L.moe_tgmm_kt(b.act_t, b.dy_t, b.group_offsets, b.rows_cap, b.dwo,
                      dev_status=b.dev_status, stream=stream, b_colwise=True)
    else:
        L.moe_tgmm(b.act, b.dy, b.group_offsets, b.dwo, dev_status=b.dev_status, stream=stream)
    mark("tgmm_dwo")
    if s.bias:
        L.moe_group_colsum(b.dy, b.group_offsets, b.dbo, stream)
        mark("colsum_dbo")
        L.moe_group_colsum(b.dh, b.group_offsets, b.dbi, stream)
        mark("colsum_dbi")
    if b.colwise:
        L.moe_transpose_act(b.xs, b.group_offsets, b.xs_t, stream)
        mark("transpose_xs")

    def tgmm_dwi(sl, name):
        if b.colwise:
            L.moe_tgmm_kt(b.xs_t[sl], b.dh_t, b.group_offsets, b.rows_cap, b.dwi[:, sl, :],
                          dev_status=b.dev_status, stream=stream, b_colwise=True)
        else:
            L.moe_tgmm(b.xs[:, sl], b.dh, b.group_offsets, b.dwi[:, sl, :],
                       dev_status=b.dev_status, stream=stream)
        mark(name)

    if s.num_chunks <= 1:
        L.moe_gmm(b.dh, wi, 1, b.group_offsets, b.dxs, L.EPI_NONE, dev_status=b.dev_status,
                  stream=stream)
        mark("gmm_dgrad_up")
        tgmm_dwi(slice(0, s.d), "tgmm_dwi")
    else:
        dc = s.d // s.num_chunks
        for c in range(s.num_chunks):
            sl = slice(c * dc, (c + 1) * dc)
            L.moe_gmm(b.dh, wi[:, sl, :], 1, b.group_offsets, b.dxs[:, sl], L.EPI_NONE,
                      dev_status=b.dev_status, stream=stream)
            mark("gmm_dgrad_up_chunk")
            tgmm_dwi(sl, "tgmm_dwi_chunk")
    L.moe_combine(b.dxs, b.f2s, None, b.dx, s.k, stream)
    mark("dispatch_bwd")
    return b.dx, b.dwi, b.dwo, b.d_topk_w


def kernels_per_step(s: LayerShape) -> int:
    """Kernels one forward + backward launches (route 1, permute 3, each GEMM 1,
    combine 1, unpermute_bwd 1, route_bwd 1, dispatch backward 1, bias gradients 2,
    auxiliary loss 2 + 1, column-wise copies of dY and Xs 2)."""
    up = max(1, s.num_chunks)
    aux = bool(s.aux_coeff)
    fwd = 1 + 3 + up + 1 + 1 + (2 if aux and s.T > 0 else 1 if aux else 0)
    bwd = 1 + 1 + 1 + 1 + 2 * up + 1 + (2 if s.bias else 0) + (1 if aux and s.T > 0 else 0)
    if s.fp8:   # amax + quantize for x, wi, wo; quantize for act (amax in the GEMM);
        fwd += 7   # amax + quantize for dy; quantize for dh
        bwd += 3
    elif s.mxfp8:  # both copies of xs, act and of the two weights; of dy and dh
        fwd += 4
        bwd += 2
    elif s.wgrad_colwise:
        bwd += 2
    return fwd + bwd


def gemm_flops(m_kept: int, d: int, f: int) -> int:
    """Algorithmic FLOPs of the expert GEMMs, forward + backward (18 M d f)."""
    return 18 * m_kept * d * f
