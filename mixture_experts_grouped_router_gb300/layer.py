"""The MoE expert layer, forward and backward, through the library's layer calls.

This module only describes the layer (LayerShape -> moe_layer_config),
allocates its device workspace through PyTorch and exposes the buffers the
library plans inside it as tensors; moe_layer_forward / moe_layer_backward
(csrc/layer.cu) issue the sequence of library calls on the current stream,
and every arithmetic step runs in libmoe_gb300.so's kernels.  The sequence
follows the single-VJP MoE block of TransformerEngine PR #2912 ("[JAX] Add
an MoE Block (Layer) that compound router, permutation, groupedGEMM and
communication", sequence diagram), without the expert-parallel all-to-all:

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
    """The device workspace of one layer instance, allocated once and reused
    every step; its buffers (planned by the library) as tensor attributes."""

    def __init__(self, s: LayerShape, device="cuda", dw_dtype=torch.bfloat16):
        self.s = s
        T, d, f, E, k = s.T, s.d, s.f, s.E, s.k
        cfg = L.LayerConfig(
            T=T, d=d, f=f, E=E, k=k, score_fn=s.score_fn, renorm=int(s.renorm),
            num_groups=s.num_groups, topk_group=s.topk_group, align=s.align,
            capacity=s.capacity, num_chunks=s.num_chunks, aux_coeff=float(s.aux_coeff),
            bias=int(bool(s.bias)),
            precision=L.PREC_MXFP8 if s.mxfp8 else L.PREC_FP8 if s.fp8 else L.PREC_BF16,
            wgrad_colwise=int(bool(s.wgrad_colwise)),
            dw_dtype=L.DTYPE_F32 if dw_dtype == torch.float32 else L.DTYPE_BF16)
        if s.mxfp8 and s.fp8:
            raise ValueError("fp8 and mxfp8 are exclusive")
        nbytes = L.moe_layer_workspace_bytes(cfg)
        if nbytes == 0:
            raise ValueError(L.last_error())
        self.cfg = cfg
        self.rows_cap = L.moe_rows_cap(T, E, k, s.align, s.capacity)
        R = self.rows_cap
        P = L.moe_fp8_padded_rows(R, E)
        self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=device)
        bf, i32, f32, u8 = torch.bfloat16, torch.int32, torch.float32, torch.uint8

        def view(name, dtype=None, shape=None):
            """The buffer as a tensor; None when the configuration does not use it
            (an empty tensor when it does but holds nothing, e.g. T = 0)."""
            off, nb = L.moe_layer_buffer(cfg, name)
            if nb == 0:
                if shape is not None and 0 in shape:
                    return torch.empty(shape, dtype=dtype, device=device)
                return None
            t = self.workspace[off:off + nb]
            if dtype is None:
                return t
            return t.view(dtype).view(shape)

        shapes = dict(
            topk_idx=(i32, (T, k)), topk_w=(f32, (T, k)), xs=(bf, (R, d)),
            group_sizes=(i32, (E,)), kept_counts=(i32, (E,)), group_offsets=(i32, (E + 1,)),
            s2f=(i32, (R,)), f2s=(i32, (T * k,)), h=(bf, (R, 2 * f)), act=(bf, (R, f)),
            y=(bf, (R, d)), out=(bf, (T, d)), p=(f32, (R, 2 * f)), dy=(bf, (R, d)),
            d_topk_w=(f32, (T, k)), d_logits=(f32, (T, E)), dh=(bf, (R, 2 * f)),
            dxs=(bf, (R, d)), dx=(bf, (T, d)), dwi=(dw_dtype, (E, d, 2 * f)),
            dwo=(dw_dtype, (E, f, d)), dbi=(f32, (E, 2 * f)), dbo=(f32, (E, d)),
            dev_status=(i32, (1,)), xs_t=(bf, (d, P)), act_t=(bf, (f, P)), dy_t=(bf, (d, P)),
            dh_t=(bf, (2 * f, P)), xs_q=(u8, (R, d)), xs_qt=(u8, (d, P)), act_q=(u8, (R, f)),
            act_qt=(u8, (f, P)), dy_q=(u8, (R, d)), dy_qt=(u8, (d, P)), dh_q=(u8, (R, 2 * f)),
            dh_qt=(u8, (2 * f, P)), wi_q=(u8, (E, d, 2 * f)), wi_qt=(u8, (E, 2 * f, d)),
            wo_q=(u8, (E, f, d)), wo_qt=(u8, (E, d, f)), f8_amax=(f32, (4 + 2 * E,)),
            f8_sinv=(f32, (4 + 2 * E,)), aux_counts=(i32, (E,)), aux_probs=(f32, (E,)),
            aux_loss=(f32, (1,)), mx_woff_d=(i32, (E + 1,)), mx_woff_f=(i32, (E + 1,)))
        # attribute name -> library buffer name where they differ
        alias = dict(p="partial", xs_q="f8_xs_q", xs_qt="f8_xs_qt", act_q="f8_act_q",
                     act_qt="f8_act_qt", dy_q="f8_dy_q", dy_qt="f8_dy_qt", dh_q="f8_dh_q",
                     dh_qt="f8_dh_qt", wi_q="f8_wi_q", wi_qt="f8_wi_qt", wo_q="f8_wo_q",
                     wo_qt="f8_wo_qt")
        for name, (dt, shape) in shapes.items():
            setattr(self, name, view(alias.get(name, name), dt, shape))
        self.ws = view("permute_ws")
        self.aux_ws = view("aux_ws")
        self.colwise = bool(s.wgrad_colwise) and not s.fp8 and not s.mxfp8
        self.f8_P = self.mx_P = P
        if s.mxfp8:
            # codes and scale atoms of every block-scaled operand
            mx_shapes = dict(xs=(R, d), act=(R, f), dy=(R, d), dh=(R, 2 * f), xs_t=(d, P),
                             act_t=(f, P), dy_t=(d, P), dh_t=(2 * f, P), wi_t=(2 * f, E * d),
                             wi=(E * d, 2 * f), wo_t=(d, E * f), wo=(E * f, d))
            self.mx = {n: (view("mx_%s_q" % n, u8, shape), view("mx_%s_sf" % n))
                       for n, shape in mx_shapes.items()}
        self.logits = None
        L.moe_layer_init(cfg, self.workspace)


def _noop(_name):
    pass


def forward(b: MoEBuffers, x, logits, wi, wo, stream=None, mark=_noop, bi=None, bo=None,
            expert_bias=None):
    """x bf16 [T,d], logits fp32 [T,E], wi bf16 [E,d,2f] ([wi_0 | wi_1]), wo bf16 [E,f,d];
    with a bias layer shape also bi bf16 [E,2f] and bo bf16 [E,d]; expert_bias fp32 [E]
    or None: DeepSeek-V3's selection bias (MaxText PR #2579, "Onboard explicit sharding
    to deepseek": the weights keep the pre-bias logits).

    ``mark(name)`` is called after each library call (the benchmark records a
    CUDA event there)."""
    if b.s.bias != (bi is not None and bo is not None):
        raise ValueError("forward: pass bi and bo exactly when the layer shape has bias=True")
    b.logits = logits
    L.moe_layer_forward(b.cfg, b.workspace, x, logits, wi, wo, bi, bo, expert_bias,
                        None if mark is _noop else mark, stream)
    return b.out


def backward(b: MoEBuffers, dout, wi, wo, stream=None, mark=_noop):
    """dout bf16 [T,d] -> (dx, dwi, dwo, d_topk_w) in b's buffers; the router-logit
    gradient lands in b.d_logits, the bias gradients (bias layers) in b.dbi, b.dbo."""
    L.moe_layer_backward(b.cfg, b.workspace, dout, b.logits, wi, wo,
                         None if mark is _noop else mark, stream)
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
