"""ctypes binding of libmoe_gb300.so: one Python function per C entry point,
same names, argument marshalling only (tensor -> pointer, shape -> sizes,
current torch stream -> cudaStream_t).  Every step of the layer runs in the
library's CUDA kernels; there is no fallback: if the library is missing the
import fails.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

_HERE = os.path.dirname(os.path.abspath(__file__))

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_CUDA = 3
MOE_ERR_TIMEOUT = 4
MOE_ERR_DEVICE = 5
SCORE_SOFTMAX = 0
SCORE_SIGMOID = 1
DTYPE_BF16 = 0
DTYPE_F32 = 1
EPI_NONE = 0
EPI_SWIGLU_FWD = 1
EPI_SWIGLU_BWD = 2


class MoEError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__("%s (status %d: %s)" % (msg, status, status_string(status)))
        self.status = status


def _load() -> ctypes.CDLL:
    path = _build.LIB_PATH
    if not os.path.exists(path):
        raise ImportError("libmoe_gb300.so is not built (%s); run "
                          "`python -m mixture_experts_grouped_router_gb300.build`" % path)
    return ctypes.CDLL(path)


LIB = _load()

_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t

_SIGS = {
    "moe_status_string": (ctypes.c_char_p, [_I]),
    "moe_last_error": (ctypes.c_char_p, []),
    "moe_version": (_I, []),
    "moe_set_wait_limit_ns": (_I, [ctypes.c_uint64]),
    "moe_wait_limit_ns": (ctypes.c_uint64, []),
    "moe_test_stall_loads": (None, [_I]),
    "moe_rows_cap": (_I64, [_I, _I, _I, _I, _I]),
    "moe_permute_workspace_bytes": (_SZ, [_I, _I]),
    "moe_route_topk": (_I, [_P, _I64, _I, _I, _I, _I, _I, _P, _I, _I, _P, _P, _P]),
    "moe_aux_loss_workspace_bytes": (_SZ, [_I, _I]),
    "moe_aux_loss": (_I, [_P, _I64, _I, _I, _I, _I, _P, ctypes.c_float, _P, _P, _P, _P, _SZ,
                          _P]),
    "moe_aux_loss_bwd": (_I, [_P, _I64, _I, _I, _I, _I, _P, ctypes.c_float, ctypes.c_float, _P,
                              _I64, _I, _P]),
    "moe_route_topk_bwd": (_I, [_P, _I64, _P, _P, _P, _I, _I, _I, _I, _I, _P, _I64, _P]),
    "moe_permute": (_I, [_P, _I64, _P, _I, _I, _I, _I, _I, _I, _P, _I64, _I64, _P, _P, _P, _P,
                         _P, _P, _SZ, _P, _P]),
    "moe_permute_noalloc": (_I, [_P, _I64, _P, _I, _I, _I, _I, _I, _I, _P, _I64, _I64, _P, _P,
                                 _P, _P, _P, _P, _P]),
    "moe_gmm": (_I, [_P, _I64, _P, _I64, _I64, _I, _P, _I, _I64, _I, _I, _I, _P, _I64, _P, _I64,
                     _P, _I64, _P, _I, _I64, _P, _I64, _P, _I64, _P, _P]),
    "moe_group_colsum": (_I, [_P, _I64, _P, _I, _I64, _I, _P, _I64, _P]),
    "moe_tgmm": (_I, [_P, _I64, _P, _I64, _P, _I, _I64, _I, _I, _P, _I, _I64, _I64, _I, _P, _P]),
    "moe_combine": (_I, [_P, _I64, _P, _P, _I, _I, _I, _P, _I64, _P]),
    "moe_fp8_amax": (_I, [_P, _I64, _I64, _I, _I, _P, _I, _P, _P]),
    "moe_fp8_padded_rows": (_I64, [_I64, _I]),
    "moe_fp8_quantize_act": (_I, [_P, _I64, _P, _I, _I64, _I, _I, _P, _P, _I64, _P, _I64, _P,
                                  _P]),
    "moe_fp8_quantize_weights": (_I, [_P, _I, _I, _I, _I, _P, _P, _P, _P, _P]),
    "moe_transpose_act": (_I, [_P, _I64, _P, _I, _I64, _I, _P, _I64, _P]),
    "moe_tgmm_kt": (_I, [_P, _I64, _P, _I64, _I, _P, _I, _I64, _I, _I, _P, _I, _I64, _I64, _I,
                         _P, _P]),
    "moe_gmm_fp8": (_I, [_P, _I64, _I, _P, _P, _I64, _I64, _I, _P, _P, _I, _I64, _I, _I, _I, _P,
                         _I64, _P, _I, _I64, _P, _I64, _P, _P, _P]),
    "moe_tgmm_fp8": (_I, [_P, _I64, _I, _P, _P, _I64, _I, _P, _P, _I, _I64, _I, _I, _P, _I, _I64,
                          _I64, _I, _P, _P]),
    "moe_unpermute_bwd": (_I, [_P, _I64, _P, _I64, _P, _P, _P, _P, _I, _I, _I, _I, _I64, _P,
                               _I64, _P, _P]),
    "moe_mx_scale_bytes": (_SZ, [_I64, _I, _I, _I]),
    "moe_mx_quantize": (_I, [_P, _I64, _I64, _I, _I, _I, _P, _I, _P, _I64, _P, _SZ, _P]),
    "moe_mx_quantize_2x": (_I, [_P, _I64, _I64, _I, _I, _P, _I, _P, _I64, _I, _P, _SZ, _P, _I64,
                                _I, _I, _P, _SZ, _P]),
    "moe_gmm_mx": (_I, [_P, _I64, _P, _I, _P, _I64, _I64, _P, _I, _I, _P, _I, _I64, _I,
                        _I, _I, _P, _I64, _P, _I, _I64, _P, _I64, _P, _P]),
    "moe_tgmm_mx": (_I, [_P, _I64, _P, _I, _P, _I64, _P, _I, _P, _I, _I64, _I, _I, _P, _I, _I64,
                         _I64, _I, _P, _P]),
    "moe_ep_recv_rows_cap": (_I64, [_I, _I, _I, _I, _I]),
    "moe_ep_a2a_params": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P]),
    "moe_ep_local_layout": (_I, [_P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P]),
    "moe_sort_chunks": (_I, [_P, _I64, _P, _I64, _I, _P, _P, _P, _I, _I64, _P]),
    "moe_layer_workspace_bytes": (_SZ, [_P]),
    "moe_layer_buffer": (_I, [_P, _I, _P, _P]),
    "moe_layer_init": (_I, [_P, _P, _SZ, _P]),
    "moe_layer_forward": (_I, [_P, _P, _SZ, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_layer_backward": (_I, [_P, _P, _SZ, _P, _P, _P, _P, _P, _P, _P]),
    "moe_layer_pipeline_workspace_bytes": (_SZ, [_P]),
    "moe_layer_pipeline_create": (_I, [_P, _P, _SZ, _P, _SZ, _P]),
    "moe_layer_pipeline_step": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
    "moe_layer_pipeline_join": (_I, [_P, _P]),
    "moe_layer_pipeline_sync": (_I, [_P]),
    "moe_layer_pipeline_destroy": (None, [_P]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(LIB, _name)
    _fn.restype = _res
    _fn.argtypes = _args

EXPORTED = tuple(_SIGS)


def status_string(status: int) -> str:
    return LIB.moe_status_string(status).decode()


def last_error() -> str:
    return LIB.moe_last_error().decode()


def _check(status: int):
    if status != MOE_OK:
        raise MoEError(status, last_error())


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ld(t):
    assert t.dim() >= 2, "matrices only"
    if t.numel() == 0:
        return t.shape[-1]
    assert t.stride(-1) == 1, "row-major tensors only"
    return t.stride(-2)


def moe_set_wait_limit_ns(limit_ns: int):
    _check(LIB.moe_set_wait_limit_ns(int(limit_ns)))


def moe_wait_limit_ns() -> int:
    return int(LIB.moe_wait_limit_ns())


def moe_test_stall_loads(enable: bool):
    LIB.moe_test_stall_loads(int(bool(enable)))


def moe_rows_cap(T: int, E: int, k: int, align: int, capacity: int = 0) -> int:
    return int(LIB.moe_rows_cap(T, E, k, align, capacity))


def moe_permute_workspace_bytes(T: int, E: int) -> int:
    return int(LIB.moe_permute_workspace_bytes(T, E))


def moe_route_topk(logits, k, score_fn, renorm, topk_idx, topk_w, stream=None,
                   expert_bias=None, num_groups=0, topk_group=0):
    T, E = logits.shape
    _check(LIB.moe_route_topk(_ptr(logits), _ld(logits), T, E, k, score_fn, int(renorm),
                              _ptr(expert_bias), int(num_groups), int(topk_group),
                              _ptr(topk_idx), _ptr(topk_w), _stream(stream)))


def moe_aux_loss_workspace_bytes(T: int, E: int) -> int:
    return int(LIB.moe_aux_loss_workspace_bytes(T, E))


def moe_aux_loss(logits, topk_idx, score_fn, coeff, counts, probs_mean, loss, workspace,
                 stream=None):
    """counts int32 [E], probs_mean fp32 [E], loss fp32 [1] (device outputs)."""
    T, E = logits.shape
    k = topk_idx.shape[1]
    _check(LIB.moe_aux_loss(_ptr(logits), _ld(logits), T, E, k, score_fn, _ptr(topk_idx),
                            float(coeff), _ptr(counts), _ptr(probs_mean), _ptr(loss),
                            _ptr(workspace), workspace.numel() * workspace.element_size(),
                            _stream(stream)))


def moe_aux_loss_bwd(logits, counts, k, score_fn, coeff, d_logits, d_loss=1.0, accumulate=True,
                     stream=None):
    T, E = logits.shape
    _check(LIB.moe_aux_loss_bwd(_ptr(logits), _ld(logits), T, E, k, score_fn, _ptr(counts),
                                float(coeff), float(d_loss), _ptr(d_logits), _ld(d_logits),
                                int(accumulate), _stream(stream)))


def moe_route_topk_bwd(logits, topk_idx, topk_w, d_topk_w, score_fn, renorm, d_logits,
                       stream=None):
    T, E = logits.shape
    k = topk_idx.shape[1]
    _check(LIB.moe_route_topk_bwd(_ptr(logits), _ld(logits), _ptr(topk_idx), _ptr(topk_w),
                                  _ptr(d_topk_w), T, E, k, score_fn, int(renorm), _ptr(d_logits),
                                  _ld(d_logits), _stream(stream)))


def moe_permute(x, topk_idx, E, align, capacity, x_sorted, group_sizes, kept_counts,
                group_offsets, sorted_to_flat, flat_to_sorted, workspace, dev_status=None,
                stream=None):
    T, d = x.shape
    k = topk_idx.shape[1]
    _check(LIB.moe_permute(_ptr(x), _ld(x), _ptr(topk_idx), T, d, E, k, align, capacity,
                           _ptr(x_sorted), _ld(x_sorted), x_sorted.shape[0], _ptr(group_sizes),
                           _ptr(kept_counts), _ptr(group_offsets), _ptr(sorted_to_flat),
                           _ptr(flat_to_sorted), _ptr(workspace),
                           workspace.numel() * workspace.element_size(), _ptr(dev_status),
                           _stream(stream)))


def moe_permute_noalloc(x, topk_idx, E, align, capacity, x_sorted, group_sizes, kept_counts,
                        group_offsets, sorted_to_flat, flat_to_sorted, dev_status=None,
                        stream=None):
    """moe_permute with the library's built-in scratch array instead of a workspace."""
    T, d = x.shape
    k = topk_idx.shape[1]
    _check(LIB.moe_permute_noalloc(_ptr(x), _ld(x), _ptr(topk_idx), T, d, E, k, align, capacity,
                                   _ptr(x_sorted), _ld(x_sorted), x_sorted.shape[0],
                                   _ptr(group_sizes), _ptr(kept_counts), _ptr(group_offsets),
                                   _ptr(sorted_to_flat), _ptr(flat_to_sorted), _ptr(dev_status),
                                   _stream(stream)))


def moe_gmm(A, B, trans_b, group_offsets, C, epilogue=EPI_NONE, aux=None, partial_sum=None,
            C2=None, dev_status=None, stream=None, K=None, N=None, bias=None, Ct=None):
    """A [rows_cap, >=K]; B [E, K, N] (trans_b=0) or [E, N, K] (trans_b=1), any
    row-major views; C bf16 or fp32; bias bf16 [E, >=N] (row e added to expert
    e's rows); Ct bf16 [F or 2F, >= moe_fp8_padded_rows(rows_cap, E)]: the
    column-wise copy of Act / dH the SwiGLU epilogues also write.  K and N
    default to the shapes of B."""
    E = B.shape[0]
    if K is None:
        K = B.shape[2] if trans_b else B.shape[1]
    if N is None:
        N = B.shape[1] if trans_b else B.shape[2]
    c_dtype = DTYPE_F32 if C.dtype == torch.float32 else DTYPE_BF16
    _check(LIB.moe_gmm(_ptr(A), _ld(A), _ptr(B), B.stride(1), B.stride(0), int(trans_b),
                       _ptr(group_offsets), E, A.shape[0], K, N, epilogue, _ptr(aux),
                       _ld(aux) if aux is not None else 0, _ptr(partial_sum),
                       _ld(partial_sum) if partial_sum is not None else 0, _ptr(bias),
                       bias.stride(0) if bias is not None else 0, _ptr(C), c_dtype,
                       _ld(C), _ptr(C2), _ld(C2) if C2 is not None else 0, _ptr(Ct),
                       _ld(Ct) if Ct is not None else 0, _ptr(dev_status), _stream(stream)))


def moe_group_colsum(G, group_offsets, out, stream=None):
    """out fp32 [E, >=N] = per-expert column sums of G bf16 [rows_cap, N]."""
    E = out.shape[0]
    N = G.shape[1]
    _check(LIB.moe_group_colsum(_ptr(G), _ld(G), _ptr(group_offsets), E, G.shape[0], N,
                                _ptr(out), out.stride(0), _stream(stream)))


def moe_tgmm(A, B, group_offsets, W, accumulate=False, dev_status=None, stream=None):
    """W [E, M, N] (bf16 or fp32, any row-major view); A [rows_cap, >=M]; B [rows_cap, >=N]."""
    E, M, N = W.shape
    w_dtype = DTYPE_F32 if W.dtype == torch.float32 else DTYPE_BF16
    _check(LIB.moe_tgmm(_ptr(A), _ld(A), _ptr(B), _ld(B), _ptr(group_offsets), E, A.shape[0], M,
                        N, _ptr(W), w_dtype, W.stride(1), W.stride(0), int(accumulate),
                        _ptr(dev_status), _stream(stream)))


FP8_E4M3 = 0
FP8_E5M2 = 1


def moe_fp8_amax(x, amax, groups=1, group_offsets=None, E=0, stream=None):
    """x bf16 2-D [rows, cols] (a [E, K, N] weight as x.view(E * K, N) with groups=E)."""
    _check(LIB.moe_fp8_amax(_ptr(x), _ld(x), x.shape[0], x.shape[1], groups, _ptr(group_offsets),
                            E, _ptr(amax), _stream(stream)))


def moe_fp8_padded_rows(rows_cap: int, E: int) -> int:
    return int(LIB.moe_fp8_padded_rows(rows_cap, E))


def moe_fp8_quantize_act(x, group_offsets, fmt, amax, q, qt, scale_inv, stream=None):
    """x bf16 [rows_cap, cols]; q uint8 [rows_cap, >=cols]; qt uint8 [cols, >=padded rows]."""
    E = group_offsets.shape[0] - 1
    _check(LIB.moe_fp8_quantize_act(_ptr(x), _ld(x), _ptr(group_offsets), E, x.shape[0],
                                    x.shape[1], fmt, _ptr(amax), _ptr(q), _ld(q), _ptr(qt),
                                    _ld(qt), _ptr(scale_inv), _stream(stream)))


def moe_fp8_quantize_weights(w, fmt, amax, q, qt, scale_inv, stream=None):
    """w bf16 [E, K, N] contiguous -> q uint8 [E, K, N], qt uint8 [E, N, K]."""
    E, K, N = w.shape
    _check(LIB.moe_fp8_quantize_weights(_ptr(w), E, K, N, fmt, _ptr(amax), _ptr(q), _ptr(qt),
                                        _ptr(scale_inv), _stream(stream)))


def moe_transpose_act(x, group_offsets, xt, stream=None):
    """x bf16 [rows_cap, cols] -> xt bf16 [cols, >= padded rows] (padded group layout)."""
    E = group_offsets.shape[0] - 1
    _check(LIB.moe_transpose_act(_ptr(x), _ld(x), _ptr(group_offsets), E, x.shape[0], x.shape[1],
                                 _ptr(xt), _ld(xt), _stream(stream)))


def moe_tgmm_kt(At, B, group_offsets, rows_cap, W, accumulate=False, dev_status=None,
                stream=None, b_colwise=False):
    """W [E, M, N] = per-expert A^T B with A given as its column-wise copy At [M, >=P];
    B row-wise [rows_cap, N], or (b_colwise) its column-wise copy [N, >=P]."""
    E, M, N = W.shape
    w_dtype = DTYPE_F32 if W.dtype == torch.float32 else DTYPE_BF16
    _check(LIB.moe_tgmm_kt(_ptr(At), _ld(At), _ptr(B), _ld(B), int(b_colwise),
                           _ptr(group_offsets), E, rows_cap,
                           M, N, _ptr(W), w_dtype, W.stride(1), W.stride(0), int(accumulate),
                           _ptr(dev_status), _stream(stream)))


def moe_gmm_fp8(A, a_fmt, a_scale_inv, B, b_fmt, b_scale_inv, group_offsets, C,
                epilogue=EPI_NONE, aux=None, C2=None, dev_status=None, stream=None,
                amax_out=None):
    """A uint8 codes [rows_cap, K]; B uint8 codes [E, N, K] (K-major); C bf16 or fp32."""
    E, N, K = B.shape
    c_dtype = DTYPE_F32 if C.dtype == torch.float32 else DTYPE_BF16
    _check(LIB.moe_gmm_fp8(_ptr(A), _ld(A), a_fmt, _ptr(a_scale_inv), _ptr(B), B.stride(1),
                           B.stride(0), b_fmt, _ptr(b_scale_inv), _ptr(group_offsets), E,
                           A.shape[0], K, N, epilogue, _ptr(aux),
                           _ld(aux) if aux is not None else 0, _ptr(C), c_dtype, _ld(C),
                           _ptr(C2), _ld(C2) if C2 is not None else 0, _ptr(amax_out),
                           _ptr(dev_status), _stream(stream)))


def moe_tgmm_fp8(At, a_fmt, a_scale_inv, Bt, b_fmt, b_scale_inv, group_offsets, rows_cap, W,
                 accumulate=False, dev_status=None, stream=None):
    """At uint8 [M, >=padded rows], Bt uint8 [N, >=padded rows]; W [E, M, N] bf16 / fp32."""
    E, M, N = W.shape
    w_dtype = DTYPE_F32 if W.dtype == torch.float32 else DTYPE_BF16
    _check(LIB.moe_tgmm_fp8(_ptr(At), _ld(At), a_fmt, _ptr(a_scale_inv), _ptr(Bt), _ld(Bt), b_fmt,
                            _ptr(b_scale_inv), _ptr(group_offsets), E, rows_cap, M, N, _ptr(W),
                            w_dtype, W.stride(1), W.stride(0), int(accumulate), _ptr(dev_status),
                            _stream(stream)))


def moe_combine(Y, flat_to_sorted, topk_w, out, k, stream=None):
    T, d = out.shape
    _check(LIB.moe_combine(_ptr(Y), _ld(Y), _ptr(flat_to_sorted), _ptr(topk_w), T, k, d,
                           _ptr(out), _ld(out), _stream(stream)))


def moe_unpermute_bwd(d_out, Y, flat_to_sorted, sorted_to_flat, group_offsets, topk_w, dY,
                      d_topk_w, stream=None):
    T, d = d_out.shape
    k = topk_w.shape[1]
    E = group_offsets.shape[0] - 1
    _check(LIB.moe_unpermute_bwd(_ptr(d_out), _ld(d_out), _ptr(Y), _ld(Y), _ptr(flat_to_sorted),
                                 _ptr(sorted_to_flat), _ptr(group_offsets), _ptr(topk_w), T, k, d,
                                 E, dY.shape[0], _ptr(dY), _ld(dY), _ptr(d_topk_w),
                                 _stream(stream)))


# ------------------------------------------------------------ block-scaled FP8
MX_ROWS_PLAIN = 0
MX_ROWS_GROUPED = 1
MX_ROWS_SWIGLU = 2
MX_ROWS_TILES = 3


def moe_mx_scale_bytes(rows: int, cols: int, row_map: int, E: int = 1) -> int:
    return int(LIB.moe_mx_scale_bytes(rows, cols, row_map, E))


def moe_mx_quantize(x, fmt, q, sf, row_map=MX_ROWS_PLAIN, group_offsets=None, stream=None,
                    groups=1):
    """x bf16 [rows, cols] -> q uint8 [rows, cols] codes, sf uint8 scale atoms;
    GROUPED takes group_offsets, TILES the number of equal row groups."""
    rows, cols = x.shape
    E = groups if group_offsets is None else group_offsets.shape[0] - 1
    _check(LIB.moe_mx_quantize(_ptr(x), _ld(x), rows, cols, fmt, row_map, _ptr(group_offsets), E,
                               _ptr(q), _ld(q), _ptr(sf), sf.numel() * sf.element_size(),
                               _stream(stream)))


def moe_mx_quantize_2x(x, fmt, group_offsets, q=None, sfq=None, q_map=MX_ROWS_GROUPED,
                       qt=None, sfqt=None, qt_map=MX_ROWS_PLAIN, qt_cols=None, stream=None):
    """Row-wise codes q [rows, cols] and column-wise codes qt [cols, qt_cols] (padded
    group layout) of x bf16 [rows, cols] from one read; either may be None."""
    rows, cols = x.shape
    E = group_offsets.shape[0] - 1
    if qt_cols is None and qt is not None:
        qt_cols = qt.shape[1]
    _check(LIB.moe_mx_quantize_2x(_ptr(x), _ld(x), rows, cols, fmt, _ptr(group_offsets), E,
                                  _ptr(q), _ld(q) if q is not None else 16, q_map, _ptr(sfq),
                                  sfq.numel() if sfq is not None else 0, _ptr(qt),
                                  _ld(qt) if qt is not None else 128,
                                  int(qt_cols or 128), qt_map, _ptr(sfqt),
                                  sfqt.numel() if sfqt is not None else 0, _stream(stream)))


def moe_gmm_mx(A, sfa, a_fmt, B, sfb, sfb_by_cols, b_fmt, group_offsets, C,
               epilogue=EPI_NONE, aux=None, C2=None, dev_status=None, stream=None, E=None, N=None,
               K=None, ldb=None, stride_b=None):
    """A uint8 codes [rows_cap, K]; B uint8 codes, K-major [E, N, K] (sfb_by_cols 0; or
    the [N, E*K] matrix given by ldb / stride_b = K with E, N, K: sfb_by_cols 1);
    C bf16 or fp32."""
    if E is None:
        E, N, K = B.shape
        ldb, stride_b = B.stride(1), B.stride(0)
    c_dtype = DTYPE_F32 if C.dtype == torch.float32 else DTYPE_BF16
    _check(LIB.moe_gmm_mx(_ptr(A), _ld(A), _ptr(sfa), a_fmt, _ptr(B), ldb, stride_b, _ptr(sfb),
                          int(sfb_by_cols), b_fmt, _ptr(group_offsets), E, A.shape[0], K,
                          N, epilogue, _ptr(aux), _ld(aux) if aux is not None else 0, _ptr(C),
                          c_dtype, _ld(C), _ptr(C2), _ld(C2) if C2 is not None else 0,
                          _ptr(dev_status), _stream(stream)))


def moe_tgmm_mx(At, sfa, a_fmt, Bt, sfb, b_fmt, group_offsets, rows_cap, W, accumulate=False,
                dev_status=None, stream=None):
    """W [E, M, N] = per-expert products of the block-scaled column-wise copies
    At [M, >=P], Bt [N, >=P]."""
    E, M, N = W.shape
    w_dtype = DTYPE_F32 if W.dtype == torch.float32 else DTYPE_BF16
    _check(LIB.moe_tgmm_mx(_ptr(At), _ld(At), _ptr(sfa), a_fmt, _ptr(Bt), _ld(Bt), _ptr(sfb),
                           b_fmt, _ptr(group_offsets), E, rows_cap, M, N, _ptr(W), w_dtype,
                           W.stride(1), W.stride(0), int(accumulate), _ptr(dev_status),
                           _stream(stream)))


# ------------------------------------------------------------ expert parallelism
def _np_ptr(a):
    return ctypes.c_void_p(a.ctypes.data)


def _gs_host(group_sizes):
    import numpy as np
    if isinstance(group_sizes, torch.Tensor):
        group_sizes = group_sizes.cpu().numpy()
    return np.ascontiguousarray(group_sizes, dtype=np.int32)


def moe_ep_recv_rows_cap(T: int, num_ep: int, E: int, k: int, align: int) -> int:
    return int(LIB.moe_ep_recv_rows_cap(T, num_ep, E, k, align))


def moe_ep_a2a_params(group_sizes, shard: int) -> dict:
    """group_sizes int32 [num_ep, E] (host) -> send_off, send_sz, out_off, recv_off,
    recv_sz: int64 numpy arrays [num_ep]."""
    import numpy as np
    gs = _gs_host(group_sizes)
    num_ep, E = gs.shape
    out = {n: np.zeros(num_ep, np.int64)
           for n in ("send_off", "send_sz", "out_off", "recv_off", "recv_sz")}
    _check(LIB.moe_ep_a2a_params(_np_ptr(gs), num_ep, E, shard, *(_np_ptr(out[n]) for n in (
        "send_off", "send_sz", "out_off", "recv_off", "recv_sz"))))
    return out


def moe_ep_local_layout(group_sizes, shard: int) -> dict:
    """group_sizes int32 [num_ep, E] (host) -> the chunk tables fwd_* / inv_* (int64
    [num_ep * El]) and local_offsets (int32 [El + 1]), numpy arrays."""
    import numpy as np
    gs = _gs_host(group_sizes)
    num_ep, E = gs.shape
    n = E  # num_ep * (E / num_ep) chunks
    names = ("fwd_src", "fwd_dst", "fwd_len", "inv_src", "inv_dst", "inv_len")
    out = {nm: np.zeros(n, np.int64) for nm in names}
    out["local_offsets"] = np.zeros(E // num_ep + 1 if E % num_ep == 0 else 1, np.int32)
    _check(LIB.moe_ep_local_layout(_np_ptr(gs), num_ep, E, shard,
                                   *(_np_ptr(out[nm]) for nm in names),
                                   _np_ptr(out["local_offsets"])))
    return out


def moe_sort_chunks(src, dst, src_off, dst_off, length, rows=None, stream=None):
    """Row mover: src / dst bf16 [rows, d] (row-major views); src_off / dst_off /
    length int64 device tensors [n_chunks]; rows defaults to src's rows."""
    d = src.shape[1]
    _check(LIB.moe_sort_chunks(_ptr(src), _ld(src), _ptr(dst), _ld(dst), d, _ptr(src_off),
                               _ptr(dst_off), _ptr(length), src_off.shape[0],
                               src.shape[0] if rows is None else rows, _stream(stream)))


# ------------------------------------------------------------ the whole layer
PREC_BF16 = 0
PREC_FP8 = 1
PREC_MXFP8 = 2

# MOE_BUF_* of include/moe_gb300.h, in order
BUFFERS = (
    "topk_idx", "topk_w", "xs", "group_sizes", "kept_counts", "group_offsets", "s2f", "f2s",
    "permute_ws", "h", "act", "y", "out", "partial", "dy", "d_topk_w", "d_logits", "dh", "dxs",
    "dx", "dwi", "dwo", "dbi", "dbo", "dev_status", "xs_t", "act_t", "dy_t", "dh_t",
    "f8_xs_q", "f8_xs_qt", "f8_act_q", "f8_act_qt", "f8_dy_q", "f8_dy_qt", "f8_dh_q",
    "f8_dh_qt", "f8_wi_q", "f8_wi_qt", "f8_wo_q", "f8_wo_qt", "f8_amax", "f8_sinv",
    "mx_xs_q", "mx_xs_sf", "mx_act_q", "mx_act_sf", "mx_dy_q", "mx_dy_sf", "mx_dh_q",
    "mx_dh_sf", "mx_xs_t_q", "mx_xs_t_sf", "mx_act_t_q", "mx_act_t_sf", "mx_dy_t_q",
    "mx_dy_t_sf", "mx_dh_t_q", "mx_dh_t_sf", "mx_wi_t_q", "mx_wi_t_sf", "mx_wi_q", "mx_wi_sf",
    "mx_wo_t_q", "mx_wo_t_sf", "mx_wo_q", "mx_wo_sf", "mx_woff_d", "mx_woff_f", "aux_counts",
    "aux_probs", "aux_loss", "aux_ws")
BUF = {n: i for i, n in enumerate(BUFFERS)}


class LayerConfig(ctypes.Structure):
    """moe_layer_config."""
    _fields_ = [(n, ctypes.c_int32) for n in (
        "T", "d", "f", "E", "k", "score_fn", "renorm", "num_groups", "topk_group", "align",
        "capacity", "num_chunks")] + [("aux_coeff", ctypes.c_float)] + [
        (n, ctypes.c_int32) for n in ("bias", "precision", "wgrad_colwise", "dw_dtype")]


MARK_FN = ctypes.CFUNCTYPE(None, ctypes.c_void_p, ctypes.c_char_p)


def _cfg(cfg):
    return ctypes.byref(cfg)


def _nbytes(t):
    return t.numel() * t.element_size()


def moe_layer_workspace_bytes(cfg: LayerConfig) -> int:
    """0 for an invalid configuration (reason: last_error())."""
    return int(LIB.moe_layer_workspace_bytes(_cfg(cfg)))


def moe_layer_buffer(cfg: LayerConfig, name: str):
    """(byte offset, bytes) of buffer `name` (BUFFERS) in the layer workspace."""
    off, nb = ctypes.c_size_t(), ctypes.c_size_t()
    _check(LIB.moe_layer_buffer(_cfg(cfg), BUF[name], ctypes.byref(off), ctypes.byref(nb)))
    return int(off.value), int(nb.value)


def moe_layer_init(cfg, workspace, stream=None):
    _check(LIB.moe_layer_init(_cfg(cfg), _ptr(workspace), _nbytes(workspace), _stream(stream)))


def _contig(*ts):
    for t in ts:
        assert t is None or t.is_contiguous(), "contiguous tensors only"


def _mark_fn(mark):
    """A C callback that calls mark(name), or None; keep it alive for the call."""
    if mark is None:
        return None
    return MARK_FN(lambda _ctx, name: mark(name.decode()))


def moe_layer_forward(cfg, workspace, x, logits, wi, wo, bi=None, bo=None, expert_bias=None,
                      mark=None, stream=None):
    _contig(x, logits, wi, wo, bi, bo, expert_bias)
    cb = _mark_fn(mark)
    _check(LIB.moe_layer_forward(_cfg(cfg), _ptr(workspace), _nbytes(workspace), _ptr(x),
                                 _ptr(logits), _ptr(wi), _ptr(wo), _ptr(bi), _ptr(bo),
                                 _ptr(expert_bias), ctypes.cast(cb, _P) if cb else None, None,
                                 _stream(stream)))


def moe_layer_backward(cfg, workspace, dout, logits, wi, wo, mark=None, stream=None):
    _contig(dout, logits, wi, wo)
    cb = _mark_fn(mark)
    _check(LIB.moe_layer_backward(_cfg(cfg), _ptr(workspace), _nbytes(workspace), _ptr(dout),
                                  _ptr(logits), _ptr(wi), _ptr(wo),
                                  ctypes.cast(cb, _P) if cb else None, None, _stream(stream)))


def moe_layer_pipeline_workspace_bytes(cfg) -> int:
    return int(LIB.moe_layer_pipeline_workspace_bytes(_cfg(cfg)))


class LayerPipeline:
    """moe_layer_pipeline: training steps from host buffers (see the header)."""

    def __init__(self, cfg, workspace, staging):
        self.cfg, self.workspace, self.staging = cfg, workspace, staging
        h = ctypes.c_void_p()
        _check(LIB.moe_layer_pipeline_create(_cfg(cfg), _ptr(workspace), _nbytes(workspace),
                                             _ptr(staging), _nbytes(staging), ctypes.byref(h)))
        self._h = h

    def step(self, wi, wo, h_x, h_logits, h_dout, h_out, h_dx, h_d_logits, bi=None, bo=None,
             expert_bias=None, stream=None):
        _contig(wi, wo, h_x, h_logits, h_dout, h_out, h_dx, h_d_logits, bi, bo, expert_bias)
        _check(LIB.moe_layer_pipeline_step(self._h, _ptr(wi), _ptr(wo), _ptr(bi), _ptr(bo),
                                           _ptr(expert_bias), _ptr(h_x), _ptr(h_logits),
                                           _ptr(h_dout), _ptr(h_out), _ptr(h_dx),
                                           _ptr(h_d_logits), _stream(stream)))

    def join(self, stream=None):
        _check(LIB.moe_layer_pipeline_join(self._h, _stream(stream)))

    def sync(self):
        _check(LIB.moe_layer_pipeline_sync(self._h))

    def close(self):
        """Synchronise the copy streams and release them (idempotent)."""
        if getattr(self, "_h", None):
            LIB.moe_layer_pipeline_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:   # interpreter shutdown: the library may already be unloaded
            pass
