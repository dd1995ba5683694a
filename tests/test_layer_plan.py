"""The whole-layer entry points on the host (no GPU): the workspace planner's
layout (every buffer the configuration needs, at least its shape's bytes,
256-byte aligned, none overlapping), the configurations it rejects, and the
argument checks of moe_layer_forward / _backward / the pipeline, which fail
before anything is enqueued."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_gb300.h")


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__._build_module().build()
    from mixture_experts_grouped_router_gb300 import _lib
    return _lib


def test_buffer_names_follow_the_header(L):
    src = open(HEADER).read()
    body = src[src.index("MOE_BUF_TOPK_IDX = 0"):src.index("MOE_BUF_COUNT")]
    names = [n.lower() for n in re.findall(r"\bMOE_BUF_([A-Z0-9_]+)", body)]
    assert tuple(names) == L.BUFFERS


def _cfg(L, **kw):
    base = dict(T=300, d=256, f=384, E=6, k=2, score_fn=0, renorm=1, num_groups=0, topk_group=0,
                align=0, capacity=0, num_chunks=1, aux_coeff=0.0, bias=0, precision=0,
                wgrad_colwise=0, dw_dtype=0)
    base.update(kw)
    return L.LayerConfig(**base)


def _expected(L, c):
    """Bytes each buffer needs, from the shapes (0 = not used)."""
    T, d, f, E, k = c.T, c.d, c.f, c.E, c.k
    R = L.moe_rows_cap(T, E, k, c.align, c.capacity)
    P = L.moe_fp8_padded_rows(R, E)
    dw = 4 if c.dw_dtype == 1 else 2
    want = dict(topk_idx=T * k * 4, topk_w=T * k * 4, xs=R * d * 2, group_sizes=E * 4,
                kept_counts=E * 4, group_offsets=(E + 1) * 4, s2f=R * 4, f2s=T * k * 4,
                permute_ws=L.moe_permute_workspace_bytes(T, E), h=R * 2 * f * 2, act=R * f * 2,
                y=R * d * 2, out=T * d * 2, dy=R * d * 2, d_topk_w=T * k * 4,
                d_logits=T * E * 4, dh=R * 2 * f * 2, dxs=R * d * 2, dx=T * d * 2,
                dwi=E * d * 2 * f * dw, dwo=E * f * d * dw, dev_status=4)
    if c.num_chunks > 1:
        want["partial"] = R * 2 * f * 4
    if c.bias:
        want.update(dbi=E * 2 * f * 4, dbo=E * d * 4)
    if c.wgrad_colwise and c.precision == 0:
        want.update(xs_t=d * P * 2, act_t=f * P * 2, dy_t=d * P * 2, dh_t=2 * f * P * 2)
    if c.precision == 1:
        want.update(f8_xs_q=R * d, f8_xs_qt=d * P, f8_act_q=R * f, f8_act_qt=f * P,
                    f8_dy_q=R * d, f8_dy_qt=d * P, f8_dh_q=R * 2 * f, f8_dh_qt=2 * f * P,
                    f8_wi_q=E * d * 2 * f, f8_wi_qt=E * d * 2 * f, f8_wo_q=E * f * d,
                    f8_wo_qt=E * f * d, f8_amax=(4 + 2 * E) * 4, f8_sinv=(4 + 2 * E) * 4)
    if c.precision == 2:
        G, PL, SW, TL = (L.MX_ROWS_GROUPED, L.MX_ROWS_PLAIN, L.MX_ROWS_SWIGLU,
                         L.MX_ROWS_TILES)
        for n, rows, cols, m, g in (("xs", R, d, G, E), ("act", R, f, G, E), ("dy", R, d, G, E),
                                    ("dh", R, 2 * f, G, E), ("xs_t", d, P, PL, E),
                                    ("act_t", f, P, PL, E), ("dy_t", d, P, TL, 1),
                                    ("dh_t", 2 * f, P, TL, 1), ("wi_t", 2 * f, E * d, SW, E),
                                    ("wi", E * d, 2 * f, TL, E), ("wo_t", d, E * f, TL, 1),
                                    ("wo", E * f, d, TL, E)):
            want["mx_%s_q" % n] = rows * cols
            want["mx_%s_sf" % n] = L.moe_mx_scale_bytes(rows, cols, m, g)
        want.update(mx_woff_d=(E + 1) * 4, mx_woff_f=(E + 1) * 4)
    if c.aux_coeff > 0:
        want.update(aux_counts=E * 4, aux_probs=E * 4, aux_loss=4,
                    aux_ws=L.moe_aux_loss_workspace_bytes(T, E))
    return want


CASES = [
    dict(),
    dict(align=16, capacity=40, bias=1, dw_dtype=1),
    dict(num_chunks=4, aux_coeff=1e-3, num_groups=3, topk_group=2, score_fn=1),
    dict(wgrad_colwise=1),
    dict(precision=1),
    dict(precision=2),
    dict(precision=2, wgrad_colwise=1, T=0),
]


@pytest.mark.parametrize("kw", CASES, ids=[str(i) for i in range(len(CASES))])
def test_plan_layout(L, kw):
    c = _cfg(L, **kw)
    total = L.moe_layer_workspace_bytes(c)
    assert total > 0, L.last_error()
    want = _expected(L, c)
    spans = []
    for name in L.BUFFERS:
        off, nb = L.moe_layer_buffer(c, name)
        assert nb == want.get(name, 0), (name, nb, want.get(name, 0))
        if nb:
            assert off % 256 == 0 and off + nb <= total, (name, off, nb, total)
            spans.append((off, off + nb, name))
    spans.sort()
    for (a0, a1, an), (b0, b1, bn) in zip(spans, spans[1:]):
        assert a1 <= b0, ("overlap", an, bn)


@pytest.mark.parametrize("kw, msg", [
    (dict(num_chunks=3), "does not divide"),
    (dict(precision=1, bias=1), "neither biases"),
    (dict(precision=2, num_chunks=2), "neither biases"),
    (dict(precision=2, d=192), "multiples of 128"),
    (dict(k=7), "bad sizes"),
    (dict(precision=5), "unknown precision"),
    (dict(dw_dtype=3), "dw_dtype"),
])
def test_plan_rejects(L, kw, msg):
    c = _cfg(L, **kw)
    assert L.moe_layer_workspace_bytes(c) == 0
    assert msg in L.last_error()
    off, nb = ctypes.c_size_t(), ctypes.c_size_t()
    assert L.LIB.moe_layer_buffer(ctypes.byref(c), 0, ctypes.byref(off),
                                  ctypes.byref(nb)) == L.MOE_ERR_INVALID_ARG


def test_entry_points_check_before_enqueueing(L):
    """Fake device addresses: every call below must fail on its arguments alone."""
    c = _cfg(L, bias=1)
    total = L.moe_layer_workspace_bytes(c)
    P = lambda v: ctypes.c_void_p(v)
    ws = P(1 << 20)
    cb = ctypes.byref(c)
    # workspace: null, unaligned, too small
    assert L.LIB.moe_layer_forward(cb, None, total, P(256), P(256), P(256), P(256), P(256),
                                   P(256), None, None, None, None) == L.MOE_ERR_INVALID_ARG
    assert "aligned" in L.last_error()
    assert L.LIB.moe_layer_forward(cb, P((1 << 20) + 16), total, P(256), P(256), P(256), P(256),
                                   P(256), P(256), None, None, None,
                                   None) == L.MOE_ERR_INVALID_ARG
    assert L.LIB.moe_layer_forward(cb, ws, total - 1, P(256), P(256), P(256), P(256), P(256),
                                   P(256), None, None, None, None) == L.MOE_ERR_INVALID_ARG
    assert "needed" in L.last_error()
    # a null input, biases missing for a bias configuration
    assert L.LIB.moe_layer_forward(cb, ws, total, None, P(256), P(256), P(256), P(256), P(256),
                                   None, None, None, None) == L.MOE_ERR_INVALID_ARG
    assert L.LIB.moe_layer_forward(cb, ws, total, P(256), P(256), P(256), P(256), None, None,
                                   None, None, None, None) == L.MOE_ERR_INVALID_ARG
    assert "bi and bo" in L.last_error()
    assert L.LIB.moe_layer_backward(cb, ws, total, None, P(256), P(256), P(256), None, None,
                                    None) == L.MOE_ERR_INVALID_ARG
    # the pipeline: staging missing or too small, step without a pipeline
    h = ctypes.c_void_p()
    need = L.moe_layer_pipeline_workspace_bytes(c)
    assert need == 2 * sum(-(-b // 256) * 256 for b in (
        c.T * c.d * 2, c.T * c.E * 4, c.T * c.d * 2, c.T * c.d * 2, c.T * c.d * 2, c.T * c.E * 4))
    assert L.LIB.moe_layer_pipeline_create(cb, ws, total, None, need,
                                           ctypes.byref(h)) == L.MOE_ERR_INVALID_ARG
    assert L.LIB.moe_layer_pipeline_create(cb, ws, total, P(1 << 30), need - 1,
                                           ctypes.byref(h)) == L.MOE_ERR_INVALID_ARG
    assert not h.value
    assert L.LIB.moe_layer_pipeline_step(None, *([P(256)] * 11), None) == L.MOE_ERR_INVALID_ARG
    L.LIB.moe_layer_pipeline_destroy(None)


def test_layer_buffers_reject_bad_id(L):
    c = _cfg(L)
    off, nb = ctypes.c_size_t(), ctypes.c_size_t()
    for bad in (-1, len(L.BUFFERS)):
        assert L.LIB.moe_layer_buffer(ctypes.byref(c), bad, ctypes.byref(off),
                                      ctypes.byref(nb)) == L.MOE_ERR_INVALID_ARG
