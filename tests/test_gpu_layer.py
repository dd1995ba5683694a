"""End-to-end GPU parity of the layer (forward + backward through the C ABI)
against the fp64 oracle.

* reduced sizes of the five workloads, compared element by element;
* the five workloads at full size, in the configuration the benchmark times:
  integer outputs compared in full, floating-point outputs on sampled tokens,
  expert columns and rows that the oracle recomputes one by one.
"""
import math

import numpy as np
import pytest
import torch

import moe_synth
from gpu_helpers import (assert_close, check_layout, host_f64, run_gpu_layer, run_oracle)
from oracle import moe_ref

pytestmark = pytest.mark.gpu
pytest.importorskip("mixture_experts_grouped_router_gb300._lib")

C = moe_synth.CONFIGS
SMALL = {
    "tiny": C["tiny"],
    "mixtral": moe_synth.scaled(C["mixtral"], T=1024, d=256, f=448),
    "dsv3": moe_synth.scaled(C["dsv3"], T=512, d=448, f=256),
    "skewed": moe_synth.scaled(C["skewed"], T=4096, d=256, f=128, capacity=64),
    "dsv3_chunked": moe_synth.scaled(C["dsv3_chunked"], T=512, d=448, f=256),
    "odd_sizes": moe_synth.MoEConfig("odd_sizes", T=999, d=200, f=136, E=7, k=3, score_fn=1,
                                     renorm=0, align=16, capacity=300),
}


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("wgrad_colwise", [False, True])
def test_layer_small(name, wgrad_colwise):
    """Every output element by element; with wgrad_colwise the weight
    gradients read the column-wise copies the epilogues write."""
    cfg = SMALL[name]
    inp = moe_synth.make_inputs(cfg, seed=0)
    b = run_gpu_layer(cfg, inp, wgrad_colwise=wgrad_colwise)
    assert int(b.dev_status.item()) == 0
    fw, bw = run_oracle(cfg, inp)
    check_layout(b, fw, cfg.T, cfg.k)
    R = fw["layout"]["R"]
    assert_close("xs", b.xs[:R], fw["xs"], rel_fro=0, max_rel=0)
    assert_close("h", b.h[:R], fw["h"])
    assert_close("act", b.act[:R], fw["act"])
    assert_close("y", b.y[:R], fw["y"])
    assert_close("out", b.out, fw["out"])
    assert_close("dy", b.dy[:R], bw["dy"])
    assert_close("d_topk_w", b.d_topk_w, bw["d_topk_w"])
    assert_close("d_logits", b.d_logits,
                 moe_ref.route_topk_bwd(inp["logits"], fw["topk_idx"], bw["d_topk_w"],
                                        cfg.score_fn, cfg.renorm))
    assert_close("dh", b.dh[:R], bw["dh"])
    assert_close("dxs", b.dxs[:R], bw["d_xs"])
    assert_close("dx", b.dx, bw["dx"])
    assert_close("dwo", b.dwo, bw["d_wo"])
    assert_close("dwi", b.dwi, bw["d_wi"])
    empty = np.nonzero(fw["layout"]["group_sizes"] == 0)[0]
    for e in empty:
        assert (b.dwi[e].float() == 0).all() and (b.dwo[e].float() == 0).all()


@pytest.mark.parametrize("name", ["dsv3", "mixtral"])
def test_layer_expert_bias(name):
    """DeepSeek-V3's selection bias through the layer (MaxText PR #2579, the
    routing that keeps pre-bias logits): experts ranked by logit + bias, the
    weights from the unbiased logits; every output against the oracle."""
    cfg = SMALL[name]
    inp = moe_synth.make_inputs(cfg, seed=3)
    bias = np.random.default_rng(11).standard_normal(cfg.E).astype(np.float32)
    b = run_gpu_layer(cfg, inp, expert_bias=bias)
    assert int(b.dev_status.item()) == 0
    fw, bw = run_oracle(cfg, inp, expert_bias=bias)
    # the bias must change the selection, or this test checks nothing new
    plain_idx, _ = moe_ref.route_topk(inp["logits"], cfg.k, cfg.score_fn, cfg.renorm)
    assert (plain_idx != fw["topk_idx"]).any()
    check_layout(b, fw, cfg.T, cfg.k)
    R = fw["layout"]["R"]
    assert_close("out", b.out, fw["out"])
    assert_close("d_topk_w", b.d_topk_w, bw["d_topk_w"])
    assert_close("d_logits", b.d_logits,
                 moe_ref.route_topk_bwd(inp["logits"], fw["topk_idx"], bw["d_topk_w"],
                                        cfg.score_fn, cfg.renorm))
    assert_close("dh", b.dh[:R], bw["dh"])
    assert_close("dx", b.dx, bw["dx"])
    assert_close("dwo", b.dwo, bw["d_wo"])
    assert_close("dwi", b.dwi, bw["d_wi"])


# ---------------------------------------------------------------------------
# full-size workloads, sampled
# ---------------------------------------------------------------------------
def _sampled_check(cfg, inp, b, n_tok=6, n_cols=3, seed=0):
    f64 = moe_synth.bits_to_f64
    T, k, f = cfg.T, cfg.k, cfg.f
    rng = np.random.default_rng(seed)
    idx, w = moe_ref.route_topk(inp["logits"], k, cfg.score_fn, cfg.renorm)
    lay = moe_ref.permute_layout(idx, cfg.E, cfg.align, cfg.capacity)
    check_layout(b, dict(topk_idx=idx, topk_w=w, layout=lay), T, k)
    f2s = lay["flat_to_sorted"].reshape(T, k)
    off = lay["group_offsets"]

    def expert_of(p):
        return int(np.searchsorted(off, p, side="right") - 1)

    # rows of sampled tokens: forward and input-gradient chain, row by row
    toks = rng.choice(T, size=n_tok, replace=False)
    dout = f64(inp["dout"][toks])
    x = f64(inp["x"][toks])
    out_ref = np.zeros((n_tok, cfg.d))
    dx_ref = np.zeros((n_tok, cfg.d))
    dw_ref = np.zeros((n_tok, k))
    rows_p, inter = [], {n: [] for n in ("h", "act", "y", "dy", "dh", "dxs")}
    for i, t in enumerate(toks):
        for j in range(k):
            p = f2s[t, j]
            if p < 0:
                continue
            e = expert_of(p)
            wi_e = f64(inp["wi"][e])
            wo_e = f64(inp["wo"][e])
            h = x[i:i + 1] @ wi_e
            act = moe_ref.swiglu(h)
            y = act @ wo_e
            out_ref[i] += w[t, j] * y[0]
            dw_ref[i, j] = dout[i] @ y[0]
            dy = w[t, j] * dout[i:i + 1]
            dh = moe_ref.swiglu_bwd(h, dy @ wo_e.T)
            dxs = dh @ wi_e.T
            dx_ref[i] += dxs[0]
            rows_p.append(p)
            for n, v in (("h", h), ("act", act), ("y", y), ("dy", dy), ("dh", dh), ("dxs", dxs)):
                inter[n].append(v[0])
    assert_close("out[sampled]", b.out[torch.from_numpy(toks).cuda()], out_ref)
    assert_close("dx[sampled]", b.dx[torch.from_numpy(toks).cuda()], dx_ref)
    assert_close("d_topk_w[sampled]", b.d_topk_w[torch.from_numpy(toks).cuda()], dw_ref)
    # the saved intermediates of the sampled tokens' rows, at full size
    if rows_p:
        prow = torch.tensor(rows_p, dtype=torch.long, device="cuda")
        for n, buf in (("h", b.h), ("act", b.act), ("y", b.y), ("dy", b.dy), ("dh", b.dh),
                       ("dxs", b.dxs)):
            assert_close("%s[sampled rows]" % n, buf[prow], np.stack(inter[n]))

    # weight-gradient columns / rows of sampled experts: whole-group reductions
    nonempty = np.nonzero(lay["group_sizes"] > 0)[0]
    for e in rng.choice(nonempty, size=min(n_cols, len(nonempty)), replace=False):
        s, t_ = int(off[e]), int(off[e + 1])
        rows = lay["sorted_to_flat"][s:t_]
        real = rows >= 0
        xs = np.zeros((t_ - s, cfg.d))
        xs[real] = f64(inp["x"][rows[real] // k])
        dy = np.zeros((t_ - s, cfg.d))
        a = rows[real]
        dy[real] = w.reshape(-1)[a][:, None] * f64(inp["dout"][a // k])
        wi_e = f64(inp["wi"][e])
        wo_e = f64(inp["wo"][e])
        c = int(rng.integers(f))
        g = xs @ wi_e[:, c]
        u = xs @ wi_e[:, f + c]
        d_act = dy @ wo_e[c, :]
        dh = moe_ref.swiglu_bwd(np.stack([g, u], 1), d_act[:, None])
        dwi_cols = xs.T @ dh          # dWi[e][:, c] and dWi[e][:, f + c]
        act_c = moe_ref.swiglu(np.stack([g, u], 1))[:, 0]
        dwo_row = act_c @ dy          # dWo[e][c, :]
        assert_close("dwi[%d][:, %d]" % (e, c), b.dwi[e][:, c], dwi_cols[:, 0])
        assert_close("dwi[%d][:, f+%d]" % (e, c), b.dwi[e][:, f + c], dwi_cols[:, 1])
        assert_close("dwo[%d][%d, :]" % (e, c), b.dwo[e][c, :], dwo_row)
    for e in np.nonzero(lay["group_sizes"] == 0)[0]:
        assert (b.dwi[e].float() == 0).all() and (b.dwo[e].float() == 0).all()
    return lay


@pytest.mark.parametrize("name", list(moe_synth.CONFIGS))
def test_layer_full_size_sampled(name):
    cfg = moe_synth.CONFIGS[name]
    inp = moe_synth.make_inputs(cfg, seed=0)
    b = run_gpu_layer(cfg, inp)
    assert int(b.dev_status.item()) == 0
    lay = _sampled_check(cfg, inp, b)
    if name == "skewed":
        assert (lay["group_sizes"] == 0).sum() >= 5
        assert math.ceil(cfg.T * cfg.k / cfg.E) == cfg.capacity
    # padded / empty rows of the permuted activations are zero
    R = lay["R"]
    pad = torch.from_numpy(lay["sorted_to_flat"] < 0).cuda()
    if pad.any():
        assert (b.xs[:R][pad].float() == 0).all()
        assert (b.dy[:R][pad].float() == 0).all()
