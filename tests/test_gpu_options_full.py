"""Full-size GPU parity of the layer's options, in the configurations the
benchmark times them in, on outputs the fp64 oracle recomputes one by one:

* expert-FFN biases (bi on [gate | up], bo on the output) on the Mixtral-like
  layer: sampled tokens' out / dx / d_topk_w, sampled experts' weight-gradient
  columns and rows, their bias-gradient entries, and the whole of dbo;
* group-limited top-k (8 groups, 4 kept) with the auxiliary load-balancing
  loss on the DeepSeek-like layer: the routing and layout of every token
  (bit-exact), the loss and its per-expert counts, and sampled tokens'
  out / dx / d_topk_w / d_logits (routing gradient plus the loss's logit
  gradient, taken over all tokens).

Integer outputs bit-exact; floating point within the layer's tolerances
(relative Frobenius <= 1e-2, max |diff| <= 5e-2 * max |ref|; routing weights
to 1e-6).
"""
import numpy as np
import pytest
import torch

import moe_synth
from gpu_helpers import assert_close, check_layout, run_gpu_layer
from oracle import moe_ref

pytestmark = pytest.mark.gpu
pytest.importorskip("mixture_experts_grouped_router_gb300._lib")

f64 = moe_synth.bits_to_f64


def _layout(cfg, inp, num_groups=0, topk_group=0):
    idx, w = moe_ref.route_topk(inp["logits"], cfg.k, cfg.score_fn, cfg.renorm,
                                num_groups=num_groups, topk_group=topk_group)
    lay = moe_ref.permute_layout(idx, cfg.E, cfg.align, cfg.capacity)
    return idx, w, lay


def _sampled_tokens(cfg, inp, b, w, lay, toks, bi=None, bo=None):
    """out, dx, d_topk_w of the sampled tokens, each (token, slot) through its
    expert's FFN in fp64 (biases added when given)."""
    T, k = cfg.T, cfg.k
    f2s = lay["flat_to_sorted"].reshape(T, k)
    off = lay["group_offsets"]
    n = len(toks)
    out_ref = np.zeros((n, cfg.d))
    dx_ref = np.zeros((n, cfg.d))
    dw_ref = np.zeros((n, k))
    x = f64(inp["x"][toks])
    dout = f64(inp["dout"][toks])
    for i, t in enumerate(toks):
        for j in range(k):
            p = f2s[t, j]
            if p < 0:
                continue
            e = int(np.searchsorted(off, p, side="right") - 1)
            wi_e, wo_e = f64(inp["wi"][e]), f64(inp["wo"][e])
            h = x[i:i + 1] @ wi_e + (0.0 if bi is None else bi[e])
            y = moe_ref.swiglu(h) @ wo_e + (0.0 if bo is None else bo[e])
            out_ref[i] += w[t, j] * y[0]
            dw_ref[i, j] = dout[i] @ y[0]
            dh = moe_ref.swiglu_bwd(h, (w[t, j] * dout[i:i + 1]) @ wo_e.T)
            dx_ref[i] += (dh @ wi_e.T)[0]
    tt = torch.from_numpy(toks).cuda()
    assert_close("out[sampled]", b.out[tt], out_ref)
    assert_close("dx[sampled]", b.dx[tt], dx_ref)
    assert_close("d_topk_w[sampled]", b.d_topk_w[tt], dw_ref)
    return dw_ref


def test_bias_full_size_sampled():
    cfg = moe_synth.CONFIGS["mixtral"]
    inp = moe_synth.make_inputs(cfg, seed=0)
    biases = moe_synth.make_biases(cfg, seed=0)
    b = run_gpu_layer(cfg, inp, biases=biases)
    assert int(b.dev_status.item()) == 0
    idx, w, lay = _layout(cfg, inp)
    check_layout(b, dict(topk_idx=idx, topk_w=w, layout=lay), cfg.T, cfg.k)
    bi, bo = f64(biases["bi"]), f64(biases["bo"])
    rng = np.random.default_rng(11)
    _sampled_tokens(cfg, inp, b, w, lay, rng.choice(cfg.T, size=5, replace=False), bi, bo)

    off = lay["group_offsets"]
    f = cfg.f
    for e in rng.choice(np.nonzero(lay["group_sizes"] > 0)[0], size=2, replace=False):
        s, t_ = int(off[e]), int(off[e + 1])
        rows = lay["sorted_to_flat"][s:t_]
        real = rows >= 0
        xs = np.zeros((t_ - s, cfg.d))
        xs[real] = f64(inp["x"][rows[real] // cfg.k])
        dy = np.zeros((t_ - s, cfg.d))
        dy[real] = w.reshape(-1)[rows[real]][:, None] * f64(inp["dout"][rows[real] // cfg.k])
        # dbo[e] = column sums of the expert's dY rows (every entry)
        assert_close("dbo[%d]" % e, b.dbo[e], dy.sum(axis=0))
        wi_e, wo_e = f64(inp["wi"][e]), f64(inp["wo"][e])
        c = int(rng.integers(f))
        g = xs @ wi_e[:, c] + bi[e, c]
        u = xs @ wi_e[:, f + c] + bi[e, f + c]
        dh = moe_ref.swiglu_bwd(np.stack([g, u], 1), (dy @ wo_e[c, :])[:, None])
        dh[~real] = 0.0                                   # padding rows carry no gradient
        dwi_cols = xs.T @ dh
        act_c = moe_ref.swiglu(np.stack([g, u], 1))[:, 0]
        act_c[~real] = 0.0
        assert_close("dwi[%d][:, %d]" % (e, c), b.dwi[e][:, c], dwi_cols[:, 0])
        assert_close("dwi[%d][:, f+%d]" % (e, c), b.dwi[e][:, f + c], dwi_cols[:, 1])
        assert_close("dwo[%d][%d, :]" % (e, c), b.dwo[e][c, :], act_c @ dy)
        got = b.dbi[e][[c, f + c]].cpu().numpy().astype(np.float64)
        assert_close("dbi[%d][c, f+c]" % e, got, dh.sum(axis=0))


def test_grouped_routing_aux_loss_full_size_sampled():
    cfg = moe_synth.CONFIGS["dsv3"]
    G, tg, coeff = 8, 4, 1e-3
    inp = moe_synth.make_inputs(cfg, seed=0)
    b = run_gpu_layer(cfg, inp, num_groups=G, topk_group=tg, aux_coeff=coeff)
    assert int(b.dev_status.item()) == 0
    idx, w, lay = _layout(cfg, inp, G, tg)
    check_layout(b, dict(topk_idx=idx, topk_w=w, layout=lay), cfg.T, cfg.k)
    # every token's experts lie in at most tg of the G groups
    groups = idx // (cfg.E // G)
    assert max(len(set(r)) for r in groups.tolist()) <= tg

    loss, counts, _ = moe_ref.aux_loss(inp["logits"], idx, cfg.E, cfg.score_fn, coeff)
    assert b.aux_counts.cpu().numpy().astype(np.int64).tolist() == counts.tolist()
    np.testing.assert_allclose(float(b.aux_loss.item()), loss, rtol=2e-5)

    rng = np.random.default_rng(12)
    toks = rng.choice(cfg.T, size=6, replace=False)
    dw_ref = _sampled_tokens(cfg, inp, b, w, lay, toks)
    d_aux = moe_ref.aux_loss_bwd(inp["logits"], counts, cfg.k, cfg.score_fn, coeff)
    d_logits = moe_ref.route_topk_bwd(inp["logits"][toks], idx[toks], dw_ref, cfg.score_fn,
                                      cfg.renorm) + d_aux[toks]
    assert_close("d_logits[sampled]", b.d_logits[torch.from_numpy(toks).cuda()], d_logits)
