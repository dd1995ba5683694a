"""GPU parity of the auxiliary load-balancing loss (moe_aux_loss) and its
logit gradient (moe_aux_loss_bwd) against the oracle, and of the layer with
group-limited routing and the loss switched on (d_logits = routing-weight
gradient + loss gradient).

The loss follows TransformerEngine PR #2912 ("[JAX] Add an MoE Block (Layer)
that compound router, permutation, groupedGEMM and communication"),
Description: the block's optional auxiliary load-balancing loss, in the
Switch-Transformer / DeepSeek-V3 form coeff * sum_e f_e P_e."""
import numpy as np
import pytest
import torch

import moe_synth
from gpu_helpers import assert_close, check_layout, dev_bf16, run_oracle
from oracle import moe_ref

pytestmark = pytest.mark.gpu
L = pytest.importorskip("mixture_experts_grouped_router_gb300._lib")

AUX_CASES = [
    # T, E, k, score_fn
    (1, 8, 2, 0), (300, 8, 2, 0), (1025, 64, 6, 1), (4096, 256, 8, 1), (777, 5, 5, 0),
    (16384, 8, 2, 0),
]


def _run_aux(lg, idx, k, sfn, coeff, d_init=None):
    T, E = lg.shape
    lgd = torch.from_numpy(lg).cuda()
    idd = torch.from_numpy(idx.astype(np.int32)).cuda()
    counts = torch.full((E,), -1, dtype=torch.int32, device="cuda")
    P = torch.full((E,), float("nan"), dtype=torch.float32, device="cuda")
    loss = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(L.moe_aux_loss_workspace_bytes(T, E), dtype=torch.uint8, device="cuda")
    L.moe_aux_loss(lgd, idd, sfn, coeff, counts, P, loss, ws)
    d = (torch.from_numpy(d_init).cuda() if d_init is not None
         else torch.full((T, E), float("nan"), dtype=torch.float32, device="cuda"))
    L.moe_aux_loss_bwd(lgd, counts, k, sfn, coeff, d, d_loss=0.5,
                       accumulate=d_init is not None)
    torch.cuda.synchronize()
    return counts.cpu().numpy(), P.cpu().numpy(), float(loss.item()), d.cpu().numpy()


@pytest.mark.parametrize("case", AUX_CASES)
def test_aux_loss_and_bwd(case):
    T, E, k, sfn = case
    rng = np.random.default_rng(T + E + k)
    lg = (rng.standard_normal((T, E)) + np.linspace(-2, 2, E)).astype(np.float32)
    idx, _ = moe_ref.route_topk(lg, k, sfn, 1)
    coeff = 0.01
    counts, P, loss, d = _run_aux(lg, idx, k, sfn, coeff)
    rloss, rcounts, rP = moe_ref.aux_loss(lg, idx, E, sfn, coeff)
    assert counts.tolist() == rcounts.tolist()
    np.testing.assert_allclose(P, rP, rtol=2e-5, atol=1e-7)
    np.testing.assert_allclose(loss, rloss, rtol=2e-5)
    rd = moe_ref.aux_loss_bwd(lg, rcounts, k, sfn, coeff, d_loss=0.5)
    # entries scale with d_loss * coeff / T; with k = E every f_e is 1 and the
    # gradient vanishes (the oracle leaves rounding residue of 1e-22 there)
    scale = max(np.abs(rd).max(), 0.5 * coeff / max(T, 1))
    np.testing.assert_allclose(d, rd, rtol=0, atol=2e-5 * scale)


def test_aux_loss_bwd_accumulates():
    T, E, k = 500, 16, 4
    rng = np.random.default_rng(5)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    idx, _ = moe_ref.route_topk(lg, k, 1, 1)
    base = rng.standard_normal((T, E)).astype(np.float32)
    _, _, _, d = _run_aux(lg, idx, k, 1, 0.1, d_init=base)
    _, rc, _ = moe_ref.aux_loss(lg, idx, E, 1, 0.1)
    rd = base + moe_ref.aux_loss_bwd(lg, rc, k, 1, 0.1, d_loss=0.5)
    np.testing.assert_allclose(d, rd, rtol=0, atol=1e-6)


def test_aux_loss_equal_logits_is_coeff():
    T, E, k = 1000, 32, 4
    lg = np.zeros((T, E), np.float32)
    idx, _ = moe_ref.route_topk(lg, k, 0, 1)
    counts, P, loss, _ = _run_aux(lg, idx, k, 0, 0.02)
    assert counts.tolist() == [T] * k + [0] * (E - k)
    np.testing.assert_allclose(loss, 0.02, rtol=1e-6)


def test_aux_loss_no_tokens():
    lg = np.zeros((0, 8), np.float32)
    counts, P, loss, _ = _run_aux(lg, np.zeros((0, 2), np.int32), 2, 0, 0.01)
    assert counts.tolist() == [0] * 8 and (P == 0).all() and loss == 0.0


def test_layer_grouped_routing_with_aux_loss():
    from mixture_experts_grouped_router_gb300 import layer
    cfg = moe_synth.MoEConfig("dsv3_grouped", T=512, d=256, f=128, E=32, k=8, score_fn=1,
                              renorm=1)
    G, tg, coeff = 8, 4, 0.01
    inp = moe_synth.make_inputs(cfg, seed=2)
    x, wi, wo, dout = (dev_bf16(inp[n]) for n in ("x", "wi", "wo", "dout"))
    logits = torch.from_numpy(inp["logits"]).cuda()
    shape = layer.LayerShape(cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.score_fn, cfg.renorm,
                             num_groups=G, topk_group=tg, aux_coeff=coeff)
    b = layer.MoEBuffers(shape)
    layer.forward(b, x, logits, wi, wo)
    layer.backward(b, dout, wi, wo)
    torch.cuda.synchronize()
    assert int(b.dev_status.item()) == 0
    # oracle: grouped routing, then the layer on that routing decision
    ridx, _ = moe_ref.route_topk(inp["logits"], cfg.k, cfg.score_fn, cfg.renorm,
                                 num_groups=G, topk_group=tg)
    assert (b.topk_idx.cpu().numpy() == ridx).all()
    fw, bw = run_oracle(cfg, inp, num_groups=G, topk_group=tg)
    check_layout(b, fw, cfg.T, cfg.k)
    assert_close("out", b.out, fw["out"])
    assert_close("dx", b.dx, bw["dx"])
    rloss, rcounts, _ = moe_ref.aux_loss(inp["logits"], ridx, cfg.E, cfg.score_fn, coeff)
    np.testing.assert_allclose(float(b.aux_loss.item()), rloss, rtol=2e-5)
    d_logits = (moe_ref.route_topk_bwd(inp["logits"], ridx, bw["d_topk_w"], cfg.score_fn,
                                       cfg.renorm) +
                moe_ref.aux_loss_bwd(inp["logits"], rcounts, cfg.k, cfg.score_fn, coeff))
    assert_close("d_logits", b.d_logits, d_logits)
