"""Degenerate and boundary cases of the layer on the GPU, against the oracle:
no tokens, a single expert, every expert selected (k = E), the largest expert
count the router takes (E = 256), and row counts that leave one-row groups."""
import numpy as np
import pytest
import torch

import moe_synth
from gpu_helpers import assert_close, check_layout, run_gpu_layer, run_oracle

pytestmark = pytest.mark.gpu
pytest.importorskip("mixture_experts_grouped_router_gb300._lib")

CASES = {
    "single_expert": moe_synth.MoEConfig("single_expert", T=300, d=128, f=192, E=1, k=1),
    "all_experts": moe_synth.MoEConfig("all_experts", T=200, d=136, f=128, E=4, k=4,
                                       score_fn=1, renorm=1),
    "many_experts": moe_synth.MoEConfig("many_experts", T=640, d=64, f=64, E=256, k=8,
                                        score_fn=1, renorm=1),
    "few_tokens": moe_synth.MoEConfig("few_tokens", T=3, d=64, f=64, E=8, k=2, align=4,
                                      capacity=1),
}


@pytest.mark.parametrize("name", list(CASES))
def test_edge_layer(name):
    cfg = CASES[name]
    inp = moe_synth.make_inputs(cfg, seed=3)
    b = run_gpu_layer(cfg, inp)
    assert int(b.dev_status.item()) == 0
    fw, bw = run_oracle(cfg, inp)
    check_layout(b, fw, cfg.T, cfg.k)
    assert_close("out", b.out, fw["out"])
    assert_close("dx", b.dx, bw["dx"])
    assert_close("dwi", b.dwi, bw["d_wi"])
    assert_close("dwo", b.dwo, bw["d_wo"])
    assert_close("d_topk_w", b.d_topk_w, bw["d_topk_w"])


def test_no_tokens():
    cfg = moe_synth.MoEConfig("empty", T=0, d=64, f=64, E=4, k=2)
    inp = moe_synth.make_inputs(cfg, seed=0)
    b = run_gpu_layer(cfg, inp)
    assert int(b.dev_status.item()) == 0
    assert b.group_offsets.cpu().tolist() == [0, 0, 0, 0, 0]
    assert (b.dwi.float() == 0).all() and (b.dwo.float() == 0).all()
    assert b.out.shape == (0, 64) and b.dx.shape == (0, 64)
