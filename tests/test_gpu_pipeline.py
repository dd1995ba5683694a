"""The layer from host buffers (moe_layer_pipeline_*): several training steps
whose inputs come from, and whose results go back to, page-locked host
memory through the double-buffered copy streams.  Each step's host results
are checked against the fp64 oracle on that step's inputs, and bit for bit
against the device-buffer entry points on the same inputs."""
import numpy as np
import pytest
import torch

import moe_synth
from gpu_helpers import assert_close, dev_bf16, layer_shape, run_oracle
from oracle import moe_ref

pytestmark = pytest.mark.gpu
L = pytest.importorskip("mixture_experts_grouped_router_gb300._lib")

C = moe_synth.CONFIGS
CASES = {
    "mixtral": moe_synth.scaled(C["mixtral"], T=1024, d=256, f=448),
    "odd_sizes": moe_synth.MoEConfig("odd_sizes", T=999, d=200, f=136, E=7, k=3, score_fn=1,
                                     renorm=0, align=16, capacity=300),
}


def _pinned_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).astype(np.int16)).view(
        torch.bfloat16).pin_memory()


@pytest.mark.parametrize("name", list(CASES))
def test_pipeline_steps(name):
    from mixture_experts_grouped_router_gb300 import layer
    cfg = CASES[name]
    steps = 4
    inps = [moe_synth.make_inputs(cfg, seed=s) for s in range(steps)]
    w = inps[0]  # one set of weights for every step
    wi, wo = dev_bf16(w["wi"]), dev_bf16(w["wo"])
    shape = layer_shape(cfg)
    b = layer.MoEBuffers(shape)
    staging = torch.empty(L.moe_layer_pipeline_workspace_bytes(b.cfg), dtype=torch.uint8,
                          device="cuda")
    pipe = L.LayerPipeline(b.cfg, b.workspace, staging)
    h_in = [dict(x=_pinned_bf16(i["x"]), logits=torch.from_numpy(i["logits"]).pin_memory(),
                 dout=_pinned_bf16(i["dout"])) for i in inps]
    h_res = [dict(out=torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16).pin_memory(),
                  dx=torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16).pin_memory(),
                  d_logits=torch.empty(cfg.T, cfg.E, dtype=torch.float32).pin_memory())
             for _ in range(steps)]
    for s in range(steps):
        pipe.step(wi, wo, h_in[s]["x"], h_in[s]["logits"], h_in[s]["dout"], h_res[s]["out"],
                  h_res[s]["dx"], h_res[s]["d_logits"])
    pipe.sync()
    torch.cuda.synchronize()
    pipe.close()
    assert int(b.dev_status.item()) == 0

    ref = layer.MoEBuffers(shape)
    for s in range(steps):
        inp = dict(inps[s], wi=w["wi"], wo=w["wo"])
        # the device entry points on the same inputs: identical bits
        x = dev_bf16(inp["x"])
        logits = torch.from_numpy(inp["logits"]).cuda()
        layer.forward(ref, x, logits, wi, wo)
        layer.backward(ref, dev_bf16(inp["dout"]), wi, wo)
        torch.cuda.synchronize()
        for key, dev in (("out", ref.out), ("dx", ref.dx), ("d_logits", ref.d_logits)):
            assert torch.equal(h_res[s][key], dev.cpu()), (s, key)
        # and the oracle
        fw, bw = run_oracle(cfg, inp)
        assert_close("out[%d]" % s, h_res[s]["out"], fw["out"])
        assert_close("dx[%d]" % s, h_res[s]["dx"], bw["dx"])
        assert_close("d_logits[%d]" % s, h_res[s]["d_logits"],
                     moe_ref.route_topk_bwd(inp["logits"], fw["topk_idx"], bw["d_topk_w"],
                                            cfg.score_fn, cfg.renorm))
    # the weight gradients left in the workspace are the last step's
    assert torch.equal(b.dwi, ref.dwi) and torch.equal(b.dwo, ref.dwo)


@pytest.mark.parametrize("opts", [
    dict(fp8=True),
    dict(mxfp8=True),
    dict(bias=True, num_groups=4, topk_group=2, aux_coeff=1e-3, num_chunks=2),
    dict(wgrad_colwise=True),
], ids=["fp8", "mxfp8", "bias_groups_aux_chunks", "colwise"])
def test_pipeline_options(opts):
    """Every layer option through the host-buffer pipeline: two steps with
    different inputs, host results bit for bit against the device-buffer calls
    (whose parity with the oracles the layer tests of each option check)."""
    import dataclasses
    from mixture_experts_grouped_router_gb300 import layer
    cfg = moe_synth.scaled(C["mixtral"], T=512, d=256, f=384)
    shape = dataclasses.replace(layer_shape(cfg), **opts)
    inps = [moe_synth.make_inputs(cfg, seed=s) for s in range(2)]
    wi, wo = dev_bf16(inps[0]["wi"]), dev_bf16(inps[0]["wo"])
    bi = bo = None
    if shape.bias:
        bs = moe_synth.make_biases(cfg, seed=0)
        bi, bo = dev_bf16(bs["bi"]), dev_bf16(bs["bo"])
    b = layer.MoEBuffers(shape)
    staging = torch.empty(L.moe_layer_pipeline_workspace_bytes(b.cfg), dtype=torch.uint8,
                          device="cuda")
    pipe = L.LayerPipeline(b.cfg, b.workspace, staging)
    h_in = [dict(x=_pinned_bf16(i["x"]), logits=torch.from_numpy(i["logits"]).pin_memory(),
                 dout=_pinned_bf16(i["dout"])) for i in inps]
    h_res = [dict(out=torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16).pin_memory(),
                  dx=torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16).pin_memory(),
                  d_logits=torch.empty(cfg.T, cfg.E, dtype=torch.float32).pin_memory())
             for _ in inps]
    for s in range(len(inps)):
        pipe.step(wi, wo, h_in[s]["x"], h_in[s]["logits"], h_in[s]["dout"], h_res[s]["out"],
                  h_res[s]["dx"], h_res[s]["d_logits"], bi=bi, bo=bo)
    pipe.sync()
    torch.cuda.synchronize()
    pipe.close()
    assert int(b.dev_status.item()) == 0
    ref = layer.MoEBuffers(shape)
    for s, inp in enumerate(inps):
        layer.forward(ref, dev_bf16(inp["x"]), torch.from_numpy(inp["logits"]).cuda(), wi, wo,
                      bi=bi, bo=bo)
        layer.backward(ref, dev_bf16(inp["dout"]), wi, wo)
        torch.cuda.synchronize()
        for key, dev in (("out", ref.out), ("dx", ref.dx), ("d_logits", ref.d_logits)):
            got = h_res[s][key]
            assert torch.isfinite(got.float()).all(), (s, key)
            assert torch.equal(got, dev.cpu()), (s, key)
    assert torch.equal(b.dwi, ref.dwi) and torch.equal(b.dwo, ref.dwo)
    if shape.bias:
        assert torch.equal(b.dbi, ref.dbi) and torch.equal(b.dbo, ref.dbo)


def test_pipeline_no_tokens():
    """A step of no tokens through the pipeline: empty host buffers, zero
    weight gradients, no error."""
    from mixture_experts_grouped_router_gb300 import layer
    cfg = moe_synth.MoEConfig("empty", T=0, d=64, f=64, E=4, k=2)
    inp = moe_synth.make_inputs(cfg, seed=0)
    wi, wo = dev_bf16(inp["wi"]), dev_bf16(inp["wo"])
    b = layer.MoEBuffers(layer_shape(cfg))
    staging = torch.empty(max(1, L.moe_layer_pipeline_workspace_bytes(b.cfg)), dtype=torch.uint8,
                          device="cuda")
    pipe = L.LayerPipeline(b.cfg, b.workspace, staging)
    empty_bf = torch.empty(0, cfg.d, dtype=torch.bfloat16).pin_memory()
    empty_f = torch.empty(0, cfg.E, dtype=torch.float32).pin_memory()
    pipe.step(wi, wo, empty_bf, empty_f, empty_bf, empty_bf, empty_bf, empty_f)
    pipe.sync()
    torch.cuda.synchronize()
    pipe.close()
    assert int(b.dev_status.item()) == 0
    assert (b.dwi.float() == 0).all() and (b.dwo.float() == 0).all()
