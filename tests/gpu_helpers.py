"""Helpers shared by the GPU parity tests: device transfer of the seeded
inputs, running the layer through the C ABI, and the acceptance tolerances.

Tolerances (stated for the layer's floating-point outputs): relative Frobenius
error <= 1e-2 and max |diff| <= 5e-2 * max |ref| against the fp64 oracle on the
same bf16 inputs; fp32 routing weights to 1e-6 absolute; integer outputs
bit-exact.
"""
import numpy as np
import torch

import moe_synth
from oracle import moe_ref

REL_FRO = 1e-2
MAX_REL = 5e-2
W_ATOL = 1e-6


def dev_bf16(bits, device="cuda"):
    return torch.from_numpy(np.ascontiguousarray(bits).astype(np.int16)).view(torch.bfloat16).to(device)


def host_f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_close(name, got, want, rel_fro=REL_FRO, max_rel=MAX_REL):
    got = host_f64(got) if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (name, got.shape, want.shape)
    assert np.isfinite(got).all(), "%s: non-finite values" % name
    nref = np.linalg.norm(want)
    err = np.linalg.norm(got - want)
    mref = np.abs(want).max() if want.size else 0.0
    mdiff = np.abs(got - want).max() if want.size else 0.0
    if nref == 0:
        assert err == 0, "%s: expected exact zeros, |err| = %g" % (name, err)
        return
    assert err <= rel_fro * nref, "%s: rel Frobenius %.3g > %g" % (name, err / nref, rel_fro)
    assert mdiff <= max_rel * mref, "%s: max diff %.3g > %g * %.3g" % (name, mdiff, max_rel, mref)


def layer_shape(cfg, bias=False, num_groups=0, topk_group=0, aux_coeff=0.0,
                wgrad_colwise=False):
    from mixture_experts_grouped_router_gb300 import layer
    return layer.LayerShape(cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.score_fn, cfg.renorm,
                            cfg.align, cfg.capacity, cfg.num_chunks, bias,
                            num_groups=num_groups, topk_group=topk_group, aux_coeff=aux_coeff,
                            wgrad_colwise=wgrad_colwise)


def run_gpu_layer(cfg, inp, device="cuda", dw_dtype=torch.bfloat16, biases=None, num_groups=0,
                  topk_group=0, aux_coeff=0.0, expert_bias=None, wgrad_colwise=False):
    """biases: None or the dict of moe_synth.make_biases; num_groups / topk_group /
    aux_coeff / expert_bias (fp32 [E] numpy or None): the routing options of the layer;
    wgrad_colwise: weight gradients from column-wise copies."""
    from mixture_experts_grouped_router_gb300 import layer
    x, wi, wo, dout = (dev_bf16(inp[n], device) for n in ("x", "wi", "wo", "dout"))
    logits = torch.from_numpy(inp["logits"]).to(device)
    shape = layer_shape(cfg, biases is not None, num_groups, topk_group, aux_coeff,
                        wgrad_colwise)
    b = layer.MoEBuffers(shape, device=device, dw_dtype=dw_dtype)
    bi = bo = None
    if biases is not None:
        bi, bo = dev_bf16(biases["bi"], device), dev_bf16(biases["bo"], device)
    eb = None if expert_bias is None else torch.from_numpy(
        np.asarray(expert_bias, np.float32)).to(device)
    layer.forward(b, x, logits, wi, wo, bi=bi, bo=bo, expert_bias=eb)
    layer.backward(b, dout, wi, wo)
    torch.cuda.synchronize()
    return b


def run_oracle(cfg, inp, biases=None, num_groups=0, topk_group=0, expert_bias=None):
    f64 = moe_synth.bits_to_f64
    x, wi, wo, dout = (f64(inp[n]) for n in ("x", "wi", "wo", "dout"))
    bi = bo = None
    if biases is not None:
        bi, bo = f64(biases["bi"]), f64(biases["bo"])
    fw = moe_ref.forward(x, inp["logits"], wi, wo, cfg.k, cfg.score_fn, cfg.renorm, cfg.align,
                         cfg.capacity, cfg.num_chunks, bi=bi, bo=bo, num_groups=num_groups,
                         topk_group=topk_group, expert_bias=expert_bias)
    bw = moe_ref.backward(fw, dout, wi, wo, cfg.k, cfg.num_chunks)
    return fw, bw


def check_layout(b, fw, T, k):
    lay = fw["layout"]
    R = lay["R"]
    assert (b.topk_idx.cpu().numpy() == fw["topk_idx"]).all()
    np.testing.assert_allclose(b.topk_w.cpu().numpy(), fw["topk_w"], rtol=0, atol=W_ATOL)
    assert b.group_sizes.cpu().numpy().tolist() == lay["group_sizes"].tolist()
    assert b.kept_counts.cpu().numpy().tolist() == lay["kept_counts"].tolist()
    assert b.group_offsets.cpu().numpy().tolist() == lay["group_offsets"].tolist()
    s2f = b.s2f.cpu().numpy()
    assert s2f[:R].tolist() == lay["sorted_to_flat"].tolist()
    assert (s2f[R:] == -1).all()
    assert b.f2s.cpu().numpy().tolist() == lay["flat_to_sorted"].tolist()
