"""Expert-parallel dispatch on one GPU (GPU).

* moe_sort_chunks (the local permute's row mover) against numpy;
* num_ep shards run as EPShard objects on one GPU, phase by phase in lockstep,
  with the exchanges played by copies between the shards' buffers (the data
  movement of the all-to-all; no kernel waits on another): every shard's
  outputs, input gradients and local weight gradients equal the single-GPU
  layer's on the whole batch (bit for bit without padding: a token's rows
  meet the same expert weights in the same order) and the oracle's.

No run here uses more than one GPU: the multi-rank exchange with real
collectives is covered on the CPU (tests/test_ep_multiprocess.py)."""
import numpy as np
import pytest
import torch

import moe_synth
from gpu_helpers import assert_close, dev_bf16, run_gpu_layer, run_oracle

pytestmark = pytest.mark.gpu
L = pytest.importorskip("mixture_experts_grouped_router_gb300._lib")


@pytest.mark.parametrize("d", [8, 136, 4096])
def test_sort_chunks(d):
    rng = np.random.default_rng(d)
    lens = rng.integers(0, 40, size=23)
    lens[[2, 3, 17]] = 0                     # empty chunks, two in a row
    src_off = np.concatenate([[0], np.cumsum(lens)[:-1]]) + np.arange(23) * 2  # gaps
    perm = rng.permutation(23)
    dst_off = np.zeros(23, np.int64)
    pos = 0
    for c in perm:
        dst_off[c] = pos
        pos += lens[c]
    rows = int(src_off[-1] + lens[-1] + 5)
    src_bits = moe_synth.bf16_bits(rng.standard_normal((rows, d)).astype(np.float32))
    src = dev_bf16(src_bits)
    dst = torch.full((pos + 3, d), 7.0, dtype=torch.bfloat16, device="cuda")
    t = lambda a: torch.from_numpy(np.asarray(a, np.int64)).cuda()
    L.moe_sort_chunks(src, dst, t(src_off), t(dst_off), t(lens), rows=rows)
    torch.cuda.synchronize()
    want = np.full((pos + 3, d), np.uint16(0x40E0))     # 7.0
    for a, b, n in zip(src_off, dst_off, lens):
        want[b:b + n] = src_bits[a:a + n]
    assert (dst.view(torch.int16).cpu().numpy().astype(np.uint16) == want).all()


def _exchange(dsts, srcs, shards, reverse):
    """The all-to-all between shards on one device: rows of shard s's send block
    for shard r land in r's receive buffer (reverse: the way back)."""
    for r, shr in enumerate(shards):
        pr = shr.plan_full
        for s, shs in enumerate(shards):
            ps = shs.plan_full
            if not reverse:   # s's block for r -> r's receive buffer at recv_off[s]
                n = int(ps["send_sz"][r])
                a, b = int(ps["send_off"][r]), int(pr["recv_off"][s])
                dsts[r][b:b + n].copy_(srcs[s][a:a + n])
            else:             # r's receive-buffer rows from s -> back into s's own order
                n = int(pr["recv_sz"][s])
                a, b = int(pr["recv_off"][s]), int(ps["send_off"][r])
                dsts[s][b:b + n].copy_(srcs[r][a:a + n])


@pytest.mark.parametrize("num_ep,align", [(2, 0), (4, 0), (4, 8)])
def test_ep_emulated_matches_single_gpu(num_ep, align):
    from mixture_experts_grouped_router_gb300 import ep, layer
    T, d, f, E, k = 384, 256, 192, 8, 2
    cfg = moe_synth.MoEConfig("ep", T=T * num_ep, d=d, f=f, E=E, k=k, score_fn=0, renorm=1,
                              align=align)
    inp = moe_synth.make_inputs(cfg, seed=5)
    x, wi, wo, dout = (dev_bf16(inp[n]) for n in ("x", "wi", "wo", "dout"))
    logits = torch.from_numpy(inp["logits"]).cuda()
    El = E // num_ep
    shape = layer.LayerShape(T, d, f, E, k, 0, 1, align)
    shards = [ep.EPShard(shape, num_ep, r) for r in range(num_ep)]
    sl = [slice(r * T, (r + 1) * T) for r in range(num_ep)]
    wl = [slice(r * El, (r + 1) * El) for r in range(num_ep)]
    gs = torch.stack([sh.route_permute(x[sl[r]], logits[sl[r]]) for r, sh in enumerate(shards)])
    for sh in shards:
        sh.set_plan(gs)
        sh.plan_full = L.moe_ep_a2a_params(gs.cpu().numpy(), sh.shard)
    _exchange([sh.recv for sh in shards], [sh.xs for sh in shards], shards, False)
    for r, sh in enumerate(shards):
        sh.to_local(sh.recv, sh.xs_loc)
        sh.ffn_forward(wi[wl[r]], wo[wl[r]])
        sh.from_local(sh.y_loc, sh.recv)
    _exchange([sh.y for sh in shards], [sh.recv for sh in shards], shards, True)
    for r, sh in enumerate(shards):
        sh.combine()
        sh.combine_bwd(dout[sl[r]])
    _exchange([sh.recv for sh in shards], [sh.dy for sh in shards], shards, False)
    for r, sh in enumerate(shards):
        sh.to_local(sh.recv, sh.dy_loc)
        sh.ffn_backward(wi[wl[r]], wo[wl[r]])
        sh.from_local(sh.dxs_loc, sh.recv)
    _exchange([sh.dxs for sh in shards], [sh.recv for sh in shards], shards, True)
    for sh in shards:
        sh.dispatch_bwd()
    torch.cuda.synchronize()
    for sh in shards:
        assert int(sh.dev_status.item()) == 0
    out = torch.cat([sh.out for sh in shards])
    dx = torch.cat([sh.dx for sh in shards])
    dwi = torch.cat([sh.dwi for sh in shards])
    dwo = torch.cat([sh.dwo for sh in shards])
    d_logits = torch.cat([sh.d_logits for sh in shards])
    b = run_gpu_layer(cfg, inp)
    bits = lambda t: t.contiguous().view(torch.int16)
    if align == 0:
        assert torch.equal(bits(out), bits(b.out))
        assert torch.equal(bits(dx), bits(b.dx))
        assert torch.equal(bits(dwi), bits(b.dwi))
        assert torch.equal(bits(dwo), bits(b.dwo))
        assert torch.equal(d_logits, b.d_logits)
    fw, bw = run_oracle(cfg, inp)
    assert_close("out", out, fw["out"])
    assert_close("dx", dx, bw["dx"])
    assert_close("dwi", dwi, bw["d_wi"])
    assert_close("dwo", dwo, bw["d_wo"])
