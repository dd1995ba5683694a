"""Expert-parallel dispatch on the CPU with gloo ranks (2 and 4 shards): the
library's exchange bookkeeping (moe_ep_a2a_params, moe_ep_local_layout) and a
real ragged all-to-all move every token row to the shard that owns its
expert and back.  The device kernels' steps are played by the oracle (route,
permute, grouped GEMMs, combine) and by numpy (the chunk moves); the check is
that every shard ends with what the single-device oracle computes for the
whole batch: its local experts' rows in the same order, its tokens' outputs
and input gradients, and its experts' full weight gradients.

TransformerEngine PR #2912, sequence diagram (_dispatch / _combine with
ragged_all_to_all, the backward with the same exchanges) and the helpers
compute_ragged_all_to_all_params / local_permute_after_a2a."""
import json
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _move(src, src_off, dst_off, length, n_dst):
    """numpy stand-in for moe_sort_chunks."""
    dst = np.full((n_dst,) + src.shape[1:], np.nan if src.dtype.kind == "f" else -7, src.dtype)
    for a, b, n in zip(src_off, dst_off, length):
        dst[b:b + n] = src[a:a + n]
    return dst


def _a2a(arr, out_splits, in_splits):
    out = torch.empty((int(sum(out_splits)),) + arr.shape[1:], dtype=torch.from_numpy(arr).dtype)
    dist.all_to_all_single(out, torch.from_numpy(np.ascontiguousarray(arr)),
                           [int(v) for v in out_splits], [int(v) for v in in_splits])
    return out.numpy()


def _ep_rank(rank, ws, port, case, out_dir):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        import moe_synth
        from mixture_experts_grouped_router_gb300 import _lib as L
        from oracle import moe_ref
        T, d, f, E, k, sfn, ren, align = case
        El = E // ws
        cfg = moe_synth.MoEConfig("ep", T=T * ws, d=d, f=f, E=E, k=k, score_fn=sfn, renorm=ren,
                                  align=align)
        inp = moe_synth.make_inputs(cfg, seed=7)
        f64 = moe_synth.bits_to_f64
        x_all, wi, wo, dout_all = (f64(inp[n]) for n in ("x", "wi", "wo", "dout"))
        # the single-device oracle over the whole batch (every shard's tokens in shard order)
        fw = moe_ref.forward(x_all, inp["logits"], wi, wo, k, sfn, ren, align)
        bw = moe_ref.backward(fw, dout_all, wi, wo, k)
        mine = slice(rank * T, (rank + 1) * T)
        x, logits, dout = x_all[mine], inp["logits"][mine], dout_all[mine]

        # shard: route and permute its own tokens over all E experts
        idx, w = moe_ref.route_topk(logits, k, sfn, ren)
        lay = moe_ref.permute_layout(idx, E, align)
        R = lay["R"]
        xs = moe_ref.permute_rows(x, lay, k)[:R]
        gid = np.where(lay["sorted_to_flat"] >= 0, lay["sorted_to_flat"] + rank * T * k, -1)
        gs = torch.from_numpy(lay["group_sizes"].astype(np.int32))
        gs_all = torch.empty(ws * E, dtype=torch.int32)
        dist.all_gather_into_tensor(gs_all, gs)
        gs_all = gs_all.view(ws, E)
        prm = L.moe_ep_a2a_params(gs_all.numpy(), rank)
        loc = L.moe_ep_local_layout(gs_all.numpy(), rank)
        # the exchange's own consistency: where I receive from s is where s sends to me
        oo = torch.from_numpy(prm["out_off"])
        oo_all = torch.empty(ws * ws, dtype=torch.int64)
        dist.all_gather_into_tensor(oo_all, oo)
        oo_all = oo_all.view(ws, ws)
        assert (oo_all[:, rank].numpy() == prm["recv_off"]).all()
        assert prm["send_sz"].sum() == R
        n_recv = int(prm["recv_sz"].sum())
        assert n_recv <= L.moe_ep_recv_rows_cap(T, ws, E, k, align)
        n_loc = int(loc["local_offsets"][-1])
        assert n_loc == n_recv

        # dispatch: ragged all-to-all, then the local permute
        recv = _a2a(xs, prm["recv_sz"], prm["send_sz"])
        rid = _a2a(gid.astype(np.int64), prm["recv_sz"], prm["send_sz"])
        xs_loc = _move(recv, loc["fwd_src"], loc["fwd_dst"], loc["fwd_len"], n_loc)
        id_loc = _move(rid, loc["fwd_src"], loc["fwd_dst"], loc["fwd_len"], n_loc)
        goff = fw["layout"]["group_offsets"]
        loff = loc["local_offsets"]
        for le in range(El):
            e = rank * El + le
            ids = id_loc[loff[le]:loff[le + 1]]
            want = fw["layout"]["sorted_to_flat"][goff[e]:goff[e + 1]]
            # the expert's assignments in the single-device order (padding apart)
            assert ids[ids >= 0].tolist() == want[want >= 0].tolist(), (rank, le)
            rows = xs_loc[loff[le]:loff[le + 1]]
            assert (rows[ids >= 0] == x_all[ids[ids >= 0] // k]).all()
            assert (rows[ids < 0] == 0).all()
            if align <= 1:
                assert (rows == fw["xs"][goff[e]:goff[e + 1]]).all()

        # the local experts' FFN, the local unpermute and the reverse exchange
        wi_l, wo_l = wi[rank * El:(rank + 1) * El], wo[rank * El:(rank + 1) * El]
        h = moe_ref.gmm(xs_loc, wi_l, loff)
        act = moe_ref.swiglu(h)
        y_loc = moe_ref.gmm(act, wo_l, loff)
        y_recv = _move(y_loc, loc["inv_src"], loc["inv_dst"], loc["inv_len"], n_recv)
        y = _a2a(y_recv, prm["send_sz"], prm["recv_sz"])
        out = moe_ref.combine(y, lay["flat_to_sorted"], w)
        np.testing.assert_allclose(out, fw["out"][mine], rtol=1e-12, atol=1e-12)

        # backward through the same exchanges
        dy, d_w = moe_ref.combine_bwd(dout, y, lay["flat_to_sorted"], w, R)
        dy_loc = _move(_a2a(dy[:R], prm["recv_sz"], prm["send_sz"]), loc["fwd_src"],
                       loc["fwd_dst"], loc["fwd_len"], n_loc)
        dh = moe_ref.swiglu_bwd(h, moe_ref.gmm(dy_loc, wo_l, loff, transpose_rhs=True))
        dwo = moe_ref.tgmm(act, dy_loc, loff, El)
        dwi = moe_ref.tgmm(xs_loc, dh, loff, El)
        dxs_loc = moe_ref.gmm(dh, wi_l, loff, transpose_rhs=True)
        dxs = _a2a(_move(dxs_loc, loc["inv_src"], loc["inv_dst"], loc["inv_len"], n_recv),
                   prm["send_sz"], prm["recv_sz"])
        dx = moe_ref.dispatch_bwd(dxs, lay["flat_to_sorted"], T, k)
        np.testing.assert_allclose(d_w, bw["d_topk_w"][mine], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(dx, bw["dx"][mine], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(dwo, bw["d_wo"][rank * El:(rank + 1) * El], rtol=1e-10,
                                   atol=1e-12)
        np.testing.assert_allclose(dwi, bw["d_wi"][rank * El:(rank + 1) * El], rtol=1e-10,
                                   atol=1e-12)
        json.dump(dict(ok=True, n_recv=n_recv), open(os.path.join(out_dir, "r%d.json" % rank), "w"))
    finally:
        dist.destroy_process_group()


CASES = {
    # T per shard, d, f, E, k, score_fn, renorm, align
    "softmax_top2": (96, 32, 48, 8, 2, 0, 1, 0),
    "sigmoid_top4_align8": (80, 24, 40, 16, 4, 1, 1, 8),
}


@pytest.mark.parametrize("ws", [2, 4])
@pytest.mark.parametrize("name", list(CASES))
def test_ep_dispatch_matches_single_device(ws, name, tmp_path):
    mp.start_processes(_ep_rank, args=(ws, _free_port(), CASES[name], str(tmp_path)),
                       nprocs=ws, start_method="spawn")
    for r in range(ws):
        assert json.load(open(tmp_path / ("r%d.json" % r)))["ok"]
