"""Expert-parallel MoE layer: each shard owns E / num_ep experts, and the
permuted rows travel to the shard that owns their expert and back.

The sequence is the single-VJP block of TransformerEngine PR #2912 ("[JAX]
Add an MoE Block (Layer) that compound router, permutation, groupedGEMM and
communication", sequence diagram) with its expert-parallel steps:

forward   route -> permute (all E experts) -> all-gather group sizes ->
          ragged all-to-all -> local permute -> grouped GEMMs of the local
          experts -> local unpermute -> reverse all-to-all -> combine
backward  combine backward -> all-to-all (dY) -> local permute -> dgrad /
          weight-gradient GEMMs -> local unpermute -> reverse all-to-all (dXs)
          -> dispatch backward

Every arithmetic step and every row move runs in libmoe_gb300.so; the
exchange bookkeeping (send / receive sizes, the local chunk tables) is the
library's host code, and the exchanges themselves are the caller's
collectives, passed in as two functions (``torch.distributed`` with NCCL
between GPUs):

    allgather(t)                         -> [num_ep, *t.shape] of every shard's t
    all_to_all(out, inp, out_splits, in_splits)   rows of inp to the shards,
                                         rows from the shards into out

The shard runs its phases in order; :func:`forward` and :func:`backward`
chain them for one shard.  Capacity dropping is not offered here (each shard
would drop by its own counts); align padding is (each source pads its groups).
"""
from __future__ import annotations

import torch

from . import _lib as L
from .layer import LayerShape


class EPShard:
    """Buffers and exchange plan of one shard (device memory through PyTorch)."""

    def __init__(self, s: LayerShape, num_ep: int, shard: int, device="cuda",
                 dw_dtype=torch.bfloat16):
        if s.E % num_ep:
            raise ValueError("E=%d is not a multiple of num_ep=%d" % (s.E, num_ep))
        if s.capacity > 0 or s.fp8 or s.bias or s.num_chunks > 1:
            raise ValueError("the expert-parallel layer takes no capacity, FP8, biases or "
                             "K-chunks")
        self.s, self.num_ep, self.shard = s, num_ep, shard
        T, d, f, E, k = s.T, s.d, s.f, s.E, s.k
        self.El = E // num_ep
        bf, i32, f32 = torch.bfloat16, torch.int32, torch.float32
        dev = device
        R = L.moe_rows_cap(T, E, k, s.align, s.capacity)
        self.rows_cap = R
        # the shard's own tokens, permuted over all E experts
        self.topk_idx = torch.empty(T, k, dtype=i32, device=dev)
        self.topk_w = torch.empty(T, k, dtype=f32, device=dev)
        self.xs = torch.empty(R, d, dtype=bf, device=dev)
        self.group_sizes = torch.empty(E, dtype=i32, device=dev)
        self.kept_counts = torch.empty(E, dtype=i32, device=dev)
        self.group_offsets = torch.empty(E + 1, dtype=i32, device=dev)
        self.s2f = torch.empty(R, dtype=i32, device=dev)
        self.f2s = torch.empty(T * k, dtype=i32, device=dev)
        self.ws = torch.empty(L.moe_permute_workspace_bytes(T, E), dtype=torch.uint8, device=dev)
        self.y = torch.empty(R, d, dtype=bf, device=dev)      # expert outputs, own order
        self.out = torch.empty(T, d, dtype=bf, device=dev)
        self.dy = torch.empty(R, d, dtype=bf, device=dev)
        self.dxs = torch.empty(R, d, dtype=bf, device=dev)
        self.dx = torch.empty(T, d, dtype=bf, device=dev)
        self.d_topk_w = torch.empty(T, k, dtype=f32, device=dev)
        self.d_logits = torch.empty(T, E, dtype=f32, device=dev)
        self.logits = None
        # rows received for the local experts: source-major (recv) and expert-major (loc)
        RC = L.moe_ep_recv_rows_cap(T, num_ep, E, k, s.align)
        self.recv_rows_cap = RC
        self.recv = torch.empty(RC, d, dtype=bf, device=dev)
        self.xs_loc = torch.empty(RC, d, dtype=bf, device=dev)
        self.h = torch.empty(RC, 2 * f, dtype=bf, device=dev)
        self.act = torch.empty(RC, f, dtype=bf, device=dev)
        self.y_loc = torch.empty(RC, d, dtype=bf, device=dev)
        self.dy_loc = torch.empty(RC, d, dtype=bf, device=dev)
        self.dh = torch.empty(RC, 2 * f, dtype=bf, device=dev)
        self.dxs_loc = torch.empty(RC, d, dtype=bf, device=dev)
        self.dwi = torch.empty(self.El, d, 2 * f, dtype=dw_dtype, device=dev)
        self.dwo = torch.empty(self.El, f, d, dtype=dw_dtype, device=dev)
        self.local_offsets = torch.empty(self.El + 1, dtype=i32, device=dev)
        self.tables = torch.empty(6, E, dtype=torch.int64, device=dev)
        self.dev_status = torch.zeros(1, dtype=i32, device=dev)
        self.plan = None

    # ------------------------------------------------------------ phases
    def route_permute(self, x, logits, stream=None, expert_bias=None):
        """Route and permute this shard's tokens over all E experts; returns the
        group sizes (device int32 [E]) that every shard must see."""
        s = self.s
        self.logits = logits
        L.moe_route_topk(logits, s.k, s.score_fn, s.renorm, self.topk_idx, self.topk_w, stream,
                         expert_bias=expert_bias, num_groups=s.num_groups,
                         topk_group=s.topk_group)
        L.moe_permute(x, self.topk_idx, s.E, s.align, s.capacity, self.xs, self.group_sizes,
                      self.kept_counts, self.group_offsets, self.s2f, self.f2s, self.ws,
                      self.dev_status, stream)
        return self.group_sizes

    def set_plan(self, all_group_sizes, stream=None):
        """all_group_sizes: int32 [num_ep, E] of every shard (host or device);
        computes the exchange sizes and the local chunk tables (host), and puts
        the tables and the local group offsets on the device."""
        gs = L._gs_host(all_group_sizes)
        if gs.shape != (self.num_ep, self.s.E):
            raise ValueError("group sizes of shape %s, expected (%d, %d)"
                             % (gs.shape, self.num_ep, self.s.E))
        prm = L.moe_ep_a2a_params(gs, self.shard)
        lay = L.moe_ep_local_layout(gs, self.shard)
        n_recv = int(prm["recv_sz"].sum())
        if n_recv > self.recv_rows_cap:
            raise RuntimeError("%d rows to receive > receive buffer of %d"
                               % (n_recv, self.recv_rows_cap))
        import numpy as np
        host = torch.from_numpy(np.stack([lay[n] for n in ("fwd_src", "fwd_dst", "fwd_len",
                                                           "inv_src", "inv_dst", "inv_len")]))
        self.tables.copy_(host, non_blocking=False)
        self.local_offsets.copy_(torch.from_numpy(lay["local_offsets"]))
        self.plan = dict(send=prm["send_sz"].tolist(), recv=prm["recv_sz"].tolist(),
                         n_send=int(prm["send_sz"].sum()), n_recv=n_recv,
                         n_loc=int(lay["local_offsets"][-1]))
        return self.plan

    def to_local(self, src, dst, stream=None):
        """Receive buffer (source-major) -> local buffer (expert-major)."""
        t = self.tables
        L.moe_sort_chunks(src, dst, t[0], t[1], t[2], rows=self.plan["n_recv"], stream=stream)

    def from_local(self, src, dst, stream=None):
        """Local buffer (expert-major) -> receive-buffer order (source-major)."""
        t = self.tables
        L.moe_sort_chunks(src, dst, t[3], t[4], t[5], rows=self.plan["n_loc"], stream=stream)

    def ffn_forward(self, wi_loc, wo_loc, stream=None):
        """Grouped GEMMs of the local experts on the local rows."""
        n = self.plan["n_loc"]
        off = self.local_offsets
        L.moe_gmm(self.xs_loc[:n], wi_loc, 0, off, self.h[:n], L.EPI_SWIGLU_FWD,
                  C2=self.act[:n], dev_status=self.dev_status, stream=stream)
        L.moe_gmm(self.act[:n], wo_loc, 0, off, self.y_loc[:n], L.EPI_NONE,
                  dev_status=self.dev_status, stream=stream)

    def combine(self, stream=None):
        L.moe_combine(self.y, self.f2s, self.topk_w, self.out, self.s.k, stream)
        return self.out

    def combine_bwd(self, dout, stream=None):
        """dY and d_topk_w on the shard's own permuted rows; d_logits."""
        s = self.s
        L.moe_unpermute_bwd(dout, self.y, self.f2s, self.s2f, self.group_offsets, self.topk_w,
                            self.dy, self.d_topk_w, stream)
        L.moe_route_topk_bwd(self.logits, self.topk_idx, self.topk_w, self.d_topk_w,
                             s.score_fn, s.renorm, self.d_logits, stream)

    def ffn_backward(self, wi_loc, wo_loc, stream=None):
        """dgrad and weight-gradient GEMMs of the local experts."""
        n = self.plan["n_loc"]
        off = self.local_offsets
        L.moe_gmm(self.dy_loc[:n], wo_loc, 1, off, self.dh[:n], L.EPI_SWIGLU_BWD,
                  aux=self.h[:n], dev_status=self.dev_status, stream=stream)
        L.moe_tgmm(self.act[:n], self.dy_loc[:n], off, self.dwo, dev_status=self.dev_status,
                   stream=stream)
        L.moe_gmm(self.dh[:n], wi_loc, 1, off, self.dxs_loc[:n], L.EPI_NONE,
                  dev_status=self.dev_status, stream=stream)
        L.moe_tgmm(self.xs_loc[:n], self.dh[:n], off, self.dwi, dev_status=self.dev_status,
                   stream=stream)

    def dispatch_bwd(self, stream=None):
        L.moe_combine(self.dxs, self.f2s, None, self.dx, self.s.k, stream)
        return self.dx


def forward(sh: EPShard, x, logits, wi_loc, wo_loc, allgather, all_to_all, stream=None):
    """One shard's forward: x bf16 [T, d], logits fp32 [T, E], wi_loc / wo_loc the
    weights of its El experts.  Returns sh.out."""
    gs = sh.route_permute(x, logits, stream)
    plan = sh.set_plan(allgather(gs), stream)
    all_to_all(sh.recv[:plan["n_recv"]], sh.xs[:plan["n_send"]], plan["recv"], plan["send"])
    sh.to_local(sh.recv, sh.xs_loc, stream)
    sh.ffn_forward(wi_loc, wo_loc, stream)
    sh.from_local(sh.y_loc, sh.recv, stream)
    all_to_all(sh.y[:plan["n_send"]], sh.recv[:plan["n_recv"]], plan["send"], plan["recv"])
    return sh.combine(stream)


def backward(sh: EPShard, dout, wi_loc, wo_loc, all_to_all, stream=None):
    """One shard's backward after forward(): dx in sh.dx, d_logits in sh.d_logits,
    the local experts' weight gradients in sh.dwi / sh.dwo."""
    plan = sh.plan
    sh.combine_bwd(dout, stream)
    all_to_all(sh.recv[:plan["n_recv"]], sh.dy[:plan["n_send"]], plan["recv"], plan["send"])
    sh.to_local(sh.recv, sh.dy_loc, stream)
    sh.ffn_backward(wi_loc, wo_loc, stream)
    sh.from_local(sh.dxs_loc, sh.recv, stream)
    all_to_all(sh.dxs[:plan["n_send"]], sh.recv[:plan["n_recv"]], plan["send"], plan["recv"])
    return sh.dispatch_bwd(stream)


def torch_collectives(group=None):
    """(allgather, all_to_all) over a torch.distributed process group."""
    import torch.distributed as dist

    def allgather(t):
        n = dist.get_world_size(group)
        out = torch.empty(n * t.numel(), dtype=t.dtype, device=t.device)
        dist.all_gather_into_tensor(out, t.contiguous().view(-1), group=group)
        return out.view((n,) + tuple(t.shape))

    def all_to_all(out, inp, out_splits, in_splits):
        dist.all_to_all_single(out, inp, [int(v) for v in out_splits],
                               [int(v) for v in in_splits], group=group)

    return allgather, all_to_all
