"""Dense one-hot brute force of the MoE layer, used only to pin the oracle.

It shares no code with ``oracle/`` and follows a different formulation: every
expert runs on every token, and a gate matrix that is zero for unselected or
dropped (token, expert) pairs masks and weights the results.  Selection is
decided by counting, for each expert, how many experts beat it; capacity by
counting earlier tokens that chose the same expert.  Gradients come from
PyTorch CPU autograd in float64 over this dense formulation.
"""
import math

import numpy as np
import torch


def route_dense(logits, k, score_fn, renorm):
    """Returns (sel [T,E] bool, slot [T,E] int (-1 if unselected), weight [T,E] float)."""
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    sel = np.zeros((T, E), dtype=bool)
    slot = np.full((T, E), -1, dtype=np.int64)
    weight = np.zeros((T, E))
    for t in range(T):
        row = [float(v) for v in logits[t]]
        for e in range(E):
            beaten_by = sum(1 for e2 in range(E)
                            if row[e2] > row[e] or (row[e2] == row[e] and e2 < e))
            if beaten_by < k:
                sel[t, e] = True
                slot[t, e] = beaten_by
        if score_fn == 0:
            mx = max(row)
            z = sum(math.exp(v - mx) for v in row)
            score = [math.exp(v - mx) / z for v in row]
        else:
            score = [1.0 / (1.0 + math.exp(-v)) for v in row]
        tot = sum(score[e] for e in range(E) if sel[t, e])
        for e in range(E):
            if sel[t, e]:
                weight[t, e] = score[e] / tot if renorm else score[e]
    return sel, slot, weight


def kept_dense(sel, capacity):
    """kept[t,e]: selected and fewer than `capacity` earlier tokens chose e."""
    T, E = sel.shape
    kept = np.zeros_like(sel)
    for e in range(E):
        seen = 0
        for t in range(T):
            if sel[t, e]:
                kept[t, e] = capacity <= 0 or seen < capacity
                seen += 1
    return kept


def layout_dense(sel, kept, align):
    """Row position of every kept (t, e), expert-major then token order."""
    T, E = sel.shape
    a = max(align, 1)
    pos = np.full((T, E), -1, dtype=np.int64)
    start = 0
    sizes = []
    for e in range(E):
        n = 0
        for t in range(T):
            if kept[t, e]:
                pos[t, e] = start + n
                n += 1
        g = -(-n // a) * a
        sizes.append(g)
        start += g
    return pos, np.array(sizes), start


def ffn_dense_torch(x, wi, wo, gate, bi=None, bo=None):
    """out[t] = sum_e gate[t,e] * ((silu(x wi_0[e] + bi_0[e]) * (x wi_1[e] + bi_1[e])) wo[e]
    + bo[e]), all torch fp64."""
    E, d, f2 = wi.shape
    f = f2 // 2
    out = torch.zeros(x.shape[0], wo.shape[2], dtype=torch.float64)
    for e in range(E):
        g = x @ wi[e, :, :f]
        u = x @ wi[e, :, f:]
        if bi is not None:
            g = g + bi[e, :f]
            u = u + bi[e, f:]
        act = g * torch.sigmoid(g) * u
        y = act @ wo[e]
        if bo is not None:
            y = y + bo[e]
        out = out + gate[:, e:e + 1] * y
    return out


def layer_dense(x, logits, wi, wo, dout, k, score_fn, renorm, capacity=0, bi=None, bo=None):
    """Forward output and gradients (dx, dwi, dwo, dgate[, dbi, dbo]) of L = <dout, out>."""
    sel, slot, weight = route_dense(logits, k, score_fn, renorm)
    kept = kept_dense(sel, capacity)
    gate_np = np.where(kept, weight, 0.0)
    xt = torch.tensor(x, dtype=torch.float64, requires_grad=True)
    wit = torch.tensor(wi, dtype=torch.float64, requires_grad=True)
    wot = torch.tensor(wo, dtype=torch.float64, requires_grad=True)
    gt = torch.tensor(gate_np, dtype=torch.float64, requires_grad=True)
    bit = None if bi is None else torch.tensor(bi, dtype=torch.float64, requires_grad=True)
    bot = None if bo is None else torch.tensor(bo, dtype=torch.float64, requires_grad=True)
    out = ffn_dense_torch(xt, wit, wot, gt, bit, bot)
    loss = (out * torch.tensor(dout, dtype=torch.float64)).sum()
    loss.backward()
    res = dict(sel=sel, slot=slot, weight=weight, kept=kept, out=out.detach().numpy(),
               dx=xt.grad.numpy(), dwi=wit.grad.numpy(), dwo=wot.grad.numpy(),
               dgate=gt.grad.numpy())
    if bit is not None:
        res["dbi"] = bit.grad.numpy()
        res["dbo"] = bot.grad.numpy()
    return res


def route_bwd_dense_torch(logits, sel, d_gate, score_fn, renorm, bias=None):
    """d_logits of L = sum d_gate * gate(logits), the selection mask held fixed:
    the gate of every (token, expert) pair is written as a dense formula in
    torch fp64 and differentiated by autograd."""
    lt = torch.tensor(np.asarray(logits, np.float64), requires_grad=True)
    mask = torch.tensor(sel, dtype=torch.float64)
    if score_fn == 0:
        score = torch.softmax(lt, dim=1)
    else:
        score = torch.sigmoid(lt)
    gate = score * mask
    if renorm:
        gate = gate / gate.sum(dim=1, keepdim=True)
    (gate * torch.tensor(d_gate, dtype=torch.float64)).sum().backward()
    return lt.grad.numpy()
