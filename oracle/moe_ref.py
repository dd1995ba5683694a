"""Plain fp64 NumPy oracle of the MoE expert layer (router top-k, permutation,
grouped SwiGLU FFN, weighted combine, and the whole backward pass).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module;
only the tests, the package's smoke check and the benchmark's CPU-baseline
leg do.  It shares no code with the CUDA path.

It follows the pages' own plain path: the pure-JAX argsort / gather / einsum
formulation of TransformerEngine PR #2912, "[JAX] Add an MoE Block (Layer)
that compound router, permutation, groupedGEMM and communication" (called
TE-2912 below), and the Pallas gmm/tgmm semantics of MaxText PR #4295,
"Overlap moe comms with collective matmul" (MT-4295 below).  Every
floating-point step runs in float64 on inputs that were rounded to bf16 (or
are fp32 logits) and then widened; intermediates are not rounded.

Readings taken where the pages are silent (each is listed with its reason in
the design notes of the repository):
  * softmax routing renormalises over the k selected experts when ``renorm``;
    sigmoid routing (DeepSeek-V3) renormalises the selected sigmoid scores;
  * experts are ranked by the fp32 logit, descending, ties to the lower id;
  * capacity C keeps the first C assignments of each expert in (expert,
    token) order, before align_size padding; dropped slots contribute 0;
  * SwiGLU is act = silu(x wi_0) * (x wi_1), silu(z) = z * sigmoid(z);
  * padding rows of the permuted activations and of dY are zero;
  * group-limited routing: a group scores the fp32 sum of its k/topk_group
    largest selection keys; the best topk_group groups stay open;
  * the auxiliary load-balancing loss is coeff * sum_e f_e P_e (Switch /
    DeepSeek-V3 form) with routing counts taken before capacity drops.
"""
from __future__ import annotations

import numpy as np

SOFTMAX = 0
SIGMOID = 1


# ----------------------------------------------------------------------------
# routing
# ----------------------------------------------------------------------------
def group_limit_mask(key: np.ndarray, k: int, num_groups: int, topk_group: int) -> np.ndarray:
    """Experts a token may choose under group-limited routing.

    TE-2912, Description ("top-K with optional grouped/sigmoid scoring (for
    DSv3 workload)") and the ``group_topk`` argument of the router.  The E
    experts form ``num_groups`` contiguous groups of E / num_groups.  A
    group's score is the sum of its m = k / topk_group largest selection keys,
    added in fp32 from the largest down (DeepSeek-V3 sums the top two of each
    of its 8 groups for k = 8 over 4 groups); the ``topk_group`` groups with
    the highest scores (ties to the lower group id) stay open.

    key: fp32 [T, E] selection keys.  Returns bool [T, E].
    """
    T, E = key.shape
    G = num_groups
    assert E % G == 0 and 1 <= topk_group <= G and k % topk_group == 0
    gs = E // G
    m = k // topk_group
    assert m <= gs
    grouped = np.sort(key.reshape(T, G, gs).astype(np.float32), axis=-1)[:, :, ::-1]
    score = grouped[:, :, 0].copy()
    for i in range(1, m):
        score = (score + grouped[:, :, i]).astype(np.float32)
    gid = np.broadcast_to(np.arange(G), (T, G))
    order = np.lexsort((gid, -score.astype(np.float64)), axis=-1)
    open_g = np.zeros((T, G), bool)
    np.put_along_axis(open_g, order[:, :topk_group], True, axis=1)
    return np.repeat(open_g, gs, axis=1)


def route_topk(logits: np.ndarray, k: int, score_fn: int, renorm: int, expert_bias=None,
               num_groups: int = 0, topk_group: int = 0):
    """Top-k expert selection and routing weights.

    TE-2912, Description ("TE's fused router ... top-K with optional
    grouped/sigmoid scoring (for DSv3 workload)").  Selection ranks the fp32
    logits (both score maps are monotone); the weights are the softmax (over
    all E) or sigmoid scores of the selected experts, optionally divided by
    their sum over the k selected.

    With ``expert_bias`` (DeepSeek-V3's per-expert bias; TE-2912, the
    ``expert_bias`` field of the body residuals; MaxText PR #2579 "Onboard
    explicit sharding to deepseek", the routing code that keeps pre-bias
    logits) the selection ranks the fp32 sums logit + bias while the weights
    still come from the unbiased logits.

    With ``num_groups`` > 1, selection is group-limited (group_limit_mask):
    only experts of the ``topk_group`` best groups compete.

    Returns (topk_idx int32 [T,k], topk_w float64 [T,k]).
    """
    logits = np.asarray(logits, dtype=np.float32)
    T, E = logits.shape
    assert np.isfinite(logits).all(), "the oracle assumes finite router logits"
    assert 1 <= k <= E
    l64 = logits.astype(np.float64)           # exact widening: same order as fp32
    key = logits if expert_bias is None else \
        (logits + np.asarray(expert_bias, dtype=np.float32)[None, :]).astype(np.float32)
    ids = np.broadcast_to(np.arange(E), (T, E))
    rank_key = -key.astype(np.float64)
    if num_groups > 1:
        closed = ~group_limit_mask(key, k, num_groups, topk_group)
        rank_key = np.where(closed, np.inf, rank_key)     # closed experts rank last
    # np.lexsort sorts by the last key first: -key descending, then expert id ascending
    order = np.lexsort((ids, rank_key), axis=-1)
    topk_idx = order[:, :k].astype(np.int32)
    if score_fn == SOFTMAX:
        m = l64.max(axis=1, keepdims=True)
        ex = np.exp(l64 - m)
        score = ex / ex.sum(axis=1, keepdims=True)
    elif score_fn == SIGMOID:
        score = 1.0 / (1.0 + np.exp(-l64))
    else:
        raise ValueError("score_fn must be 0 (softmax) or 1 (sigmoid)")
    w = np.take_along_axis(score, topk_idx.astype(np.int64), axis=1)
    if renorm:
        w = w / w.sum(axis=1, keepdims=True)
    return topk_idx, w


def route_topk_bwd(logits: np.ndarray, topk_idx: np.ndarray, d_topk_w: np.ndarray,
                   score_fn: int, renorm: int, chunk: int = 2048):
    """Gradient of the routing weights w.r.t. the router logits, selection fixed.

    TE-2912, sequence diagram / ``_moe_bwd_rule``: the block's backward returns
    the gate-kernel gradient, i.e. it carries d_w back through the router.
    Written as the chain rule with explicit Jacobians: the score Jacobian
    (softmax: diag(p) - p p^T over all E; sigmoid: diag(s (1 - s))), the rows of
    the selected experts, then the renormalisation Jacobian
    d(v_j / S)/d v_m = (delta_jm - w_j) / S with S = sum of the selected v.
    Returns d_logits float64 [T, E].
    """
    l = np.asarray(logits, dtype=np.float32).astype(np.float64)
    T, E = l.shape
    k = topk_idx.shape[1]
    out = np.zeros((T, E))
    for c0 in range(0, T, chunk):
        lc = l[c0:c0 + chunk]
        n = lc.shape[0]
        if score_fn == SOFTMAX:
            ex = np.exp(lc - lc.max(axis=1, keepdims=True))
            sc = ex / ex.sum(axis=1, keepdims=True)
            js = np.einsum("te,ef->tef", sc, np.eye(E)) - np.einsum("te,tf->tef", sc, sc)
        else:
            sc = 1.0 / (1.0 + np.exp(-lc))
            js = np.einsum("te,ef->tef", sc * (1.0 - sc), np.eye(E))
        idx = topk_idx[c0:c0 + chunk].astype(np.int64)
        jv = np.take_along_axis(js, idx[:, :, None], axis=1)          # [n, k, E]
        if renorm:
            v = np.take_along_axis(sc, idx, axis=1)                  # [n, k]
            S = v.sum(axis=1)
            w = v / S[:, None]
            jr = (np.eye(k)[None] - w[:, :, None]) / S[:, None, None]   # [n, j, m]
            jw = np.einsum("tjm,tme->tje", jr, jv)
        else:
            jw = jv
        out[c0:c0 + n] = np.einsum("tje,tj->te", jw, d_topk_w[c0:c0 + chunk])
    return out


# ----------------------------------------------------------------------------
# permutation layout
# ----------------------------------------------------------------------------
def router_probs(logits: np.ndarray, score_fn: int) -> np.ndarray:
    """Per-token expert probabilities for the load-balancing loss: the softmax
    over all E, or (sigmoid scoring) the sigmoid scores divided by their sum
    over all E (DeepSeek-V3's normalised affinities)."""
    l = np.asarray(logits, dtype=np.float64)
    if score_fn == SOFTMAX:
        ex = np.exp(l - l.max(axis=1, keepdims=True))
        return ex / ex.sum(axis=1, keepdims=True)
    s = 1.0 / (1.0 + np.exp(-l))
    return s / s.sum(axis=1, keepdims=True)


def aux_loss(logits: np.ndarray, topk_idx: np.ndarray, E: int, score_fn: int, coeff: float):
    """Auxiliary load-balancing loss (TE-2912, Description: "optional auxiliary
    load-balancing loss"; the block returns it beside the output, sequence
    diagram).  The pages name the loss but not its form; this is the standard
    one (Switch Transformer; DeepSeek-V3's balance loss):

        loss = coeff * sum_e f_e * P_e,
        f_e  = E / (k T) * (number of (token, slot) choices of expert e),
        P_e  = mean over tokens of router_probs[:, e].

    Counts come from the routing decision (before any capacity drop).
    Returns (loss, counts int64 [E], P float64 [E]).
    """
    T, k = topk_idx.shape
    p = router_probs(logits, score_fn)
    counts = np.bincount(topk_idx.reshape(-1).astype(np.int64), minlength=E)[:E]
    f = E / (k * T) * counts if T > 0 else np.zeros(E)
    P = p.mean(axis=0) if T > 0 else np.zeros(E)
    return coeff * float((f * P).sum()), counts, P


def aux_loss_bwd(logits: np.ndarray, counts: np.ndarray, k: int, score_fn: int, coeff: float,
                 d_loss: float = 1.0) -> np.ndarray:
    """Gradient of aux_loss w.r.t. the router logits (counts fixed), by the
    chain rule with explicit Jacobians: dloss/dp[t, e] = coeff f_e / T, then
    each token's probability Jacobian dp_e / dl_e' (softmax: p_e (delta_ee' -
    p_e'); normalised sigmoid p = s / S: (delta_ee' - p_e) s_e' (1 - s_e') / S).
    Returns float64 [T, E]."""
    l = np.asarray(logits, dtype=np.float64)
    T, E = l.shape
    if T == 0:
        return np.zeros((0, E))
    f = E / (k * T) * np.asarray(counts, dtype=np.float64)
    g = d_loss * coeff * f / T                        # dloss / dp[t, e], same for every t
    out = np.zeros((T, E))
    for t in range(T):
        if score_fn == SOFTMAX:
            p = router_probs(l[t:t + 1], SOFTMAX)[0]
            jac = np.diag(p) - np.outer(p, p)          # jac[e, e'] = dp_e / dl_e'
        else:
            s = 1.0 / (1.0 + np.exp(-l[t]))
            S = s.sum()
            p = s / S
            ds = s * (1.0 - s)                         # ds_e' / dl_e'
            # dp_e / dl_e' = (delta_ee' - p_e) ds_e' / S
            jac = (np.eye(E) - p[:, None]) * (ds / S)[None, :]
        out[t] = g @ jac
    return out


def rows_cap(T: int, E: int, k: int, align: int) -> int:
    """Worst-case permuted rows, T*k + E*(align-1): TE-2912, review thread on
    ``recv_buffer_rows`` ("align_size > 0 + EP are combined")."""
    return T * k + E * (align - 1 if align > 1 else 0)


def permute_layout(topk_idx: np.ndarray, E: int, align: int = 0, capacity: int = 0):
    """Group the flattened (token, slot) assignments by expert.

    TE-2912, review thread on ``_combine_bwd`` (pure-JAX path): the flat
    assignment a = t*k + j is sorted by its expert with an argsort
    (``sorted_indices``); being stable, equal experts keep token order.
    ``group_sizes`` are the aligned counts when align_size > 0 (TE-2912,
    ``recv_buffer_rows`` thread).  Capacity dropping ("token-dropping",
    MaxText PR #2319 "[Draft] Integrate TE/JAX GroupedGEMM for MoE", Tests)
    keeps the first C assignments of each expert in that order.

    Returns a dict with group_sizes, kept_counts, group_offsets [E+1] (int64),
    sorted_to_flat [R] (-1 on padding rows), flat_to_sorted [T*k] (-1 when
    dropped), and R.
    """
    topk_idx = np.asarray(topk_idx)
    T, k = topk_idx.shape
    flat = topk_idx.reshape(-1).astype(np.int64)
    assert ((flat >= 0) & (flat < E)).all()
    sorted_indices = np.argsort(flat, kind="stable")
    counts = np.bincount(flat, minlength=E)
    kept = np.minimum(counts, capacity) if capacity > 0 else counts.copy()
    a = align if align > 1 else 1
    group_sizes = (kept + a - 1) // a * a
    group_offsets = np.concatenate([[0], np.cumsum(group_sizes)]).astype(np.int64)
    R = int(group_offsets[-1])
    run_start = np.concatenate([[0], np.cumsum(counts)])
    sorted_to_flat = np.full(R, -1, dtype=np.int64)
    flat_to_sorted = np.full(T * k, -1, dtype=np.int64)
    for e in range(E):
        run = sorted_indices[run_start[e]:run_start[e + 1]]
        keep = run[:kept[e]]
        pos = group_offsets[e] + np.arange(kept[e])
        sorted_to_flat[pos] = keep
        flat_to_sorted[keep] = pos
    return dict(group_sizes=group_sizes.astype(np.int64), kept_counts=kept.astype(np.int64),
                group_offsets=group_offsets, sorted_to_flat=sorted_to_flat,
                flat_to_sorted=flat_to_sorted, R=R, sorted_indices=sorted_indices)


def permute_rows(x: np.ndarray, layout: dict, k: int) -> np.ndarray:
    """sorted_x: row p holds x[t] for the assignment a = sorted_to_flat[p] (t = a // k);
    padding rows are zero."""
    s2f = layout["sorted_to_flat"]
    xs = np.zeros((layout["R"], x.shape[1]), dtype=np.float64)
    valid = s2f >= 0
    xs[valid] = x[s2f[valid] // k]
    return xs


# ----------------------------------------------------------------------------
# expert FFN (grouped GEMMs)
# ----------------------------------------------------------------------------
def sigmoid(z):
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-z))


def silu(z):
    return z * sigmoid(z)


def swiglu(h: np.ndarray):
    """act = silu(gate) * up, with [gate | up] = x [wi_0 | wi_1] (TE-2912, commit
    fusing wi_0/wi_1 into one grouped GEMM whose output is sliced into
    gate_proj_out and up_proj_out; the SwiGLU FFN of the Description)."""
    f = h.shape[1] // 2
    return silu(h[:, :f]) * h[:, f:]


def swiglu_bwd(h: np.ndarray, d_act: np.ndarray):
    """Gradient of act = silu(g) * u w.r.t. [g | u]:
    d_g = d_act * u * s * (1 + g (1 - s)),  d_u = d_act * silu(g),  s = sigmoid(g)."""
    f = h.shape[1] // 2
    g, u = h[:, :f], h[:, f:]
    s = sigmoid(g)
    dg = d_act * u * s * (1.0 + g * (1.0 - s))
    du = d_act * g * s
    return np.concatenate([dg, du], axis=1)


def gmm(lhs: np.ndarray, rhs: np.ndarray, group_offsets, transpose_rhs: bool = False,
        partial_sum: np.ndarray | None = None):
    """Grouped matmul: rows [off_e, off_e+1) of lhs times rhs[e].

    MT-4295, review thread on the gmm kernel: ``partial_sum`` is added to the
    product in place (its rows may be fewer than lhs's padded M; rows beyond
    it are not produced); ``transpose_rhs`` multiplies by rhs[e]^T (the dgrad
    form).  Rows outside every group are left zero.
    """
    E = rhs.shape[0]
    n = rhs.shape[1] if transpose_rhs else rhs.shape[2]
    out = np.zeros((lhs.shape[0], n), dtype=np.float64)
    for e in range(E):
        s, t = int(group_offsets[e]), int(group_offsets[e + 1])
        if t > s:
            w = rhs[e].T if transpose_rhs else rhs[e]
            out[s:t] = lhs[s:t] @ w
    if partial_sum is not None:
        out[: partial_sum.shape[0]] += partial_sum
    return out


def tgmm(lhs: np.ndarray, rhs: np.ndarray, group_offsets, E: int,
         partial_sum: np.ndarray | None = None):
    """Weight-gradient grouped matmul: out[e] = lhs[g_e]^T rhs[g_e].

    MT-4295, Testing ("TGMM with zero-initialized empty expert groups"): an
    expert with no rows gets exactly zero, or its partial sum unchanged.
    """
    out = np.zeros((E, lhs.shape[1], rhs.shape[1]), dtype=np.float64)
    for e in range(E):
        s, t = int(group_offsets[e]), int(group_offsets[e + 1])
        if t > s:
            out[e] = lhs[s:t].T @ rhs[s:t]
    if partial_sum is not None:
        out += partial_sum
    return out


# ----------------------------------------------------------------------------
# combine and its backward
# ----------------------------------------------------------------------------
def combine(y: np.ndarray, flat_to_sorted: np.ndarray, topk_w: np.ndarray):
    """output[t] = sum_j w[t,j] * y[flat_to_sorted[t,j]] over kept slots.

    TE-2912, review thread on ``_combine_bwd``: un-sort the expert outputs
    with argsort(sorted_indices), strip padding, then the einsum
    output[B,E] = sum_K intermediate[B,K,E] * weights[B,K].  Here the unsort
    is the gather by flat_to_sorted and padding rows are never gathered.
    """
    T, k = topk_w.shape
    out = np.zeros((T, y.shape[1]), dtype=np.float64)
    f2s = flat_to_sorted.reshape(T, k)
    for j in range(k):
        p = f2s[:, j]
        ok = p >= 0
        out[ok] += topk_w[ok, j][:, None] * y[p[ok]]
    return out


def combine_bwd(d_out: np.ndarray, y: np.ndarray, flat_to_sorted: np.ndarray,
                topk_w: np.ndarray, R: int):
    """Backward of :func:`combine` (TE-2912, ``_combine_bwd`` thread):
    d_intermediate[B,K,E] = d_output[B,E] * w[B,K];
    d_w[B,K] = sum_E d_output[B,E] * intermediate[B,K,E];
    padding rows receive zero, then the gather by sorted order places each
    d_intermediate row at its sorted position.  Dropped slots get d_w = 0.
    """
    T, k = topk_w.shape
    dy = np.zeros((R, d_out.shape[1]), dtype=np.float64)
    dw = np.zeros((T, k), dtype=np.float64)
    f2s = flat_to_sorted.reshape(T, k)
    for j in range(k):
        p = f2s[:, j]
        ok = p >= 0
        dy[p[ok]] = topk_w[ok, j][:, None] * d_out[ok]
        dw[ok, j] = np.einsum("td,td->t", d_out[ok], y[p[ok]])
    return dy, dw


def dispatch_bwd(d_xs: np.ndarray, flat_to_sorted: np.ndarray, T: int, k: int):
    """Backward of the permutation (TE-2912, sequence diagram: ``_dispatch_bwd``
    returns d_inputs_2d): every token sums the gradients of its kept rows."""
    dx = np.zeros((T, d_xs.shape[1]), dtype=np.float64)
    f2s = flat_to_sorted.reshape(T, k)
    for j in range(k):
        p = f2s[:, j]
        ok = p >= 0
        dx[ok] += d_xs[p[ok]]
    return dx


# ----------------------------------------------------------------------------
# whole layer
# ----------------------------------------------------------------------------
def add_group_bias(m: np.ndarray, bias, group_offsets):
    """Adds bias[e] to every row of group e (padding rows included).

    MLP biases of the expert FFN: MaxText PR #4295, Testing (chunked GMM with
    ``mlp_bias=True``); TE-2912, the ``has_wi_bias`` static info of the body
    residuals."""
    if bias is None:
        return m
    out = m.copy()
    for e in range(bias.shape[0]):
        s, t = int(group_offsets[e]), int(group_offsets[e + 1])
        out[s:t] += bias[e][None, :]
    return out


def group_colsum(g: np.ndarray, group_offsets, E: int):
    """Per-expert column sums: out[e] = sum of rows [off_e, off_e+1) of g (the
    gradient of a bias that every row of the group received)."""
    out = np.zeros((E, g.shape[1]))
    for e in range(E):
        s, t = int(group_offsets[e]), int(group_offsets[e + 1])
        out[e] = g[s:t].sum(axis=0)
    return out


def forward(x, logits, wi, wo, k, score_fn, renorm, align=0, capacity=0, num_chunks=1,
            bi=None, bo=None, num_groups=0, topk_group=0, expert_bias=None):
    """The layer's forward pass (TE-2912, sequence diagram of ``_moe_fwd_rule``
    without the expert-parallel all-to-all).

    x [T,d], wi [E,d,2f], wo [E,f,d] as float64 arrays; logits fp32 [T,E].
    With num_chunks > 1 the up-projection is accumulated chunk by chunk along
    d_model into an fp32-style partial sum P (MT-4295, Description: each
    chunk's gmm adds into the partial sum in place), then SwiGLU runs on P.
    Optional MLP biases bi [E, 2f] (added to [gate | up]) and bo [E, d];
    optional group-limited routing (num_groups, topk_group) and selection
    bias (expert_bias), both as in route_topk.
    Returns a dict of every intermediate the backward needs.
    """
    T, d = x.shape
    E = wi.shape[0]
    topk_idx, topk_w = route_topk(logits, k, score_fn, renorm, expert_bias=expert_bias,
                                  num_groups=num_groups, topk_group=topk_group)
    lay = permute_layout(topk_idx, E, align, capacity)
    xs = permute_rows(x, lay, k)
    off = lay["group_offsets"]
    if num_chunks <= 1:
        h = gmm(xs, wi, off)
    else:
        assert d % num_chunks == 0
        dc = d // num_chunks
        p = None
        for c in range(num_chunks):
            sl = slice(c * dc, (c + 1) * dc)
            p = gmm(xs[:, sl], wi[:, sl, :], off, partial_sum=p)
        h = p
    h = add_group_bias(h, bi, off)
    act = swiglu(h)
    y = add_group_bias(gmm(act, wo, off), bo, off)
    out = combine(y, lay["flat_to_sorted"], topk_w)
    return dict(topk_idx=topk_idx, topk_w=topk_w, layout=lay, xs=xs, h=h, act=act, y=y,
                out=out)


def backward(fw: dict, d_out, wi, wo, k, num_chunks=1):
    """The layer's backward pass (TE-2912, sequence diagram of ``_moe_bwd_rule``):
    combine bwd -> FFN bwd (dgrad with transposed weights and tgmm weight
    gradients, fused over [wi_0 | wi_1]) -> dispatch bwd.

    With num_chunks > 1 the partial sum's cotangent is the upstream gradient
    itself (MT-4295, review thread on the gmm backward returning ``grad`` for
    ``partial_sum``), so every chunk's dgrad and tgmm see the same dH, each on
    its own slice of d_model.
    """
    lay = fw["layout"]
    off = lay["group_offsets"]
    E = wi.shape[0]
    T = d_out.shape[0]
    dy, d_topk_w = combine_bwd(d_out, fw["y"], lay["flat_to_sorted"], fw["topk_w"], lay["R"])
    d_act = gmm(dy, wo, off, transpose_rhs=True)
    dh = swiglu_bwd(fw["h"], d_act)
    d_wo = tgmm(fw["act"], dy, off, E)
    if num_chunks <= 1:
        d_xs = gmm(dh, wi, off, transpose_rhs=True)
        d_wi = tgmm(fw["xs"], dh, off, E)
    else:
        d = wi.shape[1]
        dc = d // num_chunks
        d_xs = np.zeros((lay["R"], d))
        d_wi = np.zeros_like(wi, dtype=np.float64)
        for c in range(num_chunks):
            sl = slice(c * dc, (c + 1) * dc)
            d_xs[:, sl] = gmm(dh, wi[:, sl, :], off, transpose_rhs=True)
            d_wi[:, sl, :] = tgmm(fw["xs"][:, sl], dh, off, E)
    dx = dispatch_bwd(d_xs, lay["flat_to_sorted"], T, k)
    return dict(dy=dy, d_topk_w=d_topk_w, d_act=d_act, dh=dh, d_wo=d_wo, d_xs=d_xs,
                d_wi=d_wi, dx=dx, d_bi=group_colsum(dh, off, E), d_bo=group_colsum(dy, off, E))


def flops_fwd_bwd(m_kept: int, d: int, f: int) -> int:
    """Algorithmic FLOPs of the three expert GEMMs, forward and backward:
    up (2*M*d*2f) + down (2*M*f*d) forward, twice that backward = 18*M*d*f."""
    return 18 * m_kept * d * f
