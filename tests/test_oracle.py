"""Pins of the fp64 oracle against things other than itself (CPU only).

* hand-worked golden fixtures (tests/golden/*.json, each derivation written out);
* the dense one-hot brute force of tests/brute_force.py (all experts on all
  tokens, masked), with gradients from PyTorch autograd;
* closed forms and library routines (scipy softmax / expit; E=1, k=1 is a
  plain SwiGLU MLP);
* invariants of the permutation layout;
* central finite differences of L = <dOut, out>;
* planted mistakes in the oracle that these pins must catch.
"""
import json
import os
import zlib

import numpy as np
import pytest
import scipy.special
import torch

import brute_force as bf
from oracle import moe_ref as ref

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_layer(seed, T, d, f, E, dist_logits="normal"):
    rng = np.random.default_rng(seed)
    if dist_logits == "normal":
        logits = rng.standard_normal((T, E)).astype(np.float32)
    elif dist_logits == "ties":
        logits = rng.integers(-2, 3, size=(T, E)).astype(np.float32)
    else:
        logits = np.zeros((T, E), np.float32)
    x = rng.standard_normal((T, d))
    wi = rng.standard_normal((E, d, 2 * f)) * 0.3
    wo = rng.standard_normal((E, f, d)) * 0.3
    dout = rng.standard_normal((T, d))
    return logits, x, wi, wo, dout


# ---------------------------------------------------------------------------
# golden fixtures
# ---------------------------------------------------------------------------
def test_golden_route_permute_hand():
    g = json.load(open(os.path.join(GOLDEN, "route_permute_hand.json")))
    logits = np.array(g["logits"], np.float32)
    idx, w = ref.route_topk(logits, g["k"], g["score_fn"], g["renorm"])
    assert idx.tolist() == g["topk_idx"]
    np.testing.assert_allclose(w, np.array(g["topk_w"]), rtol=0, atol=1e-15)
    lay = ref.permute_layout(idx, g["E"], g["align"], g["capacity"])
    assert lay["kept_counts"].tolist() == g["kept_counts"]
    assert lay["group_sizes"].tolist() == g["group_sizes"]
    assert lay["group_offsets"].tolist() == g["group_offsets"]
    assert lay["R"] == g["R"]
    assert lay["sorted_to_flat"].tolist() == g["sorted_to_flat"]
    assert lay["flat_to_sorted"].tolist() == g["flat_to_sorted"]
    assert ref.rows_cap(g["T"], g["E"], g["k"], g["align"]) == g["rows_cap"]


def test_golden_swiglu_scalar_hand():
    g = json.load(open(os.path.join(GOLDEN, "swiglu_scalar_hand.json")))
    x = np.array([[g["x"]]])
    wi = np.array([[[g["wi_0"], g["wi_1"]]]])
    wo = np.array([[[g["wo"]]]])
    logits = np.zeros((1, 1), np.float32)
    fw = ref.forward(x, logits, wi, wo, k=1, score_fn=0, renorm=1)
    bw = ref.backward(fw, np.array([[g["dout"]]]), wi, wo, k=1)
    assert fw["out"][0, 0] == pytest.approx(g["y"], rel=1e-15)
    assert bw["dx"][0, 0] == pytest.approx(g["dx"], rel=1e-14)
    assert bw["d_wi"][0, 0, 0] == pytest.approx(g["d_wi_0"], rel=1e-14)
    assert bw["d_wi"][0, 0, 1] == pytest.approx(g["d_wi_1"], rel=1e-14)
    assert bw["d_wo"][0, 0, 0] == pytest.approx(g["d_wo"], rel=1e-14)


# ---------------------------------------------------------------------------
# brute force
# ---------------------------------------------------------------------------
BRUTE_CASES = [
    # T, d, f, E, k, score_fn, renorm, align, capacity, logits
    (13, 6, 5, 5, 2, 0, 1, 0, 0, "normal"),
    (17, 4, 3, 6, 3, 1, 1, 0, 0, "normal"),
    (20, 5, 4, 4, 1, 0, 0, 4, 3, "normal"),
    (24, 3, 2, 5, 2, 0, 1, 3, 4, "ties"),
    (9, 4, 3, 7, 3, 1, 0, 2, 0, "ties"),
    (8, 3, 2, 4, 2, 0, 1, 0, 2, "equal"),
]


@pytest.mark.parametrize("case", BRUTE_CASES)
def test_oracle_vs_brute_force(case):
    T, d, f, E, k, sfn, ren, align, cap, dist = case
    logits, x, wi, wo, dout = _rand_layer(zlib.crc32(repr(case).encode()) % 1000, T, d, f, E, dist)
    b = bf.layer_dense(x, logits, wi, wo, dout, k, sfn, ren, cap)
    fw = ref.forward(x, logits, wi, wo, k, sfn, ren, align, cap)
    bw = ref.backward(fw, dout, wi, wo, k)
    idx, w = fw["topk_idx"], fw["topk_w"]
    # routing
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            assert b["sel"][t, e] and b["slot"][t, e] == j
            assert w[t, j] == pytest.approx(b["weight"][t, e], rel=1e-13, abs=1e-15)
    # layout
    pos, sizes, R = bf.layout_dense(b["sel"], b["kept"], align)
    lay = fw["layout"]
    assert lay["R"] == R
    assert lay["group_sizes"].tolist() == sizes.tolist()
    f2s = lay["flat_to_sorted"].reshape(T, k)
    for t in range(T):
        for j in range(k):
            assert f2s[t, j] == pos[t, idx[t, j]]
    # forward output and gradients
    np.testing.assert_allclose(fw["out"], b["out"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(bw["dx"], b["dx"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(bw["d_wi"], b["dwi"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(bw["d_wo"], b["dwo"], rtol=1e-11, atol=1e-12)
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            want = b["dgate"][t, e] if b["kept"][t, e] else 0.0
            assert bw["d_topk_w"][t, j] == pytest.approx(want, rel=1e-11, abs=1e-12)


# ---------------------------------------------------------------------------
# closed forms and library routines
# ---------------------------------------------------------------------------
def test_softmax_renorm_is_softmax_of_selected_logits():
    rng = np.random.default_rng(3)
    logits = rng.standard_normal((50, 16)).astype(np.float32)
    idx, w = ref.route_topk(logits, 4, ref.SOFTMAX, 1)
    sel = np.take_along_axis(logits.astype(np.float64), idx.astype(np.int64), 1)
    np.testing.assert_allclose(w, scipy.special.softmax(sel, axis=1), rtol=1e-14)
    # without renorm: the full-E softmax probabilities of the selected experts
    idx2, w2 = ref.route_topk(logits, 4, ref.SOFTMAX, 0)
    full = scipy.special.softmax(logits.astype(np.float64), axis=1)
    np.testing.assert_allclose(w2, np.take_along_axis(full, idx2.astype(np.int64), 1), rtol=1e-14)
    # the selected experts are the k largest: numpy's argsort on the negated logits
    ref_idx = np.argsort(-logits.astype(np.float64), axis=1, kind="stable")[:, :4]
    assert (idx == ref_idx).all()


def test_sigmoid_scores_are_expit():
    rng = np.random.default_rng(4)
    logits = rng.standard_normal((40, 32)).astype(np.float32)
    idx, w = ref.route_topk(logits, 8, ref.SIGMOID, 0)
    s = scipy.special.expit(logits.astype(np.float64))
    np.testing.assert_allclose(w, np.take_along_axis(s, idx.astype(np.int64), 1), rtol=1e-14)
    idx_r, w_r = ref.route_topk(logits, 8, ref.SIGMOID, 1)
    np.testing.assert_allclose(w_r.sum(1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(w_r, w / w.sum(1, keepdims=True), rtol=1e-14)


def test_single_expert_top1_is_dense_swiglu_mlp():
    rng = np.random.default_rng(5)
    T, d, f = 33, 12, 10
    x = rng.standard_normal((T, d))
    wi = rng.standard_normal((1, d, 2 * f))
    wo = rng.standard_normal((1, f, d))
    logits = rng.standard_normal((T, 1)).astype(np.float32)
    fw = ref.forward(x, logits, wi, wo, k=1, score_fn=0, renorm=1)
    g = np.matmul(x, wi[0, :, :f])
    u = np.matmul(x, wi[0, :, f:])
    dense = np.matmul(g * scipy.special.expit(g) * u, wo[0])
    np.testing.assert_allclose(fw["out"], dense, rtol=1e-13, atol=1e-13)
    assert (fw["topk_w"] == 1.0).all()


def test_all_equal_logits_pick_lowest_ids():
    idx, _ = ref.route_topk(np.zeros((7, 9), np.float32), 4, ref.SOFTMAX, 1)
    assert (idx == np.arange(4)).all()


# ---------------------------------------------------------------------------
# invariants of the layout
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("align,cap", [(0, 0), (1, 0), (8, 0), (8, 100), (128, 40), (0, 37)])
def test_layout_invariants(align, cap):
    rng = np.random.default_rng(align * 1000 + cap)
    T, E, k = 500, 16, 4
    logits = rng.standard_normal((T, E)).astype(np.float32) + np.linspace(0, 3, E).astype(np.float32)
    idx, _ = ref.route_topk(logits, k, 0, 1)
    lay = ref.permute_layout(idx, E, align, cap)
    counts = np.bincount(idx.reshape(-1), minlength=E)
    kept = lay["kept_counts"]
    dropped = (counts - kept).sum()
    assert kept.sum() == T * k - dropped
    if cap > 0:
        assert (kept == np.minimum(counts, cap)).all()
    else:
        assert dropped == 0
    a = max(align, 1)
    assert (lay["group_sizes"] % a == 0).all()
    assert (lay["group_sizes"] >= kept).all() and (lay["group_sizes"] - kept < a).all()
    assert lay["R"] <= ref.rows_cap(T, E, k, align)
    s2f, f2s = lay["sorted_to_flat"], lay["flat_to_sorted"]
    assert (f2s >= 0).sum() == kept.sum() and (s2f >= 0).sum() == kept.sum()
    ok = s2f >= 0
    assert (f2s[s2f[ok]] == np.nonzero(ok)[0]).all()
    off = lay["group_offsets"]
    for e in range(E):
        rows = s2f[off[e]:off[e + 1]]
        real = rows[rows >= 0]
        assert len(real) == kept[e]
        assert (rows[:kept[e]] >= 0).all() and (rows[kept[e]:] == -1).all()
        toks = real // k
        assert (np.diff(toks) > 0).all()
        assert (idx.reshape(-1)[real] == e).all()
    # dropped assignments are the latest tokens of their expert
    if cap > 0:
        for a_ in np.nonzero(f2s < 0)[0]:
            e = idx.reshape(-1)[a_]
            kept_toks = s2f[off[e]:off[e] + kept[e]] // k
            assert a_ // k > kept_toks.max()
    xs = ref.permute_rows(rng.standard_normal((T, 3)), lay, k)
    assert (xs[~ok] == 0).all()


# ---------------------------------------------------------------------------
# combine identities and gmm / tgmm semantics
# ---------------------------------------------------------------------------
def test_combine_bwd_identity():
    logits, x, wi, wo, dout = _rand_layer(11, 40, 8, 6, 6)
    fw = ref.forward(x, logits, wi, wo, 3, 1, 1, align=4, capacity=15)
    bw = ref.backward(fw, dout, wi, wo, 3)
    lhs = (fw["topk_w"] * bw["d_topk_w"]).sum()
    rhs = (dout * fw["out"]).sum()
    assert lhs == pytest.approx(rhs, rel=1e-12)
    assert (bw["dy"][fw["layout"]["sorted_to_flat"] < 0] == 0).all()


def test_tgmm_empty_group_exact_zero_and_partial_sum():
    rng = np.random.default_rng(12)
    off = np.array([0, 5, 5, 9, 9])
    a = rng.standard_normal((9, 3))
    b = rng.standard_normal((9, 4))
    out = ref.tgmm(a, b, off, 4)
    assert (out[1] == 0).all() and (out[3] == 0).all()
    np.testing.assert_allclose(out[0], sum(np.outer(a[r], b[r]) for r in range(5)), rtol=1e-14)
    ps = rng.standard_normal((4, 3, 4))
    out2 = ref.tgmm(a, b, off, 4, partial_sum=ps)
    assert (out2[1] == ps[1]).all() and (out2[3] == ps[3]).all()
    np.testing.assert_allclose(out2[2], ps[2] + a[5:9].T @ b[5:9], rtol=1e-14)


def test_gmm_partial_sum_and_transpose():
    rng = np.random.default_rng(13)
    off = np.array([0, 3, 3, 7])
    a = rng.standard_normal((7, 5))
    w = rng.standard_normal((3, 5, 6))
    ps = rng.standard_normal((7, 6))
    base = ref.gmm(a, w, off)
    np.testing.assert_allclose(ref.gmm(a, w, off, partial_sum=ps), base + ps, rtol=1e-14)
    wt = np.ascontiguousarray(np.swapaxes(w, 1, 2))
    np.testing.assert_allclose(ref.gmm(a, wt, off, transpose_rhs=True), base, rtol=1e-14)
    for r in range(7):
        e = 0 if r < 3 else 2
        np.testing.assert_allclose(base[r], a[r] @ w[e], rtol=1e-14)


def test_chunked_equals_unchunked():
    logits, x, wi, wo, dout = _rand_layer(14, 30, 16, 6, 5)
    f1 = ref.forward(x, logits, wi, wo, 2, 0, 1)
    b1 = ref.backward(f1, dout, wi, wo, 2)
    f1c = ref.forward(x, logits, wi, wo, 2, 0, 1, num_chunks=1)
    np.testing.assert_array_equal(f1["out"], f1c["out"])
    f4 = ref.forward(x, logits, wi, wo, 2, 0, 1, num_chunks=4)
    b4 = ref.backward(f4, dout, wi, wo, 2, num_chunks=4)
    np.testing.assert_allclose(f4["out"], f1["out"], rtol=1e-12, atol=1e-12)
    for key in ("dx", "d_wi", "d_wo", "d_topk_w"):
        np.testing.assert_allclose(b4[key], b1[key], rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# finite differences
# ---------------------------------------------------------------------------
def _fd_check(seed=21, T=25, d=7, f=5, E=5, k=2, sfn=0, ren=1, align=2, cap=9, chunks=1):
    logits, x, wi, wo, dout = _rand_layer(seed, T, d, f, E)
    fw = ref.forward(x, logits, wi, wo, k, sfn, ren, align, cap, chunks)
    bw = ref.backward(fw, dout, wi, wo, k, chunks)
    rng = np.random.default_rng(seed + 1)
    eps = 1e-6
    errs = {}

    def loss(x_, wi_, wo_, w_):
        lay = fw["layout"]
        xs = ref.permute_rows(x_, lay, k)
        h = ref.gmm(xs, wi_, lay["group_offsets"])
        y = ref.gmm(ref.swiglu(h), wo_, lay["group_offsets"])
        return (dout * ref.combine(y, lay["flat_to_sorted"], w_)).sum()

    base = (x, wi, wo, fw["topk_w"])
    grads = (bw["dx"], bw["d_wi"], bw["d_wo"], bw["d_topk_w"])
    for i, name in enumerate(("x", "wi", "wo", "w")):
        v = rng.standard_normal(base[i].shape)
        plus = list(base)
        minus = list(base)
        plus[i] = base[i] + eps * v
        minus[i] = base[i] - eps * v
        fd = (loss(*plus) - loss(*minus)) / (2 * eps)
        an = (grads[i] * v).sum()
        errs[name] = abs(fd - an) / max(abs(an), 1e-30)
    return errs


@pytest.mark.parametrize("kw", [dict(), dict(sfn=1, k=3, cap=0, align=0),
                                dict(k=1, ren=0, align=4, cap=6), dict(chunks=7, d=14)])
def test_finite_differences(kw):
    errs = _fd_check(**kw)
    for name, e in errs.items():
        assert e < 1e-6, (name, e)


# ---------------------------------------------------------------------------
# planted mistakes: each must be caught by one of the pins above
# ---------------------------------------------------------------------------
def _mut_swiglu_bwd_drop_term(h, d_act):
    f = h.shape[1] // 2
    g, u = h[:, :f], h[:, f:]
    s = ref.sigmoid(g)
    return np.concatenate([d_act * u * s, d_act * g * s], axis=1)     # dropped (1 + g(1-s))


def _mut_route_tie_high_id(logits, k, score_fn, renorm):
    idx, w = ORIG_ROUTE(logits[:, ::-1].copy(), k, score_fn, renorm)
    return (logits.shape[1] - 1 - idx).astype(np.int32), w


def _mut_combine_bwd_transposed(d_out, y, f2s, w, R):
    dy, dw = ORIG_CBWD(d_out, y, f2s, w, R)
    return dy, dw[:, ::-1].copy()


ORIG_ROUTE = ref.route_topk
ORIG_CBWD = ref.combine_bwd


@pytest.mark.parametrize("mutant", ["swiglu_bwd", "route_tie", "combine_bwd"])
def test_planted_mistakes_are_caught(monkeypatch, mutant):
    if mutant == "swiglu_bwd":
        monkeypatch.setattr(ref, "swiglu_bwd", _mut_swiglu_bwd_drop_term)
        errs = _fd_check()
        assert max(errs.values()) > 1e-3
    elif mutant == "route_tie":
        monkeypatch.setattr(ref, "route_topk", _mut_route_tie_high_id)
        with pytest.raises(AssertionError):
            test_golden_route_permute_hand()
    else:
        monkeypatch.setattr(ref, "combine_bwd", _mut_combine_bwd_transposed)
        errs = _fd_check()
        assert errs["w"] > 1e-3


# ---------------------------------------------------------------------------
# routing backward and expert bias
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("sfn,ren,k", [(0, 1, 2), (0, 0, 3), (1, 1, 8), (1, 0, 1), (0, 1, 1)])
def test_route_bwd_vs_autograd_and_fd(sfn, ren, k):
    rng = np.random.default_rng(31 + 7 * sfn + ren + k)
    T, E = 40, 12
    logits = rng.standard_normal((T, E)).astype(np.float32)
    idx, w = ref.route_topk(logits, k, sfn, ren)
    dw = rng.standard_normal((T, k))
    got = ref.route_topk_bwd(logits, idx, dw, sfn, ren)
    sel = np.zeros((T, E), bool)
    d_gate = np.zeros((T, E))
    for t in range(T):
        sel[t, idx[t]] = True
        d_gate[t, idx[t]] = dw[t]
    want = bf.route_bwd_dense_torch(logits, sel, d_gate, sfn, ren)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-14)

    # central differences of L(l) = <dw, w(l)> with the selection held fixed
    def weights(lg):
        if sfn == 0:
            ex = np.exp(lg - lg.max(1, keepdims=True))
            sc = ex / ex.sum(1, keepdims=True)
        else:
            sc = 1 / (1 + np.exp(-lg))
        v = np.take_along_axis(sc, idx.astype(np.int64), 1)
        return v / v.sum(1, keepdims=True) if ren else v
    l64 = logits.astype(np.float64)
    np.testing.assert_allclose(weights(l64), w, rtol=1e-14)
    v = rng.standard_normal(l64.shape)
    eps = 1e-6
    fd = ((dw * weights(l64 + eps * v)).sum() - (dw * weights(l64 - eps * v)).sum()) / (2 * eps)
    assert fd == pytest.approx((got * v).sum(), rel=1e-7, abs=1e-12)


def test_route_bwd_closed_forms():
    rng = np.random.default_rng(41)
    logits = rng.standard_normal((25, 6)).astype(np.float32)
    # top-1 with renorm: the weight is identically 1, so the gradient is exactly 0
    idx, _ = ref.route_topk(logits, 1, 0, 1)
    assert (ref.route_topk_bwd(logits, idx, rng.standard_normal((25, 1)), 0, 1) == 0).all()
    # sigmoid without renorm: d_l = dw * s (1 - s) on the selected experts (scipy expit)
    idx, w = ref.route_topk(logits, 3, 1, 0)
    dw = rng.standard_normal((25, 3))
    got = ref.route_topk_bwd(logits, idx, dw, 1, 0)
    s = scipy.special.expit(logits.astype(np.float64))
    want = np.zeros_like(got)
    np.put_along_axis(want, idx.astype(np.int64),
                      dw * np.take_along_axis(s * (1 - s), idx.astype(np.int64), 1), 1)
    np.testing.assert_allclose(got, want, rtol=1e-13)
    # softmax (renormalised or over all E) is shift invariant: rows sum to 0
    for ren in (0, 1):
        idx, _ = ref.route_topk(logits, 3, 0, ren)
        g = ref.route_topk_bwd(logits, idx, rng.standard_normal((25, 3)), 0, ren)
        np.testing.assert_allclose(g.sum(1), 0, atol=1e-14)


def test_expert_bias_changes_selection_not_weights():
    rng = np.random.default_rng(43)
    logits = rng.standard_normal((60, 8)).astype(np.float32)
    bias = np.zeros(8, np.float32)
    bias[5] = 10.0           # expert 5 always selected first
    idx, w = ref.route_topk(logits, 2, 1, 0, expert_bias=bias)
    assert (idx[:, 0] == 5).all()
    s = scipy.special.expit(logits.astype(np.float64))
    np.testing.assert_allclose(w, np.take_along_axis(s, idx.astype(np.int64), 1), rtol=1e-14)
    # brute force: rank by logit + bias in fp32, ties to the lower id
    key = (logits + bias).astype(np.float32)
    for t in range(60):
        order = sorted(range(8), key=lambda e: (-float(key[t, e]), e))
        assert idx[t].tolist() == order[:2]
    # zero bias is the unbiased router
    i0, w0 = ref.route_topk(logits, 2, 1, 0, expert_bias=np.zeros(8, np.float32))
    i1, w1 = ref.route_topk(logits, 2, 1, 0)
    assert (i0 == i1).all() and (w0 == w1).all()


# ---------------------------------------------------------------------------
# MLP biases
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("case", [(14, 5, 4, 4, 2, 0, 1, 0, 0), (20, 4, 3, 5, 1, 0, 0, 4, 3),
                                  (16, 6, 4, 6, 3, 1, 1, 2, 0)])
def test_biases_vs_brute_force(case):
    T, d, f, E, k, sfn, ren, align, cap = case
    logits, x, wi, wo, dout = _rand_layer(zlib.crc32(repr(case).encode()) % 1000, T, d, f, E)
    rng = np.random.default_rng(77)
    bi = rng.standard_normal((E, 2 * f)) * 0.5
    bo = rng.standard_normal((E, d)) * 0.5
    b = bf.layer_dense(x, logits, wi, wo, dout, k, sfn, ren, cap, bi=bi, bo=bo)
    fw = ref.forward(x, logits, wi, wo, k, sfn, ren, align, cap, bi=bi, bo=bo)
    bw = ref.backward(fw, dout, wi, wo, k)
    np.testing.assert_allclose(fw["out"], b["out"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(bw["dx"], b["dx"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(bw["d_wi"], b["dwi"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(bw["d_wo"], b["dwo"], rtol=1e-11, atol=1e-12)
    # bias gradients: only kept assignments reach the output
    np.testing.assert_allclose(bw["d_bi"], b["dbi"], rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(bw["d_bo"], b["dbo"], rtol=1e-11, atol=1e-12)


def test_bias_free_layer_is_zero_bias_layer():
    logits, x, wi, wo, dout = _rand_layer(5, 12, 4, 3, 3)
    f0 = ref.forward(x, logits, wi, wo, 2, 0, 1, bi=np.zeros((3, 6)), bo=np.zeros((3, 4)))
    f1 = ref.forward(x, logits, wi, wo, 2, 0, 1)
    np.testing.assert_array_equal(f0["out"], f1["out"])


def test_group_colsum_closed_form():
    g = np.arange(30, dtype=np.float64).reshape(10, 3)
    off = np.array([0, 4, 4, 10])
    out = ref.group_colsum(g, off, 3)
    np.testing.assert_array_equal(out[0], g[:4].sum(0))
    np.testing.assert_array_equal(out[1], 0)
    np.testing.assert_array_equal(out[2], [sum(3 * r + c for r in range(4, 10)) for c in range(3)])


# ---------------------------------------------------------------------------
# group-limited routing
# ---------------------------------------------------------------------------
def test_golden_group_limited_hand():
    g = json.load(open(os.path.join(GOLDEN, "route_group_limited_hand.json")))
    for c in g["cases"]:
        lg = np.array(c["logits"], np.float32)
        bias = None if c["expert_bias"] is None else np.array(c["expert_bias"], np.float32)
        idx, w = ref.route_topk(lg, c["k"], c["score_fn"], c["renorm"], expert_bias=bias,
                                num_groups=c["num_groups"], topk_group=c["topk_group"])
        assert idx.tolist() == c["topk_idx"], c["name"]
        np.testing.assert_allclose(w, c["topk_w"], rtol=1e-13, atol=0)


@pytest.mark.parametrize("E,G,k", [(8, 4, 2), (64, 8, 6), (256, 8, 8)])
def test_group_limited_with_every_group_open_is_plain_topk(E, G, k):
    rng = np.random.default_rng(E + k)
    lg = rng.standard_normal((200, E)).astype(np.float32)
    for sfn in (0, 1):
        a = ref.route_topk(lg, k, sfn, 1)
        b = ref.route_topk(lg, k, sfn, 1, num_groups=G, topk_group=G if k % G == 0 else 1)
        if k % G == 0:
            assert (a[0] == b[0]).all()
            np.testing.assert_array_equal(a[1], b[1])
    # one group holding all experts
    c = ref.route_topk(lg, k, 0, 1, num_groups=1, topk_group=1)
    assert (c[0] == ref.route_topk(lg, k, 0, 1)[0]).all()


def _group_scores_by_hand(keys, G, m):
    """Python-list restatement: per group, sort the keys descending and add the
    first m in fp32 one by one."""
    gs = len(keys) // G
    out = []
    for g in range(G):
        vals = sorted((float(v) for v in keys[g * gs:(g + 1) * gs]), reverse=True)
        acc = np.float32(vals[0])
        for v in vals[1:m]:
            acc = np.float32(acc + np.float32(v))
        out.append(float(acc))
    return out


@pytest.mark.parametrize("E,G,tg,k,ties", [(64, 8, 3, 6, False), (256, 8, 4, 8, False),
                                          (32, 4, 2, 4, True), (16, 16, 4, 4, True)])
def test_group_limited_properties(E, G, tg, k, ties):
    rng = np.random.default_rng(E * 3 + k)
    T = 300
    if ties:
        lg = rng.integers(-2, 3, size=(T, E)).astype(np.float32)
    else:
        lg = rng.standard_normal((T, E)).astype(np.float32)
    bias = (rng.standard_normal(E) * 0.5).astype(np.float32)
    idx, _ = ref.route_topk(lg, k, 1, 1, expert_bias=bias, num_groups=G, topk_group=tg)
    key = (lg + bias[None, :]).astype(np.float32)
    gs, m = E // G, k // tg
    for t in range(T):
        sc = _group_scores_by_hand(key[t], G, m)
        order = sorted(range(G), key=lambda g: (-sc[g], g))
        open_g = set(order[:tg])
        # (a) every chosen expert lies in an open group
        assert all(int(e) // gs in open_g for e in idx[t])
        # (b) open groups outrank closed ones
        for go in open_g:
            for gc in set(range(G)) - open_g:
                assert sc[go] > sc[gc] or (sc[go] == sc[gc] and go < gc)
        # (c) the choice is the top-k of the open experts by (key desc, id asc)
        cand = [e for e in range(E) if e // gs in open_g]
        want = sorted(cand, key=lambda e: (-float(key[t, e]), e))[:k]
        assert idx[t].tolist() == want


def test_group_limited_planted_max_instead_of_sum_is_caught(monkeypatch):
    """A group score taken as the group's maximum (a plausible misreading)
    fails the hand-worked fixture."""
    orig = ref.group_limit_mask

    def by_max(key, k, num_groups, topk_group):
        return orig(key, topk_group, num_groups, topk_group)   # m = 1: the maximum
    monkeypatch.setattr(ref, "group_limit_mask", by_max)
    with pytest.raises(AssertionError):
        test_golden_group_limited_hand()


# ---------------------------------------------------------------------------
# auxiliary load-balancing loss
# ---------------------------------------------------------------------------
def test_golden_aux_loss_hand():
    g = json.load(open(os.path.join(GOLDEN, "aux_loss_hand.json")))
    lg = np.log(np.array(g["logits_ln_of"], np.float64))
    idx, _ = ref.route_topk(lg.astype(np.float32), g["k"], g["score_fn"], 1)
    assert idx.tolist() == g["topk_idx"]
    loss, counts, _ = ref.aux_loss(lg, idx, g["E"], g["score_fn"], g["coeff"])
    assert counts.tolist() == g["counts"]
    np.testing.assert_allclose(loss, g["loss"], rtol=1e-14)
    d = ref.aux_loss_bwd(lg, counts, g["k"], g["score_fn"], g["coeff"])
    np.testing.assert_allclose(d, g["d_logits"], rtol=1e-13, atol=1e-18)


@pytest.mark.parametrize("E,k", [(4, 1), (8, 2), (64, 8), (5, 5)])
@pytest.mark.parametrize("sfn", [0, 1])
def test_aux_loss_equal_logits_closed_form(E, k, sfn):
    """Equal logits: p = 1/E for every expert and every token picks experts
    0..k-1, so sum_e f_e P_e = k * (E/k) * (1/E) = 1 and loss = coeff."""
    lg = np.full((37, E), 0.25, np.float32)
    idx, _ = ref.route_topk(lg, k, sfn, 1)
    loss, counts, P = ref.aux_loss(lg, idx, E, sfn, 0.03)
    np.testing.assert_allclose(P, 1.0 / E, rtol=1e-15)
    assert counts.tolist() == [37] * k + [0] * (E - k)
    np.testing.assert_allclose(loss, 0.03, rtol=1e-14)


def test_aux_loss_uses_scipy_softmax_and_is_permutation_invariant():
    rng = np.random.default_rng(9)
    lg = rng.standard_normal((50, 12)).astype(np.float32)
    idx, _ = ref.route_topk(lg, 3, 0, 1)
    loss, counts, P = ref.aux_loss(lg, idx, 12, 0, 1.0)
    np.testing.assert_allclose(P, scipy.special.softmax(lg.astype(np.float64), axis=1).mean(0),
                               rtol=1e-13)
    perm = rng.permutation(12)
    inv = np.argsort(perm)
    loss_p, _, _ = ref.aux_loss(lg[:, perm], inv[idx], 12, 0, 1.0)
    np.testing.assert_allclose(loss_p, loss, rtol=1e-13)
    # sigmoid probabilities are expit normalised over the experts
    _, _, Ps = ref.aux_loss(lg, idx, 12, 1, 1.0)
    s = scipy.special.expit(lg.astype(np.float64))
    np.testing.assert_allclose(Ps, (s / s.sum(1, keepdims=True)).mean(0), rtol=1e-13)


@pytest.mark.parametrize("sfn,E,k", [(0, 8, 2), (1, 16, 4), (0, 5, 1)])
def test_aux_loss_bwd_vs_fd_and_autograd(sfn, E, k):
    rng = np.random.default_rng(E + 10 * sfn)
    T = 9
    lg = rng.standard_normal((T, E))
    idx, _ = ref.route_topk(lg.astype(np.float32), k, sfn, 1)
    coeff = 0.7
    _, counts, _ = ref.aux_loss(lg, idx, E, sfn, coeff)
    d = ref.aux_loss_bwd(lg, counts, k, sfn, coeff, d_loss=1.3)
    # central differences of 1.3 * loss, routing decision held fixed
    h = 1e-6
    fd = np.zeros_like(lg)
    for t in range(T):
        for e in range(E):
            lp, lm = lg.copy(), lg.copy()
            lp[t, e] += h
            lm[t, e] -= h
            fd[t, e] = 1.3 * (ref.aux_loss(lp, idx, E, sfn, coeff)[0] -
                              ref.aux_loss(lm, idx, E, sfn, coeff)[0]) / (2 * h)
    np.testing.assert_allclose(d, fd, rtol=1e-6, atol=1e-10)
    # autograd of the loss written with torch ops
    l_t = torch.tensor(lg, dtype=torch.float64, requires_grad=True)
    p = torch.softmax(l_t, 1) if sfn == 0 else torch.sigmoid(l_t) / torch.sigmoid(l_t).sum(1, keepdim=True)
    f = torch.tensor(counts, dtype=torch.float64) * E / (k * T)
    (1.3 * coeff * (f * p.mean(0)).sum()).backward()
    np.testing.assert_allclose(d, l_t.grad.numpy(), rtol=1e-12, atol=1e-15)
