"""GPU parity of moe_route_topk and moe_permute against the oracle: indices,
group layout and permuted rows bit-exact; fp32 weights to 1e-6."""
import numpy as np
import pytest
import torch

import moe_synth
from gpu_helpers import W_ATOL, dev_bf16
from oracle import moe_ref

pytestmark = pytest.mark.gpu

L = pytest.importorskip("mixture_experts_grouped_router_gb300._lib")


def _logits(rng, T, E, kind):
    if kind == "normal":
        return rng.standard_normal((T, E)).astype(np.float32)
    if kind == "ties":
        return rng.integers(-2, 3, size=(T, E)).astype(np.float32)
    if kind == "equal":
        return np.zeros((T, E), np.float32)
    if kind == "one_expert":   # every token prefers expert E-1 by far
        lg = rng.standard_normal((T, E)).astype(np.float32)
        lg[:, -1] += 100.0
        return lg
    if kind == "skew":
        return (rng.standard_normal((T, E)) + np.linspace(-4, 4, E)).astype(np.float32)
    raise ValueError(kind)


ROUTE_CASES = [
    (1, 8, 1, 0, 1, "normal"), (257, 8, 2, 0, 1, "normal"), (300, 32, 8, 1, 1, "normal"),
    (513, 64, 1, 0, 0, "skew"), (100, 256, 16, 1, 0, "normal"), (77, 5, 5, 0, 1, "ties"),
    (64, 33, 3, 1, 1, "equal"), (129, 128, 6, 0, 0, "ties"), (1000, 160, 4, 1, 1, "normal"),
]


@pytest.mark.parametrize("case", ROUTE_CASES)
def test_route_topk(case):
    T, E, k, sfn, ren, kind = case
    rng = np.random.default_rng(T * 7 + E)
    lg = _logits(rng, T, E, kind)
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, dtype=torch.float32, device="cuda")
    L.moe_route_topk(torch.from_numpy(lg).cuda(), k, sfn, ren, idx, w)
    torch.cuda.synchronize()
    ridx, rw = moe_ref.route_topk(lg, k, sfn, ren)
    assert (idx.cpu().numpy() == ridx).all()
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=0, atol=W_ATOL)


def test_route_topk_strided_logits():
    rng = np.random.default_rng(1)
    full = rng.standard_normal((50, 40)).astype(np.float32)
    lg = torch.from_numpy(full).cuda()[:, :24]
    idx = torch.empty(50, 4, dtype=torch.int32, device="cuda")
    w = torch.empty(50, 4, dtype=torch.float32, device="cuda")
    L.moe_route_topk(lg, 4, 0, 1, idx, w)
    ridx, rw = moe_ref.route_topk(full[:, :24], 4, 0, 1)
    assert (idx.cpu().numpy() == ridx).all()
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=0, atol=W_ATOL)


def run_permute(idx_np, E, align, cap, d=64, seed=0, x_bits=None):
    T, k = idx_np.shape
    rng = np.random.default_rng(seed)
    if x_bits is None:
        x_bits = moe_synth.bf16_bits(rng.standard_normal((T, d)).astype(np.float32))
    rows_cap = L.moe_rows_cap(T, E, k, align)
    dev = "cuda"
    x = dev_bf16(x_bits)
    xs = torch.full((rows_cap, d), float("nan"), dtype=torch.bfloat16, device=dev)
    gs = torch.empty(E, dtype=torch.int32, device=dev)
    kc = torch.empty(E, dtype=torch.int32, device=dev)
    off = torch.empty(E + 1, dtype=torch.int32, device=dev)
    s2f = torch.full((rows_cap,), 12345, dtype=torch.int32, device=dev)
    f2s = torch.full((T * k,), 12345, dtype=torch.int32, device=dev)
    ws = torch.empty(L.moe_permute_workspace_bytes(T, E), dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    L.moe_permute(x, torch.from_numpy(idx_np.astype(np.int32)).to(dev), E, align, cap, xs, gs, kc,
                  off, s2f, f2s, ws, st)
    torch.cuda.synchronize()
    return dict(x_bits=x_bits, xs=xs, gs=gs, kc=kc, off=off, s2f=s2f, f2s=f2s, st=st,
                rows_cap=rows_cap)


def check_permute(r, idx_np, E, align, cap):
    T, k = idx_np.shape
    lay = moe_ref.permute_layout(idx_np, E, align, cap)
    R = lay["R"]
    assert int(r["st"].item()) == 0
    assert r["gs"].cpu().numpy().tolist() == lay["group_sizes"].tolist()
    assert r["kc"].cpu().numpy().tolist() == lay["kept_counts"].tolist()
    assert r["off"].cpu().numpy().tolist() == lay["group_offsets"].tolist()
    s2f = r["s2f"].cpu().numpy()
    assert s2f[:R].tolist() == lay["sorted_to_flat"].tolist()
    assert (s2f[R:] == -1).all()
    assert r["f2s"].cpu().numpy().tolist() == lay["flat_to_sorted"].tolist()
    # permuted rows: exact copies of x (compared bitwise), padding rows zero
    xs_bits = r["xs"][:R].view(torch.int16).cpu().numpy().astype(np.uint16)
    ref_rows = np.zeros((R, r["x_bits"].shape[1]), np.uint16)
    ok = lay["sorted_to_flat"] >= 0
    ref_rows[ok] = r["x_bits"][lay["sorted_to_flat"][ok] // k]
    assert (xs_bits == ref_rows).all()


PERMUTE_CASES = [
    # T, E, k, align, cap, logits kind
    (1, 4, 1, 0, 0, "normal"), (300, 8, 2, 0, 0, "normal"), (1025, 8, 2, 0, 0, "normal"),
    (3000, 32, 8, 0, 0, "normal"), (2500, 64, 1, 128, 40, "skew"), (2049, 16, 4, 8, 0, "ties"),
    (777, 8, 2, 1, 0, "one_expert"), (1500, 8, 2, 16, 100, "one_expert"),
    (4097, 256, 8, 4, 50, "skew"), (512, 6, 3, 2, 0, "equal"), (2000, 64, 2, 128, 0, "skew"),
]


@pytest.mark.parametrize("case", PERMUTE_CASES)
def test_permute(case):
    T, E, k, align, cap, kind = case
    rng = np.random.default_rng(T + E)
    idx, _ = moe_ref.route_topk(_logits(rng, T, E, kind), k, 0, 1)
    r = run_permute(idx, E, align, cap, d=72, seed=T)
    check_permute(r, idx, E, align, cap)


def test_permute_no_tokens():
    idx = np.zeros((0, 2), np.int32)
    r = run_permute(idx, 4, 8, 0, d=16)
    assert r["gs"].cpu().numpy().tolist() == [0, 0, 0, 0]
    assert r["off"].cpu().numpy().tolist() == [0, 0, 0, 0, 0]
    assert (r["s2f"].cpu().numpy() == -1).all()


@pytest.mark.parametrize("align", [0, 8])
def test_permute_bad_expert_sets_status_without_fault(align):
    """An id out of range and a repeated id are both dropped, by the counts as
    well as the ranks: the groups hold only the valid assignments, every kept
    row is written and padding rows are zero.  Expected layout by hand: valid
    assignments a0 (token 0, expert 0), a1 (0, 1), a2 (1, 2), a4 (2, 1); a3
    (expert 9) and a5 (token 2 repeats expert 1) are dropped."""
    idx = np.array([[0, 1], [2, 9], [1, 1]], np.int32)
    r = run_permute(idx, 4, align, 0, d=16)
    assert int(r["st"].item()) == L.MOE_ERR_DEVICE
    assert r["kc"].cpu().numpy().tolist() == [1, 2, 1, 0]
    if align == 8:
        gs, s2f = [8, 8, 8, 0], [0] + [-1] * 7 + [1, 4] + [-1] * 6 + [2] + [-1] * 7
    else:
        gs, s2f = [1, 2, 1, 0], [0, 1, 4, 2]
    assert r["gs"].cpu().numpy().tolist() == gs
    assert r["off"].cpu().numpy().tolist() == np.concatenate([[0], np.cumsum(gs)]).tolist()
    R = sum(gs)
    got_s2f = r["s2f"].cpu().numpy()
    assert got_s2f[:R].tolist() == s2f and (got_s2f[R:] == -1).all()
    f2s = r["f2s"].cpu().numpy()
    assert f2s[3] == -1 and f2s[5] == -1
    assert [f2s[a] for a in (0, 1, 2, 4)] == [s2f.index(a) for a in (0, 1, 2, 4)]
    xs_bits = r["xs"][:R].view(torch.int16).cpu().numpy().astype(np.uint16)
    for p_, a in enumerate(s2f):
        want = r["x_bits"][a // 2] if a >= 0 else np.zeros(16, np.uint16)
        assert (xs_bits[p_] == want).all(), p_


BIAS_CASES = [(300, 8, 2, 1, 1), (513, 64, 8, 1, 1), (100, 256, 4, 0, 0), (77, 32, 3, 0, 1)]


@pytest.mark.parametrize("case", BIAS_CASES)
def test_route_topk_expert_bias(case):
    T, E, k, sfn, ren = case
    rng = np.random.default_rng(T + E + k)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    bias = (rng.standard_normal(E) * 2).astype(np.float32)
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, dtype=torch.float32, device="cuda")
    L.moe_route_topk(torch.from_numpy(lg).cuda(), k, sfn, ren, idx, w,
                     expert_bias=torch.from_numpy(bias).cuda())
    torch.cuda.synchronize()
    ridx, rw = moe_ref.route_topk(lg, k, sfn, ren, expert_bias=bias)
    assert (idx.cpu().numpy() == ridx).all()
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=0, atol=W_ATOL)


ROUTE_BWD_CASES = [(257, 8, 2, 0, 1), (300, 32, 8, 1, 1), (513, 64, 1, 0, 0), (100, 256, 16, 1, 0),
                   (129, 128, 6, 0, 0), (64, 5, 5, 1, 1), (33, 40, 1, 0, 1)]


@pytest.mark.parametrize("case", ROUTE_BWD_CASES)
def test_route_topk_bwd(case):
    T, E, k, sfn, ren = case
    rng = np.random.default_rng(3 * T + E)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    lgd = torch.from_numpy(lg).cuda()
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, dtype=torch.float32, device="cuda")
    L.moe_route_topk(lgd, k, sfn, ren, idx, w)
    dw_np = rng.standard_normal((T, k)).astype(np.float32)
    dl = torch.full((T, E), float("nan"), dtype=torch.float32, device="cuda")
    L.moe_route_topk_bwd(lgd, idx, w, torch.from_numpy(dw_np).cuda(), sfn, ren, dl)
    torch.cuda.synchronize()
    ridx, _ = moe_ref.route_topk(lg, k, sfn, ren)
    assert (idx.cpu().numpy() == ridx).all()
    want = moe_ref.route_topk_bwd(lg, ridx, dw_np.astype(np.float64), sfn, ren)
    got = dl.cpu().numpy().astype(np.float64)
    # fp32 arithmetic on fp32 inputs: far tighter than the layer's bf16 tolerance
    np.testing.assert_allclose(got, want, rtol=0, atol=2e-6 * max(1.0, np.abs(want).max()))
    if not (sfn == 0 and ren == 0):
        sel = np.zeros((T, E), bool)
        np.put_along_axis(sel, ridx.astype(np.int64), True, 1)
        assert (got[~sel] == 0).all()


GROUP_CASES = [
    # T, E, k, num_groups, topk_group, score_fn, renorm, bias, logits kind
    (300, 8, 4, 4, 2, 0, 1, False, "normal"), (513, 64, 6, 8, 3, 1, 1, True, "normal"),
    (1000, 256, 8, 8, 4, 1, 1, True, "normal"), (257, 32, 4, 4, 2, 0, 0, False, "ties"),
    (129, 16, 4, 16, 4, 1, 0, False, "ties"), (100, 160, 8, 5, 2, 0, 1, True, "skew"),
    (64, 256, 16, 32, 8, 1, 1, False, "normal"), (77, 12, 3, 3, 3, 0, 1, False, "equal"),
]


@pytest.mark.parametrize("case", GROUP_CASES)
def test_route_topk_group_limited(case):
    T, E, k, G, tg, sfn, ren, with_bias, kind = case
    rng = np.random.default_rng(T + E + G)
    lg = _logits(rng, T, E, kind)
    bias = (rng.standard_normal(E) * 0.5).astype(np.float32) if with_bias else None
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, dtype=torch.float32, device="cuda")
    L.moe_route_topk(torch.from_numpy(lg).cuda(), k, sfn, ren, idx, w,
                     expert_bias=None if bias is None else torch.from_numpy(bias).cuda(),
                     num_groups=G, topk_group=tg)
    torch.cuda.synchronize()
    ridx, rw = moe_ref.route_topk(lg, k, sfn, ren, expert_bias=bias, num_groups=G,
                                  topk_group=tg)
    assert (idx.cpu().numpy() == ridx).all()
    np.testing.assert_allclose(w.cpu().numpy(), rw, rtol=0, atol=W_ATOL)
