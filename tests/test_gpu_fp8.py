"""GPU parity of the FP8 path against the FP8 oracle (oracle/moe_fp8_ref.py):
amax and scales, row-wise and column-wise codes (bit-exact; the column-wise
copy of a grouped activation with its per-group padding of zeros), the FP8
grouped GEMMs, and the FP8 layer.

The recipe is the pages' configuration of the expert GEMMs (MaxText PR #2319,
"[Draft] Integrate TE/JAX GroupedGEMM for MoE", review thread on the quantizer
settings: current tensor scaling, float8_e4m3fn forward, float8_e5m2
backward, row- and column-wise copies)."""
import dataclasses

import numpy as np
import pytest
import torch

import moe_synth
from gpu_helpers import assert_close, dev_bf16, layer_shape
from oracle import moe_fp8_ref as q8
from oracle import moe_ref

pytestmark = pytest.mark.gpu
L = pytest.importorskip("mixture_experts_grouped_router_gb300._lib")

FMTS = {0: "e4m3", 1: "e5m2"}


def _bf(rng, shape, scale=1.0):
    return moe_synth.bf16_bits((rng.standard_normal(shape) * scale).astype(np.float32))


def _f32(bits):
    return moe_synth.bits_to_f64(bits).astype(np.float32)


@pytest.mark.parametrize("E,K,N", [(1, 64, 64), (4, 128, 96), (3, 80, 208), (8, 256, 512)])
@pytest.mark.parametrize("fmt", [0, 1])
def test_quantize_weights(E, K, N, fmt):
    rng = np.random.default_rng(E * K + N + fmt)
    w_bits = np.stack([_bf(rng, (K, N), 10.0 ** rng.uniform(-3, 2)) for _ in range(E)])
    w = dev_bf16(w_bits)
    amax = torch.full((E,), -1.0, device="cuda")
    L.moe_fp8_amax(w.view(E * K, N), amax, groups=E)
    q = torch.empty(E, K, N, dtype=torch.uint8, device="cuda")
    qt = torch.empty(E, N, K, dtype=torch.uint8, device="cuda")
    sinv = torch.empty(E, device="cuda")
    L.moe_fp8_quantize_weights(w, fmt, amax, q, qt, sinv)
    torch.cuda.synchronize()
    name = FMTS[fmt]
    for e in range(E):
        x = _f32(w_bits[e])
        ra = np.abs(x).max()
        assert float(amax[e].item()) == ra
        s = q8.current_scale(ra, name)
        np.testing.assert_allclose(float(sinv[e].item()), 1.0 / float(s), rtol=1e-7)
        want = q8.quantize(x, s, name)
        got = q[e].cpu().numpy()
        assert (got == want).all(), (e, np.argwhere(got != want)[:4])
        assert (qt[e].cpu().numpy() == want.T).all()


def _offsets(sizes):
    return np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)


def _poff(sizes, pad=128):
    p = [0]
    for s in sizes:
        p.append(p[-1] + (s + pad - 1) // pad * pad)
    return p


@pytest.mark.parametrize("groups,rpg,cols", [(5, 37, 24), (3, 4099, 2056), (40, 9, 8)])
def test_amax_groups_ragged(groups, rpg, cols):
    """Per-group amax when groups straddle the blocks' row ranges (rows per
    group not a multiple of the rows a block reads at once); each group's
    maximum sits on its first or last row."""
    rng = np.random.default_rng(groups * rpg + cols)
    bits = _bf(rng, (groups * rpg, cols))
    for g in range(groups):
        r = g * rpg + (0 if g % 2 else rpg - 1)
        v = -(8.0 + g) if g % 3 else 8.0 + g
        bits[r, (g * 7) % cols] = moe_synth.bf16_bits(np.float32([v]))[0]
    x = dev_bf16(bits)
    amax = torch.full((groups,), -1.0, device="cuda")
    L.moe_fp8_amax(x, amax, groups=groups)
    got = amax.cpu().numpy()
    want = np.abs(moe_synth.bits_to_f64(bits).reshape(groups, rpg * cols)).max(axis=1)
    assert (got == want.astype(np.float32)).all(), (got, want)


def test_amax_nan_propagates():
    """A NaN element makes its group's amax NaN (the scale then falls back to 1)."""
    rng = np.random.default_rng(7)
    bits = _bf(rng, (2 * 64, 32))
    x = dev_bf16(bits)
    x[70, 5] = float("nan")                   # group 1
    amax = torch.full((2,), -1.0, device="cuda")
    L.moe_fp8_amax(x, amax, groups=2)
    got = amax.cpu().numpy()
    assert got[0] == np.abs(moe_synth.bits_to_f64(bits[:64])).max()
    assert np.isnan(got[1])


@pytest.mark.parametrize("sizes,cols", [([0, 7, 300, 128, 129, 0, 1, 640], 64),
                                        ([517], 96), ([1, 2, 3], 16), ([256, 0, 0], 512),
                                        ([0, 0], 32), ([64] * 40, 128)])
@pytest.mark.parametrize("fmt", [0, 1])
def test_quantize_act_padded_transpose(sizes, cols, fmt):
    rng = np.random.default_rng(len(sizes) * 31 + cols + fmt)
    off = _offsets(sizes)
    E, R = len(sizes), int(off[-1])
    rows_cap = R + 23
    x_bits = _bf(rng, (rows_cap, cols), 3.0)
    x = dev_bf16(x_bits)
    x[R:] = float("nan")                      # rows past the groups are never read
    offd = torch.from_numpy(off).cuda()
    pr = L.moe_fp8_padded_rows(rows_cap, E)
    assert pr % 128 == 0 and pr >= _poff(sizes)[-1]
    amax = torch.full((1,), -1.0, device="cuda")
    L.moe_fp8_amax(x, amax, group_offsets=offd, E=E)
    q = torch.full((rows_cap, cols), 0xAB, dtype=torch.uint8, device="cuda")
    qt = torch.full((cols, pr), 0xAB, dtype=torch.uint8, device="cuda")
    sinv = torch.empty(1, device="cuda")
    L.moe_fp8_quantize_act(x, offd, fmt, amax, q, qt, sinv)
    torch.cuda.synchronize()
    name = FMTS[fmt]
    xf = _f32(x_bits[:R])
    ra = np.abs(xf).max() if R else 0.0
    assert float(amax.item()) == ra
    s = q8.current_scale(ra, name)
    want = q8.quantize(xf, s, name)
    qn = q.cpu().numpy()
    assert (qn[:R] == want).all()
    assert (qn[R:] == 0xAB).all(), "rows past the groups were written"
    qtn = qt.cpu().numpy()
    po = _poff(sizes)
    for e in range(E):
        a, b = int(off[e]), int(off[e + 1])
        seg = qtn[:, po[e]:po[e + 1]]
        assert (seg[:, :b - a] == want[a:b].T).all(), e
        assert (seg[:, b - a:] == 0).all(), e
    assert (qtn[:, po[-1]:] == 0xAB).all()


# ---------------------------------------------------------------------------
# FP8 grouped GEMMs: both sides quantize the same bf16 inputs (codes are
# bit-exact, see above); the oracle multiplies the dequantized values in fp64
# ---------------------------------------------------------------------------

SIZES = {"mixed": [0, 7, 300, 128, 129, 0, 1, 640], "one": [517], "tiny": [1, 2, 3],
         "empty_tail": [256, 0, 0]}


def _act_gpu(x_bits, off, fmt):
    """GPU quantization of a permuted activation; oracle dequantized values."""
    E = len(off) - 1
    x = dev_bf16(x_bits)
    offd = torch.from_numpy(off).cuda()
    rows_cap, cols = x.shape
    amax = torch.empty(1, device="cuda")
    L.moe_fp8_amax(x, amax, group_offsets=offd, E=E)
    q = torch.zeros(rows_cap, cols, dtype=torch.uint8, device="cuda")
    pr = L.moe_fp8_padded_rows(rows_cap, E)
    qt = torch.zeros(cols, pr, dtype=torch.uint8, device="cuda")
    sinv = torch.empty(1, device="cuda")
    L.moe_fp8_quantize_act(x, offd, fmt, amax, q, qt, sinv)
    R = int(off[-1])
    xf = _f32(x_bits[:R])
    s = q8.current_scale(np.abs(xf).max() if R else 0.0, FMTS[fmt])
    deq = q8.dequantize(q8.quantize(xf, s, FMTS[fmt]), s, FMTS[fmt])
    return q, qt, sinv, deq


def _w_gpu(w_bits, fmt):
    E, K, N = w_bits.shape
    w = dev_bf16(w_bits)
    amax = torch.empty(E, device="cuda")
    L.moe_fp8_amax(w.view(E * K, N), amax, groups=E)
    q = torch.empty(E, K, N, dtype=torch.uint8, device="cuda")
    qt = torch.empty(E, N, K, dtype=torch.uint8, device="cuda")
    sinv = torch.empty(E, device="cuda")
    L.moe_fp8_quantize_weights(w, fmt, amax, q, qt, sinv)
    deq = np.stack([q8.qdq_tensor(_f32(w_bits[e]), FMTS[fmt])[0] for e in range(E)])
    return q, qt, sinv, deq


# sizes of quantized operands are multiples of 16 (codes move in 16-byte rows)
GMM8_CASES = [("mixed", 256, 384), ("one", 1024, 144), ("tiny", 128, 64), ("empty_tail", 512, 1024),
              ("mixed", 4096, 256)]
SAME_FMT = [(0, 0)]
MIXED_FMT = [(1, 0)]


@pytest.mark.parametrize("case", GMM8_CASES)
@pytest.mark.parametrize("fmts", SAME_FMT + MIXED_FMT)
@pytest.mark.parametrize("transposed_weight", [False, True])
def test_gmm_fp8_none(case, fmts, transposed_weight):
    sz, K, N = case
    fa, fb = fmts
    rng = np.random.default_rng(K + N + 10 * fa + fb)
    off = _offsets(SIZES[sz])
    E, R = len(SIZES[sz]), int(off[-1])
    rows_cap = R + 19
    a_q, _, a_sinv, a_deq = _act_gpu(_bf(rng, (rows_cap, K), 2.0), off, fa)
    if transposed_weight:   # dgrad: weight stored [E, N, K], used as is
        w_bits = _bf(rng, (E, N, K), 0.05)
        w_q, _, b_sinv, w_deq = _w_gpu(w_bits, fb)
        b_op, w_ref, tr = w_q, w_deq, True
    else:                   # forward: weight stored [E, K, N], its transposed copy
        w_bits = _bf(rng, (E, K, N), 0.05)
        _, w_qt, b_sinv, w_deq = _w_gpu(w_bits, fb)
        b_op, w_ref, tr = w_qt, w_deq, False
    C = torch.full((rows_cap, N), 7.0, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    L.moe_gmm_fp8(a_q, fa, a_sinv, b_op, fb, b_sinv, torch.from_numpy(off).cuda(), C,
                  dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    want = moe_ref.gmm(a_deq, w_ref, off, transpose_rhs=tr)
    assert_close("gmm_fp8", C[:R], want)
    assert (C[R:].float() == 7.0).all()


def test_gmm_fp8_epilogue_amax_is_the_outputs_amax():
    """amax_out of the SwiGLU forward / backward / plain epilogues is max |.| of
    the bf16 tensor the GEMM wrote (the amax that quantizes it next)."""
    rng = np.random.default_rng(77)
    off = _offsets(SIZES["mixed"])
    E, R = len(SIZES["mixed"]), int(off[-1])
    rows_cap = R + 5
    K, F = 256, 192
    offd = torch.from_numpy(off).cuda()
    a_q, _, a_sinv, _ = _act_gpu(_bf(rng, (rows_cap, K), 2.0), off, 0)
    _, w_qt, b_sinv, _ = _w_gpu(_bf(rng, (E, K, 2 * F), 0.05), 0)
    H = torch.empty(rows_cap, 2 * F, dtype=torch.bfloat16, device="cuda")
    Act = torch.full((rows_cap, F), 1e4, dtype=torch.bfloat16, device="cuda")
    amax = torch.full((1,), -1.0, device="cuda")
    L.moe_gmm_fp8(a_q, 0, a_sinv, w_qt, 0, b_sinv, offd, H, L.EPI_SWIGLU_FWD, C2=Act,
                  amax_out=amax)
    torch.cuda.synchronize()
    assert float(amax.item()) == float(Act[:R].float().abs().max().item())
    w_q, _, wsinv, _ = _w_gpu(_bf(rng, (E, F, K), 0.05), 1)
    dH = torch.full((rows_cap, 2 * F), 1e4, dtype=torch.bfloat16, device="cuda")
    L.moe_gmm_fp8(a_q, 0, a_sinv, w_q, 1, wsinv, offd, dH, L.EPI_SWIGLU_BWD, aux=H, amax_out=amax)
    torch.cuda.synchronize()
    assert float(amax.item()) == float(dH[:R].float().abs().max().item())
    C = torch.full((rows_cap, F), 1e4, dtype=torch.bfloat16, device="cuda")
    L.moe_gmm_fp8(a_q, 0, a_sinv, w_q, 1, wsinv, offd, C, amax_out=amax)
    torch.cuda.synchronize()
    assert float(amax.item()) == float(C[:R].float().abs().max().item())


@pytest.mark.parametrize("sz,K,F", [("mixed", 256, 192), ("one", 512, 200), ("tiny", 128, 64)])
def test_gmm_fp8_swiglu_fwd(sz, K, F):
    rng = np.random.default_rng(K + F)
    off = _offsets(SIZES[sz])
    E, R = len(SIZES[sz]), int(off[-1])
    rows_cap = R + 5
    a_q, _, a_sinv, a_deq = _act_gpu(_bf(rng, (rows_cap, K), 2.0), off, 0)
    _, w_qt, b_sinv, w_deq = _w_gpu(_bf(rng, (E, K, 2 * F), 0.05), 0)
    H = torch.empty(rows_cap, 2 * F, dtype=torch.bfloat16, device="cuda")
    Act = torch.empty(rows_cap, F, dtype=torch.bfloat16, device="cuda")
    L.moe_gmm_fp8(a_q, 0, a_sinv, w_qt, 0, b_sinv, torch.from_numpy(off).cuda(), H,
                  L.EPI_SWIGLU_FWD, C2=Act)
    torch.cuda.synchronize()
    h = moe_ref.gmm(a_deq, w_deq, off)
    assert_close("H", H[:R], h)
    assert_close("Act", Act[:R], moe_ref.swiglu(h))


@pytest.mark.parametrize("sz,K,F", [("mixed", 256, 192), ("one", 512, 208), ("tiny", 128, 64)])
@pytest.mark.parametrize("fmts", SAME_FMT + MIXED_FMT)
def test_gmm_fp8_swiglu_bwd(sz, K, F, fmts):
    fa, fb = fmts
    rng = np.random.default_rng(K * F + fa)
    off = _offsets(SIZES[sz])
    E, R = len(SIZES[sz]), int(off[-1])
    rows_cap = R + 5
    a_q, _, a_sinv, a_deq = _act_gpu(_bf(rng, (rows_cap, K), 1.0), off, fa)
    w_q, _, b_sinv, w_deq = _w_gpu(_bf(rng, (E, F, K), 0.05), fb)      # wo [E, F, d]
    h_bits = _bf(rng, (rows_cap, 2 * F), 2.0)
    dH = torch.empty(rows_cap, 2 * F, dtype=torch.bfloat16, device="cuda")
    L.moe_gmm_fp8(a_q, fa, a_sinv, w_q, fb, b_sinv, torch.from_numpy(off).cuda(), dH,
                  L.EPI_SWIGLU_BWD, aux=dev_bf16(h_bits))
    torch.cuda.synchronize()
    d_act = moe_ref.gmm(a_deq, w_deq, off, transpose_rhs=True)
    want = moe_ref.swiglu_bwd(moe_synth.bits_to_f64(h_bits)[:R], d_act)
    assert_close("dH", dH[:R], want)


@pytest.mark.parametrize("sz,M,N", [("mixed", 256, 384), ("one", 144, 208), ("tiny", 64, 64),
                                    ("empty_tail", 128, 528)])
@pytest.mark.parametrize("fmts", SAME_FMT + MIXED_FMT)
@pytest.mark.parametrize("w_f32", [False, True])
def test_tgmm_fp8(sz, M, N, fmts, w_f32):
    fa, fb = fmts
    rng = np.random.default_rng(M + N + fa + 3 * w_f32)
    off = _offsets(SIZES[sz])
    E, R = len(SIZES[sz]), int(off[-1])
    rows_cap = R + 11
    _, a_qt, a_sinv, a_deq = _act_gpu(_bf(rng, (rows_cap, M), 1.0), off, fa)
    _, b_qt, b_sinv, b_deq = _act_gpu(_bf(rng, (rows_cap, N), 1.0), off, fb)
    W = torch.full((E, M, N), 5.0, dtype=torch.float32 if w_f32 else torch.bfloat16, device="cuda")
    L.moe_tgmm_fp8(a_qt, fa, a_sinv, b_qt, fb, b_sinv, torch.from_numpy(off).cuda(), rows_cap, W)
    torch.cuda.synchronize()
    want = moe_ref.tgmm(a_deq, b_deq, off, E)
    assert_close("W", W, want)
    for e in np.nonzero(np.diff(off) == 0)[0]:
        assert (W[e].float() == 0).all()


# ---------------------------------------------------------------------------
# the FP8 layer against the FP8 oracle
# ---------------------------------------------------------------------------
C = moe_synth.CONFIGS
FP8_LAYERS = {
    "mixtral": moe_synth.scaled(C["mixtral"], T=1024, d=256, f=448),
    "dsv3": moe_synth.scaled(C["dsv3"], T=512, d=448, f=256),
    "skewed": moe_synth.scaled(C["skewed"], T=4096, d=256, f=128, capacity=64),
    "odd": moe_synth.MoEConfig("odd", T=999, d=208, f=144, E=7, k=3, score_fn=1, renorm=0,
                               align=16, capacity=300),
}


def _rel(a, b):
    a = a.detach().float().cpu().numpy().astype(np.float64) if isinstance(a, torch.Tensor) else a
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def _max_rel(a, b):
    """max |a - b| / max |b|: the elementwise half of the acceptance bar."""
    a = a.detach().float().cpu().numpy().astype(np.float64) if isinstance(a, torch.Tensor) else a
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-300))


@pytest.mark.parametrize("name", list(FP8_LAYERS))
def test_layer_fp8(name):
    """The GPU follows the FP8 recipe: every output is within 1e-2 (relative
    Frobenius) and 5e-2 * max|ref| (elementwise) of the FP8 oracle, and at
    most half as far from it as the FP8 oracle is from the unquantized layer.
    Both sides quantize the same bf16 tensors; the residual is fp32 against
    fp64 accumulation, which now and then moves a bf16 rounding and with it
    one code."""
    from mixture_experts_grouped_router_gb300 import layer
    cfg = FP8_LAYERS[name]
    inp = moe_synth.make_inputs(cfg, seed=4)
    f64 = moe_synth.bits_to_f64
    x, wi, wo, dout = (dev_bf16(inp[n]) for n in ("x", "wi", "wo", "dout"))
    logits = torch.from_numpy(inp["logits"]).cuda()
    shape = dataclasses.replace(layer_shape(cfg), fp8=True)
    b = layer.MoEBuffers(shape)
    layer.forward(b, x, logits, wi, wo)
    layer.backward(b, dout, wi, wo)
    torch.cuda.synchronize()
    assert int(b.dev_status.item()) == 0
    xs, wis, wos, douts = (f64(inp[n]) for n in ("x", "wi", "wo", "dout"))
    f8 = q8.forward(xs, inp["logits"], wis, wos, cfg.k, cfg.score_fn, cfg.renorm, cfg.align,
                    cfg.capacity)
    b8 = q8.backward(f8, douts, cfg.k)
    fr = moe_ref.forward(xs, inp["logits"], wis, wos, cfg.k, cfg.score_fn, cfg.renorm, cfg.align,
                         cfg.capacity)
    br = moe_ref.backward(fr, douts, wis, wos, cfg.k)
    assert (b.topk_idx.cpu().numpy() == f8["topk_idx"]).all()
    # the forward input of the up-projection is quantized from identical bf16 rows: exact codes
    R = f8["layout"]["R"]
    assert (b.xs_q[:R].cpu().numpy() ==
            q8.quantize(f8["xs"][:R].astype(np.float32), f8["scales"]["x"], "e4m3")).all()
    errs = {}
    for key, got, want8, want16 in (
            ("h", b.h[:R], f8["h"], fr["h"]), ("act", b.act[:R], f8["act"], fr["act"]),
            ("out", b.out, f8["out"], fr["out"]), ("dy", b.dy[:R], b8["dy"], br["dy"]),
            ("dh", b.dh[:R], b8["dh"], br["dh"]), ("dx", b.dx, b8["dx"], br["dx"]),
            ("dwi", b.dwi, b8["d_wi"], br["d_wi"]), ("dwo", b.dwo, b8["d_wo"], br["d_wo"]),
            ("d_topk_w", b.d_topk_w, b8["d_topk_w"], br["d_topk_w"])):
        errs[key] = (_rel(got, want8), _rel(want8, want16), _max_rel(got, want8))
    bad = {k: v for k, v in errs.items()
           if not (v[0] <= 1e-2 and v[0] <= 0.5 * v[1] and v[2] <= 5e-2)}
    assert not bad, errs


class _ExpertsF64:
    """Expert e's bf16 weights as float64, converted when asked for."""

    def __init__(self, bits):
        self.bits = bits

    def __len__(self):
        return self.bits.shape[0]

    def __getitem__(self, e):
        return moe_synth.bits_to_f64(self.bits[e])


@pytest.mark.parametrize("name", ["mixtral", "dsv3"])
def test_layer_fp8_full_size_sampled(name):
    """The FP8 layer at full size, in the configuration `bench.py --fp8` times,
    against the FP8 oracle.  The oracle derives every scale itself over all
    rows (layer_scales: Act and dH block by block in fp64, slow), then
    recomputes one by one: out and dx of sampled tokens, one row of dWo and
    one column of dWi of sampled experts; each within 1e-2 relative Frobenius
    and 5e-2 * max|ref| elementwise.  Scales of x, wi and wo are bit-exact;
    those of Act, dY and dH within one bf16 rounding of their amax."""
    from mixture_experts_grouped_router_gb300 import layer
    cfg = moe_synth.CONFIGS[name]
    inp = moe_synth.make_inputs(cfg, seed=0)
    x, wi, wo, dout = (dev_bf16(inp[n]) for n in ("x", "wi", "wo", "dout"))
    logits = torch.from_numpy(inp["logits"]).cuda()
    b = layer.MoEBuffers(dataclasses.replace(layer_shape(cfg), fp8=True))
    layer.forward(b, x, logits, wi, wo)
    layer.backward(b, dout, wi, wo)
    torch.cuda.synchronize()
    assert int(b.dev_status.item()) == 0
    del x, wi, wo, dout
    f64 = moe_synth.bits_to_f64
    E, k, f = cfg.E, cfg.k, cfg.f
    wi_b, wo_b = _ExpertsF64(inp["wi"]), _ExpertsF64(inp["wo"])
    sc = q8.layer_scales(f64(inp["x"]), inp["logits"], wi_b, wo_b, f64(inp["dout"]), k,
                         cfg.score_fn, cfg.renorm, cfg.align, cfg.capacity)
    lay, S = sc["layout"], sc["scales"]
    assert (b.topk_idx.cpu().numpy() == sc["topk_idx"]).all()
    assert b.group_offsets.cpu().numpy().tolist() == lay["group_offsets"].tolist()
    # the GPU keeps 1 / scale: slots x, act, dy, dh, wi[E], wo[E]
    g_scale = 1.0 / b.f8_sinv.double().cpu().numpy()
    g_sinv = b.f8_sinv.cpu().numpy()
    assert g_sinv[0] == np.float32(1) / S["x"]
    assert (g_sinv[4:4 + E] == np.float32(1) / S["wi"]).all()
    assert (g_sinv[4 + E:] == np.float32(1) / S["wo"]).all()
    for i, key in ((1, "act"), (2, "dy"), (3, "dh")):
        assert abs(g_scale[i] / float(S[key]) - 1) <= 2.0 ** -7, (key, g_scale[i], S[key])
    rng = np.random.default_rng(1)
    toks = rng.choice(cfg.T, size=6, replace=False)
    f2s = lay["flat_to_sorted"].reshape(cfg.T, k)
    off = lay["group_offsets"]
    col_experts = rng.choice(np.nonzero(lay["group_sizes"] > 0)[0], size=2, replace=False)
    out_ref = np.zeros((len(toks), cfg.d))
    dx_ref = np.zeros((len(toks), cfg.d))
    dwo_rows, dwo_ref, dwi_cols, dwi_ref = [], [], [], []
    xs_q, dy_q = sc["xs_q"], sc["dy_q"]
    w = sc["topk_w"]

    def qdq(v, key, fmt):
        return q8.dequantize(q8.encode_lib((np.asarray(v, np.float32) *
                                            np.float32(S[key])).astype(np.float32), fmt),
                             S[key], fmt)

    for e in range(E):
        uses = [(i, j) for i, t in enumerate(toks) for j in range(k)
                if f2s[t, j] >= 0 and off[e] <= f2s[t, j] < off[e + 1]]
        if not uses and e not in col_experts:
            continue
        wi_q = q8.dequantize(q8.encode_lib((wi_b[e].astype(np.float32) * S["wi"][e]).astype(
            np.float32), q8.E4M3), S["wi"][e], q8.E4M3)
        wo_q = q8.dequantize(q8.encode_lib((wo_b[e].astype(np.float32) * S["wo"][e]).astype(
            np.float32), q8.E4M3), S["wo"][e], q8.E4M3)
        for i, j in uses:
            p = f2s[toks[i], j]
            h = xs_q[p:p + 1] @ wi_q
            act_q = qdq(q8.round_bf16(moe_ref.swiglu(h)), "act", q8.E4M3)
            out_ref[i] += w[toks[i], j] * (act_q @ wo_q)[0]
            dh = q8.round_bf16(moe_ref.swiglu_bwd(q8.round_bf16(h), dy_q[p:p + 1] @ wo_q.T))
            dx_ref[i] += (qdq(dh, "dh", q8.E5M2) @ wi_q.T)[0]
        if e in col_experts:
            rows = slice(int(off[e]), int(off[e + 1]))
            c = int(rng.integers(f))
            h2 = xs_q[rows] @ wi_q[:, [c, f + c]]
            act_c = qdq(q8.round_bf16(moe_ref.swiglu(h2)), "act", q8.E4M3)[:, 0]
            dwo_rows.append((e, c))
            dwo_ref.append(act_c @ dy_q[rows])
            n = int(rng.integers(2 * f))
            cc = n % f
            h3 = q8.round_bf16(xs_q[rows] @ wi_q[:, [cc, f + cc]])
            dh2 = q8.round_bf16(moe_ref.swiglu_bwd(h3, dy_q[rows] @ wo_q[cc, :][:, None]))
            dh_n = qdq(dh2[:, 1 if n >= f else 0], "dh", q8.E5M2)
            dwi_cols.append((e, n))
            dwi_ref.append(xs_q[rows].T @ dh_n)
    tsel = torch.from_numpy(toks).cuda()
    assert_close("out (sampled tokens)", b.out[tsel], out_ref)
    assert_close("dx (sampled tokens)", b.dx[tsel], dx_ref)
    assert_close("dWo (sampled rows)", torch.stack([b.dwo[e][c, :] for e, c in dwo_rows]),
                 np.stack(dwo_ref))
    assert_close("dWi (sampled columns)", torch.stack([b.dwi[e][:, n] for e, n in dwi_cols]),
                 np.stack(dwi_ref))
