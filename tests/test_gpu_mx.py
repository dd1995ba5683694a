"""Block-scaled FP8 (MXFP8) on the GPU against the block-scaled oracle
(oracle/moe_mx_ref.py):

* moe_mx_quantize: codes and E8M0 scales bit-exact, in the scale-atom layout
  of every row order (plain, grouped with padded expert tiles, SwiGLU tiles),
  with zero, subnormal, saturating and non-finite blocks;
* moe_gmm_mx (each epilogue) and moe_tgmm_mx against the oracle's grouped
  GEMMs of the dequantized operands;
* the MXFP8 layer on reduced workloads element by element, and at full size
  on sampled columns and weight-gradient entries.  Every 32-element block is scaled by its
  own random power of two, so a scale applied to the wrong rows, columns or
  blocks changes the result by factors of 2 and more.

The scale-atom layout (a property of the interface, restated here): atom
(ar, ac) at byte (ar * cols / 128 + ac) * 512 holds row r0 + 32 r1 of atom
row ar, block j of column group ac at byte 16 r0 + 4 r1 + j."""
import numpy as np
import pytest
import torch

import moe_synth
from gpu_helpers import assert_close, dev_bf16
from oracle import moe_fp8_ref as q8
from oracle import moe_mx_ref as mx
from oracle import moe_ref

pytestmark = pytest.mark.gpu
L = pytest.importorskip("mixture_experts_grouped_router_gb300._lib")
FMT = {L.FP8_E4M3: q8.E4M3, L.FP8_E5M2: q8.E5M2}


def _blocky(rng, rows, cols, spread=5):
    """bf16 bits of N(0,1) values with every 32-element block of a row scaled
    by its own power of two in [2^-spread, 2^spread]."""
    p = rng.integers(-spread, spread + 1, size=(rows, cols // 32, 1))
    v = rng.standard_normal((rows, cols // 32, 32)) * np.ldexp(1.0, p)
    return moe_synth.bf16_bits(v.reshape(rows, cols).astype(np.float32))


def _atom_rows_plain(rows):
    return np.arange(rows)


def _atom_rows_grouped(off):
    """Padded position of every row of the groups."""
    pos = []
    p = 0
    for e in range(len(off) - 1):
        n = int(off[e + 1] - off[e])
        pos.extend(range(p, p + n))
        p += (n + 127) // 128 * 128
    return np.array(pos, np.int64)


def _atom_rows_swiglu(rows):
    """SwiGLU tiles of the B operand: tile t = gate rows [96t, 96t + 96) then up
    rows, at padded rows 256 t (192-row tiles take two atom rows)."""
    F = rows // 2
    r = np.arange(rows)
    n = np.where(r < F, r, r - F)
    return (n // 96) * 256 + np.where(r < F, 0, 96) + n % 96


def _atom_rows_tiles(rows, groups):
    """B operands in 192-row tiles per group of rows / groups rows."""
    G = rows // groups
    r = np.arange(rows)
    e, n = r // G, r % G
    return (e * ((G + 191) // 192) + n // 192) * 256 + n % 192


def _expected_sf(scales, pos, cols, nbytes):
    """Place the oracle's scale codes [rows, cols / 32] at their atom bytes."""
    out = np.full(nbytes, -1, np.int32)
    rows = scales.shape[0]
    for r in range(rows):
        pr = int(pos[r])
        ar, rw = pr // 128, pr % 128
        for cb in range(cols // 32):
            atom = ar * (cols // 128) + cb // 4
            out[atom * 512 + (rw % 32) * 16 + (rw // 32) * 4 + cb % 4] = scales[r, cb]
    return out


def _quantize_gpu(x_bits, fmt, row_map=L.MX_ROWS_PLAIN, off=None, groups=1):
    rows, cols = x_bits.shape
    x = dev_bf16(x_bits)
    q = torch.full((rows, cols), 0xAB, dtype=torch.uint8, device="cuda")
    E = groups if off is None else len(off) - 1
    nb = L.moe_mx_scale_bytes(rows, cols, row_map, E)
    sf = torch.full((nb,), 0xCD, dtype=torch.uint8, device="cuda")
    offd = None if off is None else torch.from_numpy(np.asarray(off, np.int32)).cuda()
    L.moe_mx_quantize(x, fmt, q, sf, row_map=row_map, group_offsets=offd, groups=groups)
    return q, sf


@pytest.mark.parametrize("fmt", [L.FP8_E4M3, L.FP8_E5M2])
@pytest.mark.parametrize("row_map", [L.MX_ROWS_PLAIN, L.MX_ROWS_GROUPED, L.MX_ROWS_SWIGLU,
                                     L.MX_ROWS_TILES])
def test_mx_quantize(fmt, row_map):
    rng = np.random.default_rng(fmt * 3 + row_map)
    rows, cols = (448, 384) if row_map == L.MX_ROWS_SWIGLU else (300, 256)
    x_bits = _blocky(rng, rows, cols, spread=40)
    # special blocks: zeros, a subnormal-range block, saturating values, NaN, infinity
    x_bits[3, 0:32] = 0
    x_bits[5, 32:64] = moe_synth.bf16_bits(np.full(32, 3e-39, np.float32))
    x_bits[7, 64:96] = moe_synth.bf16_bits((rng.standard_normal(32) * 1e30).astype(np.float32))
    x_bits[9, 96] = 0x7FC0
    x_bits[11, 128] = 0x7F80
    off = None
    if row_map == L.MX_ROWS_GROUPED:
        off = np.array([0, 7, 7, 140, 290, 290], np.int64)   # rows 290..299 are past the groups
        pos = _atom_rows_grouped(off)
        n_rows = int(off[-1])
    elif row_map == L.MX_ROWS_SWIGLU:
        pos, n_rows = _atom_rows_swiglu(rows), rows
    elif row_map == L.MX_ROWS_TILES:
        pos, n_rows = _atom_rows_tiles(rows, 3), rows      # 3 groups of 100 rows
    else:
        pos, n_rows = _atom_rows_plain(rows), rows
    q, sf = _quantize_gpu(x_bits, fmt, row_map, off, groups=3 if row_map == L.MX_ROWS_TILES else 1)
    torch.cuda.synchronize()
    codes, scales = mx.mx_quantize(moe_synth.bits_to_f64(x_bits[:n_rows]), FMT[fmt])
    got_q = q.cpu().numpy()
    assert (got_q[:n_rows] == codes).all()
    if n_rows < rows:
        assert (got_q[n_rows:] == 0xAB).all(), "rows past the groups were written"
    want = _expected_sf(scales, pos, cols, sf.numel())
    got = sf.cpu().numpy().astype(np.int32)
    written = want >= 0
    assert (got[written] == want[written]).all()


@pytest.mark.parametrize("case", ["acts_plain", "acts_tiles", "weights_swiglu",
                                  "weights_tiles"])
def test_mx_quantize_2x(case):
    """Both copies from one read equal the oracle's block quantization of the
    row-wise matrix and of the padded column-wise copy, codes and scales."""
    rng = np.random.default_rng(len(case))
    fmt = L.FP8_E5M2 if case == "acts_tiles" else L.FP8_E4M3
    if case.startswith("acts"):
        sizes = [0, 7, 300, 128, 129, 0, 1, 64]
        cols = 256
        off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)
        rows = int(off[-1]) + 21
        q_map, q_groups = L.MX_ROWS_GROUPED, len(sizes)
        qt_map = L.MX_ROWS_PLAIN if case == "acts_plain" else L.MX_ROWS_TILES
        qt_cols = L.moe_fp8_padded_rows(rows, len(sizes))
    else:
        E, G = 3, 256
        cols = 384 if case == "weights_swiglu" else 256
        off = np.arange(0, E * G + 1, G).astype(np.int64)
        rows = E * G
        q_map, q_groups = L.MX_ROWS_TILES, E
        qt_map = L.MX_ROWS_SWIGLU if case == "weights_swiglu" else L.MX_ROWS_TILES
        qt_cols = E * G
    E = len(off) - 1
    x_bits = _blocky(rng, rows, cols, spread=20)
    x_bits[2, 0:32] = 0
    x_bits[int(off[-1]) - 1, 5] = 0x7FC0                  # a NaN in the last group's last row
    R = int(off[-1])
    q = torch.full((rows, cols), 0xAB, dtype=torch.uint8, device="cuda")
    sfq = torch.full((L.moe_mx_scale_bytes(rows, cols, q_map, q_groups),), 0xCD,
                     dtype=torch.uint8, device="cuda")
    qt = torch.full((cols, qt_cols), 0xAB, dtype=torch.uint8, device="cuda")
    sfqt = torch.full((L.moe_mx_scale_bytes(cols, qt_cols, qt_map, 1),), 0xCD, dtype=torch.uint8,
                      device="cuda")
    L.moe_mx_quantize_2x(dev_bf16(x_bits), fmt, torch.from_numpy(off.astype(np.int32)).cuda(),
                         q, sfq, q_map, qt, sfqt, qt_map, qt_cols=qt_cols)
    torch.cuda.synchronize()
    # row-wise: the oracle's blocks along each row
    codes, scales = mx.mx_quantize(moe_synth.bits_to_f64(x_bits[:R]), FMT[fmt])
    assert (q.cpu().numpy()[:R] == codes).all()
    assert (q.cpu().numpy()[R:] == 0xAB).all()
    pos = _atom_rows_grouped(off) if q_map == L.MX_ROWS_GROUPED else _atom_rows_tiles(rows, E)
    want = _expected_sf(scales, pos[:R], cols, sfq.numel())
    got = sfq.cpu().numpy().astype(np.int32)
    assert (got[want >= 0] == want[want >= 0]).all()
    # column-wise: the oracle's blocks along the padded copy's rows
    ct_bits = np.zeros((cols, qt_cols), np.uint16)
    ppos = _atom_rows_grouped(off)
    ct_bits[:, ppos] = x_bits[:R].T
    used = (int(ppos[-1]) + 128) // 128 * 128 if R else 0       # through the last group's padding
    codes_t, scales_t = mx.mx_quantize(moe_synth.bits_to_f64(ct_bits[:, :used]), FMT[fmt])
    got_t = qt.cpu().numpy()
    assert (got_t[:, :used] == codes_t).all()
    assert (got_t[:, used:] == 0xAB).all()
    tpos = {L.MX_ROWS_PLAIN: _atom_rows_plain, L.MX_ROWS_TILES: lambda n: _atom_rows_tiles(n, 1),
            L.MX_ROWS_SWIGLU: _atom_rows_swiglu}[qt_map](cols)
    full_scales = np.full((cols, qt_cols // 32), -1, np.int64)
    full_scales[:, :used // 32] = scales_t
    want_t = _expected_sf(full_scales, tpos, qt_cols, sfqt.numel())
    got_t_sf = sfqt.cpu().numpy().astype(np.int32)
    assert (got_t_sf[want_t >= 0] == want_t[want_t >= 0]).all()


SIZES = {"mixed": [0, 7, 300, 128, 129, 0, 1, 640], "one": [517], "tiny": [1, 2, 3]}


def _off(sizes):
    return np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)


def _deq_rows(bits, fmt):
    return mx.mx_qdq(moe_synth.bits_to_f64(bits), FMT[fmt])


@pytest.mark.parametrize("sz,K,N", [("mixed", 256, 256), ("one", 384, 160), ("tiny", 128, 416),
                                    ("mixed", 128, 192)])
@pytest.mark.parametrize("fmts", [(L.FP8_E4M3, L.FP8_E4M3), (L.FP8_E5M2, L.FP8_E4M3)])
@pytest.mark.parametrize("c_f32", [False, True])
@pytest.mark.parametrize("by_cols", [False, True])
def test_gmm_mx_none(sz, K, N, fmts, c_f32, by_cols):
    """B [E, N, K] quantized as the [E*N, K] matrix (192-row tiles per expert),
    or (by_cols) as the [N, E*K] matrix of the transposed weights (expert e's
    K columns at e*K)."""
    rng = np.random.default_rng(K + N + fmts[0])
    off = _off(SIZES[sz])
    E, R = len(SIZES[sz]), int(off[-1])
    rows_cap = R + 29
    a_bits = _blocky(rng, rows_cap, K)
    qa, sfa = _quantize_gpu(a_bits, fmts[0], L.MX_ROWS_GROUPED, off)
    C = torch.full((rows_cap, N), 7.0, dtype=torch.float32 if c_f32 else torch.bfloat16,
                   device="cuda")
    offd = torch.from_numpy(off.astype(np.int32)).cuda()
    if by_cols:
        bt_bits = _blocky(rng, N, E * K)
        qb, sfb = _quantize_gpu(bt_bits, fmts[1], L.MX_ROWS_TILES, groups=1)
        L.moe_gmm_mx(qa, sfa, fmts[0], qb, sfb, 1, fmts[1], offd, C, E=E, N=N, K=K,
                     ldb=E * K, stride_b=K)
        bt_dq = _deq_rows(bt_bits, fmts[1])
        b_dq = np.stack([bt_dq[:, e * K:(e + 1) * K] for e in range(E)])   # [E, N, K]
    else:
        b_bits = _blocky(rng, E * N, K)             # B [E, N, K] as one [E*N, K] matrix
        qb, sfb = _quantize_gpu(b_bits, fmts[1], L.MX_ROWS_TILES, groups=E)
        L.moe_gmm_mx(qa, sfa, fmts[0], qb.view(E, N, K), sfb, 0, fmts[1], offd, C)
        b_dq = _deq_rows(b_bits, fmts[1]).reshape(E, N, K)
    torch.cuda.synchronize()
    a_dq = _deq_rows(a_bits[:R], fmts[0])
    want = moe_ref.gmm(a_dq, b_dq, off, transpose_rhs=True)
    # fp32 output: only the order of the fp32 sums differs; bf16: one rounding more
    tol = dict(rel_fro=1e-4, max_rel=1e-3) if c_f32 else dict(rel_fro=4e-3, max_rel=1e-2)
    assert_close("gmm_mx", C[:R], want, **tol)
    assert (C[R:].float() == 7.0).all()


@pytest.mark.parametrize("sz,K,F", [("mixed", 256, 128), ("one", 128, 224), ("tiny", 384, 96),
                                    ("mixed", 128, 320)])
def test_gmm_mx_swiglu_fwd(sz, K, F):
    """B is the [2F, E*K] matrix of the transposed fused weight (expert e's K
    columns at e*K), scales in SwiGLU tile order."""
    rng = np.random.default_rng(K * F)
    off = _off(SIZES[sz])
    E, R = len(SIZES[sz]), int(off[-1])
    rows_cap = R + 5
    a_bits = _blocky(rng, rows_cap, K)
    bt_bits = _blocky(rng, 2 * F, E * K)
    qa, sfa = _quantize_gpu(a_bits, L.FP8_E4M3, L.MX_ROWS_GROUPED, off)
    qb, sfb = _quantize_gpu(bt_bits, L.FP8_E4M3, L.MX_ROWS_SWIGLU)
    H = torch.empty(rows_cap, 2 * F, dtype=torch.bfloat16, device="cuda")
    Act = torch.empty(rows_cap, F, dtype=torch.bfloat16, device="cuda")
    offd = torch.from_numpy(off.astype(np.int32)).cuda()
    L.moe_gmm_mx(qa, sfa, L.FP8_E4M3, qb, sfb, 1, L.FP8_E4M3, offd, H,
                 L.EPI_SWIGLU_FWD, C2=Act, E=E, N=2 * F, K=K, ldb=E * K, stride_b=K)
    torch.cuda.synchronize()
    a_dq = _deq_rows(a_bits[:R], L.FP8_E4M3)
    bt_dq = _deq_rows(bt_bits, L.FP8_E4M3)                        # [2F, E*K]
    w = np.stack([bt_dq[:, e * K:(e + 1) * K].T for e in range(E)])  # [E, K, 2F]
    h = moe_ref.gmm(a_dq, w, off)
    assert_close("H", H[:R], h, rel_fro=4e-3, max_rel=1e-2)
    assert_close("Act", Act[:R], moe_ref.swiglu(h), rel_fro=4e-3, max_rel=1e-2)


@pytest.mark.parametrize("sz,K,F", [("mixed", 256, 128), ("one", 128, 256), ("tiny", 256, 224)])
def test_gmm_mx_swiglu_bwd(sz, K, F):
    rng = np.random.default_rng(K + 3 * F)
    off = _off(SIZES[sz])
    E, R = len(SIZES[sz]), int(off[-1])
    rows_cap = R + 3
    a_bits = _blocky(rng, rows_cap, K, spread=3)
    b_bits = _blocky(rng, E * F, K, spread=3)        # wo [E, F, K]: dgrad reads it K-major
    h_bits = moe_synth.bf16_bits((rng.standard_normal((rows_cap, 2 * F)) * 2).astype(np.float32))
    qa, sfa = _quantize_gpu(a_bits, L.FP8_E5M2, L.MX_ROWS_GROUPED, off)
    qb, sfb = _quantize_gpu(b_bits, L.FP8_E4M3, L.MX_ROWS_TILES, groups=E)
    dH = torch.empty(rows_cap, 2 * F, dtype=torch.bfloat16, device="cuda")
    offd = torch.from_numpy(off.astype(np.int32)).cuda()
    L.moe_gmm_mx(qa, sfa, L.FP8_E5M2, qb.view(E, F, K), sfb, 0, L.FP8_E4M3, offd, dH,
                 L.EPI_SWIGLU_BWD, aux=dev_bf16(h_bits))
    torch.cuda.synchronize()
    d_act = moe_ref.gmm(_deq_rows(a_bits[:R], L.FP8_E5M2),
                        _deq_rows(b_bits, L.FP8_E4M3).reshape(E, F, K), off, transpose_rhs=True)
    want = moe_ref.swiglu_bwd(moe_synth.bits_to_f64(h_bits)[:R], d_act)
    assert_close("dH", dH[:R], want, rel_fro=4e-3, max_rel=1e-2)


def _padded_colwise(bits, off):
    """Host copy of the padded column-wise layout: [cols, P] with group e's rows
    at columns [poff_e, poff_e + size_e), zeros elsewhere."""
    E = len(off) - 1
    P = L.moe_fp8_padded_rows(bits.shape[0], E)
    out = np.zeros((bits.shape[1], P), np.uint16)
    pos = _atom_rows_grouped(off)
    out[:, pos] = bits[:int(off[-1])].T
    return out, pos


@pytest.mark.parametrize("sz,M,N", [("mixed", 256, 128), ("one", 128, 256), ("tiny", 128, 416)])
@pytest.mark.parametrize("mode", ["bf16", "f32_acc"])
def test_tgmm_mx(sz, M, N, mode):
    rng = np.random.default_rng(M + N + len(mode))
    off = _off(SIZES[sz])
    E, R = len(SIZES[sz]), int(off[-1])
    rows_cap = R + 11
    a_bits = _blocky(rng, rows_cap, M, spread=3)
    b_bits = _blocky(rng, rows_cap, N, spread=3)
    At_bits, pos = _padded_colwise(a_bits, off)
    Bt_bits, _ = _padded_colwise(b_bits, off)
    qa, sfa = _quantize_gpu(At_bits, L.FP8_E4M3)
    qb, sfb = _quantize_gpu(Bt_bits, L.FP8_E5M2, L.MX_ROWS_TILES, groups=1)
    dt = torch.float32 if mode == "f32_acc" else torch.bfloat16
    W0 = rng.standard_normal((E, M, N)).astype(np.float32)
    W = torch.from_numpy(W0).cuda().to(dt)
    offd = torch.from_numpy(off.astype(np.int32)).cuda()
    L.moe_tgmm_mx(qa, sfa, L.FP8_E4M3, qb, sfb, L.FP8_E5M2, offd, rows_cap, W,
                  accumulate=mode == "f32_acc")
    torch.cuda.synchronize()
    a_dq = _deq_rows(At_bits, L.FP8_E4M3)[:, pos].T          # back to [R, M]
    b_dq = _deq_rows(Bt_bits, L.FP8_E5M2)[:, pos].T
    want = moe_ref.tgmm(a_dq, b_dq, off, E,
                        partial_sum=W0.astype(np.float64) if mode == "f32_acc" else None)
    got = W.float().cpu().numpy()
    for e in range(E):
        if SIZES[sz][e] == 0:
            assert (got[e] == (W0[e] if mode == "f32_acc" else 0)).all()
        else:
            assert_close("tgmm_mx[%d]" % e, got[e], want[e], rel_fro=4e-3, max_rel=1e-2)


# ---------------------------------------------------------------------------
# the MXFP8 layer against the MXFP8 oracle
# ---------------------------------------------------------------------------
C = moe_synth.CONFIGS
MX_LAYERS = {
    "mixtral": moe_synth.scaled(C["mixtral"], T=1024, d=256, f=384),
    "dsv3": moe_synth.scaled(C["dsv3"], T=512, d=384, f=256),
    "skewed": moe_synth.scaled(C["skewed"], T=4096, d=256, f=128, capacity=64),
    "odd": moe_synth.MoEConfig("odd", T=999, d=256, f=128, E=7, k=3, score_fn=1, renorm=0,
                               align=16, capacity=300),
}


def _rel(a, b):
    a = a.detach().float().cpu().numpy().astype(np.float64) if isinstance(a, torch.Tensor) else a
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def _max_rel(a, b):
    a = a.detach().float().cpu().numpy().astype(np.float64) if isinstance(a, torch.Tensor) else a
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-300))


@pytest.mark.parametrize("name", list(MX_LAYERS))
def test_layer_mxfp8(name):
    """The MXFP8 layer follows the block-scaled recipe: every output within
    1e-2 (relative Frobenius) and 5e-2 * max|ref| (elementwise) of the MXFP8
    oracle, and at most half as far from it as the oracle is from the
    unquantized layer; the integer layout is exact."""
    import dataclasses
    from gpu_helpers import layer_shape
    from mixture_experts_grouped_router_gb300 import layer
    cfg = MX_LAYERS[name]
    inp = moe_synth.make_inputs(cfg, seed=4)
    f64 = moe_synth.bits_to_f64
    x, wi, wo, dout = (dev_bf16(inp[n]) for n in ("x", "wi", "wo", "dout"))
    logits = torch.from_numpy(inp["logits"]).cuda()
    b = layer.MoEBuffers(dataclasses.replace(layer_shape(cfg), mxfp8=True))
    layer.forward(b, x, logits, wi, wo)
    layer.backward(b, dout, wi, wo)
    torch.cuda.synchronize()
    assert int(b.dev_status.item()) == 0
    xs, wis, wos, douts = (f64(inp[n]) for n in ("x", "wi", "wo", "dout"))
    fm = mx.forward(xs, inp["logits"], wis, wos, cfg.k, cfg.score_fn, cfg.renorm, cfg.align,
                    cfg.capacity)
    bm = mx.backward(fm, douts, wis, wos, cfg.k)
    fr = moe_ref.forward(xs, inp["logits"], wis, wos, cfg.k, cfg.score_fn, cfg.renorm,
                         cfg.align, cfg.capacity)
    br = moe_ref.backward(fr, douts, wis, wos, cfg.k)
    assert (b.topk_idx.cpu().numpy() == fm["topk_idx"]).all()
    assert b.group_offsets.cpu().numpy().tolist() == fm["layout"]["group_offsets"].tolist()
    R = fm["layout"]["R"]
    errs = {}
    for key, got, want, ref in (
            ("h", b.h[:R], fm["h"], fr["h"][:R]), ("act", b.act[:R], fm["act"], fr["act"][:R]),
            ("out", b.out, fm["out"], fr["out"]), ("dy", b.dy[:R], bm["dy"], br["dy"][:R]),
            ("dh", b.dh[:R], bm["dh"], br["dh"][:R]), ("dx", b.dx, bm["dx"], br["dx"]),
            ("dwi", b.dwi, bm["d_wi"], br["d_wi"]), ("dwo", b.dwo, bm["d_wo"], br["d_wo"]),
            ("d_topk_w", b.d_topk_w, bm["d_topk_w"], br["d_topk_w"])):
        errs[key] = (_rel(got, want), _rel(want, ref), _max_rel(got, want))
    bad = {k: v for k, v in errs.items()
           if not (v[0] <= 1e-2 and v[0] <= 0.5 * max(v[1], 1e-3) and v[2] <= 5e-2)}
    assert not bad, errs


def _qdq_rows(col, fmt):
    """Blocks of 32 along a column of one expert's rows, aligned at its first
    row and completed with zeros (the weight gradients' operands)."""
    n = col.shape[0]
    pad = np.zeros(((n + 31) // 32 * 32,) + col.shape[1:])
    pad[:n] = col
    return mx.qdq_along(pad, 0, fmt)[:n]


def test_layer_mxfp8_full_size_sampled():
    """The Mixtral-like layer at full size with block-scaled GEMMs, as
    `bench.py --mxfp8` runs it, against the MXFP8 oracle at sampled positions
    the oracle computes one by one (block scaling is local: a sampled column
    needs only its own blocks): the layout exactly; H, Act and dH of expert 0
    and 5 on sampled columns (every row of the expert); dWi and dWo on sampled
    rows x columns.  Tolerances 1e-2 (relative Frobenius) and 5e-2 * max|ref|
    over each sampled block."""
    import dataclasses
    from gpu_helpers import layer_shape
    from mixture_experts_grouped_router_gb300 import layer
    cfg = C["mixtral"]
    T, d, f, E, k = cfg.T, cfg.d, cfg.f, cfg.E, cfg.k
    inp = moe_synth.make_inputs(cfg, seed=0)
    x, wi, wo, dout = (dev_bf16(inp[n]) for n in ("x", "wi", "wo", "dout"))
    logits = torch.from_numpy(inp["logits"]).cuda()
    b = layer.MoEBuffers(dataclasses.replace(layer_shape(cfg), mxfp8=True))
    layer.forward(b, x, logits, wi, wo)
    layer.backward(b, dout, wi, wo)
    torch.cuda.synchronize()
    assert int(b.dev_status.item()) == 0
    del wi, wo, x, dout
    idx, w = moe_ref.route_topk(inp["logits"], k, cfg.score_fn, cfg.renorm)
    lay = moe_ref.permute_layout(idx, E)
    off = lay["group_offsets"]
    assert b.group_offsets.cpu().numpy().tolist() == off.tolist()
    assert b.s2f.cpu().numpy()[:lay["R"]].tolist() == lay["sorted_to_flat"].tolist()
    f64 = moe_synth.bits_to_f64
    e4, e5 = q8.E4M3, q8.E5M2
    rng = np.random.default_rng(11)
    for e in (0, 5):
        lo, hi = int(off[e]), int(off[e + 1])
        a = lay["sorted_to_flat"][lo:hi]                 # the expert's assignments, in order
        t, j = a // k, a % k
        xs = f64(inp["x"][t])                            # [n_e, d]
        xsq = mx.qdq_along(xs, 1, e4)                     # blocks along d (up-projection A)
        cg = np.sort(rng.choice(f, 4, replace=False))     # sampled gate / up columns
        cols = np.concatenate([cg, f + cg])
        ci = torch.as_tensor(cols, device="cuda")
        wiq = mx.qdq_along(f64(inp["wi"][e][:, cols]), 0, e4)  # [d, 8], blocks along d
        h = xsq @ wiq                                     # [n_e, 2 * 4]: gate cols, up cols
        assert_close("h[e=%d]" % e, b.h[lo:hi][:, ci], h)
        act = q8.round_bf16(moe_ref.swiglu(h))            # [n_e, 4]
        assert_close("act[e=%d]" % e, b.act[lo:hi][:, ci[:4]], act)
        # backward: dY rows = w * dOut of the token (bf16), blocks along d
        dy = q8.round_bf16(w[t, j][:, None] * f64(inp["dout"][t]))
        dyq = mx.qdq_along(dy, 1, e5)
        woq = mx.qdq_along(f64(inp["wo"][e][cg]), 1, e4)  # rows cg of [f, d], blocks along d
        d_act = dyq @ woq.T                               # [n_e, 4]
        dh = q8.round_bf16(moe_ref.swiglu_bwd(q8.round_bf16(h), d_act))   # [dg | du]
        assert_close("dh[e=%d]" % e, b.dh[lo:hi][:, ci], dh)
        # weight gradients on sampled rows x columns, operands blocked along the expert's rows
        rd = np.sort(rng.choice(d, 3, replace=False))
        ri = torch.as_tensor(rd, device="cuda")
        dwi = _qdq_rows(xs[:, rd], e4).T @ _qdq_rows(dh, e5)          # [3, 8]
        assert_close("dwi[e=%d]" % e, b.dwi[e][ri][:, ci], dwi)
        dwo = _qdq_rows(act, e4).T @ _qdq_rows(dy[:, rd], e5)          # [4, 3]
        assert_close("dwo[e=%d]" % e, b.dwo[e][ci[:4]][:, ri], dwo)
