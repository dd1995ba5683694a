"""Block-scaled FP8 (MXFP8) on the GPU against the block-scaled oracle
(oracle/moe_mx_ref.py):

* moe_mx_quantize: codes and E8M0 scales bit-exact, in the scale-atom layout
  of every row order (plain, grouped with padded expert tiles, SwiGLU tiles),
  with zero, subnormal, saturating and non-finite blocks;
* moe_gmm_mx (each epilogue) and moe_tgmm_mx against the oracle's grouped
  GEMMs of the dequantized operands.  Every 32-element block is scaled by its
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
    F = rows // 2
    r = np.arange(rows)
    n = np.where(r < F, r, r - F)
    return (n // 64) * 128 + np.where(r < F, 0, 64) + n % 64


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


def _quantize_gpu(x_bits, fmt, row_map=L.MX_ROWS_PLAIN, off=None):
    rows, cols = x_bits.shape
    x = dev_bf16(x_bits)
    q = torch.full((rows, cols), 0xAB, dtype=torch.uint8, device="cuda")
    E = 1 if off is None else len(off) - 1
    nb = L.moe_mx_scale_bytes(rows, cols, row_map, E)
    sf = torch.full((nb,), 0xCD, dtype=torch.uint8, device="cuda")
    offd = None if off is None else torch.from_numpy(np.asarray(off, np.int32)).cuda()
    L.moe_mx_quantize(x, fmt, q, sf, row_map=row_map, group_offsets=offd)
    return q, sf


@pytest.mark.parametrize("fmt", [L.FP8_E4M3, L.FP8_E5M2])
@pytest.mark.parametrize("row_map", [L.MX_ROWS_PLAIN, L.MX_ROWS_GROUPED, L.MX_ROWS_SWIGLU])
def test_mx_quantize(fmt, row_map):
    rng = np.random.default_rng(fmt * 3 + row_map)
    rows, cols = (256, 384) if row_map == L.MX_ROWS_SWIGLU else (300, 256)
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
    else:
        pos, n_rows = _atom_rows_plain(rows), rows
    q, sf = _quantize_gpu(x_bits, fmt, row_map, off)
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


SIZES = {"mixed": [0, 7, 300, 128, 129, 0, 1, 640], "one": [517], "tiny": [1, 2, 3]}


def _off(sizes):
    return np.concatenate([[0], np.cumsum(sizes)]).astype(np.int64)


def _deq_rows(bits, fmt):
    return mx.mx_qdq(moe_synth.bits_to_f64(bits), FMT[fmt])


@pytest.mark.parametrize("sz,K,N", [("mixed", 256, 256), ("one", 384, 128), ("tiny", 128, 384)])
@pytest.mark.parametrize("fmts", [(L.FP8_E4M3, L.FP8_E4M3), (L.FP8_E5M2, L.FP8_E4M3)])
@pytest.mark.parametrize("c_f32", [False, True])
def test_gmm_mx_none(sz, K, N, fmts, c_f32):
    rng = np.random.default_rng(K + N + fmts[0])
    off = _off(SIZES[sz])
    E, R = len(SIZES[sz]), int(off[-1])
    rows_cap = R + 29
    a_bits = _blocky(rng, rows_cap, K)
    b_bits = _blocky(rng, E * N, K)                 # B [E, N, K] as one [E*N, K] matrix
    qa, sfa = _quantize_gpu(a_bits, fmts[0], L.MX_ROWS_GROUPED, off)
    qb, sfb = _quantize_gpu(b_bits, fmts[1])
    C = torch.full((rows_cap, N), 7.0, dtype=torch.float32 if c_f32 else torch.bfloat16,
                   device="cuda")
    offd = torch.from_numpy(off.astype(np.int32)).cuda()
    L.moe_gmm_mx(qa, sfa, fmts[0], qb.view(E, N, K), sfb, K // 128, N * K // 16384, fmts[1],
                 offd, C)
    torch.cuda.synchronize()
    a_dq = _deq_rows(a_bits[:R], fmts[0])
    b_dq = _deq_rows(b_bits, fmts[1]).reshape(E, N, K)
    want = moe_ref.gmm(a_dq, b_dq, off, transpose_rhs=True)
    # fp32 output: only the order of the fp32 sums differs; bf16: one rounding more
    tol = dict(rel_fro=1e-4, max_rel=1e-3) if c_f32 else dict(rel_fro=4e-3, max_rel=1e-2)
    assert_close("gmm_mx", C[:R], want, **tol)
    assert (C[R:].float() == 7.0).all()


@pytest.mark.parametrize("sz,K,F", [("mixed", 256, 128), ("one", 128, 192), ("tiny", 384, 64)])
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
    L.moe_gmm_mx(qa, sfa, L.FP8_E4M3, qb, sfb, E * K // 128, K // 128, L.FP8_E4M3, offd, H,
                 L.EPI_SWIGLU_FWD, C2=Act, E=E, N=2 * F, K=K, ldb=E * K, stride_b=K)
    torch.cuda.synchronize()
    a_dq = _deq_rows(a_bits[:R], L.FP8_E4M3)
    bt_dq = _deq_rows(bt_bits, L.FP8_E4M3)                        # [2F, E*K]
    w = np.stack([bt_dq[:, e * K:(e + 1) * K].T for e in range(E)])  # [E, K, 2F]
    h = moe_ref.gmm(a_dq, w, off)
    assert_close("H", H[:R], h, rel_fro=4e-3, max_rel=1e-2)
    assert_close("Act", Act[:R], moe_ref.swiglu(h), rel_fro=4e-3, max_rel=1e-2)


@pytest.mark.parametrize("sz,K,F", [("mixed", 256, 128), ("one", 128, 256)])
def test_gmm_mx_swiglu_bwd(sz, K, F):
    rng = np.random.default_rng(K + 3 * F)
    off = _off(SIZES[sz])
    E, R = len(SIZES[sz]), int(off[-1])
    rows_cap = R + 3
    a_bits = _blocky(rng, rows_cap, K, spread=3)
    b_bits = _blocky(rng, E * F, K, spread=3)        # wo [E, F, K]: dgrad reads it K-major
    h_bits = moe_synth.bf16_bits((rng.standard_normal((rows_cap, 2 * F)) * 2).astype(np.float32))
    qa, sfa = _quantize_gpu(a_bits, L.FP8_E5M2, L.MX_ROWS_GROUPED, off)
    qb, sfb = _quantize_gpu(b_bits, L.FP8_E4M3)
    dH = torch.empty(rows_cap, 2 * F, dtype=torch.bfloat16, device="cuda")
    offd = torch.from_numpy(off.astype(np.int32)).cuda()
    L.moe_gmm_mx(qa, sfa, L.FP8_E5M2, qb.view(E, F, K), sfb, K // 128, F * K // 16384,
                 L.FP8_E4M3, offd, dH, L.EPI_SWIGLU_BWD, aux=dev_bf16(h_bits))
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


@pytest.mark.parametrize("sz,M,N", [("mixed", 256, 128), ("one", 128, 256), ("tiny", 128, 128)])
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
    qb, sfb = _quantize_gpu(Bt_bits, L.FP8_E5M2)
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
