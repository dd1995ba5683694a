"""GPU parity of the grouped GEMMs moe_gmm / moe_tgmm against the oracle's
gmm / tgmm on shared bf16 inputs: ragged groups (empty, below one tile,
several tiles with a ragged tail), K and N that are not tile multiples,
transposed weights, each epilogue, the in-place fp32 partial sum, and exact
zeros for empty groups in tgmm."""
import numpy as np
import pytest
import torch

import moe_synth
from gpu_helpers import assert_close, dev_bf16, host_f64
from oracle import moe_ref

pytestmark = pytest.mark.gpu
L = pytest.importorskip("mixture_experts_grouped_router_gb300._lib")

SIZES = {
    "mixed": [0, 7, 300, 128, 129, 0, 1, 640],
    "one": [517],
    "tiny": [1, 2, 3],
    "empty_tail": [256, 0, 0],
}


def _offsets(sizes):
    return np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)


def _bf(rng, shape, scale=1.0):
    return moe_synth.bf16_bits((rng.standard_normal(shape) * scale).astype(np.float32))


def _setup(sizes, K, N, trans_b, seed, extra_rows=37):
    rng = np.random.default_rng(seed)
    off = _offsets(sizes)
    E = len(sizes)
    rows_cap = int(off[-1]) + extra_rows
    a_bits = _bf(rng, (rows_cap, K))
    b_shape = (E, N, K) if trans_b else (E, K, N)
    b_bits = _bf(rng, b_shape, 0.05)
    a64 = moe_synth.bits_to_f64(a_bits)
    b64 = moe_synth.bits_to_f64(b_bits)
    return rng, off, rows_cap, a_bits, b_bits, a64, b64


GMM_CASES = [
    ("mixed", 256, 384, 0), ("mixed", 264, 200, 1), ("one", 1000, 136, 0), ("tiny", 64, 64, 1),
    ("empty_tail", 512, 1024, 0), ("mixed", 128, 520, 1),
]


@pytest.mark.parametrize("case", GMM_CASES)
@pytest.mark.parametrize("c_dtype", [torch.bfloat16, torch.float32])
def test_gmm_none(case, c_dtype):
    sz, K, N, tb = case
    rng, off, rows_cap, a_bits, b_bits, a64, b64 = _setup(SIZES[sz], K, N, tb, seed=K + N)
    C = torch.full((rows_cap, N), 7.0, dtype=c_dtype, device="cuda")
    L.moe_gmm(dev_bf16(a_bits), dev_bf16(b_bits), tb, torch.from_numpy(off).cuda(), C)
    torch.cuda.synchronize()
    R = int(off[-1])
    want = moe_ref.gmm(a64[:R], b64, off, transpose_rhs=bool(tb))
    assert_close("gmm", C[:R], want)
    assert (C[R:].float() == 7.0).all(), "rows past the last group were written"


@pytest.mark.parametrize("case", GMM_CASES[:4])
def test_gmm_partial_sum_in_place_and_out_of_place(case):
    sz, K, N, tb = case
    rng, off, rows_cap, a_bits, b_bits, a64, b64 = _setup(SIZES[sz], K, N, tb, seed=3 * K + N)
    R = int(off[-1])
    ps_np = rng.standard_normal((rows_cap, N)).astype(np.float32)
    P = torch.from_numpy(ps_np).cuda()
    offd = torch.from_numpy(off).cuda()
    out = torch.empty(rows_cap, N, dtype=torch.bfloat16, device="cuda")
    L.moe_gmm(dev_bf16(a_bits), dev_bf16(b_bits), tb, offd, out, partial_sum=P)
    L.moe_gmm(dev_bf16(a_bits), dev_bf16(b_bits), tb, offd, P, partial_sum=P)   # in place
    torch.cuda.synchronize()
    want = moe_ref.gmm(a64[:R], b64, off, transpose_rhs=bool(tb),
                       partial_sum=ps_np[:R].astype(np.float64))
    assert_close("gmm+ps (bf16 out)", out[:R], want)
    assert_close("gmm+ps (in place)", P[:R], want)
    assert (P[R:].cpu().numpy() == ps_np[R:]).all()


@pytest.mark.parametrize("sz,K,F", [("mixed", 256, 192), ("one", 136, 200), ("tiny", 64, 64),
                                    ("mixed", 520, 1024)])
@pytest.mark.parametrize("with_ps", [False, True])
def test_gmm_swiglu_fwd(sz, K, F, with_ps):
    rng, off, rows_cap, a_bits, b_bits, a64, b64 = _setup(SIZES[sz], K, 2 * F, 0, seed=K + F)
    R = int(off[-1])
    offd = torch.from_numpy(off).cuda()
    H = torch.empty(rows_cap, 2 * F, dtype=torch.bfloat16, device="cuda")
    Act = torch.empty(rows_cap, F, dtype=torch.bfloat16, device="cuda")
    ps = None
    ps64 = None
    if with_ps:
        ps_np = (rng.standard_normal((rows_cap, 2 * F)) * 0.5).astype(np.float32)
        ps = torch.from_numpy(ps_np).cuda()
        ps64 = ps_np[:R].astype(np.float64)
    L.moe_gmm(dev_bf16(a_bits), dev_bf16(b_bits), 0, offd, H, L.EPI_SWIGLU_FWD, partial_sum=ps,
              C2=Act)
    torch.cuda.synchronize()
    h = moe_ref.gmm(a64[:R], b64, off, partial_sum=ps64)
    assert_close("H", H[:R], h)
    assert_close("Act", Act[:R], moe_ref.swiglu(h))


@pytest.mark.parametrize("sz,K,F", [("mixed", 256, 192), ("one", 136, 200), ("tiny", 64, 64),
                                    ("mixed", 1024, 136)])
def test_gmm_swiglu_bwd(sz, K, F):
    # S = dY . wo^T  (trans_b: wo_e is [F, K]); aux H [rows, 2F]
    rng, off, rows_cap, a_bits, b_bits, a64, b64 = _setup(SIZES[sz], K, F, 1, seed=K * F)
    R = int(off[-1])
    h_bits = _bf(rng, (rows_cap, 2 * F), 2.0)
    dH = torch.empty(rows_cap, 2 * F, dtype=torch.bfloat16, device="cuda")
    L.moe_gmm(dev_bf16(a_bits), dev_bf16(b_bits), 1, torch.from_numpy(off).cuda(), dH,
              L.EPI_SWIGLU_BWD, aux=dev_bf16(h_bits))
    torch.cuda.synchronize()
    d_act = moe_ref.gmm(a64[:R], b64, off, transpose_rhs=True)
    want = moe_ref.swiglu_bwd(moe_synth.bits_to_f64(h_bits)[:R], d_act)
    assert_close("dH", dH[:R], want)


@pytest.mark.parametrize("sz,K,F", [("mixed", 256, 192), ("one", 136, 200), ("tiny", 64, 72),
                                    ("mixed", 520, 1024), ("empty_tail", 64, 264)])
@pytest.mark.parametrize("epi", [L.EPI_SWIGLU_FWD, L.EPI_SWIGLU_BWD])
def test_gmm_swiglu_colwise_copy(sz, K, F, epi):
    """The column-wise copy the SwiGLU epilogues write (Ct) holds exactly the
    bf16 values of the row-wise output, in the padded group layout, zeros in
    each group's padding, nothing past the last group; the row-wise outputs
    are bit-identical to a launch without the copy.  Rows of A past the groups
    are NaN: a tile's rows past its expert must reach the copy as zeros."""
    bwd = epi == L.EPI_SWIGLU_BWD
    rng, off, rows_cap, a_bits, b_bits, a64, b64 = _setup(SIZES[sz], K, F if bwd else 2 * F,
                                                          int(bwd), seed=5 * K + F)
    E, R = len(SIZES[sz]), int(off[-1])
    offd = torch.from_numpy(off).cuda()
    A = dev_bf16(a_bits)
    A[R:] = float("nan")
    Bw = dev_bf16(b_bits)
    P = L.moe_fp8_padded_rows(rows_cap, E)
    width = 2 * F if bwd else F
    outs = []
    for with_copy in (False, True):
        H = torch.full((rows_cap, 2 * F), 5.0, dtype=torch.bfloat16, device="cuda")
        Act = torch.full((rows_cap, F), 5.0, dtype=torch.bfloat16, device="cuda")
        Ct = torch.full((width, P + 8), float("nan"), dtype=torch.bfloat16, device="cuda")
        kw = dict(Ct=Ct[:, :P]) if with_copy else {}
        if bwd:
            aux = dev_bf16(_bf(rng, (rows_cap, 2 * F), 2.0)) if not outs else outs[0][3]
            L.moe_gmm(A, Bw, 1, offd, H, L.EPI_SWIGLU_BWD, aux=aux, **kw)
        else:
            aux = None
            L.moe_gmm(A, Bw, 0, offd, H, L.EPI_SWIGLU_FWD, C2=Act, **kw)
        torch.cuda.synchronize()
        outs.append((H, Act, Ct, aux))
    (H0, A0, _, _), (H1, A1, Ct, aux) = outs
    assert torch.equal(H0[:R].view(torch.int16), H1[:R].view(torch.int16))
    src = H1 if bwd else A1           # dH or Act, row-wise
    if not bwd:
        assert torch.equal(A0[:R].view(torch.int16), A1[:R].view(torch.int16))
        assert_close("Act", A1[:R], moe_ref.swiglu(moe_ref.gmm(a64[:R], b64, off)))
    else:
        d_act = moe_ref.gmm(a64[:R], b64, off, transpose_rhs=True)
        assert_close("dH", H1[:R], moe_ref.swiglu_bwd(host_f64(aux)[:R], d_act))
    got = Ct.view(torch.int16).cpu().numpy()
    rows = src.view(torch.int16).cpu().numpy()
    po = _poff(SIZES[sz])
    for e in range(E):
        a, b = int(off[e]), int(off[e + 1])
        assert (got[:, po[e]:po[e] + b - a] == rows[a:b, :width].T).all(), e
        assert (got[:, po[e] + b - a:po[e + 1]] == 0).all(), e
    # columns past the last group (and past P) are not written: still NaN (0x7fc0)
    assert (got[:, po[-1]:] == np.int16(0x7FC0)).all()


TGMM_CASES = [("mixed", 256, 384), ("one", 136, 200), ("tiny", 64, 64), ("empty_tail", 128, 520),
              ("mixed", 1024, 128)]


@pytest.mark.parametrize("sz,M,N", TGMM_CASES)
@pytest.mark.parametrize("mode", ["bf16", "f32", "f32_acc"])
def test_tgmm(sz, M, N, mode):
    sizes = SIZES[sz]
    rng = np.random.default_rng(M + N + len(mode))
    off = _offsets(sizes)
    E = len(sizes)
    rows_cap = int(off[-1]) + 19
    a_bits = _bf(rng, (rows_cap, M))
    b_bits = _bf(rng, (rows_cap, N))
    dt = torch.bfloat16 if mode == "bf16" else torch.float32
    W0 = rng.standard_normal((E, M, N)).astype(np.float32)
    W = torch.from_numpy(W0).cuda().to(dt)
    R = int(off[-1])
    A, B = dev_bf16(a_bits), dev_bf16(b_bits)
    # rows past the groups are never read: NaN there would reach W through
    # the ragged last K block of the last expert unless its tail is zeroed
    A[R:] = float("nan")
    B[R:] = float("nan")
    L.moe_tgmm(A, B, torch.from_numpy(off).cuda(), W, accumulate=(mode == "f32_acc"))
    torch.cuda.synchronize()
    ps = W0.astype(np.float64) if mode == "f32_acc" else None
    want = moe_ref.tgmm(moe_synth.bits_to_f64(a_bits)[:R], moe_synth.bits_to_f64(b_bits)[:R],
                        off, E, partial_sum=ps)
    got = host_f64(W)
    for e in range(E):
        if sizes[e] == 0:
            if mode == "f32_acc":
                assert (W[e].cpu().numpy() == W0[e]).all(), "empty group changed"
            else:
                assert (got[e] == 0).all(), "empty group not exactly zero"
        else:
            assert_close("tgmm[%d]" % e, got[e], want[e])


def test_gmm_rejects_bad_args_before_launch():
    a = torch.zeros(16, 12, dtype=torch.bfloat16, device="cuda")
    b = torch.zeros(1, 12, 16, dtype=torch.bfloat16, device="cuda")
    off = torch.zeros(2, dtype=torch.int32, device="cuda")
    c = torch.zeros(16, 16, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(L.MoEError) as ei:
        L.moe_gmm(a, b, 0, off, c)     # K = 12 is not a multiple of 8
    assert ei.value.status == L.MOE_ERR_UNSUPPORTED


# ---------------------------------------------------------------------------
# weight gradients from the column-wise copy of A (K-major operand)
# ---------------------------------------------------------------------------
def _poff(sizes, pad=128):
    p = [0]
    for s in sizes:
        p.append(p[-1] + (s + pad - 1) // pad * pad)
    return p


@pytest.mark.parametrize("sz,cols", [("mixed", 64), ("one", 200), ("tiny", 8), ("empty_tail", 136)])
def test_transpose_act_padded(sz, cols):
    rng = np.random.default_rng(cols + len(SIZES[sz]))
    off = _offsets(SIZES[sz])
    E, R = len(SIZES[sz]), int(off[-1])
    rows_cap = R + 9
    x_bits = _bf(rng, (rows_cap, cols))
    x = dev_bf16(x_bits)
    x[R:] = float("nan")
    P = L.moe_fp8_padded_rows(rows_cap, E)
    xt = torch.full((cols, P), 3.0, dtype=torch.bfloat16, device="cuda")
    L.moe_transpose_act(x, torch.from_numpy(off).cuda(), xt)
    torch.cuda.synchronize()
    got = xt.view(torch.int16).cpu().numpy().astype(np.uint16)
    po = _poff(SIZES[sz])
    for e in range(E):
        a, b = int(off[e]), int(off[e + 1])
        assert (got[:, po[e]:po[e] + b - a] == x_bits[a:b].T).all(), e
        assert (got[:, po[e] + b - a:po[e + 1]] == 0).all(), e


@pytest.mark.parametrize("sz,M,N", TGMM_CASES)
@pytest.mark.parametrize("mode", ["bf16", "f32", "f32_acc"])
@pytest.mark.parametrize("b_colwise", [False, True])
def test_tgmm_kt(sz, M, N, mode, b_colwise):
    rng = np.random.default_rng(M * 7 + N)
    off = _offsets(SIZES[sz])
    E, R = len(SIZES[sz]), int(off[-1])
    rows_cap = R + 37
    a_bits = _bf(rng, (rows_cap, M))
    b_bits = _bf(rng, (rows_cap, N))
    A = dev_bf16(a_bits)
    B = dev_bf16(b_bits)
    A[R:] = float("nan")          # rows past the groups are never read
    B[R:] = float("nan")
    offd = torch.from_numpy(off).cuda()
    At = torch.empty(M, L.moe_fp8_padded_rows(rows_cap, E), dtype=torch.bfloat16, device="cuda")
    L.moe_transpose_act(A, offd, At)
    dt = torch.bfloat16 if mode == "bf16" else torch.float32
    W = torch.full((E, M, N), 0.0, dtype=dt, device="cuda")
    init = None
    if mode == "f32_acc":
        init = rng.standard_normal((E, M, N)).astype(np.float32)
        W.copy_(torch.from_numpy(init))
    if b_colwise:
        Bt = torch.empty(N, L.moe_fp8_padded_rows(rows_cap, E), dtype=torch.bfloat16,
                         device="cuda")
        L.moe_transpose_act(B, offd, Bt)
        L.moe_tgmm_kt(At, Bt, offd, rows_cap, W, accumulate=mode == "f32_acc", b_colwise=True)
    else:
        L.moe_tgmm_kt(At, B, offd, rows_cap, W, accumulate=mode == "f32_acc")
    torch.cuda.synchronize()
    a64 = moe_synth.bits_to_f64(a_bits)
    b64 = moe_synth.bits_to_f64(b_bits)
    want = moe_ref.tgmm(a64[:R], b64[:R], off, E,
                        partial_sum=None if init is None else init.astype(np.float64))
    assert_close("tgmm_kt", W, want)
    if mode != "f32_acc":
        for e in np.nonzero(np.diff(off) == 0)[0]:
            assert (W[e].float() == 0).all()
