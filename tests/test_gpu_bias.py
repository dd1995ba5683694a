"""GPU parity of the expert-FFN biases against the oracle: the bias epilogue
of moe_gmm (plain and SwiGLU forward, with and without a partial sum,
transposed weights), the per-expert column sums of moe_group_colsum (empty
experts give exact zeros; rows past the last group are never read), and the
whole layer with biases, forward and backward.

The biases follow the MLP-bias variant of the chunked grouped matmul
(MaxText PR #4295, "Overlap moe comms with collective matmul", Testing):
bi on [gate | up] after the up-projection, bo on the down-projection's output,
every row of expert e's group (padding rows included) receiving row e."""
import numpy as np
import pytest
import torch

import moe_synth
from gpu_helpers import assert_close, check_layout, dev_bf16, run_gpu_layer, run_oracle
from oracle import moe_ref

pytestmark = pytest.mark.gpu
L = pytest.importorskip("mixture_experts_grouped_router_gb300._lib")

SIZES = {
    "mixed": [0, 7, 300, 128, 129, 0, 1, 640],
    "one": [517],
    "tiny": [1, 2, 3],
}


def _offsets(sizes):
    return np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)


def _bf(rng, shape, scale=1.0):
    return moe_synth.bf16_bits((rng.standard_normal(shape) * scale).astype(np.float32))


GMM_BIAS_CASES = [("mixed", 256, 384, 0), ("mixed", 264, 200, 1), ("one", 1000, 136, 0),
                  ("tiny", 64, 64, 1)]


@pytest.mark.parametrize("case", GMM_BIAS_CASES)
@pytest.mark.parametrize("c_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("with_ps", [False, True])
def test_gmm_bias_none(case, c_dtype, with_ps):
    sz, K, N, tb = case
    rng = np.random.default_rng(K * 3 + N)
    off = _offsets(SIZES[sz])
    E, R = len(SIZES[sz]), int(off[-1])
    rows_cap = R + 21
    a_bits = _bf(rng, (rows_cap, K))
    b_bits = _bf(rng, (E, N, K) if tb else (E, K, N), 0.05)
    # bias rows padded to a stride of N + 24 (a view that is not contiguous in N)
    bias_full = _bf(rng, (E, N + 24), 0.7)
    bias = dev_bf16(bias_full)[:, :N]
    ps = ps64 = None
    if with_ps:
        ps_np = rng.standard_normal((rows_cap, N)).astype(np.float32)
        ps, ps64 = torch.from_numpy(ps_np).cuda(), ps_np[:R].astype(np.float64)
    C = torch.full((rows_cap, N), 7.0, dtype=c_dtype, device="cuda")
    L.moe_gmm(dev_bf16(a_bits), dev_bf16(b_bits), tb, torch.from_numpy(off).cuda(), C,
              partial_sum=ps, bias=bias)
    torch.cuda.synchronize()
    f64 = moe_synth.bits_to_f64
    want = moe_ref.gmm(f64(a_bits)[:R], f64(b_bits), off, transpose_rhs=bool(tb),
                       partial_sum=ps64)
    want = moe_ref.add_group_bias(want, f64(bias_full)[:, :N], off)
    assert_close("gmm+bias", C[:R], want)
    assert (C[R:].float() == 7.0).all(), "rows past the last group were written"


@pytest.mark.parametrize("sz,K,F", [("mixed", 256, 192), ("one", 136, 200), ("tiny", 64, 64)])
@pytest.mark.parametrize("with_ps", [False, True])
def test_gmm_bias_swiglu_fwd(sz, K, F, with_ps):
    rng = np.random.default_rng(K + 7 * F)
    off = _offsets(SIZES[sz])
    E, R = len(SIZES[sz]), int(off[-1])
    rows_cap = R + 9
    a_bits = _bf(rng, (rows_cap, K))
    b_bits = _bf(rng, (E, K, 2 * F), 0.05)
    bi_bits = _bf(rng, (E, 2 * F), 0.7)
    ps = ps64 = None
    if with_ps:
        ps_np = (rng.standard_normal((rows_cap, 2 * F)) * 0.5).astype(np.float32)
        ps, ps64 = torch.from_numpy(ps_np).cuda(), ps_np[:R].astype(np.float64)
    H = torch.empty(rows_cap, 2 * F, dtype=torch.bfloat16, device="cuda")
    Act = torch.empty(rows_cap, F, dtype=torch.bfloat16, device="cuda")
    L.moe_gmm(dev_bf16(a_bits), dev_bf16(b_bits), 0, torch.from_numpy(off).cuda(), H,
              L.EPI_SWIGLU_FWD, partial_sum=ps, C2=Act, bias=dev_bf16(bi_bits))
    torch.cuda.synchronize()
    f64 = moe_synth.bits_to_f64
    h = moe_ref.gmm(f64(a_bits)[:R], f64(b_bits), off, partial_sum=ps64)
    h = moe_ref.add_group_bias(h, f64(bi_bits), off)
    assert_close("H", H[:R], h)
    assert_close("Act", Act[:R], moe_ref.swiglu(h))


@pytest.mark.parametrize("sz,N,ld_extra", [("mixed", 200, 0), ("mixed", 1032, 8), ("one", 520, 0),
                                           ("tiny", 8, 16), ("mixed", 4096, 0)])
def test_group_colsum(sz, N, ld_extra):
    rng = np.random.default_rng(N + ld_extra)
    off = _offsets(SIZES[sz])
    E, R = len(SIZES[sz]), int(off[-1])
    rows_cap = R + 13
    g_bits = _bf(rng, (rows_cap, N + ld_extra), 2.0)
    G = dev_bf16(g_bits)
    G[R:] = float("nan")          # rows past the last group must not be read
    out = torch.full((E, N + 4), 123.0, dtype=torch.float32, device="cuda")
    L.moe_group_colsum(G[:, :N], torch.from_numpy(off).cuda(), out[:, :N])
    torch.cuda.synchronize()
    want = moe_ref.group_colsum(moe_synth.bits_to_f64(g_bits)[:R, :N], off, E)
    got = out[:, :N]
    assert_close("colsum", got, want, rel_fro=1e-5, max_rel=1e-5)
    for e in np.nonzero(np.diff(off) == 0)[0]:
        assert (got[e] == 0).all()
    assert (out[:, N:] == 123.0).all()


def test_group_colsum_no_rows():
    off = torch.zeros(4, dtype=torch.int32, device="cuda")
    out = torch.full((3, 16), 5.0, dtype=torch.float32, device="cuda")
    G = torch.empty(0, 16, dtype=torch.bfloat16, device="cuda")
    L.moe_group_colsum(G, off, out)
    torch.cuda.synchronize()
    assert (out == 0).all()


C = moe_synth.CONFIGS
LAYER_CASES = {
    "mixtral": moe_synth.scaled(C["mixtral"], T=1024, d=256, f=448),
    "dsv3_chunked": moe_synth.scaled(C["dsv3_chunked"], T=512, d=448, f=256),
    "odd_sizes": moe_synth.MoEConfig("odd_sizes", T=999, d=200, f=136, E=7, k=3, score_fn=1,
                                     renorm=0, align=16, capacity=300),
}


@pytest.mark.parametrize("name", list(LAYER_CASES))
def test_layer_with_biases(name):
    cfg = LAYER_CASES[name]
    inp = moe_synth.make_inputs(cfg, seed=1)
    biases = moe_synth.make_biases(cfg, seed=1)
    b = run_gpu_layer(cfg, inp, biases=biases)
    assert int(b.dev_status.item()) == 0
    fw, bw = run_oracle(cfg, inp, biases=biases)
    check_layout(b, fw, cfg.T, cfg.k)
    R = fw["layout"]["R"]
    assert_close("h", b.h[:R], fw["h"])
    assert_close("y", b.y[:R], fw["y"])
    assert_close("out", b.out, fw["out"])
    assert_close("d_topk_w", b.d_topk_w, bw["d_topk_w"])
    assert_close("dh", b.dh[:R], bw["dh"])
    assert_close("dx", b.dx, bw["dx"])
    assert_close("dwo", b.dwo, bw["d_wo"])
    assert_close("dwi", b.dwi, bw["d_wi"])
    assert_close("dbi", b.dbi, bw["d_bi"])
    assert_close("dbo", b.dbo, bw["d_bo"])
