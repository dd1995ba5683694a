"""GPU parity of the FP8 path against the FP8 oracle (oracle/moe_fp8_ref.py):
amax and scales, row-wise and column-wise codes (bit-exact; the column-wise
copy of a grouped activation with its per-group padding of zeros), the FP8
grouped GEMMs, and the FP8 layer.

The recipe is the pages' configuration of the expert GEMMs (MaxText PR #2319,
"[Draft] Integrate TE/JAX GroupedGEMM for MoE", review thread on the quantizer
settings: current tensor scaling, float8_e4m3fn forward, float8_e5m2
backward, row- and column-wise copies)."""
import numpy as np
import pytest
import torch

import moe_synth
from gpu_helpers import dev_bf16
from oracle import moe_fp8_ref as q8

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
