"""GPU parity of moe_combine (weighted and weight-less) and moe_unpermute_bwd
against the oracle, on bf16 inputs shared by both sides."""
import numpy as np
import pytest
import torch

import moe_synth
from gpu_helpers import assert_close, dev_bf16
from oracle import moe_ref

pytestmark = pytest.mark.gpu
L = pytest.importorskip("mixture_experts_grouped_router_gb300._lib")

CASES = [
    # T, d, E, k, align, cap
    (1, 8, 2, 1, 0, 0), (333, 200, 8, 2, 0, 0), (1000, 1024, 32, 8, 0, 0),
    (777, 520, 64, 1, 128, 20), (500, 64, 16, 4, 8, 40), (64, 4096, 4, 2, 0, 0),
]


def _setup(T, d, E, k, align, cap, seed):
    rng = np.random.default_rng(seed)
    lg = (rng.standard_normal((T, E)) + np.linspace(-2, 2, E)).astype(np.float32)
    idx, w = moe_ref.route_topk(lg, k, 1, 1)
    lay = moe_ref.permute_layout(idx, E, align, cap)
    rows_cap = moe_ref.rows_cap(T, E, k, align)
    y_bits = moe_synth.bf16_bits(rng.standard_normal((rows_cap, d)).astype(np.float32))
    dout_bits = moe_synth.bf16_bits(rng.standard_normal((T, d)).astype(np.float32))
    s2f = np.full(rows_cap, -1, np.int32)
    s2f[:lay["R"]] = lay["sorted_to_flat"]
    off = lay["group_offsets"].astype(np.int32)
    return lg, idx, w.astype(np.float32), lay, rows_cap, y_bits, dout_bits, s2f, off


@pytest.mark.parametrize("case", CASES)
def test_combine_and_dispatch_bwd(case):
    T, d, E, k, align, cap = case
    lg, idx, w32, lay, rows_cap, y_bits, _, _, _ = _setup(*case, seed=T + d)
    Y = dev_bf16(y_bits)
    f2s = torch.from_numpy(lay["flat_to_sorted"].astype(np.int32)).cuda()
    wt = torch.from_numpy(w32).cuda()
    out = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    L.moe_combine(Y, f2s, wt, out, k)
    dx = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    L.moe_combine(Y, f2s, None, dx, k)
    torch.cuda.synchronize()
    y64 = moe_synth.bits_to_f64(y_bits)
    assert_close("combine", out, moe_ref.combine(y64, lay["flat_to_sorted"], w32.astype(np.float64)))
    assert_close("dispatch_bwd", dx, moe_ref.dispatch_bwd(y64, lay["flat_to_sorted"], T, k))


@pytest.mark.parametrize("case", CASES)
def test_unpermute_bwd(case):
    T, d, E, k, align, cap = case
    lg, idx, w32, lay, rows_cap, y_bits, dout_bits, s2f, off = _setup(*case, seed=T * 3 + d)
    Y = dev_bf16(y_bits)
    dout = dev_bf16(dout_bits)
    dY = torch.full((rows_cap, d), float("nan"), dtype=torch.bfloat16, device="cuda")
    dw = torch.full((T, k), float("nan"), dtype=torch.float32, device="cuda")
    L.moe_unpermute_bwd(dout, Y, torch.from_numpy(lay["flat_to_sorted"].astype(np.int32)).cuda(),
                        torch.from_numpy(s2f).cuda(), torch.from_numpy(off).cuda(),
                        torch.from_numpy(w32).cuda(), dY, dw)
    torch.cuda.synchronize()
    R = lay["R"]
    rdy, rdw = moe_ref.combine_bwd(moe_synth.bits_to_f64(dout_bits), moe_synth.bits_to_f64(y_bits),
                                   lay["flat_to_sorted"], w32.astype(np.float64), R)
    assert_close("dY", dY[:R], rdy)
    assert_close("d_topk_w", dw, rdw)
    # padding rows exactly zero, dropped slots exactly zero
    pad = lay["sorted_to_flat"] < 0
    assert (dY[:R].float().cpu().numpy()[pad] == 0).all()
    drop = lay["flat_to_sorted"].reshape(T, k) < 0
    assert (dw.cpu().numpy()[drop] == 0).all()
