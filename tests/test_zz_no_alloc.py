"""moe_permute_noalloc against moe_permute (GPU).

moe_permute_noalloc serves callers that cannot allocate device memory where
they permute (operator plugins that receive only their input and output
buffers, processes whose device memory is reserved up front by their own
pool): it keeps its scratch counters in an array owned by the library instead
of a caller-provided workspace.  This file is named so that pytest collects it
last; it must pass alone in a fresh process and after the other tests.
"""
import numpy as np
import pytest
import torch

import moe_synth
from gpu_helpers import dev_bf16
from oracle import moe_ref

pytestmark = pytest.mark.gpu
L = pytest.importorskip("mixture_experts_grouped_router_gb300._lib")


def _buffers(T, d, E, k, align):
    rows_cap = L.moe_rows_cap(T, E, k, align)
    dev = "cuda"
    return dict(
        xs=torch.full((rows_cap, d), float("nan"), dtype=torch.bfloat16, device=dev),
        gs=torch.full((E,), -7, dtype=torch.int32, device=dev),
        kc=torch.full((E,), -7, dtype=torch.int32, device=dev),
        off=torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
        s2f=torch.full((rows_cap,), -7, dtype=torch.int32, device=dev),
        f2s=torch.full((T * k,), -7, dtype=torch.int32, device=dev),
        st=torch.zeros(1, dtype=torch.int32, device=dev))


def _case(seed, T, d, E, k, align, cap):
    rng = np.random.default_rng(seed)
    lg = (rng.standard_normal((T, E)) + np.linspace(-3, 3, E)).astype(np.float32)
    idx, _ = moe_ref.route_topk(lg, k, 0, 1)
    x_bits = moe_synth.bf16_bits(rng.standard_normal((T, d)).astype(np.float32))
    return torch.from_numpy(idx.astype(np.int32)).cuda(), dev_bf16(x_bits)


def _compare(a, b, R):
    for key in ("gs", "kc", "off", "f2s", "st"):
        assert torch.equal(a[key], b[key]), key
    assert torch.equal(a["s2f"], b["s2f"])
    assert torch.equal(a["xs"][:R].view(torch.int16), b["xs"][:R].view(torch.int16))


@pytest.mark.parametrize("T,d,E,k,align,cap", [(3000, 136, 64, 2, 16, 80),
                                              (32512, 64, 256, 4, 8, 0)])
def test_noalloc_matches_workspace_version_twice(T, d, E, k, align, cap):
    for call, seed in enumerate((11, 12)):   # two calls in a row, different inputs
        idx, x = _case(seed + T, T, d, E, k, align, cap)
        ref = _buffers(T, d, E, k, align)
        ws = torch.empty(L.moe_permute_workspace_bytes(T, E), dtype=torch.uint8, device="cuda")
        L.moe_permute(x, idx, E, align, cap, ref["xs"], ref["gs"], ref["kc"], ref["off"],
                      ref["s2f"], ref["f2s"], ws, ref["st"])
        got = _buffers(T, d, E, k, align)
        L.moe_permute_noalloc(x, idx, E, align, cap, got["xs"], got["gs"], got["kc"],
                              got["off"], got["s2f"], got["f2s"], got["st"])
        torch.cuda.synchronize()
        assert int(got["st"].item()) == 0, "call %d" % call
        _compare(got, ref, int(ref["off"][-1].item()))


def test_noalloc_rejects_sizes_beyond_its_array():
    T, E, k, d = 40000, 256, 1, 8   # 157 count blocks * 256 experts > 32704 counters
    b = _buffers(8, d, E, k, 0)
    idx = torch.zeros(T, k, dtype=torch.int32, device="cuda")
    x = torch.zeros(T, d, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(L.MoEError) as ei:
        L.moe_permute_noalloc(x, idx, E, 0, 0, torch.empty(T * k, d, dtype=torch.bfloat16,
                                                          device="cuda"),
                              b["gs"], b["kc"], b["off"],
                              torch.empty(T * k, dtype=torch.int32, device="cuda"),
                              torch.empty(T * k, dtype=torch.int32, device="cuda"))
    assert ei.value.status == L.MOE_ERR_UNSUPPORTED
    assert "scratch" in str(ei.value)
