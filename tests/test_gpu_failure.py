"""Failure detection on the GPU without a GPU fault.

The grouped-GEMM kernels bound every pipeline wait.  A test hook makes their
copy role issue no loads, so the first wait runs out (a barrier that nothing
completes): the kernel must wind down, report MOE_ERR_TIMEOUT through the
device status word within about the configured limit, and leave the CUDA
context usable, which the next launch on the same stream checks against the
oracle.
"""
import time

import numpy as np
import pytest
import torch

import moe_synth
from gpu_helpers import assert_close, dev_bf16
from oracle import moe_ref

pytestmark = pytest.mark.gpu
L = pytest.importorskip("mixture_experts_grouped_router_gb300._lib")


def _case(seed=5):
    rng = np.random.default_rng(seed)
    sizes = [130, 0, 257, 64]
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    rows = int(off[-1]) + 16
    a = moe_synth.bf16_bits(rng.standard_normal((rows, 128)).astype(np.float32))
    b = moe_synth.bf16_bits((rng.standard_normal((4, 128, 256)) * 0.05).astype(np.float32))
    h = moe_synth.bf16_bits(rng.standard_normal((rows, 512)).astype(np.float32))
    return off, rows, a, b, h


def _run(kind, off, rows, a, b, h, st):
    offd = torch.from_numpy(off).cuda()
    if kind == "gmm":
        C = torch.zeros(rows, 256, dtype=torch.bfloat16, device="cuda")
        L.moe_gmm(dev_bf16(a), dev_bf16(b), 0, offd, C, dev_status=st)
    elif kind == "gmm_swiglu_bwd":
        C = torch.zeros(rows, 512, dtype=torch.bfloat16, device="cuda")
        L.moe_gmm(dev_bf16(a), dev_bf16(b), 0, offd, C, L.EPI_SWIGLU_BWD, aux=dev_bf16(h),
                  dev_status=st)
    else:
        C = torch.zeros(4, 128, 256, dtype=torch.bfloat16, device="cuda")
        L.moe_tgmm(dev_bf16(a), dev_bf16(h[:, :256]), offd, C, dev_status=st)
    return C


@pytest.mark.parametrize("kind", ["gmm", "gmm_swiglu_bwd", "tgmm"])
def test_wait_timeout_reports_status_and_context_survives(kind):
    off, rows, a, b, h = _case()
    default = L.moe_wait_limit_ns()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    L.moe_set_wait_limit_ns(20_000_000)          # 20 ms
    L.moe_test_stall_loads(True)
    try:
        t0 = time.perf_counter()
        _run(kind, off, rows, a, b, h, st)
        torch.cuda.synchronize()
        elapsed = time.perf_counter() - t0
    finally:
        L.moe_test_stall_loads(False)
        L.moe_set_wait_limit_ns(default)
    assert int(st.item()) == L.MOE_ERR_TIMEOUT
    assert elapsed < 5.0
    # the context is still usable: the same call now completes and is right
    st2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    C = _run(kind, off, rows, a, b, h, st2)
    torch.cuda.synchronize()
    assert int(st2.item()) == 0
    R = int(off[-1])
    a64, b64, h64 = (moe_synth.bits_to_f64(v) for v in (a, b, h))
    if kind == "gmm":
        assert_close("gmm after timeout", C[:R], moe_ref.gmm(a64[:R], b64, off))
    elif kind == "gmm_swiglu_bwd":
        d_act = moe_ref.gmm(a64[:R], b64, off)
        assert_close("dH after timeout", C[:R], moe_ref.swiglu_bwd(h64[:R], d_act))
    else:
        assert_close("tgmm after timeout", C,
                     moe_ref.tgmm(a64[:R], h64[:R, :256], off, 4))
