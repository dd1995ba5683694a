"""The benchmark's roofline accounting (CPU): algorithmic bytes of the
data-moving kernels and FLOPs of the expert GEMMs, pinned to the figures the
layer's definition gives for two workloads, and to the rows and indices each
kernel must read and write on a small routed layout.

Formulas (bf16 = 2 bytes, index = 4 bytes): permute (T_kept + R)·d·2 + 8·T·k + 4·R;
combine M·d·2 + T·d·2 + 8·T·k; combine backward T_kept·d·2 + 2·M·d·2 + (R−M)·d·2 + 8·T·k;
dispatch backward M·d·2 + T·d·2 + 4·T·k; GEMMs 18·M·d·f per forward + backward.
"""
import pytest

import bench
import moe_synth
from oracle import moe_ref

pytestmark = pytest.mark.filterwarnings("ignore")


@pytest.mark.parametrize("name,mb", [
    # no token dropped, no padding: T_kept = T, M = R = T k
    ("mixtral", dict(permute=403.0, combine=403.0, unpermute_bwd=671.0, dispatch_bwd=403.0)),
    ("dsv3", dict(permute=1058.0, combine=1057.0, unpermute_bwd=1997.0, dispatch_bwd=1057.0)),
])
def test_bytes_of_the_full_workloads(name, mb):
    cfg = moe_synth.CONFIGS[name]
    M = R = cfg.T * cfg.k
    got = bench.algorithmic_bytes(cfg, M, R, cfg.T)
    for kernel, want in mb.items():
        assert abs(got[kernel] / 1e6 - want) < 1.0, (kernel, got[kernel] / 1e6, want)


@pytest.mark.parametrize("name,tflop", [("mixtral", 34.63), ("dsv3", 17.32)])
def test_gemm_flops_of_the_full_workloads(name, tflop):
    cfg = moe_synth.CONFIGS[name]
    M = cfg.T * cfg.k
    fl = bench.gemm_flops_per_launch(cfg, M)
    step = sum(fl[n] for n in ("gmm_up_swiglu", "gmm_down", "gmm_dgrad_down_swiglu_bwd",
                               "tgmm_dwo", "gmm_dgrad_up", "tgmm_dwi"))
    assert step == 18 * M * cfg.d * cfg.f
    assert abs(step / 1e12 - tflop) < 0.01


def test_bytes_match_the_counts_of_a_routed_layout():
    """The bytes each kernel must move, summed from the counts of a small routed
    layout with capacity drops and align padding (rows read and written, index
    arrays), against the benchmark's formulas."""
    cfg = moe_synth.MoEConfig("count", T=40, d=16, f=8, E=4, k=2, score_fn=0, renorm=1,
                              align=8, capacity=9)
    inp = moe_synth.make_inputs(cfg, seed=3)
    idx, _ = moe_ref.route_topk(inp["logits"], cfg.k, cfg.score_fn, cfg.renorm)
    lay = moe_ref.permute_layout(idx, cfg.E, cfg.align, cfg.capacity)
    T, k, d = cfg.T, cfg.k, cfg.d
    f2s = lay["flat_to_sorted"].reshape(T, k)
    R = int(lay["R"])
    M = int((f2s >= 0).sum())
    t_kept = int((f2s >= 0).any(axis=1).sum())
    assert M < T * k and R > M                          # drops and padding present
    row = d * 2
    permute = t_kept * row + R * row + T * k * 4 + T * k * 4 + R * 4   # x rows in, Xs rows out
    combine = M * row + T * row + T * k * 4 + T * k * 4                  # Y rows, out, f2s, w
    unperm = t_kept * row + M * row + M * row + (R - M) * row + T * k * 4 + T * k * 4
    dispatch = M * row + T * row + T * k * 4
    got = bench.algorithmic_bytes(cfg, M, R, t_kept)
    assert got["permute"] == permute
    assert got["combine"] == combine
    assert got["unpermute_bwd"] == unperm
    assert got["dispatch_bwd"] == dispatch


def test_gemm_bytes_and_bound():
    """Least DRAM bytes of the GEMM launches (operands read once, outputs written
    once): at Mixtral size every GEMM is far above the ridge point of the measured
    peaks (tensor-bound); in the skewed workload (about 100 rows per expert) the
    weight gradients fall below it (HBM-bound: writing 64 bf16 weight gradients
    takes longer than their FLOPs)."""
    cfg = moe_synth.CONFIGS["mixtral"]
    R = M = cfg.T * cfg.k
    d, f, E = cfg.d, cfg.f, cfg.E
    gb = bench.gemm_bytes_per_launch(cfg, R)
    # dWi: Xs and dH read, dWi written
    assert gb["tgmm_dwi"] == 2 * (R * d + R * 2 * f) + 2 * E * d * 2 * f
    assert abs(gb["tgmm_dwi"] / 1e9 - 4.027) < 1e-3   # 0.268 + 1.879 + 1.879 GB
    # SwiGLU backward: dY, wo and H read, dH written
    assert gb["gmm_dgrad_down_swiglu_bwd"] == 2 * (R * d + E * f * d) + 4 * R * 2 * f
    pk, _ = bench.peaks()
    ridge = pk["bf16_tflops_sustained"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    fl = bench.gemm_flops_per_launch(cfg, M)
    assert all(fl[n] / gb[n] > 4 * ridge for n in ("gmm_up_swiglu", "gmm_down", "tgmm_dwo",
                                                   "gmm_dgrad_up", "tgmm_dwi"))
    sk = moe_synth.CONFIGS["skewed"]
    M_sk, R_sk = 5405, 53 * 128          # kept rows and aligned rows of the skewed layer
    fl_sk = bench.gemm_flops_per_launch(sk, M_sk)
    gb_sk = bench.gemm_bytes_per_launch(sk, R_sk)
    assert fl_sk["tgmm_dwi"] / gb_sk["tgmm_dwi"] < ridge / 2
    # 8-bit operands halve the operand bytes, not the bf16 outputs
    gb8 = bench.gemm_bytes_per_launch(cfg, R, 1)
    assert gb["tgmm_dwi"] - gb8["tgmm_dwi"] == R * d + R * 2 * f
