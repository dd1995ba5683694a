"""Benchmark of the MoE expert layer, forward + backward, on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl reference]

One step is one pass of the whole hot path over one batch of synthetic input:
route top-k -> permute -> grouped GEMM up (SwiGLU fused) -> grouped GEMM down
-> combine, then unpermute backward -> dgrad down (SwiGLU backward fused) ->
tgmm dWo -> dgrad up -> tgmm dWi -> dispatch backward.  The default workload
is the Mixtral-like expert layer (T=16384, d=4096, f=14336, E=8, top-2).

Prints one JSON line.  `value` is the expert-GEMM TFLOP/s of the whole job
(18 * M_kept * d * f per step, kept rows only) with inputs resident in HBM;
`e2e` is the same metric through the library's host-buffer entry point
(moe_layer_pipeline_step): each step's inputs are copied from pinned host memory
and its results copied back inside the timed region.  With --gpus N > 1 the
script runs under torchrun as N independent replicas (one per GPU, no data
exchange), timing is the max over ranks and `value` sums the work of all ranks.
--impl reference times the fp64 CPU oracle on a bounded sample of the same
workload instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import moe_synth  # noqa: E402

METRIC = "MoE FFN fwd+bwd TFLOP/s and tokens/s on 1 GB300; % of BF16 peak / HBM BW"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
GEMM_SOURCES = ["mixture_experts_grouped_router_gb300/csrc/gmm_sm103.cu",
                "mixture_experts_grouped_router_gb300/csrc/tc_sm103.cuh"]


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def gemm_source_hash():
    h = hashlib.sha256()
    for rel in GEMM_SOURCES:
        h.update(open(os.path.join(ROOT, rel), "rb").read())
    return h.hexdigest()[:16]


def reduce_over_ranks(ms_total, ms_e2e, flops_step, dist, device):
    """Replicas: the job's timed regions are the slowest rank's, its work the sum
    of every rank's (whole-job throughput = summed work / max time)."""
    import torch
    if dist is None:
        return ms_total, ms_e2e, flops_step
    t = torch.tensor([ms_total, ms_e2e], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    f = torch.tensor([flops_step], device=device, dtype=torch.float64)
    dist.all_reduce(f)
    return float(t[0].item()), float(t[1].item()), float(f.item())


def job_value(flops_job, steps, ms_total):
    """Whole-job TFLOP/s of `steps` steps that took ms_total (max over ranks)."""
    return flops_job * steps / (ms_total * 1e-3) / 1e12


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# ---------------------------------------------------------------------------
# CPU oracle sample (the cpu_baseline leg and --impl reference)
# ---------------------------------------------------------------------------
def oracle_sample(cfg, inp, n_tok, w64=None, groups=(0, 0)):
    """Run the oracle's forward + backward on the first n_tok tokens; returns
    (seconds, kept assignments, weights-in-fp64)."""
    from oracle import moe_ref
    f64 = moe_synth.bits_to_f64
    if w64 is None:
        w64 = (f64(inp["wi"]), f64(inp["wo"]))
    wi, wo = w64
    x = f64(inp["x"][:n_tok])
    dout = f64(inp["dout"][:n_tok])
    logits = inp["logits"][:n_tok]
    cap = cfg.capacity
    if cap > 0:   # same capacity factor on the sample
        cap = max(1, -(-cap * n_tok // cfg.T))
    t0 = time.perf_counter()
    fw = moe_ref.forward(x, logits, wi, wo, cfg.k, cfg.score_fn, cfg.renorm, cfg.align, cap,
                         cfg.num_chunks, num_groups=groups[0], topk_group=groups[1])
    moe_ref.backward(fw, dout, wi, wo, cfg.k, cfg.num_chunks)
    dt = time.perf_counter() - t0
    m_kept = int(fw["layout"]["kept_counts"].sum())
    return dt, m_kept, w64


def cpu_baseline(cfg, inp, target_s=12.0, groups=(0, 0)):
    """Time the oracle on a growing token sample until one run takes ~target_s
    (its cost is not linear in the tokens: every expert's weights are read)."""
    cores = len(os.sched_getaffinity(0))
    n = min(cfg.T, 64)
    dt, m_kept, w64 = oracle_sample(cfg, inp, n, groups=groups)
    while dt < target_s and n < cfg.T:
        n = int(min(cfg.T, n * max(2.0, min(8.0, 0.8 * target_s / max(dt, 1e-3)))))
        dt, m_kept, _ = oracle_sample(cfg, inp, n, w64, groups)
    flops = 18.0 * m_kept * cfg.d * cfg.f
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "tokens_per_s": n / dt, "seconds": dt,
            "sample": "fp64 NumPy oracle, forward+backward of the first %d of %d tokens with "
                      "the full expert weights (%d kept assignments)" % (n, cfg.T, m_kept)}


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", "moe_bench_clocks_%d_%d.csv" % (os.getpid(), gpu_index))

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, mx, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [c.strip() for c in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(mx),
                "power_w_median": float(np.median(power)), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def algorithmic_bytes(cfg, m_kept, R, t_kept):
    T, d, k, f, E = cfg.T, cfg.d, cfg.k, cfg.f, cfg.E
    return {
        # FP8: amax read + quantize read (bf16) + row-wise and column-wise codes;
        # Act and dH take their amax from the GEMM that wrote them (no amax read)
        "transpose_act": 4 * R * f, "transpose_xs": 4 * R * d, "transpose_dy": 4 * R * d,
        "quant_x": 6 * R * d, "quant_act": 4 * R * f, "quant_dy": 6 * R * d,
        "quant_dh": 4 * R * 2 * f, "quant_wi": 6 * E * d * 2 * f, "quant_wo": 6 * E * f * d,
        "colsum_dbo": R * d * 2 + E * d * 4,
        "colsum_dbi": R * 2 * f * 2 + E * 2 * f * 4,
        "permute": (t_kept + R) * d * 2 + 8 * T * k + 4 * R,
        "combine": m_kept * d * 2 + T * d * 2 + 8 * T * k,
        "unpermute_bwd": t_kept * d * 2 + 2 * m_kept * d * 2 + (R - m_kept) * d * 2 + 8 * T * k,
        "dispatch_bwd": m_kept * d * 2 + T * d * 2 + 4 * T * k,
    }


def gemm_bytes_per_launch(cfg, R, op_bytes=2):
    """Least DRAM bytes of each GEMM launch: every operand read once (op_bytes per
    element: 2 for bf16, 1 for 8-bit codes), every output written once in bf16
    (the weight gradients too).  R = the permuted rows the GEMMs run over."""
    d, f, E = cfg.d, cfg.f, cfg.E
    dc = d // max(1, cfg.num_chunks)
    o = op_bytes
    return {
        "gmm_up_swiglu": o * (R * d + E * d * 2 * f) + 2 * (R * 2 * f + R * f),
        "gmm_up_chunk": o * (R * dc + E * dc * 2 * f) + 4 * R * 2 * f * 2,
        "gmm_up_chunk_swiglu": o * (R * dc + E * dc * 2 * f) + 4 * R * 2 * f + 2 * 3 * R * f,
        "gmm_down": o * (R * f + E * f * d) + 2 * R * d,
        "gmm_dgrad_down_swiglu_bwd": o * (R * d + E * f * d) + 2 * (R * 2 * f * 2),
        "tgmm_dwo": o * (R * f + R * d) + 2 * E * f * d,
        "gmm_dgrad_up": o * (R * 2 * f + E * d * 2 * f) + 2 * R * d,
        "gmm_dgrad_up_chunk": o * (R * 2 * f + E * dc * 2 * f) + 2 * R * dc,
        "tgmm_dwi": o * (R * d + R * 2 * f) + 2 * E * d * 2 * f,
        "tgmm_dwi_chunk": o * (R * dc + R * 2 * f) + 2 * E * dc * 2 * f,
    }


def gemm_flops_per_launch(cfg, m_kept):
    M, d, f = m_kept, cfg.d, cfg.f
    dc = d // max(1, cfg.num_chunks)
    return {
        "gmm_up_swiglu": 4 * M * d * f,
        "gmm_up_chunk": 4 * M * dc * f,
        "gmm_up_chunk_swiglu": 4 * M * dc * f,
        "gmm_down": 2 * M * f * d,
        "gmm_dgrad_down_swiglu_bwd": 2 * M * d * f,
        "tgmm_dwo": 2 * M * f * d,
        "gmm_dgrad_up": 4 * M * d * f,
        "gmm_dgrad_up_chunk": 4 * M * dc * f,
        "tgmm_dwi": 4 * M * d * f,
        "tgmm_dwi_chunk": 4 * M * dc * f,
    }


def run_ours(args, cfg, ws, rank, local):
    import torch
    from mixture_experts_grouped_router_gb300 import _lib as L, layer

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    dist = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    inp = moe_synth.make_inputs(cfg, seed=rank)

    def bf16(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).astype(np.int16)).view(torch.bfloat16)

    x = bf16(inp["x"]).to(dev)
    wi = bf16(inp["wi"]).to(dev)
    wo = bf16(inp["wo"]).to(dev)
    dout = bf16(inp["dout"]).to(dev)
    logits = torch.from_numpy(inp["logits"]).to(dev)
    shape = layer.LayerShape(cfg.T, cfg.d, cfg.f, cfg.E, cfg.k, cfg.score_fn, cfg.renorm,
                             cfg.align, cfg.capacity, cfg.num_chunks, args.bias,
                             num_groups=args.num_groups, topk_group=args.topk_group,
                             aux_coeff=args.aux_coeff, fp8=args.fp8,
                             wgrad_colwise=args.wgrad_colwise, mxfp8=args.mxfp8)
    b = layer.MoEBuffers(shape, device=dev)
    stream = torch.cuda.current_stream(dev)
    bi = bo = None
    if args.bias:
        bias_inp = moe_synth.make_biases(cfg, seed=rank)
        bi, bo = bf16(bias_inp["bi"]).to(dev), bf16(bias_inp["bo"]).to(dev)

    def step(mark=layer._noop):
        layer.forward(b, x, logits, wi, wo, mark=mark, bi=bi, bo=bo)
        layer.backward(b, dout, wi, wo, mark=mark)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize(dev)
    status = int(b.dev_status.item())
    if status != 0:
        raise RuntimeError("device status %d after warm-up" % status)
    kept = b.kept_counts.cpu().numpy()
    m_kept = int(kept.sum())
    R = int(b.group_offsets[-1].item())
    f2s = b.f2s.view(cfg.T, cfg.k).cpu().numpy()
    t_kept = int((f2s >= 0).any(axis=1).sum())
    empty = int((b.group_sizes.cpu().numpy() == 0).sum())
    flops_step = 18.0 * m_kept * cfg.d * cfg.f

    # ---- timed region: K steps, inputs resident, events after every call
    marks = []

    def mark(name):
        e = torch.cuda.Event(enable_timing=True)
        e.record(stream)
        marks.append((name, e))

    sampler = ClockSampler(local if "CUDA_VISIBLE_DEVICES" not in os.environ else
                           int(os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local]))
    sampler.start()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    mark("start")
    for _ in range(args.steps):
        step(mark)
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    clocks = sampler.stop()
    ms_total = t_start.elapsed_time(t_end)
    per_kernel = {}
    for (_, e0), (name, e1) in zip(marks[:-1], marks[1:]):
        per_kernel.setdefault(name, []).append(e0.elapsed_time(e1))
    status = int(b.dev_status.item())
    if status != 0:
        raise RuntimeError("device status %d after the timed steps" % status)

    # ---- end to end, through the library's host-buffer entry point
    # (moe_layer_pipeline_step): every step's inputs are copied in from pinned
    # host memory and its results (out, dx, router-logit gradient) copied back
    # to pinned host memory, inside the timed region.  The library
    # double-buffers them on its own copy streams, so that step i+1's inputs
    # and step i's results move while the neighbouring steps compute.
    hx = bf16(inp["x"]).pin_memory()
    hlog = torch.from_numpy(inp["logits"]).pin_memory()
    hdout = bf16(inp["dout"]).pin_memory()
    hres = [dict(out=torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16).pin_memory(),
                 dx=torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16).pin_memory(),
                 d_logits=torch.empty(cfg.T, cfg.E, dtype=torch.float32).pin_memory())
            for _ in range(2)]
    staging = torch.empty(L.moe_layer_pipeline_workspace_bytes(b.cfg), dtype=torch.uint8,
                          device=dev)
    pipe = L.LayerPipeline(b.cfg, b.workspace, staging)

    def host_step(i):
        r = hres[i % 2]
        pipe.step(wi, wo, hx, hlog, hdout, r["out"], r["dx"], r["d_logits"], bi=bi, bo=bo,
                  stream=stream)

    for i in range(2):
        host_step(i)
    pipe.sync()
    torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        host_step(i)
    pipe.join(stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    pipe.close()
    ms_e2e = e0.elapsed_time(e1)
    status = int(b.dev_status.item())
    if status != 0:
        raise RuntimeError("device status %d after the end-to-end steps" % status)
    h2d_bytes = hx.numel() * 2 + hlog.numel() * 4 + hdout.numel() * 2
    d2h_bytes = sum(t.numel() * t.element_size() for t in hres[0].values())

    # ---- max over ranks
    ms_total, ms_e2e, flops_job = reduce_over_ranks(ms_total, ms_e2e, flops_step, dist, dev)
    if rank != 0:
        dist.destroy_process_group()
        return None

    ms_step = ms_total / args.steps
    value = job_value(flops_job, args.steps, ms_total)
    tokens_s = cfg.T * ws * args.steps / (ms_total * 1e-3)
    pk, pk_kind = peaks()
    kernels = {}
    fl = gemm_flops_per_launch(cfg, m_kept)
    by = algorithmic_bytes(cfg, m_kept, R, t_kept)
    for name, ts in per_kernel.items():
        launches_per_step = len(ts) / args.steps
        avg = float(np.mean(ts))
        ent = {"avg_ms": avg, "launches_per_step": launches_per_step,
               "share": sum(ts) / ms_total}
        if name in fl:
            ent["tflops"] = fl[name] / (avg * 1e-3) / 1e12
        if name in by:
            ent["gbs"] = by[name] / (avg * 1e-3) / 1e9
        kernels[name] = ent
    gemm_names = [n for n in kernels if n in fl]
    dom = max(gemm_names, key=lambda n: kernels[n]["share"])
    peak_t = pk.get("bf16_tflops_sustained", pk["bf16_tflops"])
    low = args.fp8 or args.mxfp8
    if low:   # measured bf16 peak x the nominal dense fp8 / bf16 ratio (4.5 / 2.25)
        peak_t *= 2.0
    traffic = None
    tp = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tp):
        tj = json.load(open(tp))
        ent = tj.get(cfg.name, {}).get(dom)
        if ent and ent.get("source_hash") == gemm_source_hash() and not args.bias \
                and not low:
            traffic = ent["dram_bytes_per_launch"]
    # the dominant GEMM's bound: its FLOPs per least DRAM byte against the ridge
    # point of the two peaks (few rows per expert make the weight gradient a
    # stream of weight-sized writes: HBM-bound)
    gb = gemm_bytes_per_launch(cfg, R, 1 if low else 2)
    ridge = peak_t * 1e12 / (pk["hbm_gbs"] * 1e9)
    if fl[dom] / gb[dom] >= ridge:
        roofline = {"bound": "tensor", "kernel": dom, "achieved": kernels[dom]["tflops"],
                    "peak": peak_t, "unit": "TFLOP/s", "frac": kernels[dom]["tflops"] / peak_t,
                    "traffic": traffic, "peak_kind": "%s sustained bf16 (burst %.1f)%s"
                    % (pk_kind, pk["bf16_tflops"], " x 2 (nominal fp8 / bf16)" if low else ""),
                    "algorithmic_per_launch": fl[dom], "algorithmic_unit": "FLOP"}
    else:
        gbs = gb[dom] / (kernels[dom]["avg_ms"] * 1e-3) / 1e9
        roofline = {"bound": "hbm", "kernel": dom, "achieved": gbs, "peak": pk["hbm_gbs"],
                    "unit": "GB/s", "frac": gbs / pk["hbm_gbs"], "traffic": traffic,
                    "peak_kind": "%s copy bandwidth" % pk_kind,
                    "algorithmic_per_launch": gb[dom], "algorithmic_unit": "byte",
                    "intensity_flop_per_byte": fl[dom] / gb[dom], "ridge_flop_per_byte": ridge,
                    "tflops": kernels[dom]["tflops"]}
    gemm_ms = sum(kernels[n]["avg_ms"] * kernels[n]["launches_per_step"] for n in gemm_names)
    mem = {}
    for n in by:
        if n in kernels:
            mem[n] = {"gbs": kernels[n]["gbs"], "frac": kernels[n]["gbs"] / pk["hbm_gbs"],
                      "bytes": by[n]}
    out = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "tokens_per_s": tokens_s,
        "n_gpus": ws, "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ("mxfp8 (e4m3 forward, e5m2 gradients, e8m0 scale per 32 elements), fp32 "
                  "accumulation" if args.mxfp8 else
                  "fp8 (e4m3 forward, e5m2 gradients), fp32 accumulation" if args.fp8 else "bf16"),
        "data": "synthetic (seeded N(0,1) activations / N(0,0.02) weights, rank-seeded)",
        "config": {"workload": cfg.name, "T": cfg.T, "d_model": cfg.d, "d_ff": cfg.f,
                   "experts": cfg.E, "top_k": cfg.k,
                   "score": "sigmoid" if cfg.score_fn else "softmax", "renorm": cfg.renorm,
                   "align": cfg.align, "capacity": cfg.capacity, "num_chunks": cfg.num_chunks,
                   "mlp_bias": bool(args.bias), "fp8": bool(args.fp8), "mxfp8": bool(args.mxfp8),
                   "wgrad_operands": ("column-wise FP8 codes (K-major)" if low else
                                      "column-wise bf16 copies (K-major)"
                                      if args.wgrad_colwise else "row-wise (MN-major)"),
                   "num_groups": args.num_groups, "topk_group": args.topk_group,
                   "aux_coeff": args.aux_coeff,
                   "m_kept": m_kept, "rows": R, "empty_experts": empty,
                   "gemm_tflop_per_step": flops_step / 1e12,
                   "l2": "inputs larger than L2 (weights %.2f GB)" % ((inp["wi"].nbytes +
                                                                     inp["wo"].nbytes) / 1e9),
                   "parallelism": "replicas" if ws > 1 else "single GPU"},
        "gemm_tflops": flops_step / (gemm_ms * 1e-3) / 1e12,
        "clocks": clocks,
        "e2e": {"value": flops_job * args.steps / (ms_e2e * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes,
                "ms_per_step": ms_e2e / args.steps,
                "api": "moe_layer_pipeline_step (C ABI, host buffers; the library's copy "
                       "streams overlap step i+1's inputs and step i's results with compute)"},
        "gpu_launches": layer.kernels_per_step(shape) * args.steps,
        "roofline": roofline,
        "hbm_kernels": mem,
        "kernels": kernels,
    }
    if not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline(cfg, inp, groups=(args.num_groups, args.topk_group))
    if dist is not None:
        dist.destroy_process_group()
    return out


def run_reference(args, cfg, ws, rank):
    if rank != 0:
        return None
    inp = moe_synth.make_inputs(cfg, seed=0)
    cores = len(os.sched_getaffinity(0))
    # size the per-step sample so that warm-up + steps end within a few minutes
    n0 = min(cfg.T, 32)
    groups = (args.num_groups, args.topk_group)
    dt0, _, w64 = oracle_sample(cfg, inp, n0, groups=groups)
    budget = 150.0 / max(1, args.steps + args.warmup)
    n = int(min(cfg.T, max(n0, n0 * budget / max(dt0, 1e-3))))
    for _ in range(args.warmup):
        oracle_sample(cfg, inp, n, w64, groups)
    secs, kept = 0.0, 0
    for _ in range(args.steps):
        dt, m_kept, _ = oracle_sample(cfg, inp, n, w64, groups)
        secs += dt
        kept = m_kept
    flops = 18.0 * kept * cfg.d * cfg.f
    value = flops * args.steps / secs / 1e12
    sample = ("fp64 NumPy oracle, forward+backward of the first %d of %d tokens with the full "
              "expert weights per step" % (n, cfg.T))
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
            "tokens_per_s": n * args.steps / secs, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": cfg.name, "T_sample": n},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="mixtral",
                    choices=sorted(moe_synth.CONFIGS) + sorted(moe_synth.PROFILE_CONFIGS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--num-groups", type=int, default=0,
                    help="group-limited routing: expert groups (0: off)")
    ap.add_argument("--topk-group", type=int, default=0,
                    help="group-limited routing: groups kept per token")
    ap.add_argument("--aux-coeff", type=float, default=0.0,
                    help="auxiliary load-balancing loss coefficient (0: off)")
    ap.add_argument("--fp8", action="store_true",
                    help="FP8 expert GEMMs with current tensor scaling")
    ap.add_argument("--bias", action="store_true",
                    help="expert FFN with biases (bi on [gate | up], bo on the output)")
    ap.add_argument("--mxfp8", action="store_true",
                    help="block-scaled FP8 expert GEMMs (one E8M0 scale per 32 elements)")
    ap.add_argument("--wgrad-colwise", action="store_true",
                    help="bf16 weight gradients read K-major column-wise copies written "
                         "by the SwiGLU epilogues (default: the row-wise tensors)")
    args = ap.parse_args()
    cfg = {**moe_synth.CONFIGS, **moe_synth.PROFILE_CONFIGS}[args.config]
    ws, rank, local = dist_env()
    if args.impl == "reference":
        res = run_reference(args, cfg, ws, rank)
    else:
        res = run_ours(args, cfg, ws, rank, local)
    if res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
