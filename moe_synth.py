"""Seeded synthetic inputs for the MoE expert layer.

This module is shared by the oracle's tests, the GPU parity tests and the
benchmark.  It holds random draws, the workload presets and the bf16 storage
format, and none of the layer's arithmetic: no routing, permutation, GEMM or
combine step lives here.

Recipe (one ``numpy.random.default_rng(seed)`` per workload, draws in this
order): [skewed preset only: a random permutation giving each expert its
popularity rank], router logits, x, wi_0, wi_1, wo, dOut.

* router logits: fp32, N(0, 1); the skewed preset adds a per-expert bias
  ``-kappa * s * ln(rank_e)`` (Zipf-like popularity with exponent s).
* x, dOut: N(0, 1); expert weights: N(0, 0.02).
* every bf16 tensor is rounded on the host with round-to-nearest-even, so the
  GPU and the oracle consume the very same bytes.

The workloads are the ones the pages describe for this layer: a tiny layer, a
Mixtral-like layer, a DeepSeek-V3-shaped local expert layer, a skewed-routing
stress case with align_size padding and capacity dropping, and the chunked-K
partial-sum variant ("Overlap moe comms with collective matmul", MaxText
PR #4295, Description).  The pages trained on MaxText's synthetic dataset
("[Draft] Integrate TE/JAX GroupedGEMM for MoE", MaxText PR #2319, the
command under Tests), so synthetic data stands in for no public dataset.
"""
from __future__ import annotations

import dataclasses
import numpy as np

SOFTMAX = 0
SIGMOID = 1


@dataclasses.dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int            # tokens
    d: int            # d_model
    f: int            # per-expert d_ff
    E: int            # experts
    k: int            # top-k
    score_fn: int = SOFTMAX
    renorm: int = 1   # renormalise the k selected weights to sum to 1
    align: int = 0    # align_size (0 or 1: no padding)
    capacity: int = 0  # per-expert capacity C in assignments (0: no dropping)
    num_chunks: int = 1  # K-chunks of the up-projection (partial-sum path)
    zipf_s: float = 0.0   # > 0: skewed router logits
    zipf_kappa: float = 0.0

    @property
    def rows_cap(self) -> int:
        """Worst-case number of permuted rows: T*k plus E*(align-1) padding."""
        pad = self.align - 1 if self.align > 1 else 0
        return self.T * self.k + self.E * pad


CONFIGS = {
    # tiny MoE layer
    "tiny": MoEConfig("tiny", T=256, d=128, f=256, E=8, k=2, score_fn=SOFTMAX, renorm=1),
    # Mixtral-like expert layer
    "mixtral": MoEConfig("mixtral", T=16384, d=4096, f=14336, E=8, k=2,
                         score_fn=SOFTMAX, renorm=1),
    # DeepSeek-V3-shaped local expert layer: sigmoid scores renormalised over the 8 selected
    "dsv3": MoEConfig("dsv3", T=8192, d=7168, f=2048, E=32, k=8, score_fn=SIGMOID, renorm=1),
    # skewed-routing stress: Zipf-ranked bias, align 128, capacity factor 1.0
    # => C = ceil(1.0 * T * k / E) = ceil(32768 / 64) = 512
    "skewed": MoEConfig("skewed", T=32768, d=4096, f=2048, E=64, k=1, score_fn=SOFTMAX,
                        renorm=0, align=128, capacity=512, zipf_s=1.2, zipf_kappa=0.92),
    # chunked-K partial-sum path on the DeepSeek-shaped layer
    "dsv3_chunked": MoEConfig("dsv3_chunked", T=8192, d=7168, f=2048, E=32, k=8,
                              score_fn=SIGMOID, renorm=1, num_chunks=4),
}


# Reduced workloads used for profiling captures: the GEMM kernels at the same
# per-expert shapes on a few GB of device memory.
PROFILE_CONFIGS = {
    "mixtral_e2": MoEConfig("mixtral_e2", T=8192, d=4096, f=14336, E=2, k=1, score_fn=SOFTMAX,
                            renorm=0),
    "dsv3_e8": MoEConfig("dsv3_e8", T=2048, d=7168, f=2048, E=8, k=8, score_fn=SIGMOID,
                         renorm=1),
    "dsv3_e8_chunked": MoEConfig("dsv3_e8_chunked", T=2048, d=7168, f=2048, E=8, k=8,
                                 score_fn=SIGMOID, renorm=1, num_chunks=4),
    # the skewed-routing layer's expert shape and routing on 16 experts
    "skewed_e16": MoEConfig("skewed_e16", T=8192, d=4096, f=2048, E=16, k=1, score_fn=SOFTMAX,
                            renorm=0, align=128, capacity=512, zipf_s=1.2, zipf_kappa=0.92),
}


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 (round to nearest, ties to even); return the uint16 bits."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)
    return r.astype(np.uint16)


def bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Decode bf16 bits into fp32 values (exact)."""
    return (np.asarray(bits).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return bits_to_f32(bits).astype(np.float64)


def _normal_bf16(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    """Draw N(0, std^2) in fp32 and round to bf16 bits, in slabs to bound host memory."""
    out = np.empty(shape, dtype=np.uint16)
    flat = out.reshape(-1)
    n = flat.size
    slab = 1 << 26
    for s in range(0, n, slab):
        e = min(n, s + slab)
        v = rng.standard_normal(e - s, dtype=np.float32)
        if std != 1.0:
            v *= np.float32(std)
        flat[s:e] = bf16_bits(v)
    return out


def make_inputs(cfg: MoEConfig, seed: int = 0) -> dict:
    """Return the seeded inputs of one workload.

    Keys: ``logits`` fp32 [T,E]; ``x`` bf16 bits [T,d]; ``wi`` bf16 bits
    [E,d,2f] holding [wi_0 | wi_1] on the last axis; ``wo`` bf16 bits [E,f,d];
    ``dout`` bf16 bits [T,d]; ``expert_rank`` (skewed preset only).
    """
    rng = np.random.default_rng(seed)
    T, d, f, E = cfg.T, cfg.d, cfg.f, cfg.E
    res = {}
    bias = np.zeros(E, dtype=np.float32)
    if cfg.zipf_s > 0:
        rank = rng.permutation(E) + 1
        res["expert_rank"] = rank
        bias = (-cfg.zipf_kappa * cfg.zipf_s * np.log(rank.astype(np.float64))).astype(np.float32)
    logits = rng.standard_normal((T, E), dtype=np.float32) + bias[None, :]
    res["logits"] = logits.astype(np.float32)
    res["x"] = _normal_bf16(rng, (T, d), 1.0)
    wi = np.empty((E, d, 2 * f), dtype=np.uint16)
    wi[:, :, :f] = _normal_bf16(rng, (E, d, f), 0.02)
    wi[:, :, f:] = _normal_bf16(rng, (E, d, f), 0.02)
    res["wi"] = wi
    res["wo"] = _normal_bf16(rng, (E, f, d), 0.02)
    res["dout"] = _normal_bf16(rng, (T, d), 1.0)
    return res


def make_biases(cfg: MoEConfig, seed: int = 0, std: float = 0.5) -> dict:
    """Seeded expert-FFN biases, drawn from their own stream so that the
    bias-free inputs of ``make_inputs`` stay unchanged.

    Keys: ``bi`` bf16 bits [E, 2f] ([gate | up]); ``bo`` bf16 bits [E, d]."""
    rng = np.random.default_rng([seed, 0xB1A5])
    return {"bi": _normal_bf16(rng, (cfg.E, 2 * cfg.f), std),
            "bo": _normal_bf16(rng, (cfg.E, cfg.d), std)}


def scaled(cfg: MoEConfig, **kw) -> MoEConfig:
    """A copy of a preset with some sizes replaced (used for small parity cases)."""
    return dataclasses.replace(cfg, **kw)
