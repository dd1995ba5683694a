// Top-k router: one warp per token, logits held in registers, k rounds of a
// warp-shuffle argmax.  TransformerEngine PR #2912 "[JAX] Add an MoE Block
// (Layer) that compound router, permutation, groupedGEMM and communication",
// Description: the fused top-K router with softmax or (DeepSeek-V3) sigmoid
// scoring.
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kRouteThreads = 256;  // 8 tokens per block

// NaN ranks below every number so that the order stays total.
MOE_DEVINL float rank_key(float v) { return v != v ? -INFINITY : v; }

// (va, ia) outranks (vb, ib): larger logit, ties to the lower expert id.
// ids >= E mark empty candidates and never win.
MOE_DEVINL bool outranks(float va, int ia, float vb, int ib, int E) {
  if (ia >= E) return false;
  if (ib >= E) return true;
  return va > vb || (va == vb && ia < ib);
}

template <int EPL>
__global__ void __launch_bounds__(kRouteThreads)
route_topk_kernel(const float *__restrict__ logits, int64_t ld, int T, int E, int k,
                  int score_fn, int renorm, int32_t *__restrict__ topk_idx,
                  float *__restrict__ topk_w) {
  const int lane = threadIdx.x & 31;
  const int t = (blockIdx.x * kRouteThreads + threadIdx.x) >> 5;
  if (t >= T) return;
  const float *row = logits + (int64_t)t * ld;
  float v[EPL];
  bool taken[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    v[i] = e < E ? rank_key(__ldg(row + e)) : -INFINITY;
    taken[i] = e >= E;
  }
  // max over all experts (softmax shift) and the softmax denominator
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < EPL; ++i)
    if (!taken[i]) m = fmaxf(m, v[i]);
  m = warp_max(m);
  float denom = 0.f;
  if (score_fn == MOE_SCORE_SOFTMAX) {
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (!taken[i]) denom += expf(v[i] - m);
    denom = warp_sum(denom);
  }
  // k rounds of a warp argmax; lane j keeps the j-th selection
  float my_v = -INFINITY;
  int my_id = 0;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bid = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (!taken[i] && outranks(v[i], e, bv, bid, E)) {
        bv = v[i];
        bid = e;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int oid = __shfl_xor_sync(0xffffffffu, bid, o);
      if (outranks(ov, oid, bv, bid, E)) {
        bv = ov;
        bid = oid;
      }
    }
    if ((bid & 31) == lane) {
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (lane + 32 * i == bid) taken[i] = true;
    }
    if (lane == j) {
      my_v = bv;
      my_id = bid;
    }
  }
  float s = 0.f;
  if (lane < k) {
    s = score_fn == MOE_SCORE_SOFTMAX ? expf(my_v - m) : 1.0f / (1.0f + expf(-my_v));
  }
  float norm;
  if (renorm) {
    norm = warp_sum(lane < k ? s : 0.f);
  } else {
    norm = score_fn == MOE_SCORE_SOFTMAX ? denom : 1.0f;
  }
  if (lane < k) {
    topk_idx[(int64_t)t * k + lane] = my_id;
    topk_w[(int64_t)t * k + lane] = s / norm;
  }
}

}  // namespace

cudaError_t launch_route_topk(const float *logits, int64_t ld, int T, int E, int k, int score_fn,
                              int renorm, int32_t *idx, float *w, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int blocks = (T + kRouteThreads / 32 - 1) / (kRouteThreads / 32);
  if (E <= 32)
    route_topk_kernel<1><<<blocks, kRouteThreads, 0, s>>>(logits, ld, T, E, k, score_fn, renorm, idx, w);
  else if (E <= 64)
    route_topk_kernel<2><<<blocks, kRouteThreads, 0, s>>>(logits, ld, T, E, k, score_fn, renorm, idx, w);
  else if (E <= 128)
    route_topk_kernel<4><<<blocks, kRouteThreads, 0, s>>>(logits, ld, T, E, k, score_fn, renorm, idx, w);
  else
    route_topk_kernel<8><<<blocks, kRouteThreads, 0, s>>>(logits, ld, T, E, k, score_fn, renorm, idx, w);
  return cudaGetLastError();
}

}  // namespace moe
