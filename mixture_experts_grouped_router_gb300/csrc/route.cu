// Top-k router and its backward: one warp per token, logits held in
// registers, k rounds of a warp-shuffle argmax.  TransformerEngine PR #2912
// "[JAX] Add an MoE Block (Layer) that compound router, permutation,
// groupedGEMM and communication", Description: the fused top-K router with
// softmax or (DeepSeek-V3) sigmoid scoring; sequence diagram: the backward
// carries the routing-weight gradient back to the gate.
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

// Selection ranks key = logit (+ expert_bias[e] when given, the DeepSeek-V3
// bias that steers selection only); the weights use the unbiased logits.
template <int EPL>
__global__ void __launch_bounds__(kRouteThreads)
route_topk_kernel(const float *__restrict__ logits, int64_t ld, int T, int E, int k,
                  int score_fn, int renorm, const float *__restrict__ expert_bias,
                  int32_t *__restrict__ topk_idx, float *__restrict__ topk_w) {
  const int lane = threadIdx.x & 31;
  const int t = (blockIdx.x * kRouteThreads + threadIdx.x) >> 5;
  if (t >= T) return;
  const float *row = logits + (int64_t)t * ld;
  float v[EPL], lg[EPL];
  bool taken[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    lg[i] = e < E ? rank_key(__ldg(row + e)) : -INFINITY;
    v[i] = (e < E && expert_bias != nullptr) ? rank_key(lg[i] + __ldg(expert_bias + e)) : lg[i];
    taken[i] = e >= E;
  }
  // max over all experts (softmax shift) and the softmax denominator
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < EPL; ++i)
    if (!taken[i]) m = fmaxf(m, lg[i]);
  m = warp_max(m);
  float denom = 0.f;
  if (score_fn == MOE_SCORE_SOFTMAX) {
#pragma unroll
    for (int i = 0; i < EPL; ++i)
      if (!taken[i]) denom += expf(lg[i] - m);
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
    const float l = expert_bias != nullptr ? rank_key(__ldg(row + my_id)) : my_v;
    s = score_fn == MOE_SCORE_SOFTMAX ? expf(l - m) : 1.0f / (1.0f + expf(-l));
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

// Backward of the routing weights (selection fixed), one warp per token:
//   softmax + renorm:  d_l[i_j] = w_j (dw_j - c),               c = sum_m dw_m w_m
//   softmax:           d_l[e]   = p_e ([e = i_j] dw_j - c)        for every e
//   sigmoid + renorm:  d_l[i_j] = s_j (1 - s_j) (dw_j - c) / S,  S = sum_m s_m
//   sigmoid:           d_l[i_j] = dw_j s_j (1 - s_j)
// other entries are 0.
template <int EPL>
__global__ void __launch_bounds__(kRouteThreads)
route_topk_bwd_kernel(const float *__restrict__ logits, int64_t ld,
                      const int32_t *__restrict__ topk_idx, const float *__restrict__ topk_w,
                      const float *__restrict__ d_topk_w, int T, int E, int k, int score_fn,
                      int renorm, float *__restrict__ d_logits, int64_t ld_out) {
  const int lane = threadIdx.x & 31;
  const int t = (blockIdx.x * kRouteThreads + threadIdx.x) >> 5;
  if (t >= T) return;
  const float *row = logits + (int64_t)t * ld;
  int id = -1;
  float w = 0.f, dw = 0.f, l = 0.f;
  if (lane < k) {
    id = __ldg(topk_idx + (int64_t)t * k + lane);
    w = __ldg(topk_w + (int64_t)t * k + lane);
    dw = __ldg(d_topk_w + (int64_t)t * k + lane);
    if (id >= 0 && id < E) l = __ldg(row + id);
    else id = -1;
  }
  const float c = warp_sum(lane < k ? dw * w : 0.f);
  float val = 0.f;  // gradient of the selected expert held by lane j
  if (score_fn == MOE_SCORE_SOFTMAX) {
    if (renorm) val = w * (dw - c);
  } else {
    const float sj = 1.0f / (1.0f + expf(-l));
    if (renorm) {
      const float S = warp_sum(lane < k ? sj : 0.f);
      val = sj * (1.0f - sj) * (dw - c) / S;
    } else {
      val = dw * sj * (1.0f - sj);
    }
  }
  // softmax over all E without renorm: every expert gets -p_e c, the selected +p_e dw_j
  float m = 0.f, denom = 1.f;
  const bool dense = score_fn == MOE_SCORE_SOFTMAX && !renorm;
  if (dense) {
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E) mx = fmaxf(mx, rank_key(__ldg(row + e)));
    }
    m = warp_max(mx);
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E) sum += expf(rank_key(__ldg(row + e)) - m);
    }
    denom = warp_sum(sum);
  }
  float out[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    float p = 0.f;
    if (dense && e < E) p = expf(rank_key(__ldg(row + e)) - m) / denom;
    out[i] = dense ? -p * c : 0.f;
    for (int j = 0; j < k; ++j) {
      const int ij = __shfl_sync(0xffffffffu, id, j);
      const float vj = __shfl_sync(0xffffffffu, val, j);
      const float dwj = __shfl_sync(0xffffffffu, dw, j);
      if (ij == e) out[i] = dense ? p * (dwj - c) : vj;
    }
  }
  float *orow = d_logits + (int64_t)t * ld_out;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E) orow[e] = out[i];
  }
}

}  // namespace

cudaError_t launch_route_topk_bwd(const float *logits, int64_t ld, const int32_t *idx,
                                  const float *w, const float *dw, int T, int E, int k,
                                  int score_fn, int renorm, float *d_logits, int64_t ld_out,
                                  cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int blocks = (T + kRouteThreads / 32 - 1) / (kRouteThreads / 32);
#define MOE_ROUTE_BWD(EPL)                                                                   \
  route_topk_bwd_kernel<EPL><<<blocks, kRouteThreads, 0, s>>>(logits, ld, idx, w, dw, T, E, k, \
                                                              score_fn, renorm, d_logits, ld_out)
  if (E <= 32) MOE_ROUTE_BWD(1);
  else if (E <= 64) MOE_ROUTE_BWD(2);
  else if (E <= 128) MOE_ROUTE_BWD(4);
  else MOE_ROUTE_BWD(8);
#undef MOE_ROUTE_BWD
  return cudaGetLastError();
}

cudaError_t launch_route_topk(const float *logits, int64_t ld, int T, int E, int k, int score_fn,
                              int renorm, const float *bias, int32_t *idx, float *w,
                              cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int blocks = (T + kRouteThreads / 32 - 1) / (kRouteThreads / 32);
#define MOE_ROUTE(EPL)                                                                        \
  route_topk_kernel<EPL><<<blocks, kRouteThreads, 0, s>>>(logits, ld, T, E, k, score_fn, renorm, \
                                                          bias, idx, w)
  if (E <= 32) MOE_ROUTE(1);
  else if (E <= 64) MOE_ROUTE(2);
  else if (E <= 128) MOE_ROUTE(4);
  else MOE_ROUTE(8);
#undef MOE_ROUTE
  return cudaGetLastError();
}

}  // namespace moe
