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

// (va, ia) outranks (vb, ib) in (value desc, id asc) order, no sentinel ids.
MOE_DEVINL bool before(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// Group-limited selection (DeepSeek-V3 style): the warp's token keys are in
// `keys` (shared memory); lane-strided groups of gs experts each score the
// fp32 sum of their m largest keys, added from the largest down; the
// topk_group best groups (ties to the lower group id) are marked open in
// `open_g`.
MOE_DEVINL void open_groups(const float *keys, unsigned char *open_g, int G, int gs, int m,
                            int topk_group, int lane) {
  constexpr int kMaxGPL = 8;  // groups per lane: G <= 256
  float sc[kMaxGPL];
  bool chosen[kMaxGPL];
#pragma unroll
  for (int j = 0; j < kMaxGPL; ++j) {
    const int g = lane + 32 * j;
    chosen[j] = g >= G;
    sc[j] = -INFINITY;
    if (g < G) {
      const float *kg = keys + g * gs;
      // m passes, each taking the next key in (value desc, index asc) order
      float pv = INFINITY;
      int pi = -1;
      float acc = 0.f;
      for (int r = 0; r < m; ++r) {
        float bv = -INFINITY;
        int bi = gs;
        for (int i = 0; i < gs; ++i) {
          const float v = kg[i];
          const bool after_prev = v < pv || (v == pv && i > pi);
          if (after_prev && (bi == gs || before(v, i, bv, bi))) {
            bv = v;
            bi = i;
          }
        }
        acc = r == 0 ? bv : __fadd_rn(acc, bv);
        pv = bv;
        pi = bi;
      }
      sc[j] = acc;
    }
  }
  for (int r = 0; r < topk_group; ++r) {
    float bv = -INFINITY;
    int bg = 0x7fffffff;
#pragma unroll
    for (int j = 0; j < kMaxGPL; ++j) {
      const int g = lane + 32 * j;
      if (!chosen[j] && (bg == 0x7fffffff || before(sc[j], g, bv, bg))) {
        bv = sc[j];
        bg = g;
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      const int og = __shfl_xor_sync(0xffffffffu, bg, o);
      if (og != 0x7fffffff && (bg == 0x7fffffff || before(ov, og, bv, bg))) {
        bv = ov;
        bg = og;
      }
    }
    if ((bg & 31) == lane) {
#pragma unroll
      for (int j = 0; j < kMaxGPL; ++j)
        if (lane + 32 * j == bg) chosen[j] = true;
    }
    if (lane == 0) open_g[bg] = 1;
  }
}

// Selection ranks key = logit (+ expert_bias[e] when given, the DeepSeek-V3
// bias that steers selection only); the weights use the unbiased logits.
// GROUPED: only experts of the topk_group best of num_groups groups compete.
template <int EPL, bool GROUPED>
__global__ void __launch_bounds__(kRouteThreads)
route_topk_kernel(const float *__restrict__ logits, int64_t ld, int T, int E, int k,
                  int score_fn, int renorm, const float *__restrict__ expert_bias,
                  int num_groups, int topk_group,
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
  if (GROUPED) {
    __shared__ float s_keys[kRouteThreads / 32][256];
    __shared__ unsigned char s_open[kRouteThreads / 32][256];
    const int w = threadIdx.x >> 5;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E) s_keys[w][e] = v[i];
      if (e < num_groups) s_open[w][e] = 0;
    }
    __syncwarp();
    const int gs = E / num_groups;
    open_groups(s_keys[w], s_open[w], num_groups, gs, k / topk_group, topk_group, lane);
    __syncwarp();
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !s_open[w][e / gs]) taken[i] = true;  // closed group: never chosen
    }
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

// Router probabilities of one token for the load-balancing loss: softmax over
// all E, or sigmoid scores normalised by their sum over all E.  Lane-strided
// experts in registers; s_out (sigmoid only) receives the raw sigmoid scores.
template <int EPL>
MOE_DEVINL void token_probs(const float *row, int E, int score_fn, int lane, float *p,
                            float *s_out, float *S_out) {
  float l[EPL];
  float mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    l[i] = e < E ? rank_key(__ldg(row + e)) : -INFINITY;
    mx = fmaxf(mx, l[i]);
  }
  float sum = 0.f;
  if (score_fn == MOE_SCORE_SOFTMAX) {
    mx = warp_max(mx);
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      p[i] = lane + 32 * i < E ? expf(l[i] - mx) : 0.f;
      sum += p[i];
    }
  } else {
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      p[i] = lane + 32 * i < E ? 1.0f / (1.0f + expf(-l[i])) : 0.f;
      s_out[i] = p[i];
      sum += p[i];
    }
  }
  sum = warp_sum(sum);
#pragma unroll
  for (int i = 0; i < EPL; ++i) p[i] /= sum;
  *S_out = sum;
}

constexpr int kAuxTokens = 256;  // tokens per block of the loss kernel (32 per warp)

// Per block: column sums of the router probabilities over its tokens and the
// histogram of its tokens' choices, written to the block's workspace row.
template <int EPL>
__global__ void __launch_bounds__(kRouteThreads)
aux_partial_kernel(const float *__restrict__ logits, int64_t ld, int T, int E, int k,
                   int score_fn, const int32_t *__restrict__ topk_idx,
                   float *__restrict__ part_p, int32_t *__restrict__ part_c) {
  __shared__ float s_p[kRouteThreads / 32][256];
  __shared__ int s_c[256];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  for (int e = threadIdx.x; e < E; e += kRouteThreads) s_c[e] = 0;
  __syncthreads();
  float acc[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) acc[i] = 0.f;
  const int t0 = blockIdx.x * kAuxTokens + w * (kAuxTokens / (kRouteThreads / 32));
  for (int u = 0; u < kAuxTokens / (kRouteThreads / 32); ++u) {
    const int t = t0 + u;
    if (t >= T) break;
    float p[EPL], sg[EPL], S;
    token_probs<EPL>(logits + (int64_t)t * ld, E, score_fn, lane, p, sg, &S);
#pragma unroll
    for (int i = 0; i < EPL; ++i) acc[i] += p[i];
    if (lane < k) {
      const int e = __ldg(topk_idx + (int64_t)t * k + lane);
      if (e >= 0 && e < E) atomicAdd(&s_c[e], 1);   // integer: order-free
    }
  }
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    if (e < E) s_p[w][e] = acc[i];
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += kRouteThreads) {
    float v = 0.f;
    for (int ww = 0; ww < kRouteThreads / 32; ++ww) v += s_p[ww][e];   // fixed order
    part_p[(int64_t)blockIdx.x * E + e] = v;
    part_c[(int64_t)blockIdx.x * E + e] = s_c[e];
  }
}

// One block: block partials summed in block order; P_e, counts, and
// loss = coeff * sum_e f_e P_e with f_e = E count_e / (k T).
__global__ void __launch_bounds__(256)
aux_finish_kernel(const float *__restrict__ part_p, const int32_t *__restrict__ part_c,
                  int nblk, int T, int E, int k, float coeff, int32_t *__restrict__ counts,
                  float *__restrict__ P, float *__restrict__ loss) {
  __shared__ float s_t[256];
  const int e = threadIdx.x;
  float term = 0.f;
  if (e < E) {
    float ps = 0.f;
    int c = 0;
    for (int b = 0; b < nblk; ++b) {
      ps += part_p[(int64_t)b * E + e];
      c += part_c[(int64_t)b * E + e];
    }
    const float Pe = T > 0 ? ps / (float)T : 0.f;
    const float fe = T > 0 ? (float)E * (float)c / ((float)k * (float)T) : 0.f;
    counts[e] = c;
    P[e] = Pe;
    term = fe * Pe;
  }
  s_t[threadIdx.x] = term;
  __syncthreads();
  for (int h = 128; h > 0; h >>= 1) {
    if (threadIdx.x < h) s_t[threadIdx.x] += s_t[threadIdx.x + h];
    __syncthreads();
  }
  if (threadIdx.x == 0) *loss = coeff * s_t[0];
}

// Logit gradient of the load-balancing loss, one warp per token:
//   softmax:           d_l[e] = g p_e (f_e - c)
//   normalised sigmoid: d_l[e] = g s_e (1 - s_e) / S (f_e - c)
// with g = d_loss coeff / T and c = sum_j f_j p_j.
template <int EPL>
__global__ void __launch_bounds__(kRouteThreads)
aux_bwd_kernel(const float *__restrict__ logits, int64_t ld, int T, int E, int k, int score_fn,
               const int32_t *__restrict__ counts, float coeff, float d_loss,
               float *__restrict__ d_logits, int64_t ld_out, int accumulate) {
  const int lane = threadIdx.x & 31;
  const int t = (blockIdx.x * kRouteThreads + threadIdx.x) >> 5;
  if (t >= T) return;
  float p[EPL], sg[EPL], S;
  token_probs<EPL>(logits + (int64_t)t * ld, E, score_fn, lane, p, sg, &S);
  const float fscale = (float)E / ((float)k * (float)T);
  float f[EPL];
  float c = 0.f;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    f[i] = e < E ? fscale * (float)__ldg(counts + e) : 0.f;
    c += f[i] * p[i];
  }
  c = warp_sum(c);
  const float g = d_loss * coeff / (float)T;
  float *orow = d_logits + (int64_t)t * ld_out;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    const int e = lane + 32 * i;
    if (e >= E) continue;
    const float jac = score_fn == MOE_SCORE_SOFTMAX ? p[i] : sg[i] * (1.0f - sg[i]) / S;
    const float v = g * jac * (f[i] - c);
    orow[e] = accumulate ? orow[e] + v : v;
  }
}

}  // namespace

size_t aux_loss_workspace_bytes(int T, int E) {
  const size_t nblk = (size_t)(T + kAuxTokens - 1) / kAuxTokens;
  return (nblk > 0 ? nblk : 1) * (size_t)E * 8;
}

cudaError_t launch_aux_loss(const float *logits, int64_t ld, int T, int E, int k, int score_fn,
                            const int32_t *idx, float coeff, int32_t *counts, float *P,
                            float *loss, void *ws, cudaStream_t s) {
  const int nblk = (T + kAuxTokens - 1) / kAuxTokens;
  float *part_p = static_cast<float *>(ws);
  int32_t *part_c = reinterpret_cast<int32_t *>(part_p + (size_t)(nblk > 0 ? nblk : 1) * E);
  if (nblk > 0) {
#define MOE_AUX(EPL)                                                                      \
  aux_partial_kernel<EPL><<<nblk, kRouteThreads, 0, s>>>(logits, ld, T, E, k, score_fn, idx, \
                                                         part_p, part_c)
    if (E <= 32) MOE_AUX(1);
    else if (E <= 64) MOE_AUX(2);
    else if (E <= 128) MOE_AUX(4);
    else MOE_AUX(8);
#undef MOE_AUX
  }
  aux_finish_kernel<<<1, 256, 0, s>>>(part_p, part_c, nblk, T, E, k, coeff, counts, P, loss);
  return cudaGetLastError();
}

cudaError_t launch_aux_loss_bwd(const float *logits, int64_t ld, int T, int E, int k,
                                int score_fn, const int32_t *counts, float coeff, float d_loss,
                                float *d_logits, int64_t ld_out, int accumulate, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int blocks = (T + kRouteThreads / 32 - 1) / (kRouteThreads / 32);
#define MOE_AUX_BWD(EPL)                                                                 \
  aux_bwd_kernel<EPL><<<blocks, kRouteThreads, 0, s>>>(logits, ld, T, E, k, score_fn, counts, \
                                                       coeff, d_loss, d_logits, ld_out, accumulate)
  if (E <= 32) MOE_AUX_BWD(1);
  else if (E <= 64) MOE_AUX_BWD(2);
  else if (E <= 128) MOE_AUX_BWD(4);
  else MOE_AUX_BWD(8);
#undef MOE_AUX_BWD
  return cudaGetLastError();
}

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
                              int renorm, const float *bias, int num_groups, int topk_group,
                              int32_t *idx, float *w, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int blocks = (T + kRouteThreads / 32 - 1) / (kRouteThreads / 32);
  const bool grouped = num_groups > 1;
#define MOE_ROUTE(EPL)                                                                          \
  do {                                                                                          \
    if (grouped)                                                                                \
      route_topk_kernel<EPL, true><<<blocks, kRouteThreads, 0, s>>>(                            \
          logits, ld, T, E, k, score_fn, renorm, bias, num_groups, topk_group, idx, w);         \
    else                                                                                        \
      route_topk_kernel<EPL, false><<<blocks, kRouteThreads, 0, s>>>(                           \
          logits, ld, T, E, k, score_fn, renorm, bias, num_groups, topk_group, idx, w);         \
  } while (0)
  if (E <= 32) MOE_ROUTE(1);
  else if (E <= 64) MOE_ROUTE(2);
  else if (E <= 128) MOE_ROUTE(4);
  else MOE_ROUTE(8);
#undef MOE_ROUTE
  return cudaGetLastError();
}

}  // namespace moe
