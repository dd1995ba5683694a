// Routing-weighted combine, its backward, and the dispatch backward.
//
// TransformerEngine PR #2912 "[JAX] Add an MoE Block (Layer) that compound
// router, permutation, groupedGEMM and communication", review thread on
// _combine_bwd (pure-JAX path):
//   forward   output[t] = sum_j intermediate[t, j] * w[t, j]
//   backward  d_intermediate[t, j] = d_output[t] * w[t, j]
//             d_w[t, j] = sum over hidden of d_output[t] * intermediate[t, j]
// with intermediate[t, j] = Y[flat_to_sorted[t*k + j]] (the un-sort) and zero
// gradient on padding rows.  One warp per token; rows move in 16-byte words;
// sums are fp32 in slot order.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kThreads = 256;  // 8 warps = 8 tokens per block

// KT: compile-time slot bound (k <= KT), so the per-slot arrays stay in registers.
template <bool kWeighted, int KT>
__global__ void __launch_bounds__(kThreads)
combine_kernel(const uint16_t *__restrict__ Y, int64_t ldy, const int32_t *__restrict__ f2s,
               const float *__restrict__ w, int T, int k, int d, uint16_t *__restrict__ out,
               int64_t ldo) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
  if (t >= T) return;
  const int pl = lane < k ? __ldg(f2s + (int64_t)t * k + lane) : -1;
  const float wl = (kWeighted && lane < k) ? __ldg(w + (int64_t)t * k + lane) : 1.0f;
  int p[KT];
  float wj[KT];
#pragma unroll
  for (int j = 0; j < KT; ++j) {
    p[j] = __shfl_sync(0xffffffffu, pl, j);
    wj[j] = __shfl_sync(0xffffffffu, wl, j);
  }
  const int nvec = d >> 3;
  uint4 *dst = reinterpret_cast<uint4 *>(out + (int64_t)t * ldo);
  for (int i = lane; i < nvec; i += 64) {
    const bool two = i + 32 < nvec;
    // every slot's loads in flight before the first is used
    uint4 yq[KT][2];
#pragma unroll
    for (int j = 0; j < KT; ++j) {
      if (j < k && p[j] >= 0) {
        const uint4 *src = reinterpret_cast<const uint4 *>(Y + (int64_t)p[j] * ldy);
        yq[j][0] = ld_nc_v4(src + i);
        if (two) yq[j][1] = ld_nc_v4(src + i + 32);
      }
    }
    float acc0[8], acc1[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) acc0[q] = acc1[q] = 0.f;
#pragma unroll
    for (int j = 0; j < KT; ++j) {
      if (j < k && p[j] >= 0) {
        float f[8];
        bf16x8_to_f32(yq[j][0], f);
#pragma unroll
        for (int q = 0; q < 8; ++q) acc0[q] = fmaf(wj[j], f[q], acc0[q]);
        if (two) {
          bf16x8_to_f32(yq[j][1], f);
#pragma unroll
          for (int q = 0; q < 8; ++q) acc1[q] = fmaf(wj[j], f[q], acc1[q]);
        }
      }
    }
    st_v4(dst + i, f32_to_bf16x8(acc0));
    if (two) st_v4(dst + i + 32, f32_to_bf16x8(acc1));
  }
}

// Part A (blocks < nb_tok): one warp per token, two 16-byte chunks per lane
// in flight per slot.  Part B: zero dY on padding rows, 32 rows of
// sorted_to_flat per warp.
template <int KT>
__global__ void __launch_bounds__(kThreads)
unpermute_bwd_kernel(const uint16_t *__restrict__ dout, int64_t ld_dout,
                     const uint16_t *__restrict__ Y, int64_t ldy,
                     const int32_t *__restrict__ f2s, const int32_t *__restrict__ s2f,
                     const int32_t *__restrict__ offsets, const float *__restrict__ w, int T,
                     int k, int d, int E, int64_t rows_cap, uint16_t *__restrict__ dY,
                     int64_t ld_dy, float *__restrict__ dw, int nb_tok) {
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  const int nvec = d >> 3;
  if ((int)blockIdx.x < nb_tok) {
    const int t = blockIdx.x * (kThreads / 32) + wib;
    if (t >= T) return;
    int pl = lane < k ? __ldg(f2s + (int64_t)t * k + lane) : -1;
    if (pl >= rows_cap) pl = -1;
    const float wl = lane < k ? __ldg(w + (int64_t)t * k + lane) : 0.f;
    int p[KT];
    float wj[KT], dot[KT];
#pragma unroll
    for (int j = 0; j < KT; ++j) {
      p[j] = __shfl_sync(0xffffffffu, pl, j);
      wj[j] = __shfl_sync(0xffffffffu, wl, j);
      dot[j] = 0.f;
    }
    const uint4 *g = reinterpret_cast<const uint4 *>(dout + (int64_t)t * ld_dout);
    // a token whose assignments were all dropped reads nothing (its d_w are 0)
    const int nv = __any_sync(0xffffffffu, pl >= 0) ? nvec : 0;
    for (int i = lane; i < nv; i += 64) {
      const bool two = i + 32 < nvec;
      uint4 gq[2], yq[KT][2];
      gq[0] = ld_nc_v4(g + i);
      if (two) gq[1] = ld_nc_v4(g + i + 32);
#pragma unroll
      for (int j = 0; j < KT; ++j) {
        if (j < k && p[j] >= 0) {
          const uint4 *yr = reinterpret_cast<const uint4 *>(Y + (int64_t)p[j] * ldy);
          yq[j][0] = ld_nc_v4(yr + i);
          if (two) yq[j][1] = ld_nc_v4(yr + i + 32);
        }
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (h == 1 && !two) break;
        float gf[8];
        bf16x8_to_f32(gq[h], gf);
#pragma unroll
        for (int j = 0; j < KT; ++j) {
          if (j < k && p[j] >= 0) {
            float yf[8], o[8];
            bf16x8_to_f32(yq[j][h], yf);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              dot[j] = fmaf(gf[q], yf[q], dot[j]);
              o[q] = wj[j] * gf[q];
            }
            st_v4(reinterpret_cast<uint4 *>(dY + (int64_t)p[j] * ld_dy) + i + 32 * h,
                  f32_to_bf16x8(o));
          }
        }
      }
    }
#pragma unroll
    for (int j = 0; j < KT; ++j) {
      if (j < k) {
        const float s = warp_sum(dot[j]);
        if (lane == 0) dw[(int64_t)t * k + j] = p[j] >= 0 ? s : 0.f;
      }
    }
  } else {
    const int64_t wg = (int64_t)(blockIdx.x - nb_tok) * (kThreads / 32) + wib;
    const int64_t R = min((int64_t)__ldg(offsets + E), rows_cap);
    const int64_t p0 = wg * 32;
    if (p0 >= R) return;
    const int64_t pr = p0 + lane;
    const bool pad = pr < R && __ldg(s2f + pr) < 0;
    uint32_t m = __ballot_sync(0xffffffffu, pad);
    const uint4 z = make_uint4(0, 0, 0, 0);
    while (m) {
      const int bit = __ffs(m) - 1;
      m &= m - 1;
      uint4 *dst = reinterpret_cast<uint4 *>(dY + (p0 + bit) * ld_dy);
      for (int i = lane; i < nvec; i += 32) st_v4(dst + i, z);
    }
  }
}

// Per-expert column sums (bias gradients): block (column block, expert e)
// sums every row of group e over 8*CW columns.  CW threads cover one row
// segment with 16-byte loads; the other 256/CW thread rows stride down the
// group, four rows in flight each; the partial sums meet in shared memory in
// a fixed order (deterministic, no atomics).  CW is picked per call so that
// the grid has a few blocks per SM even when N*E is small.
template <int CW>
__global__ void __launch_bounds__(256)
group_colsum_kernel(const uint16_t *__restrict__ G, int64_t ldg,
                    const int32_t *__restrict__ offsets, int64_t rows_cap, int N,
                    float *__restrict__ out, int64_t ld_out) {
  constexpr int RL = 256 / CW;  // row lanes
  __shared__ float part[RL - 1][CW][8];
  const int e = blockIdx.y;
  const int tx = threadIdx.x % CW, ty = threadIdx.x / CW;
  const int col = blockIdx.x * (8 * CW) + tx * 8;
  const int64_t r0 = min(max((int64_t)__ldg(offsets + e), (int64_t)0), rows_cap);
  const int64_t r1 = max(min((int64_t)__ldg(offsets + e + 1), rows_cap), r0);
  float acc[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) acc[q] = 0.f;
  if (col < N) {
    const uint16_t *base = G + col;
    int64_t r = r0 + ty;
    for (; r + 3 * RL < r1; r += 4 * RL) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = ld_nc_v4(base + (r + u * RL) * ldg);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        float f[8];
        bf16x8_to_f32(v[u], f);
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] += f[q];
      }
    }
    for (; r < r1; r += RL) {
      float f[8];
      bf16x8_to_f32(ld_nc_v4(base + r * ldg), f);
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] += f[q];
    }
  }
  if (ty > 0) {
#pragma unroll
    for (int q = 0; q < 8; ++q) part[ty - 1][tx][q] = acc[q];
  }
  __syncthreads();
  if (ty == 0 && col < N) {
    for (int w = 0; w < RL - 1; ++w)
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] += part[w][tx][q];
    float *o = out + (int64_t)e * ld_out + col;
    *reinterpret_cast<float4 *>(o) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    *reinterpret_cast<float4 *>(o + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

}  // namespace

cudaError_t launch_group_colsum(const uint16_t *G, int64_t ldg, const int32_t *offsets, int E,
                               int64_t rows_cap, int N, float *out, int64_t ld_out,
                               cudaStream_t s) {
  if ((ld_out & 3) != 0 || (reinterpret_cast<uintptr_t>(out) & 15) != 0) {
    // fp32 output written with 16-byte stores
    return cudaErrorMisalignedAddress;
  }
  // widest column block that still gives >= 2 blocks per SM
  const int64_t want = 2 * (int64_t)num_sms();
  int cw = 64;
  while (cw > 8 && (int64_t)((N + 8 * cw - 1) / (8 * cw)) * E < want) cw >>= 1;
  dim3 grid((N + 8 * cw - 1) / (8 * cw), E);
  switch (cw) {
    case 64: group_colsum_kernel<64><<<grid, 256, 0, s>>>(G, ldg, offsets, rows_cap, N, out, ld_out); break;
    case 32: group_colsum_kernel<32><<<grid, 256, 0, s>>>(G, ldg, offsets, rows_cap, N, out, ld_out); break;
    case 16: group_colsum_kernel<16><<<grid, 256, 0, s>>>(G, ldg, offsets, rows_cap, N, out, ld_out); break;
    default: group_colsum_kernel<8><<<grid, 256, 0, s>>>(G, ldg, offsets, rows_cap, N, out, ld_out); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_combine(const uint16_t *Y, int64_t ldy, const int32_t *f2s, const float *w,
                           int T, int k, int d, uint16_t *out, int64_t ldo, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int blocks = (T + kThreads / 32 - 1) / (kThreads / 32);
#define MOE_COMBINE(KT)                                                                   \
  do {                                                                                    \
    if (w != nullptr)                                                                     \
      combine_kernel<true, KT><<<blocks, kThreads, 0, s>>>(Y, ldy, f2s, w, T, k, d, out, ldo); \
    else                                                                                  \
      combine_kernel<false, KT><<<blocks, kThreads, 0, s>>>(Y, ldy, f2s, w, T, k, d, out, ldo); \
  } while (0)
  if (k <= 1) MOE_COMBINE(1);
  else if (k <= 2) MOE_COMBINE(2);
  else if (k <= 4) MOE_COMBINE(4);
  else if (k <= 8) MOE_COMBINE(8);
  else MOE_COMBINE(16);
#undef MOE_COMBINE
  return cudaGetLastError();
}

cudaError_t launch_unpermute_bwd(const uint16_t *dout, int64_t ld_dout, const uint16_t *Y,
                                 int64_t ldy, const int32_t *f2s, const int32_t *s2f,
                                 const int32_t *offsets, const float *w, int T, int k, int d,
                                 int E, int64_t rows_cap, uint16_t *dY, int64_t ld_dy,
                                 float *dw, cudaStream_t s) {
  const int wpb = kThreads / 32;
  const int nb_tok = (T + wpb - 1) / wpb;
  const int64_t pad_warps = (rows_cap + 31) / 32;
  const int nb_pad = (int)((pad_warps + wpb - 1) / wpb);
  if (nb_tok + nb_pad == 0) return cudaSuccess;
#define MOE_UNPERMUTE(KT)                                                               \
  unpermute_bwd_kernel<KT><<<nb_tok + nb_pad, kThreads, 0, s>>>(                        \
      dout, ld_dout, Y, ldy, f2s, s2f, offsets, w, T, k, d, E, rows_cap, dY, ld_dy, dw, nb_tok)
  if (k <= 1) MOE_UNPERMUTE(1);
  else if (k <= 2) MOE_UNPERMUTE(2);
  else if (k <= 4) MOE_UNPERMUTE(4);
  else if (k <= 8) MOE_UNPERMUTE(8);
  else MOE_UNPERMUTE(16);
#undef MOE_UNPERMUTE
  return cudaGetLastError();
}

}  // namespace moe
