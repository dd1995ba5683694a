// Plain CUDA-core grouped GEMMs (64x64 tiles, fp32 accumulation): the first,
// simple implementation of moe_gmm / moe_tgmm semantics, used to bring the
// whole layer up end to end.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int BM = 64, BN = 64, BK = 16;

MOE_DEVINL float bf(const uint16_t *p) {
  return __uint_as_float(((uint32_t)__ldg(reinterpret_cast<const unsigned short *>(p))) << 16);
}

template <int EPI>
__global__ void __launch_bounds__(256) gmm_simt_kernel(GmmArgs a) {
  __shared__ float As[BK][BM + 1];
  __shared__ float Bs[2][BK][BN + 1];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  // m-tile slot -> (expert, row range)
  int slot = blockIdx.y, e = -1, row0 = 0, row1 = 0;
  for (int g = 0; g < a.E; ++g) {
    const int s = min((int64_t)a.offsets[g], a.rows_cap);
    const int t = min((int64_t)a.offsets[g + 1], a.rows_cap);
    const int nt = t > s ? (t - s + BM - 1) / BM : 0;
    if (slot < nt) {
      e = g;
      row0 = s + slot * BM;
      row1 = min(t, row0 + BM);
      break;
    }
    slot -= nt;
  }
  if (e < 0) return;
  const int F = (EPI == MOE_EPI_SWIGLU_FWD) ? a.N / 2 : a.N;  // output columns of the tile grid
  const int n0 = blockIdx.x * BN;
  if (n0 >= F) return;
  const uint16_t *Be = a.B + (int64_t)e * a.stride_b;
  constexpr int NB = (EPI == MOE_EPI_SWIGLU_FWD) ? 2 : 1;
  float acc[NB][4][4];
#pragma unroll
  for (int h = 0; h < NB; ++h)
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[h][i][j] = 0.f;
  for (int k0 = 0; k0 < a.K; k0 += BK) {
    for (int q = threadIdx.x; q < BM * BK; q += 256) {
      const int m = q / BK, kk = q % BK;
      const int r = row0 + m, kc = k0 + kk;
      As[kk][m] = (r < row1 && kc < a.K) ? bf(a.A + (int64_t)r * a.lda + kc) : 0.f;
    }
    for (int h = 0; h < NB; ++h) {
      for (int q = threadIdx.x; q < BN * BK; q += 256) {
        const int kk = q / BN, nn = q % BN;
        const int kc = k0 + kk, n = n0 + nn + h * F;
        float v = 0.f;
        if (kc < a.K && n0 + nn < F)
          v = a.trans_b ? bf(Be + (int64_t)n * a.ldb + kc) : bf(Be + (int64_t)kc * a.ldb + n);
        Bs[h][kk][nn] = v;
      }
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
#pragma unroll
      for (int h = 0; h < NB; ++h)
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int j = 0; j < 4; ++j) acc[h][i][j] += As[kk][ty * 4 + i] * Bs[h][kk][tx * 4 + j];
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = row0 + ty * 4 + i;
    if (r >= row1) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= F) continue;
      if (EPI == MOE_EPI_NONE) {
        float v = acc[0][i][j];
        if (a.ps) v += a.ps[(int64_t)r * a.ld_ps + n];
        if (a.c_dtype == MOE_DTYPE_F32)
          static_cast<float *>(a.C)[(int64_t)r * a.ldc + n] = v;
        else
          static_cast<bf16_t *>(a.C)[(int64_t)r * a.ldc + n] = __float2bfloat16_rn(v);
      } else if (EPI == MOE_EPI_SWIGLU_FWD) {
        float g = acc[0][i][j], u = acc[NB - 1][i][j];
        if (a.ps) {
          g += a.ps[(int64_t)r * a.ld_ps + n];
          u += a.ps[(int64_t)r * a.ld_ps + F + n];
        }
        bf16_t *H = static_cast<bf16_t *>(a.C);
        H[(int64_t)r * a.ldc + n] = __float2bfloat16_rn(g);
        H[(int64_t)r * a.ldc + F + n] = __float2bfloat16_rn(u);
        reinterpret_cast<bf16_t *>(a.C2)[(int64_t)r * a.ldc2 + n] =
            __float2bfloat16_rn(g * sigmoid_f(g) * u);
      } else {
        const float da = acc[0][i][j];
        const float g = bf(a.aux + (int64_t)r * a.ld_aux + n);
        const float u = bf(a.aux + (int64_t)r * a.ld_aux + F + n);
        const float s = sigmoid_f(g);
        bf16_t *dH = static_cast<bf16_t *>(a.C);
        dH[(int64_t)r * a.ldc + n] = __float2bfloat16_rn(da * u * s * (1.f + g * (1.f - s)));
        dH[(int64_t)r * a.ldc + F + n] = __float2bfloat16_rn(da * g * s);
      }
    }
  }
}

__global__ void __launch_bounds__(256) tgmm_simt_kernel(TgmmArgs a) {
  __shared__ float As[BK][BM + 1];
  __shared__ float Bs[BK][BN + 1];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int e = blockIdx.z, m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  const int s = min((int64_t)a.offsets[e], a.rows_cap);
  const int t = min((int64_t)a.offsets[e + 1], a.rows_cap);
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
  for (int r0 = s; r0 < t; r0 += BK) {
    for (int q = threadIdx.x; q < BM * BK; q += 256) {
      const int rr = q / BM, mm = q % BM;
      const int r = r0 + rr;
      As[rr][mm] = (r < t && m0 + mm < a.M) ? bf(a.A + (int64_t)r * a.lda + m0 + mm) : 0.f;
      Bs[rr][mm] = (r < t && n0 + mm < a.N) ? bf(a.B + (int64_t)r * a.ldb + n0 + mm) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int rr = 0; rr < BK; ++rr)
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] += As[rr][ty * 4 + i] * Bs[rr][tx * 4 + j];
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty * 4 + i;
    if (m >= a.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= a.N) continue;
      const int64_t o = (int64_t)e * a.stride_w + (int64_t)m * a.ldw + n;
      if (a.w_dtype == MOE_DTYPE_F32) {
        float *W = static_cast<float *>(a.W);
        W[o] = a.accumulate ? W[o] + acc[i][j] : acc[i][j];
      } else {
        static_cast<bf16_t *>(a.W)[o] = __float2bfloat16_rn(acc[i][j]);
      }
    }
  }
}

}  // namespace

moe_status_t launch_gmm(const GmmArgs &a, cudaStream_t s) {
  const int F = a.epilogue == MOE_EPI_SWIGLU_FWD ? a.N / 2 : a.N;
  const int64_t slots = (a.rows_cap + BM - 1) / BM + a.E;
  if (slots > 65535) {
    set_error("moe_gmm: too many row tiles for the grid");
    return MOE_ERR_UNSUPPORTED;
  }
  dim3 grid((F + BN - 1) / BN, (unsigned)slots);
  if (a.epilogue == MOE_EPI_NONE)
    gmm_simt_kernel<MOE_EPI_NONE><<<grid, 256, 0, s>>>(a);
  else if (a.epilogue == MOE_EPI_SWIGLU_FWD)
    gmm_simt_kernel<MOE_EPI_SWIGLU_FWD><<<grid, 256, 0, s>>>(a);
  else
    gmm_simt_kernel<MOE_EPI_SWIGLU_BWD><<<grid, 256, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("moe_gmm launch: %s", cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

moe_status_t launch_tgmm(const TgmmArgs &a, cudaStream_t s) {
  dim3 grid((a.N + BN - 1) / BN, (a.M + BM - 1) / BM, a.E);
  tgmm_simt_kernel<<<grid, 256, 0, s>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("moe_tgmm launch: %s", cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

}  // namespace moe
