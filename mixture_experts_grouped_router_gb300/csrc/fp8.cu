// FP8 quantization with current tensor scaling: amax, and bf16 -> 8-bit
// float codes in a row-wise and a column-wise (transposed) copy.
// MaxText PR #2319 "[Draft] Integrate TE/JAX GroupedGEMM for MoE", review
// thread on the quantizer settings of moe.py: current tensor scaling,
// float8_e4m3fn forward, float8_e5m2 backward, 2x (row- and column-wise)
// quantization; TransformerEngine PR #2912, wi-fusion commit: one amax per
// expert for the fused weight.
//
// scale = fp8_max / amax (fp32, 1 when amax is 0 or not finite); code =
// round-to-nearest-even of fp32(x * scale), saturated (cvt.rn.satfinite).
// The column-wise copy of a grouped activation puts group e's rows at columns
// [poff_e, poff_e + size_e) with poff_e = sum over e' < e of the sizes rounded
// up to kF8PadRows, and zeros up to the next group: a weight-gradient GEMM then
// reads whole K blocks of one group with no ragged tail.
#include <float.h>

#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kQT = 64;   // tile: 64 rows x 64 columns
constexpr int kQCT = 8;   // column tiles per block (amortises the group-offset scan)

MOE_DEVINL float fp8_max_of(int fmt) { return fmt == MOE_FP8_E4M3 ? 448.0f : 57344.0f; }

MOE_DEVINL float scale_of(float amax, int fmt) {
  return (amax > 0.0f && amax <= FLT_MAX) ? __fdiv_rn(fp8_max_of(fmt), amax) : 1.0f;
}

// codes of (lo, hi) in the low / high byte
MOE_DEVINL uint32_t cvt_fp8x2(float lo, float hi, int fmt) {
  uint16_t r;
  if (fmt == MOE_FP8_E4M3)
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  else
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// 8 bf16 -> 8 codes (little-endian in a uint2)
MOE_DEVINL uint2 quant8(const uint4 &v, float scale, int fmt) {
  float f[8];
  bf16x8_to_f32(v, f);
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    w[i] = cvt_fp8x2(__fmul_rn(f[2 * i], scale), __fmul_rn(f[2 * i + 1], scale), fmt);
  return make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
}

// amax over rows [g * rpg, g * rpg + limit) of group g = blockIdx.y, where
// limit = rpg, or group_offsets[E] (clamped) when offsets are given.
__global__ void __launch_bounds__(256)
amax_kernel(const uint16_t *__restrict__ x, int64_t ldx, int64_t rpg, int cols,
            const int32_t *__restrict__ offsets, int E, float *__restrict__ amax) {
  const int g = blockIdx.y;
  int64_t rows = rpg;
  if (offsets != nullptr) rows = min(max((int64_t)__ldg(offsets + E), (int64_t)0), rpg);
  const uint16_t *base = x + (int64_t)g * rpg * ldx;
  float m = 0.0f;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const uint16_t *row = base + r * ldx;
    for (int c = threadIdx.x * 8; c < cols; c += 256 * 8) {
      float f[8];
      bf16x8_to_f32(ld_nc_v4(row + c), f);
#pragma unroll
      for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
    }
  }
  m = warp_max(m);
  __shared__ float s_m[8];
  if ((threadIdx.x & 31) == 0) s_m[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
#pragma unroll
    for (int w = 1; w < 8; ++w) m = fmaxf(m, s_m[w]);
    // non-negative floats order like their bit patterns
    if (m > 0.0f) atomicMax(reinterpret_cast<unsigned int *>(amax + g), __float_as_uint(m));
  }
}

// One 64 x 64 tile: row-wise codes to q, column-wise codes to qt.
//   PADDED (grouped activations, one scale): blockIdx.x walks the padded row
//   space; the tile's 64 padded rows belong to one group e and map to source
//   rows off_e + (j - poff_e) (zeros past the group's end).
//   else (weights, one scale per expert g = blockIdx.z): plain transpose of
//   each [rpg, cols] slab.
template <bool PADDED>
__global__ void __launch_bounds__(256)
quant_kernel(const uint16_t *__restrict__ x, int64_t ldx, int64_t rpg, int cols,
             const int32_t *__restrict__ offsets, int E, int64_t rows_cap,
             const float *__restrict__ amax, int fmt, uint8_t *__restrict__ q, int64_t ldq,
             int64_t stride_q, uint8_t *__restrict__ qt, int64_t ldqt, int64_t stride_qt,
             float *__restrict__ scale_inv) {
  __shared__ uint8_t tile[kQT][kQT + 16];
  __shared__ int s_poff[kMaxGroups + 1];
  const int g = PADDED ? 0 : blockIdx.z;
  const int64_t j0 = (int64_t)blockIdx.x * kQT;  // first (padded) row of the tile
  const float scale = scale_of(__ldg(amax + g), fmt);
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) scale_inv[g] = __frcp_rn(scale);

  int64_t src0;      // source row of padded row j0
  int64_t src_end;   // first source row past the tile's group
  if (PADDED) {
    // padded group starts: inclusive scan (one thread per group) of the
    // rounded-up sizes into s_poff[1..E]
    {
      const int t = threadIdx.x;
      int v = 0;
      if (t < E) {
        const int a = min(max(__ldg(offsets + t), 0), (int)rows_cap);
        const int b = max(min(__ldg(offsets + t + 1), (int)rows_cap), a);
        v = (b - a + kF8PadRows - 1) / kF8PadRows * kF8PadRows;
      }
      if (t == 0) s_poff[0] = 0;
      s_poff[t + 1] = v;
      __syncthreads();
      for (int o = 1; o < kMaxGroups; o <<= 1) {
        const int add = t >= o ? s_poff[t + 1 - o] : 0;
        __syncthreads();
        s_poff[t + 1] += add;
        __syncthreads();
      }
    }
    if (j0 >= s_poff[E]) return;
    int lo = 0, hi = E - 1;  // last group with s_poff[e] <= j0
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_poff[mid] <= j0) lo = mid;
      else hi = mid - 1;
    }
    const int e = lo;
    const int a = min(max(__ldg(offsets + e), 0), (int)rows_cap);
    const int b = max(min(__ldg(offsets + e + 1), (int)rows_cap), a);
    src0 = a + (j0 - s_poff[e]);
    src_end = b;
  } else {
    src0 = j0;
    src_end = rpg;
  }
  const uint16_t *xg = x + (int64_t)g * rpg * ldx;
  uint8_t *qg = q + (int64_t)g * stride_q;
  for (int ct = 0; ct < kQCT; ++ct) {
    const int c0 = (blockIdx.y * kQCT + ct) * kQT;
    if (c0 >= cols) break;
    if (ct > 0) __syncthreads();  // the previous tile's column-wise reads are done
    // load, quantize, write row-wise codes, keep the tile in shared memory
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int v = threadIdx.x + h * 256;
      const int i = v >> 3;            // tile row
      const int cc = (v & 7) * 8;      // tile column
      const int64_t r = src0 + i;
      const int c = c0 + cc;
      uint2 codes = make_uint2(0, 0);
      if (r < src_end && c < cols) {
        codes = quant8(ld_nc_v4(xg + r * ldx + c), scale, fmt);
        *reinterpret_cast<uint2 *>(qg + r * ldq + c) = codes;
      }
      *reinterpret_cast<uint2 *>(&tile[i][cc]) = codes;
    }
    __syncthreads();
    // column-wise: output row c (= input column), 16 consecutive padded rows
    {
      const int cr = threadIdx.x >> 2;       // tile column -> output row
      const int k16 = (threadIdx.x & 3) * 16;
      const int c = c0 + cr;
      const int64_t jj = j0 + k16;
      if (c < cols && (PADDED || jj < rpg)) {
        uint32_t w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          w[u] = 0;
#pragma unroll
          for (int b = 0; b < 4; ++b) w[u] |= (uint32_t)tile[k16 + 4 * u + b][cr] << (8 * b);
        }
        *reinterpret_cast<uint4 *>(qt + (int64_t)g * stride_qt + (int64_t)c * ldqt + jj) =
            make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
  }
}

}  // namespace

int64_t f8_padded_rows(int64_t rows_cap, int E) {
  const int64_t p = rows_cap + (int64_t)E * (kF8PadRows - 1);
  return (p + kF8PadRows - 1) / kF8PadRows * kF8PadRows;
}

cudaError_t launch_fp8_amax(const uint16_t *x, int64_t ldx, int64_t rows, int cols, int groups,
                            const int32_t *offsets, int E, float *amax, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(amax, 0, sizeof(float) * groups, s);
  if (e != cudaSuccess) return e;
  const int64_t rpg = rows / groups;
  if (rpg == 0) return cudaSuccess;
  const int want = 4 * num_sms() / groups + 1;
  dim3 grid((unsigned)std::min<int64_t>(rpg, std::max(want, 1)), groups);
  amax_kernel<<<grid, 256, 0, s>>>(x, ldx, rpg, cols, offsets, E, amax);
  return cudaGetLastError();
}

cudaError_t launch_fp8_quant_act(const uint16_t *x, int64_t ldx, const int32_t *offsets, int E,
                                 int64_t rows_cap, int cols, int fmt, const float *amax,
                                 uint8_t *q, int64_t ldq, uint8_t *qt, int64_t ldqt,
                                 float *scale_inv, cudaStream_t s) {
  const int64_t pr = f8_padded_rows(rows_cap, E);
  dim3 grid((unsigned)(pr / kQT), (cols + kQT * kQCT - 1) / (kQT * kQCT), 1);
  quant_kernel<true><<<grid, 256, 0, s>>>(x, ldx, rows_cap, cols, offsets, E, rows_cap, amax,
                                          fmt, q, ldq, 0, qt, ldqt, 0, scale_inv);
  return cudaGetLastError();
}

cudaError_t launch_fp8_quant_weights(const uint16_t *w, int E, int K, int N, int fmt,
                                     const float *amax, uint8_t *q, uint8_t *qt,
                                     float *scale_inv, cudaStream_t s) {
  dim3 grid((K + kQT - 1) / kQT, (N + kQT * kQCT - 1) / (kQT * kQCT), E);
  quant_kernel<false><<<grid, 256, 0, s>>>(w, N, K, N, nullptr, E, K, amax, fmt, q, N,
                                           (int64_t)K * N, qt, K, (int64_t)N * K, scale_inv);
  return cudaGetLastError();
}

}  // namespace moe
