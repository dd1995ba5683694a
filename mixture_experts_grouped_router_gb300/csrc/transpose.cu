// Column-wise (transposed) bf16 copy of a permuted activation, in the padded
// group layout the weight-gradient GEMM reads K-major: group e's rows land in
// columns [poff_e, poff_e + size_e) with poff_e the sum of the previous group
// sizes each rounded up to kF8PadRows, and the columns up to the next group
// are zero (the same layout as the FP8 column-wise codes).
//   MaxText PR #4295 "Overlap moe comms with collective matmul", Testing: the
//   tgmm W_e = A_e^T B_e over each expert's rows; here A_e^T is read from
//   this copy so that its operand tiles are K-major.
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kTT = 64;   // tile: 64 rows x 64 columns
constexpr int kTCT = 8;   // column tiles per block (amortises the group-offset scan)

__global__ void __launch_bounds__(256)
transpose_pad_kernel(const uint16_t *__restrict__ x, int64_t ldx, int cols,
                     const int32_t *__restrict__ offsets, int E, int64_t rows_cap,
                     uint16_t *__restrict__ xt, int64_t ldxt) {
  __shared__ uint16_t tile[kTT][kTT + 8];
  __shared__ int s_poff[kMaxGroups + 1];
  const int64_t j0 = (int64_t)blockIdx.x * kTT;  // first padded row (output column)
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
  int lo = 0, hi = E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_poff[mid] <= j0) lo = mid;
    else hi = mid - 1;
  }
  const int a = min(max(__ldg(offsets + lo), 0), (int)rows_cap);
  const int b = max(min(__ldg(offsets + lo + 1), (int)rows_cap), a);
  const int64_t src0 = a + (j0 - s_poff[lo]);
  for (int ct = 0; ct < kTCT; ++ct) {
    const int c0 = (blockIdx.y * kTCT + ct) * kTT;
    if (c0 >= cols) break;
    if (ct > 0) __syncthreads();  // the previous tile's transposed reads are done
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int v = threadIdx.x + h * 256;
      const int i = v >> 3;            // tile row
      const int cc = (v & 7) * 8;      // tile column
      const int64_t r = src0 + i;
      const int c = c0 + cc;
      uint4 val = make_uint4(0, 0, 0, 0);
      if (r < b && c < cols) val = ld_nc_v4(x + r * ldx + c);
      *reinterpret_cast<uint4 *>(&tile[i][cc]) = val;
    }
    __syncthreads();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int v = threadIdx.x + h * 256;
      const int cr = v >> 3;            // output row within the tile (= input column)
      const int k8 = (v & 7) * 8;       // 8 consecutive output columns
      const int c = c0 + cr;
      if (c < cols) {
        uint32_t w[4];
#pragma unroll
        for (int u = 0; u < 4; ++u)
          w[u] = (uint32_t)tile[k8 + 2 * u][cr] | ((uint32_t)tile[k8 + 2 * u + 1][cr] << 16);
        st_v4(xt + (int64_t)c * ldxt + j0 + k8, make_uint4(w[0], w[1], w[2], w[3]));
      }
    }
  }
}

}  // namespace

cudaError_t launch_transpose_act(const uint16_t *x, int64_t ldx, const int32_t *offsets, int E,
                                 int64_t rows_cap, int cols, uint16_t *xt, int64_t ldxt,
                                 cudaStream_t s) {
  const int64_t pr = f8_padded_rows(rows_cap, E);
  dim3 grid((unsigned)(pr / kTT), (cols + kTT * kTCT - 1) / (kTT * kTCT), 1);
  transpose_pad_kernel<<<grid, 256, 0, s>>>(x, ldx, cols, offsets, E, rows_cap, xt, ldxt);
  return cudaGetLastError();
}

}  // namespace moe
