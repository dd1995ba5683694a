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

// The 64 x 64 tile sits in shared memory as 64 rows of 32 words (two bf16 a
// word), the 16-byte chunk j of row i stored at chunk j ^ ((i >> 3) & 7).
// Row phase: a thread loads 8 values of each of two rows (the next tile's
// loads are issued before the barrier) and stores them as one chunk each
// (a warp's four rows fill all 32 banks).  Column phase: thread (row octet
// ro, column pair cp) reads the pair's word from 8 rows (ro = lane & 7 and
// the warp's four column pairs share a chunk index that the swizzle spreads
// over all 32 banks), splits the words into two 8-row column pieces with byte
// permutes and stores each as 16 bytes (8 lanes write one 128-byte line).
MOE_DEVINL uint32_t tile_word(int i, int w) { return i * 32 + ((((w >> 2) ^ (i >> 3)) & 7) << 2) + (w & 3); }

__global__ void __launch_bounds__(256)
transpose_pad_kernel(const uint16_t *__restrict__ x, int64_t ldx, int cols,
                     const int32_t *__restrict__ offsets, int E, int64_t rows_cap,
                     uint16_t *__restrict__ xt, int64_t ldxt) {
  __shared__ __align__(16) uint32_t tile[kTT * kTT / 2];
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
  const int cbase = blockIdx.y * kTCT * kTT;
  const int ntiles = min(kTCT, (cols - cbase + kTT - 1) / kTT);

  // row phase: element v = threadIdx.x + h * 256 is tile row v >> 3, chunk v & 7
  auto load = [&](int ct, uint4 raw[2]) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int v = threadIdx.x + h * 256;
      const int64_t r = src0 + (v >> 3);
      const int c = cbase + ct * kTT + (v & 7) * 8;
      raw[h] = r < b && c < cols ? ld_nc_v4(x + r * ldx + c) : make_uint4(0, 0, 0, 0);
    }
  };
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ro = lane & 7;               // output columns 8 ro .. 8 ro + 7 of the tile
  const int cp = 4 * warp + (lane >> 3); // input columns 2 cp, 2 cp + 1

  uint4 raw[2];
  load(0, raw);
  for (int ct = 0; ct < ntiles; ++ct) {
    const int c0 = cbase + ct * kTT;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int v = threadIdx.x + h * 256;
      *reinterpret_cast<uint4 *>(&tile[tile_word(v >> 3, (v & 7) * 4)]) = raw[h];
    }
    if (ct + 1 < ntiles) load(ct + 1, raw);
    __syncthreads();
    {
      uint32_t w[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) w[r] = tile[tile_word(8 * ro + r, cp)];
      uint32_t lo4[4], hi4[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        lo4[m] = __byte_perm(w[2 * m], w[2 * m + 1], 0x5410);  // column 2 cp
        hi4[m] = __byte_perm(w[2 * m], w[2 * m + 1], 0x7632);  // column 2 cp + 1
      }
      const int c = c0 + 2 * cp;
      uint16_t *dst = xt + (int64_t)c * ldxt + j0 + 8 * ro;
      if (c < cols) st_v4(dst, make_uint4(lo4[0], lo4[1], lo4[2], lo4[3]));
      if (c + 1 < cols) st_v4(dst + ldxt, make_uint4(hi4[0], hi4[1], hi4[2], hi4[3]));
    }
    __syncthreads();  // the tile is read before the next row phase writes it
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
