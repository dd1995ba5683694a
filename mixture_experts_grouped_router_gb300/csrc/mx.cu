// Block-scaled 8-bit quantization (MXFP8): one power-of-two scale per 32
// consecutive elements of a row, the codes of the elements divided by it.
//
// TransformerEngine PR #2912, wi-fusion commit, FP8 note: the block-scaled
// recipes (MXFP8, NVFP4) keep one scale per block, so fusing wi_0 and wi_1
// leaves them unaffected.  The arithmetic is the OCP Microscaling (MX) v1.0
// definition: scale X = 2^s, s = floor(log2 amax) - emax (emax 8 for E4M3,
// 15 for E5M2), clamped to [-127, 127] and stored as the E8M0 code s + 127;
// element code = round-to-nearest-even of x / X saturated to the largest
// finite value.  A block of zeros takes the smallest scale (code 0); a block
// holding a NaN or an infinity takes the NaN scale (0xFF) and zero codes.
//
// Scale layout: the tensor cores read a tile's scales from tensor memory,
// copied there from shared memory in 512-byte atoms of 128 rows x 4 blocks:
// row r = r0 + 32 r1 (r0 < 32, r1 < 4), block j < 4 at byte 16 r0 + 4 r1 + j.
// Atom (ar, ac) covers atom row ar (128 rows) and columns [128 ac, 128 ac +
// 128) and sits at byte (ar * cols / 128 + ac) * 512.  The atom row of a
// matrix row depends on how the GEMM tiles it (row_map; the B operands are
// tiled by 192 rows, which take two atom rows each, the second half used):
//   PLAIN    r / 128 (A operands: weight-gradient copies of activations)
//   GROUPED  the expert's padded tile: rows of group e start at atom row
//            poff_e / 128 (poff_e = the group starts rounded up to 128, as in
//            the column-wise copies), so a GEMM row tile of one expert reads
//            one atom row
//   TILES    E equal groups of G = rows / E rows (experts' weights, or one
//            group): row n of group e in tile t = n / 192 at padded row
//            256 (e ceil(G / 192) + t) + n % 192
//   SWIGLU   a fused [gate | up] weight (2F rows) in the order of the SwiGLU
//            tiles: tile t holds gate rows [96 t, 96 t + 96) then up rows
//            [F + 96 t, F + 96 t + 96), at padded rows 256 t ...
#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kMxThreads = 256;  // one thread per 32-element block
constexpr int kMxMaxE = 256;

MOE_DEVINL uint32_t cvt_f8x2(float lo, float hi, int fmt) {
  uint16_t r;
  if (fmt == MOE_FP8_E4M3)
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  else
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// floor(log2(a)) of a finite a > 0 from its bit fields (subnormals included).
MOE_DEVINL int floor_log2(float a) {
  const uint32_t b = __float_as_uint(a);
  const int e = (int)((b >> 23) & 0xFF);
  if (e > 0) return e - 127;
  return (31 - __clz(b & 0x7FFFFF)) - 149;
}

__global__ void __launch_bounds__(kMxThreads)
mx_quantize_kernel(const uint16_t *__restrict__ x, int64_t ldx, int64_t rows, int cols, int fmt,
                   int row_map, const int32_t *__restrict__ offsets, int E,
                   uint8_t *__restrict__ q, int64_t ldq, uint8_t *__restrict__ sf) {
  __shared__ int s_poff[kMxMaxE];  // padded start of each group (GROUPED)
  const int nb = cols >> 5;  // blocks per row
  const int64_t b = (int64_t)blockIdx.x * kMxThreads + threadIdx.x;
  const int64_t r = b / nb;
  const int cb = (int)(b - r * nb);
  if (row_map == MOE_MX_ROWS_GROUPED) {
    // the group starts rounded up to whole atoms, summed (warp-shuffle scan)
    if (threadIdx.x < 32) {
      int carry = 0;
      for (int c0 = 0; c0 < E; c0 += 32) {
        const int e = c0 + threadIdx.x;
        const int sz = e < E ? max(__ldg(offsets + e + 1) - __ldg(offsets + e), 0) : 0;
        const int pad = (sz + 127) / 128 * 128;
        int incl = pad;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          if ((int)threadIdx.x >= o) incl += y;
        }
        if (e < E) s_poff[e] = carry + incl - pad;
        carry += __shfl_sync(0xffffffffu, incl, 31);
      }
    }
    __syncthreads();
  }
  if (r >= rows) return;
  // the row's place in the scale atoms
  int64_t pr = r;
  if (row_map == MOE_MX_ROWS_GROUPED) {
    const int R = min(max(__ldg(offsets + E), 0), (int)rows);
    if (r >= R) return;
    int lo = 0, hi = E - 1;  // last group starting at or before r
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (__ldg(offsets + mid) <= r) lo = mid;
      else hi = mid - 1;
    }
    pr = s_poff[lo] + (r - __ldg(offsets + lo));
  } else if (row_map == MOE_MX_ROWS_SWIGLU) {
    const int64_t F = rows / 2;
    const int64_t n = r < F ? r : r - F;
    pr = (n / 96) * 256 + (r < F ? 0 : 96) + n % 96;
  } else if (row_map == MOE_MX_ROWS_TILES) {
    const int64_t G = rows / E;
    const int64_t e = r / G, n = r - e * G;
    pr = (e * ((G + 191) / 192) + n / 192) * 256 + n % 192;
  }
  const uint4 *src = reinterpret_cast<const uint4 *>(x + r * ldx + cb * 32);
  float v[32];
#pragma unroll
  for (int i = 0; i < 4; ++i) bf16x8_to_f32(ld_nc_v4(src + i), v + 8 * i);
  float amax = 0.0f;
  bool finite = true;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float a = fabsf(v[i]);
    finite &= a <= 3.402823466e38f;  // false for inf and NaN
    amax = fmaxf(amax, a);
  }
  uint8_t code;
  uint32_t w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  if (!finite) {
    code = 0xFF;
  } else {
    const int emax = fmt == MOE_FP8_E4M3 ? 8 : 15;
    const int s = amax > 0.0f ? max(-127, min(127, floor_log2(amax) - emax)) : -127;
    code = (uint8_t)(s + 127);
    // 2^-s is a normal float for every scale a finite bf16 block can take
    // (s <= 128 - emax); x * 2^-s is exact
    const float inv = __uint_as_float((uint32_t)(127 - s) << 23);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      w[i] = cvt_f8x2(v[4 * i] * inv, v[4 * i + 1] * inv, fmt) |
             (cvt_f8x2(v[4 * i + 2] * inv, v[4 * i + 3] * inv, fmt) << 16);
  }
  uint4 *dst = reinterpret_cast<uint4 *>(q + r * ldq + cb * 32);
  dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
  dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
  const int64_t atom = (pr >> 7) * (cols >> 7) + (cb >> 2);
  const int rw = (int)(pr & 127);
  sf[atom * 512 + (rw & 31) * 16 + (rw >> 5) * 4 + (cb & 3)] = code;
}

}  // namespace

int64_t mx_atom_rows(int64_t rows, int row_map, int E) {
  if (row_map == MOE_MX_ROWS_GROUPED) return f8_padded_rows(rows, E) / 128;
  if (row_map == MOE_MX_ROWS_SWIGLU) return 2 * ((rows / 2 + 95) / 96);
  if (row_map == MOE_MX_ROWS_TILES) return 2 * (int64_t)E * ((rows / E + 191) / 192);
  return (rows + 127) / 128;
}

cudaError_t launch_mx_quantize(const uint16_t *x, int64_t ldx, int64_t rows, int cols, int fmt,
                               int row_map, const int32_t *offsets, int E, uint8_t *q,
                               int64_t ldq, uint8_t *sf, cudaStream_t s) {
  const int64_t blocks = rows * (cols / 32);
  if (blocks == 0) return cudaSuccess;
  mx_quantize_kernel<<<(unsigned)((blocks + kMxThreads - 1) / kMxThreads), kMxThreads, 0, s>>>(
      x, ldx, rows, cols, fmt, row_map, offsets, E, q, ldq, sf);
  return cudaGetLastError();
}

}  // namespace moe
