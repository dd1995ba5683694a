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

// amax over rows [g * rpg, g * rpg + limit) of every group g, where limit =
// rpg, or group_offsets[E] (clamped) when offsets are given (groups == 1).
// The groups' rows, laid end to end, are split into one contiguous range per
// block (a persistent grid of the resident blocks); a block reduces and
// publishes its maximum once per group its range touches.
// |x| of a bf16 is its bit pattern with the sign cleared, and non-negative
// floats order like their bit patterns, so the max is an unsigned max of the
// 16-bit patterns (two per word, __vmaxu2); a NaN pattern is above every
// finite one and infinity, so a NaN input makes amax NaN.  Each thread keeps
// kAmaxRows rows of loads in flight.
constexpr int kAmaxRows = 4;
constexpr int kAmaxThreads = 256;

__global__ void __launch_bounds__(kAmaxThreads)
amax_kernel(const uint16_t *__restrict__ x, int64_t ldx, int64_t rpg, int cols, int groups,
            const int32_t *__restrict__ offsets, int E, float *__restrict__ amax) {
  __shared__ uint32_t s_m[kAmaxThreads / 32];
  int64_t limit = rpg;
  if (offsets != nullptr) limit = min(max((int64_t)__ldg(offsets + E), (int64_t)0), rpg);
  const int64_t total = offsets != nullptr ? limit : (int64_t)groups * rpg;
  // this block's range of rows, in whole kAmaxRows steps
  const int64_t steps = (total + kAmaxRows - 1) / kAmaxRows;
  const int64_t per = (steps + gridDim.x - 1) / gridDim.x * kAmaxRows;
  const int64_t begin = (int64_t)blockIdx.x * per;
  const int64_t end = min(begin + per, total);
  if (begin >= end) return;
  for (int g = (int)(begin / rpg); (int64_t)g * rpg < end; ++g) {
    const int64_t lo = max(begin - (int64_t)g * rpg, (int64_t)0);
    const int64_t hi = min(end - (int64_t)g * rpg, limit);
    const uint16_t *base = x + (int64_t)g * rpg * ldx;
    uint32_t m2 = 0;  // two running maxima of 16-bit patterns
    for (int64_t r0 = lo; r0 < hi; r0 += kAmaxRows) {
      for (int c = threadIdx.x * 8; c < cols; c += kAmaxThreads * 8) {
        uint4 v[kAmaxRows];
#pragma unroll
        for (int u = 0; u < kAmaxRows; ++u)
          v[u] = r0 + u < hi ? ld_nc_v4(base + (r0 + u) * ldx + c) : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int u = 0; u < kAmaxRows; ++u) {
          m2 = __vmaxu2(m2, v[u].x & 0x7FFF7FFFu);
          m2 = __vmaxu2(m2, v[u].y & 0x7FFF7FFFu);
          m2 = __vmaxu2(m2, v[u].z & 0x7FFF7FFFu);
          m2 = __vmaxu2(m2, v[u].w & 0x7FFF7FFFu);
        }
      }
    }
    uint32_t m = max(m2 & 0xFFFFu, m2 >> 16);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
    __syncthreads();  // s_m is free (the previous group's reduction is read)
    if ((threadIdx.x & 31) == 0) s_m[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
#pragma unroll
      for (int w = 1; w < kAmaxThreads / 32; ++w) m = max(m, s_m[w]);
      // the fp32 bit pattern of the bf16 value orders the same way
      if (m != 0) atomicMax(reinterpret_cast<unsigned int *>(amax + g), m << 16);
    }
  }
}

// 4 x 4 byte transpose: row[r] holds the codes of one row, column c at byte
// c; col[c] gets column c, row r at byte r.
MOE_DEVINL void transpose4x4(const uint32_t row[4], uint32_t col[4]) {
  const uint32_t t0 = __byte_perm(row[0], row[1], 0x5140);  // a0 b0 a1 b1
  const uint32_t t1 = __byte_perm(row[2], row[3], 0x5140);  // c0 d0 c1 d1
  const uint32_t t2 = __byte_perm(row[0], row[1], 0x7362);  // a2 b2 a3 b3
  const uint32_t t3 = __byte_perm(row[2], row[3], 0x7362);  // c2 d2 c3 d3
  col[0] = __byte_perm(t0, t1, 0x5410);
  col[1] = __byte_perm(t0, t1, 0x7632);
  col[2] = __byte_perm(t2, t3, 0x5410);
  col[3] = __byte_perm(t2, t3, 0x7632);
}

// 64 x 64 tiles, kQCT of them along the columns per block: row-wise codes to
// q, column-wise codes to qt.
//   PADDED (grouped activations, one scale): blockIdx.x walks the padded row
//   space; the tile's 64 padded rows belong to one group e and map to source
//   rows off_e + (j - poff_e) (zeros past the group's end).
//   else (weights, one scale per expert g = blockIdx.z): plain transpose of
//   each [rpg, cols] slab.
// Row phase: a thread quantizes 8 codes of each of two rows, stores them
// row-wise and as words into the tile (rows of 17 words); the next tile's
// loads are issued before the barrier.  Column phase: a thread reads a 4 x 4
// block of codes as four words (the 17-word rows make the warp's reads
// conflict-free), transposes it with byte permutes and stores four 4-byte
// column pieces (8 lanes per column piece: whole 32-byte sectors).
template <bool PADDED>
__global__ void __launch_bounds__(256)
quant_kernel(const uint16_t *__restrict__ x, int64_t ldx, int64_t rpg, int cols,
             const int32_t *__restrict__ offsets, int E, int64_t rows_cap,
             const float *__restrict__ amax, int fmt, uint8_t *__restrict__ q, int64_t ldq,
             int64_t stride_q, uint8_t *__restrict__ qt, int64_t ldqt, int64_t stride_qt,
             float *__restrict__ scale_inv) {
  constexpr int kRowWords = kQT / 4 + 1;
  __shared__ uint32_t tile[kQT][kRowWords];
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
  uint8_t *qtg = qt + (int64_t)g * stride_qt;
  const int cbase = blockIdx.y * kQCT * kQT;
  const int ntiles = min(kQCT, (cols - cbase + kQT - 1) / kQT);

  // row phase: element v = threadIdx.x + h * 256 is tile row v >> 3, columns
  // (v & 7) * 8 .. + 7
  auto load = [&](int ct, uint4 raw[2]) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int v = threadIdx.x + h * 256;
      const int64_t r = src0 + (v >> 3);
      const int c = cbase + ct * kQT + (v & 7) * 8;
      raw[h] = r < src_end && c < cols ? ld_nc_v4(xg + r * ldx + c) : make_uint4(0, 0, 0, 0);
    }
  };
  // column phase: rows 4 rq .. 4 rq + 3, columns 4 cq .. 4 cq + 3 of the tile
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cq = 4 * (warp & 3) + (lane >> 3);
  const int rq = 8 * (warp >> 2) + (lane & 7);
  const int64_t jj = j0 + 4 * rq;
  const bool rows_ok = PADDED || jj < rpg;

  uint4 raw[2];
  load(0, raw);
  for (int ct = 0; ct < ntiles; ++ct) {
    const int c0 = cbase + ct * kQT;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int v = threadIdx.x + h * 256;
      const int i = v >> 3;
      const int cc = (v & 7) * 8;
      const int64_t r = src0 + i;
      const int c = c0 + cc;
      uint2 codes = make_uint2(0, 0);
      if (r < src_end && c < cols) {
        codes = quant8(raw[h], scale, fmt);
        *reinterpret_cast<uint2 *>(qg + r * ldq + c) = codes;
      }
      tile[i][cc / 4] = codes.x;
      tile[i][cc / 4 + 1] = codes.y;
    }
    if (ct + 1 < ntiles) load(ct + 1, raw);
    __syncthreads();
    {
      uint32_t rw[4], cw[4];
#pragma unroll
      for (int r = 0; r < 4; ++r) rw[r] = tile[4 * rq + r][cq];
      transpose4x4(rw, cw);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int c = c0 + 4 * cq + i;
        if (c < cols && rows_ok)
          *reinterpret_cast<uint32_t *>(qtg + (int64_t)c * ldqt + jj) = cw[i];
      }
    }
    __syncthreads();  // the tile is read before the next row phase writes it
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
  // one wave: every block resident at once
  static int per_sm = 0;
  if (per_sm == 0) {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, amax_kernel, kAmaxThreads, 0) !=
            cudaSuccess ||
        n < 1)
      n = 1;
    per_sm = n;
  }
  const int64_t steps = (rows + kAmaxRows - 1) / kAmaxRows;
  const unsigned grid = (unsigned)std::max<int64_t>(
      1, std::min<int64_t>(steps, (int64_t)per_sm * num_sms()));
  amax_kernel<<<grid, kAmaxThreads, 0, s>>>(x, ldx, rpg, cols, groups, offsets, E, amax);
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
