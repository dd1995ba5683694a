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
#include <algorithm>

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

// Padded (atom-layout) row of row r of a [rows, .] matrix under the row maps
// that need no group offsets (PLAIN, TILES with E groups, SWIGLU).
MOE_DEVINL int64_t mapped_row(int64_t r, int64_t rows, int row_map, int E) {
  if (row_map == MOE_MX_ROWS_SWIGLU) {
    const int64_t F = rows / 2;
    const int64_t n = r < F ? r : r - F;
    return (n / 96) * 256 + (r < F ? 0 : 96) + n % 96;
  }
  if (row_map == MOE_MX_ROWS_TILES) {
    const int64_t G = rows / E;
    const int64_t e = r / G, n = r - e * G;
    return (e * ((G + 191) / 192) + n / 192) * 256 + n % 192;
  }
  return r;
}

// Byte of the scale of (padded row pr, 32-column block cb) in atoms of a
// matrix with `cols` columns.
MOE_DEVINL int64_t scale_byte(int64_t pr, int cb, int cols) {
  const int64_t atom = (pr >> 7) * (cols >> 7) + (cb >> 2);
  const int rw = (int)(pr & 127);
  return atom * 512 + (rw & 31) * 16 + (rw >> 5) * 4 + (cb & 3);
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
  } else {
    pr = mapped_row(r, rows, row_map, E);
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
  sf[scale_byte(pr, cb, cols)] = code;
}

// One 32-element block: its E8M0 code and the codes of its elements (8
// little-endian words); v is overwritten.
MOE_DEVINL uint8_t quant_block(float *v, int fmt, uint32_t *w) {
  float amax = 0.0f;
  bool finite = true;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const float a = fabsf(v[i]);
    finite &= a <= 3.402823466e38f;
    amax = fmaxf(amax, a);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) w[i] = 0;
  if (!finite) return 0xFF;
  const int emax = fmt == MOE_FP8_E4M3 ? 8 : 15;
  const int s = amax > 0.0f ? max(-127, min(127, floor_log2(amax) - emax)) : -127;
  const float inv = __uint_as_float((uint32_t)(127 - s) << 23);
#pragma unroll
  for (int i = 0; i < 8; ++i)
    w[i] = cvt_f8x2(v[4 * i] * inv, v[4 * i + 1] * inv, fmt) |
           (cvt_f8x2(v[4 * i + 2] * inv, v[4 * i + 3] * inv, fmt) << 16);
  return (uint8_t)(s + 127);
}

// Both block-scaled copies of a grouped matrix from one read.  Block = a
// tile of 64 padded rows x 128 columns (padded rows: group e's rows at poff_e
// + i, zeros past the group; 16 KB, four 16-byte loads in flight per thread),
// staged in shared memory; then every thread quantizes one row's 32-column
// block (row-wise codes q, blocks along the columns) and one column's 32-row
// block (column-wise codes qt [cols, padded rows], blocks along each group's
// rows).
constexpr int kMx2Rows = 64, kMx2Cols = 128;
constexpr int kMx2Pitch = kMx2Cols * 2 + 16;  // bytes per staged row: 16 spare keep banks apart

// Loads tile (tile_x, tile_y) of x into a staging buffer with 16-byte
// asynchronous copies, rows past the group as zeros (a copy of 0 source bytes
// fills its 16 bytes with zeros).
MOE_DEVINL void mx2_load_tile(uint8_t *buf, const uint16_t *x, int64_t ldx, int64_t g0,
                              int64_t gsz, int64_t i0, int c0, int tid) {
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    const int idx = tid + 256 * h;
    const int rr = idx >> 4, ch = idx & 15;
    const bool in = i0 + rr < gsz;
    const uint16_t *src = in ? x + (g0 + i0 + rr) * ldx + c0 + ch * 8 : x;
    const uint32_t dst = static_cast<uint32_t>(__cvta_generic_to_shared(buf + rr * kMx2Pitch + ch * 16));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
                 "r"(in ? 16 : 0)
                 : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// Persistent: block b quantizes tiles b, b + grid, ... (64 padded rows x 128
// columns each, tile t at column tile t % col_tiles, row tile t / col_tiles);
// the next tile's load runs while this one is quantized (two staging buffers).
__global__ void __launch_bounds__(256, 4)
mx_quantize_2x_kernel(const uint16_t *__restrict__ x, int64_t ldx, int64_t rows, int cols,
                      int fmt, const int32_t *__restrict__ offsets, int E,
                      uint8_t *__restrict__ q, int64_t ldq, int q_map, uint8_t *__restrict__ sfq,
                      uint8_t *__restrict__ qt, int64_t ldqt, int qt_cols, int qt_map,
                      uint8_t *__restrict__ sfqt, int64_t n_tiles) {
  __shared__ int s_poff[kMxMaxE + 1];
  __shared__ __align__(16) uint8_t tiles[2][kMx2Rows * kMx2Pitch];
  __shared__ __align__(16) uint8_t s_code[kMx2Rows][4];  // row-wise scale codes of a tile
  const int tid = threadIdx.x;
  // TILES (the weights): a tile's 64 rows are 64 consecutive padded rows
  // from a multiple of 64, so its row-wise scale codes fill 8 consecutive
  // bytes of each of 32 atom lines (rows r0 and r0 + 32, blocks 0-3): written
  // as 32 8-byte stores instead of 256 single bytes (weights 6% faster; the
  // same for GROUPED, whose rows share that property, measured 1-2% slower)
  const bool sc_packed = q_map == MOE_MX_ROWS_TILES;
  if (tid < 32) {  // padded group starts (warp-shuffle scan)
    int carry = 0;
    for (int c0 = 0; c0 < E; c0 += 32) {
      const int e = c0 + tid;
      const int sz = e < E ? max(__ldg(offsets + e + 1) - __ldg(offsets + e), 0) : 0;
      const int pad = (sz + 127) / 128 * 128;
      int incl = pad;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (tid >= o) incl += y;
      }
      if (e < E) s_poff[e] = carry + incl - pad;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (tid == 0) s_poff[E] = carry;
  }
  __syncthreads();
  const int col_tiles = cols / kMx2Cols;
  const int64_t prows = s_poff[E];
  // tile t -> (group, its first row in the group, first padded row, first column)
  struct Tile {
    int64_t g0, gsz, i0, pr0;
    int c0;
    bool live;
  };
  auto locate = [&](int64_t t) {
    Tile ti;
    ti.pr0 = (t / col_tiles) * kMx2Rows;
    ti.c0 = (int)(t % col_tiles) * kMx2Cols;
    ti.live = t < n_tiles && ti.pr0 < prows;
    int lo = 0, hi = E - 1;  // the group of the tile (tiles never straddle groups)
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_poff[mid] <= ti.pr0) lo = mid;
      else hi = mid - 1;
    }
    ti.g0 = min(max((int64_t)__ldg(offsets + lo), (int64_t)0), rows);
    ti.gsz = min(max((int64_t)__ldg(offsets + lo + 1), ti.g0), rows) - ti.g0;
    ti.i0 = ti.pr0 - s_poff[lo];
    return ti;
  };
  int64_t t = blockIdx.x;
  Tile cur = locate(t);
  if (cur.live) mx2_load_tile(tiles[0], x, ldx, cur.g0, cur.gsz, cur.i0, cur.c0, tid);
  for (int it = 0; cur.live; ++it) {
    uint8_t *tile = tiles[it & 1];
    const Tile nxt = locate(t + gridDim.x);
    // this tile's copies landed (every thread's), and every thread is done
    // with the buffer the next load overwrites (quantized one iteration ago)
    asm volatile("cp.async.wait_group 0;" ::: "memory");
    __syncthreads();
    if (nxt.live) mx2_load_tile(tiles[(it + 1) & 1], x, ldx, nxt.g0, nxt.gsz, nxt.i0, nxt.c0, tid);
    const int64_t g0 = cur.g0, gsz = cur.gsz, i0 = cur.i0, pr0 = cur.pr0;
    const int c0 = cur.c0;
    float v[32];
    uint32_t w[8];
    if (q != nullptr) {
      const int rr = tid >> 2, blk = tid & 3;
      uint8_t code = 0;  // rows past the group: the smallest scale, no codes written
      if (i0 + rr < gsz) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
          bf16x8_to_f32(
              *reinterpret_cast<const uint4 *>(tile + rr * kMx2Pitch + blk * 64 + i * 16),
              v + 8 * i);
        code = quant_block(v, fmt, w);
        const int64_t r = g0 + i0 + rr;
        uint4 *dst = reinterpret_cast<uint4 *>(q + r * ldq + c0 + blk * 32);
        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
        if (!sc_packed) {
          const int64_t pr =
              q_map == MOE_MX_ROWS_GROUPED ? pr0 + rr : mapped_row(r, rows, q_map, E);
          sfq[scale_byte(pr, (c0 >> 5) + blk, cols)] = code;
        }
      }
      if (sc_packed) {
        s_code[rr][blk] = code;
        __syncthreads();
        if (tid < 32) {
          // the tile's first padded row (a multiple of 64) and its atom line
          const int64_t pf = mapped_row(g0 + i0, rows, q_map, E);
          const uint32_t lo = *reinterpret_cast<const uint32_t *>(s_code[tid]);
          const uint32_t hi = *reinterpret_cast<const uint32_t *>(s_code[tid + 32]);
          // byte of (row pf + tid, block c0 / 32), 8-byte aligned; the next
          // four bytes hold row pf + tid + 32
          *reinterpret_cast<uint2 *>(sfq + scale_byte(pf + tid, c0 >> 5, cols)) =
              make_uint2(lo, hi);
        }
      }
    }
    const int c = tid & 127, half = tid >> 7;  // column, and which 32 of the 64 rows
    const int64_t pb = pr0 + 32 * half;        // the block's first padded row
    if (qt != nullptr && pb + 32 <= qt_cols) {
      const uint16_t *col = reinterpret_cast<const uint16_t *>(tile + 32 * half * kMx2Pitch) + c;
#pragma unroll
      for (int rr = 0; rr < 32; ++rr)
        v[rr] = __uint_as_float((uint32_t)col[rr * (kMx2Pitch / 2)] << 16);
      const uint8_t code = quant_block(v, fmt, w);
      const int64_t n = c0 + c;  // row of qt
      uint4 *dst = reinterpret_cast<uint4 *>(qt + n * ldqt + pb);
      dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
      dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
      const int64_t pr = mapped_row(n, cols, qt_map, 1);
      sfqt[scale_byte(pr, (int)(pb >> 5), qt_cols)] = code;
    }
    cur = nxt;
    t += gridDim.x;
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}

}  // namespace

int64_t mx_atom_rows(int64_t rows, int row_map, int E) {
  if (row_map == MOE_MX_ROWS_GROUPED) return f8_padded_rows(rows, E) / 128;
  if (row_map == MOE_MX_ROWS_SWIGLU) return 2 * ((rows / 2 + 95) / 96);
  if (row_map == MOE_MX_ROWS_TILES) return 2 * (int64_t)E * ((rows / E + 191) / 192);
  return (rows + 127) / 128;
}

cudaError_t launch_mx_quantize_2x(const uint16_t *x, int64_t ldx, int64_t rows, int cols, int fmt,
                                  const int32_t *offsets, int E, uint8_t *q, int64_t ldq,
                                  int q_map, uint8_t *sfq, uint8_t *qt, int64_t ldqt,
                                  int qt_cols, int qt_map, uint8_t *sfqt, cudaStream_t s) {
  if (rows == 0) return cudaSuccess;
  // tiles over the padded rows (an upper bound: the groups' padded total is
  // known on the device only), a persistent grid of resident blocks
  const int64_t n_tiles = (int64_t)(cols / kMx2Cols) * (f8_padded_rows(rows, E) / kMx2Rows);
  static int per_sm = 0;
  if (per_sm == 0 &&
      cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, mx_quantize_2x_kernel, 256, 0) !=
          cudaSuccess)
    per_sm = 1;
  const int64_t grid = std::min<int64_t>(n_tiles, (int64_t)std::max(per_sm, 1) * num_sms());
  if (grid == 0) return cudaSuccess;
  mx_quantize_2x_kernel<<<(unsigned)grid, 256, 0, s>>>(x, ldx, rows, cols, fmt, offsets, E, q, ldq,
                                                       q_map, sfq, qt, ldqt, qt_cols, qt_map,
                                                       sfqt, n_tiles);
  return cudaGetLastError();
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
