// Grouped GEMMs of the MoE expert FFN on the sm_103a tensor cores.
//
// moe_gmm  (ragged M): for every expert e, rows [off_e, off_e+1) of A times
//          B_e, with the SwiGLU forward / backward or plain epilogue fused.
//          TransformerEngine PR #2912 "[JAX] Add an MoE Block (Layer) that
//          compound router, permutation, groupedGEMM and communication":
//          the expert FFN's grouped GEMMs, [wi_0 | wi_1] fused into one
//          up-projection (wi-fusion commit); MaxText PR #4295 "Overlap moe
//          comms with collective matmul", review threads on the gmm kernel:
//          transposed rhs and the in-place partial sum.
// moe_tgmm (ragged K): W_e = A_e^T B_e over the rows of expert e; an expert
//          without rows gets exact zeros (MaxText PR #4295, Testing).
//
// Design (persistent, one CTA per SM, CTAs in clusters of two whose pair
// issues 2-SM MMAs (tcgen05 cta_group::2, M = 256) on adjacent 128-row tiles
// of the same expert and one 256-column tile; warp-specialised):
//   warp 0      TMA producer: each CTA loads its own 128-row A tile and its
//               half (128 columns) of the B tile for every K block, both
//               completing on the leader CTA's barrier (32 KB per CTA and
//               stage, 6 stages; 5 for the SwiGLU forward that adds a
//               partial sum, whose epilogue needs more staging).  128-byte
//               swizzle throughout; a K block is one 128-byte row per tile
//               row (64 bf16 or 128 8-bit codes).
//   warp 1      TMEM owner; in the leader CTA the MMA issuer: kind::f16
//               (bf16) or kind::f8f6f4 (E4M3 / E5M2 codes), fp32 accumulators
//               in TMEM (two 256-column accumulators so that the epilogue of
//               one tile overlaps the mainloop of the next).  Stages and
//               finished accumulators are signalled to both CTAs by
//               multicast commits.
//   warps 2-5   epilogue, one warp per TMEM lane quarter (every GEMM):
//               tcgen05.ld of one
//               TMEM lane (= one output row) per thread, fused SwiGLU /
//               partial-sum / bias / FP8-dequantization / cast; each warp
//               stages its 32x32 output blocks (32x64 for a bf16 weight
//               gradient) in swizzled shared memory and writes them with TMA
//               bulk stores (bulk reduce-add for fp32 partial sums), so that
//               outputs leave as whole lines and never contend with the
//               mainloop's operand loads (a block that straddles the expert's
//               last row is written with plain stores); the SwiGLU backward's
//               H blocks and a partial sum's blocks arrive by TMA loads one
//               chunk ahead.
// Tiles never straddle two experts.  The tile list is derived on the device
// from group_offsets (no host synchronisation); tiles are visited expert by
// expert in groups of 32 row tiles so that concurrently running CTAs share
// their A rows and B columns in L2.  Every wait is bounded: on time-out the
// CTA raises an abort flag, winds down, drains its in-flight copies and
// MMAs, frees TMEM and reports MOE_ERR_TIMEOUT through dev_status.
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"
#include "tc_sm103.cuh"

namespace moe {
namespace {

constexpr int BM = 128, BK = 64, UK = 16;
// output tile width (columns of the pair's 256 x BN tile): 256 for the bf16
// and current-scaling FP8 GEMMs, 192 for the block-scaled ones: their scale
// factors need tensor-memory columns beside the two accumulators (2 x 192 +
// 6 stages x 12), and a SwiGLU tile's gate and up halves stay whole 32-column
// chunks
constexpr int kBN = 256;
constexpr int kBNmx = 192;  // tile width of the block-scaled GEMMs
constexpr int kStages = 8;  // ring slots of the barrier book (5 or 6 in use, see Ring)
constexpr int kMaxEpiWarps = 4;
constexpr int kPadRows = kF8PadRows;  // group padding of column-wise copies (128 rows)
constexpr int kStgBytes = 8192;  // per epilogue warp: up to four 32x32 bf16 blocks (or two fp32)
// Internal epilogue: the SwiGLU forward that adds an fp32 partial sum (the last
// K-chunk of a chunked up-projection), its partial-sum blocks brought into the
// warp's staging by TMA loads one chunk ahead (16 KB of staging per warp, so 5
// stages)
constexpr int kEpiSwigluPs = 3;
constexpr bool is_swiglu_fwd(int epi) { return epi == MOE_EPI_SWIGLU_FWD || epi == kEpiSwigluPs; }
constexpr int A_BYTES = BM * BK * 2;   // 16 KB
constexpr int BOX_BYTES = 64 * 64 * 2; // one 64x64 MN-major box, 8 KB
constexpr int kMaxE = 256;
constexpr int kGroupPairs = 16;  // raster group: 16 row-tile pairs x all column tiles

constexpr int kTmemCols = 512;  // two accumulators of BN columns (+ block-scale factors)

// Operand elements: bf16 (K blocks of 64, MMA K = 16) or 8-bit float codes
// (K blocks of 128, MMA K = 32).  Either way a K block of one tile row is one
// 128-byte swizzle row, so stages, boxes and descriptors keep their byte sizes.
template <bool F8>
struct Elem {
  static constexpr int BKE = F8 ? 128 : 64;
  static constexpr int UKE = F8 ? 32 : 16;
};

enum { KIND_GMM = 0, KIND_TGMM = 1 };

struct Book {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint64_t aux_full[kMaxEpiWarps];  // SwiGLU backward: H blocks landed in a warp's staging
  uint32_t tmem_base;
  int abort_flag;
  int total_tiles;
  int cum[kMaxE + 1];            // per-expert tile prefix
  // weight gradients from column-wise copies: start of each expert's
  // zero-padded K range in units of kPadRows (the copies hold < 2^16 of them)
  uint16_t poff[kMaxE + 1];
};

// Per-kernel layout.  Every GEMM runs as 2-SM MMAs whose stage holds this
// CTA's 128-row (tgmm: 128-column) A tile and half of the B tile (BN = 256:
// 32 KB; block-scaled, BN = 192: 28 KB plus 1.5 KB of scale factors, padded
// to whole KB), 6 stages, and 4 epilogue warps (one per TMEM lane quarter).
template <int KIND, int EPI, bool F8, int BN, bool MX>
struct Ring {
  static constexpr int epi_warps = 4;
  static constexpr int stages = EPI == kEpiSwigluPs ? 5 : 6;
  static constexpr int stg_bytes = EPI == kEpiSwigluPs ? 2 * kStgBytes : kStgBytes;  // per warp
  static constexpr int b_bytes = BN * BK;  // this CTA's BN / 2 columns of B, 128-byte rows
  // block scaling: the scale factors of the stage's K block, A's 128 rows (one
  // 512-byte atom) and the tile's 192 columns (two atoms)
  static constexpr int sf_bytes = MX ? 1536 : 0;
  static constexpr int tx_bytes = A_BYTES + b_bytes + sf_bytes;  // copied per CTA and stage
  static constexpr int stage_bytes = (tx_bytes + 1023) / 1024 * 1024;
  static_assert(!MX || (F8 && BN == kBNmx), "block scaling: 8-bit operands, 192-column tiles");
  static_assert(stages <= kStages, "barrier book");
  static constexpr int threads = 64 + 32 * epi_warps;  // producer, MMA, epilogue
  static constexpr int stg_offset = stages * stage_bytes;  // 1024-aligned
  static constexpr int book_offset = stg_offset + epi_warps * stg_bytes;
  static constexpr int smem_bytes =
      1024 + book_offset + (int)((sizeof(Book) + 127) / 128 * 128);
  static_assert(stg_offset % 1024 == 0, "staging alignment");
  static_assert(smem_bytes <= 232448, "shared memory budget of one CTA");
};

struct TcParams {
  int E;
  int rows_cap;
  int K;        // contraction (gmm)
  int N;        // columns of the accumulated product (F for SWIGLU_BWD)
  int F;        // SwiGLU half width (SWIGLU_FWD: N / 2)
  int M;        // tgmm output rows
  int n_tiles;
  int m_tiles;  // tgmm: row tiles of the output
  const int32_t *offsets;
  void *C;
  int64_t ldc;
  int c_f32;
  uint16_t *C2;
  int64_t ldc2;
  uint16_t *Ct;   // column-wise copy of Act (SwiGLU forward) / dH (backward), or null
  int64_t ldct;
  const float *ps;
  int64_t ld_ps;
  const uint16_t *bias;   // expert e's vector at bias + e * stride_bias, or null
  int64_t stride_bias;
  const uint16_t *aux;
  int64_t ld_aux;
  int64_t stride_w;
  int accumulate;
  int32_t *dev_status;
  uint64_t wait_limit_ns;  // bound of every wait before the CTA gives up
  int stall_loads;         // test hook: the producer issues no loads
  // FP8: 1 / scale of A (one) and of B (one per expert), operand formats
  const float *a_sinv;
  const float *b_sinv;
  int a_fmt, b_fmt;
  float *amax_out;  // or null: max |value| of the bf16 output the epilogue writes
  // block scaling: where a tile's scale atoms sit for its K block kb
  //   A: atom (row tile) * sfa_stride + kb, the row tile being the expert's
  //      padded tile (gmm) or the output row tile (tgmm)
  //   B: atom rows 2 n_idx + e * sfb_erow (and the next), atom column
  //      e * sfb_ecol + kb (each 192-column tile owns two atom rows)
  int64_t sfa_stride;
  int sfb_ecol, sfb_erow;
};

struct TileInfo {
  int e, m_idx, n_idx, row0, row_end, kblocks;
  int k0;  // weight gradients from a column-wise copy of A: the expert's first column
  int pcol0;  // ragged-M GEMM: column of the tile's first row in a column-wise copy
};

// Group offsets read from global memory (through L1), clamped to [0, rows_cap].
MOE_DEVINL int group_offset(const TcParams &p, int e) {
  return min(max(__ldg(p.offsets + e), 0), p.rows_cap);
}

// Tiles are handed out in pairs: the two CTAs of a cluster take row tiles
// 2*pm and 2*pm + 1 of the same expert and column tile (the second one may lie
// past the expert's rows; it then runs through the pipeline and stores nothing).
template <int KIND, bool F8, bool AK>
MOE_DEVINL TileInfo decode_tile(const Book &bk, const TcParams &p, int t, int crank) {
  int lo = 0, hi = p.E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (bk.cum[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  TileInfo ti;
  ti.e = lo;
  const int local = t - bk.cum[lo];
  ti.row0 = group_offset(p, lo);
  ti.row_end = max(group_offset(p, lo + 1), ti.row0);
  const int size = ti.row_end - ti.row0;
  const int mt = KIND == KIND_GMM ? (size + BM - 1) / BM : p.m_tiles;
  const int mp = (mt + 1) / 2;                   // row-tile pairs
  const int group = kGroupPairs * p.n_tiles;
  const int g = local / group;
  const int within = local - g * group;
  const int gm = min(kGroupPairs, mp - g * kGroupPairs);
  ti.n_idx = within / gm;
  ti.m_idx = 2 * (g * kGroupPairs + (within - ti.n_idx * gm)) + crank;
  constexpr int BKE = Elem<F8>::BKE;
  if (KIND == KIND_GMM) {
    ti.row0 += ti.m_idx * BM;
    ti.kblocks = (p.K + BKE - 1) / BKE;
    ti.pcol0 = (int)bk.poff[lo] * kPadRows + ti.m_idx * BM;
  } else if (F8) {
    // FP8 weight gradients read the column-wise copies, where expert e's rows
    // fill whole K blocks from poff[e] on (zero padded to 128 rows)
    ti.row0 = (int)bk.poff[lo] * kPadRows;
    ti.row_end = (int)bk.poff[lo + 1] * kPadRows;
    ti.kblocks = (ti.row_end - ti.row0) / BKE;
    ti.k0 = ti.row0;
  } else {
    ti.kblocks = (size + BKE - 1) / BKE;
    ti.k0 = AK ? (int)bk.poff[lo] * kPadRows : 0;
  }
  return ti;
}

// --------------------------------------------------------------- epilogues
MOE_DEVINL void st_bf16x8(uint16_t *dst, const float *v) { st_v4(dst, f32_to_bf16x8(v)); }

MOE_DEVINL void st_f32x8(float *dst, const float *v) {
  st_v4(dst, make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]),
                        __float_as_uint(v[3])));
  st_v4(dst + 4, make_uint4(__float_as_uint(v[4]), __float_as_uint(v[5]), __float_as_uint(v[6]),
                            __float_as_uint(v[7])));
}

MOE_DEVINL uint4 ld_v4_no_l1(const void *ptr) {
  uint4 r;
  asm volatile("ld.global.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(ptr));
  return r;
}

MOE_DEVINL void prefetch_l2(const void *ptr) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(ptr));
}

// Staging of one thread's 32-value row segment in the layout the TMA store
// reads: bf16 rows of 64 bytes under the 64-byte swizzle (16-byte chunk c of
// row r at chunk c ^ ((r >> 1) & 3)), fp32 rows of 128 bytes under the
// 128-byte swizzle (chunk c ^ (r & 7)).  Both are free of bank conflicts
// when the 32 lanes of a warp write the same chunk of their 32 rows.
MOE_DEVINL void stage_bf16(uint8_t *buf, int r, const float *v) {
#pragma unroll
  for (int c = 0; c < 4; ++c)
    *reinterpret_cast<uint4 *>(buf + r * 64 + ((c ^ ((r >> 1) & 3)) << 4)) =
        f32_to_bf16x8(v + 8 * c);
}

// 64 bf16 values of row r as one 128-byte row under the 128-byte swizzle (the
// layout of stage_f32, 8 values per 16-byte chunk).
MOE_DEVINL void stage_bf16_64(uint8_t *buf, int r, const float *v) {
#pragma unroll
  for (int c = 0; c < 8; ++c)
    *reinterpret_cast<uint4 *>(buf + r * 128 + ((c ^ (r & 7)) << 4)) = f32_to_bf16x8(v + 8 * c);
}

MOE_DEVINL void stage_f32(uint8_t *buf, int r, const float *v) {
#pragma unroll
  for (int c = 0; c < 8; ++c)
    *reinterpret_cast<uint4 *>(buf + r * 128 + ((c ^ (r & 7)) << 4)) =
        make_uint4(__float_as_uint(v[4 * c]), __float_as_uint(v[4 * c + 1]),
                   __float_as_uint(v[4 * c + 2]), __float_as_uint(v[4 * c + 3]));
}

// The transposed layout of stage_bf16: thread r's 32 values become column r
// of the 32 x 32 block (block row n = value n), rows of 64 bytes under the
// 64-byte swizzle.  Lanes r and r^1 trade one value per row pair so that each
// writes 32-bit words (the even lane rows 2m, the odd lane rows 2m+1): every
// store instruction fills two whole 64-byte rows, free of bank conflicts.
MOE_DEVINL void stage_bf16_t(uint8_t *buf, int r, const float *v) {
  const bool odd = r & 1;
  const int off = ((r >> 1) & 3) * 4;  // byte of the word within its 16-byte chunk
  const int chunk = r >> 3;
#pragma unroll
  for (int m = 0; m < 16; ++m) {
    const float recv = __shfl_xor_sync(0xffffffffu, odd ? v[2 * m] : v[2 * m + 1], 1);
    const int n = 2 * m + (odd ? 1 : 0);
    const __nv_bfloat162 w = odd ? __floats2bfloat162_rn(recv, v[2 * m + 1])
                                 : __floats2bfloat162_rn(v[2 * m], recv);
    *reinterpret_cast<__nv_bfloat162 *>(buf + n * 64 + ((chunk ^ ((n >> 1) & 3)) << 4) + off) = w;
  }
}

// The same transposed block written straight to global memory: column-wise
// copy rows [nc, nc + 32) (those below nmax) at columns [pc0, pc0 + 32); each
// store instruction writes two contiguous 64-byte row segments.
MOE_DEVINL void store_bf16_t(uint16_t *Ct, int64_t ldct, int64_t pc0, int nc, int nmax, int r,
                             const float *v) {
  const bool odd = r & 1;
  uint16_t *base = Ct + pc0 + (r & ~1);
#pragma unroll
  for (int m = 0; m < 16; ++m) {
    const float recv = __shfl_xor_sync(0xffffffffu, odd ? v[2 * m] : v[2 * m + 1], 1);
    const int n = 2 * m + (odd ? 1 : 0);
    const __nv_bfloat162 w = odd ? __floats2bfloat162_rn(recv, v[2 * m + 1])
                                 : __floats2bfloat162_rn(v[2 * m], recv);
    if (nc + n < nmax) *reinterpret_cast<__nv_bfloat162 *>(base + (int64_t)(nc + n) * ldct) = w;
  }
}

// The warp's staging buffers may be rewritten once the previous bulk stores
// have read them.
MOE_DEVINL void stage_acquire(int lane) {
  if (lane == 0) tc::bulk_wait_read0();
  __syncwarp();
}

// Staged writes become visible to the TMA engine; lane 0 then issues the stores.
MOE_DEVINL void stage_release() {
  tc::fence_proxy_async_smem();
  __syncwarp();
}

// Output maps of an epilogue warp (m0..m2), the H maps it loads from in the
// SwiGLU backward (m2 = gate, m3 = up), its aux barrier and that barrier's
// phase count, and the evict-first L2 policy of the tensors it streams (H
// written by the SwiGLU forward; H read and dH written by the backward).
struct OutMaps {
  const CUtensorMap *m0, *m1, *m2, *m3;
  uint64_t *aux_bar;
  uint32_t aux_phase;   // H loads waited for
  uint32_t aux_issued;  // H loads issued
  uint64_t stream_pol;
};

// Before a tile's accumulator is ready: pull the epilogue's global inputs
// (SwiGLU-backward H, partial sums) into L2 so that the epilogue's loads do
// not wait on HBM one after another.  Thread = one output row.
template <int KIND, int EPI, int BN>
MOE_DEVINL void epilogue_prefetch(const TcParams &p, const TileInfo &ti, int rit, int c_begin,
                                  int c_end) {
  if (KIND == KIND_GMM) {
    const int64_t row = (int64_t)ti.row0 + rit;
    if (row >= ti.row_end) return;
    if (EPI == MOE_EPI_SWIGLU_BWD) {
      const uint16_t *h = p.aux + row * p.ld_aux;
      const int n0 = ti.n_idx * BN + c_begin * 32;
      for (int n = n0; n < min(ti.n_idx * BN + c_end * 32, p.N); n += 64) {
        prefetch_l2(h + n);
        prefetch_l2(h + p.N + n);
      }
    } else if (p.ps != nullptr) {
      const float *q = p.ps + row * p.ld_ps;
      if (is_swiglu_fwd(EPI)) {
        const int n0 = ti.n_idx * (BN / 2);
        for (int n = n0; n < min(n0 + BN / 2, p.F); n += 32) {
          prefetch_l2(q + n);
          prefetch_l2(q + p.F + n);
        }
      } else {
        const int n0 = ti.n_idx * BN;
        for (int n = n0; n < min(n0 + BN, p.N); n += 32) prefetch_l2(q + n);
      }
    }
  } else if (p.accumulate) {
    const int m = ti.m_idx * BM + rit;
    if (m >= p.M) return;
    const float *w = static_cast<const float *>(p.C) + (int64_t)ti.e * p.stride_w +
                     (int64_t)m * p.ldc;
    const int n0 = ti.n_idx * BN;
    for (int n = n0; n < min(n0 + BN, p.N); n += 32) prefetch_l2(w + n);
  }
}

// amx = max(amx, |v[0]|, ..., |v[n - 1]|) over a 32-value chunk, by a tree
// of pairwise maxima (max is exact, so the order does not matter); the
// bounds check only on a ragged last chunk.
MOE_DEVINL float chunk_amax(float amx, const float *v, int n) {
  float m[16];
  if (n >= 32) {
#pragma unroll
    for (int i = 0; i < 16; ++i) m[i] = fmaxf(fabsf(v[2 * i]), fabsf(v[2 * i + 1]));
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i)
      m[i] = fmaxf(2 * i < n ? fabsf(v[2 * i]) : 0.0f, 2 * i + 1 < n ? fabsf(v[2 * i + 1]) : 0.0f);
  }
#pragma unroll
  for (int w = 8; w > 0; w >>= 1)
#pragma unroll
    for (int i = 0; i < w; ++i) m[i] = fmaxf(m[i], m[i + w]);
  return fmaxf(amx, m[0]);
}

// One tile's epilogue for the ragged-M GEMM.  Warp q owns tile rows
// [32q, 32q+32), thread = one row; 32-column chunks.  The global inputs of a
// chunk are loaded one chunk ahead so that their latency overlaps the work
// of the previous chunk.
// SwiGLU backward: TMA loads of the warp's 32x32 gate and up blocks of H for
// the chunk starting at column nc into its staging area (lane 0 issues).
MOE_DEVINL void issue_aux_load(OutMaps &om, uint8_t *stg, int nc, int wrow0) {
  ++om.aux_issued;
  tc::mbar_expect_tx(om.aux_bar, 4096);
  tc::tma_load_2d_hint(stg + 4096, om.m2, om.aux_bar, nc, wrow0, om.stream_pol);
  tc::tma_load_2d_hint(stg + 6144, om.m3, om.aux_bar, nc, wrow0, om.stream_pol);
}

// SwiGLU forward with a partial sum: TMA loads of the warp's 32 x 32 fp32
// blocks of P (gate columns nc.., up columns F + nc..) into the second half of
// its staging (lane 0 issues; m3 is the map of P).
MOE_DEVINL void issue_ps_load(OutMaps &om, uint8_t *stg, int nc, int F, int wrow0) {
  ++om.aux_issued;
  tc::mbar_expect_tx(om.aux_bar, 8192);
  tc::tma_load_2d_hint(stg + kStgBytes, om.m3, om.aux_bar, nc, wrow0, om.stream_pol);
  tc::tma_load_2d_hint(stg + kStgBytes + 4096, om.m3, om.aux_bar, F + nc, wrow0, om.stream_pol);
}

// Row r's 32 fp32 values of a 32 x 32 block staged under the 128-byte swizzle
// (the inverse of stage_f32).
MOE_DEVINL void unstage_f32(const uint8_t *buf, int r, float *v) {
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 w = *reinterpret_cast<const uint4 *>(buf + r * 128 + ((c ^ (r & 7)) << 4));
    v[4 * c] = __uint_as_float(w.x);
    v[4 * c + 1] = __uint_as_float(w.y);
    v[4 * c + 2] = __uint_as_float(w.z);
    v[4 * c + 3] = __uint_as_float(w.w);
  }
}

// One tile's epilogue for the ragged-M GEMM.  Warp q owns tile rows
// [32q, 32q+32), thread = one row; 32-column chunks.
// Chunks [c_begin, c_end) of the tile's 32-column chunks are this warp's.
// amx: the warp thread's running max |value| over the outputs it wrote
// (Act for the SwiGLU forward, dH for the SwiGLU backward), when amax_out.
template <int EPI, bool F8, int BN, bool MX, bool CT>
MOE_DEVINL void epilogue_gmm(const TcParams &p, const TileInfo &ti, uint32_t taddr, int q,
                             int lane, uint8_t *stg, OutMaps &om, volatile int *abort_flag,
                             int c_begin, int c_end, float &amx) {
  // FP8 with current scaling: the accumulator holds code products; dequantize
  // with both scales (block-scaled MMAs apply their scales themselves)
  constexpr bool kDeq = F8 && !MX;
  const float sc = kDeq ? __ldg(p.a_sinv) * __ldg(p.b_sinv + ti.e) : 1.0f;
  const int wrow0 = ti.row0 + q * 32;
  const int64_t row = (int64_t)wrow0 + lane;
  const bool valid = row < ti.row_end;
  const bool bulk = wrow0 + 32 <= ti.row_end;  // every row of the block is this expert's
  // FP8 GEMMs track their output amax and take no partial sum or bias; bf16
  // ones the reverse (compile-time, so neither pays the other's registers)
  const bool track = F8 && p.amax_out != nullptr && valid;
  // column-wise copy of the activation output: every 32-row block of a tile
  // that starts inside the expert, rows past the expert as zeros (they are the
  // expert's padding in the copy); a tile past the expert writes nothing
  const bool colwise = CT && ti.row0 < ti.row_end;
  const int64_t pc0 = (int64_t)ti.pcol0 + q * 32;
  if (is_swiglu_fwd(EPI)) {
    // kPsTma: the partial sum arrives by TMA in the staging (first chunk's
    // load issued at the tile's start); the column-wise-copy instance, whose
    // fourth map is the copy's, loads it into registers one chunk ahead (the
    // plain instance never gets one: the host sends partial sums to kPsTma)
    constexpr bool kPsTma = EPI == kEpiSwigluPs;
    const int F = p.F;
    const int n0 = ti.n_idx * (BN / 2);
    const bool has_ps = CT && !F8 && valid && p.ps != nullptr;
    auto load_ps = [&](int c, uint4 *g4, uint4 *u4) {
      const int nc = n0 + c * 32;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (nc + j * 4 < F) {
          g4[j] = ld_v4_no_l1(p.ps + row * p.ld_ps + nc + j * 4);
          u4[j] = ld_v4_no_l1(p.ps + row * p.ld_ps + F + nc + j * 4);
        }
      }
    };
    uint4 pg[8], pu[8], ng[8], nu[8];
    if (has_ps) load_ps(c_begin, pg, pu);
#pragma unroll 1
    for (int c = c_begin; c < min(c_end, BN / 2 / 32); ++c) {
      const int nc = n0 + c * 32;
      if (nc >= F) break;
      if (has_ps && c + 1 < min(c_end, BN / 2 / 32) && nc + 32 < F) load_ps(c + 1, ng, nu);
      float pgv[32], puv[32];
      if (kPsTma) {
        // this chunk's P blocks -> registers, then the next chunk's loads
        if (!tc::mbar_wait_warp(om.aux_bar, om.aux_phase & 1, abort_flag, p.wait_limit_ns))
          return;
        ++om.aux_phase;
        unstage_f32(stg + kStgBytes, lane, pgv);
        unstage_f32(stg + kStgBytes + 4096, lane, puv);
        __syncwarp();
        if (lane == 0 && c + 1 < min(c_end, BN / 2 / 32) && nc + 32 < F) {
          tc::fence_proxy_async_smem();
          issue_ps_load(om, stg, nc + 32, F, wrow0);
        }
      }
      float g[32], u[32], act[32];
      {  // both halves in flight, one wait
        uint32_t rg[32], ru[32];
        tc::tmem_ld32_issue(taddr + c * 32, rg);
        tc::tmem_ld32_issue(taddr + BN / 2 + c * 32, ru);
        tc::tmem_wait_ld(rg);
        tc::reg_after(ru);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          g[j] = __uint_as_float(rg[j]);
          u[j] = __uint_as_float(ru[j]);
        }
      }
      if (kDeq) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          g[j] *= sc;
          u[j] *= sc;
        }
      }
      if (kPsTma) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          g[j] += pgv[j];
          u[j] += puv[j];
        }
      }
      if (has_ps) {
        const float *fg = reinterpret_cast<const float *>(pg);
        const float *fu = reinterpret_cast<const float *>(pu);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          g[j] += fg[j];
          u[j] += fu[j];
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          pg[j] = ng[j];
          pu[j] = nu[j];
        }
      }
      if (!F8 && p.bias != nullptr) {
        const uint16_t *be = p.bias + (int64_t)ti.e * p.stride_bias;
#pragma unroll
        for (int j8 = 0; j8 < 4; ++j8) {
          if (nc + j8 * 8 < F) {
            float bg[8], bu[8];
            bf16x8_to_f32(__ldg(reinterpret_cast<const uint4 *>(be + nc + j8 * 8)), bg);
            bf16x8_to_f32(__ldg(reinterpret_cast<const uint4 *>(be + F + nc + j8 * 8)), bu);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              g[j8 * 8 + i] += bg[i];
              u[j8 * 8 + i] += bu[i];
            }
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 32; ++j) act[j] = g[j] * sigmoid_f(g[j]) * u[j];
      if (track) amx = chunk_amax(amx, act, F - nc);
      if (!CT) {  // (kept apart: the shared form below costs this instance registers)
        if (bulk) {
          stage_acquire(lane);
          stage_bf16(stg, lane, g);
          stage_bf16(stg + 2048, lane, u);
          stage_bf16(stg + 4096, lane, act);
          stage_release();
          if (lane == 0) {
            tc::tma_store_2d_hint(om.m0, stg, nc, wrow0, om.stream_pol);
            tc::tma_store_2d_hint(om.m1, stg + 2048, nc, wrow0, om.stream_pol);
            tc::tma_store_2d(om.m2, stg + 4096, nc, wrow0);
            tc::bulk_commit();
          }
        } else if (valid) {
          uint16_t *H = static_cast<uint16_t *>(p.C) + row * p.ldc;
          uint16_t *A = p.C2 + row * p.ldc2;
#pragma unroll
          for (int j8 = 0; j8 < 4; ++j8) {
            const int n = nc + j8 * 8;
            if (n >= F) break;
            st_bf16x8(H + n, g + j8 * 8);
            st_bf16x8(H + F + n, u + j8 * 8);
            st_bf16x8(A + n, act + j8 * 8);
          }
        }
        continue;
      }
      if (bulk || colwise) {
        stage_acquire(lane);
        if (bulk) {
          stage_bf16(stg, lane, g);
          stage_bf16(stg + 2048, lane, u);
          stage_bf16(stg + 4096, lane, act);
        }
        if (colwise) {
          if (!valid) {
#pragma unroll
            for (int j = 0; j < 32; ++j) act[j] = 0.0f;
          }
          stage_bf16_t(stg + 6144, lane, act);
        }
        stage_release();
        if (lane == 0) {
          if (bulk) {
            tc::tma_store_2d_hint(om.m0, stg, nc, wrow0, om.stream_pol);
            tc::tma_store_2d_hint(om.m1, stg + 2048, nc, wrow0, om.stream_pol);
            tc::tma_store_2d(om.m2, stg + 4096, nc, wrow0);
          }
          if (colwise) tc::tma_store_2d(om.m3, stg + 6144, (int)pc0, nc);
          tc::bulk_commit();
        }
      }
      if (!bulk && valid) {
        uint16_t *H = static_cast<uint16_t *>(p.C) + row * p.ldc;
        uint16_t *A = p.C2 + row * p.ldc2;
#pragma unroll
        for (int j8 = 0; j8 < 4; ++j8) {
          const int n = nc + j8 * 8;
          if (n >= F) break;
          st_bf16x8(H + n, g + j8 * 8);
          st_bf16x8(H + F + n, u + j8 * 8);
          st_bf16x8(A + n, act + j8 * 8);
        }
      }
    }
  } else if (EPI == MOE_EPI_SWIGLU_BWD) {
    const int N = p.N;
    const int n0 = ti.n_idx * BN;
    const uint8_t *aux_g = stg + 4096;
    const uint8_t *aux_u = stg + 6144;
#pragma unroll 1
    for (int c = c_begin; c < c_end; ++c) {
      const int nc = n0 + c * 32;
      if (nc >= N) break;
      // this chunk's H blocks (issued one chunk ahead) -> registers, while
      // its TMEM load is in flight
      if (!tc::mbar_wait_warp(om.aux_bar, om.aux_phase & 1, abort_flag, p.wait_limit_ns)) return;
      ++om.aux_phase;
      uint32_t rv[32];
      tc::tmem_ld32_issue(taddr + c * 32, rv);
      float g[32], u[32];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const int off = lane * 64 + ((cc ^ ((lane >> 1) & 3)) << 4);
        bf16x8_to_f32(*reinterpret_cast<const uint4 *>(aux_g + off), g + 8 * cc);
        bf16x8_to_f32(*reinterpret_cast<const uint4 *>(aux_u + off), u + 8 * cc);
      }
      __syncwarp();
      if (lane == 0 && c + 1 < c_end && nc + 32 < N) {
        tc::fence_proxy_async_smem();
        issue_aux_load(om, stg, nc + 32, wrow0);
      }
      tc::tmem_wait_ld(rv);
      float v[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(rv[j]);
      if (kDeq) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] *= sc;
      }
      float dg[32], du[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const float sg = sigmoid_f(g[k]);
        const float vs = v[k] * sg;
        du[k] = vs * g[k];
        dg[k] = vs * u[k] * (1.0f + g[k] * (1.0f - sg));
      }
      if (track) {
        amx = chunk_amax(amx, dg, N - nc);
        amx = chunk_amax(amx, du, N - nc);
      }
      if (colwise) {
        if (!valid) {
#pragma unroll
          for (int j = 0; j < 32; ++j) dg[j] = du[j] = 0.0f;
        }
        store_bf16_t(p.Ct, p.ldct, pc0, nc, N, lane, dg);
        store_bf16_t(p.Ct + (int64_t)N * p.ldct, p.ldct, pc0, nc, N, lane, du);
      }
      if (bulk) {
        stage_acquire(lane);
        stage_bf16(stg, lane, dg);
        stage_bf16(stg + 2048, lane, du);
        stage_release();
        if (lane == 0) {
          tc::tma_store_2d_hint(om.m0, stg, nc, wrow0, om.stream_pol);
          tc::tma_store_2d_hint(om.m1, stg + 2048, nc, wrow0, om.stream_pol);
          tc::bulk_commit();
        }
      } else if (valid) {
        uint16_t *dH = static_cast<uint16_t *>(p.C) + row * p.ldc;
#pragma unroll
        for (int j8 = 0; j8 < 4; ++j8) {
          const int n = nc + j8 * 8;
          if (n >= N) break;
          st_bf16x8(dH + n, dg + j8 * 8);
          st_bf16x8(dH + N + n, du + j8 * 8);
        }
      }
    }
  } else {  // MOE_EPI_NONE
    const int N = p.N;
    const int n0 = ti.n_idx * BN;
    // in place (C is the fp32 partial sum): the TMA engine adds the block in L2
    const bool in_place = p.ps != nullptr && static_cast<const void *>(p.ps) == p.C;
    const bool has_in = !F8 && valid && p.ps != nullptr && !(in_place && bulk);
    auto load_chunk = [&](int c, uint4 *buf) {
      const int nc = n0 + c * 32;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int n = nc + j * 4;
        if (n < N) buf[j] = ld_v4_no_l1(p.ps + row * p.ld_ps + n);
      }
    };
    uint4 cur[8], nxt[8];
    if (has_in) load_chunk(c_begin, cur);
#pragma unroll 1
    for (int c = c_begin; c < c_end; ++c) {
      const int nc = n0 + c * 32;
      if (nc >= N) break;
      if (has_in && c + 1 < c_end && nc + 32 < N) load_chunk(c + 1, nxt);
      float v[32];
      tc::tmem_ld32(taddr + c * 32, v);
      if (kDeq) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] *= sc;
      }
      if (has_in) {
        const float *pv = reinterpret_cast<const float *>(cur);
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] += pv[j];
#pragma unroll
        for (int j = 0; j < 8; ++j) cur[j] = nxt[j];
      }
      if (!F8 && p.bias != nullptr) {
        const uint16_t *be = p.bias + (int64_t)ti.e * p.stride_bias;
#pragma unroll
        for (int j8 = 0; j8 < 4; ++j8) {
          if (nc + j8 * 8 < N) {
            float bv[8];
            bf16x8_to_f32(__ldg(reinterpret_cast<const uint4 *>(be + nc + j8 * 8)), bv);
#pragma unroll
            for (int i = 0; i < 8; ++i) v[j8 * 8 + i] += bv[i];
          }
        }
      }
      if (track) amx = chunk_amax(amx, v, N - nc);
      if (bulk) {
        stage_acquire(lane);
        if (p.c_f32) stage_f32(stg, lane, v);
        else stage_bf16(stg, lane, v);
        stage_release();
        if (lane == 0) {
          if (in_place) tc::tma_reduce_add_2d(om.m0, stg, nc, wrow0);
          else tc::tma_store_2d(om.m0, stg, nc, wrow0);
          tc::bulk_commit();
        }
      } else if (valid) {
#pragma unroll
        for (int j8 = 0; j8 < 4; ++j8) {
          const int n = nc + j8 * 8;
          if (n >= N) break;
          if (p.c_f32) st_f32x8(static_cast<float *>(p.C) + row * p.ldc + n, v + j8 * 8);
          else st_bf16x8(static_cast<uint16_t *>(p.C) + row * p.ldc + n, v + j8 * 8);
        }
      }
    }
  }
}

// tgmm epilogue: warp q owns output rows m in [m_idx*128 + 32q, +32) of W_e.
// `zero`: the expert had no rows, so TMEM is not read.  Bulk stores, or bulk
// fp32 reduce-adds into W when accumulating; the box is clipped at M and N.
// A bf16 W leaves in 32 x 64 boxes (128-byte rows, two TMEM loads in flight
// per box): with few rows per expert this epilogue sets the pace, and half as
// many boxes per tile means half the staging waits, fences and store issues.
// The warp's 8 KB of staging holds two such boxes, used in turn (`slot`
// counts the warp's boxes across tiles), so that the previous box's store may
// still be reading shared memory while the next one is staged.
template <bool F8, int BN, bool MX>
MOE_DEVINL void epilogue_tgmm(const TcParams &p, const TileInfo &ti, uint32_t taddr, int q,
                              int lane, uint8_t *stg, const OutMaps &om, bool zero,
                              uint32_t &slot) {
  constexpr bool kDeq = F8 && !MX;
  const float sc = kDeq && !zero ? __ldg(p.a_sinv) * __ldg(p.b_sinv) : 1.0f;
  const int wm0 = ti.m_idx * BM + q * 32;
  const int n0 = ti.n_idx * BN;
  if (!p.c_f32) {
#pragma unroll 1
    for (int c = 0; c < BN / 64; ++c) {
      const int nc = n0 + c * 64;
      if (nc >= p.N) break;
      float v[64];
      if (zero) {
#pragma unroll
        for (int j = 0; j < 64; ++j) v[j] = 0.f;
      } else {
        uint32_t r0[32], r1[32];
        tc::tmem_ld32_issue(taddr + c * 64, r0);
        tc::tmem_ld32_issue(taddr + c * 64 + 32, r1);
        tc::tmem_wait_ld(r0);
        tc::reg_after(r1);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          v[j] = __uint_as_float(r0[j]) * sc;
          v[32 + j] = __uint_as_float(r1[j]) * sc;
        }
      }
      uint8_t *buf = stg + (slot & 1) * 4096;
      if (lane == 0) tc::bulk_wait_read<1>();
      __syncwarp();
      stage_bf16_64(buf, lane, v);
      stage_release();
      if (lane == 0) {
        tc::tma_store_3d(om.m0, buf, nc, wm0, ti.e);
        tc::bulk_commit();
      }
      ++slot;
    }
    return;
  }
#pragma unroll 1
  for (int c = 0; c < BN / 32; ++c) {
    const int nc = n0 + c * 32;
    if (nc >= p.N) break;
    float v[32];
    if (zero) {
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = 0.f;
    } else {
      tc::tmem_ld32(taddr + c * 32, v);
      if (kDeq) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] *= sc;
      }
    }
    stage_acquire(lane);
    if (p.c_f32) stage_f32(stg, lane, v);
    else stage_bf16(stg, lane, v);
    stage_release();
    if (lane == 0) {
      if (p.accumulate) tc::tma_reduce_add_3d(om.m0, stg, nc, wm0, ti.e);
      else tc::tma_store_3d(om.m0, stg, nc, wm0, ti.e);
      tc::bulk_commit();
    }
  }
}

// ------------------------------------------------------------------ kernel
template <int KIND, bool B_MN, int EPI, bool F8, bool AK, int BN, bool MX, bool CT>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(Ring<KIND, EPI, F8, BN, MX>::threads, 1)
gmm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              const __grid_constant__ CUtensorMap tmC0, const __grid_constant__ CUtensorMap tmC1,
              const __grid_constant__ CUtensorMap tmC2, const __grid_constant__ CUtensorMap tmC3,
              const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
              const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Book &bk = *reinterpret_cast<Book *>(smem + Ring<KIND, EPI, F8, BN, MX>::book_offset);
  volatile int *abort_flag = &bk.abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int crank = (int)tc::cluster_ctarank();
  const int cid = (int)tc::cluster_id_x();
  const int ncl = (int)tc::nclusters_x();
  constexpr uint16_t kPair = 0x3;
  constexpr int kSt = Ring<KIND, EPI, F8, BN, MX>::stages;
  constexpr int kStageB = Ring<KIND, EPI, F8, BN, MX>::stage_bytes;
  constexpr int BKE = Elem<F8>::BKE;
  constexpr int kEW = Ring<KIND, EPI, F8, BN, MX>::epi_warps;
  constexpr int kSfOff = A_BYTES + Ring<KIND, EPI, F8, BN, MX>::b_bytes;  // scale factors in a stage
  // bf16 weight gradients read A as stored (MN-major) unless AK: then from a
  // zero-padded column-wise copy (K-major), like FP8 always does
  constexpr bool A_MN = KIND == KIND_TGMM && !AK;
  const bool leader = crank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kSt; ++s) {
      tc::mbar_init(&bk.full[s], 1);
      // 2-SM: the leader's MMA commit releases a stage in both CTAs once;
      // else both CTAs' MMA warps release it
      tc::mbar_init(&bk.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(&bk.tfull[a], 1);
      // 2-SM: the leader's accumulator is free once both CTAs' epilogues are done
      tc::mbar_init(&bk.tempty[a], 2 * kEW);
    }
    tc::mbar_init(&bk.drain, 1);
    for (int w = 0; w < kEW; ++w) tc::mbar_init(&bk.aux_full[w], 1);
    bk.abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch(&tmA);
    tc::tma_prefetch(&tmB);
    tc::tma_prefetch(&tmC0);
  }
  __syncthreads();
  if (warp == 0) {
    // per-expert tile counts and their exclusive scan (warp shuffles); FP8
    // weight gradients also scan the sizes rounded up to whole K blocks
    int carry = 0, pcarry = 0;
    for (int c0 = 0; c0 < p.E; c0 += 32) {
      const int e = c0 + lane;
      int tiles = 0, padded = 0;
      if (e < p.E) {
        const int size = max(group_offset(p, e + 1) - group_offset(p, e), 0);
        const int mt = KIND == KIND_GMM ? (size + BM - 1) / BM : p.m_tiles;
        tiles = (mt + 1) / 2 * p.n_tiles;
        padded = (size + kPadRows - 1) / kPadRows;
      }
      int incl = tiles, pincl = padded;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        const int py = __shfl_up_sync(0xffffffffu, pincl, o);
        if (lane >= o) {
          incl += y;
          pincl += py;
        }
      }
      if (e < p.E) {
        bk.cum[e] = carry + incl - tiles;
        bk.poff[e] = (uint16_t)(pcarry + pincl - padded);
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
      pcarry += __shfl_sync(0xffffffffu, pincl, 31);
    }
    if (lane == 0) {
      bk.cum[p.E] = carry;
      bk.poff[p.E] = (uint16_t)pcarry;
      bk.total_tiles = carry;
    }
    // offsets must be non-decreasing; clamp a bad table to empty groups
    for (int e = lane; e < p.E; e += 32)
      if (group_offset(p, e + 1) < group_offset(p, e)) moe_set_status(p.dev_status, MOE_ERR_DEVICE);
  }
  if (warp == 1) {
    tc::tmem_alloc_2sm(&bk.tmem_base, kTmemCols);
    tc::tmem_relinquish_2sm();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::cluster_sync();  // both CTAs' barriers exist before any multicast lands
  tc::tc_fence_after();
  const uint32_t tmem = bk.tmem_base;
  const int total = bk.total_tiles;

  uint32_t issued = 0;  // producer: k-blocks issued (ring position)
  if (warp == 0) {
    if (lane == 0 && !p.stall_loads) {
      int s = 0;         // ring slot of the next K block
      uint32_t ph = 0;   // its pass over the ring (parity)
      for (int t = cid; t < total; t += ncl) {
        const TileInfo ti = decode_tile<KIND, F8, AK>(bk, p, t, crank);
        bool ok = true;
        for (int kb = 0; kb < ti.kblocks; ++kb) {
          if (!tc::mbar_wait(&bk.empty[s], ph ^ 1, abort_flag, p.wait_limit_ns)) {
            ok = false;
            break;
          }
          uint8_t *sa = smem + s * kStageB;
          uint8_t *sb = sa + A_BYTES;
          uint64_t *fb = &bk.full[s];
          // both CTAs' copies complete on the leader's full barrier, which
          // expects the whole pair's stage
          const uint32_t fbl = tc::mapa_shared(tc::smem_u32(fb), 0);
          if (leader) tc::mbar_expect_tx(fb, 2 * Ring<KIND, EPI, F8, BN, MX>::tx_bytes);
          if (KIND == KIND_TGMM && (F8 || (AK && !B_MN))) {
            // K-major column-wise copies: this CTA's 128 rows of A^T (output
            // rows) and of B^T (its half of the 256 output columns)
            const int k = ti.k0 + kb * BKE;
            tc::tma_load_2d_2sm(sa, &tmA, fbl, k, ti.m_idx * BM);
            tc::tma_load_2d_2sm(sb, &tmB, fbl, k, ti.n_idx * BN + crank * (BN / 2));
          } else if (KIND == KIND_TGMM && AK) {
            // K-major A from the column-wise copy (zero padded past the
            // expert's rows); MN-major B rows as stored (tail zeroed below)
            const int r = ti.row0 + kb * BKE;
            const int nb = ti.n_idx * BN + crank * (BN / 2);
            tc::tma_load_2d_2sm(sa, &tmA, fbl, ti.k0 + kb * BKE, ti.m_idx * BM);
            tc::tma_load_2d_2sm(sb, &tmB, fbl, nb, r);
            tc::tma_load_2d_2sm(sb + BOX_BYTES, &tmB, fbl, nb + 64, r);
          } else if (KIND == KIND_TGMM) {
            // this CTA's 128 output rows of A (two 64-column boxes) and its
            // 128 columns of B, both over the K block's 64 rows
            const int r = ti.row0 + kb * BK;
            const int m0 = ti.m_idx * BM;
            const int nb = ti.n_idx * BN + crank * (BN / 2);
            tc::tma_load_2d_2sm(sa, &tmA, fbl, m0, r);
            tc::tma_load_2d_2sm(sa + BOX_BYTES, &tmA, fbl, m0 + 64, r);
            tc::tma_load_2d_2sm(sb, &tmB, fbl, nb, r);
            tc::tma_load_2d_2sm(sb + BOX_BYTES, &tmB, fbl, nb + 64, r);
          } else {
            tc::tma_load_2d_2sm(sa, &tmA, fbl, kb * BKE, ti.row0);
            if (B_MN) {
              // this CTA's 128 columns of B: two 64-column boxes
              const int n0 = is_swiglu_fwd(EPI) ? ti.n_idx * (BN / 2) : ti.n_idx * BN;
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                const int i = 2 * crank + j;
                const int x = is_swiglu_fwd(EPI)
                                  ? (i < 2 ? n0 + 64 * i : p.F + n0 + 64 * (i - 2))
                                  : n0 + 64 * i;
                tc::tma_load_3d_2sm(sb + j * BOX_BYTES, &tmB, fbl, x, kb * BKE, ti.e);
              }
            } else {
              // K-major B: this CTA's 128 of the tile's 256 columns (SwiGLU
              // forward: gate columns in the first CTA, up columns in the second)
              const int nrow = is_swiglu_fwd(EPI)
                                   ? (crank == 0 ? 0 : p.F) + ti.n_idx * (BN / 2)
                                   : ti.n_idx * BN + crank * (BN / 2);
              tc::tma_load_3d_2sm(sb, &tmB, fbl, kb * BKE, nrow, ti.e);
            }
          }
          if (MX) {
            // the K block's scale-factor atoms: this CTA's 128 A rows, and the
            // tile's 128 B columns (both CTAs load the same B atom)
            int64_t ia;
            int bc, br;  // B's atom column and first atom row
            if (KIND == KIND_GMM) {
              ia = ((int64_t)bk.poff[ti.e] + ti.m_idx) * p.sfa_stride + kb;
              bc = ti.e * p.sfb_ecol + kb;
              br = 2 * ti.n_idx + ti.e * p.sfb_erow;
            } else {
              const int kb0 = ti.k0 / BKE + kb;
              ia = (int64_t)ti.m_idx * p.sfa_stride + kb0;
              bc = kb0;
              br = 2 * ti.n_idx;
            }
            tc::tma_load_2d_2sm(sa + kSfOff, &tmSA, fbl, 0, (int)ia);
            tc::tma_load_3d_2sm(sa + kSfOff + 512, &tmSB, fbl, 0, bc, br);
          }
          ++issued;
          if (++s == kSt) {
            s = 0;
            ph ^= 1;
          }
        }
        if (!ok) break;
      }
      // drain: every issued copy has landed before the CTA may exit
      // (2-SM: a CTA's copies complete on the leader's barrier; the leader's
      // MMA consumed them all before the pair's final cluster barrier)
      if (leader)
        for (uint32_t i = issued > (uint32_t)kSt ? issued - kSt : 0; i < issued; ++i)
          tc::mbar_wait_drain(&bk.full[i % kSt], (i / kSt) & 1, p.wait_limit_ns / 4);
    }
  } else if (warp == 1 && leader) {
    const uint32_t IDESC = F8 ? tc::idesc_f8(2 * BM, BN, p.a_fmt, p.b_fmt)
                              : tc::idesc_bf16(2 * BM, BN, A_MN, B_MN);
    // block scaling: the kk-th MMA of a K block reads byte kk of the scale words
    uint32_t IDESC_MX[4];
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) IDESC_MX[kk] = tc::idesc_mxf8(2 * BM, BN, p.a_fmt, p.b_fmt, kk, kk);
    uint32_t acc_it = 0;
    int s = 0;         // ring slot of the next K block
    uint32_t ph = 0;   // its pass over the ring (parity)
    bool ok = true;
    for (int t = cid; t < total && ok; t += ncl) {
      const TileInfo ti = decode_tile<KIND, F8, AK>(bk, p, t, crank);
      if (ti.kblocks == 0) continue;
      const uint32_t a = acc_it & 1;
      const uint32_t aph = (acc_it >> 1) & 1;
      if (!tc::mbar_wait_warp(&bk.tempty[a], aph ^ 1, abort_flag, p.wait_limit_ns)) break;
      tc::tc_fence_after();
      const uint32_t d_tmem = tmem + a * BN;
      for (int kb = 0; kb < ti.kblocks; ++kb) {

        if (!tc::mbar_wait_warp(&bk.full[s], ph, abort_flag, p.wait_limit_ns)) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
        uint8_t *sa = smem + s * kStageB;
        uint8_t *sb = sa + A_BYTES;
        if (KIND == KIND_TGMM && !F8 && (!AK || B_MN)) {
          // rows past the expert's last row belong to the next expert: zero
          // them in both operands (one 128-byte row per K index per box).
          // 2-SM: this CTA's four boxes and the same four in the partner
          // CTA, whose copies have landed too (they complete on this CTA's
          // full barrier) and whose boxes this MMA reads.
          // (AK: A's copy is zero past the rows already; only B's boxes)
          const int valid = ti.row_end - (ti.row0 + kb * BK);
          if (valid < BK) {
            // lane = (row phase, 16-byte chunk): 4 rows per step, every box
            constexpr int kBox0 = AK ? 2 : 0;
            constexpr int kBoxes = AK ? 2 : 4;
            const int chunk = lane & 7;
            for (int rr = valid + (lane >> 3); rr < BK; rr += 4) {
#pragma unroll
              for (int box = kBox0; box < kBox0 + kBoxes; ++box) {
                uint8_t *base = box < 2 ? sa + box * BOX_BYTES : sb + (box - 2) * BOX_BYTES;
                const uint32_t off = rr * 128 + chunk * 16;
                *reinterpret_cast<uint4 *>(base + off) = make_uint4(0, 0, 0, 0);
                tc::st_cluster_zero16(tc::mapa_shared(tc::smem_u32(base), 1) + off);
              }
            }
            tc::fence_proxy_async_smem();
            tc::fence_proxy_async_smem_cluster();
          }
          __syncwarp();
        }
        if (lane == 0) {
          // descriptors of the stage's first MMA; the kk-th MMA starts 32 bytes
          // further along the row (K-major: 16 bf16 or 32 codes) or 16 rows of
          // 128 bytes further (MN-major), i.e. 2 or 128 in the address field
          const uint64_t ad0 = A_MN ? tc::sdesc(tc::smem_u32(sa), BOX_BYTES, 1024)
                                    : tc::sdesc(tc::smem_u32(sa), 16, 1024);
          const uint64_t bd0 = B_MN ? tc::sdesc(tc::smem_u32(sb), BOX_BYTES, 1024)
                                    : tc::sdesc(tc::smem_u32(sb), 16, 1024);
          constexpr uint64_t kAStep = A_MN ? (UK * 128) >> 4 : 32 >> 4;
          constexpr uint64_t kBStep = B_MN ? (UK * 128) >> 4 : 32 >> 4;
          if (MX) {
            // the stage's scale factors -> tensor memory, 12 columns per ring
            // slot after the two accumulators (A's atom, then B's two); the
            // copies and the MMAs run in issue order, and a slot is rewritten
            // only after the MMAs that read it released the stage
            const uint32_t sft = tmem + 2 * BN + s * 12;
            const uint32_t sfs = tc::smem_u32(sa + kSfOff);
#pragma unroll
            for (int j = 0; j < 3; ++j)
              tc::tmem_cp_32x128b_x4_2sm(sft + 4 * j, tc::sdesc_plain(sfs + 512 * j, 0, 128));
#pragma unroll
            for (int kk = 0; kk < BK / UK; ++kk)
              tc::umma_mxf8_2sm(d_tmem, ad0 + kk * kAStep, bd0 + kk * kBStep, IDESC_MX[kk], sft,
                                sft + 4, (kb | kk) != 0);
          } else {
#pragma unroll
            for (int kk = 0; kk < BK / UK; ++kk) {
              const uint64_t ad = ad0 + kk * kAStep;
              const uint64_t bd = bd0 + kk * kBStep;
              if (F8) tc::umma_f8_2sm(d_tmem, ad, bd, IDESC, (kb | kk) != 0);
              else tc::umma_bf16_2sm(d_tmem, ad, bd, IDESC, (kb | kk) != 0);
            }
          }
          // release the stage in both CTAs
          tc::umma_commit_2sm_mc(&bk.empty[s], kPair);
        }
        __syncwarp();
        if (++s == kSt) {
          s = 0;
          ph ^= 1;
        }
      }
      if (!ok) break;
      if (lane == 0) {
        tc::umma_commit_2sm_mc(&bk.tfull[a], kPair);  // both CTAs' epilogues
      }
      __syncwarp();
      ++acc_it;
    }
    // drain: no MMA of this CTA is in flight once `drain` completes
    if (lane == 0) {
      tc::umma_commit_2sm_mc(&bk.drain, 0x1);
    }
    __syncwarp();
    tc::mbar_wait_drain(&bk.drain, 0, p.wait_limit_ns);
  } else if (warp >= 2) {
    const int q = warp & 3;  // TMEM lane quarter this warp may read = its tile rows
    const int rit = q * 32 + lane;
    uint8_t *stg = smem + Ring<KIND, EPI, F8, BN, MX>::stg_offset +
                   (warp - 2) * Ring<KIND, EPI, F8, BN, MX>::stg_bytes;
    constexpr int kChunks = BN / 32;  // the tile's 32-column chunks, all this warp's
    const int c_begin = 0;
    OutMaps om{&tmC0, &tmC1, &tmC2, &tmC3, &bk.aux_full[warp - 2], 0u, 0u,
               tc::l2_evict_first_policy()};
    uint32_t acc_it = 0;
    uint32_t stg_slot = 0;  // tgmm: boxes staged so far (which half of the staging is next)
    float amx = 0.0f;
    for (int t = cid; t < total; t += ncl) {
      const TileInfo ti = decode_tile<KIND, F8, AK>(bk, p, t, crank);
      if (KIND == KIND_TGMM && ti.kblocks == 0) {
        if (!p.accumulate) epilogue_tgmm<F8, BN, MX>(p, ti, 0, q, lane, stg, om, true, stg_slot);
        continue;
      }
      epilogue_prefetch<KIND, EPI, BN>(p, ti, rit, c_begin, c_begin + kChunks);
      if (KIND == KIND_GMM && EPI == MOE_EPI_SWIGLU_BWD && lane == 0)
        issue_aux_load(om, stg, ti.n_idx * BN + c_begin * 32, ti.row0 + q * 32);  // first chunk
      if (KIND == KIND_GMM && EPI == kEpiSwigluPs && lane == 0) {
        tc::fence_proxy_async_smem();  // the previous tile's reads of the P blocks came first
        issue_ps_load(om, stg, ti.n_idx * (BN / 2) + c_begin * 32, p.F, ti.row0 + q * 32);
      }
      const uint32_t a = acc_it & 1;
      const uint32_t aph = (acc_it >> 1) & 1;
      if (!tc::mbar_wait_warp(&bk.tfull[a], aph, abort_flag, p.wait_limit_ns)) break;
      tc::tc_fence_after();
      const uint32_t taddr = tmem + a * BN + (static_cast<uint32_t>(q * 32) << 16);
      if (KIND == KIND_GMM)
        epilogue_gmm<EPI, F8, BN, MX, CT>(p, ti, taddr, q, lane, stg, om, abort_flag, c_begin,
                              c_begin + kChunks, amx);
      else
        epilogue_tgmm<F8, BN, MX>(p, ti, taddr, q, lane, stg, om, false, stg_slot);
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        tc::mbar_arrive_cluster(tc::mapa_shared(tc::smem_u32(&bk.tempty[a]), 0));
      }
      ++acc_it;
    }
    // the warp's output amax, once per kernel (bf16 rounding is monotone: the
    // rounded maximum is the maximum of the rounded outputs)
    if (KIND == KIND_GMM && F8 && p.amax_out != nullptr) {
      amx = warp_max(amx);
      if (lane == 0 && amx > 0.0f) {
        const float r = p.c_f32 && EPI == MOE_EPI_NONE
                            ? amx
                            : __bfloat162float(__float2bfloat16_rn(amx));
        atomicMax(reinterpret_cast<unsigned int *>(p.amax_out), __float_as_uint(r));
      }
    }
    // every bulk store and H load of this warp has completed before the CTA exits
    if (lane == 0) tc::bulk_wait0();
    if (KIND == KIND_GMM && (EPI == MOE_EPI_SWIGLU_BWD || EPI == kEpiSwigluPs) &&
        __shfl_sync(0xffffffffu, om.aux_issued, 0) != om.aux_phase)
      tc::mbar_wait_drain(om.aux_bar, om.aux_phase & 1, p.wait_limit_ns / 4);
    __syncwarp();
  }
  tc::tc_fence_before();
  __syncthreads();
  // the pair is done with each other's barriers, shared memory and TMEM
  tc::cluster_sync();
  tc::tc_fence_after();
  if (warp == 1) {
    tc::tmem_dealloc_2sm(tmem, kTmemCols);
  }
  if (threadIdx.x == 0 && bk.abort_flag) moe_set_status(p.dev_status, MOE_ERR_TIMEOUT);
}

// --------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// bf16 tensor map with 128-byte swizzle; dims[0] is the contiguous dimension.
bool make_map(CUtensorMap *m, const void *base, int rank, const uint64_t *dims,
              const uint64_t *strides_bytes, const uint32_t *box,
              CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t d[3], st[2];
  cuuint32_t b[3], es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
  }
  for (int i = 0; i < rank - 1; ++i) st[i] = strides_bytes[i];
  return fn(m, dtype, rank, const_cast<void *>(base), d, st, b, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Output map of a [rows, cols] row-major matrix written in 32 x 32 blocks
// (bf16: 64-byte rows, 64-byte swizzle; fp32: 128-byte rows, 128-byte swizzle).
bool make_out_map(CUtensorMap *m, const void *base, bool f32, int64_t cols, int64_t rows,
                  int64_t ld) {
  const uint64_t dims[2] = {(uint64_t)cols, (uint64_t)rows};
  const uint64_t st[1] = {(uint64_t)ld * (f32 ? 4 : 2)};
  const uint32_t box[2] = {32, 32};
  return make_map(m, base, 2, dims, st, box,
                  f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                  f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B);
}

template <int KIND, bool B_MN, int EPI, bool F8 = false, bool AK = F8, int BN = kBN,
          bool MX = false, bool CT = false>
moe_status_t launch_tc(const CUtensorMap &ma, const CUtensorMap &mb, const CUtensorMap *mc,
                       const TcParams &p, int64_t tiles_upper, cudaStream_t s,
                       const CUtensorMap *msf = nullptr) {
  constexpr int kSmem = Ring<KIND, EPI, F8, BN, MX>::smem_bytes;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  static int max_clusters = 0;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(gmm_tc_kernel<KIND, B_MN, EPI, F8, AK, BN, MX, CT>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (attr_err != cudaSuccess) return;
    // clusters of two CTAs (one per SM) that can be resident at once
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * (unsigned)num_sms());
    cfg.blockDim = dim3(Ring<KIND, EPI, F8, BN, MX>::threads);
    cfg.dynamicSmemBytes = kSmem;
    if (cudaOccupancyMaxActiveClusters(&max_clusters, gmm_tc_kernel<KIND, B_MN, EPI, F8, AK, BN, MX, CT>, &cfg) !=
            cudaSuccess ||
        max_clusters <= 0) {
      cudaGetLastError();
      max_clusters = num_sms() / 2;
    }
  });
  if (attr_err != cudaSuccess) {
    set_error("grouped GEMM: cannot reserve %d bytes of shared memory: %s", kSmem,
              cudaGetErrorString(attr_err));
    return MOE_ERR_CUDA;
  }
  const int64_t pairs = (tiles_upper + 1) / 2;
  const int grid = 2 * (int)std::max<int64_t>(1, std::min<int64_t>(max_clusters, pairs));
  gmm_tc_kernel<KIND, B_MN, EPI, F8, AK, BN, MX, CT><<<grid, Ring<KIND, EPI, F8, BN, MX>::threads, kSmem, s>>>(
      ma, mb, mc[0], mc[1], mc[2], mc[3], msf != nullptr ? msf[0] : ma,
      msf != nullptr ? msf[1] : ma, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("grouped GEMM launch: %s", cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

}  // namespace

moe_status_t launch_gmm(const GmmArgs &a, cudaStream_t s) {
  if (a.E > kMaxE) {
    set_error("moe_gmm: E=%d > %d", a.E, kMaxE);
    return MOE_ERR_UNSUPPORTED;
  }
  if (a.epilogue == MOE_EPI_SWIGLU_FWD && a.trans_b) {
    set_error("moe_gmm: the SwiGLU forward epilogue needs trans_b = 0 ([K, N] weights)");
    return MOE_ERR_UNSUPPORTED;
  }
  const bool b_mn = !a.trans_b;
  const int64_t stride_b = a.E > 1 ? a.stride_b : (a.trans_b ? (int64_t)a.N : (int64_t)a.K) * a.ldb;
  CUtensorMap ma, mb;
  {
    const uint64_t dims[2] = {(uint64_t)a.K, (uint64_t)a.rows_cap};
    const uint64_t st[1] = {(uint64_t)a.lda * 2};
    const uint32_t box[2] = {BK, BM};
    if (!make_map(&ma, a.A, 2, dims, st, box)) {
      set_error("moe_gmm: cannot encode the TMA descriptor of A");
      return MOE_ERR_CUDA;
    }
  }
  if (b_mn) {
    const uint64_t dims[3] = {(uint64_t)a.N, (uint64_t)a.K, (uint64_t)a.E};
    const uint64_t st[2] = {(uint64_t)a.ldb * 2, (uint64_t)stride_b * 2};
    const uint32_t box[3] = {64, BK, 1};
    if (!make_map(&mb, a.B, 3, dims, st, box)) {
      set_error("moe_gmm: cannot encode the TMA descriptor of B");
      return MOE_ERR_CUDA;
    }
  } else {
    const uint64_t dims[3] = {(uint64_t)a.K, (uint64_t)a.N, (uint64_t)a.E};
    const uint64_t st[2] = {(uint64_t)a.ldb * 2, (uint64_t)stride_b * 2};
    const uint32_t box[3] = {BK, kBN / 2, 1};
    if (!make_map(&mb, a.B, 3, dims, st, box)) {
      set_error("moe_gmm: cannot encode the TMA descriptor of B");
      return MOE_ERR_CUDA;
    }
  }
  TcParams p{};
  p.E = a.E;
  p.rows_cap = (int)a.rows_cap;
  p.K = a.K;
  p.N = a.N;
  p.F = a.epilogue == MOE_EPI_SWIGLU_FWD ? a.N / 2 : a.N;
  p.n_tiles = a.epilogue == MOE_EPI_SWIGLU_FWD ? (p.F + kBN / 2 - 1) / (kBN / 2) : (a.N + kBN - 1) / kBN;
  p.offsets = a.offsets;
  p.C = a.C;
  p.ldc = a.ldc;
  p.c_f32 = a.c_dtype == MOE_DTYPE_F32;
  p.C2 = a.C2;
  p.ldc2 = a.ldc2;
  p.Ct = a.Ct;
  p.ldct = a.ldct;
  p.ps = a.ps;
  p.ld_ps = a.ld_ps;
  p.bias = a.bias;
  p.stride_bias = a.stride_bias;
  p.aux = a.aux;
  p.ld_aux = a.ld_aux;
  p.dev_status = a.dev_status;
  p.wait_limit_ns = wait_limit_ns();
  p.stall_loads = test_stall_loads();
  // output maps (unused slots repeat the first)
  CUtensorMap mc[4];
  bool ok = true;
  const bool f32 = a.c_dtype == MOE_DTYPE_F32;
  if (a.epilogue == MOE_EPI_SWIGLU_FWD) {
    const uint16_t *H = static_cast<const uint16_t *>(a.C);
    ok = make_out_map(&mc[0], H, false, p.F, a.rows_cap, a.ldc) &&
         make_out_map(&mc[1], H + p.F, false, p.F, a.rows_cap, a.ldc) &&
         make_out_map(&mc[2], a.C2, false, p.F, a.rows_cap, a.ldc2);
    // m3: the column-wise copy Act^T [F, padded rows] (transposed 32 x 32 blocks)
    if (a.Ct != nullptr)
      ok = ok && make_out_map(&mc[3], a.Ct, false, f8_padded_rows(a.rows_cap, a.E), p.F, a.ldct);
    else
      mc[3] = mc[0];
  } else if (a.epilogue == MOE_EPI_SWIGLU_BWD) {
    const uint16_t *dH = static_cast<const uint16_t *>(a.C);
    // m0/m1: dH gate / up (stores); m2/m3: H gate / up (loads, same block shape)
    ok = make_out_map(&mc[0], dH, false, a.N, a.rows_cap, a.ldc) &&
         make_out_map(&mc[1], dH + a.N, false, a.N, a.rows_cap, a.ldc) &&
         make_out_map(&mc[2], a.aux, false, a.N, a.rows_cap, a.ld_aux) &&
         make_out_map(&mc[3], a.aux + a.N, false, a.N, a.rows_cap, a.ld_aux);
  } else {
    ok = make_out_map(&mc[0], a.C, f32, a.N, a.rows_cap, a.ldc);
    mc[1] = mc[2] = mc[3] = mc[0];
  }
  if (!ok) {
    set_error("moe_gmm: cannot encode the TMA descriptor of the output");
    return MOE_ERR_CUDA;
  }
  const int64_t tiles_upper = ((a.rows_cap + BM - 1) / BM + a.E) * p.n_tiles;
  // the column-wise copies (Ct) come from instances of their own, so that the
  // default epilogues keep their registers
  if (a.Ct != nullptr) {
    if (a.epilogue == MOE_EPI_SWIGLU_FWD && b_mn)
      return launch_tc<KIND_GMM, true, MOE_EPI_SWIGLU_FWD, false, false, kBN, false, true>(
          ma, mb, mc, p, tiles_upper, s);
    if (a.epilogue == MOE_EPI_SWIGLU_BWD)
      return b_mn ? launch_tc<KIND_GMM, true, MOE_EPI_SWIGLU_BWD, false, false, kBN, false, true>(
                        ma, mb, mc, p, tiles_upper, s)
                  : launch_tc<KIND_GMM, false, MOE_EPI_SWIGLU_BWD, false, false, kBN, false,
                              true>(ma, mb, mc, p, tiles_upper, s);
    set_error("moe_gmm: no column-wise copy for this epilogue / layout");
    return MOE_ERR_UNSUPPORTED;
  }
  if (a.epilogue == MOE_EPI_SWIGLU_FWD && a.ps != nullptr && b_mn) {
    // m3: the partial sum P [rows_cap, 2F] fp32, read in 32 x 32 blocks
    if (!make_out_map(&mc[3], a.ps, true, 2 * p.F, a.rows_cap, a.ld_ps)) {
      set_error("moe_gmm: cannot encode the TMA descriptor of the partial sum");
      return MOE_ERR_CUDA;
    }
    return launch_tc<KIND_GMM, true, kEpiSwigluPs>(ma, mb, mc, p, tiles_upper, s);
  }
  switch (a.epilogue * 2 + (b_mn ? 1 : 0)) {
    case MOE_EPI_NONE * 2 + 1:
      return launch_tc<KIND_GMM, true, MOE_EPI_NONE>(ma, mb, mc, p, tiles_upper, s);
    case MOE_EPI_NONE * 2 + 0:
      return launch_tc<KIND_GMM, false, MOE_EPI_NONE>(ma, mb, mc, p, tiles_upper, s);
    case MOE_EPI_SWIGLU_FWD * 2 + 1:
      return launch_tc<KIND_GMM, true, MOE_EPI_SWIGLU_FWD>(ma, mb, mc, p, tiles_upper, s);
    case MOE_EPI_SWIGLU_BWD * 2 + 1:
      return launch_tc<KIND_GMM, true, MOE_EPI_SWIGLU_BWD>(ma, mb, mc, p, tiles_upper, s);
    case MOE_EPI_SWIGLU_BWD * 2 + 0:
      return launch_tc<KIND_GMM, false, MOE_EPI_SWIGLU_BWD>(ma, mb, mc, p, tiles_upper, s);
    default:
      set_error("moe_gmm: unsupported epilogue / layout");
      return MOE_ERR_UNSUPPORTED;
  }
}

// At == nullptr: A read as stored (MN-major); else K-major from its
// column-wise copy At [M, ldat] (zero-padded group layout).
static moe_status_t tgmm_impl(const TgmmArgs &a, const uint16_t *At, int64_t ldat,
                              bool b_colwise, cudaStream_t s) {
  if (a.E > kMaxE) {
    set_error("moe_tgmm: E=%d > %d", a.E, kMaxE);
    return MOE_ERR_UNSUPPORTED;
  }
  CUtensorMap ma, mb;
  const uint32_t box[2] = {64, BK};
  if (At != nullptr) {
    const uint64_t dims[2] = {(uint64_t)f8_padded_rows(a.rows_cap, a.E), (uint64_t)a.M};
    const uint64_t st[1] = {(uint64_t)ldat * 2};
    const uint32_t abox[2] = {BK, BM};
    if (!make_map(&ma, At, 2, dims, st, abox)) {
      set_error("moe_tgmm: cannot encode the TMA descriptor of A");
      return MOE_ERR_CUDA;
    }
  } else {
    const uint64_t dims[2] = {(uint64_t)a.M, (uint64_t)a.rows_cap};
    const uint64_t st[1] = {(uint64_t)a.lda * 2};
    if (!make_map(&ma, a.A, 2, dims, st, box)) {
      set_error("moe_tgmm: cannot encode the TMA descriptor of A");
      return MOE_ERR_CUDA;
    }
  }
  if (b_colwise) {
    const uint64_t dims[2] = {(uint64_t)f8_padded_rows(a.rows_cap, a.E), (uint64_t)a.N};
    const uint64_t st[1] = {(uint64_t)a.ldb * 2};
    const uint32_t bbox[2] = {BK, kBN / 2};
    if (!make_map(&mb, a.B, 2, dims, st, bbox)) {
      set_error("moe_tgmm: cannot encode the TMA descriptor of B");
      return MOE_ERR_CUDA;
    }
  } else {
    const uint64_t dims[2] = {(uint64_t)a.N, (uint64_t)a.rows_cap};
    const uint64_t st[1] = {(uint64_t)a.ldb * 2};
    if (!make_map(&mb, a.B, 2, dims, st, box)) {
      set_error("moe_tgmm: cannot encode the TMA descriptor of B");
      return MOE_ERR_CUDA;
    }
  }
  TcParams p{};
  p.E = a.E;
  p.rows_cap = (int)a.rows_cap;
  p.M = a.M;
  p.N = a.N;
  p.m_tiles = (a.M + BM - 1) / BM;
  p.n_tiles = (a.N + kBN - 1) / kBN;
  p.offsets = a.offsets;
  p.C = a.W;
  p.ldc = a.ldw;
  p.c_f32 = a.w_dtype == MOE_DTYPE_F32;
  p.stride_w = a.stride_w;
  p.accumulate = a.accumulate;
  p.dev_status = a.dev_status;
  p.wait_limit_ns = wait_limit_ns();
  p.stall_loads = test_stall_loads();
  CUtensorMap mc[4];
  {
    const bool f32 = a.w_dtype == MOE_DTYPE_F32;
    const int64_t es = f32 ? 4 : 2;
    const int64_t stride_w = a.E > 1 ? a.stride_w : (int64_t)a.M * a.ldw;
    const uint64_t dims[3] = {(uint64_t)a.N, (uint64_t)a.M, (uint64_t)a.E};
    const uint64_t st[2] = {(uint64_t)(a.ldw * es), (uint64_t)(stride_w * es)};
    const uint32_t box[3] = {f32 ? 32u : 64u, 32, 1};
    if (!make_map(&mc[0], a.W, 3, dims, st, box,
                  f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                  CU_TENSOR_MAP_SWIZZLE_128B)) {
      set_error("moe_tgmm: cannot encode the TMA descriptor of W");
      return MOE_ERR_CUDA;
    }
    mc[1] = mc[2] = mc[3] = mc[0];
  }
  const int64_t tiles_upper = (int64_t)a.E * p.m_tiles * p.n_tiles;
  if (At != nullptr && b_colwise)
    return launch_tc<KIND_TGMM, false, MOE_EPI_NONE, false, true>(ma, mb, mc, p, tiles_upper, s);
  if (At != nullptr)
    return launch_tc<KIND_TGMM, true, MOE_EPI_NONE, false, true>(ma, mb, mc, p, tiles_upper, s);
  return launch_tc<KIND_TGMM, true, MOE_EPI_NONE>(ma, mb, mc, p, tiles_upper, s);
}

moe_status_t launch_tgmm(const TgmmArgs &a, cudaStream_t s) {
  return tgmm_impl(a, nullptr, 0, false, s);
}

moe_status_t launch_tgmm_kt(const TgmmArgs &a, const uint16_t *At, int64_t ldat, bool b_colwise,
                            cudaStream_t s) {
  return tgmm_impl(a, At, ldat, b_colwise, s);
}

// Output maps shared by the bf16 and FP8 ragged-M GEMMs (unused slots repeat
// the first).
static bool gmm_out_maps(CUtensorMap *mc, int epilogue, void *C, int c_dtype, int64_t ldc,
                         uint16_t *C2, int64_t ldc2, const uint16_t *aux, int64_t ld_aux, int N,
                         int F, int64_t rows_cap) {
  const bool f32 = c_dtype == MOE_DTYPE_F32;
  if (epilogue == MOE_EPI_SWIGLU_FWD) {
    const uint16_t *H = static_cast<const uint16_t *>(C);
    if (!make_out_map(&mc[0], H, false, F, rows_cap, ldc) ||
        !make_out_map(&mc[1], H + F, false, F, rows_cap, ldc) ||
        !make_out_map(&mc[2], C2, false, F, rows_cap, ldc2))
      return false;
    mc[3] = mc[0];
    return true;
  }
  if (epilogue == MOE_EPI_SWIGLU_BWD) {
    const uint16_t *dH = static_cast<const uint16_t *>(C);
    return make_out_map(&mc[0], dH, false, N, rows_cap, ldc) &&
           make_out_map(&mc[1], dH + N, false, N, rows_cap, ldc) &&
           make_out_map(&mc[2], aux, false, N, rows_cap, ld_aux) &&
           make_out_map(&mc[3], aux + N, false, N, rows_cap, ld_aux);
  }
  if (!make_out_map(&mc[0], C, f32, N, rows_cap, ldc)) return false;
  mc[1] = mc[2] = mc[3] = mc[0];
  return true;
}

moe_status_t launch_gmm_f8(const GmmF8Args &a, cudaStream_t s) {
  if (a.E > kMaxE) {
    set_error("moe_gmm_fp8: E=%d > %d", a.E, kMaxE);
    return MOE_ERR_UNSUPPORTED;
  }
  const int64_t stride_b = a.E > 1 ? a.stride_b : (int64_t)a.N * a.ldb;
  CUtensorMap ma, mb;
  {
    const uint64_t dims[2] = {(uint64_t)a.K, (uint64_t)a.rows_cap};
    const uint64_t st[1] = {(uint64_t)a.lda};
    const uint32_t box[2] = {Elem<true>::BKE, BM};
    if (!make_map(&ma, a.A, 2, dims, st, box, CU_TENSOR_MAP_DATA_TYPE_UINT8)) {
      set_error("moe_gmm_fp8: cannot encode the TMA descriptor of A");
      return MOE_ERR_CUDA;
    }
  }
  {
    const uint64_t dims[3] = {(uint64_t)a.K, (uint64_t)a.N, (uint64_t)a.E};
    const uint64_t st[2] = {(uint64_t)a.ldb, (uint64_t)stride_b};
    const uint32_t box[3] = {Elem<true>::BKE, kBN / 2, 1};
    if (!make_map(&mb, a.B, 3, dims, st, box, CU_TENSOR_MAP_DATA_TYPE_UINT8)) {
      set_error("moe_gmm_fp8: cannot encode the TMA descriptor of B");
      return MOE_ERR_CUDA;
    }
  }
  TcParams p{};
  p.E = a.E;
  p.rows_cap = (int)a.rows_cap;
  p.K = a.K;
  p.N = a.N;
  p.F = a.epilogue == MOE_EPI_SWIGLU_FWD ? a.N / 2 : a.N;
  p.n_tiles = a.epilogue == MOE_EPI_SWIGLU_FWD ? (p.F + kBN / 2 - 1) / (kBN / 2) : (a.N + kBN - 1) / kBN;
  p.offsets = a.offsets;
  p.C = a.C;
  p.ldc = a.ldc;
  p.c_f32 = a.c_dtype == MOE_DTYPE_F32;
  p.C2 = a.C2;
  p.ldc2 = a.ldc2;
  p.aux = a.aux;
  p.ld_aux = a.ld_aux;
  p.dev_status = a.dev_status;
  p.wait_limit_ns = wait_limit_ns();
  p.stall_loads = test_stall_loads();
  p.a_sinv = a.a_sinv;
  p.b_sinv = a.b_sinv;
  p.a_fmt = a.a_fmt;
  p.b_fmt = a.b_fmt;
  p.amax_out = a.amax_out;
  if (a.amax_out != nullptr) {
    const cudaError_t e = cudaMemsetAsync(a.amax_out, 0, sizeof(float), s);
    if (e != cudaSuccess) {
      set_error("moe_gmm_fp8: amax reset: %s", cudaGetErrorString(e));
      return MOE_ERR_CUDA;
    }
  }
  CUtensorMap mc[4];
  if (!gmm_out_maps(mc, a.epilogue, a.C, a.c_dtype, a.ldc, a.C2, a.ldc2, a.aux, a.ld_aux, a.N,
                    p.F, a.rows_cap)) {
    set_error("moe_gmm_fp8: cannot encode the TMA descriptor of the output");
    return MOE_ERR_CUDA;
  }
  const int64_t tiles_upper = ((a.rows_cap + BM - 1) / BM + a.E) * p.n_tiles;
  switch (a.epilogue) {
    case MOE_EPI_NONE:
      return launch_tc<KIND_GMM, false, MOE_EPI_NONE, true>(ma, mb, mc, p, tiles_upper, s);
    case MOE_EPI_SWIGLU_FWD:
      return launch_tc<KIND_GMM, false, MOE_EPI_SWIGLU_FWD, true>(ma, mb, mc, p, tiles_upper, s);
    case MOE_EPI_SWIGLU_BWD:
      return launch_tc<KIND_GMM, false, MOE_EPI_SWIGLU_BWD, true>(ma, mb, mc, p, tiles_upper, s);
    default:
      set_error("moe_gmm_fp8: unsupported epilogue");
      return MOE_ERR_UNSUPPORTED;
  }
}

moe_status_t launch_tgmm_f8(const TgmmF8Args &a, cudaStream_t s) {
  if (a.E > kMaxE) {
    set_error("moe_tgmm_fp8: E=%d > %d", a.E, kMaxE);
    return MOE_ERR_UNSUPPORTED;
  }
  const int64_t P = f8_padded_rows(a.rows_cap, a.E);  // columns the copies may use
  CUtensorMap ma, mb;
  const uint32_t box[2] = {Elem<true>::BKE, BM};
  {
    const uint64_t dims[2] = {(uint64_t)P, (uint64_t)a.M};
    const uint64_t st[1] = {(uint64_t)a.ldat};
    if (!make_map(&ma, a.At, 2, dims, st, box, CU_TENSOR_MAP_DATA_TYPE_UINT8)) {
      set_error("moe_tgmm_fp8: cannot encode the TMA descriptor of A");
      return MOE_ERR_CUDA;
    }
  }
  {
    const uint64_t dims[2] = {(uint64_t)P, (uint64_t)a.N};
    const uint64_t st[1] = {(uint64_t)a.ldbt};
    if (!make_map(&mb, a.Bt, 2, dims, st, box, CU_TENSOR_MAP_DATA_TYPE_UINT8)) {
      set_error("moe_tgmm_fp8: cannot encode the TMA descriptor of B");
      return MOE_ERR_CUDA;
    }
  }
  TcParams p{};
  p.E = a.E;
  p.rows_cap = (int)a.rows_cap;
  p.M = a.M;
  p.N = a.N;
  p.m_tiles = (a.M + BM - 1) / BM;
  p.n_tiles = (a.N + kBN - 1) / kBN;
  p.offsets = a.offsets;
  p.C = a.W;
  p.ldc = a.ldw;
  p.c_f32 = a.w_dtype == MOE_DTYPE_F32;
  p.stride_w = a.stride_w;
  p.accumulate = a.accumulate;
  p.dev_status = a.dev_status;
  p.wait_limit_ns = wait_limit_ns();
  p.stall_loads = test_stall_loads();
  p.a_sinv = a.a_sinv;
  p.b_sinv = a.b_sinv;
  p.a_fmt = a.a_fmt;
  p.b_fmt = a.b_fmt;
  CUtensorMap mc[4];
  {
    const bool f32 = a.w_dtype == MOE_DTYPE_F32;
    const int64_t es = f32 ? 4 : 2;
    const int64_t stride_w = a.E > 1 ? a.stride_w : (int64_t)a.M * a.ldw;
    const uint64_t dims[3] = {(uint64_t)a.N, (uint64_t)a.M, (uint64_t)a.E};
    const uint64_t st[2] = {(uint64_t)(a.ldw * es), (uint64_t)(stride_w * es)};
    const uint32_t wbox[3] = {f32 ? 32u : 64u, 32, 1};
    if (!make_map(&mc[0], a.W, 3, dims, st, wbox,
                  f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                  CU_TENSOR_MAP_SWIZZLE_128B)) {
      set_error("moe_tgmm_fp8: cannot encode the TMA descriptor of W");
      return MOE_ERR_CUDA;
    }
    mc[1] = mc[2] = mc[3] = mc[0];
  }
  const int64_t tiles_upper = (int64_t)a.E * p.m_tiles * p.n_tiles;
  return launch_tc<KIND_TGMM, false, MOE_EPI_NONE, true>(ma, mb, mc, p, tiles_upper, s);
}

// Scale-factor maps of the block-scaled operands: 512-byte atoms viewed as
// 32-bit words.  A: [atoms, 128] (one atom per box).  B: [atom rows, atom
// columns, 128] (the two atom rows of a 192-column tile per box).
static bool make_sf_map(CUtensorMap *m, const uint8_t *sf, int64_t atoms) {
  const uint64_t dims[2] = {128, (uint64_t)atoms};
  const uint64_t st[1] = {512};
  const uint32_t box[2] = {128, 1};
  return make_map(m, sf, 2, dims, st, box, CU_TENSOR_MAP_DATA_TYPE_UINT32,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
}

static bool make_sf_map_b(CUtensorMap *m, const uint8_t *sf, int64_t atom_cols,
                          int64_t atom_rows) {
  const uint64_t dims[3] = {128, (uint64_t)atom_cols, (uint64_t)atom_rows};
  const uint64_t st[2] = {512, (uint64_t)atom_cols * 512};
  const uint32_t box[3] = {128, 1, 2};
  return make_map(m, sf, 3, dims, st, box, CU_TENSOR_MAP_DATA_TYPE_UINT32,
                  CU_TENSOR_MAP_SWIZZLE_NONE);
}

moe_status_t launch_gmm_mx(const GmmMxArgs &a, cudaStream_t s) {
  if (a.E > kMaxE) {
    set_error("moe_gmm_mx: E=%d > %d", a.E, kMaxE);
    return MOE_ERR_UNSUPPORTED;
  }
  const bool swiglu = a.epilogue == MOE_EPI_SWIGLU_FWD;
  const int64_t stride_b = a.E > 1 ? a.stride_b : (int64_t)a.N * a.ldb;
  const int KB = a.K / 128;
  CUtensorMap ma, mb, msf[2];
  {
    const uint64_t dims[2] = {(uint64_t)a.K, (uint64_t)a.rows_cap};
    const uint64_t st[1] = {(uint64_t)a.lda};
    const uint32_t box[2] = {Elem<true>::BKE, BM};
    if (!make_map(&ma, a.A, 2, dims, st, box, CU_TENSOR_MAP_DATA_TYPE_UINT8)) {
      set_error("moe_gmm_mx: cannot encode the TMA descriptor of A");
      return MOE_ERR_CUDA;
    }
  }
  {
    const uint64_t dims[3] = {(uint64_t)a.K, (uint64_t)a.N, (uint64_t)a.E};
    const uint64_t st[2] = {(uint64_t)a.ldb, (uint64_t)stride_b};
    const uint32_t box[3] = {Elem<true>::BKE, kBNmx / 2, 1};
    if (!make_map(&mb, a.B, 3, dims, st, box, CU_TENSOR_MAP_DATA_TYPE_UINT8)) {
      set_error("moe_gmm_mx: cannot encode the TMA descriptor of B");
      return MOE_ERR_CUDA;
    }
  }
  // A: the expert-padded row tiles.  B: quantized as [E N, K] (tiles of each
  // expert's N rows, sfb_by_cols = 0) or as [N, E K] (expert e's K columns at
  // e K; MOE_MX_ROWS_SWIGLU for the up-projection, sfb_by_cols = 1)
  const int64_t a_atoms = f8_padded_rows(a.rows_cap, a.E) / 128 * KB;
  const int64_t tiles_n = swiglu ? (a.N / 2 + kBNmx / 2 - 1) / (kBNmx / 2)
                                 : (a.N + kBNmx - 1) / kBNmx;
  const int64_t b_cols = a.sfb_by_cols ? (int64_t)a.E * KB : KB;
  const int64_t b_rows = a.sfb_by_cols ? 2 * tiles_n : (int64_t)a.E * 2 * tiles_n;
  if (!make_sf_map(&msf[0], a.sfa, a_atoms) || !make_sf_map_b(&msf[1], a.sfb, b_cols, b_rows)) {
    set_error("moe_gmm_mx: cannot encode the TMA descriptors of the scale factors");
    return MOE_ERR_CUDA;
  }
  TcParams p{};
  p.E = a.E;
  p.rows_cap = (int)a.rows_cap;
  p.K = a.K;
  p.N = a.N;
  p.F = swiglu ? a.N / 2 : a.N;
  p.n_tiles = (int)tiles_n;
  p.offsets = a.offsets;
  p.C = a.C;
  p.ldc = a.ldc;
  p.c_f32 = a.c_dtype == MOE_DTYPE_F32;
  p.C2 = a.C2;
  p.ldc2 = a.ldc2;
  p.aux = a.aux;
  p.ld_aux = a.ld_aux;
  p.dev_status = a.dev_status;
  p.wait_limit_ns = wait_limit_ns();
  p.stall_loads = test_stall_loads();
  p.a_fmt = a.a_fmt;
  p.b_fmt = a.b_fmt;
  p.sfa_stride = KB;
  p.sfb_ecol = a.sfb_by_cols ? KB : 0;
  p.sfb_erow = a.sfb_by_cols ? 0 : (int)(2 * tiles_n);
  CUtensorMap mc[4];
  if (!gmm_out_maps(mc, a.epilogue, a.C, a.c_dtype, a.ldc, a.C2, a.ldc2, a.aux, a.ld_aux, a.N,
                    p.F, a.rows_cap)) {
    set_error("moe_gmm_mx: cannot encode the TMA descriptor of the output");
    return MOE_ERR_CUDA;
  }
  const int64_t tiles_upper = ((a.rows_cap + BM - 1) / BM + a.E) * p.n_tiles;
  switch (a.epilogue) {
    case MOE_EPI_NONE:
      return launch_tc<KIND_GMM, false, MOE_EPI_NONE, true, true, kBNmx, true>(
          ma, mb, mc, p, tiles_upper, s, msf);
    case MOE_EPI_SWIGLU_FWD:
      return launch_tc<KIND_GMM, false, MOE_EPI_SWIGLU_FWD, true, true, kBNmx, true>(
          ma, mb, mc, p, tiles_upper, s, msf);
    case MOE_EPI_SWIGLU_BWD:
      return launch_tc<KIND_GMM, false, MOE_EPI_SWIGLU_BWD, true, true, kBNmx, true>(
          ma, mb, mc, p, tiles_upper, s, msf);
    default:
      set_error("moe_gmm_mx: unsupported epilogue");
      return MOE_ERR_UNSUPPORTED;
  }
}

moe_status_t launch_tgmm_mx(const TgmmMxArgs &a, cudaStream_t s) {
  if (a.E > kMaxE) {
    set_error("moe_tgmm_mx: E=%d > %d", a.E, kMaxE);
    return MOE_ERR_UNSUPPORTED;
  }
  const int64_t P = f8_padded_rows(a.rows_cap, a.E);
  CUtensorMap ma, mb, msf[2];
  const uint32_t abox[2] = {Elem<true>::BKE, BM};
  const uint32_t bbox[2] = {Elem<true>::BKE, kBNmx / 2};
  {
    const uint64_t dims[2] = {(uint64_t)P, (uint64_t)a.M};
    const uint64_t st[1] = {(uint64_t)a.ldat};
    if (!make_map(&ma, a.At, 2, dims, st, abox, CU_TENSOR_MAP_DATA_TYPE_UINT8)) {
      set_error("moe_tgmm_mx: cannot encode the TMA descriptor of A");
      return MOE_ERR_CUDA;
    }
  }
  {
    const uint64_t dims[2] = {(uint64_t)P, (uint64_t)a.N};
    const uint64_t st[1] = {(uint64_t)a.ldbt};
    if (!make_map(&mb, a.Bt, 2, dims, st, bbox, CU_TENSOR_MAP_DATA_TYPE_UINT8)) {
      set_error("moe_tgmm_mx: cannot encode the TMA descriptor of B");
      return MOE_ERR_CUDA;
    }
  }
  // At [M, P] quantized PLAIN (atom per 128 rows), Bt [N, P] quantized in
  // 192-row tiles (MOE_MX_ROWS_TILES, one group)
  const int64_t pk = P / 128;
  const int64_t tiles_n = (a.N + kBNmx - 1) / kBNmx;
  if (!make_sf_map(&msf[0], a.sfa, (a.M + 127) / 128 * pk) ||
      !make_sf_map_b(&msf[1], a.sfb, pk, 2 * tiles_n)) {
    set_error("moe_tgmm_mx: cannot encode the TMA descriptors of the scale factors");
    return MOE_ERR_CUDA;
  }
  TcParams p{};
  p.E = a.E;
  p.rows_cap = (int)a.rows_cap;
  p.M = a.M;
  p.N = a.N;
  p.m_tiles = (a.M + BM - 1) / BM;
  p.n_tiles = (int)tiles_n;
  p.offsets = a.offsets;
  p.C = a.W;
  p.ldc = a.ldw;
  p.c_f32 = a.w_dtype == MOE_DTYPE_F32;
  p.stride_w = a.stride_w;
  p.accumulate = a.accumulate;
  p.dev_status = a.dev_status;
  p.wait_limit_ns = wait_limit_ns();
  p.stall_loads = test_stall_loads();
  p.a_fmt = a.a_fmt;
  p.b_fmt = a.b_fmt;
  p.sfa_stride = pk;
  CUtensorMap mc[4];
  {
    const bool f32 = a.w_dtype == MOE_DTYPE_F32;
    const int64_t es = f32 ? 4 : 2;
    const int64_t stride_w = a.E > 1 ? a.stride_w : (int64_t)a.M * a.ldw;
    const uint64_t dims[3] = {(uint64_t)a.N, (uint64_t)a.M, (uint64_t)a.E};
    const uint64_t st[2] = {(uint64_t)(a.ldw * es), (uint64_t)(stride_w * es)};
    const uint32_t wbox[3] = {f32 ? 32u : 64u, 32, 1};
    if (!make_map(&mc[0], a.W, 3, dims, st, wbox,
                  f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                  CU_TENSOR_MAP_SWIZZLE_128B)) {
      set_error("moe_tgmm_mx: cannot encode the TMA descriptor of W");
      return MOE_ERR_CUDA;
    }
    mc[1] = mc[2] = mc[3] = mc[0];
  }
  const int64_t tiles_upper = (int64_t)a.E * p.m_tiles * p.n_tiles;
  return launch_tc<KIND_TGMM, false, MOE_EPI_NONE, true, true, kBNmx, true>(
      ma, mb, mc, p, tiles_upper, s, msf);
}

}  // namespace moe
