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
// Design (one persistent CTA per SM, 320 threads, warp-specialised):
//   warp 0      TMA producer: 128x64 A tiles and 256x64 B tiles (bf16,
//               128-byte swizzle) into a 4-stage shared-memory ring;
//   warp 1      TMEM owner and MMA issuer: tcgen05.mma kind::f16,
//               M=128 N=256 K=16, fp32 accumulators in TMEM, two 256-column
//               accumulators so the epilogue of one tile overlaps the
//               mainloop of the next;
//   warps 2-9   epilogue: tcgen05.ld of one TMEM lane (= one output row) per
//               thread, fused SwiGLU / partial-sum / cast, 16-byte stores; two
//               warps per TMEM lane quarter, each taking half of the columns,
//               so that the SwiGLU math keeps pace with the mainloop.
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

constexpr int BM = 128, BN = 256, BK = 64, UK = 16;
constexpr int kStages = 4;
constexpr int kThreads = 320;  // producer, MMA, 8 epilogue warps
constexpr int kEpiWarps = 8;
constexpr int A_BYTES = BM * BK * 2;   // 16 KB
constexpr int B_BYTES = BN * BK * 2;   // 32 KB
constexpr int BOX_BYTES = 64 * 64 * 2; // one 64x64 MN-major box, 8 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int kMaxE = 256;
constexpr int kGroupM = 32;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr int kTmemCols = 2 * BN;                 // two accumulators

enum { KIND_GMM = 0, KIND_TGMM = 1 };

struct Book {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
  int total_tiles;
  int off[kMaxE + 1];
  int cum[kMaxE + 1];
};
constexpr int SMEM_BYTES = 1024 + kStages * STAGE_BYTES + (int)((sizeof(Book) + 127) / 128 * 128);

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
  const float *ps;
  int64_t ld_ps;
  const uint16_t *aux;
  int64_t ld_aux;
  int64_t stride_w;
  int accumulate;
  int32_t *dev_status;
};

struct TileInfo {
  int e, m_idx, n_idx, row0, row_end, kblocks;
};

template <int KIND>
MOE_DEVINL TileInfo decode_tile(const Book &bk, const TcParams &p, int t) {
  int lo = 0, hi = p.E - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (bk.cum[mid] <= t) lo = mid;
    else hi = mid - 1;
  }
  TileInfo ti;
  ti.e = lo;
  const int local = t - bk.cum[lo];
  ti.row0 = bk.off[lo];
  ti.row_end = bk.off[lo + 1];
  const int size = ti.row_end - ti.row0;
  const int mt = KIND == KIND_GMM ? (size + BM - 1) / BM : p.m_tiles;
  const int group = kGroupM * p.n_tiles;
  const int g = local / group;
  const int within = local - g * group;
  const int gm = min(kGroupM, mt - g * kGroupM);
  ti.n_idx = within / gm;
  ti.m_idx = g * kGroupM + (within - ti.n_idx * gm);
  if (KIND == KIND_GMM) {
    ti.row0 += ti.m_idx * BM;
    ti.kblocks = (p.K + BK - 1) / BK;
  } else {
    ti.kblocks = (size + BK - 1) / BK;
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

MOE_DEVINL void ld_f32x8(const float *src, float *v) {
  const float4 a = *reinterpret_cast<const float4 *>(src);
  const float4 b = *reinterpret_cast<const float4 *>(src + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
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

// Before a tile's accumulator is ready: pull the epilogue's global inputs
// (SwiGLU-backward H, partial sums) into L2 so that the epilogue's loads do
// not wait on HBM one after another.  Thread = one output row.
template <int KIND, int EPI>
MOE_DEVINL void epilogue_prefetch(const TcParams &p, const TileInfo &ti, int rit, int half) {
  if (KIND == KIND_GMM) {
    const int64_t row = (int64_t)ti.row0 + rit;
    if (row >= ti.row_end) return;
    if (EPI == MOE_EPI_SWIGLU_BWD) {
      const uint16_t *h = p.aux + row * p.ld_aux;
      const int n0 = ti.n_idx * BN + half * (BN / 2);
      for (int n = n0; n < min(n0 + BN / 2, p.N); n += 64) {
        prefetch_l2(h + n);
        prefetch_l2(h + p.N + n);
      }
    } else if (p.ps != nullptr) {
      const float *q = p.ps + row * p.ld_ps;
      if (EPI == MOE_EPI_SWIGLU_FWD) {
        const int n0 = ti.n_idx * (BN / 2) + half * (BN / 4);
        for (int n = n0; n < min(n0 + BN / 4, p.F); n += 32) {
          prefetch_l2(q + n);
          prefetch_l2(q + p.F + n);
        }
      } else {
        const int n0 = ti.n_idx * BN + half * (BN / 2);
        for (int n = n0; n < min(n0 + BN / 2, p.N); n += 32) prefetch_l2(q + n);
      }
    }
  } else if (p.accumulate) {
    const int m = ti.m_idx * BM + rit;
    if (m >= p.M) return;
    const float *w = static_cast<const float *>(p.C) + (int64_t)ti.e * p.stride_w +
                     (int64_t)m * p.ldc;
    const int n0 = ti.n_idx * BN + half * (BN / 2);
    for (int n = n0; n < min(n0 + BN / 2, p.N); n += 32) prefetch_l2(w + n);
  }
}

// One tile's epilogue for the ragged-M GEMM.  Thread = one output row.  The
// global inputs of a 32-column chunk are loaded before its TMEM read so that
// the two latencies overlap.
template <int EPI>
MOE_DEVINL void epilogue_gmm(const TcParams &p, const TileInfo &ti, uint32_t taddr, int rit,
                             int half) {
  const int64_t row = (int64_t)ti.row0 + rit;
  const bool valid = row < ti.row_end;
  if (EPI == MOE_EPI_SWIGLU_FWD) {
    const int F = p.F;
    const int n0 = ti.n_idx * (BN / 2);
#pragma unroll 1
    for (int c = half * (BN / 2 / 32 / 2); c < (half + 1) * (BN / 2 / 32 / 2); ++c) {
      const int nc = n0 + c * 32;
      if (nc >= F) break;
      float pg[32], pu[32];
      const bool has_ps = valid && p.ps != nullptr;
      if (has_ps) {
#pragma unroll
        for (int j8 = 0; j8 < 4; ++j8) {
          if (nc + j8 * 8 < F) {
            ld_f32x8(p.ps + row * p.ld_ps + nc + j8 * 8, pg + j8 * 8);
            ld_f32x8(p.ps + row * p.ld_ps + F + nc + j8 * 8, pu + j8 * 8);
          }
        }
      }
      float g[32], u[32];
      tc::tmem_ld32(taddr + c * 32, g);
      tc::tmem_ld32(taddr + BN / 2 + c * 32, u);
      if (!valid) continue;
      uint16_t *H = static_cast<uint16_t *>(p.C) + row * p.ldc;
      uint16_t *A = p.C2 + row * p.ldc2;
#pragma unroll
      for (int j8 = 0; j8 < 4; ++j8) {
        const int n = nc + j8 * 8;
        if (n >= F) break;
        float *gv = g + j8 * 8, *uv = u + j8 * 8;
        if (has_ps) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            gv[q] += pg[j8 * 8 + q];
            uv[q] += pu[j8 * 8 + q];
          }
        }
        float act[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) act[q] = gv[q] * sigmoid_f(gv[q]) * uv[q];
        st_bf16x8(H + n, gv);
        st_bf16x8(H + F + n, uv);
        st_bf16x8(A + n, act);
      }
    }
  } else {
    const int N = p.N;
    const int n0 = ti.n_idx * BN;
    const int c_begin = half * (BN / 32 / 2);
    const int c_end = c_begin + BN / 32 / 2;
    // Global inputs of a 32-column chunk (SwiGLU backward: 4 x 16 B of gate and
    // 4 x 16 B of up from H; partial sum: 8 x 16 B of fp32), loaded one chunk
    // ahead so that their latency overlaps the previous chunk's work.
    const bool has_in = valid && (EPI == MOE_EPI_SWIGLU_BWD || p.ps != nullptr);
    auto load_chunk = [&](int c, uint4 *buf) {
      const int nc = n0 + c * 32;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (EPI == MOE_EPI_SWIGLU_BWD) {
          const int n = nc + (q & 3) * 8;
          if (n < N) buf[q] = ld_nc_v4(p.aux + row * p.ld_aux + (q < 4 ? 0 : N) + n);
        } else {
          const int n = nc + q * 4;
          if (n < N) buf[q] = ld_v4_no_l1(p.ps + row * p.ld_ps + n);
        }
      }
    };
    uint4 cur[8], nxt[8];
    if (has_in && n0 + c_begin * 32 < N) load_chunk(c_begin, cur);
#pragma unroll 1
    for (int c = c_begin; c < c_end; ++c) {
      const int nc = n0 + c * 32;
      if (nc >= N) break;
      if (has_in && c + 1 < c_end && nc + 32 < N) load_chunk(c + 1, nxt);
      float v[32];
      tc::tmem_ld32(taddr + c * 32, v);
      if (valid) {
#pragma unroll
        for (int j8 = 0; j8 < 4; ++j8) {
          const int n = nc + j8 * 8;
          if (n >= N) break;
          float *x = v + j8 * 8;
          if (EPI == MOE_EPI_NONE) {
            if (p.ps != nullptr) {
              const float *pv = reinterpret_cast<const float *>(&cur[2 * j8]);
#pragma unroll
              for (int q = 0; q < 8; ++q) x[q] += pv[q];
            }
            if (p.c_f32)
              st_f32x8(static_cast<float *>(p.C) + row * p.ldc + n, x);
            else
              st_bf16x8(static_cast<uint16_t *>(p.C) + row * p.ldc + n, x);
          } else {  // SWIGLU_BWD: x = dAct, aux = H = [gate | up]
            float g[8], u[8], dg[8], du[8];
            bf16x8_to_f32(cur[j8], g);
            bf16x8_to_f32(cur[4 + j8], u);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
              const float sg = sigmoid_f(g[q]);
              dg[q] = x[q] * u[q] * sg * (1.0f + g[q] * (1.0f - sg));
              du[q] = x[q] * g[q] * sg;
            }
            uint16_t *dH = static_cast<uint16_t *>(p.C) + row * p.ldc;
            st_bf16x8(dH + n, dg);
            st_bf16x8(dH + N + n, du);
          }
        }
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) cur[q] = nxt[q];
    }
  }
}

// tgmm epilogue: thread = one output row m of W_e.  `zero`: the expert had no
// rows, so TMEM is not read.
MOE_DEVINL void epilogue_tgmm(const TcParams &p, const TileInfo &ti, uint32_t taddr, int rit,
                              int half, bool zero) {
  const int m = ti.m_idx * BM + rit;
  const bool valid = m < p.M;
  const int n0 = ti.n_idx * BN;
  const int64_t base = (int64_t)ti.e * p.stride_w + (int64_t)m * p.ldc;
#pragma unroll 1
  for (int c = half * (BN / 32 / 2); c < (half + 1) * (BN / 32 / 2); ++c) {
    const int nc = n0 + c * 32;
    if (nc >= p.N) break;
    float v[32];
    if (zero) {
#pragma unroll
      for (int q = 0; q < 32; ++q) v[q] = 0.f;
    } else {
      tc::tmem_ld32(taddr + c * 32, v);
    }
    if (!valid) continue;
#pragma unroll
    for (int j8 = 0; j8 < 4; ++j8) {
      const int n = nc + j8 * 8;
      if (n >= p.N) break;
      float *x = v + j8 * 8;
      if (p.c_f32) {
        float *W = static_cast<float *>(p.C) + base + n;
        if (p.accumulate) {
          float o[8];
          ld_f32x8(W, o);
#pragma unroll
          for (int q = 0; q < 8; ++q) x[q] += o[q];
        }
        st_f32x8(W, x);
      } else {
        st_bf16x8(static_cast<uint16_t *>(p.C) + base + n, x);
      }
    }
  }
}

// ------------------------------------------------------------------ kernel
template <int KIND, bool B_MN, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
gmm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
              const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Book &bk = *reinterpret_cast<Book *>(smem + kStages * STAGE_BYTES);
  volatile int *abort_flag = &bk.abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&bk.full[s], 1);
      tc::mbar_init(&bk.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      tc::mbar_init(&bk.tfull[a], 1);
      tc::mbar_init(&bk.tempty[a], kEpiWarps);
    }
    tc::mbar_init(&bk.drain, 1);
    bk.abort_flag = 0;
    tc::fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch(&tmA);
    tc::tma_prefetch(&tmB);
  }
  for (int i = threadIdx.x; i <= p.E; i += kThreads)
    bk.off[i] = min(max(__ldg(p.offsets + i), 0), p.rows_cap);
  __syncthreads();
  if (warp == 0) {
    // per-expert tile counts and their exclusive scan (warp shuffles)
    int carry = 0;
    for (int c0 = 0; c0 < p.E; c0 += 32) {
      const int e = c0 + lane;
      int tiles = 0;
      if (e < p.E) {
        const int size = max(bk.off[e + 1] - bk.off[e], 0);
        tiles = (KIND == KIND_GMM ? (size + BM - 1) / BM : p.m_tiles) * p.n_tiles;
      }
      int incl = tiles;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (e < p.E) bk.cum[e] = carry + incl - tiles;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      bk.cum[p.E] = carry;
      bk.total_tiles = carry;
    }
    // offsets must be non-decreasing; clamp a bad table to empty groups
    for (int e = lane; e < p.E; e += 32)
      if (bk.off[e + 1] < bk.off[e]) moe_set_status(p.dev_status, MOE_ERR_DEVICE);
  }
  if (warp == 1) {
    tc::tmem_alloc(&bk.tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem = bk.tmem_base;
  const int total = bk.total_tiles;

  uint32_t issued = 0;  // producer: k-blocks issued (ring position)
  if (warp == 0) {
    if (lane == 0) {
      for (int t = blockIdx.x; t < total; t += gridDim.x) {
        const TileInfo ti = decode_tile<KIND>(bk, p, t);
        if (ti.row_end <= ti.row0 && KIND == KIND_GMM) continue;
        bool ok = true;
        for (int kb = 0; kb < ti.kblocks; ++kb) {
          const int s = issued % kStages;
          const uint32_t ph = (issued / kStages) & 1;
          if (!tc::mbar_wait(&bk.empty[s], ph ^ 1, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          uint8_t *sa = smem + s * STAGE_BYTES;
          uint8_t *sb = sa + A_BYTES;
          uint64_t *fb = &bk.full[s];
          tc::mbar_expect_tx(fb, STAGE_BYTES);
          if (KIND == KIND_GMM) {
            tc::tma_load_2d(sa, &tmA, fb, kb * BK, ti.row0);
            if (B_MN) {
              if (EPI == MOE_EPI_SWIGLU_FWD) {
                const int n0 = ti.n_idx * (BN / 2);
                tc::tma_load_3d(sb, &tmB, fb, n0, kb * BK, ti.e);
                tc::tma_load_3d(sb + BOX_BYTES, &tmB, fb, n0 + 64, kb * BK, ti.e);
                tc::tma_load_3d(sb + 2 * BOX_BYTES, &tmB, fb, p.F + n0, kb * BK, ti.e);
                tc::tma_load_3d(sb + 3 * BOX_BYTES, &tmB, fb, p.F + n0 + 64, kb * BK, ti.e);
              } else {
                const int n0 = ti.n_idx * BN;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                  tc::tma_load_3d(sb + i * BOX_BYTES, &tmB, fb, n0 + 64 * i, kb * BK, ti.e);
              }
            } else {
              tc::tma_load_3d(sb, &tmB, fb, kb * BK, ti.n_idx * BN, ti.e);
            }
          } else {
            const int r = ti.row0 + kb * BK;
            const int m0 = ti.m_idx * BM;
            const int n0 = ti.n_idx * BN;
            tc::tma_load_2d(sa, &tmA, fb, m0, r);
            tc::tma_load_2d(sa + BOX_BYTES, &tmA, fb, m0 + 64, r);
#pragma unroll
            for (int i = 0; i < 4; ++i) tc::tma_load_2d(sb + i * BOX_BYTES, &tmB, fb, n0 + 64 * i, r);
          }
          ++issued;
        }
        if (!ok) break;
      }
      // drain: every issued copy has landed before the CTA may exit
      for (uint32_t i = issued > (uint32_t)kStages ? issued - kStages : 0; i < issued; ++i)
        tc::mbar_wait_drain(&bk.full[i % kStages], (i / kStages) & 1, kWaitLimitNs / 4);
    }
  } else if (warp == 1) {
    constexpr uint32_t IDESC = tc::idesc_bf16(BM, BN, KIND == KIND_TGMM, B_MN);
    uint32_t it = 0, acc_it = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      const TileInfo ti = decode_tile<KIND>(bk, p, t);
      if (ti.kblocks == 0 || (KIND == KIND_GMM && ti.row_end <= ti.row0)) continue;
      const uint32_t a = acc_it & 1;
      const uint32_t aph = (acc_it >> 1) & 1;
      if (!tc::mbar_wait(&bk.tempty[a], aph ^ 1, abort_flag, kWaitLimitNs)) break;
      tc::tc_fence_after();
      const uint32_t d_tmem = tmem + a * BN;
      for (int kb = 0; kb < ti.kblocks; ++kb) {
        const int s = it % kStages;
        const uint32_t ph = (it / kStages) & 1;
        if (!tc::mbar_wait(&bk.full[s], ph, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        tc::tc_fence_after();
        uint8_t *sa = smem + s * STAGE_BYTES;
        uint8_t *sb = sa + A_BYTES;
        if (KIND == KIND_TGMM) {
          // rows past the expert's last row belong to the next expert: zero
          // them in both operands (one 128-byte row per K index per box)
          const int valid = ti.row_end - (ti.row0 + kb * BK);
          if (valid < BK) {
            const int nrows = BK - valid;
            for (int i = lane; i < nrows * 6 * 8; i += 32) {
              const int chunk = i & 7;
              const int rr = valid + ((i >> 3) % nrows);
              const int box = (i >> 3) / nrows;
              uint8_t *base = box < 2 ? sa + box * BOX_BYTES : sb + (box - 2) * BOX_BYTES;
              *reinterpret_cast<uint4 *>(base + rr * 128 + chunk * 16) = make_uint4(0, 0, 0, 0);
            }
            tc::fence_proxy_async_smem();
          }
          __syncwarp();
        }
        if (lane == 0) {
          const uint32_t a_base = tc::smem_u32(sa);
          const uint32_t b_base = tc::smem_u32(sb);
#pragma unroll
          for (int kk = 0; kk < BK / UK; ++kk) {
            const uint64_t ad = KIND == KIND_TGMM ? tc::sdesc(a_base + kk * UK * 128, BOX_BYTES, 1024)
                                                  : tc::sdesc(a_base + kk * UK * 2, 16, 1024);
            const uint64_t bd = B_MN ? tc::sdesc(b_base + kk * UK * 128, BOX_BYTES, 1024)
                                     : tc::sdesc(b_base + kk * UK * 2, 16, 1024);
            tc::umma_bf16(d_tmem, ad, bd, IDESC, (kb | kk) != 0);
          }
          tc::umma_commit(&bk.empty[s]);
        }
        __syncwarp();
        ++it;
      }
      if (!ok) break;
      if (lane == 0) tc::umma_commit(&bk.tfull[a]);
      __syncwarp();
      ++acc_it;
    }
    // drain: no MMA of this CTA is in flight once `drain` completes
    if (lane == 0) tc::umma_commit(&bk.drain);
    __syncwarp();
    tc::mbar_wait_drain(&bk.drain, 0, kWaitLimitNs);
  } else {
    const int q = warp & 3;              // TMEM lane quarter this warp may read
    const int half = (warp - 2) >> 2;    // column half of the tile
    const int rit = q * 32 + lane;
    uint32_t acc_it = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x) {
      const TileInfo ti = decode_tile<KIND>(bk, p, t);
      if (KIND == KIND_GMM && ti.row_end <= ti.row0) continue;
      if (KIND == KIND_TGMM && ti.kblocks == 0) {
        if (!p.accumulate) epilogue_tgmm(p, ti, 0, rit, half, true);
        continue;
      }
      epilogue_prefetch<KIND, EPI>(p, ti, rit, half);
      const uint32_t a = acc_it & 1;
      const uint32_t aph = (acc_it >> 1) & 1;
      if (!tc::mbar_wait(&bk.tfull[a], aph, abort_flag, kWaitLimitNs)) break;
      tc::tc_fence_after();
      const uint32_t taddr = tmem + a * BN + (static_cast<uint32_t>(q * 32) << 16);
      if (KIND == KIND_GMM)
        epilogue_gmm<EPI>(p, ti, taddr, rit, half);
      else
        epilogue_tgmm(p, ti, taddr, rit, half, false);
      tc::tc_fence_before();
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&bk.tempty[a]);
      ++acc_it;
    }
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
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
              const uint64_t *strides_bytes, const uint32_t *box) {
  auto fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t d[3], st[2];
  cuuint32_t b[3], es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
  }
  for (int i = 0; i < rank - 1; ++i) st[i] = strides_bytes[i];
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(base), d, st, b, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int KIND, bool B_MN, int EPI>
moe_status_t launch_tc(const CUtensorMap &ma, const CUtensorMap &mb, const TcParams &p,
                       int64_t tiles_upper, cudaStream_t s) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(gmm_tc_kernel<KIND, B_MN, EPI>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
  });
  if (attr_err != cudaSuccess) {
    set_error("grouped GEMM: cannot reserve %d bytes of shared memory: %s", SMEM_BYTES,
              cudaGetErrorString(attr_err));
    return MOE_ERR_CUDA;
  }
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(num_sms(), tiles_upper));
  gmm_tc_kernel<KIND, B_MN, EPI><<<grid, kThreads, SMEM_BYTES, s>>>(ma, mb, p);
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
    const uint32_t box[3] = {BK, BN, 1};
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
  p.n_tiles = a.epilogue == MOE_EPI_SWIGLU_FWD ? (p.F + BN / 2 - 1) / (BN / 2) : (a.N + BN - 1) / BN;
  p.offsets = a.offsets;
  p.C = a.C;
  p.ldc = a.ldc;
  p.c_f32 = a.c_dtype == MOE_DTYPE_F32;
  p.C2 = a.C2;
  p.ldc2 = a.ldc2;
  p.ps = a.ps;
  p.ld_ps = a.ld_ps;
  p.aux = a.aux;
  p.ld_aux = a.ld_aux;
  p.dev_status = a.dev_status;
  const int64_t tiles_upper = ((a.rows_cap + BM - 1) / BM + a.E) * p.n_tiles;
  switch (a.epilogue * 2 + (b_mn ? 1 : 0)) {
    case MOE_EPI_NONE * 2 + 1: return launch_tc<KIND_GMM, true, MOE_EPI_NONE>(ma, mb, p, tiles_upper, s);
    case MOE_EPI_NONE * 2 + 0: return launch_tc<KIND_GMM, false, MOE_EPI_NONE>(ma, mb, p, tiles_upper, s);
    case MOE_EPI_SWIGLU_FWD * 2 + 1:
      return launch_tc<KIND_GMM, true, MOE_EPI_SWIGLU_FWD>(ma, mb, p, tiles_upper, s);
    case MOE_EPI_SWIGLU_BWD * 2 + 1:
      return launch_tc<KIND_GMM, true, MOE_EPI_SWIGLU_BWD>(ma, mb, p, tiles_upper, s);
    case MOE_EPI_SWIGLU_BWD * 2 + 0:
      return launch_tc<KIND_GMM, false, MOE_EPI_SWIGLU_BWD>(ma, mb, p, tiles_upper, s);
    default:
      set_error("moe_gmm: unsupported epilogue / layout");
      return MOE_ERR_UNSUPPORTED;
  }
}

moe_status_t launch_tgmm(const TgmmArgs &a, cudaStream_t s) {
  if (a.E > kMaxE) {
    set_error("moe_tgmm: E=%d > %d", a.E, kMaxE);
    return MOE_ERR_UNSUPPORTED;
  }
  CUtensorMap ma, mb;
  const uint32_t box[2] = {64, BK};
  {
    const uint64_t dims[2] = {(uint64_t)a.M, (uint64_t)a.rows_cap};
    const uint64_t st[1] = {(uint64_t)a.lda * 2};
    if (!make_map(&ma, a.A, 2, dims, st, box)) {
      set_error("moe_tgmm: cannot encode the TMA descriptor of A");
      return MOE_ERR_CUDA;
    }
  }
  {
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
  p.n_tiles = (a.N + BN - 1) / BN;
  p.offsets = a.offsets;
  p.C = a.W;
  p.ldc = a.ldw;
  p.c_f32 = a.w_dtype == MOE_DTYPE_F32;
  p.stride_w = a.stride_w;
  p.accumulate = a.accumulate;
  p.dev_status = a.dev_status;
  const int64_t tiles_upper = (int64_t)a.E * p.m_tiles * p.n_tiles;
  return launch_tc<KIND_TGMM, true, MOE_EPI_NONE>(ma, mb, p, tiles_upper, s);
}

}  // namespace moe
