// Token permutation into per-expert contiguous groups.
//
// TransformerEngine PR #2912 "[JAX] Add an MoE Block (Layer) that compound
// router, permutation, groupedGEMM and communication", review thread on
// _combine_bwd: the flat (token, slot) assignments are ordered by a stable
// argsort on their expert, i.e. by (expert, token).  Here that order is
// produced by a counting sort instead of a comparison sort:
//   1. count:  per block of `tpb` tokens (a multiple of 256 chosen so that
//              there are at most 256 blocks), a shared-memory histogram over E;
//   2. rank:   every block derives the per-expert base of its tokens from the
//              earlier blocks' counts (a warp per expert, lanes over the
//              blocks), the kept counts (capacity), the aligned
//              group sizes and their exclusive scan (warp-shuffle scan), then
//              ranks its tokens 256 at a time with one ballot per expert per
//              warp: rank = base + earlier warps + popc(ballot & lanes below);
//   3. gather: one warp per token reads the row once (16-byte loads) and
//              writes it to each of its k kept positions; padding rows are
//              zero-filled by warps that scan sorted_to_flat 32 rows at a time.
// Capacity (MaxText PR #2319, Tests: token-dropping) keeps rank < C; align
// padding follows the aligned group_sizes of the recv_buffer_rows thread.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kMaxPermBlocks = 256;  // count / rank blocks per call
constexpr int kRankThreads = 256;    // 8 warps, 256 tokens per round
constexpr int kRankWarps = kRankThreads / 32;
constexpr int kMaxE = 256;
constexpr int kMaxK = 16;
constexpr int kGatherThreads = 256;  // 8 warps

// Tokens per count / rank block: a multiple of 256, at most kMaxPermBlocks blocks.
inline int perm_tokens_per_block(int T) {
  const int64_t per = ((int64_t)T + kMaxPermBlocks - 1) / kMaxPermBlocks;
  return (int)std::max<int64_t>(256, (per + 255) / 256 * 256);
}

__global__ void __launch_bounds__(256)
permute_count_kernel(const int32_t *__restrict__ topk_idx, int T, int E, int k, int tpb,
                     int32_t *__restrict__ counts, int32_t *dev_status) {
  __shared__ int32_t hist[kMaxE];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  // thread = token: an expert id out of range, or one the token already
  // listed in an earlier slot, is not counted (the rank kernel drops the same
  // assignments, so every counted assignment gets a row)
  const int t0 = blockIdx.x * tpb;
  const int t1 = (int)min((int64_t)T, (int64_t)t0 + tpb);
  for (int t = t0 + threadIdx.x; t < t1; t += blockDim.x) {
    const int32_t *ids = topk_idx + (int64_t)t * k;
    for (int j = 0; j < k; ++j) {
      const int e = __ldg(ids + j);
      bool ok = e >= 0 && e < E;
      for (int i = 0; i < j && ok; ++i) ok = __ldg(ids + i) != e;
      if (ok)
        atomicAdd(&hist[e], 1);
      else
        moe_set_status(dev_status, MOE_ERR_DEVICE);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) counts[(int64_t)blockIdx.x * E + e] = hist[e];
}

__global__ void __launch_bounds__(kRankThreads)
permute_rank_kernel(const int32_t *__restrict__ topk_idx, int T, int E, int k, int align,
                    int capacity, int tpb, const int32_t *__restrict__ counts, int nb,
                    int64_t rows_cap,
                    int32_t *__restrict__ group_sizes, int32_t *__restrict__ kept_counts,
                    int32_t *__restrict__ group_offsets, int32_t *__restrict__ s2f,
                    int32_t *__restrict__ f2s, int32_t *dev_status) {
  __shared__ int32_t run[kMaxE];       // running rank base per expert
  __shared__ int32_t tot[kMaxE];
  __shared__ int32_t kept[kMaxE];
  __shared__ int32_t off[kMaxE + 1];
  __shared__ uint32_t smask[kRankWarps][kMaxE];
  __shared__ int32_t pre[kRankWarps][kMaxE];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.x;
  grid_dependency_wait();  // the counts of the previous kernel

  // 1. this block's base and the totals, from the count blocks: one warp per
  //    expert, its lanes over the blocks (loads in parallel, shuffle sums)
  for (int e = warp; e < E; e += kRankWarps) {
    int base = 0, all = 0;
    for (int bb = lane; bb < nb; bb += 32) {
      const int c = counts[(int64_t)bb * E + e];
      if (bb < b) base += c;
      all += c;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      base += __shfl_xor_sync(0xffffffffu, base, o);
      all += __shfl_xor_sync(0xffffffffu, all, o);
    }
    if (lane == 0) {
      run[e] = base;
      tot[e] = all;
    }
  }
  __syncthreads();
  // 2. kept counts, aligned sizes and their exclusive scan (one warp)
  if (warp == 0) {
    const int a = align > 1 ? align : 1;
    int carry = 0;
    for (int c0 = 0; c0 < E; c0 += 32) {
      const int e = c0 + lane;
      int kp = 0;
      if (e < E) kp = capacity > 0 ? min(tot[e], capacity) : tot[e];
      const int gs = (kp + a - 1) / a * a;
      int incl = gs;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      if (e < E) {
        kept[e] = kp;
        off[e] = carry + incl - gs;
        if (b == 0) {
          group_sizes[e] = gs;
          kept_counts[e] = kp;
          group_offsets[e] = carry + incl - gs;
        }
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      off[E] = carry;
      if (b == 0) group_offsets[E] = carry;
    }
  }
  __syncthreads();
  // 3. sorted_to_flat = -1 on padding rows (experts spread over blocks) and on rows >= R
  const int R = off[E];
  for (int e = b; e < E; e += nb)
    for (int p = off[e] + kept[e] + tid; p < off[e + 1]; p += kRankThreads) s2f[p] = -1;
  for (int64_t p = R + (int64_t)b * kRankThreads + tid; p < rows_cap;
       p += (int64_t)nb * kRankThreads)
    s2f[p] = -1;

  // 4. rank this block's tokens, 256 per round
  const int tok0 = b * tpb;
  const int tok1 = (int)min((int64_t)T, (int64_t)tok0 + tpb);
  for (int r0 = tok0; r0 < tok1; r0 += kRankThreads) {
    const int t = r0 + tid;
    const bool valid = t < tok1;
    int ex[kMaxK];
#pragma unroll
    for (int j = 0; j < kMaxK; ++j) {
      ex[j] = -1;
      if (j < k && valid) {
        const int e = __ldg(topk_idx + (int64_t)t * k + j);
        ex[j] = (e >= 0 && e < E) ? e : -1;
      }
    }
#pragma unroll
    for (int j = 1; j < kMaxK; ++j) {
#pragma unroll
      for (int i = 0; i < j; ++i)
        if (ex[j] >= 0 && ex[j] == ex[i]) {
          moe_set_status(dev_status, MOE_ERR_DEVICE);
          ex[j] = -1;
        }
    }
    for (int e = 0; e < E; ++e) {
      bool has = false;
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) has |= (ex[j] == e);
      const uint32_t m = __ballot_sync(0xffffffffu, has);
      if (lane == 0) smask[warp][e] = m;
    }
    __syncthreads();
    for (int e = tid; e < E; e += kRankThreads) {
      int running = run[e];
#pragma unroll
      for (int w = 0; w < kRankWarps; ++w) {
        pre[w][e] = running;
        running += __popc(smask[w][e]);
      }
      run[e] = running;
    }
    __syncthreads();
    if (valid) {
      const uint32_t lt = lanemask_lt();
#pragma unroll
      for (int j = 0; j < kMaxK; ++j) {
        if (j < k) {
          const int e = ex[j];
          const int64_t a = (int64_t)t * k + j;
          int pos = -1;
          if (e >= 0) {
            const int r = pre[warp][e] + __popc(smask[warp][e] & lt);
            if (r < kept[e]) {
              pos = off[e] + r;
              s2f[pos] = (int32_t)a;
            }
          }
          f2s[a] = pos;
        }
      }
    }
    __syncthreads();
  }
}

template <int KT>
__global__ void __launch_bounds__(kGatherThreads)
permute_gather_kernel(const uint16_t *__restrict__ x, int64_t ldx,
                      const int32_t *__restrict__ f2s, int T, int k, int d,
                      uint16_t *__restrict__ xs, int64_t ld_xs, const int32_t *__restrict__ s2f,
                      const int32_t *__restrict__ offsets, int E, int64_t rows_cap, int nb_tok,
                      int32_t *dev_status) {
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  const int nvec = d >> 3;
  grid_dependency_wait();  // the layout of the rank kernel
  if ((int)blockIdx.x < nb_tok) {
    const int t = blockIdx.x * (kGatherThreads / 32) + wib;
    if (t >= T) return;
    int pl = lane < k ? __ldg(f2s + (int64_t)t * k + lane) : -1;
    if (pl >= rows_cap) {
      moe_set_status(dev_status, MOE_ERR_DEVICE);
      pl = -1;
    }
    // a token whose assignments were all dropped is not read
    if (!__any_sync(0xffffffffu, pl >= 0)) return;
    int p[KT];
#pragma unroll
    for (int j = 0; j < KT; ++j) p[j] = __shfl_sync(0xffffffffu, pl, j);
    const uint4 *src = reinterpret_cast<const uint4 *>(x + (int64_t)t * ldx);
    int i = lane;
    for (; i + 96 < nvec; i += 128) {
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) v[u] = ld_nc_v4(src + i + 32 * u);
#pragma unroll
      for (int j = 0; j < KT; ++j) {
        if (j < k && p[j] >= 0) {
          uint4 *dst = reinterpret_cast<uint4 *>(xs + (int64_t)p[j] * ld_xs);
#pragma unroll
          for (int u = 0; u < 4; ++u) st_v4(dst + i + 32 * u, v[u]);
        }
      }
    }
    for (; i < nvec; i += 32) {
      const uint4 v = ld_nc_v4(src + i);
#pragma unroll
      for (int j = 0; j < KT; ++j)
        if (j < k && p[j] >= 0) st_v4(reinterpret_cast<uint4 *>(xs + (int64_t)p[j] * ld_xs) + i, v);
    }
  } else {
    // padding rows: each warp checks 32 consecutive rows
    const int64_t w = (int64_t)(blockIdx.x - nb_tok) * (kGatherThreads / 32) + wib;
    const int64_t R = min((int64_t)__ldg(offsets + E), rows_cap);
    const int64_t p0 = w * 32;
    if (p0 >= R) return;
    const int64_t pr = p0 + lane;
    const bool pad = pr < R && __ldg(s2f + pr) < 0;
    uint32_t m = __ballot_sync(0xffffffffu, pad);
    const uint4 z = make_uint4(0, 0, 0, 0);
    while (m) {
      const int bit = __ffs(m) - 1;
      m &= m - 1;
      uint4 *dst = reinterpret_cast<uint4 *>(xs + (p0 + bit) * ld_xs);
      for (int i = lane; i < nvec; i += 32) st_v4(dst + i, z);
    }
  }
}

}  // namespace

size_t permute_workspace_bytes(int T, int E) {
  const int tpb = perm_tokens_per_block(T);
  const int64_t nb = T > 0 ? ((int64_t)T + tpb - 1) / tpb : 1;
  return (size_t)(nb * E * sizeof(int32_t) + 256);
}

cudaError_t launch_permute(const uint16_t *x, int64_t ldx, const int32_t *topk_idx, int T, int d,
                           int E, int k, int align, int capacity, uint16_t *xs, int64_t ld_xs,
                           int64_t rows_cap, int32_t *group_sizes, int32_t *kept,
                           int32_t *offsets, int32_t *s2f, int32_t *f2s, int32_t *counts_ws,
                           int32_t *dev_status, cudaStream_t s) {
  const int tpb = perm_tokens_per_block(T);
  const int nb = T > 0 ? (int)(((int64_t)T + tpb - 1) / tpb) : 1;
  if (T > 0)
    permute_count_kernel<<<nb, 256, 0, s>>>(topk_idx, T, E, k, tpb, counts_ws, dev_status);
  else {
    cudaError_t e = cudaMemsetAsync(counts_ws, 0, sizeof(int32_t) * E, s);
    if (e != cudaSuccess) return e;
  }
  // the rank and gather kernels launch while their predecessor finishes and
  // wait for its results in their first instruction (programmatic dependent
  // launch), which hides the launch gaps of this three-kernel chain
  cudaLaunchAttribute pdl[1];
  pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = s;
  cfg.attrs = pdl;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3(nb);
  cfg.blockDim = dim3(kRankThreads);
  cudaError_t e = cudaLaunchKernelEx(&cfg, permute_rank_kernel, topk_idx, T, E, k, align,
                                     capacity, tpb, (const int32_t *)counts_ws, nb, rows_cap,
                                     group_sizes, kept, offsets, s2f, f2s, dev_status);
  if (e != cudaSuccess) return e;
  const int wpb = kGatherThreads / 32;
  const int nb_tok = (T + wpb - 1) / wpb;
  const int64_t pad_warps = (rows_cap + 31) / 32;
  const int nb_pad = (int)((pad_warps + wpb - 1) / wpb);
  if (nb_tok + nb_pad > 0) {
    cfg.gridDim = dim3(nb_tok + nb_pad);
    cfg.blockDim = dim3(kGatherThreads);
#define MOE_GATHER(KT)                                                                      \
  e = cudaLaunchKernelEx(&cfg, permute_gather_kernel<KT>, x, ldx, (const int32_t *)f2s, T, k, d, \
                         xs, ld_xs, (const int32_t *)s2f, (const int32_t *)offsets, E,          \
                         rows_cap, nb_tok, dev_status)
    if (k <= 1) MOE_GATHER(1);
    else if (k <= 2) MOE_GATHER(2);
    else if (k <= 4) MOE_GATHER(4);
    else if (k <= 8) MOE_GATHER(8);
    else MOE_GATHER(16);
#undef MOE_GATHER
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

}  // namespace moe
