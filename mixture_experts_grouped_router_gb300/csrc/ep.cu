// Expert-parallel dispatch: the exchange parameters of the ragged
// all-to-all, the local re-sort after it, and the row mover that applies it.
//
// TransformerEngine PR #2912 "[JAX] Add an MoE Block (Layer) that compound
// router, permutation, groupedGEMM and communication": the sequence diagram's
// _dispatch (global permute -> ragged_all_to_all -> local permute) and
// _combine (the reverse), with the helpers compute_ragged_all_to_all_params /
// local_permute_after_a2a / local_unpermute_before_a2a named in its
// description, and the recv_buffer_rows review thread (receive-buffer bound).
//
// Layout.  num_ep shards; shard r owns the El = E / num_ep consecutive experts
// [r*El, (r+1)*El).  Every shard permutes its own tokens over all E experts
// (moe_permute), so its rows for shard r's experts form one contiguous block
// of its permuted buffer.  The group sizes of every shard (all-gathered, on
// the host: the collective needs its split sizes there) fix everything else:
//   send block to r   rows [sum_{e < r*El} gs[me][e], + sum_{le} gs[me][r*El+le])
//   receive buffer    source-major: the block from shard 0, then from 1, ...,
//                     each ordered by local expert
//   local buffer      expert-major: local expert 0's rows from every source
//                     (source order), then local expert 1's, ...
// The local permute moves chunk (source s, local expert le) from its place in
// the receive buffer to its place in the local buffer; the combine side moves
// it back.  Rows keep their order inside a chunk, so a token keeps the
// (expert, token) rank it had in its own shard.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int kChunkThreads = 256;  // 8 warps, one row each

// Row mover: source row i belongs to the chunk c with src_off[c] <= i <
// src_off[c] + len[c] (src_off non-decreasing; found by binary search) and
// goes to destination row dst_off[c] + i - src_off[c].  One warp per row,
// 16-byte loads and stores; rows outside every chunk are not touched.
__global__ void __launch_bounds__(kChunkThreads)
sort_chunks_kernel(const uint16_t *__restrict__ src, int64_t ld_src, uint16_t *__restrict__ dst,
                   int64_t ld_dst, int d, const int64_t *__restrict__ src_off,
                   const int64_t *__restrict__ dst_off, const int64_t *__restrict__ len,
                   int n_chunks, int64_t rows) {
  const int lane = threadIdx.x & 31;
  const int64_t i = (int64_t)blockIdx.x * (kChunkThreads / 32) + (threadIdx.x >> 5);
  if (i >= rows) return;
  int lo = 0, hi = n_chunks - 1;
  while (lo < hi) {  // last chunk starting at or before row i
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(src_off + mid) <= i) lo = mid;
    else hi = mid - 1;
  }
  const int64_t rel = i - __ldg(src_off + lo);
  if (rel < 0 || rel >= __ldg(len + lo)) return;
  const uint4 *s = reinterpret_cast<const uint4 *>(src + i * ld_src);
  uint4 *t = reinterpret_cast<uint4 *>(dst + (__ldg(dst_off + lo) + rel) * ld_dst);
  const int nvec = d >> 3;
  for (int v = lane; v < nvec; v += 32) st_v4(t + v, ld_nc_v4(s + v));
}

}  // namespace

int64_t ep_recv_rows_cap(int T, int num_ep, int E, int k, int align) {
  const int El = E / num_ep;
  return (int64_t)num_ep * ((int64_t)T * std::min(k, El) + (int64_t)El * (align > 1 ? align - 1 : 0));
}

void ep_a2a_params(const int32_t *gs, int num_ep, int E, int shard, int64_t *send_off,
                   int64_t *send_sz, int64_t *out_off, int64_t *recv_off, int64_t *recv_sz) {
  const int El = E / num_ep;
  // rows that shard s sends to shard r: its groups of r's experts
  auto block = [&](int s, int r) {
    int64_t n = 0;
    for (int le = 0; le < El; ++le) n += gs[(int64_t)s * E + (int64_t)r * El + le];
    return n;
  };
  int64_t off = 0;
  for (int r = 0; r < num_ep; ++r) {
    send_off[r] = off;
    send_sz[r] = block(shard, r);
    off += send_sz[r];
    // in r's receive buffer, the blocks of the shards before this one come first
    int64_t o = 0;
    for (int s = 0; s < shard; ++s) o += block(s, r);
    out_off[r] = o;
  }
  off = 0;
  for (int s = 0; s < num_ep; ++s) {
    recv_off[s] = off;
    recv_sz[s] = block(s, shard);
    off += recv_sz[s];
  }
}

void ep_local_layout(const int32_t *gs, int num_ep, int E, int shard, int64_t *fwd_src,
                     int64_t *fwd_dst, int64_t *fwd_len, int64_t *inv_src, int64_t *inv_dst,
                     int64_t *inv_len, int32_t *local_offsets) {
  const int El = E / num_ep;
  const int e0 = shard * El;
  // local group offsets: local expert le gathers its rows from every source
  local_offsets[0] = 0;
  for (int le = 0; le < El; ++le) {
    int64_t n = 0;
    for (int s = 0; s < num_ep; ++s) n += gs[(int64_t)s * E + e0 + le];
    local_offsets[le + 1] = (int32_t)(local_offsets[le] + n);
  }
  // chunk (s, le): in the receive buffer at (rows of earlier sources) + (this
  // source's rows of earlier local experts); in the local buffer at the local
  // group's start + (rows of this expert from earlier sources)
  int64_t src = 0;
  for (int s = 0; s < num_ep; ++s) {
    for (int le = 0; le < El; ++le) {
      int64_t before = 0;
      for (int s2 = 0; s2 < s; ++s2) before += gs[(int64_t)s2 * E + e0 + le];
      const int64_t n = gs[(int64_t)s * E + e0 + le];
      const int c = s * El + le;          // receive-buffer order
      const int ci = le * num_ep + s;     // local-buffer order
      fwd_src[c] = src;
      fwd_dst[c] = local_offsets[le] + before;
      fwd_len[c] = n;
      inv_src[ci] = fwd_dst[c];
      inv_dst[ci] = fwd_src[c];
      inv_len[ci] = n;
      src += n;
    }
  }
}

cudaError_t launch_sort_chunks(const uint16_t *src, int64_t ld_src, uint16_t *dst, int64_t ld_dst,
                               int d, const int64_t *src_off, const int64_t *dst_off,
                               const int64_t *len, int n_chunks, int64_t rows, cudaStream_t s) {
  if (rows <= 0 || n_chunks <= 0) return cudaSuccess;
  const int64_t wpb = kChunkThreads / 32;
  const int64_t blocks = (rows + wpb - 1) / wpb;
  sort_chunks_kernel<<<(unsigned)blocks, kChunkThreads, 0, s>>>(src, ld_src, dst, ld_dst, d,
                                                               src_off, dst_off, len, n_chunks,
                                                               rows);
  return cudaGetLastError();
}

}  // namespace moe
