// Host-side launchers shared between the C-ABI layer (api.cu) and the kernel
// translation units.  Arguments are validated by api.cu before these run.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_gb300.h"

namespace moe {

void set_error(const char *fmt, ...);
int num_sms();
uint64_t wait_limit_ns();  // bound of the kernels' waits (moe_set_wait_limit_ns)
int test_stall_loads();    // test hook (moe_test_stall_loads)

// route.cu
cudaError_t launch_route_topk(const float *logits, int64_t ld, int T, int E, int k, int score_fn,
                              int renorm, const float *bias, int num_groups, int topk_group,
                              int32_t *idx, float *w, cudaStream_t s);
size_t aux_loss_workspace_bytes(int T, int E);
cudaError_t launch_aux_loss(const float *logits, int64_t ld, int T, int E, int k, int score_fn,
                            const int32_t *idx, float coeff, int32_t *counts, float *P,
                            float *loss, void *ws, cudaStream_t s);
cudaError_t launch_aux_loss_bwd(const float *logits, int64_t ld, int T, int E, int k,
                                int score_fn, const int32_t *counts, float coeff, float d_loss,
                                float *d_logits, int64_t ld_out, int accumulate, cudaStream_t s);
cudaError_t launch_route_topk_bwd(const float *logits, int64_t ld, const int32_t *idx,
                                  const float *w, const float *dw, int T, int E, int k,
                                  int score_fn, int renorm, float *d_logits, int64_t ld_out,
                                  cudaStream_t s);

// fp8.cu
constexpr int kF8PadRows = 128;  // group padding of column-wise FP8 copies
constexpr int kMaxGroups = 256;
int64_t f8_padded_rows(int64_t rows_cap, int E);
cudaError_t launch_fp8_amax(const uint16_t *x, int64_t ldx, int64_t rows, int cols, int groups,
                            const int32_t *offsets, int E, float *amax, cudaStream_t s);
cudaError_t launch_fp8_quant_act(const uint16_t *x, int64_t ldx, const int32_t *offsets, int E,
                                 int64_t rows_cap, int cols, int fmt, const float *amax,
                                 uint8_t *q, int64_t ldq, uint8_t *qt, int64_t ldqt,
                                 float *scale_inv, cudaStream_t s);
cudaError_t launch_fp8_quant_weights(const uint16_t *w, int E, int K, int N, int fmt,
                                     const float *amax, uint8_t *q, uint8_t *qt,
                                     float *scale_inv, cudaStream_t s);

// transpose.cu
cudaError_t launch_transpose_act(const uint16_t *x, int64_t ldx, const int32_t *offsets, int E,
                                 int64_t rows_cap, int cols, uint16_t *xt, int64_t ldxt,
                                 cudaStream_t s);

// permute.cu
size_t permute_workspace_bytes(int T, int E);
cudaError_t launch_permute(const uint16_t *x, int64_t ldx, const int32_t *topk_idx, int T, int d,
                           int E, int k, int align, int capacity, uint16_t *xs, int64_t ld_xs,
                           int64_t rows_cap, int32_t *group_sizes, int32_t *kept,
                           int32_t *offsets, int32_t *s2f, int32_t *f2s, int32_t *counts_ws,
                           int32_t *dev_status, cudaStream_t s);

// combine.cu
cudaError_t launch_combine(const uint16_t *Y, int64_t ldy, const int32_t *f2s, const float *w,
                           int T, int k, int d, uint16_t *out, int64_t ldo, cudaStream_t s);
cudaError_t launch_unpermute_bwd(const uint16_t *dout, int64_t ld_dout, const uint16_t *Y,
                                 int64_t ldy, const int32_t *f2s, const int32_t *s2f,
                                 const int32_t *offsets, const float *w, int T, int k, int d,
                                 int E, int64_t rows_cap, uint16_t *dY, int64_t ld_dy,
                                 float *dw, cudaStream_t s);

cudaError_t launch_group_colsum(const uint16_t *G, int64_t ldg, const int32_t *offsets, int E,
                               int64_t rows_cap, int N, float *out, int64_t ld_out,
                               cudaStream_t s);

// ep.cu (expert-parallel exchange: host bookkeeping and the row mover)
int64_t ep_recv_rows_cap(int T, int num_ep, int E, int k, int align);
void ep_a2a_params(const int32_t *gs, int num_ep, int E, int shard, int64_t *send_off,
                   int64_t *send_sz, int64_t *out_off, int64_t *recv_off, int64_t *recv_sz);
void ep_local_layout(const int32_t *gs, int num_ep, int E, int shard, int64_t *fwd_src,
                     int64_t *fwd_dst, int64_t *fwd_len, int64_t *inv_src, int64_t *inv_dst,
                     int64_t *inv_len, int32_t *local_offsets);
cudaError_t launch_sort_chunks(const uint16_t *src, int64_t ld_src, uint16_t *dst, int64_t ld_dst,
                               int d, const int64_t *src_off, const int64_t *dst_off,
                               const int64_t *len, int n_chunks, int64_t rows, cudaStream_t s);

// mx.cu (block-scaled 8-bit quantization)
int64_t mx_atom_rows(int64_t rows, int row_map, int E);
cudaError_t launch_mx_quantize(const uint16_t *x, int64_t ldx, int64_t rows, int cols, int fmt,
                               int row_map, const int32_t *offsets, int E, uint8_t *q,
                               int64_t ldq, uint8_t *sf, cudaStream_t s);
cudaError_t launch_mx_quantize_2x(const uint16_t *x, int64_t ldx, int64_t rows, int cols, int fmt,
                                  const int32_t *offsets, int E, uint8_t *q, int64_t ldq,
                                  int q_map, uint8_t *sfq, uint8_t *qt, int64_t ldqt,
                                  int qt_cols, int qt_map, uint8_t *sfqt, cudaStream_t s);

// gmm_sm103.cu
struct GmmArgs {
  const uint16_t *A; int64_t lda;
  const uint16_t *B; int64_t ldb; int64_t stride_b; int trans_b;
  const int32_t *offsets; int E; int64_t rows_cap; int K; int N;
  int epilogue;
  const uint16_t *aux; int64_t ld_aux;
  const float *ps; int64_t ld_ps;
  const uint16_t *bias; int64_t stride_bias;
  void *C; int c_dtype; int64_t ldc;
  uint16_t *C2; int64_t ldc2;
  uint16_t *Ct; int64_t ldct;  // column-wise copy of Act / dH (SwiGLU epilogues), or null
  int32_t *dev_status;
};
moe_status_t launch_gmm(const GmmArgs &a, cudaStream_t s);

struct TgmmArgs {
  const uint16_t *A; int64_t lda;
  const uint16_t *B; int64_t ldb;
  const int32_t *offsets; int E; int64_t rows_cap; int M; int N;
  void *W; int w_dtype; int64_t ldw; int64_t stride_w; int accumulate;
  int32_t *dev_status;
};
moe_status_t launch_tgmm(const TgmmArgs &a, cudaStream_t s);
// the same with A read K-major from its column-wise copy At [M, ldat]
moe_status_t launch_tgmm_kt(const TgmmArgs &a, const uint16_t *At, int64_t ldat, bool b_colwise,
                            cudaStream_t s);

// FP8 (8-bit float codes, K-major operands, fp32 accumulation; the epilogue
// multiplies by the scales' inverses)
struct GmmF8Args {
  const uint8_t *A; int64_t lda; int a_fmt; const float *a_sinv;
  const uint8_t *B; int64_t ldb; int64_t stride_b; int b_fmt; const float *b_sinv;
  const int32_t *offsets; int E; int64_t rows_cap; int K; int N;
  int epilogue;
  const uint16_t *aux; int64_t ld_aux;
  void *C; int c_dtype; int64_t ldc;
  uint16_t *C2; int64_t ldc2;
  float *amax_out;
  int32_t *dev_status;
};
moe_status_t launch_gmm_f8(const GmmF8Args &a, cudaStream_t s);

struct TgmmF8Args {
  const uint8_t *At; int64_t ldat; int a_fmt; const float *a_sinv;
  const uint8_t *Bt; int64_t ldbt; int b_fmt; const float *b_sinv;
  const int32_t *offsets; int E; int64_t rows_cap; int M; int N;
  void *W; int w_dtype; int64_t ldw; int64_t stride_w; int accumulate;
  int32_t *dev_status;
};
moe_status_t launch_tgmm_f8(const TgmmF8Args &a, cudaStream_t s);

// block-scaled (MXFP8): scale atoms beside the codes (mx.cu layout)
struct GmmMxArgs {
  const uint8_t *A; int64_t lda; const uint8_t *sfa; int a_fmt;
  const uint8_t *B; int64_t ldb; int64_t stride_b; const uint8_t *sfb;
  int sfb_by_cols; int b_fmt;
  const int32_t *offsets; int E; int64_t rows_cap; int K; int N;
  int epilogue;
  const uint16_t *aux; int64_t ld_aux;
  void *C; int c_dtype; int64_t ldc;
  uint16_t *C2; int64_t ldc2;
  int32_t *dev_status;
};
moe_status_t launch_gmm_mx(const GmmMxArgs &a, cudaStream_t s);

struct TgmmMxArgs {
  const uint8_t *At; int64_t ldat; const uint8_t *sfa; int a_fmt;
  const uint8_t *Bt; int64_t ldbt; const uint8_t *sfb; int b_fmt;
  const int32_t *offsets; int E; int64_t rows_cap; int M; int N;
  void *W; int w_dtype; int64_t ldw; int64_t stride_w; int accumulate;
  int32_t *dev_status;
};
moe_status_t launch_tgmm_mx(const TgmmMxArgs &a, cudaStream_t s);

}  // namespace moe
