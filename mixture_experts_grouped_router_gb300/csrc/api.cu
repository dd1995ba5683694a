// C ABI of libmoe_gb300.so: argument validation, error reporting and the
// launches.  Every check here runs on the host before anything is enqueued.
#include <stdarg.h>
#include <stdio.h>

#include <algorithm>
#include <atomic>

#include "internal.h"

namespace moe {

static thread_local char g_err[512] = "";

void set_error(const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
}

static std::atomic<uint64_t> g_wait_limit_ns{2000000000ull};
static std::atomic<int> g_stall_loads{0};

uint64_t wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }
int test_stall_loads() { return g_stall_loads.load(std::memory_order_relaxed); }

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
  return n;
}

}  // namespace moe

using moe::set_error;

#define REQUIRE(cond, code, ...)   \
  do {                             \
    if (!(cond)) {                 \
      set_error(__VA_ARGS__);      \
      return (code);               \
    }                              \
  } while (0)

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static moe_status_t cuda_status(cudaError_t e, const char *what) {
  if (e == cudaSuccess) return MOE_OK;
  set_error("%s: %s", what, cudaGetErrorString(e));
  return MOE_ERR_CUDA;
}

extern "C" {

const char *moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported size or alignment";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_DEVICE: return "bad data met on the device";
    default: return "unknown status";
  }
}

const char *moe_last_error(void) { return moe::g_err; }

int moe_version(void) { return 200; }

moe_status_t moe_set_wait_limit_ns(uint64_t limit_ns) {
  set_error("");
  REQUIRE(limit_ns >= 1000000ull && limit_ns <= 600000000000ull, MOE_ERR_INVALID_ARG,
          "moe_set_wait_limit_ns: %llu ns outside [1 ms, 600 s]", (unsigned long long)limit_ns);
  moe::g_wait_limit_ns.store(limit_ns);
  return MOE_OK;
}

uint64_t moe_wait_limit_ns(void) { return moe::wait_limit_ns(); }

void moe_test_stall_loads(int enable) { moe::g_stall_loads.store(enable ? 1 : 0); }

int64_t moe_rows_cap(int T, int E, int k, int align, int capacity) {
  if (T < 0 || E <= 0 || k <= 0) return -1;
  int64_t kept = (int64_t)T * k;
  if (capacity > 0) kept = std::min<int64_t>(kept, (int64_t)E * capacity);
  return kept + (int64_t)E * (align > 1 ? align - 1 : 0);
}

size_t moe_permute_workspace_bytes(int T, int E) {
  if (T < 0 || E <= 0) return 0;
  return moe::permute_workspace_bytes(T, E);
}

moe_status_t moe_route_topk(const float *logits, int64_t ld_logits, int T, int E, int k,
                            int score_fn, int renorm, const float *expert_bias, int num_groups,
                            int topk_group, int32_t *topk_idx, float *topk_w,
                            moe_stream_t stream) {
  set_error("");
  REQUIRE(T >= 0 && E > 0 && k > 0, MOE_ERR_INVALID_ARG, "moe_route_topk: T=%d E=%d k=%d", T, E, k);
  REQUIRE(k <= E, MOE_ERR_INVALID_ARG, "moe_route_topk: k=%d > E=%d", k, E);
  REQUIRE(E <= 256 && k <= 16, MOE_ERR_UNSUPPORTED, "moe_route_topk: needs E <= 256, k <= 16");
  REQUIRE(ld_logits >= E, MOE_ERR_INVALID_ARG, "moe_route_topk: ld_logits < E");
  REQUIRE(score_fn == MOE_SCORE_SOFTMAX || score_fn == MOE_SCORE_SIGMOID, MOE_ERR_INVALID_ARG,
          "moe_route_topk: bad score_fn %d", score_fn);
  REQUIRE(T == 0 || (logits && topk_idx && topk_w), MOE_ERR_INVALID_ARG,
          "moe_route_topk: null pointer");
  REQUIRE(num_groups >= 0 && topk_group >= 0, MOE_ERR_INVALID_ARG,
          "moe_route_topk: num_groups=%d topk_group=%d", num_groups, topk_group);
  if (num_groups > 1) {
    REQUIRE(E % num_groups == 0, MOE_ERR_INVALID_ARG,
            "moe_route_topk: E=%d not a multiple of num_groups=%d", E, num_groups);
    REQUIRE(topk_group >= 1 && topk_group <= num_groups && k % topk_group == 0 &&
                k / topk_group <= E / num_groups,
            MOE_ERR_INVALID_ARG,
            "moe_route_topk: topk_group=%d must divide k=%d, be <= num_groups=%d, and "
            "k/topk_group <= E/num_groups", topk_group, k, num_groups);
  }
  return cuda_status(moe::launch_route_topk(logits, ld_logits, T, E, k, score_fn, renorm,
                                            expert_bias, num_groups, topk_group, topk_idx,
                                            topk_w, (cudaStream_t)stream),
                     "moe_route_topk launch");
}

size_t moe_aux_loss_workspace_bytes(int T, int E) {
  if (T < 0 || E <= 0) return 0;
  return moe::aux_loss_workspace_bytes(T, E);
}

moe_status_t moe_aux_loss(const float *logits, int64_t ld_logits, int T, int E, int k,
                          int score_fn, const int32_t *topk_idx, float coeff, int32_t *counts,
                          float *probs_mean, float *loss, void *workspace,
                          size_t workspace_bytes, moe_stream_t stream) {
  set_error("");
  REQUIRE(T >= 0 && E > 0 && k > 0 && k <= E, MOE_ERR_INVALID_ARG,
          "moe_aux_loss: T=%d E=%d k=%d", T, E, k);
  REQUIRE(E <= 256 && k <= 16, MOE_ERR_UNSUPPORTED, "moe_aux_loss: needs E <= 256, k <= 16");
  REQUIRE(ld_logits >= E, MOE_ERR_INVALID_ARG, "moe_aux_loss: ld_logits < E");
  REQUIRE(score_fn == MOE_SCORE_SOFTMAX || score_fn == MOE_SCORE_SIGMOID, MOE_ERR_INVALID_ARG,
          "moe_aux_loss: bad score_fn %d", score_fn);
  REQUIRE(counts && probs_mean && loss && workspace && (T == 0 || (logits && topk_idx)),
          MOE_ERR_INVALID_ARG, "moe_aux_loss: null pointer");
  REQUIRE(workspace_bytes >= moe::aux_loss_workspace_bytes(T, E), MOE_ERR_INVALID_ARG,
          "moe_aux_loss: workspace of %zu bytes < %zu", workspace_bytes,
          moe::aux_loss_workspace_bytes(T, E));
  REQUIRE((reinterpret_cast<uintptr_t>(workspace) & 3u) == 0, MOE_ERR_INVALID_ARG,
          "moe_aux_loss: workspace must be 4-byte aligned");
  return cuda_status(moe::launch_aux_loss(logits, ld_logits, T, E, k, score_fn, topk_idx, coeff,
                                          counts, probs_mean, loss, workspace,
                                          (cudaStream_t)stream),
                     "moe_aux_loss launch");
}

moe_status_t moe_aux_loss_bwd(const float *logits, int64_t ld_logits, int T, int E, int k,
                              int score_fn, const int32_t *counts, float coeff, float d_loss,
                              float *d_logits, int64_t ld_dlogits, int accumulate,
                              moe_stream_t stream) {
  set_error("");
  REQUIRE(T >= 0 && E > 0 && k > 0 && k <= E, MOE_ERR_INVALID_ARG,
          "moe_aux_loss_bwd: T=%d E=%d k=%d", T, E, k);
  REQUIRE(E <= 256, MOE_ERR_UNSUPPORTED, "moe_aux_loss_bwd: needs E <= 256");
  REQUIRE(ld_logits >= E && ld_dlogits >= E, MOE_ERR_INVALID_ARG,
          "moe_aux_loss_bwd: leading dimension < E");
  REQUIRE(score_fn == MOE_SCORE_SOFTMAX || score_fn == MOE_SCORE_SIGMOID, MOE_ERR_INVALID_ARG,
          "moe_aux_loss_bwd: bad score_fn %d", score_fn);
  REQUIRE(T == 0 || (logits && counts && d_logits), MOE_ERR_INVALID_ARG,
          "moe_aux_loss_bwd: null pointer");
  return cuda_status(moe::launch_aux_loss_bwd(logits, ld_logits, T, E, k, score_fn, counts, coeff,
                                              d_loss, d_logits, ld_dlogits, accumulate,
                                              (cudaStream_t)stream),
                     "moe_aux_loss_bwd launch");
}

moe_status_t moe_route_topk_bwd(const float *logits, int64_t ld_logits, const int32_t *topk_idx,
                                const float *topk_w, const float *d_topk_w, int T, int E, int k,
                                int score_fn, int renorm, float *d_logits, int64_t ld_dlogits,
                                moe_stream_t stream) {
  set_error("");
  REQUIRE(T >= 0 && E > 0 && k > 0 && k <= E, MOE_ERR_INVALID_ARG,
          "moe_route_topk_bwd: T=%d E=%d k=%d", T, E, k);
  REQUIRE(E <= 256 && k <= 16, MOE_ERR_UNSUPPORTED, "moe_route_topk_bwd: needs E <= 256, k <= 16");
  REQUIRE(ld_logits >= E && ld_dlogits >= E, MOE_ERR_INVALID_ARG,
          "moe_route_topk_bwd: leading dimension < E");
  REQUIRE(score_fn == MOE_SCORE_SOFTMAX || score_fn == MOE_SCORE_SIGMOID, MOE_ERR_INVALID_ARG,
          "moe_route_topk_bwd: bad score_fn %d", score_fn);
  REQUIRE(T == 0 || (logits && topk_idx && topk_w && d_topk_w && d_logits), MOE_ERR_INVALID_ARG,
          "moe_route_topk_bwd: null pointer");
  return cuda_status(moe::launch_route_topk_bwd(logits, ld_logits, topk_idx, topk_w, d_topk_w, T,
                                                E, k, score_fn, renorm, d_logits, ld_dlogits,
                                                (cudaStream_t)stream),
                     "moe_route_topk_bwd launch");
}

moe_status_t moe_permute(const uint16_t *x, int64_t ldx, const int32_t *topk_idx, int T, int d,
                         int E, int k, int align, int capacity, uint16_t *x_sorted,
                         int64_t ld_xs, int64_t rows_cap, int32_t *group_sizes,
                         int32_t *kept_counts, int32_t *group_offsets,
                         int32_t *sorted_to_flat, int32_t *flat_to_sorted, void *workspace,
                         size_t workspace_bytes, int32_t *dev_status, moe_stream_t stream) {
  set_error("");
  REQUIRE(T >= 0 && d > 0 && E > 0 && k > 0 && align >= 0, MOE_ERR_INVALID_ARG,
          "moe_permute: T=%d d=%d E=%d k=%d align=%d", T, d, E, k, align);
  REQUIRE(E <= 256 && k <= 16 && k <= E, MOE_ERR_UNSUPPORTED,
          "moe_permute: needs E <= 256 and k <= min(E, 16)");
  REQUIRE(d % 8 == 0 && ldx % 8 == 0 && ld_xs % 8 == 0, MOE_ERR_UNSUPPORTED,
          "moe_permute: d, ldx, ld_xs must be multiples of 8");
  REQUIRE(ldx >= d && ld_xs >= d, MOE_ERR_INVALID_ARG, "moe_permute: leading dimension < d");
  REQUIRE(rows_cap >= moe_rows_cap(T, E, k, align, capacity), MOE_ERR_INVALID_ARG,
          "moe_permute: rows_cap %lld < %lld", (long long)rows_cap,
          (long long)moe_rows_cap(T, E, k, align, capacity));
  REQUIRE(rows_cap < (1ll << 31) && (int64_t)T * k < (1ll << 31), MOE_ERR_UNSUPPORTED,
          "moe_permute: more than 2^31 rows");
  REQUIRE(group_sizes && kept_counts && group_offsets && workspace &&
              (rows_cap == 0 || sorted_to_flat),
          MOE_ERR_INVALID_ARG, "moe_permute: null pointer");
  REQUIRE(T == 0 || (x && topk_idx && flat_to_sorted && x_sorted), MOE_ERR_INVALID_ARG,
          "moe_permute: null pointer");
  REQUIRE(T == 0 || (aligned16(x) && aligned16(x_sorted)), MOE_ERR_UNSUPPORTED,
          "moe_permute: x and x_sorted must be 16-byte aligned");
  REQUIRE(workspace_bytes >= moe::permute_workspace_bytes(T, E), MOE_ERR_INVALID_ARG,
          "moe_permute: workspace of %zu bytes < %zu", workspace_bytes,
          moe::permute_workspace_bytes(T, E));
  return cuda_status(moe::launch_permute(x, ldx, topk_idx, T, d, E, k, align, capacity, x_sorted,
                                         ld_xs, rows_cap, group_sizes, kept_counts, group_offsets,
                                         sorted_to_flat, flat_to_sorted,
                                         static_cast<int32_t *>(workspace), dev_status,
                                         (cudaStream_t)stream),
                     "moe_permute launch");
}

moe_status_t moe_gmm(const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
                     int64_t stride_b, int trans_b, const int32_t *group_offsets, int E,
                     int64_t rows_cap, int K, int N, int epilogue, const uint16_t *aux,
                     int64_t ld_aux, const float *partial_sum, int64_t ld_ps,
                     const uint16_t *bias, int64_t stride_bias, void *C, int c_dtype,
                     int64_t ldc, uint16_t *C2, int64_t ldc2, uint16_t *Ct, int64_t ldct,
                     int32_t *dev_status, moe_stream_t stream) {
  set_error("");
  REQUIRE(E > 0 && rows_cap >= 0 && K > 0 && N > 0, MOE_ERR_INVALID_ARG,
          "moe_gmm: E=%d rows_cap=%lld K=%d N=%d", E, (long long)rows_cap, K, N);
  REQUIRE(Ct == nullptr || epilogue != MOE_EPI_NONE, MOE_ERR_INVALID_ARG,
          "moe_gmm: a column-wise copy (Ct) is written by the SwiGLU epilogues only");
  REQUIRE(Ct == nullptr || (aligned16(Ct) && ldct % 8 == 0 &&
                            ldct >= moe::f8_padded_rows(rows_cap, E)),
          MOE_ERR_INVALID_ARG,
          "moe_gmm: Ct needs a 16-byte aligned base and ldct >= moe_fp8_padded_rows(rows_cap, "
          "E), a multiple of 8");
  REQUIRE(epilogue >= MOE_EPI_NONE && epilogue <= MOE_EPI_SWIGLU_BWD, MOE_ERR_INVALID_ARG,
          "moe_gmm: bad epilogue %d", epilogue);
  REQUIRE(c_dtype == MOE_DTYPE_BF16 || c_dtype == MOE_DTYPE_F32, MOE_ERR_INVALID_ARG,
          "moe_gmm: bad c_dtype");
  REQUIRE(B && group_offsets && (rows_cap == 0 || (A && C)), MOE_ERR_INVALID_ARG,
          "moe_gmm: null pointer");
  REQUIRE(K % 8 == 0 && N % 8 == 0 && lda % 8 == 0 && ldb % 8 == 0 && stride_b % 8 == 0,
          MOE_ERR_UNSUPPORTED, "moe_gmm: K, N, lda, ldb, stride_b must be multiples of 8");
  REQUIRE(E <= 256, MOE_ERR_UNSUPPORTED, "moe_gmm: E=%d > 256", E);
  REQUIRE(aligned16(A) && aligned16(B) && aligned16(C) && aligned16(C2) && aligned16(aux) &&
              aligned16(partial_sum),
          MOE_ERR_UNSUPPORTED, "moe_gmm: A, B, C, C2, aux and partial_sum must be 16-byte aligned");
  REQUIRE(lda >= K, MOE_ERR_INVALID_ARG, "moe_gmm: lda < K");
  REQUIRE(trans_b ? ldb >= K : ldb >= N, MOE_ERR_INVALID_ARG, "moe_gmm: ldb too small");
  REQUIRE(stride_b >= (trans_b ? (int64_t)N * ldb : (int64_t)K * ldb) || E == 1,
          MOE_ERR_INVALID_ARG, "moe_gmm: stride_b overlaps experts");
  int outN = N;
  if (epilogue == MOE_EPI_SWIGLU_FWD) {
    REQUIRE(N % 16 == 0, MOE_ERR_UNSUPPORTED, "moe_gmm: SWIGLU_FWD needs N = 2F with F %% 8 == 0");
    REQUIRE((C2 != nullptr || rows_cap == 0) && ldc2 >= N / 2 && ldc2 % 8 == 0, MOE_ERR_INVALID_ARG,
            "moe_gmm: SWIGLU_FWD needs C2 with ldc2 >= F");
    REQUIRE(c_dtype == MOE_DTYPE_BF16, MOE_ERR_INVALID_ARG, "moe_gmm: SWIGLU_FWD writes bf16 H");
    REQUIRE(!trans_b, MOE_ERR_UNSUPPORTED, "moe_gmm: SWIGLU_FWD needs trans_b = 0");
  }
  if (epilogue == MOE_EPI_SWIGLU_BWD) {
    outN = 2 * N;
    REQUIRE((aux != nullptr || rows_cap == 0) && ld_aux >= 2 * N && ld_aux % 8 == 0,
            MOE_ERR_INVALID_ARG,
            "moe_gmm: SWIGLU_BWD needs aux = H with ld_aux >= 2N");
    REQUIRE(partial_sum == nullptr, MOE_ERR_INVALID_ARG,
            "moe_gmm: SWIGLU_BWD takes no partial sum");
    REQUIRE(c_dtype == MOE_DTYPE_BF16, MOE_ERR_INVALID_ARG, "moe_gmm: SWIGLU_BWD writes bf16 dH");
  }
  REQUIRE(ldc >= outN && ldc % 4 == 0, MOE_ERR_INVALID_ARG, "moe_gmm: ldc too small");
  REQUIRE(partial_sum == nullptr || (ld_ps >= N && ld_ps % 4 == 0), MOE_ERR_INVALID_ARG,
          "moe_gmm: ld_ps < N");
  REQUIRE(partial_sum == nullptr || (const void *)partial_sum != C ||
              (c_dtype == MOE_DTYPE_F32 && ld_ps == ldc),
          MOE_ERR_INVALID_ARG, "moe_gmm: in-place partial sum needs fp32 C with ld_ps == ldc");
  REQUIRE(bias == nullptr || epilogue != MOE_EPI_SWIGLU_BWD, MOE_ERR_INVALID_ARG,
          "moe_gmm: SWIGLU_BWD takes no bias");
  REQUIRE(bias == nullptr || (stride_bias >= N && stride_bias % 8 == 0 && aligned16(bias)) ||
              (bias != nullptr && E == 1 && aligned16(bias)),
          MOE_ERR_INVALID_ARG, "moe_gmm: bias needs stride_bias >= N (multiple of 8) and a "
          "16-byte aligned pointer");
  REQUIRE(rows_cap < (1ll << 31), MOE_ERR_UNSUPPORTED, "moe_gmm: more than 2^31 rows");
  if (rows_cap == 0) return MOE_OK;
  moe::GmmArgs a{A, lda, B, ldb, stride_b, trans_b, group_offsets, E, rows_cap, K, N, epilogue,
                 aux, ld_aux, partial_sum, ld_ps, bias, stride_bias, C, c_dtype, ldc, C2, ldc2,
                 Ct, ldct, dev_status};
  return moe::launch_gmm(a, (cudaStream_t)stream);
}

moe_status_t moe_tgmm(const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
                      const int32_t *group_offsets, int E, int64_t rows_cap, int M, int N,
                      void *W, int w_dtype, int64_t ldw, int64_t stride_w, int accumulate,
                      int32_t *dev_status, moe_stream_t stream) {
  set_error("");
  REQUIRE(E > 0 && rows_cap >= 0 && M > 0 && N > 0, MOE_ERR_INVALID_ARG,
          "moe_tgmm: E=%d rows_cap=%lld M=%d N=%d", E, (long long)rows_cap, M, N);
  REQUIRE(group_offsets && W && (rows_cap == 0 || (A && B)), MOE_ERR_INVALID_ARG,
          "moe_tgmm: null pointer");
  REQUIRE(w_dtype == MOE_DTYPE_BF16 || w_dtype == MOE_DTYPE_F32, MOE_ERR_INVALID_ARG,
          "moe_tgmm: bad w_dtype");
  REQUIRE(!accumulate || w_dtype == MOE_DTYPE_F32, MOE_ERR_INVALID_ARG,
          "moe_tgmm: accumulate needs fp32 W");
  REQUIRE(M % 8 == 0 && N % 8 == 0 && lda % 8 == 0 && ldb % 8 == 0, MOE_ERR_UNSUPPORTED,
          "moe_tgmm: M, N, lda, ldb must be multiples of 8");
  REQUIRE(E <= 256, MOE_ERR_UNSUPPORTED, "moe_tgmm: E=%d > 256", E);
  REQUIRE(aligned16(A) && aligned16(B) && aligned16(W), MOE_ERR_UNSUPPORTED,
          "moe_tgmm: A, B and W must be 16-byte aligned");
  REQUIRE(lda >= M && ldb >= N && ldw >= N && ldw % 4 == 0, MOE_ERR_INVALID_ARG,
          "moe_tgmm: leading dimension too small");
  REQUIRE(stride_w >= (int64_t)M * ldw || E == 1, MOE_ERR_INVALID_ARG,
          "moe_tgmm: stride_w overlaps experts");
  REQUIRE(rows_cap < (1ll << 31), MOE_ERR_UNSUPPORTED, "moe_tgmm: more than 2^31 rows");
  if (rows_cap == 0) {  // no rows at all: every expert is empty
    if (accumulate) return MOE_OK;
    const size_t es = w_dtype == MOE_DTYPE_F32 ? 4 : 2;
    for (int e = 0; e < E; ++e) {
      const cudaError_t ce =
          cudaMemset2DAsync(static_cast<char *>(W) + (size_t)e * stride_w * es, (size_t)ldw * es,
                            0, (size_t)N * es, (size_t)M, (cudaStream_t)stream);
      if (ce != cudaSuccess) return cuda_status(ce, "moe_tgmm zero fill");
    }
    return MOE_OK;
  }
  moe::TgmmArgs a{A, lda, B, ldb, group_offsets, E, rows_cap, M, N, W, w_dtype, ldw, stride_w,
                  accumulate, dev_status};
  return moe::launch_tgmm(a, (cudaStream_t)stream);
}

moe_status_t moe_transpose_act(const uint16_t *x, int64_t ldx, const int32_t *group_offsets,
                               int E, int64_t rows_cap, int cols, uint16_t *xt, int64_t ldxt,
                               moe_stream_t stream) {
  set_error("");
  REQUIRE(E > 0 && E <= moe::kMaxGroups && rows_cap >= 0 && cols > 0, MOE_ERR_INVALID_ARG,
          "moe_transpose_act: E=%d rows_cap=%lld cols=%d", E, (long long)rows_cap, cols);
  REQUIRE(cols % 8 == 0 && ldx % 8 == 0 && ldxt % 8 == 0, MOE_ERR_UNSUPPORTED,
          "moe_transpose_act: cols, ldx, ldxt must be multiples of 8");
  REQUIRE(ldx >= cols && ldxt >= moe::f8_padded_rows(rows_cap, E), MOE_ERR_INVALID_ARG,
          "moe_transpose_act: leading dimension too small");
  REQUIRE(rows_cap < (1ll << 31), MOE_ERR_UNSUPPORTED, "moe_transpose_act: 2^31 rows");
  REQUIRE(group_offsets && xt && (rows_cap == 0 || x), MOE_ERR_INVALID_ARG,
          "moe_transpose_act: null pointer");
  REQUIRE(aligned16(x) && aligned16(xt), MOE_ERR_UNSUPPORTED,
          "moe_transpose_act: x and xt must be 16-byte aligned");
  return cuda_status(moe::launch_transpose_act(x, ldx, group_offsets, E, rows_cap, cols, xt, ldxt,
                                               (cudaStream_t)stream),
                     "moe_transpose_act launch");
}

moe_status_t moe_tgmm_kt(const uint16_t *At, int64_t ldat, const uint16_t *B, int64_t ldb,
                         int b_colwise, const int32_t *group_offsets, int E, int64_t rows_cap, int M, int N,
                         void *W, int w_dtype, int64_t ldw, int64_t stride_w, int accumulate,
                         int32_t *dev_status, moe_stream_t stream) {
  set_error("");
  REQUIRE(E > 0 && rows_cap >= 0 && M > 0 && N > 0, MOE_ERR_INVALID_ARG,
          "moe_tgmm_kt: E=%d rows_cap=%lld M=%d N=%d", E, (long long)rows_cap, M, N);
  REQUIRE(w_dtype == MOE_DTYPE_BF16 || w_dtype == MOE_DTYPE_F32, MOE_ERR_INVALID_ARG,
          "moe_tgmm_kt: bad w_dtype");
  REQUIRE(!accumulate || w_dtype == MOE_DTYPE_F32, MOE_ERR_INVALID_ARG,
          "moe_tgmm_kt: accumulate needs fp32 W");
  const int64_t P = moe::f8_padded_rows(rows_cap, E);
  REQUIRE(P / moe::kF8PadRows < 65536, MOE_ERR_UNSUPPORTED,
          "moe_tgmm_kt: more than 2^16 blocks of 128 rows");
  REQUIRE(ldat >= P && ldat % 8 == 0, MOE_ERR_INVALID_ARG,
          "moe_tgmm_kt: ldat must be >= moe_fp8_padded_rows (%lld) and a multiple of 8",
          (long long)P);
  REQUIRE(N % 8 == 0 && ldb % 8 == 0 && ldw % 8 == 0, MOE_ERR_UNSUPPORTED,
          "moe_tgmm_kt: N, ldb, ldw must be multiples of 8");
  REQUIRE((b_colwise ? ldb >= P : ldb >= N) && ldw >= N, MOE_ERR_INVALID_ARG,
          "moe_tgmm_kt: leading dimension too small");
  REQUIRE(stride_w >= (int64_t)M * ldw || E == 1, MOE_ERR_INVALID_ARG,
          "moe_tgmm_kt: stride_w overlaps experts");
  REQUIRE(group_offsets && W && (rows_cap == 0 || (At && B)), MOE_ERR_INVALID_ARG,
          "moe_tgmm_kt: null pointer");
  REQUIRE(aligned16(At) && aligned16(B) && aligned16(W), MOE_ERR_UNSUPPORTED,
          "moe_tgmm_kt: operands must be 16-byte aligned");
  REQUIRE(rows_cap < (1ll << 31), MOE_ERR_UNSUPPORTED, "moe_tgmm_kt: more than 2^31 rows");
  if (rows_cap == 0) {  // no rows at all: every expert is empty
    if (accumulate) return MOE_OK;
    const size_t es = w_dtype == MOE_DTYPE_F32 ? 4 : 2;
    for (int e = 0; e < E; ++e) {
      const cudaError_t ce =
          cudaMemset2DAsync(static_cast<char *>(W) + (size_t)e * stride_w * es, (size_t)ldw * es,
                            0, (size_t)N * es, (size_t)M, (cudaStream_t)stream);
      if (ce != cudaSuccess) return cuda_status(ce, "moe_tgmm_kt zero fill");
    }
    return MOE_OK;
  }
  moe::TgmmArgs a{nullptr, 0, B, ldb, group_offsets, E, rows_cap, M, N, W, w_dtype, ldw,
                  stride_w, accumulate, dev_status};
  return moe::launch_tgmm_kt(a, At, ldat, b_colwise != 0, (cudaStream_t)stream);
}

moe_status_t moe_group_colsum(const uint16_t *G, int64_t ldg, const int32_t *group_offsets,
                              int E, int64_t rows_cap, int N, float *out, int64_t ld_out,
                              moe_stream_t stream) {
  set_error("");
  REQUIRE(E > 0 && rows_cap >= 0 && N > 0, MOE_ERR_INVALID_ARG,
          "moe_group_colsum: E=%d rows_cap=%lld N=%d", E, (long long)rows_cap, N);
  REQUIRE(E <= 65535, MOE_ERR_UNSUPPORTED, "moe_group_colsum: E > 65535");
  REQUIRE(N % 8 == 0 && ldg % 8 == 0, MOE_ERR_UNSUPPORTED,
          "moe_group_colsum: N and ldg must be multiples of 8");
  REQUIRE(ldg >= N && ld_out >= N, MOE_ERR_INVALID_ARG, "moe_group_colsum: leading dimension < N");
  REQUIRE(group_offsets && out && (rows_cap == 0 || G), MOE_ERR_INVALID_ARG,
          "moe_group_colsum: null pointer");
  REQUIRE(aligned16(G) && aligned16(out) && ld_out % 4 == 0, MOE_ERR_UNSUPPORTED,
          "moe_group_colsum: G and out must be 16-byte aligned, ld_out a multiple of 4");
  REQUIRE(rows_cap < (1ll << 31), MOE_ERR_UNSUPPORTED, "moe_group_colsum: more than 2^31 rows");
  return cuda_status(moe::launch_group_colsum(G, ldg, group_offsets, E, rows_cap, N, out, ld_out,
                                              (cudaStream_t)stream),
                     "moe_group_colsum launch");
}

moe_status_t moe_fp8_amax(const uint16_t *x, int64_t ldx, int64_t rows, int cols, int groups,
                          const int32_t *group_offsets, int E, float *amax,
                          moe_stream_t stream) {
  set_error("");
  REQUIRE(rows >= 0 && cols > 0 && groups >= 1, MOE_ERR_INVALID_ARG,
          "moe_fp8_amax: rows=%lld cols=%d groups=%d", (long long)rows, cols, groups);
  REQUIRE(rows % groups == 0, MOE_ERR_INVALID_ARG, "moe_fp8_amax: rows %% groups != 0");
  REQUIRE(cols % 8 == 0 && ldx % 8 == 0 && ldx >= cols, MOE_ERR_UNSUPPORTED,
          "moe_fp8_amax: cols and ldx must be multiples of 8, ldx >= cols");
  REQUIRE(group_offsets == nullptr || (groups == 1 && E > 0), MOE_ERR_INVALID_ARG,
          "moe_fp8_amax: group_offsets needs groups == 1 and E > 0");
  REQUIRE(amax && (rows == 0 || x), MOE_ERR_INVALID_ARG, "moe_fp8_amax: null pointer");
  REQUIRE(aligned16(x), MOE_ERR_UNSUPPORTED, "moe_fp8_amax: x must be 16-byte aligned");
  return cuda_status(moe::launch_fp8_amax(x, ldx, rows, cols, groups, group_offsets, E, amax,
                                          (cudaStream_t)stream),
                     "moe_fp8_amax launch");
}

int64_t moe_fp8_padded_rows(int64_t rows_cap, int E) {
  if (rows_cap < 0 || E <= 0) return -1;
  return moe::f8_padded_rows(rows_cap, E);
}

moe_status_t moe_fp8_quantize_act(const uint16_t *x, int64_t ldx, const int32_t *group_offsets,
                                  int E, int64_t rows_cap, int cols, int fmt, const float *amax,
                                  uint8_t *q, int64_t ldq, uint8_t *qt, int64_t ldqt,
                                  float *scale_inv, moe_stream_t stream) {
  set_error("");
  REQUIRE(E > 0 && E <= moe::kMaxGroups && rows_cap >= 0 && cols > 0, MOE_ERR_INVALID_ARG,
          "moe_fp8_quantize_act: E=%d rows_cap=%lld cols=%d", E, (long long)rows_cap, cols);
  REQUIRE(fmt == MOE_FP8_E4M3 || fmt == MOE_FP8_E5M2, MOE_ERR_INVALID_ARG,
          "moe_fp8_quantize_act: bad fmt %d", fmt);
  REQUIRE(cols % 16 == 0 && ldx % 8 == 0 && ldq % 16 == 0 && ldqt % 16 == 0, MOE_ERR_UNSUPPORTED,
          "moe_fp8_quantize_act: cols, ldq, ldqt must be multiples of 16, ldx of 8");
  REQUIRE(ldx >= cols && ldq >= cols && ldqt >= moe::f8_padded_rows(rows_cap, E),
          MOE_ERR_INVALID_ARG, "moe_fp8_quantize_act: leading dimension too small");
  REQUIRE(rows_cap < (1ll << 31), MOE_ERR_UNSUPPORTED, "moe_fp8_quantize_act: 2^31 rows");
  REQUIRE(group_offsets && amax && scale_inv && (rows_cap == 0 || (x && q && qt)),
          MOE_ERR_INVALID_ARG, "moe_fp8_quantize_act: null pointer");
  REQUIRE(aligned16(x) && aligned16(q) && aligned16(qt), MOE_ERR_UNSUPPORTED,
          "moe_fp8_quantize_act: x, q, qt must be 16-byte aligned");
  return cuda_status(moe::launch_fp8_quant_act(x, ldx, group_offsets, E, rows_cap, cols, fmt,
                                               amax, q, ldq, qt, ldqt, scale_inv,
                                               (cudaStream_t)stream),
                     "moe_fp8_quantize_act launch");
}

moe_status_t moe_fp8_quantize_weights(const uint16_t *w, int E, int K, int N, int fmt,
                                      const float *amax, uint8_t *q, uint8_t *qt,
                                      float *scale_inv, moe_stream_t stream) {
  set_error("");
  REQUIRE(E > 0 && E <= 65535 && K > 0 && N > 0, MOE_ERR_INVALID_ARG,
          "moe_fp8_quantize_weights: E=%d K=%d N=%d", E, K, N);
  REQUIRE(fmt == MOE_FP8_E4M3 || fmt == MOE_FP8_E5M2, MOE_ERR_INVALID_ARG,
          "moe_fp8_quantize_weights: bad fmt %d", fmt);
  REQUIRE(K % 16 == 0 && N % 16 == 0, MOE_ERR_UNSUPPORTED,
          "moe_fp8_quantize_weights: K and N must be multiples of 16");
  REQUIRE(w && amax && q && qt && scale_inv, MOE_ERR_INVALID_ARG,
          "moe_fp8_quantize_weights: null pointer");
  REQUIRE(aligned16(w) && aligned16(q) && aligned16(qt), MOE_ERR_UNSUPPORTED,
          "moe_fp8_quantize_weights: w, q, qt must be 16-byte aligned");
  return cuda_status(moe::launch_fp8_quant_weights(w, E, K, N, fmt, amax, q, qt, scale_inv,
                                                   (cudaStream_t)stream),
                     "moe_fp8_quantize_weights launch");
}

moe_status_t moe_gmm_fp8(const uint8_t *A, int64_t lda, int a_fmt, const float *a_scale_inv,
                         const uint8_t *B, int64_t ldb, int64_t stride_b, int b_fmt,
                         const float *b_scale_inv, const int32_t *group_offsets, int E,
                         int64_t rows_cap, int K, int N, int epilogue, const uint16_t *aux,
                         int64_t ld_aux, void *C, int c_dtype, int64_t ldc, uint16_t *C2,
                         int64_t ldc2, float *amax_out, int32_t *dev_status,
                         moe_stream_t stream) {
  set_error("");
  REQUIRE(E > 0 && rows_cap >= 0 && K > 0 && N > 0, MOE_ERR_INVALID_ARG,
          "moe_gmm_fp8: E=%d rows_cap=%lld K=%d N=%d", E, (long long)rows_cap, K, N);
  REQUIRE(E <= 256, MOE_ERR_UNSUPPORTED, "moe_gmm_fp8: E=%d > 256", E);
  REQUIRE((a_fmt == MOE_FP8_E4M3 || a_fmt == MOE_FP8_E5M2) &&
              (b_fmt == MOE_FP8_E4M3 || b_fmt == MOE_FP8_E5M2),
          MOE_ERR_INVALID_ARG, "moe_gmm_fp8: bad operand format");
  REQUIRE(epilogue >= MOE_EPI_NONE && epilogue <= MOE_EPI_SWIGLU_BWD, MOE_ERR_INVALID_ARG,
          "moe_gmm_fp8: bad epilogue %d", epilogue);
  REQUIRE(c_dtype == MOE_DTYPE_BF16 || c_dtype == MOE_DTYPE_F32, MOE_ERR_INVALID_ARG,
          "moe_gmm_fp8: bad c_dtype");
  REQUIRE(K % 16 == 0 && lda % 16 == 0 && ldb % 16 == 0 && stride_b % 16 == 0 && N % 8 == 0,
          MOE_ERR_UNSUPPORTED,
          "moe_gmm_fp8: K, lda, ldb, stride_b must be multiples of 16, N of 8");
  REQUIRE(lda >= K && ldb >= K && (E == 1 || stride_b >= (int64_t)N * ldb), MOE_ERR_INVALID_ARG,
          "moe_gmm_fp8: leading dimension or expert stride too small");
  REQUIRE(B && group_offsets && a_scale_inv && b_scale_inv && (rows_cap == 0 || (A && C)),
          MOE_ERR_INVALID_ARG, "moe_gmm_fp8: null pointer");
  REQUIRE(aligned16(A) && aligned16(B) && aligned16(C) && aligned16(C2) && aligned16(aux),
          MOE_ERR_UNSUPPORTED, "moe_gmm_fp8: operands must be 16-byte aligned");
  int outN = N;
  if (epilogue == MOE_EPI_SWIGLU_FWD) {
    REQUIRE(N % 16 == 0, MOE_ERR_UNSUPPORTED, "moe_gmm_fp8: SWIGLU_FWD needs N = 2F, F %% 8 == 0");
    REQUIRE((C2 != nullptr || rows_cap == 0) && ldc2 >= N / 2 && ldc2 % 8 == 0,
            MOE_ERR_INVALID_ARG, "moe_gmm_fp8: SWIGLU_FWD needs C2 with ldc2 >= F");
    REQUIRE(c_dtype == MOE_DTYPE_BF16, MOE_ERR_INVALID_ARG, "moe_gmm_fp8: SWIGLU_FWD writes bf16");
  }
  if (epilogue == MOE_EPI_SWIGLU_BWD) {
    outN = 2 * N;
    REQUIRE((aux != nullptr || rows_cap == 0) && ld_aux >= 2 * N && ld_aux % 8 == 0,
            MOE_ERR_INVALID_ARG, "moe_gmm_fp8: SWIGLU_BWD needs aux = H with ld_aux >= 2N");
    REQUIRE(c_dtype == MOE_DTYPE_BF16, MOE_ERR_INVALID_ARG, "moe_gmm_fp8: SWIGLU_BWD writes bf16");
  }
  REQUIRE(ldc >= (epilogue == MOE_EPI_SWIGLU_FWD ? N : outN) && ldc % 8 == 0, MOE_ERR_INVALID_ARG,
          "moe_gmm_fp8: ldc too small or not a multiple of 8");
  REQUIRE(rows_cap < (1ll << 31), MOE_ERR_UNSUPPORTED, "moe_gmm_fp8: more than 2^31 rows");
  if (rows_cap == 0) {
    if (amax_out != nullptr)
      return cuda_status(cudaMemsetAsync(amax_out, 0, sizeof(float), (cudaStream_t)stream),
                         "moe_gmm_fp8 amax reset");
    return MOE_OK;
  }
  moe::GmmF8Args a{A, lda, a_fmt, a_scale_inv, B, ldb, stride_b, b_fmt, b_scale_inv,
                   group_offsets, E, rows_cap, K, N, epilogue, aux, ld_aux, C, c_dtype, ldc,
                   C2, ldc2, amax_out, dev_status};
  return moe::launch_gmm_f8(a, (cudaStream_t)stream);
}

moe_status_t moe_tgmm_fp8(const uint8_t *At, int64_t ldat, int a_fmt, const float *a_scale_inv,
                          const uint8_t *Bt, int64_t ldbt, int b_fmt, const float *b_scale_inv,
                          const int32_t *group_offsets, int E, int64_t rows_cap, int M, int N,
                          void *W, int w_dtype, int64_t ldw, int64_t stride_w, int accumulate,
                          int32_t *dev_status, moe_stream_t stream) {
  set_error("");
  REQUIRE(E > 0 && rows_cap >= 0 && M > 0 && N > 0, MOE_ERR_INVALID_ARG,
          "moe_tgmm_fp8: E=%d rows_cap=%lld M=%d N=%d", E, (long long)rows_cap, M, N);
  REQUIRE(E <= 256, MOE_ERR_UNSUPPORTED, "moe_tgmm_fp8: E=%d > 256", E);
  REQUIRE((a_fmt == MOE_FP8_E4M3 || a_fmt == MOE_FP8_E5M2) &&
              (b_fmt == MOE_FP8_E4M3 || b_fmt == MOE_FP8_E5M2),
          MOE_ERR_INVALID_ARG, "moe_tgmm_fp8: bad operand format");
  REQUIRE(w_dtype == MOE_DTYPE_BF16 || w_dtype == MOE_DTYPE_F32, MOE_ERR_INVALID_ARG,
          "moe_tgmm_fp8: bad w_dtype");
  REQUIRE(!accumulate || w_dtype == MOE_DTYPE_F32, MOE_ERR_INVALID_ARG,
          "moe_tgmm_fp8: accumulate needs fp32 W");
  const int64_t P = moe::f8_padded_rows(rows_cap, E);
  REQUIRE(P / moe::kF8PadRows < 65536, MOE_ERR_UNSUPPORTED,
          "moe_tgmm_fp8: more than 2^16 blocks of 128 rows");
  REQUIRE(ldat >= P && ldbt >= P && ldat % 16 == 0 && ldbt % 16 == 0, MOE_ERR_INVALID_ARG,
          "moe_tgmm_fp8: ldat, ldbt must be >= moe_fp8_padded_rows (%lld) and multiples of 16",
          (long long)P);
  REQUIRE(N % 8 == 0 && ldw >= N && ldw % 8 == 0, MOE_ERR_UNSUPPORTED,
          "moe_tgmm_fp8: N and ldw must be multiples of 8, ldw >= N");
  REQUIRE(stride_w >= (int64_t)M * ldw || E == 1, MOE_ERR_INVALID_ARG,
          "moe_tgmm_fp8: stride_w overlaps experts");
  REQUIRE(At && Bt && a_scale_inv && b_scale_inv && group_offsets && W, MOE_ERR_INVALID_ARG,
          "moe_tgmm_fp8: null pointer");
  REQUIRE(aligned16(At) && aligned16(Bt) && aligned16(W), MOE_ERR_UNSUPPORTED,
          "moe_tgmm_fp8: operands must be 16-byte aligned");
  moe::TgmmF8Args a{At, ldat, a_fmt, a_scale_inv, Bt, ldbt, b_fmt, b_scale_inv, group_offsets, E,
                    rows_cap, M, N, W, w_dtype, ldw, stride_w, accumulate, dev_status};
  return moe::launch_tgmm_f8(a, (cudaStream_t)stream);
}

size_t moe_mx_scale_bytes(int64_t rows, int cols, int row_map, int E) {
  if (rows < 0 || cols <= 0 || cols % 128 != 0 || row_map < MOE_MX_ROWS_PLAIN ||
      row_map > MOE_MX_ROWS_TILES ||
      ((row_map == MOE_MX_ROWS_GROUPED || row_map == MOE_MX_ROWS_TILES) && E <= 0) ||
      (row_map == MOE_MX_ROWS_TILES && rows % E != 0) ||
      (row_map == MOE_MX_ROWS_SWIGLU && rows % 2 != 0))
    return 0;
  return (size_t)moe::mx_atom_rows(rows, row_map, E) * (size_t)(cols / 128) * 512u;
}

moe_status_t moe_mx_quantize(const uint16_t *x, int64_t ldx, int64_t rows, int cols, int fmt,
                             int row_map, const int32_t *group_offsets, int E, uint8_t *q,
                             int64_t ldq, uint8_t *sf, size_t sf_bytes, moe_stream_t stream) {
  set_error("");
  REQUIRE(rows >= 0 && cols > 0, MOE_ERR_INVALID_ARG, "moe_mx_quantize: rows=%lld cols=%d",
          (long long)rows, cols);
  REQUIRE(fmt == MOE_FP8_E4M3 || fmt == MOE_FP8_E5M2, MOE_ERR_INVALID_ARG,
          "moe_mx_quantize: bad format %d", fmt);
  REQUIRE(row_map >= MOE_MX_ROWS_PLAIN && row_map <= MOE_MX_ROWS_TILES, MOE_ERR_INVALID_ARG,
          "moe_mx_quantize: bad row_map %d", row_map);
  REQUIRE(cols % 128 == 0 && ldx % 8 == 0 && ldq % 16 == 0, MOE_ERR_UNSUPPORTED,
          "moe_mx_quantize: cols must be a multiple of 128, ldx of 8, ldq of 16");
  REQUIRE(ldx >= cols && ldq >= cols, MOE_ERR_INVALID_ARG, "moe_mx_quantize: ld < cols");
  REQUIRE(rows < (1ll << 31), MOE_ERR_UNSUPPORTED, "moe_mx_quantize: more than 2^31 rows");
  if (row_map == MOE_MX_ROWS_GROUPED)
    REQUIRE(group_offsets != nullptr && E > 0 && E <= 256, MOE_ERR_INVALID_ARG,
            "moe_mx_quantize: GROUPED needs group_offsets and 0 < E <= 256");
  if (row_map == MOE_MX_ROWS_SWIGLU)
    REQUIRE(rows % 64 == 0, MOE_ERR_UNSUPPORTED,
            "moe_mx_quantize: SWIGLU needs 2F rows with F a multiple of 32");
  if (row_map == MOE_MX_ROWS_TILES)
    REQUIRE(E > 0 && rows % E == 0, MOE_ERR_INVALID_ARG,
            "moe_mx_quantize: TILES needs E > 0 groups of equal rows");
  if (rows == 0) return MOE_OK;
  REQUIRE(x && q && sf, MOE_ERR_INVALID_ARG, "moe_mx_quantize: null pointer");
  REQUIRE(aligned16(x) && aligned16(q), MOE_ERR_UNSUPPORTED,
          "moe_mx_quantize: x and q must be 16-byte aligned");
  REQUIRE(sf_bytes >= moe_mx_scale_bytes(rows, cols, row_map, E), MOE_ERR_INVALID_ARG,
          "moe_mx_quantize: sf of %zu bytes < %zu", sf_bytes,
          moe_mx_scale_bytes(rows, cols, row_map, E));
  return cuda_status(moe::launch_mx_quantize(x, ldx, rows, cols, fmt, row_map, group_offsets, E,
                                             q, ldq, sf, (cudaStream_t)stream),
                     "moe_mx_quantize launch");
}

moe_status_t moe_mx_quantize_2x(const uint16_t *x, int64_t ldx, int64_t rows, int cols, int fmt,
                                const int32_t *group_offsets, int E, uint8_t *q, int64_t ldq,
                                int q_map, uint8_t *sfq, size_t sfq_bytes, uint8_t *qt,
                                int64_t ldqt, int qt_cols, int qt_map, uint8_t *sfqt,
                                size_t sfqt_bytes, moe_stream_t stream) {
  set_error("");
  REQUIRE(rows >= 0 && cols > 0 && E > 0 && E <= 256, MOE_ERR_INVALID_ARG,
          "moe_mx_quantize_2x: rows=%lld cols=%d E=%d", (long long)rows, cols, E);
  REQUIRE(fmt == MOE_FP8_E4M3 || fmt == MOE_FP8_E5M2, MOE_ERR_INVALID_ARG,
          "moe_mx_quantize_2x: bad format %d", fmt);
  REQUIRE(q_map == MOE_MX_ROWS_GROUPED || q_map == MOE_MX_ROWS_TILES, MOE_ERR_INVALID_ARG,
          "moe_mx_quantize_2x: q_map must be GROUPED or TILES");
  REQUIRE(qt_map == MOE_MX_ROWS_PLAIN || qt_map == MOE_MX_ROWS_TILES ||
              qt_map == MOE_MX_ROWS_SWIGLU,
          MOE_ERR_INVALID_ARG, "moe_mx_quantize_2x: qt_map must be PLAIN, TILES or SWIGLU");
  REQUIRE(cols % 128 == 0 && ldx % 8 == 0 && ldq % 16 == 0 && ldqt % 16 == 0 &&
              qt_cols % 128 == 0,
          MOE_ERR_UNSUPPORTED,
          "moe_mx_quantize_2x: cols and qt_cols multiples of 128, ldx of 8, ldq and ldqt of 16");
  REQUIRE(ldx >= cols && ldq >= cols && ldqt >= qt_cols, MOE_ERR_INVALID_ARG,
          "moe_mx_quantize_2x: leading dimension too small");
  REQUIRE(q_map != MOE_MX_ROWS_TILES || rows % E == 0, MOE_ERR_INVALID_ARG,
          "moe_mx_quantize_2x: TILES needs E equal groups");
  REQUIRE(qt_map != MOE_MX_ROWS_SWIGLU || cols % 64 == 0, MOE_ERR_UNSUPPORTED,
          "moe_mx_quantize_2x: SWIGLU needs 2F columns with F a multiple of 32");
  REQUIRE(rows < (1ll << 31), MOE_ERR_UNSUPPORTED, "moe_mx_quantize_2x: more than 2^31 rows");
  if (rows == 0 || (q == nullptr && qt == nullptr)) return MOE_OK;
  REQUIRE(x && group_offsets && (q == nullptr || sfq) && (qt == nullptr || sfqt),
          MOE_ERR_INVALID_ARG, "moe_mx_quantize_2x: null pointer");
  REQUIRE(aligned16(x) && aligned16(q) && aligned16(qt), MOE_ERR_UNSUPPORTED,
          "moe_mx_quantize_2x: x, q and qt must be 16-byte aligned");
  REQUIRE(q == nullptr || sfq_bytes >= moe_mx_scale_bytes(rows, cols, q_map, E),
          MOE_ERR_INVALID_ARG, "moe_mx_quantize_2x: sfq of %zu bytes < %zu", sfq_bytes,
          moe_mx_scale_bytes(rows, cols, q_map, E));
  REQUIRE(qt == nullptr || sfqt_bytes >= moe_mx_scale_bytes(cols, qt_cols, qt_map, 1),
          MOE_ERR_INVALID_ARG, "moe_mx_quantize_2x: sfqt of %zu bytes < %zu", sfqt_bytes,
          moe_mx_scale_bytes(cols, qt_cols, qt_map, 1));
  return cuda_status(moe::launch_mx_quantize_2x(x, ldx, rows, cols, fmt, group_offsets, E, q, ldq,
                                                q_map, sfq, qt, ldqt, qt_cols, qt_map, sfqt,
                                                (cudaStream_t)stream),
                     "moe_mx_quantize_2x launch");
}

moe_status_t moe_gmm_mx(const uint8_t *A, int64_t lda, const uint8_t *sfa, int a_fmt,
                        const uint8_t *B, int64_t ldb, int64_t stride_b, const uint8_t *sfb,
                        int sfb_by_cols, int b_fmt,
                        const int32_t *group_offsets, int E, int64_t rows_cap, int K, int N,
                        int epilogue, const uint16_t *aux, int64_t ld_aux, void *C, int c_dtype,
                        int64_t ldc, uint16_t *C2, int64_t ldc2, int32_t *dev_status,
                        moe_stream_t stream) {
  set_error("");
  REQUIRE(E > 0 && rows_cap >= 0 && K > 0 && N > 0, MOE_ERR_INVALID_ARG,
          "moe_gmm_mx: E=%d rows_cap=%lld K=%d N=%d", E, (long long)rows_cap, K, N);
  REQUIRE(E <= 256, MOE_ERR_UNSUPPORTED, "moe_gmm_mx: E=%d > 256", E);
  REQUIRE((a_fmt == MOE_FP8_E4M3 || a_fmt == MOE_FP8_E5M2) &&
              (b_fmt == MOE_FP8_E4M3 || b_fmt == MOE_FP8_E5M2),
          MOE_ERR_INVALID_ARG, "moe_gmm_mx: bad operand format");
  REQUIRE(epilogue >= MOE_EPI_NONE && epilogue <= MOE_EPI_SWIGLU_BWD, MOE_ERR_INVALID_ARG,
          "moe_gmm_mx: bad epilogue %d", epilogue);
  REQUIRE(c_dtype == MOE_DTYPE_BF16 || c_dtype == MOE_DTYPE_F32, MOE_ERR_INVALID_ARG,
          "moe_gmm_mx: bad c_dtype");
  REQUIRE(K % 128 == 0 && N % 32 == 0 && lda % 16 == 0 && ldb % 16 == 0 && stride_b % 16 == 0,
          MOE_ERR_UNSUPPORTED,
          "moe_gmm_mx: K must be a multiple of 128, N of 32, lda, ldb, stride_b of 16");
  REQUIRE(lda >= K && ldb >= K, MOE_ERR_INVALID_ARG, "moe_gmm_mx: lda, ldb < K");
  REQUIRE(sfb_by_cols == 0 || sfb_by_cols == 1, MOE_ERR_INVALID_ARG,
          "moe_gmm_mx: sfb_by_cols must be 0 or 1");
  REQUIRE(sfb_by_cols ? (stride_b == K && ldb >= (int64_t)E * K)
                      : (stride_b >= (int64_t)N * ldb || E == 1),
          MOE_ERR_INVALID_ARG,
          "moe_gmm_mx: B must be [E*N, K] (sfb_by_cols 0) or [N, E*K] with stride_b = K (1)");
  REQUIRE(epilogue != MOE_EPI_SWIGLU_FWD || (sfb_by_cols && N % 64 == 0), MOE_ERR_UNSUPPORTED,
          "moe_gmm_mx: SWIGLU_FWD needs the [2F, E*K] weight (sfb_by_cols 1), F % 32 == 0");
  int outN = N;
  if (epilogue == MOE_EPI_SWIGLU_FWD) {
    REQUIRE((C2 != nullptr || rows_cap == 0) && ldc2 >= N / 2 && ldc2 % 8 == 0,
            MOE_ERR_INVALID_ARG, "moe_gmm_mx: SWIGLU_FWD needs C2 with ldc2 >= F");
    REQUIRE(c_dtype == MOE_DTYPE_BF16, MOE_ERR_INVALID_ARG, "moe_gmm_mx: SWIGLU_FWD writes bf16");
  }
  if (epilogue == MOE_EPI_SWIGLU_BWD) {
    outN = 2 * N;
    REQUIRE((aux != nullptr || rows_cap == 0) && ld_aux >= 2 * N && ld_aux % 8 == 0,
            MOE_ERR_INVALID_ARG, "moe_gmm_mx: SWIGLU_BWD needs aux = H with ld_aux >= 2N");
    REQUIRE(c_dtype == MOE_DTYPE_BF16, MOE_ERR_INVALID_ARG, "moe_gmm_mx: SWIGLU_BWD writes bf16");
  }
  REQUIRE(ldc >= outN && ldc % 4 == 0, MOE_ERR_INVALID_ARG, "moe_gmm_mx: ldc too small");
  REQUIRE(rows_cap < (1ll << 31), MOE_ERR_UNSUPPORTED, "moe_gmm_mx: more than 2^31 rows");
  if (rows_cap == 0) return MOE_OK;
  REQUIRE(A && sfa && B && sfb && group_offsets && C, MOE_ERR_INVALID_ARG,
          "moe_gmm_mx: null pointer");
  REQUIRE(aligned16(A) && aligned16(B) && aligned16(C) && aligned16(C2) && aligned16(aux) &&
              aligned16(sfa) && aligned16(sfb),
          MOE_ERR_UNSUPPORTED, "moe_gmm_mx: operands must be 16-byte aligned");
  moe::GmmMxArgs a{A, lda, sfa, a_fmt, B, ldb, stride_b, sfb, sfb_by_cols, b_fmt,
                   group_offsets, E, rows_cap, K, N, epilogue, aux, ld_aux, C, c_dtype, ldc, C2,
                   ldc2, dev_status};
  return moe::launch_gmm_mx(a, (cudaStream_t)stream);
}

moe_status_t moe_tgmm_mx(const uint8_t *At, int64_t ldat, const uint8_t *sfa, int a_fmt,
                         const uint8_t *Bt, int64_t ldbt, const uint8_t *sfb, int b_fmt,
                         const int32_t *group_offsets, int E, int64_t rows_cap, int M, int N,
                         void *W, int w_dtype, int64_t ldw, int64_t stride_w, int accumulate,
                         int32_t *dev_status, moe_stream_t stream) {
  set_error("");
  REQUIRE(E > 0 && rows_cap >= 0 && M > 0 && N > 0, MOE_ERR_INVALID_ARG,
          "moe_tgmm_mx: E=%d rows_cap=%lld M=%d N=%d", E, (long long)rows_cap, M, N);
  REQUIRE(E <= 256, MOE_ERR_UNSUPPORTED, "moe_tgmm_mx: E=%d > 256", E);
  REQUIRE((a_fmt == MOE_FP8_E4M3 || a_fmt == MOE_FP8_E5M2) &&
              (b_fmt == MOE_FP8_E4M3 || b_fmt == MOE_FP8_E5M2),
          MOE_ERR_INVALID_ARG, "moe_tgmm_mx: bad operand format");
  REQUIRE(w_dtype == MOE_DTYPE_BF16 || w_dtype == MOE_DTYPE_F32, MOE_ERR_INVALID_ARG,
          "moe_tgmm_mx: bad w_dtype");
  REQUIRE(!accumulate || w_dtype == MOE_DTYPE_F32, MOE_ERR_INVALID_ARG,
          "moe_tgmm_mx: accumulate needs fp32 W");
  const int64_t P = moe::f8_padded_rows(rows_cap, E);
  REQUIRE(P / moe::kF8PadRows < 65536, MOE_ERR_UNSUPPORTED,
          "moe_tgmm_mx: more than 2^16 blocks of 128 rows");
  REQUIRE(ldat >= P && ldbt >= P && ldat % 16 == 0 && ldbt % 16 == 0, MOE_ERR_INVALID_ARG,
          "moe_tgmm_mx: ldat, ldbt must be >= moe_fp8_padded_rows (%lld) and multiples of 16",
          (long long)P);
  REQUIRE(M % 128 == 0 && N % 32 == 0 && ldw >= N && ldw % 8 == 0, MOE_ERR_UNSUPPORTED,
          "moe_tgmm_mx: M must be a multiple of 128, N of 32, ldw >= N a multiple of 8");
  REQUIRE(stride_w >= (int64_t)M * ldw || E == 1, MOE_ERR_INVALID_ARG,
          "moe_tgmm_mx: stride_w overlaps experts");
  REQUIRE(At && sfa && Bt && sfb && group_offsets && W, MOE_ERR_INVALID_ARG,
          "moe_tgmm_mx: null pointer");
  REQUIRE(aligned16(At) && aligned16(Bt) && aligned16(W) && aligned16(sfa) && aligned16(sfb),
          MOE_ERR_UNSUPPORTED, "moe_tgmm_mx: operands must be 16-byte aligned");
  moe::TgmmMxArgs a{At, ldat, sfa, a_fmt, Bt, ldbt, sfb, b_fmt, group_offsets, E, rows_cap, M, N,
                    W, w_dtype, ldw, stride_w, accumulate, dev_status};
  return moe::launch_tgmm_mx(a, (cudaStream_t)stream);
}

int64_t moe_ep_recv_rows_cap(int T, int num_ep, int E, int k, int align) {
  if (T < 0 || num_ep <= 0 || E <= 0 || k <= 0 || E % num_ep != 0) return -1;
  return moe::ep_recv_rows_cap(T, num_ep, E, k, align);
}

static moe_status_t ep_check(const char *what, const int32_t *group_sizes, int num_ep, int E,
                             int shard) {
  REQUIRE(group_sizes != nullptr, MOE_ERR_INVALID_ARG, "%s: null group_sizes", what);
  REQUIRE(num_ep >= 1 && num_ep <= 1024 && E >= 1 && E <= 65536 && E % num_ep == 0,
          MOE_ERR_INVALID_ARG, "%s: E=%d must be a multiple of num_ep=%d (<= 1024)", what, E,
          num_ep);
  REQUIRE(shard >= 0 && shard < num_ep, MOE_ERR_INVALID_ARG, "%s: shard %d of %d", what, shard,
          num_ep);
  for (int64_t i = 0; i < (int64_t)num_ep * E; ++i)
    REQUIRE(group_sizes[i] >= 0, MOE_ERR_INVALID_ARG, "%s: group_sizes[%lld] = %d < 0", what,
            (long long)i, group_sizes[i]);
  return MOE_OK;
}

moe_status_t moe_ep_a2a_params(const int32_t *group_sizes, int num_ep, int E, int shard,
                               int64_t *send_off, int64_t *send_sz, int64_t *out_off,
                               int64_t *recv_off, int64_t *recv_sz) {
  set_error("");
  const moe_status_t st = ep_check("moe_ep_a2a_params", group_sizes, num_ep, E, shard);
  if (st != MOE_OK) return st;
  REQUIRE(send_off && send_sz && out_off && recv_off && recv_sz, MOE_ERR_INVALID_ARG,
          "moe_ep_a2a_params: null output");
  moe::ep_a2a_params(group_sizes, num_ep, E, shard, send_off, send_sz, out_off, recv_off,
                     recv_sz);
  return MOE_OK;
}

moe_status_t moe_ep_local_layout(const int32_t *group_sizes, int num_ep, int E, int shard,
                                 int64_t *fwd_src, int64_t *fwd_dst, int64_t *fwd_len,
                                 int64_t *inv_src, int64_t *inv_dst, int64_t *inv_len,
                                 int32_t *local_offsets) {
  set_error("");
  const moe_status_t st = ep_check("moe_ep_local_layout", group_sizes, num_ep, E, shard);
  if (st != MOE_OK) return st;
  REQUIRE(fwd_src && fwd_dst && fwd_len && inv_src && inv_dst && inv_len && local_offsets,
          MOE_ERR_INVALID_ARG, "moe_ep_local_layout: null output");
  const int El = E / num_ep;
  int64_t rows = 0;
  for (int s = 0; s < num_ep; ++s)
    for (int le = 0; le < El; ++le) rows += group_sizes[(int64_t)s * E + (int64_t)shard * El + le];
  REQUIRE(rows < (1ll << 31), MOE_ERR_UNSUPPORTED, "moe_ep_local_layout: %lld rows >= 2^31",
          (long long)rows);
  moe::ep_local_layout(group_sizes, num_ep, E, shard, fwd_src, fwd_dst, fwd_len, inv_src, inv_dst,
                       inv_len, local_offsets);
  return MOE_OK;
}

moe_status_t moe_sort_chunks(const uint16_t *src, int64_t ld_src, uint16_t *dst, int64_t ld_dst,
                             int d, const int64_t *src_off, const int64_t *dst_off,
                             const int64_t *len, int n_chunks, int64_t rows,
                             moe_stream_t stream) {
  set_error("");
  REQUIRE(d > 0 && n_chunks >= 0 && rows >= 0, MOE_ERR_INVALID_ARG,
          "moe_sort_chunks: d=%d n_chunks=%d rows=%lld", d, n_chunks, (long long)rows);
  REQUIRE(ld_src >= d && ld_dst >= d, MOE_ERR_INVALID_ARG, "moe_sort_chunks: ld < d");
  REQUIRE(d % 8 == 0 && ld_src % 8 == 0 && ld_dst % 8 == 0, MOE_ERR_UNSUPPORTED,
          "moe_sort_chunks: d, ld_src, ld_dst must be multiples of 8");
  if (rows == 0 || n_chunks == 0) return MOE_OK;
  REQUIRE(src && dst && src_off && dst_off && len, MOE_ERR_INVALID_ARG,
          "moe_sort_chunks: null pointer");
  REQUIRE(aligned16(src) && aligned16(dst), MOE_ERR_UNSUPPORTED,
          "moe_sort_chunks: src and dst must be 16-byte aligned");
  return cuda_status(moe::launch_sort_chunks(src, ld_src, dst, ld_dst, d, src_off, dst_off, len,
                                             n_chunks, rows, (cudaStream_t)stream),
                     "moe_sort_chunks launch");
}

moe_status_t moe_combine(const uint16_t *Y, int64_t ldy, const int32_t *flat_to_sorted,
                         const float *topk_w, int T, int k, int d, uint16_t *out, int64_t ldo,
                         moe_stream_t stream) {
  set_error("");
  REQUIRE(T >= 0 && k > 0 && d > 0, MOE_ERR_INVALID_ARG, "moe_combine: T=%d k=%d d=%d", T, k, d);
  REQUIRE(k <= 16, MOE_ERR_UNSUPPORTED, "moe_combine: k > 16");
  REQUIRE(d % 8 == 0 && ldy % 8 == 0 && ldo % 8 == 0, MOE_ERR_UNSUPPORTED,
          "moe_combine: d, ldy, ldo must be multiples of 8");
  REQUIRE(ldy >= d && ldo >= d, MOE_ERR_INVALID_ARG, "moe_combine: leading dimension < d");
  REQUIRE(T == 0 || (Y && flat_to_sorted && out), MOE_ERR_INVALID_ARG, "moe_combine: null pointer");
  REQUIRE(T == 0 || (aligned16(Y) && aligned16(out)), MOE_ERR_UNSUPPORTED,
          "moe_combine: Y and out must be 16-byte aligned");
  return cuda_status(moe::launch_combine(Y, ldy, flat_to_sorted, topk_w, T, k, d, out, ldo,
                                         (cudaStream_t)stream),
                     "moe_combine launch");
}

moe_status_t moe_unpermute_bwd(const uint16_t *d_out, int64_t ld_dout, const uint16_t *Y,
                               int64_t ldy, const int32_t *flat_to_sorted,
                               const int32_t *sorted_to_flat, const int32_t *group_offsets,
                               const float *topk_w, int T, int k, int d, int E,
                               int64_t rows_cap, uint16_t *dY, int64_t ld_dy, float *d_topk_w,
                               moe_stream_t stream) {
  set_error("");
  REQUIRE(T >= 0 && k > 0 && d > 0 && E > 0 && rows_cap >= 0, MOE_ERR_INVALID_ARG,
          "moe_unpermute_bwd: T=%d k=%d d=%d E=%d", T, k, d, E);
  REQUIRE(k <= 16, MOE_ERR_UNSUPPORTED, "moe_unpermute_bwd: k > 16");
  REQUIRE(d % 8 == 0 && ld_dout % 8 == 0 && ldy % 8 == 0 && ld_dy % 8 == 0, MOE_ERR_UNSUPPORTED,
          "moe_unpermute_bwd: d and leading dimensions must be multiples of 8");
  REQUIRE(ld_dout >= d && ldy >= d && ld_dy >= d, MOE_ERR_INVALID_ARG,
          "moe_unpermute_bwd: leading dimension < d");
  REQUIRE(rows_cap < (1ll << 31), MOE_ERR_UNSUPPORTED, "moe_unpermute_bwd: more than 2^31 rows");
  REQUIRE(group_offsets && (rows_cap == 0 || (sorted_to_flat && dY)), MOE_ERR_INVALID_ARG,
          "moe_unpermute_bwd: null pointer");
  REQUIRE(T == 0 || (d_out && Y && flat_to_sorted && topk_w && d_topk_w), MOE_ERR_INVALID_ARG,
          "moe_unpermute_bwd: null pointer");
  REQUIRE(aligned16(dY) && (T == 0 || (aligned16(d_out) && aligned16(Y))), MOE_ERR_UNSUPPORTED,
          "moe_unpermute_bwd: d_out, Y, dY must be 16-byte aligned");
  return cuda_status(moe::launch_unpermute_bwd(d_out, ld_dout, Y, ldy, flat_to_sorted,
                                               sorted_to_flat, group_offsets, topk_w, T, k, d, E,
                                               rows_cap, dY, ld_dy, d_topk_w,
                                               (cudaStream_t)stream),
                     "moe_unpermute_bwd launch");
}

}  // extern "C"
