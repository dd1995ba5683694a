// The whole layer behind two calls: a workspace planner, the forward and
// backward sequences of the library's calls, and a double-buffered host
// pipeline.  Host code apart from one table-filling kernel; every step of the
// layer runs in the kernels behind the calls it makes.
//
// The sequence is the single-VJP MoE block of TransformerEngine PR #2912 ("[JAX]
// Add an MoE Block (Layer) that compound router, permutation, groupedGEMM and
// communication", sequence diagram) on one GPU: route -> permute -> grouped
// GEMM (up, SwiGLU) -> grouped GEMM (down) -> combine, and its VJP.

#include <new>

#include "internal.h"

using moe::set_error;

namespace {

constexpr size_t kAlign = 256;

struct Slot {
  size_t off = 0, bytes = 0;
};

struct Plan {
  Slot buf[MOE_BUF_COUNT];
  size_t total = 0;
  int64_t R = 0, P = 0;
};

// Shapes of the configuration in elements, and the checks every entry point
// shares.  Returns false (reason in moe_last_error) for an invalid one.
bool check_config(const moe_layer_config *c) {
  if (c == nullptr) {
    set_error("moe_layer: null configuration");
    return false;
  }
  if (c->T < 0 || c->d <= 0 || c->f <= 0 || c->E <= 0 || c->k <= 0 || c->k > c->E) {
    set_error("moe_layer: bad sizes T=%d d=%d f=%d E=%d k=%d", c->T, c->d, c->f, c->E, c->k);
    return false;
  }
  if (c->precision < MOE_PREC_BF16 || c->precision > MOE_PREC_MXFP8) {
    set_error("moe_layer: unknown precision %d", c->precision);
    return false;
  }
  if (c->num_chunks > 1 && c->d % c->num_chunks != 0) {
    // the chunks tile d_model exactly (MaxText PR #4295, Description: the
    // up-projection is split evenly along d_model)
    set_error("moe_layer: num_chunks=%d does not divide d_model=%d", c->num_chunks, c->d);
    return false;
  }
  if (c->precision != MOE_PREC_BF16 && (c->bias || c->num_chunks > 1)) {
    set_error("moe_layer: the FP8 and MXFP8 layers take neither biases nor K-chunks");
    return false;
  }
  if (c->precision == MOE_PREC_MXFP8 && (c->d % 128 || c->f % 128)) {
    set_error("moe_layer: MXFP8 needs d_model and d_ff multiples of 128");
    return false;
  }
  if (c->dw_dtype != MOE_DTYPE_BF16 && c->dw_dtype != MOE_DTYPE_F32) {
    set_error("moe_layer: dw_dtype %d is neither bf16 nor f32", c->dw_dtype);
    return false;
  }
  if (c->aux_coeff < 0.f) {
    set_error("moe_layer: negative aux_coeff");
    return false;
  }
  return true;
}

bool colwise(const moe_layer_config *c) {
  return c->wgrad_colwise && c->precision == MOE_PREC_BF16;
}

bool make_plan(const moe_layer_config *c, Plan *p) {
  if (!check_config(c)) return false;
  const int64_t T = c->T, d = c->d, f = c->f, E = c->E, k = c->k;
  const int64_t R = moe_rows_cap(c->T, c->E, c->k, c->align, c->capacity);
  if (R < 0) {
    set_error("moe_layer: moe_rows_cap failed for align=%d capacity=%d", c->align, c->capacity);
    return false;
  }
  const int64_t P = moe_fp8_padded_rows(R, c->E);
  p->R = R;
  p->P = P;
  const size_t bf = 2, i32 = 4, f32 = 4, u8 = 1;
  const size_t dw = c->dw_dtype == MOE_DTYPE_F32 ? 4 : 2;
  size_t sz[MOE_BUF_COUNT] = {};
  sz[MOE_BUF_TOPK_IDX] = T * k * i32;
  sz[MOE_BUF_TOPK_W] = T * k * f32;
  sz[MOE_BUF_XS] = R * d * bf;
  sz[MOE_BUF_GROUP_SIZES] = E * i32;
  sz[MOE_BUF_KEPT_COUNTS] = E * i32;
  sz[MOE_BUF_GROUP_OFFSETS] = (E + 1) * i32;
  sz[MOE_BUF_S2F] = R * i32;
  sz[MOE_BUF_F2S] = T * k * i32;
  sz[MOE_BUF_PERMUTE_WS] = moe_permute_workspace_bytes(c->T, c->E);
  sz[MOE_BUF_H] = R * 2 * f * bf;
  sz[MOE_BUF_ACT] = R * f * bf;
  sz[MOE_BUF_Y] = R * d * bf;
  sz[MOE_BUF_OUT] = T * d * bf;
  if (c->num_chunks > 1) sz[MOE_BUF_PARTIAL] = R * 2 * f * f32;
  sz[MOE_BUF_DY] = R * d * bf;
  sz[MOE_BUF_D_TOPK_W] = T * k * f32;
  sz[MOE_BUF_D_LOGITS] = T * E * f32;
  sz[MOE_BUF_DH] = R * 2 * f * bf;
  sz[MOE_BUF_DXS] = R * d * bf;
  sz[MOE_BUF_DX] = T * d * bf;
  sz[MOE_BUF_DWI] = E * d * 2 * f * dw;
  sz[MOE_BUF_DWO] = E * f * d * dw;
  if (c->bias) {
    sz[MOE_BUF_DBI] = E * 2 * f * f32;
    sz[MOE_BUF_DBO] = E * d * f32;
  }
  sz[MOE_BUF_DEV_STATUS] = i32;
  if (colwise(c)) {
    sz[MOE_BUF_XS_T] = d * P * bf;
    sz[MOE_BUF_ACT_T] = f * P * bf;
    sz[MOE_BUF_DY_T] = d * P * bf;
    sz[MOE_BUF_DH_T] = 2 * f * P * bf;
  }
  if (c->precision == MOE_PREC_FP8) {
    sz[MOE_BUF_F8_XS_Q] = R * d * u8;
    sz[MOE_BUF_F8_XS_QT] = d * P * u8;
    sz[MOE_BUF_F8_ACT_Q] = R * f * u8;
    sz[MOE_BUF_F8_ACT_QT] = f * P * u8;
    sz[MOE_BUF_F8_DY_Q] = R * d * u8;
    sz[MOE_BUF_F8_DY_QT] = d * P * u8;
    sz[MOE_BUF_F8_DH_Q] = R * 2 * f * u8;
    sz[MOE_BUF_F8_DH_QT] = 2 * f * P * u8;
    sz[MOE_BUF_F8_WI_Q] = E * d * 2 * f * u8;
    sz[MOE_BUF_F8_WI_QT] = E * 2 * f * d * u8;
    sz[MOE_BUF_F8_WO_Q] = E * f * d * u8;
    sz[MOE_BUF_F8_WO_QT] = E * d * f * u8;
    sz[MOE_BUF_F8_AMAX] = (4 + 2 * E) * f32;
    sz[MOE_BUF_F8_SINV] = (4 + 2 * E) * f32;
  }
  if (c->precision == MOE_PREC_MXFP8) {
    struct Q {
      int q;
      int64_t rows, cols;
      int map, groups;
    } qs[] = {
        {MOE_BUF_MX_XS_Q, R, d, MOE_MX_ROWS_GROUPED, c->E},
        {MOE_BUF_MX_ACT_Q, R, f, MOE_MX_ROWS_GROUPED, c->E},
        {MOE_BUF_MX_DY_Q, R, d, MOE_MX_ROWS_GROUPED, c->E},
        {MOE_BUF_MX_DH_Q, R, 2 * f, MOE_MX_ROWS_GROUPED, c->E},
        {MOE_BUF_MX_XS_T_Q, d, P, MOE_MX_ROWS_PLAIN, c->E},
        {MOE_BUF_MX_ACT_T_Q, f, P, MOE_MX_ROWS_PLAIN, c->E},
        {MOE_BUF_MX_DY_T_Q, d, P, MOE_MX_ROWS_TILES, 1},
        {MOE_BUF_MX_DH_T_Q, 2 * f, P, MOE_MX_ROWS_TILES, 1},
        {MOE_BUF_MX_WI_T_Q, 2 * f, E * d, MOE_MX_ROWS_SWIGLU, c->E},
        {MOE_BUF_MX_WI_Q, E * d, 2 * f, MOE_MX_ROWS_TILES, c->E},
        {MOE_BUF_MX_WO_T_Q, d, E * f, MOE_MX_ROWS_TILES, 1},
        {MOE_BUF_MX_WO_Q, E * f, d, MOE_MX_ROWS_TILES, c->E},
    };
    for (const Q &q : qs) {
      sz[q.q] = q.rows * q.cols * u8;
      const size_t sf = moe_mx_scale_bytes(q.rows, (int)q.cols, q.map, q.groups);
      if (sf == 0) {
        set_error("moe_layer: no block-scale layout for a [%lld, %lld] operand",
                  (long long)q.rows, (long long)q.cols);
        return false;
      }
      sz[q.q + 1] = sf;  // the scale atoms follow their codes in the enum
    }
    sz[MOE_BUF_MX_WOFF_D] = (E + 1) * i32;
    sz[MOE_BUF_MX_WOFF_F] = (E + 1) * i32;
  }
  if (c->aux_coeff > 0.f) {
    sz[MOE_BUF_AUX_COUNTS] = E * i32;
    sz[MOE_BUF_AUX_PROBS] = E * f32;
    sz[MOE_BUF_AUX_LOSS] = f32;
    sz[MOE_BUF_AUX_WS] = moe_aux_loss_workspace_bytes(c->T, c->E);
  }
  size_t off = 0;
  for (int i = 0; i < MOE_BUF_COUNT; ++i) {
    p->buf[i].off = sz[i] ? off : 0;
    p->buf[i].bytes = sz[i];
    off += (sz[i] + kAlign - 1) / kAlign * kAlign;
  }
  p->total = off;
  return true;
}

// The layer's tensors resolved in one workspace, plus the step's inputs and
// results (the workspace's own buffers, or a pipeline's staging slots).
struct View {
  const moe_layer_config *c;
  Plan plan;
  uint8_t *ws;
  template <class T>
  T *at(int id) const {
    return plan.buf[id].bytes ? reinterpret_cast<T *>(ws + plan.buf[id].off) : nullptr;
  }
  uint16_t *bf(int id) const { return at<uint16_t>(id); }
  uint8_t *u8(int id) const { return at<uint8_t>(id); }
  int32_t *i32(int id) const { return at<int32_t>(id); }
  float *f32(int id) const { return at<float>(id); }
};

struct Io {
  const uint16_t *x = nullptr, *dout = nullptr;
  const float *logits = nullptr;
  uint16_t *out = nullptr, *dx = nullptr;
  float *d_logits = nullptr;
};

bool make_view(const moe_layer_config *c, void *ws, size_t ws_bytes, View *v) {
  v->c = c;
  if (!make_plan(c, &v->plan)) return false;
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & (kAlign - 1)) != 0) {
    set_error("moe_layer: workspace null or not 256-byte aligned");
    return false;
  }
  if (ws_bytes < v->plan.total) {
    set_error("moe_layer: workspace of %zu bytes, %zu needed", ws_bytes, v->plan.total);
    return false;
  }
  v->ws = static_cast<uint8_t *>(ws);
  return true;
}

#define CALL(expr)                          \
  do {                                      \
    const moe_status_t st_ = (expr);        \
    if (st_ != MOE_OK) return st_;          \
  } while (0)

void mark(moe_mark_fn fn, void *ctx, const char *name) {
  if (fn != nullptr) fn(ctx, name);
}

// ---------------------------------------------------------------- forward
moe_status_t forward_fp8(const View &v, const uint16_t *wi, const uint16_t *wo, cudaStream_t s,
                         moe_mark_fn mk, void *ctx) {
  const moe_layer_config &c = *v.c;
  const int E = c.E, d = c.d, f = c.f;
  const int64_t R = v.plan.R, P = v.plan.P;
  const int32_t *off = v.i32(MOE_BUF_GROUP_OFFSETS);
  int32_t *st = v.i32(MOE_BUF_DEV_STATUS);
  float *amax = v.f32(MOE_BUF_F8_AMAX), *sinv = v.f32(MOE_BUF_F8_SINV);
  // slots: 0 Xs, 1 Act, 2 dY, 3 dH, 4.. wi (E), 4 + E.. wo (E)
  CALL(moe_fp8_amax(v.bf(MOE_BUF_XS), d, R, d, 1, off, E, amax + 0, s));
  CALL(moe_fp8_quantize_act(v.bf(MOE_BUF_XS), d, off, E, R, d, MOE_FP8_E4M3, amax + 0,
                            v.u8(MOE_BUF_F8_XS_Q), d, v.u8(MOE_BUF_F8_XS_QT), P, sinv + 0, s));
  mark(mk, ctx, "quant_x");
  CALL(moe_fp8_amax(wi, 2 * f, (int64_t)E * d, 2 * f, E, nullptr, 0, amax + 4, s));
  CALL(moe_fp8_quantize_weights(wi, E, d, 2 * f, MOE_FP8_E4M3, amax + 4,
                                v.u8(MOE_BUF_F8_WI_Q), v.u8(MOE_BUF_F8_WI_QT), sinv + 4, s));
  mark(mk, ctx, "quant_wi");
  CALL(moe_fp8_amax(wo, d, (int64_t)E * f, d, E, nullptr, 0, amax + 4 + E, s));
  CALL(moe_fp8_quantize_weights(wo, E, f, d, MOE_FP8_E4M3, amax + 4 + E,
                                v.u8(MOE_BUF_F8_WO_Q), v.u8(MOE_BUF_F8_WO_QT), sinv + 4 + E, s));
  mark(mk, ctx, "quant_wo");
  // up-projection on [E, 2f, d] codes, the SwiGLU epilogue leaves Act's amax
  CALL(moe_gmm_fp8(v.u8(MOE_BUF_F8_XS_Q), d, MOE_FP8_E4M3, sinv + 0, v.u8(MOE_BUF_F8_WI_QT), d,
                   (int64_t)2 * f * d, MOE_FP8_E4M3, sinv + 4, off, E, R, d, 2 * f,
                   MOE_EPI_SWIGLU_FWD, nullptr, 0, v.bf(MOE_BUF_H), MOE_DTYPE_BF16, 2 * f,
                   v.bf(MOE_BUF_ACT), f, amax + 1, st, s));
  mark(mk, ctx, "gmm_up_swiglu");
  CALL(moe_fp8_quantize_act(v.bf(MOE_BUF_ACT), f, off, E, R, f, MOE_FP8_E4M3, amax + 1,
                            v.u8(MOE_BUF_F8_ACT_Q), f, v.u8(MOE_BUF_F8_ACT_QT), P, sinv + 1, s));
  mark(mk, ctx, "quant_act");
  CALL(moe_gmm_fp8(v.u8(MOE_BUF_F8_ACT_Q), f, MOE_FP8_E4M3, sinv + 1, v.u8(MOE_BUF_F8_WO_QT), f,
                   (int64_t)d * f, MOE_FP8_E4M3, sinv + 4 + E, off, E, R, f, d, MOE_EPI_NONE,
                   nullptr, 0, v.bf(MOE_BUF_Y), MOE_DTYPE_BF16, d, nullptr, 0, nullptr, st, s));
  mark(mk, ctx, "gmm_down");
  return MOE_OK;
}

// Row-wise and column-wise block-scaled codes of a permuted activation from
// one read (blocks along its row's d_model / d_ff, and along each expert's
// rows; qt_map PLAIN for a weight gradient's A operand, TILES for its B).
moe_status_t mx_both(const View &v, const char *name, const uint16_t *x, int cols, int fmt,
                     int q_id, int qt_id, int qt_map, cudaStream_t s, moe_mark_fn mk, void *ctx) {
  const moe_layer_config &c = *v.c;
  const Plan &p = v.plan;
  CALL(moe_mx_quantize_2x(x, cols, p.R, cols, fmt, v.i32(MOE_BUF_GROUP_OFFSETS), c.E, v.u8(q_id),
                          cols, MOE_MX_ROWS_GROUPED, v.u8(q_id + 1), p.buf[q_id + 1].bytes,
                          v.u8(qt_id), p.P, p.P, qt_map, v.u8(qt_id + 1),
                          p.buf[qt_id + 1].bytes, s));
  mark(mk, ctx, name);
  return MOE_OK;
}

moe_status_t forward_mx(const View &v, const uint16_t *wi, const uint16_t *wo, cudaStream_t s,
                        moe_mark_fn mk, void *ctx) {
  const moe_layer_config &c = *v.c;
  const Plan &p = v.plan;
  const int E = c.E, d = c.d, f = c.f;
  const int64_t R = p.R;
  const int32_t *off = v.i32(MOE_BUF_GROUP_OFFSETS);
  int32_t *st = v.i32(MOE_BUF_DEV_STATUS);
  const int e4 = MOE_FP8_E4M3;
  CALL(mx_both(v, "mxquant_xs", v.bf(MOE_BUF_XS), d, e4, MOE_BUF_MX_XS_Q, MOE_BUF_MX_XS_T_Q,
               MOE_MX_ROWS_PLAIN, s, mk, ctx));
  // the weights along both contractions from one read each: wi as [E d, 2f]
  // (dgrad-up B, blocks along 2f) and wi^T [2f, E d] (up-projection B, blocks
  // along d, SwiGLU tile order); wo as [E f, d] and wo^T [d, E f]
  CALL(moe_mx_quantize_2x(wi, 2 * f, (int64_t)E * d, 2 * f, e4, v.i32(MOE_BUF_MX_WOFF_D), E,
                          v.u8(MOE_BUF_MX_WI_Q), 2 * f, MOE_MX_ROWS_TILES,
                          v.u8(MOE_BUF_MX_WI_SF), p.buf[MOE_BUF_MX_WI_SF].bytes,
                          v.u8(MOE_BUF_MX_WI_T_Q), (int64_t)E * d, (int64_t)E * d,
                          MOE_MX_ROWS_SWIGLU, v.u8(MOE_BUF_MX_WI_T_SF),
                          p.buf[MOE_BUF_MX_WI_T_SF].bytes, s));
  CALL(moe_mx_quantize_2x(wo, d, (int64_t)E * f, d, e4, v.i32(MOE_BUF_MX_WOFF_F), E,
                          v.u8(MOE_BUF_MX_WO_Q), d, MOE_MX_ROWS_TILES, v.u8(MOE_BUF_MX_WO_SF),
                          p.buf[MOE_BUF_MX_WO_SF].bytes, v.u8(MOE_BUF_MX_WO_T_Q),
                          (int64_t)E * f, (int64_t)E * f, MOE_MX_ROWS_TILES,
                          v.u8(MOE_BUF_MX_WO_T_SF), p.buf[MOE_BUF_MX_WO_T_SF].bytes, s));
  mark(mk, ctx, "mxquant_weights");
  CALL(moe_gmm_mx(v.u8(MOE_BUF_MX_XS_Q), d, v.u8(MOE_BUF_MX_XS_SF), e4, v.u8(MOE_BUF_MX_WI_T_Q),
                  (int64_t)E * d, d, v.u8(MOE_BUF_MX_WI_T_SF), 1, e4, off, E, R, d, 2 * f,
                  MOE_EPI_SWIGLU_FWD, nullptr, 0, v.bf(MOE_BUF_H), MOE_DTYPE_BF16, 2 * f,
                  v.bf(MOE_BUF_ACT), f, st, s));
  mark(mk, ctx, "gmm_up_swiglu");
  CALL(mx_both(v, "mxquant_act", v.bf(MOE_BUF_ACT), f, e4, MOE_BUF_MX_ACT_Q, MOE_BUF_MX_ACT_T_Q,
               MOE_MX_ROWS_PLAIN, s, mk, ctx));
  CALL(moe_gmm_mx(v.u8(MOE_BUF_MX_ACT_Q), f, v.u8(MOE_BUF_MX_ACT_SF), e4,
                  v.u8(MOE_BUF_MX_WO_T_Q), (int64_t)E * f, f, v.u8(MOE_BUF_MX_WO_T_SF), 1, e4, off,
                  E, R, f, d, MOE_EPI_NONE, nullptr, 0, v.bf(MOE_BUF_Y), MOE_DTYPE_BF16, d,
                  nullptr, 0, st, s));
  mark(mk, ctx, "gmm_down");
  return MOE_OK;
}

moe_status_t forward(const View &v, const Io &io, const uint16_t *wi, const uint16_t *wo,
                     const uint16_t *bi, const uint16_t *bo, const float *expert_bias,
                     cudaStream_t s, moe_mark_fn mk, void *ctx) {
  const moe_layer_config &c = *v.c;
  const int T = c.T, E = c.E, k = c.k, d = c.d, f = c.f;
  const int64_t R = v.plan.R, P = v.plan.P;
  if ((T > 0 && (io.x == nullptr || io.logits == nullptr)) || wi == nullptr || wo == nullptr) {
    set_error("moe_layer_forward: null x, logits or weights");
    return MOE_ERR_INVALID_ARG;
  }
  if ((c.bias != 0) != (bi != nullptr && bo != nullptr)) {
    set_error("moe_layer_forward: pass bi and bo exactly when the configuration has biases");
    return MOE_ERR_INVALID_ARG;
  }
  int32_t *topk_idx = v.i32(MOE_BUF_TOPK_IDX);
  float *topk_w = v.f32(MOE_BUF_TOPK_W);
  const int32_t *off = v.i32(MOE_BUF_GROUP_OFFSETS);
  int32_t *st = v.i32(MOE_BUF_DEV_STATUS);
  CALL(moe_route_topk(io.logits, E, T, E, k, c.score_fn, c.renorm, expert_bias, c.num_groups,
                      c.topk_group, topk_idx, topk_w, s));
  mark(mk, ctx, "route");
  if (c.aux_coeff > 0.f) {
    CALL(moe_aux_loss(io.logits, E, T, E, k, c.score_fn, topk_idx, c.aux_coeff,
                      v.i32(MOE_BUF_AUX_COUNTS), v.f32(MOE_BUF_AUX_PROBS),
                      v.f32(MOE_BUF_AUX_LOSS), v.u8(MOE_BUF_AUX_WS),
                      v.plan.buf[MOE_BUF_AUX_WS].bytes, s));
    mark(mk, ctx, "aux_loss");
  }
  CALL(moe_permute(io.x, d, topk_idx, T, d, E, k, c.align, c.capacity, v.bf(MOE_BUF_XS), d, R,
                   v.i32(MOE_BUF_GROUP_SIZES), v.i32(MOE_BUF_KEPT_COUNTS),
                   v.i32(MOE_BUF_GROUP_OFFSETS), v.i32(MOE_BUF_S2F), v.i32(MOE_BUF_F2S),
                   v.u8(MOE_BUF_PERMUTE_WS), v.plan.buf[MOE_BUF_PERMUTE_WS].bytes, st, s));
  mark(mk, ctx, "permute");
  if (c.precision == MOE_PREC_MXFP8) {
    CALL(forward_mx(v, wi, wo, s, mk, ctx));
  } else if (c.precision == MOE_PREC_FP8) {
    CALL(forward_fp8(v, wi, wo, s, mk, ctx));
  } else {
    uint16_t *act_t = colwise(&c) ? v.bf(MOE_BUF_ACT_T) : nullptr;
    const int64_t ld_act_t = act_t ? P : 0;
    const uint16_t *xs = v.bf(MOE_BUF_XS);
    if (c.num_chunks <= 1) {
      CALL(moe_gmm(xs, d, wi, 2 * f, (int64_t)d * 2 * f, 0, off, E, R, d, 2 * f,
                   MOE_EPI_SWIGLU_FWD, nullptr, 0, nullptr, 0, bi, bi ? 2 * f : 0,
                   v.bf(MOE_BUF_H), MOE_DTYPE_BF16, 2 * f, v.bf(MOE_BUF_ACT), f, act_t, ld_act_t,
                   st, s));
      mark(mk, ctx, "gmm_up_swiglu");
    } else {
      // K-chunks of d_model into the fp32 partial sum in place, SwiGLU fused
      // into the last chunk (MaxText PR #4295, Description)
      const int dc = d / c.num_chunks;
      float *ps = v.f32(MOE_BUF_PARTIAL);
      for (int ch = 0; ch < c.num_chunks; ++ch) {
        const uint16_t *a_c = xs + (int64_t)ch * dc;
        const uint16_t *w_c = wi + (int64_t)ch * dc * 2 * f;
        const float *ps_in = ch == 0 ? nullptr : ps;
        const int64_t ld_ps = ch == 0 ? 0 : 2 * f;
        if (ch == c.num_chunks - 1) {
          CALL(moe_gmm(a_c, d, w_c, 2 * f, (int64_t)d * 2 * f, 0, off, E, R, dc, 2 * f,
                       MOE_EPI_SWIGLU_FWD, nullptr, 0, ps_in, ld_ps, bi, bi ? 2 * f : 0,
                       v.bf(MOE_BUF_H), MOE_DTYPE_BF16, 2 * f, v.bf(MOE_BUF_ACT), f, act_t,
                       ld_act_t, st, s));
          mark(mk, ctx, "gmm_up_chunk_swiglu");
        } else {
          CALL(moe_gmm(a_c, d, w_c, 2 * f, (int64_t)d * 2 * f, 0, off, E, R, dc, 2 * f,
                       MOE_EPI_NONE, nullptr, 0, ps_in, ld_ps, nullptr, 0, ps, MOE_DTYPE_F32,
                       2 * f, nullptr, 0, nullptr, 0, st, s));
          mark(mk, ctx, "gmm_up_chunk");
        }
      }
    }
    CALL(moe_gmm(v.bf(MOE_BUF_ACT), f, wo, d, (int64_t)f * d, 0, off, E, R, f, d, MOE_EPI_NONE,
                 nullptr, 0, nullptr, 0, bo, bo ? d : 0, v.bf(MOE_BUF_Y), MOE_DTYPE_BF16, d,
                 nullptr, 0, nullptr, 0, st, s));
    mark(mk, ctx, "gmm_down");
  }
  CALL(moe_combine(v.bf(MOE_BUF_Y), d, v.i32(MOE_BUF_F2S), topk_w, T, k, d, io.out, d, s));
  mark(mk, ctx, "combine");
  return MOE_OK;
}

// ---------------------------------------------------------------- backward
moe_status_t backward_fp8(const View &v, cudaStream_t s, moe_mark_fn mk, void *ctx) {
  const moe_layer_config &c = *v.c;
  const int E = c.E, d = c.d, f = c.f;
  const int64_t R = v.plan.R, P = v.plan.P;
  const int32_t *off = v.i32(MOE_BUF_GROUP_OFFSETS);
  int32_t *st = v.i32(MOE_BUF_DEV_STATUS);
  float *amax = v.f32(MOE_BUF_F8_AMAX), *sinv = v.f32(MOE_BUF_F8_SINV);
  const int dw = c.dw_dtype;
  CALL(moe_fp8_amax(v.bf(MOE_BUF_DY), d, R, d, 1, off, E, amax + 2, s));
  CALL(moe_fp8_quantize_act(v.bf(MOE_BUF_DY), d, off, E, R, d, MOE_FP8_E5M2, amax + 2,
                            v.u8(MOE_BUF_F8_DY_Q), d, v.u8(MOE_BUF_F8_DY_QT), P, sinv + 2, s));
  mark(mk, ctx, "quant_dy");
  // dgrad down on wo's [E, f, d] codes (K-major: K = d), SwiGLU backward
  CALL(moe_gmm_fp8(v.u8(MOE_BUF_F8_DY_Q), d, MOE_FP8_E5M2, sinv + 2, v.u8(MOE_BUF_F8_WO_Q), d,
                   (int64_t)f * d, MOE_FP8_E4M3, sinv + 4 + E, off, E, R, d, f,
                   MOE_EPI_SWIGLU_BWD, v.bf(MOE_BUF_H), 2 * f, v.bf(MOE_BUF_DH), MOE_DTYPE_BF16,
                   2 * f, nullptr, 0, amax + 3, st, s));
  mark(mk, ctx, "gmm_dgrad_down_swiglu_bwd");
  CALL(moe_tgmm_fp8(v.u8(MOE_BUF_F8_ACT_QT), P, MOE_FP8_E4M3, sinv + 1, v.u8(MOE_BUF_F8_DY_QT), P,
                    MOE_FP8_E5M2, sinv + 2, off, E, R, f, d, v.at<void>(MOE_BUF_DWO), dw, d,
                    (int64_t)f * d, 0, st, s));
  mark(mk, ctx, "tgmm_dwo");
  CALL(moe_fp8_quantize_act(v.bf(MOE_BUF_DH), 2 * f, off, E, R, 2 * f, MOE_FP8_E5M2, amax + 3,
                            v.u8(MOE_BUF_F8_DH_Q), 2 * f, v.u8(MOE_BUF_F8_DH_QT), P, sinv + 3,
                            s));
  mark(mk, ctx, "quant_dh");
  CALL(moe_gmm_fp8(v.u8(MOE_BUF_F8_DH_Q), 2 * f, MOE_FP8_E5M2, sinv + 3, v.u8(MOE_BUF_F8_WI_Q),
                   2 * f, (int64_t)d * 2 * f, MOE_FP8_E4M3, sinv + 4, off, E, R, 2 * f, d,
                   MOE_EPI_NONE, nullptr, 0, v.bf(MOE_BUF_DXS), MOE_DTYPE_BF16, d, nullptr, 0,
                   nullptr, st, s));
  mark(mk, ctx, "gmm_dgrad_up");
  CALL(moe_tgmm_fp8(v.u8(MOE_BUF_F8_XS_QT), P, MOE_FP8_E4M3, sinv + 0, v.u8(MOE_BUF_F8_DH_QT), P,
                    MOE_FP8_E5M2, sinv + 3, off, E, R, d, 2 * f, v.at<void>(MOE_BUF_DWI), dw,
                    2 * f, (int64_t)d * 2 * f, 0, st, s));
  mark(mk, ctx, "tgmm_dwi");
  return MOE_OK;
}

moe_status_t backward_mx(const View &v, cudaStream_t s, moe_mark_fn mk, void *ctx) {
  const moe_layer_config &c = *v.c;
  const int E = c.E, d = c.d, f = c.f;
  const int64_t R = v.plan.R, P = v.plan.P;
  const int32_t *off = v.i32(MOE_BUF_GROUP_OFFSETS);
  int32_t *st = v.i32(MOE_BUF_DEV_STATUS);
  const int e4 = MOE_FP8_E4M3, e5 = MOE_FP8_E5M2, dw = c.dw_dtype;
  CALL(mx_both(v, "mxquant_dy", v.bf(MOE_BUF_DY), d, e5, MOE_BUF_MX_DY_Q, MOE_BUF_MX_DY_T_Q,
               MOE_MX_ROWS_TILES, s, mk, ctx));
  CALL(moe_gmm_mx(v.u8(MOE_BUF_MX_DY_Q), d, v.u8(MOE_BUF_MX_DY_SF), e5, v.u8(MOE_BUF_MX_WO_Q), d,
                  (int64_t)f * d, v.u8(MOE_BUF_MX_WO_SF), 0, e4, off, E, R, d, f,
                  MOE_EPI_SWIGLU_BWD, v.bf(MOE_BUF_H), 2 * f, v.bf(MOE_BUF_DH), MOE_DTYPE_BF16,
                  2 * f, nullptr, 0, st, s));
  mark(mk, ctx, "gmm_dgrad_down_swiglu_bwd");
  CALL(moe_tgmm_mx(v.u8(MOE_BUF_MX_ACT_T_Q), P, v.u8(MOE_BUF_MX_ACT_T_SF), e4,
                   v.u8(MOE_BUF_MX_DY_T_Q), P, v.u8(MOE_BUF_MX_DY_T_SF), e5, off, E, R, f, d,
                   v.at<void>(MOE_BUF_DWO), dw, d, (int64_t)f * d, 0, st, s));
  mark(mk, ctx, "tgmm_dwo");
  CALL(mx_both(v, "mxquant_dh", v.bf(MOE_BUF_DH), 2 * f, e5, MOE_BUF_MX_DH_Q, MOE_BUF_MX_DH_T_Q,
               MOE_MX_ROWS_TILES, s, mk, ctx));
  CALL(moe_gmm_mx(v.u8(MOE_BUF_MX_DH_Q), 2 * f, v.u8(MOE_BUF_MX_DH_SF), e5,
                  v.u8(MOE_BUF_MX_WI_Q), 2 * f, (int64_t)d * 2 * f, v.u8(MOE_BUF_MX_WI_SF), 0, e4,
                  off, E, R, 2 * f, d, MOE_EPI_NONE, nullptr, 0, v.bf(MOE_BUF_DXS),
                  MOE_DTYPE_BF16, d, nullptr, 0, st, s));
  mark(mk, ctx, "gmm_dgrad_up");
  CALL(moe_tgmm_mx(v.u8(MOE_BUF_MX_XS_T_Q), P, v.u8(MOE_BUF_MX_XS_T_SF), e4,
                   v.u8(MOE_BUF_MX_DH_T_Q), P, v.u8(MOE_BUF_MX_DH_T_SF), e5, off, E, R, d, 2 * f,
                   v.at<void>(MOE_BUF_DWI), dw, 2 * f, (int64_t)d * 2 * f, 0, st, s));
  mark(mk, ctx, "tgmm_dwi");
  return MOE_OK;
}

moe_status_t backward(const View &v, const Io &io, const uint16_t *wi, const uint16_t *wo,
                      cudaStream_t s, moe_mark_fn mk, void *ctx) {
  const moe_layer_config &c = *v.c;
  const int T = c.T, E = c.E, k = c.k, d = c.d, f = c.f;
  const int64_t R = v.plan.R, P = v.plan.P;
  if ((T > 0 && (io.dout == nullptr || io.logits == nullptr)) || wi == nullptr ||
      wo == nullptr) {
    set_error("moe_layer_backward: null dout, logits or weights");
    return MOE_ERR_INVALID_ARG;
  }
  const int32_t *off = v.i32(MOE_BUF_GROUP_OFFSETS);
  int32_t *st = v.i32(MOE_BUF_DEV_STATUS);
  const int32_t *f2s = v.i32(MOE_BUF_F2S);
  const float *topk_w = v.f32(MOE_BUF_TOPK_W);
  float *d_topk_w = v.f32(MOE_BUF_D_TOPK_W);
  const int dw = c.dw_dtype;
  const size_t dwsz = dw == MOE_DTYPE_F32 ? 4 : 2;
  CALL(moe_unpermute_bwd(io.dout, d, v.bf(MOE_BUF_Y), d, f2s, v.i32(MOE_BUF_S2F), off, topk_w, T,
                         k, d, E, R, v.bf(MOE_BUF_DY), d, d_topk_w, s));
  mark(mk, ctx, "unpermute_bwd");
  CALL(moe_route_topk_bwd(io.logits, E, v.i32(MOE_BUF_TOPK_IDX), topk_w, d_topk_w, T, E, k,
                          c.score_fn, c.renorm, io.d_logits, E, s));
  mark(mk, ctx, "route_bwd");
  if (c.aux_coeff > 0.f) {
    CALL(moe_aux_loss_bwd(io.logits, E, T, E, k, c.score_fn, v.i32(MOE_BUF_AUX_COUNTS),
                          c.aux_coeff, 1.0f, io.d_logits, E, 1, s));
    mark(mk, ctx, "aux_loss_bwd");
  }
  if (c.precision == MOE_PREC_MXFP8) {
    CALL(backward_mx(v, s, mk, ctx));
  } else if (c.precision == MOE_PREC_FP8) {
    CALL(backward_fp8(v, s, mk, ctx));
  } else {
    const bool cw = colwise(&c);
    uint8_t *dwi = v.u8(MOE_BUF_DWI);
    // dAct = dY . wo^T fused with the SwiGLU backward into dH = [dgate | dup]
    CALL(moe_gmm(v.bf(MOE_BUF_DY), d, wo, d, (int64_t)f * d, 1, off, E, R, d, f,
                 MOE_EPI_SWIGLU_BWD, v.bf(MOE_BUF_H), 2 * f, nullptr, 0, nullptr, 0,
                 v.bf(MOE_BUF_DH), MOE_DTYPE_BF16, 2 * f, nullptr, 0,
                 cw ? v.bf(MOE_BUF_DH_T) : nullptr, cw ? P : 0, st, s));
    mark(mk, ctx, "gmm_dgrad_down_swiglu_bwd");
    if (cw) {
      CALL(moe_transpose_act(v.bf(MOE_BUF_DY), d, off, E, R, d, v.bf(MOE_BUF_DY_T), P, s));
      mark(mk, ctx, "transpose_dy");
      CALL(moe_tgmm_kt(v.bf(MOE_BUF_ACT_T), P, v.bf(MOE_BUF_DY_T), P, 1, off, E, R, f, d,
                       v.at<void>(MOE_BUF_DWO), dw, d, (int64_t)f * d, 0, st, s));
    } else {
      CALL(moe_tgmm(v.bf(MOE_BUF_ACT), f, v.bf(MOE_BUF_DY), d, off, E, R, f, d,
                    v.at<void>(MOE_BUF_DWO), dw, d, (int64_t)f * d, 0, st, s));
    }
    mark(mk, ctx, "tgmm_dwo");
    if (c.bias) {
      CALL(moe_group_colsum(v.bf(MOE_BUF_DY), d, off, E, R, d, v.f32(MOE_BUF_DBO), d, s));
      mark(mk, ctx, "colsum_dbo");
      CALL(moe_group_colsum(v.bf(MOE_BUF_DH), 2 * f, off, E, R, 2 * f, v.f32(MOE_BUF_DBI), 2 * f,
                            s));
      mark(mk, ctx, "colsum_dbi");
    }
    if (cw) {
      CALL(moe_transpose_act(v.bf(MOE_BUF_XS), d, off, E, R, d, v.bf(MOE_BUF_XS_T), P, s));
      mark(mk, ctx, "transpose_xs");
    }
    // dWi over the d_model rows [r0, r0 + m)
    auto tgmm_dwi = [&](int r0, int m, const char *name) -> moe_status_t {
      void *w = dwi + (size_t)r0 * 2 * f * dwsz;
      if (cw)
        CALL(moe_tgmm_kt(v.bf(MOE_BUF_XS_T) + (int64_t)r0 * P, P, v.bf(MOE_BUF_DH_T), P, 1, off,
                         E, R, m, 2 * f, w, dw, 2 * f, (int64_t)d * 2 * f, 0, st, s));
      else
        CALL(moe_tgmm(v.bf(MOE_BUF_XS) + r0, d, v.bf(MOE_BUF_DH), 2 * f, off, E, R, m, 2 * f, w,
                      dw, 2 * f, (int64_t)d * 2 * f, 0, st, s));
      mark(mk, ctx, name);
      return MOE_OK;
    };
    if (c.num_chunks <= 1) {
      CALL(moe_gmm(v.bf(MOE_BUF_DH), 2 * f, wi, 2 * f, (int64_t)d * 2 * f, 1, off, E, R, 2 * f,
                   d, MOE_EPI_NONE, nullptr, 0, nullptr, 0, nullptr, 0, v.bf(MOE_BUF_DXS),
                   MOE_DTYPE_BF16, d, nullptr, 0, nullptr, 0, st, s));
      mark(mk, ctx, "gmm_dgrad_up");
      CALL(tgmm_dwi(0, d, "tgmm_dwi"));
    } else {
      const int dc = d / c.num_chunks;
      for (int ch = 0; ch < c.num_chunks; ++ch) {
        CALL(moe_gmm(v.bf(MOE_BUF_DH), 2 * f, wi + (int64_t)ch * dc * 2 * f, 2 * f,
                     (int64_t)d * 2 * f, 1, off, E, R, 2 * f, dc, MOE_EPI_NONE, nullptr, 0,
                     nullptr, 0, nullptr, 0, v.bf(MOE_BUF_DXS) + (int64_t)ch * dc,
                     MOE_DTYPE_BF16, d, nullptr, 0, nullptr, 0, st, s));
        mark(mk, ctx, "gmm_dgrad_up_chunk");
        CALL(tgmm_dwi(ch * dc, dc, "tgmm_dwi_chunk"));
      }
    }
  }
  CALL(moe_combine(v.bf(MOE_BUF_DXS), d, f2s, nullptr, T, k, d, io.dx, d, s));
  mark(mk, ctx, "dispatch_bwd");
  return MOE_OK;
}

__global__ void iota_kernel(int32_t *o, int n, int step) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) o[i] = i * step;
}

// ---------------------------------------------------------------- pipeline
enum { kSlotX, kSlotLogits, kSlotDout, kSlotOut, kSlotDx, kSlotDLogits, kSlotKinds };

void slot_sizes(const moe_layer_config *c, size_t sz[kSlotKinds]) {
  const size_t Td = (size_t)c->T * c->d, TE = (size_t)c->T * c->E;
  sz[kSlotX] = Td * 2;
  sz[kSlotLogits] = TE * 4;
  sz[kSlotDout] = Td * 2;
  sz[kSlotOut] = Td * 2;
  sz[kSlotDx] = Td * 2;
  sz[kSlotDLogits] = TE * 4;
}

size_t rounded(size_t b) { return (b + kAlign - 1) / kAlign * kAlign; }

}  // namespace

struct moe_layer_pipeline {
  moe_layer_config cfg;
  View view;
  uint8_t *slot[2][kSlotKinds];
  cudaStream_t in_stream = nullptr, out_stream = nullptr;
  cudaEvent_t in_ready[2] = {}, step_done[2] = {}, out_done[2] = {};
  bool out_used[2] = {false, false};
  uint64_t steps = 0;
};

extern "C" {

size_t moe_layer_workspace_bytes(const moe_layer_config *cfg) {
  set_error("");
  Plan p;
  return make_plan(cfg, &p) ? p.total : 0;
}

moe_status_t moe_layer_buffer(const moe_layer_config *cfg, int id, size_t *offset,
                              size_t *bytes) {
  set_error("");
  if (id < 0 || id >= MOE_BUF_COUNT || offset == nullptr || bytes == nullptr) {
    set_error("moe_layer_buffer: bad id %d or null output", id);
    return MOE_ERR_INVALID_ARG;
  }
  Plan p;
  if (!make_plan(cfg, &p)) return MOE_ERR_INVALID_ARG;
  *offset = p.buf[id].off;
  *bytes = p.buf[id].bytes;
  return MOE_OK;
}

moe_status_t moe_layer_init(const moe_layer_config *cfg, void *workspace,
                            size_t workspace_bytes, moe_stream_t stream) {
  set_error("");
  View v;
  if (!make_view(cfg, workspace, workspace_bytes, &v)) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemsetAsync(v.i32(MOE_BUF_DEV_STATUS), 0, 4, s);
  if (e != cudaSuccess) {
    set_error("moe_layer_init: %s", cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  if (cfg->precision == MOE_PREC_MXFP8) {
    const int n = cfg->E + 1;
    iota_kernel<<<(n + 127) / 128, 128, 0, s>>>(v.i32(MOE_BUF_MX_WOFF_D), n, cfg->d);
    iota_kernel<<<(n + 127) / 128, 128, 0, s>>>(v.i32(MOE_BUF_MX_WOFF_F), n, cfg->f);
    e = cudaGetLastError();
    if (e != cudaSuccess) {
      set_error("moe_layer_init: %s", cudaGetErrorString(e));
      return MOE_ERR_CUDA;
    }
  }
  return MOE_OK;
}

moe_status_t moe_layer_forward(const moe_layer_config *cfg, void *workspace,
                               size_t workspace_bytes, const uint16_t *x, const float *logits,
                               const uint16_t *wi, const uint16_t *wo, const uint16_t *bi,
                               const uint16_t *bo, const float *expert_bias, moe_mark_fn mark_fn,
                               void *mark_ctx, moe_stream_t stream) {
  set_error("");
  View v;
  if (!make_view(cfg, workspace, workspace_bytes, &v)) return MOE_ERR_INVALID_ARG;
  Io io;
  io.x = x;
  io.logits = logits;
  io.out = v.bf(MOE_BUF_OUT);
  return forward(v, io, wi, wo, bi, bo, expert_bias, reinterpret_cast<cudaStream_t>(stream),
                 mark_fn, mark_ctx);
}

moe_status_t moe_layer_backward(const moe_layer_config *cfg, void *workspace,
                                size_t workspace_bytes, const uint16_t *dout,
                                const float *logits, const uint16_t *wi, const uint16_t *wo,
                                moe_mark_fn mark_fn, void *mark_ctx, moe_stream_t stream) {
  set_error("");
  View v;
  if (!make_view(cfg, workspace, workspace_bytes, &v)) return MOE_ERR_INVALID_ARG;
  Io io;
  io.dout = dout;
  io.logits = logits;
  io.dx = v.bf(MOE_BUF_DX);
  io.d_logits = v.f32(MOE_BUF_D_LOGITS);
  return backward(v, io, wi, wo, reinterpret_cast<cudaStream_t>(stream), mark_fn, mark_ctx);
}

size_t moe_layer_pipeline_workspace_bytes(const moe_layer_config *cfg) {
  set_error("");
  if (!check_config(cfg)) return 0;
  size_t sz[kSlotKinds];
  slot_sizes(cfg, sz);
  size_t total = 0;
  for (int i = 0; i < kSlotKinds; ++i) total += 2 * rounded(sz[i]);
  return total;
}

void moe_layer_pipeline_destroy(moe_layer_pipeline *p) {
  if (p == nullptr) return;
  if (p->in_stream) cudaStreamSynchronize(p->in_stream);
  if (p->out_stream) cudaStreamSynchronize(p->out_stream);
  for (int i = 0; i < 2; ++i) {
    if (p->in_ready[i]) cudaEventDestroy(p->in_ready[i]);
    if (p->step_done[i]) cudaEventDestroy(p->step_done[i]);
    if (p->out_done[i]) cudaEventDestroy(p->out_done[i]);
  }
  if (p->in_stream) cudaStreamDestroy(p->in_stream);
  if (p->out_stream) cudaStreamDestroy(p->out_stream);
  delete p;
}

moe_status_t moe_layer_pipeline_create(const moe_layer_config *cfg, void *workspace,
                                       size_t workspace_bytes, void *staging,
                                       size_t staging_bytes, moe_layer_pipeline **out) {
  set_error("");
  if (out == nullptr) {
    set_error("moe_layer_pipeline_create: null output");
    return MOE_ERR_INVALID_ARG;
  }
  *out = nullptr;
  moe_layer_pipeline *p = new (std::nothrow) moe_layer_pipeline();
  if (p == nullptr) {
    set_error("moe_layer_pipeline_create: out of host memory");
    return MOE_ERR_CUDA;
  }
  p->cfg = *cfg;
  if (!make_view(&p->cfg, workspace, workspace_bytes, &p->view)) {
    delete p;
    return MOE_ERR_INVALID_ARG;
  }
  const size_t need = moe_layer_pipeline_workspace_bytes(&p->cfg);
  if (staging == nullptr || (reinterpret_cast<uintptr_t>(staging) & (kAlign - 1)) != 0 ||
      staging_bytes < need) {
    set_error("moe_layer_pipeline_create: staging null, unaligned or below %zu bytes", need);
    delete p;
    return MOE_ERR_INVALID_ARG;
  }
  size_t sz[kSlotKinds];
  slot_sizes(&p->cfg, sz);
  uint8_t *b = static_cast<uint8_t *>(staging);
  for (int i = 0; i < kSlotKinds; ++i)
    for (int j = 0; j < 2; ++j) {
      p->slot[j][i] = b;
      b += rounded(sz[i]);
    }
  bool ok = cudaStreamCreateWithFlags(&p->in_stream, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&p->out_stream, cudaStreamNonBlocking) == cudaSuccess;
  for (int i = 0; ok && i < 2; ++i)
    ok = cudaEventCreateWithFlags(&p->in_ready[i], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&p->step_done[i], cudaEventDisableTiming) == cudaSuccess &&
         cudaEventCreateWithFlags(&p->out_done[i], cudaEventDisableTiming) == cudaSuccess;
  if (!ok) {
    set_error("moe_layer_pipeline_create: %s", cudaGetErrorString(cudaGetLastError()));
    moe_layer_pipeline_destroy(p);
    return MOE_ERR_CUDA;
  }
  *out = p;
  return MOE_OK;
}

moe_status_t moe_layer_pipeline_step(moe_layer_pipeline *p, const uint16_t *wi,
                                     const uint16_t *wo, const uint16_t *bi, const uint16_t *bo,
                                     const float *expert_bias, const uint16_t *h_x,
                                     const float *h_logits, const uint16_t *h_dout,
                                     uint16_t *h_out, uint16_t *h_dx, float *h_d_logits,
                                     moe_stream_t stream) {
  set_error("");
  if (p == nullptr ||
      (p->cfg.T > 0 && (h_x == nullptr || h_logits == nullptr || h_dout == nullptr ||
                        h_out == nullptr || h_dx == nullptr || h_d_logits == nullptr))) {
    set_error("moe_layer_pipeline_step: null pipeline or host buffer");
    return MOE_ERR_INVALID_ARG;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int j = (int)(p->steps & 1);
  uint8_t *const *sl = p->slot[j];
  size_t sz[kSlotKinds];
  slot_sizes(&p->cfg, sz);
  auto fail = [](cudaError_t e) {
    set_error("moe_layer_pipeline_step: %s", cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  };
  cudaError_t e;
  // inputs: the slot is free once the step that last read it (two back) ended
  if (p->steps >= 2 && (e = cudaStreamWaitEvent(p->in_stream, p->step_done[j], 0)) != cudaSuccess)
    return fail(e);
  const void *src[3] = {h_x, h_logits, h_dout};
  const int kind[3] = {kSlotX, kSlotLogits, kSlotDout};
  for (int i = 0; i < 3; ++i)
    if (sz[kind[i]] > 0 &&
        (e = cudaMemcpyAsync(sl[kind[i]], src[i], sz[kind[i]], cudaMemcpyHostToDevice,
                             p->in_stream)) != cudaSuccess)
      return fail(e);
  if ((e = cudaEventRecord(p->in_ready[j], p->in_stream)) != cudaSuccess) return fail(e);
  // compute: after the inputs landed and the slot's results of two steps back
  // were copied out
  if ((e = cudaStreamWaitEvent(s, p->in_ready[j], 0)) != cudaSuccess) return fail(e);
  if (p->out_used[j] && (e = cudaStreamWaitEvent(s, p->out_done[j], 0)) != cudaSuccess)
    return fail(e);
  Io io;
  io.x = reinterpret_cast<const uint16_t *>(sl[kSlotX]);
  io.logits = reinterpret_cast<const float *>(sl[kSlotLogits]);
  io.dout = reinterpret_cast<const uint16_t *>(sl[kSlotDout]);
  io.out = reinterpret_cast<uint16_t *>(sl[kSlotOut]);
  io.dx = reinterpret_cast<uint16_t *>(sl[kSlotDx]);
  io.d_logits = reinterpret_cast<float *>(sl[kSlotDLogits]);
  CALL(forward(p->view, io, wi, wo, bi, bo, expert_bias, s, nullptr, nullptr));
  CALL(backward(p->view, io, wi, wo, s, nullptr, nullptr));
  if ((e = cudaEventRecord(p->step_done[j], s)) != cudaSuccess) return fail(e);
  // results
  if ((e = cudaStreamWaitEvent(p->out_stream, p->step_done[j], 0)) != cudaSuccess) return fail(e);
  void *dst[3] = {h_out, h_dx, h_d_logits};
  const int okind[3] = {kSlotOut, kSlotDx, kSlotDLogits};
  for (int i = 0; i < 3; ++i)
    if (sz[okind[i]] > 0 &&
        (e = cudaMemcpyAsync(dst[i], sl[okind[i]], sz[okind[i]], cudaMemcpyDeviceToHost,
                             p->out_stream)) != cudaSuccess)
      return fail(e);
  if ((e = cudaEventRecord(p->out_done[j], p->out_stream)) != cudaSuccess) return fail(e);
  p->out_used[j] = true;
  ++p->steps;
  return MOE_OK;
}

moe_status_t moe_layer_pipeline_join(moe_layer_pipeline *p, moe_stream_t stream) {
  set_error("");
  if (p == nullptr) {
    set_error("moe_layer_pipeline_join: null pipeline");
    return MOE_ERR_INVALID_ARG;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  for (int j = 0; j < 2; ++j) {
    if (!p->out_used[j]) continue;
    const cudaError_t e = cudaStreamWaitEvent(s, p->out_done[j], 0);
    if (e != cudaSuccess) {
      set_error("moe_layer_pipeline_join: %s", cudaGetErrorString(e));
      return MOE_ERR_CUDA;
    }
  }
  return MOE_OK;
}

moe_status_t moe_layer_pipeline_sync(moe_layer_pipeline *p) {
  set_error("");
  if (p == nullptr) {
    set_error("moe_layer_pipeline_sync: null pipeline");
    return MOE_ERR_INVALID_ARG;
  }
  cudaError_t e = cudaStreamSynchronize(p->in_stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(p->out_stream);
  if (e != cudaSuccess) {
    set_error("moe_layer_pipeline_sync: %s", cudaGetErrorString(e));
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

}  // extern "C"
