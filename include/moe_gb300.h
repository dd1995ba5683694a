/*
 * moe_gb300.h -- C ABI of the GB300 (sm_103a) MoE expert-layer library
 * (libmoe_gb300.so).
 *
 * The layer is the router -> permutation -> grouped-GEMM SwiGLU FFN ->
 * combine block of TransformerEngine PR #2912, "[JAX] Add an MoE Block
 * (Layer) that compound router, permutation, groupedGEMM and communication"
 * (TE-2912 below), on one GPU without the expert-parallel all-to-all, plus
 * the chunked-K partial-sum grouped GEMM of MaxText PR #4295, "Overlap moe
 * comms with collective matmul" (MT-4295 below).
 *
 * Conventions shared by every call
 *   - Every tensor argument is DEVICE memory owned by the caller; the library
 *     never allocates, frees or retains a pointer after the call returns.
 *   - Matrices are dense row-major with an explicit leading dimension (in
 *     elements).  bf16 tensors are passed as uint16_t (bf16 bit patterns).
 *     bf16 matrices need ld % 8 == 0 and 16-byte aligned base pointers.
 *   - Every call enqueues its kernels on `stream` and returns without a host
 *     synchronisation.  A non-OK status means nothing was enqueued, except
 *     MOE_ERR_CUDA, which reports a failed launch (text via moe_last_error()).
 *   - Device-side faults are never raised.  Kernels that can meet bad data
 *     (an expert id out of range, a wait that runs past its time limit) write
 *     a MOE_ERR_* code into the optional caller-provided int32 `dev_status`
 *     word (first error wins, 0 = no error) and skip the bad item; the caller
 *     reads the word after synchronising.
 *   - Group layout: experts own contiguous row ranges of the permuted
 *     matrices, group e = rows [group_offsets[e], group_offsets[e+1]).
 *     group_offsets lives on the device and is read by the kernels directly:
 *     ragged sizes never travel to the host.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *moe_stream_t;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* null pointer, negative size, ld too small, ... */
  MOE_ERR_UNSUPPORTED = 2, /* valid but outside what the kernels handle (sizes, alignment) */
  MOE_ERR_CUDA = 3,        /* a CUDA launch or runtime call failed */
  MOE_ERR_TIMEOUT = 4,     /* device word only: a bounded wait ran out */
  MOE_ERR_DEVICE = 5       /* device word only: bad data met on the device */
} moe_status_t;

enum { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 };
enum { MOE_DTYPE_BF16 = 0, MOE_DTYPE_F32 = 1 };
enum { MOE_EPI_NONE = 0, MOE_EPI_SWIGLU_FWD = 1, MOE_EPI_SWIGLU_BWD = 2 };
/* 8-bit float formats (OCP): E4M3FN (max 448, no infinities), E5M2 (max 57344) */
enum { MOE_FP8_E4M3 = 0, MOE_FP8_E5M2 = 1 };
/* row orders of block-scale atoms (moe_mx_quantize) */
enum { MOE_MX_ROWS_PLAIN = 0, MOE_MX_ROWS_GROUPED = 1, MOE_MX_ROWS_SWIGLU = 2,
       MOE_MX_ROWS_TILES = 3 };

/* Static description of a status code. */
const char *moe_status_string(int status);
/* Message of the last failing call made by this host thread ("" if none). */
const char *moe_last_error(void);
/* Library ABI version (major*100 + minor); 200 since moe_rows_cap takes the capacity. */
int moe_version(void);

/*
 * Failure detection (no counterpart on the pages).  Every wait inside the
 * grouped-GEMM kernels (pipeline barriers between the copy, tensor-core and
 * epilogue roles) gives up after this many nanoseconds: the kernel then winds
 * down without faulting, frees its tensor memory and writes MOE_ERR_TIMEOUT to
 * dev_status, and the CUDA context stays usable.  Default 2 s; accepted range
 * 1 ms .. 600 s (else MOE_ERR_INVALID_ARG).  Applies to launches made after the
 * call, process-wide.
 */
moe_status_t moe_set_wait_limit_ns(uint64_t limit_ns);
uint64_t moe_wait_limit_ns(void);
/*
 * Test hook for the above: while enabled, the grouped-GEMM kernels launched
 * issue no operand loads, so their first pipeline wait runs out.  Only tests
 * use it.
 */
void moe_test_stall_loads(int enable);

/*
 * Worst-case number of permuted rows: min(T*k, E*capacity) + E*(align-1)
 * (capacity <= 0: T*k kept assignments; align <= 1: no padding rows).
 * TE-2912, review thread on recv_buffer_rows ("align_size > 0 + EP are
 * combined"): aligned group sizes can add up to align-1 rows per expert;
 * with token dropping no expert keeps more than `capacity` assignments.
 * Returns -1 for T < 0, E <= 0 or k <= 0.
 */
int64_t moe_rows_cap(int T, int E, int k, int align, int capacity);

/* Bytes of device workspace that moe_permute needs for T tokens and E experts. */
size_t moe_permute_workspace_bytes(int T, int E);

/*
 * moe_route_topk -- top-k expert selection and routing weights.
 * TE-2912, Description: the fused router, "top-K with optional
 * grouped/sigmoid scoring (for DSv3 workload)"; the router's group_topk
 * argument (the commit passing None as group_topk).
 *   logits    fp32 [T, ld_logits >= E]      router logits
 *   k         1 <= k <= min(E, 16); E <= 256
 *   score_fn  MOE_SCORE_SOFTMAX: softmax over all E experts;
 *             MOE_SCORE_SIGMOID: 1/(1+exp(-logit)) per expert
 *   renorm    nonzero: divide the k selected scores by their sum
 *   expert_bias fp32 [E] or NULL: DeepSeek-V3's per-expert selection bias
 *             (TE-2912, the expert_bias residual; MaxText PR #2579 "Onboard
 *             explicit sharding to deepseek", pre-bias logits): experts are
 *             ranked by the fp32 sum logit + bias, weights use the logits
 *   num_groups, topk_group  group-limited selection when num_groups > 1
 *             (0 or 1: off): the E experts form num_groups contiguous groups
 *             (E % num_groups == 0); a group scores the fp32 sum of its
 *             m = k / topk_group largest keys, added from the largest down
 *             (topk_group must divide k, m <= E / num_groups); only experts of
 *             the topk_group best groups (ties to the lower group id) compete
 *   topk_idx  int32 [T, k] out: experts by descending key, ties to the lower id
 *   topk_w    fp32  [T, k] out: the selected (renormalised) scores, same order
 * Selection compares fp32 keys (the score maps are monotone); a NaN key ranks
 * below every number.
 */
moe_status_t moe_route_topk(const float *logits, int64_t ld_logits, int T, int E, int k,
                            int score_fn, int renorm, const float *expert_bias, int num_groups,
                            int topk_group, int32_t *topk_idx, float *topk_w,
                            moe_stream_t stream);

/*
 * moe_aux_loss -- auxiliary load-balancing loss of the routing decision.
 * TE-2912, Description ("optional auxiliary load-balancing loss") and the
 * sequence diagram (the block returns it beside the output).  The pages do
 * not print the formula; this is the Switch-Transformer / DeepSeek-V3 form:
 *     loss = coeff * sum_e f_e P_e,   f_e = E / (k T) * counts[e],
 *     P_e  = mean over tokens of p[t, e],
 * p = softmax of the logits over all E (MOE_SCORE_SOFTMAX) or the sigmoid
 * scores divided by their sum over all E (MOE_SCORE_SIGMOID).
 *   logits      fp32 [T, ld_logits >= E]; topk_idx int32 [T, k] (the routing
 *               decision, before any capacity drop)
 *   counts      int32 [E] out: choices of each expert
 *   probs_mean  fp32 [E] out: P_e
 *   loss        fp32 [1] out (device)
 *   workspace   >= moe_aux_loss_workspace_bytes(T, E) bytes of device memory
 *               (4-byte aligned), caller-owned scratch
 * fp32 sums in a fixed order: the result does not vary between runs.
 * E <= 256, k <= 16.  T = 0 gives zeros.
 */
size_t moe_aux_loss_workspace_bytes(int T, int E);
moe_status_t moe_aux_loss(const float *logits, int64_t ld_logits, int T, int E, int k,
                          int score_fn, const int32_t *topk_idx, float coeff, int32_t *counts,
                          float *probs_mean, float *loss, void *workspace,
                          size_t workspace_bytes, moe_stream_t stream);

/*
 * moe_aux_loss_bwd -- logit gradient of moe_aux_loss (counts fixed), scaled
 * by d_loss (host scalar):
 *     softmax:  d_l[t, e] = g p_e (f_e - c_t)
 *     sigmoid:  d_l[t, e] = g s_e (1 - s_e) / S_t (f_e - c_t)
 * with g = d_loss coeff / T, c_t = sum_j f_j p[t, j], S_t = sum_j s_j.
 *   counts    int32 [E] as moe_aux_loss wrote them
 *   d_logits  fp32 [T, ld_dlogits >= E]: written, or added to when
 *             accumulate != 0 (e.g. on top of moe_route_topk_bwd's output)
 */
moe_status_t moe_aux_loss_bwd(const float *logits, int64_t ld_logits, int T, int E, int k,
                              int score_fn, const int32_t *counts, float coeff, float d_loss,
                              float *d_logits, int64_t ld_dlogits, int accumulate,
                              moe_stream_t stream);

/*
 * moe_route_topk_bwd -- gradient of the routing weights w.r.t. the logits,
 * the selection held fixed (TE-2912, sequence diagram: the block's backward
 * carries d_w back to the gate kernel):
 *   softmax, renorm:   d_l[i_j] = w_j (dw_j - c),   c = sum_j dw_j w_j
 *   softmax:           d_l[e] = p_e ([e = i_j] dw_j - c) for all e
 *   sigmoid, renorm:   d_l[i_j] = s_j (1 - s_j) (dw_j - c) / sum_m s_m
 *   sigmoid:           d_l[i_j] = dw_j s_j (1 - s_j)
 * other entries 0.  logits, topk_idx, topk_w as moe_route_topk produced them;
 * d_topk_w fp32 [T, k]; d_logits fp32 [T, ld_dlogits >= E] out (every entry
 * written).  E <= 256, k <= 16.
 */
moe_status_t moe_route_topk_bwd(const float *logits, int64_t ld_logits, const int32_t *topk_idx,
                                const float *topk_w, const float *d_topk_w, int T, int E, int k,
                                int score_fn, int renorm, float *d_logits, int64_t ld_dlogits,
                                moe_stream_t stream);

/*
 * moe_permute -- group the T*k (token, slot) assignments by expert and gather
 * the token rows into per-expert contiguous groups.
 * TE-2912, review thread on _combine_bwd (pure-JAX path): the flat
 * assignment a = t*k + j is ordered by a stable argsort on its expert
 * (sorted_indices), i.e. by (expert, token); group_sizes are the aligned
 * counts when align_size > 0 (thread on recv_buffer_rows); token dropping
 * (MaxText PR #2319, "[Draft] Integrate TE/JAX GroupedGEMM for MoE", Tests)
 * keeps the first `capacity` assignments of each expert in that order.
 *   x              bf16 [T, ldx >= d]            token activations (d % 8 == 0)
 *   topk_idx       int32 [T, k]                  expert ids, distinct within a token
 *   align          group-size multiple (0 or 1: none)
 *   capacity       per-expert kept assignments (<= 0: no dropping)
 *   x_sorted       bf16 [rows_cap, ld_xs >= d] out: row p = x[token of
 *                  sorted_to_flat[p]]; padding rows are zero; rows >= R
 *                  (R = group_offsets[E]) are not written
 *   rows_cap       rows of x_sorted / sorted_to_flat,
 *                  >= moe_rows_cap(T, E, k, align, capacity)
 *   group_sizes    int32 [E] out: aligned group sizes
 *   kept_counts    int32 [E] out: kept (not dropped) assignments per expert
 *   group_offsets  int32 [E+1] out: exclusive scan of group_sizes
 *   sorted_to_flat int32 [rows_cap] out: flat assignment of row p, -1 on
 *                  padding rows and on rows >= R
 *   flat_to_sorted int32 [T*k] out: row of assignment a, -1 if dropped
 *   workspace      device scratch of >= moe_permute_workspace_bytes(T, E) bytes
 *                  (contents on entry are ignored)
 * An out-of-range expert id or a repeated expert within one token sets
 * MOE_ERR_DEVICE in dev_status; such assignments are treated as dropped.
 */
moe_status_t moe_permute(const uint16_t *x, int64_t ldx, const int32_t *topk_idx, int T, int d,
                         int E, int k, int align, int capacity, uint16_t *x_sorted,
                         int64_t ld_xs, int64_t rows_cap, int32_t *group_sizes,
                         int32_t *kept_counts, int32_t *group_offsets,
                         int32_t *sorted_to_flat, int32_t *flat_to_sorted, void *workspace,
                         size_t workspace_bytes, int32_t *dev_status, moe_stream_t stream);

/*
 * moe_permute_noalloc -- moe_permute without a caller-provided workspace.
 * The pages have no counterpart of this call; it exists for callers that
 * cannot allocate device memory where they permute (plugin-style interfaces
 * that receive only their input and output buffers, or processes whose device
 * memory is reserved up front by their own pool, where an extra cudaMalloc
 * fails or fragments the pool).  Arguments and results are those of
 * moe_permute without `workspace` / `workspace_bytes`.
 * Scratch: a fixed 128 KB array of library-owned device memory, held by every
 * GPU that loads the library until the process exits.  Sizes that need more
 * (moe_permute_workspace_bytes(T, E) > 131072: with E = 256, T > 32512;
 * E <= 64 always fits) return MOE_ERR_UNSUPPORTED.  The call allocates and frees nothing.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  After cudaDeviceReset() the array belongs to the device's new
 * context, and the first call made there looks the address up again (make it
 * before any capture too).  All calls share the array: calls whose kernels
 * overlap on the GPU race and must be serialised by the caller.
 */
moe_status_t moe_permute_noalloc(const uint16_t *x, int64_t ldx, const int32_t *topk_idx, int T,
                                 int d, int E, int k, int align, int capacity,
                                 uint16_t *x_sorted, int64_t ld_xs, int64_t rows_cap,
                                 int32_t *group_sizes, int32_t *kept_counts,
                                 int32_t *group_offsets, int32_t *sorted_to_flat,
                                 int32_t *flat_to_sorted, int32_t *dev_status,
                                 moe_stream_t stream);

/*
 * moe_gmm -- grouped GEMM over ragged per-expert row groups (tcgen05 tensor
 * cores, fp32 accumulation).  For every row r of group e:
 *     S[r, :] = A[r, :] . B_e  (+ partial_sum[r, :]) (+ bias_e)
 * TE-2912: the grouped_gemm calls of the expert FFN (Description), with
 * [wi_0 | wi_1] fused into one up-projection (wi-fusion commit); MT-4295,
 * review threads on the gmm kernel: `transpose_rhs` and the in-place
 * `partial_sum`.
 *   A         bf16 [rows_cap, lda >= K]   permuted activations
 *   B         bf16 expert weights, expert e at B + e*stride_b:
 *               trans_b == 0: B_e is [K, N] row-major (ldb >= N)   S = A . B_e
 *               trans_b != 0: B_e is [N, K] row-major (ldb >= K)   S = A . B_e^T
 *   group_offsets int32 [E+1] device; rows_cap bounds group_offsets[E]
 *   K, N      multiples of 8, > 0
 *   epilogue  MOE_EPI_NONE:       C = S, stored as c_dtype (bf16 or fp32)
 *             MOE_EPI_SWIGLU_FWD: N = 2F (F % 8 == 0); C = bf16(S) = H and
 *                                 C2 = bf16(silu(S[:, :F]) * S[:, F:]) = Act
 *                                 (C2 bf16 [rows_cap, ldc2 >= F])
 *             MOE_EPI_SWIGLU_BWD: S is dAct [., N = F]; aux = H bf16
 *                                 [rows_cap, ld_aux >= 2F]; C = bf16 dH
 *                                 [., 2F]: dH[:, :F] = S * u * s * (1 + g(1-s)),
 *                                 dH[:, F:] = S * silu(g), g = H[:, :F],
 *                                 u = H[:, F:], s = sigmoid(g)
 *   partial_sum fp32 [rows_cap, ld_ps >= N] or NULL (NONE / SWIGLU_FWD only);
 *             may alias C when c_dtype is fp32 and ld_ps == ldc (in place)
 *   bias      bf16 or NULL (NONE / SWIGLU_FWD only): expert e's N-vector at
 *             bias + e*stride_bias, added to every row of group e after the
 *             partial sum (SWIGLU_FWD: [gate | up] bias, before the SwiGLU)
 *   C         [rows_cap, ldc] (ldc >= N, or >= 2F for SWIGLU_BWD)
 *   Ct        bf16 or NULL (SWIGLU_FWD / SWIGLU_BWD only): the epilogue also
 *             writes a column-wise copy of its activation output in the padded
 *             group layout of moe_transpose_act, the K-major operand of the
 *             weight gradient (moe_tgmm_kt):
 *               SWIGLU_FWD: Act^T [F, ldct],  Ct[n, poff_e + i] = Act[off_e + i, n]
 *               SWIGLU_BWD: dH^T [2F, ldct], Ct[n, poff_e + i] = dH[off_e + i, n]
 *             with zeros in each group's padding up to its next multiple of 128
 *             columns; ldct >= moe_fp8_padded_rows(rows_cap, E), ldct % 8 == 0
 * Only rows r < group_offsets[E] are written.  E <= 256; A, B, C, C2, Ct, aux
 * and partial_sum 16-byte aligned; SWIGLU_FWD needs trans_b == 0.
 */
moe_status_t moe_gmm(const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
                     int64_t stride_b, int trans_b, const int32_t *group_offsets, int E,
                     int64_t rows_cap, int K, int N, int epilogue, const uint16_t *aux,
                     int64_t ld_aux, const float *partial_sum, int64_t ld_ps,
                     const uint16_t *bias, int64_t stride_bias, void *C, int c_dtype,
                     int64_t ldc, uint16_t *C2, int64_t ldc2, uint16_t *Ct, int64_t ldct,
                     int32_t *dev_status, moe_stream_t stream);

/*
 * moe_transpose_act -- column-wise bf16 copy of a permuted activation in the
 * padded group layout (see moe_fp8_padded_rows): xt[c, poff_e + i] =
 * x[group_offsets[e] + i, c] for the rows of group e, zeros up to poff_e+1.
 *   x   bf16 [rows_cap, ldx >= cols], cols % 8 == 0
 *   xt  bf16 [cols, ldxt >= moe_fp8_padded_rows(rows_cap, E)] out (columns
 *       [0, poff_E) written)
 * The K-major A operand of moe_tgmm_kt (MaxText PR #4295, Testing: tgmm).
 */
moe_status_t moe_transpose_act(const uint16_t *x, int64_t ldx, const int32_t *group_offsets,
                               int E, int64_t rows_cap, int cols, uint16_t *xt, int64_t ldxt,
                               moe_stream_t stream);

/*
 * moe_tgmm_kt -- moe_tgmm with A given as its column-wise copy At [M, ldat]
 * (moe_transpose_act of A); B bf16 [rows_cap, ldb] as in moe_tgmm, or with
 * b_colwise != 0 its column-wise copy Bt [N, ldb >= moe_fp8_padded_rows].
 * Reading operands K-major feeds the tensor cores faster than the row-major
 * operands of moe_tgmm.  Same result, zeros for empty experts, same W.
 */
moe_status_t moe_tgmm_kt(const uint16_t *At, int64_t ldat, const uint16_t *B, int64_t ldb,
                         int b_colwise, const int32_t *group_offsets, int E, int64_t rows_cap, int M, int N,
                         void *W, int w_dtype, int64_t ldw, int64_t stride_w, int accumulate,
                         int32_t *dev_status, moe_stream_t stream);

/*
 * moe_group_colsum -- per-expert column sums, the gradient of a bias that
 * every row of a group received (the expert-FFN biases: MT-4295, Testing,
 * `mlp_bias`; TE-2912, `has_wi_bias`):
 *     out[e, n] = sum over rows r of group e of G[r, n]
 *   summed in fp32 in a fixed order (the result does not vary between runs);
 *   G bf16 [rows_cap, ldg >= N] (16-byte aligned, ldg % 8 == 0), N % 8 == 0;
 *   out fp32 [E, ld_out >= N] (16-byte aligned, ld_out % 4 == 0; columns < N
 *   of every row written, empty experts get 0).  Rows at or past
 *   group_offsets[E] are not read.  E <= 65535.
 */
moe_status_t moe_group_colsum(const uint16_t *G, int64_t ldg, const int32_t *group_offsets,
                              int E, int64_t rows_cap, int N, float *out, int64_t ld_out,
                              moe_stream_t stream);

/* ------------------------------------------------------------------ FP8 --
 * Current tensor scaling for the FP8 expert GEMMs.  MaxText PR #2319
 * "[Draft] Integrate TE/JAX GroupedGEMM for MoE", review thread on the
 * quantizer settings of moe.py: current tensor scaling, float8_e4m3fn
 * forward, float8_e5m2 backward, 2x (row- and column-wise) quantization;
 * TE-2912, wi-fusion commit: one amax per expert for the fused weight.
 *   scale = fp8_max / amax (fp32; 1 when amax is 0 or not finite)
 *   code  = round-to-nearest-even(fp32(x * scale)), saturated to +-fp8_max
 *   value = code / scale
 */

/*
 * moe_fp8_amax -- amax[g] = max |x| over the rows of group g (NaN when one of
 *   them is NaN, 0 for a group with no rows).
 *   x        bf16 [rows, ldx >= cols] (16-byte aligned, ldx % 8 == 0, cols % 8 == 0)
 *   groups   1, or E for per-expert weights (rows % groups == 0: group g is
 *            rows [g * rows / groups, (g + 1) * rows / groups))
 *   group_offsets (groups == 1 only; may be NULL): only rows < group_offsets[E]
 *            are read (permuted activations)
 *   amax     fp32 [groups] out (device)
 */
moe_status_t moe_fp8_amax(const uint16_t *x, int64_t ldx, int64_t rows, int cols, int groups,
                          const int32_t *group_offsets, int E, float *amax,
                          moe_stream_t stream);

/*
 * moe_fp8_padded_rows -- columns of the column-wise copy of a grouped
 * activation with rows_cap rows: group e occupies columns [poff_e, poff_e +
 * size_e) with poff_e the sum of the previous sizes each rounded up to 128,
 * zeros up to the next group; the result is rows_cap + 127 E rounded up to 128.
 */
int64_t moe_fp8_padded_rows(int64_t rows_cap, int E);

/*
 * moe_fp8_quantize_act -- row-wise and column-wise codes of a permuted
 * activation (rows [0, group_offsets[E]) of x), one scale from amax[0].
 *   x        bf16 [rows_cap, ldx >= cols]; cols % 16 == 0
 *   q        uint8 [rows_cap, ldq >= cols] out (ldq % 16 == 0); rows past
 *            group_offsets[E] are not written
 *   qt       uint8 [cols, ldqt >= moe_fp8_padded_rows(rows_cap, E)] out
 *            (ldqt % 16 == 0): columns [0, poff_E) written, padding zero
 *   scale_inv fp32 [1] out: 1 / scale
 */
moe_status_t moe_fp8_quantize_act(const uint16_t *x, int64_t ldx, const int32_t *group_offsets,
                                  int E, int64_t rows_cap, int cols, int fmt, const float *amax,
                                  uint8_t *q, int64_t ldq, uint8_t *qt, int64_t ldqt,
                                  float *scale_inv, moe_stream_t stream);

/*
 * moe_fp8_quantize_weights -- per-expert codes of w bf16 [E, K, N]
 * (contiguous), scale of expert e from amax[e]:
 *   q  uint8 [E, K, N] out (row-wise), qt uint8 [E, N, K] out (transposed),
 *   scale_inv fp32 [E] out.  K % 16 == 0, N % 16 == 0.
 */
moe_status_t moe_fp8_quantize_weights(const uint16_t *w, int E, int K, int N, int fmt,
                                      const float *amax, uint8_t *q, uint8_t *qt,
                                      float *scale_inv, moe_stream_t stream);

/*
 * moe_gmm_fp8 -- moe_gmm on 8-bit float codes (tcgen05 kind::f8f6f4, fp32
 * accumulation), the row-wise copies of the 2x quantization:
 *     S[r, :] = (A_q[r, :] . B_q,e^T) * a_scale_inv[0] * b_scale_inv[e]
 * then the epilogue of moe_gmm (NONE, SWIGLU_FWD, SWIGLU_BWD; no partial sum,
 * no bias).
 *   A     uint8 codes [rows_cap, lda >= K] (format a_fmt), K-major
 *   B     uint8 codes [E, N, K] K-major: row n of expert e at B + e*stride_b +
 *         n*ldb (the transposed copy for [K, N] weights, the row-wise copy of
 *         a [N, K] weight for dgrad); SWIGLU_FWD: rows [0, F) gate, [F, 2F) up
 *   a_scale_inv fp32 [1], b_scale_inv fp32 [E] (device)
 *   amax_out  fp32 [1] (device) or NULL: set to max |x| over the values the
 *             epilogue writes (Act for SWIGLU_FWD, dH for SWIGLU_BWD, C for
 *             NONE; NaN values are skipped; 0 with no rows), the amax that
 *             quantizes them next (no extra pass)
 *   K, lda, ldb, stride_b multiples of 16; other arguments as moe_gmm.
 * FP8 recipe (TE-2912, the fused up-projection; MaxText PR #2319, quantizer
 * settings): E4M3 operands forward, E5M2 gradients backward.
 */
moe_status_t moe_gmm_fp8(const uint8_t *A, int64_t lda, int a_fmt, const float *a_scale_inv,
                         const uint8_t *B, int64_t ldb, int64_t stride_b, int b_fmt,
                         const float *b_scale_inv, const int32_t *group_offsets, int E,
                         int64_t rows_cap, int K, int N, int epilogue, const uint16_t *aux,
                         int64_t ld_aux, void *C, int c_dtype, int64_t ldc, uint16_t *C2,
                         int64_t ldc2, float *amax_out, int32_t *dev_status,
                         moe_stream_t stream);

/*
 * moe_tgmm_fp8 -- moe_tgmm on the column-wise copies of two permuted
 * activations (moe_fp8_quantize_act's qt):
 *     W_e = (At_e . Bt_e^T) * a_scale_inv[0] * b_scale_inv[0]
 * where At_e / Bt_e are columns [poff_e, poff_e+1) of At [M, ldat] and Bt
 * [N, ldbt] (group e's rows, zero padded to a multiple of 128); an expert
 * without rows gets zeros (or nothing when accumulating).  ldat, ldbt >=
 * moe_fp8_padded_rows(rows_cap, E); W as moe_tgmm.
 */
moe_status_t moe_tgmm_fp8(const uint8_t *At, int64_t ldat, int a_fmt, const float *a_scale_inv,
                          const uint8_t *Bt, int64_t ldbt, int b_fmt, const float *b_scale_inv,
                          const int32_t *group_offsets, int E, int64_t rows_cap, int M, int N,
                          void *W, int w_dtype, int64_t ldw, int64_t stride_w, int accumulate,
                          int32_t *dev_status, moe_stream_t stream);

/* --------------------------------------------------- block-scaled FP8 --
 * MXFP8: one power-of-two scale per 32 consecutive elements along the
 * contraction axis, read by the tensor cores themselves (tcgen05.mma
 * kind::mxf8f6f4.block_scale).  TE-2912, wi-fusion commit, FP8 note (the
 * block-scaled recipes keep one scale per block); the arithmetic is the OCP
 * Microscaling (MX) v1.0 definition: scale 2^s, s = floor(log2 amax) - emax
 * (8 for E4M3, 15 for E5M2) clamped to [-127, 127], stored as the E8M0 code
 * s + 127; code = round-to-nearest-even of x / 2^s, saturated; a block of
 * zeros takes code 0, a block holding a NaN or infinity the NaN scale 0xFF
 * (and zero codes).
 * Scales are kept in 512-byte atoms of 128 rows x 4 blocks (128 columns):
 * row r0 + 32 r1 (r0 < 32, r1 < 4), block j at byte 16 r0 + 4 r1 + j; atom
 * (ar, ac) at byte (ar * cols / 128 + ac) * 512.  The atom row of a matrix
 * row follows how the GEMMs tile it (row_map).  A operands come in tiles of
 * 128 rows, B operands in tiles of 192 rows (the GEMMs' 192-column output
 * tiles), each B tile taking two atom rows (padded row 256 t + i):
 *   MOE_MX_ROWS_PLAIN    r / 128: the column-wise activation copy that is a
 *                        weight gradient's A operand
 *   MOE_MX_ROWS_GROUPED  permuted activations (A operands): the rows of group
 *                        e start at atom row poff_e / 128, poff_e the group
 *                        starts rounded up to 128 (moe_fp8_padded_rows layout)
 *   MOE_MX_ROWS_TILES    B operands: E equal groups of G = rows / E rows (the
 *                        experts' weights, or E = 1: a weight gradient's B
 *                        copy); row n of group e in tile t = n / 192 at
 *                        padded row 256 (e ceil(G/192) + t) + n % 192
 *   MOE_MX_ROWS_SWIGLU   the fused [gate | up] up-projection weight, 2F rows,
 *                        in SwiGLU tiles: tile t holds gate rows [96t, 96t +
 *                        96) then up rows [F + 96t, F + 96t + 96)
 */

/* Bytes of scale atoms for a [rows, cols] matrix (cols % 128 == 0); 0 for bad arguments. */
size_t moe_mx_scale_bytes(int64_t rows, int cols, int row_map, int E);

/*
 * moe_mx_quantize -- block-scaled codes of x bf16 [rows, ldx >= cols]
 * (blocks along each row), codes q uint8 [rows, ldq >= cols] (ldq % 16 == 0),
 * scales sf (>= moe_mx_scale_bytes bytes, device).  GROUPED: group_offsets
 * int32 [E + 1] on the device, rows at or past group_offsets[E] are not
 * written; scale bytes of padding rows are not written either.
 */
moe_status_t moe_mx_quantize(const uint16_t *x, int64_t ldx, int64_t rows, int cols, int fmt,
                             int row_map, const int32_t *group_offsets, int E, uint8_t *q,
                             int64_t ldq, uint8_t *sf, size_t sf_bytes, moe_stream_t stream);

/*
 * moe_mx_quantize_2x -- both block-scaled copies of a grouped bf16 matrix x
 * [rows, ldx >= cols] from one read (the GEMM operands that the forward /
 * dgrad and the weight gradient take from one tensor):
 *   q   (or NULL) row-wise codes [rows, ldq >= cols], blocks of 32 along each
 *       row; scales sfq in the atoms of q_map: GROUPED (permuted activations,
 *       groups of group_offsets) or TILES (E equal groups: weights)
 *   qt  (or NULL) column-wise codes [cols, ldqt >= qt_cols]: qt[c, poff_e + i]
 *       = code of x[group_offsets[e] + i, c], blocks of 32 along each group's
 *       rows from its first one, zeros past the group up to its next multiple
 *       of 128 (poff_e: the group starts rounded up to 128, the layout of
 *       moe_transpose_act); scales sfqt for the [cols, qt_cols] matrix in the
 *       atoms of qt_map: PLAIN (a weight gradient's A), TILES with one group
 *       (a B operand) or SWIGLU (the up-projection's transposed weight)
 *   group_offsets int32 [E+1] on the device (TILES: 0, G, 2G, ... with G =
 *   rows / E); qt_cols % 128 == 0 and at least the padded extent of the
 *   groups (e.g. moe_fp8_padded_rows(rows, E); E*G for 128-aligned equal
 *   groups): column blocks past qt_cols are not written.
 * Codes and scales are those of moe_mx_quantize of the two matrices.
 */
moe_status_t moe_mx_quantize_2x(const uint16_t *x, int64_t ldx, int64_t rows, int cols, int fmt,
                                const int32_t *group_offsets, int E, uint8_t *q, int64_t ldq,
                                int q_map, uint8_t *sfq, size_t sfq_bytes, uint8_t *qt,
                                int64_t ldqt, int qt_cols, int qt_map, uint8_t *sfqt,
                                size_t sfqt_bytes, moe_stream_t stream);

/*
 * moe_gmm_mx -- moe_gmm on block-scaled codes (fp32 accumulation of
 * (a * 2^sa) (b * 2^sb) in the tensor cores; 256 x 192 output tiles):
 *   A    uint8 codes [rows_cap, lda >= K] with scales sfa from moe_mx_quantize
 *        (GROUPED, E groups of group_offsets)
 *   B    uint8 codes, K-major: row n of expert e at B + e*stride_b + n*ldb,
 *        scales sfb from moe_mx_quantize of either
 *          sfb_by_cols = 0: the [E*N, K] matrix (stride_b = N*ldb), TILES
 *            with E groups;
 *          sfb_by_cols = 1: the [N, E*K] matrix of the transposed weights
 *            (expert e's K columns at e*K, stride_b = K), SWIGLU for the
 *            SWIGLU_FWD epilogue (N = 2F), else TILES with one group
 *   K % 128 == 0, N % 32 == 0 (SWIGLU_FWD: N = 2F, F % 32 == 0, and
 *   sfb_by_cols = 1); epilogues, aux, C, C2 as moe_gmm (no partial sum, no bias).
 */
moe_status_t moe_gmm_mx(const uint8_t *A, int64_t lda, const uint8_t *sfa, int a_fmt,
                        const uint8_t *B, int64_t ldb, int64_t stride_b, const uint8_t *sfb,
                        int sfb_by_cols, int b_fmt,
                        const int32_t *group_offsets, int E, int64_t rows_cap, int K, int N,
                        int epilogue, const uint16_t *aux, int64_t ld_aux, void *C, int c_dtype,
                        int64_t ldc, uint16_t *C2, int64_t ldc2, int32_t *dev_status,
                        moe_stream_t stream);

/*
 * moe_tgmm_mx -- moe_tgmm on block-scaled codes of the column-wise copies
 * (moe_transpose_act layout, P = moe_fp8_padded_rows(rows_cap, E); blocks of
 * 32 along the expert's rows, zeros in its padding): At [M, P] quantized
 * PLAIN, Bt [N, P] quantized TILES with one group.  M % 128 == 0, N % 32 ==
 * 0; W as moe_tgmm (exact zeros for experts without rows, or W kept when
 * accumulating).
 */
moe_status_t moe_tgmm_mx(const uint8_t *At, int64_t ldat, const uint8_t *sfa, int a_fmt,
                         const uint8_t *Bt, int64_t ldbt, const uint8_t *sfb, int b_fmt,
                         const int32_t *group_offsets, int E, int64_t rows_cap, int M, int N,
                         void *W, int w_dtype, int64_t ldw, int64_t stride_w, int accumulate,
                         int32_t *dev_status, moe_stream_t stream);

/*
 * moe_tgmm -- weight-gradient grouped GEMM, ragged along the contraction:
 *     W_e = A_e^T . B_e   (+ W_e when accumulate),  A_e / B_e = rows of group e
 * MT-4295, Testing: "TGMM with zero-initialized empty expert groups": an
 * expert with no rows gets exact zeros (or keeps W_e when accumulating).
 *   A  bf16 [rows_cap, lda >= M];  B  bf16 [rows_cap, ldb >= N];  M, N % 8 == 0
 *   W  expert e at W + e*stride_w, [M, ldw >= N] row-major, w_dtype bf16 or
 *      fp32 (accumulate requires fp32); E <= 256; A, B, W 16-byte aligned
 */
moe_status_t moe_tgmm(const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
                      const int32_t *group_offsets, int E, int64_t rows_cap, int M, int N,
                      void *W, int w_dtype, int64_t ldw, int64_t stride_w, int accumulate,
                      int32_t *dev_status, moe_stream_t stream);

/*
 * moe_combine -- routing-weighted un-permute:
 *     out[t] = sum_j w[t,j] * Y[flat_to_sorted[t*k+j]]   (slots with -1 skipped)
 * summed in fp32 in slot order.  With topk_w == NULL every weight is 1, which
 * is the backward of moe_permute's row gather (dispatch backward).
 * TE-2912, review thread on _combine_bwd: the forward combine is
 * output[B,E] = sum_K intermediate[B,K,E] * weights[B,K] after the un-sort.
 *   Y bf16 [rows, ldy >= d]; out bf16 [T, ldo >= d]; d % 8 == 0
 */
moe_status_t moe_combine(const uint16_t *Y, int64_t ldy, const int32_t *flat_to_sorted,
                         const float *topk_w, int T, int k, int d, uint16_t *out, int64_t ldo,
                         moe_stream_t stream);

/*
 * moe_unpermute_bwd -- backward of moe_combine (TE-2912, review thread on
 * _combine_bwd: d_intermediate = d_output * w, d_w = sum over hidden of
 * d_output * intermediate, zero on padding, placed back in sorted order):
 *     dY[p]      = w[t,j] * d_out[t]        for p = flat_to_sorted[t*k+j] >= 0
 *     d_topk_w[t,j] = <d_out[t], Y[p]>   (0 for dropped slots)
 *     dY[p]      = 0 for padding rows p < group_offsets[E]
 *   d_out bf16 [T, ld_dout]; Y bf16 [rows_cap, ldy]; dY bf16 [rows_cap, ld_dy];
 *   sorted_to_flat int32 [rows_cap]; group_offsets int32 [E+1]
 */
moe_status_t moe_unpermute_bwd(const uint16_t *d_out, int64_t ld_dout, const uint16_t *Y,
                               int64_t ldy, const int32_t *flat_to_sorted,
                               const int32_t *sorted_to_flat, const int32_t *group_offsets,
                               const float *topk_w, int T, int k, int d, int E,
                               int64_t rows_cap, uint16_t *dY, int64_t ld_dy, float *d_topk_w,
                               moe_stream_t stream);

/* ---------------------------------------------------- expert parallelism --
 * Dispatch of the permuted rows to the shards that own their experts with a
 * ragged all-to-all, and the local re-sort after it: TE-2912, sequence
 * diagram (_dispatch -> ragged_all_to_all -> local permute; _combine the
 * reverse; the backward re-runs the same exchanges with swapped roles) and
 * its helpers compute_ragged_all_to_all_params / local_permute_after_a2a /
 * local_unpermute_before_a2a; the receive-buffer bound of the recv_buffer_rows
 * review thread.
 * num_ep shards; shard r owns the El = E / num_ep experts [r*El, (r+1)*El).
 * Every shard permutes its own tokens over all E experts (moe_permute), so
 * the rows it sends to shard r are one contiguous block of its permuted
 * buffer.  The exchange itself is the caller's collective (e.g. an NCCL
 * all-to-all with these sizes); it needs the sizes on the host, so
 * group_sizes of every shard (an all-gather of moe_permute's group_sizes) are
 * HOST arrays here.
 */

/* Rows of the receive buffer (and of the local buffer) that suffice for any
 * routing of T tokens per shard: num_ep * (T * min(k, El) + El * (align - 1));
 * -1 for bad arguments. */
int64_t moe_ep_recv_rows_cap(int T, int num_ep, int E, int k, int align);

/*
 * moe_ep_a2a_params -- sizes and offsets of the exchange for shard `shard`
 * (host computation, no GPU work).
 *   group_sizes  int32 [num_ep, E] HOST: row s = the group sizes of shard s
 *   send_off, send_sz  int64 [num_ep] out: rows [send_off[r], +send_sz[r]) of
 *                this shard's permuted buffer go to shard r
 *   out_off      int64 [num_ep] out: where those rows start in shard r's
 *                receive buffer
 *   recv_off, recv_sz  int64 [num_ep] out: the rows from shard s land at
 *                [recv_off[s], +recv_sz[s]) of this shard's receive buffer
 *                (source-major, each source's rows by local expert)
 * The reverse exchange (combine, dispatch backward) sends (recv_off, recv_sz)
 * and receives (send_off, send_sz).  E % num_ep == 0, num_ep <= 1024, sizes
 * >= 0, else MOE_ERR_INVALID_ARG.
 */
moe_status_t moe_ep_a2a_params(const int32_t *group_sizes, int num_ep, int E, int shard,
                               int64_t *send_off, int64_t *send_sz, int64_t *out_off,
                               int64_t *recv_off, int64_t *recv_sz);

/*
 * moe_ep_local_layout -- the local permute after the exchange (host
 * computation).  Chunk (source s, local expert le) holds shard s's rows of
 * expert shard*El + le, in their order; the local buffer is expert-major
 * (local expert 0's rows from every source in source order, then local
 * expert 1's, ...), the layout the grouped GEMMs take.
 *   fwd_src, fwd_dst, fwd_len  int64 [num_ep * El] out: the chunks in
 *        receive-buffer order (chunk s*El + le): moe_sort_chunks receive -> local
 *   inv_src, inv_dst, inv_len  int64 [num_ep * El] out: the same chunks in
 *        local-buffer order (chunk le*num_ep + s): moe_sort_chunks local -> receive
 *   local_offsets  int32 [El + 1] out: group offsets of the local experts
 * Aligned group sizes stay aligned: each source pads its own groups.
 */
moe_status_t moe_ep_local_layout(const int32_t *group_sizes, int num_ep, int E, int shard,
                                 int64_t *fwd_src, int64_t *fwd_dst, int64_t *fwd_len,
                                 int64_t *inv_src, int64_t *inv_dst, int64_t *inv_len,
                                 int32_t *local_offsets);

/*
 * moe_sort_chunks -- move rows chunk by chunk (device): for every chunk c and
 * 0 <= i < len[c], row src_off[c] + i of src is copied to row dst_off[c] + i
 * of dst.  src_off, dst_off, len: int64 [n_chunks] DEVICE arrays, src_off
 * non-decreasing, chunks disjoint in src and in dst; rows: src rows to scan
 * (>= the end of the last chunk).  src, dst bf16 (16-byte aligned), d, ld_src,
 * ld_dst multiples of 8.  Rows of dst outside every chunk are not written.
 */
moe_status_t moe_sort_chunks(const uint16_t *src, int64_t ld_src, uint16_t *dst, int64_t ld_dst,
                             int d, const int64_t *src_off, const int64_t *dst_off,
                             const int64_t *len, int n_chunks, int64_t rows,
                             moe_stream_t stream);

/* ------------------------------------------------------------------------
 * The whole layer: one forward and one backward call
 * ------------------------------------------------------------------------
 * moe_layer_forward / moe_layer_backward run the layer's sequence of the
 * calls above on `stream` (TE-2912, sequence diagram: route -> permute ->
 * grouped GEMM (up, SwiGLU) -> grouped GEMM (down) -> combine, and its VJP:
 * combine backward -> router backward -> dgrad (down, SwiGLU backward) ->
 * tgmm (dWo) -> dgrad (up) -> tgmm (dWi) -> dispatch backward), every
 * intermediate in one caller-owned device workspace whose layout the library
 * plans.  The options are those of the calls above: group-limited routing,
 * DeepSeek-V3's selection bias (MaxText PR #2579, "Onboard explicit sharding
 * to deepseek"), the auxiliary load-balancing loss, align_size padding,
 * capacity dropping, K-chunked up-projection (MT-4295), expert-FFN biases,
 * FP8 current scaling or block-scaled (MXFP8) GEMMs, and weight gradients
 * from column-wise copies.
 */
enum { MOE_PREC_BF16 = 0, MOE_PREC_FP8 = 1, MOE_PREC_MXFP8 = 2 };

typedef struct moe_layer_config {
  int32_t T, d, f, E, k;       /* tokens, d_model, d_ff, experts, top-k */
  int32_t score_fn, renorm;    /* MOE_SCORE_*, renormalise the top-k weights */
  int32_t num_groups, topk_group; /* group-limited routing (0, 0: off) */
  int32_t align, capacity;     /* align_size padding, per-expert capacity (0: off) */
  int32_t num_chunks;          /* K-chunks of the up-projection (<= 1: one GEMM) */
  float aux_coeff;             /* auxiliary load-balancing loss weight (0: off) */
  int32_t bias;                /* expert-FFN biases bi [E, 2f], bo [E, d] */
  int32_t precision;           /* MOE_PREC_* of the expert GEMMs */
  int32_t wgrad_colwise;       /* bf16: weight gradients from column-wise copies */
  int32_t dw_dtype;            /* MOE_DTYPE_* of dWi / dWo */
} moe_layer_config;

/* Buffers of the workspace (moe_layer_buffer).  Shapes: R = rows_cap
 * (moe_rows_cap), P = moe_fp8_padded_rows(R, E); bf16 unless noted. */
enum {
  MOE_BUF_TOPK_IDX = 0,   /* int32 [T, k] */
  MOE_BUF_TOPK_W,         /* f32 [T, k] */
  MOE_BUF_XS,             /* [R, d] permuted tokens */
  MOE_BUF_GROUP_SIZES,    /* int32 [E] */
  MOE_BUF_KEPT_COUNTS,    /* int32 [E] */
  MOE_BUF_GROUP_OFFSETS,  /* int32 [E + 1] */
  MOE_BUF_S2F,            /* int32 [R] sorted_to_flat */
  MOE_BUF_F2S,            /* int32 [T k] flat_to_sorted */
  MOE_BUF_PERMUTE_WS,     /* moe_permute_workspace_bytes(T, E) */
  MOE_BUF_H,              /* [R, 2f] up-projection [gate | up] */
  MOE_BUF_ACT,            /* [R, f] SwiGLU activation */
  MOE_BUF_Y,              /* [R, d] expert outputs */
  MOE_BUF_OUT,            /* [T, d] layer output */
  MOE_BUF_PARTIAL,        /* f32 [R, 2f] K-chunk partial sum (num_chunks > 1) */
  MOE_BUF_DY,             /* [R, d] */
  MOE_BUF_D_TOPK_W,       /* f32 [T, k] */
  MOE_BUF_D_LOGITS,       /* f32 [T, E] router-logit gradient */
  MOE_BUF_DH,             /* [R, 2f] */
  MOE_BUF_DXS,            /* [R, d] */
  MOE_BUF_DX,             /* [T, d] input gradient */
  MOE_BUF_DWI,            /* dw_dtype [E, d, 2f] */
  MOE_BUF_DWO,            /* dw_dtype [E, f, d] */
  MOE_BUF_DBI,            /* f32 [E, 2f] (bias) */
  MOE_BUF_DBO,            /* f32 [E, d] (bias) */
  MOE_BUF_DEV_STATUS,     /* int32 [1] device status word */
  MOE_BUF_XS_T,           /* [d, P] column-wise copies (wgrad_colwise) */
  MOE_BUF_ACT_T,          /* [f, P] */
  MOE_BUF_DY_T,           /* [d, P] */
  MOE_BUF_DH_T,           /* [2f, P] */
  MOE_BUF_F8_XS_Q,        /* uint8 [R, d]   FP8: row-wise codes ... */
  MOE_BUF_F8_XS_QT,       /* uint8 [d, P]   ... and column-wise codes */
  MOE_BUF_F8_ACT_Q,       /* uint8 [R, f] */
  MOE_BUF_F8_ACT_QT,      /* uint8 [f, P] */
  MOE_BUF_F8_DY_Q,        /* uint8 [R, d] */
  MOE_BUF_F8_DY_QT,       /* uint8 [d, P] */
  MOE_BUF_F8_DH_Q,        /* uint8 [R, 2f] */
  MOE_BUF_F8_DH_QT,       /* uint8 [2f, P] */
  MOE_BUF_F8_WI_Q,        /* uint8 [E, d, 2f] */
  MOE_BUF_F8_WI_QT,       /* uint8 [E, 2f, d] */
  MOE_BUF_F8_WO_Q,        /* uint8 [E, f, d] */
  MOE_BUF_F8_WO_QT,       /* uint8 [E, d, f] */
  MOE_BUF_F8_AMAX,        /* f32 [4 + 2E]: Xs, Act, dY, dH, wi (E), wo (E) */
  MOE_BUF_F8_SINV,        /* f32 [4 + 2E]: the matching 1 / scale */
  /* MXFP8: codes (uint8) and scale atoms of each block-scaled operand; the
   * atom bytes are moe_mx_scale_bytes(rows, cols, map, groups) */
  MOE_BUF_MX_XS_Q,        /* [R, d], GROUPED */
  MOE_BUF_MX_XS_SF,
  MOE_BUF_MX_ACT_Q,       /* [R, f], GROUPED */
  MOE_BUF_MX_ACT_SF,
  MOE_BUF_MX_DY_Q,        /* [R, d], GROUPED */
  MOE_BUF_MX_DY_SF,
  MOE_BUF_MX_DH_Q,        /* [R, 2f], GROUPED */
  MOE_BUF_MX_DH_SF,
  MOE_BUF_MX_XS_T_Q,      /* [d, P], PLAIN, E groups */
  MOE_BUF_MX_XS_T_SF,
  MOE_BUF_MX_ACT_T_Q,     /* [f, P], PLAIN, E groups */
  MOE_BUF_MX_ACT_T_SF,
  MOE_BUF_MX_DY_T_Q,      /* [d, P], TILES, 1 group */
  MOE_BUF_MX_DY_T_SF,
  MOE_BUF_MX_DH_T_Q,      /* [2f, P], TILES, 1 group */
  MOE_BUF_MX_DH_T_SF,
  MOE_BUF_MX_WI_T_Q,      /* [2f, E d], SWIGLU, E groups */
  MOE_BUF_MX_WI_T_SF,
  MOE_BUF_MX_WI_Q,        /* [E d, 2f], TILES, E groups */
  MOE_BUF_MX_WI_SF,
  MOE_BUF_MX_WO_T_Q,      /* [d, E f], TILES, 1 group */
  MOE_BUF_MX_WO_T_SF,
  MOE_BUF_MX_WO_Q,        /* [E f, d], TILES, E groups */
  MOE_BUF_MX_WO_SF,
  MOE_BUF_MX_WOFF_D,      /* int32 [E + 1]: e * d (the weights' rows as groups) */
  MOE_BUF_MX_WOFF_F,      /* int32 [E + 1]: e * f */
  MOE_BUF_AUX_COUNTS,     /* int32 [E] (aux_coeff > 0) */
  MOE_BUF_AUX_PROBS,      /* f32 [E] */
  MOE_BUF_AUX_LOSS,       /* f32 [1] */
  MOE_BUF_AUX_WS,         /* moe_aux_loss_workspace_bytes(T, E) */
  MOE_BUF_COUNT
};

/* Called after each enqueued call with the call's name (e.g. "permute",
 * "gmm_up_swiglu", "tgmm_dwi"), on the calling thread; a profiler records an
 * event on the stream there.  May be NULL. */
typedef void (*moe_mark_fn)(void *ctx, const char *name);

/*
 * moe_layer_workspace_bytes -- bytes of the layer's device workspace for `cfg`
 * (0 and the reason in moe_last_error() for an invalid configuration).
 * moe_layer_buffer -- where buffer `id` (MOE_BUF_*) lives in it: byte offset
 * (a multiple of 256) and size; size 0 for a buffer the configuration does
 * not use.  Both are host computations.
 */
size_t moe_layer_workspace_bytes(const moe_layer_config *cfg);
moe_status_t moe_layer_buffer(const moe_layer_config *cfg, int id, size_t *offset,
                              size_t *bytes);

/*
 * moe_layer_init -- once per workspace, before the first forward: zeroes the
 * device status word and writes the constant tables (MXFP8 weight-row
 * offsets).  workspace: 256-byte aligned, >= moe_layer_workspace_bytes(cfg).
 */
moe_status_t moe_layer_init(const moe_layer_config *cfg, void *workspace,
                            size_t workspace_bytes, moe_stream_t stream);

/*
 * moe_layer_forward -- x bf16 [T, d], logits f32 [T, E], wi bf16 [E, d, 2f]
 * ([wi_0 | wi_1] along the last axis), wo bf16 [E, f, d], all contiguous;
 * bi bf16 [E, 2f] and bo bf16 [E, d] exactly when cfg->bias; expert_bias f32
 * [E] or NULL (selection bias: experts ranked by logit + bias, weights from
 * the unbiased logits).  The output is MOE_BUF_OUT of the workspace (and, with
 * aux_coeff, the loss in MOE_BUF_AUX_LOSS).  The backward reads `logits`
 * again (pass the same, unchanged array) and the tensors the forward saved in
 * the workspace; x is not read after the forward.
 */
moe_status_t moe_layer_forward(const moe_layer_config *cfg, void *workspace,
                               size_t workspace_bytes, const uint16_t *x, const float *logits,
                               const uint16_t *wi, const uint16_t *wo, const uint16_t *bi,
                               const uint16_t *bo, const float *expert_bias, moe_mark_fn mark,
                               void *mark_ctx, moe_stream_t stream);

/*
 * moe_layer_backward -- dout bf16 [T, d] (contiguous), logits the forward's;
 * writes MOE_BUF_DX, MOE_BUF_DWI, MOE_BUF_DWO, MOE_BUF_D_LOGITS (the router
 * gradient, with the auxiliary loss's part when aux_coeff > 0),
 * MOE_BUF_D_TOPK_W and, with biases, MOE_BUF_DBI / MOE_BUF_DBO.
 */
moe_status_t moe_layer_backward(const moe_layer_config *cfg, void *workspace,
                                size_t workspace_bytes, const uint16_t *dout,
                                const float *logits, const uint16_t *wi, const uint16_t *wo,
                                moe_mark_fn mark, void *mark_ctx, moe_stream_t stream);

/*
 * The layer from HOST buffers: a training step's inputs (x, logits, dout) are
 * copied in from host memory and its results (out, dx, d_logits) copied back,
 * double-buffered so that step i + 1's input copies and step i's result
 * copies overlap the compute of the steps next to them.  The weights, the
 * weight gradients and every intermediate stay on the device (the layer's
 * workspace).
 *
 * moe_layer_pipeline_workspace_bytes -- device bytes of the staging slots
 *   (two of each: x, logits, dout, out, dx, d_logits).
 * moe_layer_pipeline_create -- a pipeline over one layer workspace (set up
 *   by moe_layer_init) and one staging workspace (both caller-owned device
 *   memory; the pipeline keeps the pointers until destroyed).  Unlike the calls above it holds state:
 *   two copy streams and its events on the current device (no device memory).
 * moe_layer_pipeline_step -- enqueue one step: host -> device copies of h_x
 *   bf16 [T, d], h_logits f32 [T, E], h_dout bf16 [T, d] on the input copy
 *   stream; forward + backward on `stream` once they have landed; device ->
 *   host copies into h_out bf16 [T, d], h_dx bf16 [T, d], h_d_logits f32
 *   [T, E] on the output copy stream once the step has finished.  Returns
 *   without waiting.  Host buffers should be page-locked (cudaHostAlloc /
 *   pinned) for the copies to overlap; the caller keeps them unchanged (inputs)
 *   and unread (results) until moe_layer_pipeline_join's stream has passed or
 *   moe_layer_pipeline_sync returned.  dWi / dWo are the workspace's and are
 *   overwritten by every step.
 * moe_layer_pipeline_join -- make `stream` wait for every copy enqueued so far.
 * moe_layer_pipeline_sync -- block the host until every copy has completed.
 * moe_layer_pipeline_destroy -- synchronise the copy streams and release them
 *   and the events (the caller synchronises its compute stream before it frees
 *   the workspaces).
 */
typedef struct moe_layer_pipeline moe_layer_pipeline;
size_t moe_layer_pipeline_workspace_bytes(const moe_layer_config *cfg);
moe_status_t moe_layer_pipeline_create(const moe_layer_config *cfg, void *workspace,
                                       size_t workspace_bytes, void *staging,
                                       size_t staging_bytes, moe_layer_pipeline **out);
moe_status_t moe_layer_pipeline_step(moe_layer_pipeline *pipe, const uint16_t *wi,
                                     const uint16_t *wo, const uint16_t *bi, const uint16_t *bo,
                                     const float *expert_bias, const uint16_t *h_x,
                                     const float *h_logits, const uint16_t *h_dout,
                                     uint16_t *h_out, uint16_t *h_dx, float *h_d_logits,
                                     moe_stream_t stream);
moe_status_t moe_layer_pipeline_join(moe_layer_pipeline *pipe, moe_stream_t stream);
moe_status_t moe_layer_pipeline_sync(moe_layer_pipeline *pipe);
void moe_layer_pipeline_destroy(moe_layer_pipeline *pipe);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
