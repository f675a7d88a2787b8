/*
 * moe.h -- C ABI of the GB300 (sm_103a) single-GPU Mixture-of-Experts layer.
 *
 * The layer pass follows "Scalable Training of Mixture-of-Experts Models with
 * Megatron Core" (paper review page), §2.1 "MoE layer architecture and forward
 * pass": Route -> Dispatch -> Expert computation -> Combine, with the router of
 * §2.2 and the grouped expert GEMM of §4.3.1.  The layer computes
 *
 *     p(x) = Score(W_r^T x + b_r)                        (review §1.1, §2.2)
 *     MoE(x) = sum_{i in TopK} p_i(x) E_i(x)  [+ S(x)]   (review §1.1)
 *
 * Conventions shared by every entry point:
 *  - Pointers named as device buffers are device pointers (cudaMalloc'd or
 *    torch-allocated).  The caller owns every buffer; no call allocates device
 *    memory.  Scratch lives in a caller-provided workspace of
 *    moe_workspace_size(cfg) bytes (256-byte aligned).
 *  - All calls are asynchronous on `stream` (a cudaStream_t, NULL = the legacy
 *    default stream) and never synchronise or read device memory on the host,
 *    except moe_get_error.  Per-expert counts and offsets stay on the device.
 *  - Argument errors return MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED /
 *    MOE_ERR_WORKSPACE before anything is enqueued.  A failed launch returns
 *    MOE_ERR_CUDA.  Conditions found on the device (a bounded wait that gave
 *    up) are recorded in a per-device status word read by moe_get_error.
 *  - Layouts are row-major.  "act" tensors (x, expert weights, biases,
 *    x_perm, y_perm, y) have the config's dtype (fp32 or bf16); the router
 *    weight, router biases, logits and probabilities are always fp32; index
 *    tensors are int32.  Row strides are the dense widths stated per argument.
 *  - Alignment: every buffer must be 16-byte aligned; bf16 configs need h and
 *    F to be multiples of 8 and fp32 configs multiples of 4 (16-byte rows).
 *  - Limits: 1 <= E <= 256, 1 <= K <= min(E, 16), T*K < 2^31, n_shared 0 or 1.
 *    SwiGLU experts are bias-free.  Anything else: MOE_ERR_UNSUPPORTED.
 *
 * Shapes (P = T*K permuted rows; R1 = 2F for SwiGLU, F for GELU):
 *   x [T,h]  w_r [E,h] (the review's W_r in R^{h x E}, stored transposed)
 *   w1 [E][R1][h] (SwiGLU: rows 0..F-1 gate, F..2F-1 up)   b1 [E][F]
 *   w2 [E][h][F]   b2 [E][h]   w1_shared [R1][h]   w2_shared [h][F]
 */
#ifndef MOE_GB300_H_
#define MOE_GB300_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef void* moe_stream_t; /* cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misaligned buffer   */
  MOE_ERR_UNSUPPORTED = 2,   /* valid but outside this library's limits     */
  MOE_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required  */
  MOE_ERR_CUDA = 4,          /* a CUDA runtime/driver call or launch failed */
  MOE_ERR_TIMEOUT = 5,       /* a bounded device-side wait gave up          */
  MOE_ERR_DEVICE_BOUNDS = 6  /* a device-side index check failed            */
} moe_status_t;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype_t;
typedef enum { MOE_SCORE_SOFTMAX = 0, MOE_SCORE_SIGMOID = 1 } moe_score_t;
typedef enum { MOE_ACT_GELU = 0, MOE_ACT_SWIGLU = 1 } moe_act_t;

enum {
  /* Divide the selected experts' scores by their sum (the skill page
   * "emerging-techniques-moe-training", "Top-2 Routing (Mixtral)").  Without
   * it: softmax is the full softmax over E at the selected experts, sigmoid is
   * normalised over all E (review §2.2). */
  MOE_FLAG_RENORM = 1u,
  /* Force-balanced routing (review §2.2): slot k of token t goes to expert
   * (t*K + k) mod E; probs are the scores at those experts. */
  MOE_FLAG_FORCE_BALANCE = 2u,
  /* Validate arguments and return without enqueuing anything. */
  MOE_FLAG_VALIDATE_ONLY = 8u,
  /* moe_layer_fwd keeps, in the workspace, what moe_layer_bwd needs. */
  MOE_FLAG_SAVE_FOR_BWD = 16u,
  /* Use the SIMT grouped GEMM for bf16 too (slow; a cross-check path). */
  MOE_FLAG_GEMM_SIMT = 32u,
  /* Tensor-core expert GEMM tiling: by default CTA pairs (256-row tiles,
   * tcgen05 cta_group::2) when experts average >= 512 rows, single CTAs
   * (128-row tiles) otherwise.  These force one or the other. */
  MOE_FLAG_GEMM_1CTA = 64u,
  MOE_FLAG_GEMM_2CTA = 128u,
  /* Route -> Dispatch hand-off (review §4.3.1, permutation fusion):
   * moe_router_topk also leaves the per-chunk expert histograms of the
   * topk_idx it writes (tokens in chunks of 32: the first step of the
   * dispatch maps) in the workspace, computed by the router's own epilogue
   * where it can (bf16, E <= 8) and by one extra step otherwise; moe_permute
   * and moe_permute_mxfp8 given the same flag, the same workspace and that
   * unmodified topk_idx start from them instead of counting again.  The
   * caller promises the hand-off: a histogram that does not match topk_idx
   * gives wrong maps (out-of-range rows are never written: they are reported
   * as MOE_ERR_DEVICE_BOUNDS).  moe_layer_fwd does this internally.
   * moe_permute_noalloc ignores the flag (it has no workspace). */
  MOE_FLAG_HIST_FROM_ROUTER = 256u
};

typedef struct {
  int32_t T;        /* tokens                                   */
  int32_t h;        /* hidden size                              */
  int32_t E;        /* routed experts                           */
  int32_t K;        /* experts per token (top-k)                */
  int32_t F;        /* expert FFN width (per SwiGLU branch)     */
  int32_t dtype;    /* moe_dtype_t of activations and weights   */
  int32_t score;    /* moe_score_t                              */
  int32_t act;      /* moe_act_t                                */
  int32_t has_bias; /* experts carry b1, b2 (GELU only)         */
  int32_t n_shared; /* 0 or 1 always-on shared expert           */
  uint32_t flags;   /* MOE_FLAG_*                               */
  /* Weights of the router's load-balancing losses (see moe_router_aux_loss)
   * in the training backward: with either nonzero, moe_layer_fwd also
   * computes both losses (read them with moe_layer_losses) and moe_layer_bwd
   * adds their gradient to the router's.  Must be finite; 0 = off. */
  float aux_loss_coeff;
  float z_loss_coeff;
  /* Expert capacity in (token, slot) pairs (skill page "emerging-techniques-
   * moe-training", "Capacity Factor Tuning"; see moe_expert_capacity): each
   * expert keeps its first `capacity` slots in ascending token order and
   * drops the rest (their dst_row is -1; they add nothing to y; the kept
   * weights are not renormalised).  0 = dropless. */
  int32_t capacity;
} moe_config_t;

/* floor(capacity_factor * T * K / E), at least min_capacity: the capacity of
 * the skill page's formula, int(tokens / experts * capacity_factor), counted
 * in top-K slots.  Host-only arithmetic; -1 if an argument is out of range
 * (T < 0, K < 1, E < 1, capacity_factor not finite and > 0) or the result
 * does not fit an int32. */
int32_t moe_expert_capacity(int32_t T, int32_t K, int32_t E, float capacity_factor,
                            int32_t min_capacity);

/* Bytes of workspace every call below needs for `cfg` (the same figure for
 * all of them; it grows with MOE_FLAG_SAVE_FOR_BWD).  0 if cfg is invalid. */
size_t moe_workspace_size(const moe_config_t* cfg);

/* Route (review §2.2 "Gating" and "Top-k selection"; §5.1 keeps the router
 * in FP32).  Computes l = W_r^T x + b_r in fp32, selects the K experts with
 * the largest key (softmax: l + sel_bias; sigmoid: fp32(sigma(l)) + sel_bias,
 * sigma evaluated in double), ties to the lower expert index, listed in
 * descending key order, and their probabilities.
 *   x [T,h] dtype; w_r [E,h] f32; gate_bias [E] f32 or NULL (b_r);
 *   sel_bias [E] f32 or NULL (selection only, never enters p);
 *   logits [T,E] f32 out or NULL; topk_idx [T,K] i32 out; topk_prob [T,K] f32 out;
 *   routing_map [T,E] u8 out or NULL (1 where selected). */
moe_status_t moe_router_topk(const moe_config_t* cfg, const void* x, const float* w_r,
                             const float* gate_bias, const float* sel_bias, float* logits,
                             int32_t* topk_idx, float* topk_prob, uint8_t* routing_map,
                             void* ws, size_t ws_bytes, moe_stream_t stream);

/* The scoring / top-k / normalisation half of the router on given fp32
 * logits [T,E]; same outputs and rules as moe_router_topk. */
moe_status_t moe_router_topk_from_logits(const moe_config_t* cfg, const float* logits,
                                         const float* sel_bias, int32_t* topk_idx,
                                         float* topk_prob, uint8_t* routing_map,
                                         moe_stream_t stream);

/* Dispatch (review §2.1 "Dispatch"; permutation fusion, §4.3.1): the T*K
 * (token, slot) pairs in expert-contiguous order, tokens ascending within an
 * expert.  counts[e] = pairs routed to e; offsets = exclusive prefix sum
 * (E+1 entries); dst_row[t,k] = offsets[e] + #{t' < t routed to e};
 * src_token[r] / perm_prob[r] invert it; x_perm[dst_row[t,k]] = x[t].
 *   x [T,h]; topk_idx [T,K]; topk_prob [T,K] or NULL (then perm_prob unused);
 *   outputs x_perm [P,h] (NULL: maps only), counts [E], offsets [E+1],
 *   dst_row [T,K], src_token [P], perm_prob [P] or NULL.
 * Bit-exact and deterministic (no atomics decide a position). */
moe_status_t moe_permute(const moe_config_t* cfg, const void* x, const int32_t* topk_idx,
                         const float* topk_prob, void* x_perm, int32_t* counts, int32_t* offsets,
                         int32_t* dst_row, int32_t* src_token, float* perm_prob, void* ws,
                         size_t ws_bytes, moe_stream_t stream);

/* moe_permute without a workspace, for callers that cannot allocate device
 * memory: plugins hosted by a framework that owns all device memory and
 * offers them no allocator, and serving loops that must not allocate after
 * start-up.  The pages have no counterpart of this entry point; it is a
 * deployment convenience.  Same arguments (minus ws), rules and results as
 * moe_permute.
 *  - Scratch: a fixed 2 MiB array inside the library (two tables of
 *    ceil(T/32) * E int32), held by every GPU that loads the library until the
 *    process exits.  Configurations with ceil(T/32) * E > 262144 return
 *    MOE_ERR_UNSUPPORTED.  Nothing in it needs clearing between calls.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current); make that first call
 *    before capturing any stream.
 *  - Every call on a device shares the one array: calls whose kernels can
 *    overlap on the GPU (different streams without ordering) race.
 *  - Allocates nothing: no cudaMalloc, cudaFree or allocating library call. */
moe_status_t moe_permute_noalloc(const moe_config_t* cfg, const void* x, const int32_t* topk_idx,
                                 const float* topk_prob, void* x_perm, int32_t* counts,
                                 int32_t* offsets, int32_t* dst_row, int32_t* src_token,
                                 float* perm_prob, moe_stream_t stream);

/* Expert computation (review §2.1 "Expert computation": every expert in one
 * grouped GEMM call; §4.1.1 memory-efficient permutation).  For every row r
 * of expert e (offsets[e] <= r < offsets[e+1]):
 *   bias-free:  a = p_r * phi(x_perm[r] W1_e^T),   y_perm[r] = a W2_e^T
 *   biased:     a = GELU(x_perm[r] W1_e^T + b1_e), y_perm[r] = p_r (a W2_e^T + b2_e)
 * phi = silu(gate) * up (SwiGLU) or GELU (exact erf); p_r = perm_prob[r]
 * (NULL: 1).  bf16 runs on the tensor cores (tcgen05, fp32 accumulate),
 * fp32 on the SIMT FMA units.
 *   x_perm [P,h]; offsets [E+1] device; w1, b1, w2, b2 as above;
 *   act_save [P,R1] out or NULL: the pre-activation x_perm W1^T (+ b1);
 *   y_perm [P,h] out. */
moe_status_t moe_grouped_mlp_fwd(const moe_config_t* cfg, const void* x_perm,
                                 const int32_t* offsets, const float* perm_prob, const void* w1,
                                 const void* b1, const void* w2, const void* b2, void* act_save,
                                 void* y_perm, void* ws, size_t ws_bytes, moe_stream_t stream);

/* The two halves of moe_grouped_mlp_fwd, one grouped GEMM launch each.
 * FC1: a[r] = p_r * phi(x_perm[r] W1_e^T) (bias-free experts) or
 *      a[r] = GELU(x_perm[r] W1_e^T + b1_e) (biased experts);
 *      act_save [P,R1] out or NULL (pre-activation); a [P,F] out.
 * FC2: y_perm[r] = a[r] W2_e^T (bias-free) or p_r (a[r] W2_e^T + b2_e). */
moe_status_t moe_expert_fc1(const moe_config_t* cfg, const void* x_perm, const int32_t* offsets,
                            const float* perm_prob, const void* w1, const void* b1,
                            void* act_save, void* a, moe_stream_t stream);
moe_status_t moe_expert_fc2(const moe_config_t* cfg, const void* a, const int32_t* offsets,
                            const float* perm_prob, const void* w2, const void* b2,
                            void* y_perm, moe_stream_t stream);

/* FC1 with the dispatch gather fused in (review §4.3.1 "permutation fusion";
 * §2.1 Dispatch then Expert computation): GEMM row r reads the token row
 * x[src_token[r]] directly instead of x_perm[r], so the permuted copy of x is
 * never written.  Same outputs and rules as moe_expert_fc1 otherwise.
 *   x [T,h] bf16; src_token [T*K] i32 and offsets [E+1] from moe_permute
 *   (called with x = NULL: maps only); perm_prob, w1, b1, act_save, a as in
 *   moe_expert_fc1.  Tensor-core (bf16) configurations only, else
 *   MOE_ERR_UNSUPPORTED.  The rows are fetched by TMA tile::gather4 loads;
 *   since FC1 reads each row block once per N tile, this is slower on GB300
 *   than moe_permute's one-pass scatter followed by moe_expert_fc1 (which
 *   moe_layer_fwd uses), but it needs no x_perm buffer. */
moe_status_t moe_expert_fc1_gather(const moe_config_t* cfg, const void* x,
                                   const int32_t* src_token, const int32_t* offsets,
                                   const float* perm_prob, const void* w1, const void* b1,
                                   void* act_save, void* a, moe_stream_t stream);

/* ---- MXFP8 expert GEMMs (review §5.3.3 "MXFP8 (Blackwell)") ----------------
 * Activations and weights quantised in 1 x 32 blocks along the GEMM's K
 * dimension, each block one E8M0 scale, elements FP8 E4M3 (OCP Microscaling
 * v1.0: X = floor(log2 max|x|) - 8, element = x / 2^X rounded to nearest even,
 * saturated to +-448); the GEMMs run as block-scaled tensor-core MMAs with
 * fp32 accumulation.  Forward only, SwiGLU experts without biases.
 *
 * MXFP8 tensor format: codes [rows, K] uint8 (E4M3, row-major) and a scale
 * buffer of moe_mxfp8_scale_bytes(rows, K, groups) bytes.  The rows form
 * groups (experts); each group's rows are cut into 128-row tiles, numbered
 * group after group; the scales of tile t and K columns kb*128..kb*128+127
 * form one 512-byte atom at byte (t * K/128 + kb) * 512, where row i of the
 * tile (i = 0..127), block j (j = 0..3) sits at byte 16 (i % 32) + 4 (i / 32)
 * + j.  K must be a multiple of 128.  Scale bytes of rows past a group's end
 * inside its last tile are unspecified.
 *
 * Errors: NULL or 16-byte-misaligned tensors -> MOE_ERR_INVALID_ARG; K or the
 * config's h / F not multiples of 128, act not SwiGLU, has_bias, fp32 dtype ->
 * MOE_ERR_UNSUPPORTED; bounded-wait timeouts on the device -> reported by
 * moe_get_error. */

/* Bytes of the scale buffer of an MXFP8 tensor of `rows` rows in `groups`
 * groups with K columns (K a multiple of 128); 0 on bad arguments. */
size_t moe_mxfp8_scale_bytes(int64_t rows, int32_t K, int32_t groups);

/* Quantise x [rows, K] bf16 (device) to MXFP8: codes q [rows, K] and scales sf
 * (device, caller-owned).  offsets [groups+1] (device): group g holds rows
 * offsets[g] .. offsets[g+1]-1 (rows outside every group get codes but no
 * scales); NULL: groups of rows/groups rows each (rows % groups == 0), as for
 * expert weights [E][N][K].  Deterministic and exact: the decisions depend
 * only on the bf16 values. */
moe_status_t moe_mxfp8_quantize(int64_t rows, int32_t K, int32_t groups, const int32_t* offsets,
                                const void* x, uint8_t* q, uint8_t* sf, moe_stream_t stream);

/* Dispatch with the MXFP8 quantisation fused in: the maps of moe_permute
 * (counts, offsets, dst_row, src_token, perm_prob; same rules, capacity
 * included) and, instead of x_perm, x_perm in MXFP8 -- x_q [P,h] codes and
 * x_sf scales (moe_mxfp8_scale_bytes(T*K, h, E) bytes, groups = the experts of
 * `offsets`).  Each token row is read and quantised once (blocks along h) and
 * its codes and scales written to its K rows: the same bytes as
 * moe_permute followed by moe_mxfp8_quantize(offsets), in one pass over x.
 * bf16 configurations with h % 128 == 0, else MOE_ERR_UNSUPPORTED; ws as for
 * moe_permute.  Rows of dropped slots are not written. */
moe_status_t moe_permute_mxfp8(const moe_config_t* cfg, const void* x, const int32_t* topk_idx,
                               const float* topk_prob, uint8_t* x_q, uint8_t* x_sf,
                               int32_t* counts, int32_t* offsets, int32_t* dst_row,
                               int32_t* src_token, float* perm_prob, void* ws, size_t ws_bytes,
                               moe_stream_t stream);

/* MXFP8 FC1 with the SwiGLU epilogue: H = x_perm W1_e^T over the dequantised
 * operands (fp32), a[r] = p_r silu(H[r, :F]) H[r, F:] (p_r = perm_prob[r], 1
 * when NULL).  Outputs, any non-NULL subset:
 *   a [P,F] bf16;  a_q [P,F] + a_sf = a quantised to MXFP8 from fp32 (blocks
 *   along F, groups = the experts of `offsets`), FC2's left operand.
 *   x_q [P,h] + x_sf: x_perm in MXFP8 (groups = experts, from offsets);
 *   w1_q [E*2F, h] + w1_sf: W1 in MXFP8 (uniform groups of 2F rows).
 * cfg gives T, K (P = T*K rows), h, E, F; offsets [E+1] as from moe_permute. */
moe_status_t moe_expert_fc1_mxfp8(const moe_config_t* cfg, const uint8_t* x_q,
                                  const uint8_t* x_sf, const int32_t* offsets,
                                  const float* perm_prob, const uint8_t* w1_q,
                                  const uint8_t* w1_sf, void* a, uint8_t* a_q, uint8_t* a_sf,
                                  moe_stream_t stream);

/* MXFP8 FC2: y_perm[r] = a[r] W2_e^T over the dequantised operands, bf16 out.
 *   a_q [P,F] + a_sf (from moe_expert_fc1_mxfp8 or moe_mxfp8_quantize with the
 *   experts' offsets); w2_q [E*h, F] + w2_sf (uniform groups of h rows);
 *   y_perm [P,h] out. */
moe_status_t moe_expert_fc2_mxfp8(const moe_config_t* cfg, const uint8_t* a_q,
                                  const uint8_t* a_sf, const int32_t* offsets,
                                  const uint8_t* w2_q, const uint8_t* w2_sf, void* y_perm,
                                  moe_stream_t stream);

/* Combine (review §2.1 "Combine"; the skill page's index_add_):
 *   y[t] = sum_{k=0}^{K-1} w[t,k] * y_perm[dst_row[t,k]]  (+ shared_y[t])
 * with w = topk_prob, or 1 when topk_prob is NULL (probabilities already
 * applied in the expert GEMM).  fp32 accumulation in fixed k order, rounded
 * once: bitwise deterministic.
 *   y_perm [P,h]; dst_row [T,K]; topk_prob [T,K] or NULL; shared_y [T,h] or NULL;
 *   y [T,h] out. */
moe_status_t moe_unpermute_combine(const moe_config_t* cfg, const void* y_perm,
                                   const int32_t* dst_row, const float* topk_prob,
                                   const void* shared_y, void* y, moe_stream_t stream);

/* The whole forward layer pass: Route, Dispatch, grouped expert GEMMs (plus
 * the shared expert when n_shared = 1, weight 1, not routed), Combine.
 *   y [T,h] out; topk_idx_out [T,K] and topk_prob_out [T,K] optional copies of
 *   the routing.  With MOE_FLAG_SAVE_FOR_BWD the workspace keeps the routing,
 *   maps and activations for moe_layer_bwd. */
moe_status_t moe_layer_fwd(const moe_config_t* cfg, const void* x, const float* w_r,
                           const float* gate_bias, const float* sel_bias, const void* w1,
                           const void* b1, const void* w2, const void* b2,
                           const void* w1_shared, const void* w2_shared, void* y,
                           int32_t* topk_idx_out, float* topk_prob_out, void* ws,
                           size_t ws_bytes, moe_stream_t stream);

/* ---- Backward (the training configuration: bf16, SwiGLU experts, a
 * renormalised softmax or sigmoid router; others return MOE_ERR_UNSUPPORTED).
 * The pages give no backward formulas ("Scalable Training of Mixture-of-Experts
 * Models with Megatron Core", review §4.1.2, only names the recomputed
 * activations); these calls compute the reverse-mode derivatives of the
 * forward above with the expert selection held fixed.  The selection bias
 * receives no gradient.  Weight gradients are written (not accumulated). */

/* Expert FFNs over permuted rows, from the forward's saved pre-activation
 * (act_save [P,2F]) and FC2 input (a [P,F] = p * silu(gate) * up):
 *   G = dy_perm W2_e;  dprob_perm[r] = <G_r, silu(g_r) * u_r> = <dy_perm_r, E_e(x_r)>;
 *   dH = [p G u silu'(g), p G silu(g)];  dW2_e = dy_perm_e^T a_e;
 *   dx_perm = dH W1_e;  dW1_e = dH_e^T x_perm_e.
 *   dy_perm, x_perm [P,h]; offsets [E+1]; perm_prob [P]; w1 [E][2F][h]; w2 [E][h][F];
 *   outputs dx_perm [P,h], dw1 [E][2F][h], dw2 [E][h][F] (bf16, fp32 accumulate;
 *   experts without rows get zeros), dprob_perm [P] f32 or NULL.
 *   ws: moe_workspace_size of cfg with MOE_FLAG_SAVE_FOR_BWD. */
moe_status_t moe_grouped_mlp_bwd(const moe_config_t* cfg, const void* dy_perm, const void* x_perm,
                                 const void* act_save, const void* a, const int32_t* offsets,
                                 const float* perm_prob, const void* w1, const void* w2,
                                 void* dx_perm, void* dw1, void* dw2, float* dprob_perm, void* ws,
                                 size_t ws_bytes, moe_stream_t stream);

/* Route backward from dprob_perm (permuted order, as moe_grouped_mlp_bwd
 * gives it): for each token's selected experts
 *   softmax: dl_k = p_k (dp_k - sum_j p_j dp_j)
 *   sigmoid: dl_k = s_k (1 - s_k) (dp_k - sum_j p_j dp_j) / sum_sel s
 * then dW_r[e] = sum over e's tokens of dl x_t (fp32), db_r[e] = sum dl, and
 * optionally dx_router[t] = sum_k dl_k W_r[e_k] (fp32 [T,h]).
 *   x [T,h]; logits [T,E]; topk_idx/topk_prob [T,K]; offsets, dst_row, src_token
 *   from moe_permute; outputs dl_topk [T,K], dw_r [E,h], db_r [E] or NULL,
 *   dx_router or NULL (then w_r may be NULL).  Dropless configs only
 *   (capacity 0, else MOE_ERR_UNSUPPORTED: moe_layer_bwd covers capacity). */
moe_status_t moe_router_bwd(const moe_config_t* cfg, const void* x, const float* logits,
                            const int32_t* topk_idx, const float* topk_prob,
                            const int32_t* offsets, const int32_t* dst_row,
                            const int32_t* src_token, const float* dprob_perm, const float* w_r,
                            float* dl_topk, float* dw_r, float* db_r, float* dx_router, void* ws,
                            size_t ws_bytes, moe_stream_t stream);

/* Load-balancing losses of the router (skill page "emerging-techniques-moe-
 * training", "Load Balancing": "Auxiliary Loss" and "Router Z-Loss"; the
 * review page's training configuration weights the auxiliary loss by 1e-3):
 *   f_e = (slots of topk_idx routed to e) / (T*K)   (no gradient: a count)
 *   P_e = (1/T) sum_t softmax(l_t)_e                 (full softmax, any scoring)
 *   losses[0] = aux = E * sum_e f_e P_e
 *   losses[1] = z   = (1/T) sum_t (logsumexp_e l_te)^2
 * and, when dlogits is given, adds the weighted gradients in place:
 *   dlogits[t,j] += aux_coeff * (E/T) s_tj (f_j - sum_e f_e s_te)
 *                 + z_coeff * (2/T) lse_t s_tj          (s_t = softmax(l_t))
 *   logits [T,E] f32; topk_idx [T,K] i32 (ids outside [0,E) are reported as
 *   MOE_ERR_DEVICE_BOUNDS and not counted); losses: 2 f32 (device, out);
 *   dlogits [T,E] f32 (in/out) or NULL; ws: moe_workspace_size(cfg) bytes.
 *   Sums in fp64 and in a fixed order: bitwise reproducible.  T = 0 writes
 *   zero losses. */
moe_status_t moe_router_aux_loss(const moe_config_t* cfg, const float* logits,
                                 const int32_t* topk_idx, float aux_coeff, float z_coeff,
                                 float* losses, float* dlogits, void* ws, size_t ws_bytes,
                                 moe_stream_t stream);

/* The two load-balancing losses of the last moe_layer_fwd on this workspace
 * (losses[0] = auxiliary loss, losses[1] = z-loss; 2 f32, device, out),
 * copied on the stream.  Only a forward whose config has a nonzero
 * aux_loss_coeff or z_loss_coeff computes them: otherwise
 * MOE_ERR_INVALID_ARG. */
moe_status_t moe_layer_losses(const moe_config_t* cfg, float* losses, void* ws, size_t ws_bytes,
                              moe_stream_t stream);

/* The whole backward layer pass after moe_layer_fwd with MOE_FLAG_SAVE_FOR_BWD
 * on the same workspace and inputs: dy [T,h] -> dx [T,h] (routed experts +
 * shared expert + router), dw_r [E,h] f32, db_r [E] f32 or NULL (gradient of
 * the gate bias), dw1, dw2 and, with a shared expert, dw1_shared [2F][h],
 * dw2_shared [h][F]. */
moe_status_t moe_layer_bwd(const moe_config_t* cfg, const void* x, const float* w_r,
                           const void* w1, const void* w2, const void* w1_shared,
                           const void* w2_shared, const void* dy, void* dx, float* dw_r,
                           float* db_r, void* dw1, void* dw2, void* dw1_shared, void* dw2_shared,
                           void* ws, size_t ws_bytes, moe_stream_t stream);

/* Bytes of host-visible state: none.  Reports (and clears) the per-device
 * status word written by device-side checks, after synchronising `stream`.
 * Returns MOE_OK, MOE_ERR_TIMEOUT, MOE_ERR_DEVICE_BOUNDS or MOE_ERR_CUDA. */
moe_status_t moe_get_error(moe_stream_t stream);

/* A static string naming a status code. */
const char* moe_status_string(moe_status_t status);

/* Library version, "major.minor.patch". */
const char* moe_version(void);

/* Stage timing for profilers and benchmarks (a measurement aid, not part of
 * the method; the pages' counterpart is the per-stage time breakdown of the
 * review page, §1.3 and §8).  Registers, for the calling host thread, up to
 * 16 CUDA events (cudaEvent_t, created by the caller on the device the layer
 * runs on) that moe_layer_fwd (pass MOE_PASS_FWD) or moe_layer_bwd
 * (MOE_PASS_BWD) record with cudaEventRecord on their own stream at stage
 * boundary i, for i < n and events[i] != NULL:
 *   forward:  0 start, 1 after route, 2 after dispatch, 3 after FC1,
 *             4 after FC2, 5 after the shared expert, 6 after combine;
 *   backward: 0 start, 1 after the dy scatter, 2 after the FC2 data gradient,
 *             3 after dW2, 4 after the FC1 data gradient, 5 after dW1,
 *             6 after the shared expert, 7 after the router, 8 after combine.
 * So the time between events 4 and 5 of the backward is the dW1 grouped GEMM
 * alone, on the stream that launched it.  n = 0 clears the pass.  The events
 * stay registered until replaced; a failed record returns MOE_ERR_CUDA from
 * the layer call.  Only the layer calls record; other entry points ignore the
 * registration.  Errors: MOE_ERR_INVALID_ARG for an unknown pass, n outside
 * [0, 16], or events NULL with n > 0. */
typedef enum { MOE_PASS_FWD = 0, MOE_PASS_BWD = 1 } moe_pass_t;
moe_status_t moe_set_stage_events(int32_t pass, void* const* events, int32_t n);

/* Test hook for the bounded-wait machinery: launches one block that waits on
 * an mbarrier nothing will ever complete, with the same bounded wait the
 * tensor-core GEMM uses, capped at `max_polls` polls.  The kernel gives up,
 * records MOE_ERR_TIMEOUT in the status word and returns; read it with
 * moe_get_error.  Never faults or hangs the device. */
moe_status_t moe_test_bounded_wait(int64_t max_polls, moe_stream_t stream);

/* Test hook (host-side fault injection, no device involvement): the next n
 * calls that would enqueue GPU work fail as if their first CUDA runtime call
 * had failed -- they return MOE_ERR_CUDA after validating their arguments and
 * before anything is enqueued.  Returns the number of injected failures that
 * were still pending (-1 if n < 0); n = 0 clears them. */
int32_t moe_test_inject_cuda_failure(int32_t n);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_H_ */
