/*
 * moe_b300.h -- C ABI of a single-GPU top-k gated Mixture-of-Experts FFN
 * layer for NVIDIA B300 (sm_103a).
 *
 * The layer is the one described by the deepspeed.moe overview page
 * (adg.csdn.net/694deb285b9f5f31781ae763, §2.1 "MoE 层": the constructor
 * MoE(hidden_size, expert, num_experts, k, capacity_factor, min_capacity,
 * drop_tokens, ...) returning (output, gate_loss, expert_count); §3.1 "MoE 层
 * 前向传播": gate -> top-k -> dispatch -> experts -> weighted merge -> balance
 * loss) and by the MoELayer pseudocode of the MoE explainer page
 * (lpnh.cn/news/725941, §3.1, Steps 1-5).  Expert-parallel communication is
 * not part of this library: every stage runs on one GPU.
 *
 * Conventions for every entry point
 * ---------------------------------
 *  - S = num_tokens, d = hidden_size, f = ffn_size, E = num_experts.
 *  - All tensors are dense, row-major and contiguous.  Weights use the
 *    nn.Linear layout (out x in):  w_gate[E,d], w1[E,f,d], w2[E,d,f],
 *    b1[E,f], b2[E,d].
 *  - "T" below is the configuration's element type (cfg->dtype): float for
 *    MOE_F32, __nv_bfloat16 for MOE_BF16.  Routing tensors are int32/float.
 *  - Every pointer except the config is a DEVICE pointer, allocated and owned
 *    by the caller.  The library never allocates device memory, never frees,
 *    never synchronises the stream and never reads device results on the
 *    host.  Work is enqueued on `stream` (0 = legacy default stream).
 *  - Buffers indexed by "rows" hold the expert-major copy of kept tokens and
 *    must have room for moe_max_rows(cfg) rows; the number actually used is
 *    expert_offsets[E], which stays on the device.
 *  - Argument checks run on the host before anything is enqueued; a failed
 *    check returns MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED /
 *    MOE_ERR_WORKSPACE and enqueues nothing.  A CUDA launch error returns
 *    MOE_ERR_CUDA.  Kernels that detect a fault on the device (a bounded wait
 *    that gave up) record it in a device error word read by
 *    moe_get_device_error().
 *  - Requirements: 1 <= k <= 2, k <= E <= 256, d and f multiples of 8,
 *    d, f >= 8, S < 2^31 / k, every pointer 16-byte aligned.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t. */
typedef struct CUstream_st *moe_stream_t;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size or config */
  MOE_ERR_UNSUPPORTED = 2, /* valid but outside this build's limits        */
  MOE_ERR_WORKSPACE = 3,   /* workspace smaller than moe_workspace_size()  */
  MOE_ERR_CUDA = 4,        /* a CUDA call or launch failed                 */
  MOE_ERR_DEVICE = 5       /* a kernel recorded a device-side fault        */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

typedef enum {
  MOE_ACT_RELU = 0,      /* max(0, z)                                       */
  MOE_ACT_GELU_TANH = 1, /* 0.5 z (1 + tanh(sqrt(2/pi) (z + 0.044715 z^3)))  */
  MOE_ACT_GELU_ERF = 2   /* 0.5 z (1 + erf(z / sqrt 2))                      */
} moe_act;

typedef enum {
  MOE_AUX_LOAD = 0, /* l_aux = E * sum_e mean_s(p[s,e]) * first[e] / S           */
  MOE_AUX_STD = 1   /* l_aux = std_e(mean_s p[s,e]) + 1e-6 (population std)    */
} moe_aux_loss;

typedef enum {
  MOE_NOISE_NONE = 0,
  MOE_NOISE_JITTER = 1,  /* router input x * U(1-eps, 1+eps)                   */
  MOE_NOISE_RSAMPLE = 2  /* choose the top-k of logits + Gumbel noise          */
} moe_noise_policy;

/* Mirrors MoE(hidden_size, num_experts, k, capacity_factor, min_capacity,
 * drop_tokens) of the deepspeed.moe overview, §2.1, plus the expert FFN
 * width, activation, element type and the weight of l_aux in the training
 * loss L = <dY, y> + aux_loss_weight * l_aux, and three gating variants:
 *  - gate_temperature T (the gating_softmax_temp of the DeepSpeed config on
 *    the ZeRO-3 + MoE page): p = softmax(logits / T); T = 0 means 1.  The
 *    top-k choice is unchanged for any T > 0.
 *  - aux_loss_type: the balance loss of the layer's specification, or the
 *    DeepSeek-MoE page's std-based alternative lambda * (std(usage) + 1e-6)
 *    with usage[e] = mean over tokens of p[s,e] (ch.1 load-balancing table).
 *  - logit_bias_per_token: logit_bias is [S,E] instead of [E]: noise the
 *    caller draws itself and adds to the gate logits.  A per-token bias gets
 *    no gradient.
 * and the randomised gate options the overview names in §2.1 without
 * formulas, drawn inside the layer from Philox4x32-10 (Salmon et al., SC
 * 2011) keyed by noise_seed and noise_offset, so a run is reproducible:
 *  - noise_policy (noisy_gate_policy): MOE_NOISE_RSAMPLE chooses the experts
 *    as the top-k of the float32 keys logits + g, g standard Gumbel noise
 *    (a sample of the softmax); probabilities and combine weights stay those
 *    of the noise-free logits.  MOE_NOISE_JITTER feeds the router x * f,
 *    f = 1 + jitter_eps * (2u - 1) per element (float32, then rounded to the
 *    layer type); the experts see x.
 *  - second_expert_sampling (top2_2nd_expert_sampling, k = 2): the first
 *    choice stays the arg-max logit, the second is the arg-max of logits + g
 *    over the other experts.
 *  - use_rts (random token selection): each expert's capacity queue takes
 *    the first choices, then the second choices, each in a keyed random
 *    order of the tokens (a Philox Feistel permutation) instead of token
 *    order, so which tokens are dropped is random.
 * The noise is a constant of the backward (jitter: dW_g uses x * f and the
 * router's part of dX is multiplied by f).  moe_gate_noise returns the draws
 * of a configuration. */
typedef struct {
  int64_t num_tokens;      /* S >= 0                                        */
  int32_t hidden_size;     /* d                                             */
  int32_t ffn_size;        /* f                                             */
  int32_t num_experts;     /* E                                             */
  int32_t k;               /* experts per token, 1 or 2                      */
  double capacity_factor;  /* > 0; read as a decimal with 6 fraction digits  */
  int32_t min_capacity;    /* >= 0                                          */
  int32_t drop_tokens;     /* nonzero: cap each expert at the capacity       */
  int32_t act;             /* moe_act                                        */
  int32_t dtype;           /* moe_dtype                                      */
  float aux_loss_weight;   /* backward only                                  */
  float gate_temperature;  /* >= 0; 0 or 1 = plain softmax                   */
  int32_t aux_loss_type;   /* moe_aux_loss                                   */
  int32_t logit_bias_per_token; /* nonzero: logit_bias is [S,E], else [E]    */
  int32_t noise_policy;    /* moe_noise_policy                               */
  int32_t second_expert_sampling; /* nonzero (k = 2 only): sampled 2nd choice */
  int32_t use_rts;         /* nonzero: random token selection                */
  float jitter_eps;        /* MOE_NOISE_JITTER half-width; 0 means 0.01      */
  uint64_t noise_seed;     /* Philox key                                     */
  uint64_t noise_offset;   /* Philox counter words 2-3 (a new draw per step) */
} moe_config;

/* Saved state of one forward pass (all device pointers, caller-owned).
 * Written by moe_forward, read by moe_backward. */
typedef struct {
  float *logits;          /* [S,E] fp32 router logits (nullable in forward) */
  float *probs;           /* [S,E] fp32 softmax (required for backward)     */
  int32_t *topk_idx;      /* [S,k] chosen experts, choice 0 = arg-max       */
  float *topk_w;          /* [S,k] combine weights                          */
  int32_t *slot;          /* [S,k] slot in the expert's queue, -1 = dropped */
  int32_t *routed_cnt;    /* [E] tokens that chose the expert               */
  int32_t *kept_cnt;      /* [E] tokens kept = expert_count                 */
  int32_t *expert_offsets;/* [E+1] exclusive scan of kept_cnt               */
  int32_t *row_src;       /* [rows] s*k+j of the choice stored in each row  */
  float *l_aux;           /* [1] load-balancing loss                        */
  void *x_disp;           /* [rows,d] T expert-major token copy; NULL in a
                             bf16 forward: the dispatch is then fused into
                             the first expert GEMM (moe_expert_ffn_gather)
                             and no copy is made.  moe_backward needs it. */
  void *h_pre;            /* [rows,f] T pre-activation (nullable forward)   */
  void *h;                /* [rows,f] T activation                          */
  void *out_disp;         /* [rows,d] T expert outputs                      */
} moe_buffers;

/* Status name, e.g. "MOE_ERR_INVALID_ARG".  Never NULL. */
const char *moe_status_string(moe_status st);

/* Per-expert capacity C = max(min_capacity, ceil(S*k*cf/E)), exact for cf
 * with at most 6 decimal digits (capacity table of the DeepSeek-MoE page,
 * lnwmold.com/news/1162317 ch.1; min_capacity and drop_tokens of the
 * deepspeed.moe overview §2.1).  *cap = -1 when drop_tokens is 0 (no cap).
 * Host only. */
moe_status moe_capacity(const moe_config *cfg, int64_t *cap);

/* Rows the expert-major buffers need: min(S*k, E*C) with a cap, S*k
 * without.  Host only. */
moe_status moe_max_rows(const moe_config *cfg, int64_t *rows);

/* Bytes of scratch the entry points need for this config: forward-only
 * entry points when for_backward == 0, moe_backward when nonzero.  The
 * caller passes a device buffer of at least this size (16-byte aligned). */
moe_status moe_workspace_size(const moe_config *cfg, int for_backward,
                              size_t *bytes);

/* Gate (MoE explainer §3.1 Steps 1-2; DeepSeek-MoE page ch.1 moe_forward and
 * capacity table; deepspeed.moe overview §2.1 drop_tokens / expert_count):
 *   logits = x w_gate^T + logit_bias          (fp32 accumulation)
 *   probs = softmax(logits / T), T = cfg->gate_temperature
 *   topk_idx: arg-max logit, then arg-max of the rest; ties -> lower index
 *   topk_w: k=2 -> p_j / (p_1 + p_2);  k=1 -> p_1
 *   slot: queue position per expert, all first choices in token order before
 *         any second choice; slot >= capacity -> -1 (dropped)
 *   routed_cnt[e], kept_cnt[e], expert_offsets = exclusive scan of kept_cnt,
 *   row_src[offsets[e]+slot] = s*k+j,
 *   l_aux = E * sum_e mean_s(p[s,e]) * (first-choice count of e)/S, or the
 *           std form when cfg->aux_loss_type is MOE_AUX_STD.
 * x: [S,d] T.  w_gate: [E,d] T.  logit_bias: fp32, [E] (or [S,E] when
 * cfg->logit_bias_per_token), or NULL.
 * logits, probs: [S,E] fp32 or NULL (not written).  Other outputs as in
 * moe_buffers.  workspace: moe_workspace_size(cfg, 0) bytes. */
moe_status moe_gate_topk(const moe_config *cfg, const void *x,
                         const void *w_gate, const float *logit_bias,
                         float *logits, float *probs, int32_t *topk_idx,
                         float *topk_w, int32_t *slot, int32_t *routed_cnt,
                         int32_t *kept_cnt, int32_t *expert_offsets,
                         int32_t *row_src, float *l_aux, void *workspace,
                         size_t workspace_bytes, moe_stream_t stream);

/* moe_gate_topk without a workspace argument, for callers that cannot
 * allocate device memory: code that is handed only its input and output
 * buffers and a stream (a plugin inside another engine, a server that
 * forbids allocation after start-up) and so cannot supply the scratch
 * moe_gate_topk needs.  The pages have no counterpart to this entry point.
 * Same arguments, outputs and results as moe_gate_topk; the caller still
 * passes every input and output.  The scratch is a 16 MiB array compiled
 * into the library, held by every GPU that loads the library until the
 * process exits.  Configurations whose moe_workspace_size(cfg, 0) exceeds
 * 16 MiB (about S*E > 4.1 million) are rejected with MOE_ERR_WORKSPACE
 * before anything is enqueued.  The first call on each device looks up the
 * array's device address (cudaGetSymbolAddress, with that device current);
 * make that first call before any stream capture.  Allocates nothing: no
 * cudaMalloc, cudaFree or allocating library call.  All calls on a device
 * share the one array, so calls that can overlap on the GPU (different
 * streams, or different host threads) race and must be serialised by the
 * caller; results never depend on what an earlier call left there. */
moe_status moe_gate_topk_static(const moe_config *cfg, const void *x,
                                const void *w_gate, const float *logit_bias,
                                float *logits, float *probs,
                                int32_t *topk_idx, float *topk_w,
                                int32_t *slot, int32_t *routed_cnt,
                                int32_t *kept_cnt, int32_t *expert_offsets,
                                int32_t *row_src, float *l_aux,
                                moe_stream_t stream);

/* The random draws the gate makes for this configuration (no other
 * output): uniform [S,E] fp32, the uniforms u of the gate-noise stream;
 * gumbel [S,E] fp32, -ln(-ln u) as the gate adds them to the logits under
 * MOE_NOISE_RSAMPLE or second-expert sampling; position [S] int32, the
 * queue position of each token under random token selection.  Each may be
 * NULL.  The values do not depend on the noise options that are set; the
 * gate uses them only where its options say so. */
moe_status moe_gate_noise(const moe_config *cfg, float *uniform, float *gumbel,
                          int32_t *position, moe_stream_t stream);

/* The routing half of moe_gate_topk, taking the logits as input instead of
 * computing them (the same kernels; used to check routing bit for bit
 * against a reference that is fed identical fp32 logits).
 * logits: [S,E] fp32 input.  probs may be NULL. */
moe_status moe_route_from_logits(const moe_config *cfg, const float *logits,
                                 float *probs, int32_t *topk_idx,
                                 float *topk_w, int32_t *slot,
                                 int32_t *routed_cnt, int32_t *kept_cnt,
                                 int32_t *expert_offsets, int32_t *row_src,
                                 float *l_aux, void *workspace,
                                 size_t workspace_bytes, moe_stream_t stream);

/* Dispatch (MoE explainer §3.1 Step 3, "flatten & scatter"):
 * x_disp[expert_offsets[e] + slot[s,j]] = x[s] for every kept (s,j).
 * x: [S,d] T; x_disp: [rows,d] T.  Rows past expert_offsets[E] untouched. */
moe_status moe_dispatch(const moe_config *cfg, const void *x,
                        const int32_t *topk_idx, const int32_t *slot,
                        const int32_t *expert_offsets, void *x_disp,
                        moe_stream_t stream);

/* Grouped expert FFN (MoE explainer §3.1 Step 4, Linear -> act -> Linear)
 * over the contiguous row block [expert_offsets[e], expert_offsets[e+1]) of
 * each expert e:
 *   h_pre = x_disp W1_e^T + b1_e ;  h = act(h_pre) ;  out = h W2_e^T + b2_e
 * with fp32 accumulation; h_pre, h, out_disp are stored as T.
 * x_disp: [rows,d]; w1: [E,f,d]; b1: [E,f]; w2: [E,d,f]; b2: [E,d];
 * h_pre: [rows,f] or NULL; h: [rows,f]; out_disp: [rows,d]. */
moe_status moe_expert_ffn(const moe_config *cfg, const void *x_disp,
                          const int32_t *expert_offsets, const void *w1,
                          const void *b1, const void *w2, const void *b2,
                          void *h_pre, void *h, void *out_disp,
                          moe_stream_t stream);

/* Dispatch fused into the grouped expert FFN, for bf16 layers: the same
 * h_pre, h and out_disp as moe_dispatch followed by moe_expert_ffn, bit for
 * bit, without the expert-major copy x_disp.  The first GEMM reads row r of
 * expert e's block straight from token row_src[r] / k of x into its operand
 * ring (MoE explainer §3.1: dispatch, expert compute and combine fused, no
 * flattened intermediate buffer; deepspeed.moe overview §3.4, fused
 * kernels).  x: [S,d] T; row_src, expert_offsets: moe_gate_topk's outputs;
 * the other arguments as moe_expert_ffn.  MOE_ERR_UNSUPPORTED for fp32
 * layers and on a device with fewer than two SMs. */
moe_status moe_expert_ffn_gather(const moe_config *cfg, const void *x,
                                 const int32_t *row_src,
                                 const int32_t *expert_offsets, const void *w1,
                                 const void *b1, const void *w2, const void *b2,
                                 void *h_pre, void *h, void *out_disp,
                                 moe_stream_t stream);

/* Combine (MoE explainer §3.1 Step 5 "gather weighted sum"; deepspeed.moe
 * overview §3.1 item 4): y[s] = sum over kept j of topk_w[s,j] *
 * out_disp[expert_offsets[e]+slot[s,j]], fp32 accumulation; a token with no
 * kept choice gets y[s] = 0.  out_disp: [rows,d] T; y: [S,d] T. */
moe_status moe_combine(const moe_config *cfg, const void *out_disp,
                       const int32_t *topk_idx, const int32_t *slot,
                       const int32_t *expert_offsets, const float *topk_w,
                       void *y, moe_stream_t stream);

/* The whole forward pass (gate, dispatch, expert FFN, combine) on `stream`;
 * returns (y, l_aux, kept_cnt) like MoE.forward's (output, gate_loss,
 * expert_count), deepspeed.moe overview §2.1.  Every non-nullable field of
 * `buf` must be set (h_pre may be NULL when no backward follows; x_disp may
 * be NULL for a bf16 layer, which fuses the dispatch into the first expert
 * GEMM -- keep it set when moe_backward follows).
 * workspace: moe_workspace_size(cfg, 0) bytes. */
moe_status moe_forward(const moe_config *cfg, const void *x,
                       const void *w_gate, const float *logit_bias,
                       const void *w1, const void *b1, const void *w2,
                       const void *b2, void *y, const moe_buffers *buf,
                       void *workspace, size_t workspace_bytes,
                       moe_stream_t stream);

/* The forward pass with PR-MoE's residual expert (deepspeed.moe overview
 * §2.3 / §3.3, MoE(..., use_residual=True), where a fixed dense MLP works
 * beside the routed experts).  The page does not say how the two outputs
 * are mixed; two readings are offered:
 *   mix_w == NULL:  y = MoE(x) + MLP(x)                       (a sum)
 *   mix_w != NULL:  c[s] = softmax over 2 of (x[s] mix_w^T + mix_b),
 *                   y[s] = c[s,0] MoE(x)[s] + c[s,1] MLP(x)[s]
 * with MLP(x) = act(x rw1^T + rb1) rw2^T + rb2 (the shape and activation of
 * one expert) applied to every token.  rw1: [f,d]; rb1: [f]; rw2: [d,f];
 * rb2: [d]; mix_w: [2,d]; mix_b: [2] (all T).  mix: [S,2] fp32 receives c
 * (required with mix_w; mix_b and mix must both be NULL without it, else
 * MOE_ERR_INVALID_ARG).  res_h: [S,f] T and res_out: [S,d] T receive the
 * MLP's activation and output (caller-owned scratch); the other arguments
 * are moe_forward's.  The MLP's output is mixed in inside the combine, in
 * fp32; c is computed with fp32 dot products. */
moe_status moe_forward_residual(const moe_config *cfg, const void *x,
                                const void *w_gate, const float *logit_bias,
                                const void *w1, const void *b1, const void *w2,
                                const void *b2, const void *rw1, const void *rb1,
                                const void *rw2, const void *rb2,
                                const void *mix_w, const void *mix_b, float *mix,
                                void *y, const moe_buffers *buf, void *res_h,
                                void *res_out, void *workspace,
                                size_t workspace_bytes, moe_stream_t stream);

/* Backward of L = <dy, y> + aux_loss_weight * l_aux with the routing held
 * fixed (DeepSeek-MoE page §3.1 TopKRouter: the gradient reaches only the
 * selected logits; §2.1/§2.3: an expert that got no token has zero weight
 * gradient, written out).
 *   dx [S,d] T, dw_gate [E,d] T, dw1 [E,f,d] T, db1 [E,f] T,
 *   dw2 [E,d,f] T, db2 [E,d] T  (fp32 accumulation, stored once as T).
 * `saved` is the moe_buffers of the matching moe_forward, with probs and
 * h_pre set.  workspace: moe_workspace_size(cfg, 1) bytes. */
moe_status moe_backward(const moe_config *cfg, const void *x,
                        const void *w_gate, const void *w1, const void *w2,
                        const moe_buffers *saved, const void *dy, void *dx,
                        void *dw_gate, void *dw1, void *db1, void *dw2,
                        void *db2, void *workspace, size_t workspace_bytes,
                        moe_stream_t stream);

/* Debugging aid: the time limit, on the current device, of the waits of
 * the single-launch bf16 gate kernel that follow its progress (a copy, an
 * MMA, the grid-wide barrier); ns = 0 restores the default of 2 s.  A
 * limit short enough to run out makes the kernel give up, record its code in
 * the device error word (moe_get_device_error), drain its own copies and
 * MMAs and return, leaving its outputs unspecified but in range; the next
 * call with the default limit computes normally.  Synchronous. */
moe_status moe_debug_set_wait_limit(uint64_t ns);

/* Reads and clears the device error word on the current device
 * (synchronous).  *code == 0 means no kernel recorded a fault; otherwise it
 * names the kernel and wait that gave up.  Returns MOE_ERR_DEVICE when
 * *code != 0. */
moe_status moe_get_device_error(uint32_t *code);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */
