// Host-side launchers of the MoE layer kernels.  Internal header shared by
// the kernel translation units and the C ABI (api.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

#include "moe_b300.h"

namespace moe {

constexpr int kMaxDevices = 64;

// Host state kept per CUDA device (a raised shared-memory limit, an
// occupancy figure, a symbol address): one value per device, filled the
// first time that device asks for it, under a lock, so host threads on the
// same or on different devices never see a half-written entry.
template <typename T>
class PerDevice {
 public:
  // The value for the current device.  On first use `init(T &)` fills it;
  // when init fails its error is returned and nothing is kept.
  template <typename F>
  cudaError_t get(T *out, F init) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu_);
    if (!set_[dev]) {
      T v{};
      e = init(v);
      if (e != cudaSuccess) return e;
      val_[dev] = v;
      set_[dev] = true;
    }
    *out = val_[dev];
    return cudaSuccess;
  }

 private:
  std::mutex mu_;
  bool set_[kMaxDevices] = {};
  T val_[kMaxDevices] = {};
};

// Tokens per gate/routing CTA; the slot scan works on per-CTA histograms.
constexpr int kRouteTokensPerCta = 128;

// 2-D bf16 TMA tensor map over a row-major [outer, inner] matrix with a box
// of [box_outer, box_inner] elements, 128-byte swizzle and zero fill out of
// bounds.  False when the driver entry point is missing or the encoding is
// rejected (misaligned base or stride, box too large).
bool make_bf16_map(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer,
                   uint32_t box_inner, uint32_t box_outer);

// ---------------------------------------------------------------- routing
// In-layer randomness of the gate (see rng.cuh): the noise policy, the
// second-choice sampling and random token selection, and the Philox key.
struct RouteNoise {
  int policy;        // MOE_NOISE_*
  int second;        // sampled second choice (k = 2)
  int rts;           // random token selection
  float jitter_eps;
  uint64_t seed, offset;
  __host__ __device__ bool any() const { return policy != 0 || second != 0 || rts != 0; }
  __host__ __device__ bool gumbel(int k) const {
    return policy == MOE_NOISE_RSAMPLE || (second != 0 && k == 2);
  }
};

struct RouteArgs {
  const float *logits;  // [S,E] fp32 (bias included)
  int64_t S;
  int E, k;
  int64_t cap;          // -1: no capacity limit
  float inv_temp;       // 1 / gate temperature: p = softmax(logits * inv_temp)
  int aux_type;         // MOE_AUX_LOAD or MOE_AUX_STD
  float *probs;         // [S,E] or null
  int32_t *idx;         // [S,k]
  float *w;             // [S,k]
  int32_t *slot;        // [S,k]
  int32_t *routed, *kept, *offsets;  // [E], [E], [E+1]
  int32_t *row_src;     // [rows]
  float *l_aux;
  RouteNoise noise;      // zero: plain top-k in token order
  // workspace views
  int32_t *hist;        // [nblk][k][E] per-CTA counts, then their scan
  float *psum;          // [nblk][E] per-CTA probability sums
  int32_t *first_cnt;   // [E]
};
size_t route_workspace_bytes(int64_t S, int E, int k);
void route_carve_workspace(RouteArgs &a, void *ws);
// steps 1-3 from fp32 logits in memory
cudaError_t launch_route(const RouteArgs &a, cudaStream_t st);
// steps 2-3 only (after the fused gate wrote the per-CTA counts)
cudaError_t launch_route_finish(const RouteArgs &a, cudaStream_t st);

// Fused bf16 gate: router GEMM on the tensor cores + routing step 1.
struct GateTcArgs {
  const void *x, *w_gate;   // bf16 [S,d], [E,d]
  int64_t S;
  int d, E, k;
  const float *logit_bias;  // [E] (bias_ld 0) or [S,E] (bias_ld E), or null
  int bias_ld;
  float inv_temp;           // 1 / gate temperature
  float *logits, *probs;    // [S,E] or null
  int32_t *idx;
  float *w;
  int32_t *rank;            // the slot buffer, holding CTA ranks until step 3
  int32_t *hist;
  float *psum;
  unsigned int *err;
};
cudaError_t launch_gate_tc(const GateTcArgs &a, cudaStream_t st);

// Single-launch bf16 gate: the fused gate above plus the slot scan and
// assignment, counts, offsets and l_aux, with a grid-wide barrier between
// the two halves.  Returns cudaErrorNotSupported (enqueueing nothing) when
// the batch does not fit one wave of tiles of at most 128 tokens per SM or
// the workspace is too small; the caller then takes the three-launch path.
struct GateRouteArgs {
  const void *x, *w_gate;   // bf16 [S,d], [E,d]
  int64_t S;
  int d, E, k;
  int64_t cap;              // -1: no capacity limit
  int64_t rows_alloc;       // rows of the expert-major buffers (moe_max_rows)
  const float *logit_bias;  // [E] (bias_ld 0) or [S,E] (bias_ld E), or null
  int bias_ld;
  float inv_temp;
  int aux_type;
  float *logits, *probs;    // [S,E] or null
  int32_t *idx;
  float *w;
  int32_t *slot;
  int32_t *routed, *kept, *offsets, *row_src;
  float *l_aux;
  void *ws;                 // per-tile counts and probability sums
  size_t ws_bytes;
  unsigned int *err;
};
cudaError_t launch_gate_route(const GateRouteArgs &a, cudaStream_t st);
// The single-launch gate's progress-wait limit on the current device
// (0: the default 2 s); synchronous.
cudaError_t set_gate_wait_limit(uint64_t ns);

// ------------------------------------------------------ SIMT grouped GEMM
// C(m,n) = epilogue( sum_k A(m,k) * B(n,k) ) with arbitrary element strides.
//  mode 0: one GEMM of M x N x K.
//  mode 1: row-grouped.  Rows [offsets[g], offsets[g+1]) of A and C use
//          B + g*b_g and bias + g*bias_g.  M is unused; grid covers max_rows.
//  mode 2: K-grouped.  C_g = sum over rows r in [offsets[g], offsets[g+1])
//          of A(m,r) B(n,r), stored at C + g*c_g (zero when the group is
//          empty).
// Epilogue order: + bias (+ bias_f32), store pre (if set), act (if >= 0),
// times act'(grad_src(m,n)) (if grad_src set, derivative of dact).
struct SimtGemm {
  int a_dtype, b_dtype, c_dtype;
  const void *A; int64_t a_m, a_k;
  const void *B; int64_t b_n, b_k, b_g;
  void *C; int64_t c_m, c_n, c_g;
  int64_t M; int N, K;
  int mode;
  const int32_t *offsets; int G;
  int64_t max_rows;
  const void *bias; int64_t bias_g;     // element type b_dtype
  const float *bias_f32;                // fp32 bias over n (mode 0): bias_f32[m*ld + n]
  int64_t bias_f32_ld;                  // 0: one row for all m
  int act;                              // -1 none
  void *pre;                            // same layout/type as C
  const void *grad_src; int dact;       // same layout/type as C
};
cudaError_t launch_simt_gemm(const SimtGemm &g, cudaStream_t st);

// ------------------------------------------------ tcgen05 grouped GEMM
// Row-grouped bf16 GEMM on the 5th-generation tensor cores:
//   C[r, n] = epi( sum_k A[r, k] * B_g(n, k) )  for r in group g's rows,
// A: [rows, K] bf16 row-major.  B_g: rows g*N .. g*N+N-1 of a [G*N, K]
// (b_kmajor) or columns of a [G*K, N] (!b_kmajor) bf16 matrix.
// Epilogue: + bias[g*N + n] (bf16, nullable), store pre (bf16, nullable),
// act (>= 0), times act'(grad_src[r, n]) when grad_src is set; C bf16.
// Gather form (row_src set): A is the token matrix x [rows_alloc = S, K]
// and row r of the grouped operand is token row_src[r] / k_choices of it
// (the dispatch copy fused into the GEMM); C, pre and the groups keep the
// expert-major row order.  Needs b_kmajor and CTA pairs.
// Router form (c_f32 set; one group, !b_kmajor, CTA pairs): row k of B is
// row k mod b_wrap of a [b_rows, N] matrix (rows past b_rows read as zero)
// and the epilogue stores the fp32 accumulator to c_f32 [rows, N] (no bias,
// activation or bf16 output).
struct TcGemm {
  const void *A; int64_t rows_alloc;   // rows of the A/C allocations
  const void *B; bool b_kmajor;
  void *C;
  int N, K, G;
  const int32_t *offsets;  // [G+1] on the device; null: one group of rows_alloc rows
  const void *bias;
  int act;
  void *pre;
  const void *grad_src; int dact;
  unsigned int *err;
  const int32_t *row_src;  // gather form: [rows] s*k+j of each row, else null
  int k_choices;
  int b_wrap, b_rows;      // router form: K rows of B repeat every b_wrap rows (0: off)
  float *c_f32;
  // data-gradient form with grad_src (CTA pairs): the epilogue also writes
  // partial column sums of its (fp32) output, bias_grad_part_bytes() of
  // them, which launch_bias_grad_reduce adds into the bias gradient
  float *col_part;
};
size_t bias_grad_part_bytes(int64_t max_rows, int G, int N);
cudaError_t launch_bias_grad_reduce(const float *part, const int32_t *offsets, int G, int N,
                                    void *db, cudaStream_t st);
cudaError_t launch_tc_gemm(const TcGemm &g, cudaStream_t st);

// K-grouped bf16 weight-gradient GEMM on the tensor cores:
//   C_g[m, n] = sum over rows r of group g of A[r, m] * B[r, n]
// A: [rows, M] bf16, B: [rows, N] bf16 (both row-major), C: [G, M, N] bf16.
// colsum (nullable): [G, M] bf16, the column sums of A over each group's
// rows (the bias gradient that goes with the weight gradient).
// Cf (fp32, nullable) replaces C; offsets == null makes group g the rows
// [g * chunk_rows, min((g + 1) * chunk_rows, rows_alloc)) (a split of one
// long reduction into partial sums, each written to its own C_g); single
// takes the one-CTA kernel.  group_maps (nullable, CTA pairs): device
// memory for 2 * G tensor maps (128 bytes each, 128-byte aligned) that a
// setup launch fills with the operands' maps cut to each group's end row,
// so the groups' partial last K blocks load with zeros past the group.
constexpr size_t kTensorMapBytes = 128;
struct TcWgrad {
  const void *A; const void *B; int64_t rows_alloc;
  void *C;
  int M, N, G;
  const int32_t *offsets;
  void *colsum;
  unsigned int *err;
  float *Cf;
  int chunk_rows;
  bool single;
  void *group_maps;
};
cudaError_t launch_tc_wgrad(const TcWgrad &g, cudaStream_t st);

// ------------------------------------------------ dispatch / combine
cudaError_t launch_dispatch(const void *x, int dtype, int64_t S, int d, int k,
                            const int32_t *idx, const int32_t *slot,
                            const int32_t *offsets, void *x_disp, cudaStream_t st);
// y[s] = res[s] (when res is not null) + sum_j w[s,j] * out_disp[row(s,j)];
// with mix ([S,2] fp32) set as well: y[s] = mix[s,1] res[s] + mix[s,0] sum_j ...
cudaError_t launch_combine(const void *out_disp, int dtype, int64_t S, int d,
                           int k, const int32_t *idx, const int32_t *slot,
                           const int32_t *offsets, const float *w, void *y,
                           cudaStream_t st, const void *res = nullptr,
                           const float *mix = nullptr);
// mix[s] = softmax over two of (x[s] . cw[j] + cb[j]); cw [2,d], cb [2] in
// the layer dtype, mix [S,2] fp32.
cudaError_t launch_residual_mix(const void *x, int dtype, int64_t S, int d,
                                const void *cw, const void *cb, float *mix,
                                cudaStream_t st);

// ------------------------------------------------ backward helpers
// dO[row] = w * dY[s], dw[s,j] = <dY[s], out[row]> (0 when dropped);
// rows (nullable): [S, k] the row of each choice, -1 when dropped.
cudaError_t launch_combine_bwd(const void *dy, const void *out_disp, int dtype,
                               int64_t S, int d, int k, const int32_t *idx,
                               const int32_t *slot, const int32_t *offsets,
                               const float *w, void *d_out, float *dw,
                               cudaStream_t st, int32_t *rows = nullptr);
// db[g, n] = sum over group rows of M[r, n]  (zero for empty groups).
cudaError_t launch_group_colsum(const void *M, int dtype, int N, int G,
                                const int32_t *offsets, void *db,
                                cudaStream_t st);
// coef[e] = d l_aux / d p[s,e] (the same for every token): E*first[e]/S^2
// for MOE_AUX_LOAD, (u_e - mean u) / (E * S * std u) with u_e = mean_s
// p[s,e] for MOE_AUX_STD (0 when std u = 0).
cudaError_t launch_aux_coef(const int32_t *idx, const float *probs, int64_t S, int k, int E,
                            int aux_type, float *coef, cudaStream_t st);
// dlogits = inv_temp * p * (dp - <dp,p>), dp from dw through the weights
// and the l_aux term aux_w * coef[e]: the gradient of the logits the gate
// GEMM produced (before the 1/T scaling).
// dlogits (fp32, nullable); dl2 (bf16, nullable): [S, 2P] rows holding
// hi = bf16(dlogits) in columns [0, E) and lo = bf16(dlogits - hi) in
// [P, P + E), zeros elsewhere -- the tensor-core operand of the router's
// backward products (hi + lo carries dlogits to about 2^-17).
cudaError_t launch_gate_bwd(const float *probs, const int32_t *idx,
                            const float *dw, const float *coef, int64_t S,
                            int E, int k, float aux_w, float inv_temp, float *dlogits,
                            void *dl2, int P, cudaStream_t st);
// ---- router backward on the tensor cores (bf16 layers)
// P = E rounded up to 64: the half width of the [S, 2P] hi/lo operand.
inline int router_pad(int E) { return (E + 63) / 64 * 64; }
// dW_g = dlogits^T x as x^T [hi | lo] over token chunks (fp32 partial sums
// [chunks, d, 2P], one-CTA K-grouped tensor-core GEMM), then a fixed-order
// sum of the chunks and of the two halves.
int gate_wgrad_tc_chunks(int64_t S, int d);
size_t gate_wgrad_tc_partial_bytes(int64_t S, int E, int d);
cudaError_t launch_gate_wgrad_tc(const void *x, const void *dl2, int64_t S, int d, int E,
                                 float *partial, void *dw_gate, unsigned int *err,
                                 cudaStream_t st);
// dX = r * f + sum_j dx_disp[rows[s, j]] with the router term
// r = [hi | lo] [W_g; W_g] (fp32 [S, d], the CTA-pair GEMM's router form)
// and f the jitter factor (1 without jitter).
cudaError_t launch_dx_router_tc(const void *dl2, const void *w_gate, const void *dx_disp,
                                int64_t S, int d, int E, int k, const int32_t *rows,
                                float *rterm, void *dx, const RouteNoise *jitter,
                                unsigned int *err, cudaStream_t st);
// dW_g = dlogits^T x: token-split fp32 partial sums, then a fixed-order sum.
int64_t gate_wgrad_splits(int64_t S);
size_t gate_wgrad_partial_bytes(int64_t S, int E, int d);
cudaError_t launch_gate_wgrad(const float *dlogits, const void *x, int dtype, int64_t S, int d,
                              int E, float *partial, void *dw_gate, cudaStream_t st);
// dx[s] = sum_j dx_disp[row(s,j)] + (dlogits[s] . w_gate) (* f[s] when
// `jitter` is set: the router saw x * f)
cudaError_t launch_dx_combine(const void *dx_disp, const float *dlogits,
                              const void *w_gate, int dtype, int64_t S, int d,
                              int E, int k, const int32_t *idx,
                              const int32_t *slot, const int32_t *offsets,
                              void *dx, cudaStream_t st, const RouteNoise *jitter = nullptr);

// The gate's draws for a configuration (moe_gate_noise): uniforms and
// Gumbel noise [S,E], random-token-selection positions [S]; each nullable.
cudaError_t launch_gate_noise(int64_t S, int E, const RouteNoise &n, float *uniform,
                              float *gumbel, int32_t *position, cudaStream_t st);
// The jittered router input xj = x * f (float32 product, rounded to the
// layer type), [S,d].
cudaError_t launch_jitter(const void *x, int dtype, int64_t S, int d, const RouteNoise &n,
                          void *xj, cudaStream_t st);

int num_sms();

}  // namespace moe
