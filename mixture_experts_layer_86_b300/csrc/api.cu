// C ABI of the MoE layer library: argument checks, capacity arithmetic,
// workspace layout and the order of kernel launches for each entry point.
// The entry points and their contracts are documented in moe_b300.h.
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "moe_b300.h"

namespace moe {

__device__ unsigned int g_device_error = 0;

namespace {

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

float inv_temperature(const moe_config *c) {
  return c->gate_temperature > 0.0f ? 1.0f / c->gate_temperature : 1.0f;
}

RouteNoise noise_of(const moe_config *c) {
  RouteNoise n{};
  n.policy = c->noise_policy;
  n.second = c->k == 2 ? c->second_expert_sampling : 0;
  n.rts = c->use_rts;
  n.jitter_eps = c->jitter_eps;
  n.seed = c->noise_seed;
  n.offset = c->noise_offset;
  return n;
}

// bytes of the jittered router input (only under MOE_NOISE_JITTER)
size_t jitter_bytes(const moe_config *c) {
  return c->noise_policy == MOE_NOISE_JITTER
             ? align256(size_t(c->num_tokens) * c->hidden_size * elem_bytes(c->dtype))
             : 0;
}

unsigned int *device_error_ptr() {
  static PerDevice<unsigned int *> ptrs;
  unsigned int *p = nullptr;
  if (ptrs.get(&p, [](unsigned int *&v) {
        void *a = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&a, g_device_error);
        v = static_cast<unsigned int *>(a);
        return e;
      }) != cudaSuccess)
    return nullptr;
  return p;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool ok_ptr(const void *p) { return p != nullptr && aligned16(p); }
bool ok_opt(const void *p) { return p == nullptr || aligned16(p); }

moe_status check_config(const moe_config *c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->num_tokens < 0 || c->hidden_size < 8 || c->ffn_size < 8) return MOE_ERR_INVALID_ARG;
  if (c->hidden_size % 8 || c->ffn_size % 8) return MOE_ERR_INVALID_ARG;
  if (c->k < 1 || c->k > 2 || c->num_experts < c->k) return MOE_ERR_INVALID_ARG;
  if (!(c->capacity_factor > 0.0) || c->capacity_factor > 1e6) return MOE_ERR_INVALID_ARG;
  if (c->min_capacity < 0) return MOE_ERR_INVALID_ARG;
  if (c->act < MOE_ACT_RELU || c->act > MOE_ACT_GELU_ERF) return MOE_ERR_INVALID_ARG;
  if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (!(c->gate_temperature >= 0.0f) || c->gate_temperature > 1e30f) return MOE_ERR_INVALID_ARG;
  if (c->aux_loss_type != MOE_AUX_LOAD && c->aux_loss_type != MOE_AUX_STD)
    return MOE_ERR_INVALID_ARG;
  if (c->logit_bias_per_token != 0 && c->logit_bias_per_token != 1) return MOE_ERR_INVALID_ARG;
  if (c->noise_policy < MOE_NOISE_NONE || c->noise_policy > MOE_NOISE_RSAMPLE)
    return MOE_ERR_INVALID_ARG;
  if ((c->second_expert_sampling != 0 && c->second_expert_sampling != 1) ||
      (c->use_rts != 0 && c->use_rts != 1))
    return MOE_ERR_INVALID_ARG;
  if (!(c->jitter_eps >= 0.0f && c->jitter_eps < 1.0f)) return MOE_ERR_INVALID_ARG;
  if (c->num_experts > kMaxExperts) return MOE_ERR_UNSUPPORTED;
  if (c->num_tokens * c->k >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

int64_t capacity_of(const moe_config *c) {
  if (!c->drop_tokens) return -1;
  // cf as an exact decimal with 6 fraction digits: C = ceil(S*k*cf_u / (E*1e6))
  const long long cf_u = llround(c->capacity_factor * 1e6);
  const __int128 num = __int128(c->num_tokens) * c->k * cf_u;
  const __int128 den = __int128(c->num_experts) * 1000000;
  const int64_t cap = int64_t((num + den - 1) / den);
  return cap > c->min_capacity ? cap : int64_t(c->min_capacity);
}

int64_t max_rows_of(const moe_config *c) {
  const int64_t sk = c->num_tokens * c->k;
  const int64_t cap = capacity_of(c);
  if (cap < 0) return sk;
  const int64_t ec = cap * c->num_experts;
  return ec < sk ? ec : sk;
}

// forward workspace: routing scratch | logits scratch | jittered input
size_t fwd_ws_bytes(const moe_config *c) {
  return route_workspace_bytes(c->num_tokens, c->num_experts, c->k) +
         align256(size_t(c->num_tokens) * c->num_experts * 4) + jitter_bytes(c);
}
float *fwd_ws_logits(const moe_config *c, void *ws) {
  return reinterpret_cast<float *>(static_cast<char *>(ws) +
                                   route_workspace_bytes(c->num_tokens, c->num_experts, c->k));
}
void *fwd_ws_jitter(const moe_config *c, void *ws) {
  return static_cast<char *>(ws) + route_workspace_bytes(c->num_tokens, c->num_experts, c->k) +
         align256(size_t(c->num_tokens) * c->num_experts * 4);
}

struct BwdWs {
  void *d_out, *dh_pre, *dx_disp;
  float *dw, *dlogits, *gate_partial;
  float *aux_coef;
  void *xj;       // the jittered router input (MOE_NOISE_JITTER only)
  int32_t *rows;  // [S, k] row of each choice in the expert-major buffers, -1 when dropped
  void *maps;     // per-expert tensor maps of the two weight-gradient GEMMs (bf16)
  float *colpart; // partial column sums of dh_pre from the data-gradient epilogue (bf16)
};

// The router's backward: fp32 layers keep dlogits [S,E] fp32 and CUDA-core
// partials; bf16 layers keep the [S, 2P] hi/lo operand (in the dlogits
// slot) and the tensor-core chunk partials.
size_t bwd_ws_carve(const moe_config *c, void *base, BwdWs *w) {
  const int64_t R = max_rows_of(c);
  const size_t eb = elem_bytes(c->dtype);
  const int64_t S = c->num_tokens;
  const bool tc = c->dtype == MOE_BF16;
  // slot 0 (dO) also holds the router term r [S, d] fp32 of bf16 layers,
  // which is formed after the last use of dO
  const size_t sz[11] = {align256(std::max(size_t(R) * c->hidden_size * eb,
                                          tc ? size_t(S) * c->hidden_size * 4 : size_t(0))),
                        align256(size_t(R) * c->ffn_size * eb),
                        align256(size_t(R) * c->hidden_size * eb),
                        align256(size_t(S) * c->k * 4),
                        align256(tc ? size_t(S) * 2 * router_pad(c->num_experts) * 2
                                    : size_t(S) * c->num_experts * 4),
                        align256(tc ? gate_wgrad_tc_partial_bytes(S, c->num_experts,
                                                                  c->hidden_size)
                                    : gate_wgrad_partial_bytes(S, c->num_experts,
                                                               c->hidden_size)),
                        align256(size_t(c->num_experts) * 4),
                        jitter_bytes(c),
                        align256(size_t(S) * c->k * 4),
                        tc ? align256(size_t(4) * c->num_experts * kTensorMapBytes) : 0,
                        tc ? align256(bias_grad_part_bytes(R, c->num_experts, c->ffn_size)) : 0};
  if (w) {
    char *p = static_cast<char *>(base);
    w->d_out = p; p += sz[0];
    w->dh_pre = p; p += sz[1];
    w->dx_disp = p; p += sz[2];
    w->dw = reinterpret_cast<float *>(p); p += sz[3];
    w->dlogits = reinterpret_cast<float *>(p); p += sz[4];
    w->gate_partial = reinterpret_cast<float *>(p); p += sz[5];
    w->aux_coef = reinterpret_cast<float *>(p); p += sz[6];
    w->xj = sz[7] ? p : nullptr; p += sz[7];
    w->rows = reinterpret_cast<int32_t *>(p); p += sz[8];
    w->maps = sz[9] ? p : nullptr; p += sz[9];
    w->colpart = sz[10] ? reinterpret_cast<float *>(p) : nullptr;
  }
  size_t total = 0;
  for (size_t v : sz) total += v;
  return total;
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

#define MOE_TRY(expr)                       \
  do {                                      \
    const moe_status st__ = (expr);         \
    if (st__ != MOE_OK) return st__;        \
  } while (0)
#define MOE_CUDA(expr) MOE_TRY(cuda_status(expr))

// logits = x w_gate^T (+ bias), fp32 out
moe_status gate_gemm(const moe_config *c, const void *x, const void *w_gate,
                     const float *logit_bias, float *logits, cudaStream_t st) {
  SimtGemm g{};
  g.a_dtype = g.b_dtype = c->dtype;
  g.c_dtype = MOE_F32;
  g.A = x; g.a_m = c->hidden_size; g.a_k = 1;
  g.B = w_gate; g.b_n = c->hidden_size; g.b_k = 1;
  g.C = logits; g.c_m = c->num_experts; g.c_n = 1;
  g.M = c->num_tokens; g.N = c->num_experts; g.K = c->hidden_size;
  g.mode = 0;
  g.bias_f32 = logit_bias;
  g.bias_f32_ld = c->logit_bias_per_token ? c->num_experts : 0;
  g.act = -1;
  return cuda_status(launch_simt_gemm(g, st));
}

moe_status route(const moe_config *c, const float *logits, float *probs, int32_t *idx, float *w,
                 int32_t *slot, int32_t *routed, int32_t *kept, int32_t *offsets,
                 int32_t *row_src, float *l_aux, void *ws, cudaStream_t st) {
  RouteArgs a{};
  a.logits = logits; a.S = c->num_tokens; a.E = c->num_experts; a.k = c->k;
  a.cap = capacity_of(c);
  a.inv_temp = inv_temperature(c);
  a.aux_type = c->aux_loss_type;
  a.probs = probs; a.idx = idx; a.w = w; a.slot = slot;
  a.routed = routed; a.kept = kept; a.offsets = offsets; a.row_src = row_src; a.l_aux = l_aux;
  a.noise = noise_of(c);
  route_carve_workspace(a, ws);
  return cuda_status(launch_route(a, st));
}

moe_status expert_ffn(const moe_config *c, const void *x_disp, const int32_t *offsets,
                      const void *w1, const void *b1, const void *w2, const void *b2, void *h_pre,
                      void *h, void *out, cudaStream_t st) {
  const int64_t R = max_rows_of(c);
  const int d = c->hidden_size, f = c->ffn_size, E = c->num_experts;
  if (R == 0) return MOE_OK;
  if (c->dtype == MOE_BF16) {
    TcGemm g1{};
    g1.A = x_disp; g1.rows_alloc = R; g1.B = w1; g1.b_kmajor = true; g1.C = h;
    g1.N = f; g1.K = d; g1.G = E; g1.offsets = offsets; g1.bias = b1; g1.act = c->act;
    g1.pre = h_pre; g1.grad_src = nullptr; g1.dact = 0; g1.err = device_error_ptr();
    MOE_CUDA(launch_tc_gemm(g1, st));
    TcGemm g2 = g1;
    g2.A = h; g2.B = w2; g2.C = out; g2.N = d; g2.K = f; g2.bias = b2; g2.act = -1;
    g2.pre = nullptr;
    return cuda_status(launch_tc_gemm(g2, st));
  }
  SimtGemm g{};
  g.a_dtype = g.b_dtype = g.c_dtype = c->dtype;
  g.A = x_disp; g.a_m = d; g.a_k = 1;
  g.B = w1; g.b_n = d; g.b_k = 1; g.b_g = int64_t(f) * d;
  g.C = h; g.c_m = f; g.c_n = 1;
  g.N = f; g.K = d; g.mode = 1; g.offsets = offsets; g.G = E; g.max_rows = R;
  g.bias = b1; g.bias_g = f; g.act = c->act; g.pre = h_pre;
  MOE_CUDA(launch_simt_gemm(g, st));
  SimtGemm g2{};
  g2.a_dtype = g2.b_dtype = g2.c_dtype = c->dtype;
  g2.A = h; g2.a_m = f; g2.a_k = 1;
  g2.B = w2; g2.b_n = f; g2.b_k = 1; g2.b_g = int64_t(d) * f;
  g2.C = out; g2.c_m = d; g2.c_n = 1;
  g2.N = d; g2.K = f; g2.mode = 1; g2.offsets = offsets; g2.G = E; g2.max_rows = R;
  g2.bias = b2; g2.bias_g = d; g2.act = -1;
  return cuda_status(launch_simt_gemm(g2, st));
}

// The expert FFN with the dispatch fused into its first GEMM: row r of the
// grouped operand is token row_src[r] / k of x (bf16 layers only).
moe_status expert_ffn_gather(const moe_config *c, const void *x, const int32_t *row_src,
                             const int32_t *offsets, const void *w1, const void *b1,
                             const void *w2, const void *b2, void *h_pre, void *h, void *out,
                             cudaStream_t st) {
  if (c->dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
  const int64_t R = max_rows_of(c);
  const int d = c->hidden_size, f = c->ffn_size, E = c->num_experts;
  if (R == 0) return MOE_OK;
  TcGemm g1{};
  g1.A = x; g1.rows_alloc = c->num_tokens; g1.B = w1; g1.b_kmajor = true; g1.C = h;
  g1.N = f; g1.K = d; g1.G = E; g1.offsets = offsets; g1.bias = b1; g1.act = c->act;
  g1.pre = h_pre; g1.grad_src = nullptr; g1.dact = 0; g1.err = device_error_ptr();
  g1.row_src = row_src; g1.k_choices = c->k;
  const cudaError_t e = launch_tc_gemm(g1, st);
  if (e == cudaErrorNotSupported) return MOE_ERR_UNSUPPORTED;
  MOE_CUDA(e);
  TcGemm g2{};
  g2.A = h; g2.rows_alloc = R; g2.B = w2; g2.b_kmajor = true; g2.C = out;
  g2.N = d; g2.K = f; g2.G = E; g2.offsets = offsets; g2.bias = b2; g2.act = -1;
  g2.err = device_error_ptr();
  return cuda_status(launch_tc_gemm(g2, st));
}

// Dispatch then the expert FFN, or -- when the caller passes no x_disp --
// the FFN with the dispatch fused into its first GEMM.
moe_status dispatch_and_ffn(const moe_config *c, const void *x, const moe_buffers *buf,
                            const void *w1, const void *b1, const void *w2, const void *b2,
                            cudaStream_t st) {
  if (!buf->x_disp)
    return expert_ffn_gather(c, x, buf->row_src, buf->expert_offsets, w1, b1, w2, b2, buf->h_pre,
                             buf->h, buf->out_disp, st);
  MOE_CUDA(launch_dispatch(x, c->dtype, c->num_tokens, c->hidden_size, c->k, buf->topk_idx,
                           buf->slot, buf->expert_offsets, buf->x_disp, st));
  return expert_ffn(c, buf->x_disp, buf->expert_offsets, w1, b1, w2, b2, buf->h_pre, buf->h,
                    buf->out_disp, st);
}

// The residual expert of PR-MoE on every token: h = act(x rw1^T + rb1),
// out = h rw2^T + rb2 -- the grouped GEMM with one group of all S rows.
moe_status dense_mlp(const moe_config *c, const void *x, const void *rw1, const void *rb1,
                     const void *rw2, const void *rb2, void *h, void *out, cudaStream_t st) {
  const int64_t S = c->num_tokens;
  const int d = c->hidden_size, f = c->ffn_size;
  if (S == 0) return MOE_OK;
  if (c->dtype == MOE_BF16) {
    TcGemm g1{};
    g1.A = x; g1.rows_alloc = S; g1.B = rw1; g1.b_kmajor = true; g1.C = h;
    g1.N = f; g1.K = d; g1.G = 1; g1.offsets = nullptr; g1.bias = rb1; g1.act = c->act;
    g1.pre = nullptr; g1.grad_src = nullptr; g1.dact = 0; g1.err = device_error_ptr();
    MOE_CUDA(launch_tc_gemm(g1, st));
    TcGemm g2 = g1;
    g2.A = h; g2.B = rw2; g2.C = out; g2.N = d; g2.K = f; g2.bias = rb2; g2.act = -1;
    return cuda_status(launch_tc_gemm(g2, st));
  }
  SimtGemm g{};
  g.a_dtype = g.b_dtype = g.c_dtype = c->dtype;
  g.A = x; g.a_m = d; g.a_k = 1;
  g.B = rw1; g.b_n = d; g.b_k = 1;
  g.C = h; g.c_m = f; g.c_n = 1;
  g.M = S; g.N = f; g.K = d; g.mode = 0; g.bias = rb1; g.act = c->act;
  MOE_CUDA(launch_simt_gemm(g, st));
  SimtGemm g2 = g;
  g2.A = h; g2.a_m = f;
  g2.B = rw2; g2.b_n = f;
  g2.C = out; g2.c_m = d;
  g2.N = d; g2.K = f; g2.bias = rb2; g2.act = -1;
  return cuda_status(launch_simt_gemm(g2, st));
}

}  // namespace

int num_sms() {
  static PerDevice<int> cached;
  int n = 0;
  if (cached.get(&n, [](int &v) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess && v <= 0) e = cudaErrorInvalidValue;
        return e;
      }) != cudaSuccess)
    return 148;
  return n;
}

}  // namespace moe

using namespace moe;

extern "C" {

const char *moe_status_string(moe_status st) {
  switch (st) {
    case MOE_OK: return "MOE_OK";
    case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
    case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
    case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
    case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
    case MOE_ERR_DEVICE: return "MOE_ERR_DEVICE";
  }
  return "MOE_ERR_UNKNOWN";
}

moe_status moe_capacity(const moe_config *cfg, int64_t *cap) {
  MOE_TRY(check_config(cfg));
  if (!cap) return MOE_ERR_INVALID_ARG;
  *cap = capacity_of(cfg);
  return MOE_OK;
}

moe_status moe_max_rows(const moe_config *cfg, int64_t *rows) {
  MOE_TRY(check_config(cfg));
  if (!rows) return MOE_ERR_INVALID_ARG;
  *rows = max_rows_of(cfg);
  return MOE_OK;
}

moe_status moe_workspace_size(const moe_config *cfg, int for_backward, size_t *bytes) {
  MOE_TRY(check_config(cfg));
  if (!bytes) return MOE_ERR_INVALID_ARG;
  *bytes = for_backward ? bwd_ws_carve(cfg, nullptr, nullptr) : fwd_ws_bytes(cfg);
  return MOE_OK;
}

moe_status moe_gate_noise(const moe_config *cfg, float *uniform, float *gumbel,
                          int32_t *position, moe_stream_t stream) {
  MOE_TRY(check_config(cfg));
  if (!ok_opt(uniform) || !ok_opt(gumbel) || !ok_opt(position)) return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_gate_noise(cfg->num_tokens, cfg->num_experts, noise_of(cfg), uniform,
                                       gumbel, position, stream));
}

moe_status moe_route_from_logits(const moe_config *cfg, const float *logits, float *probs,
                                 int32_t *topk_idx, float *topk_w, int32_t *slot,
                                 int32_t *routed_cnt, int32_t *kept_cnt, int32_t *expert_offsets,
                                 int32_t *row_src, float *l_aux, void *workspace,
                                 size_t workspace_bytes, moe_stream_t stream) {
  MOE_TRY(check_config(cfg));
  if (!ok_ptr(logits) || !ok_opt(probs) || !ok_ptr(topk_idx) || !ok_ptr(topk_w) ||
      !ok_ptr(slot) || !ok_ptr(routed_cnt) || !ok_ptr(kept_cnt) || !ok_ptr(expert_offsets) ||
      !ok_ptr(row_src) || !ok_ptr(l_aux) || !ok_ptr(workspace))
    return MOE_ERR_INVALID_ARG;
  if (workspace_bytes < fwd_ws_bytes(cfg)) return MOE_ERR_WORKSPACE;
  return route(cfg, logits, probs, topk_idx, topk_w, slot, routed_cnt, kept_cnt, expert_offsets,
               row_src, l_aux, workspace, stream);
}

moe_status moe_gate_topk(const moe_config *cfg, const void *x, const void *w_gate,
                         const float *logit_bias, float *logits, float *probs, int32_t *topk_idx,
                         float *topk_w, int32_t *slot, int32_t *routed_cnt, int32_t *kept_cnt,
                         int32_t *expert_offsets, int32_t *row_src, float *l_aux, void *workspace,
                         size_t workspace_bytes, moe_stream_t stream) {
  MOE_TRY(check_config(cfg));
  if (!ok_ptr(x) || !ok_ptr(w_gate) || !ok_opt(logit_bias) || !ok_opt(logits) ||
      !ok_opt(probs) || !ok_ptr(topk_idx) || !ok_ptr(topk_w) || !ok_ptr(slot) ||
      !ok_ptr(routed_cnt) || !ok_ptr(kept_cnt) || !ok_ptr(expert_offsets) || !ok_ptr(row_src) ||
      !ok_ptr(l_aux) || !ok_ptr(workspace))
    return MOE_ERR_INVALID_ARG;
  if (workspace_bytes < fwd_ws_bytes(cfg)) return MOE_ERR_WORKSPACE;
  const RouteNoise noise = noise_of(cfg);
  if (noise.any()) {
    // randomised gate: (jitter the router input,) the router GEMM writes
    // the logits, then the routing kernels draw the noise / take the
    // random queue order
    const void *xr = x;
    if (noise.policy == MOE_NOISE_JITTER) {
      void *xj = fwd_ws_jitter(cfg, workspace);
      MOE_CUDA(launch_jitter(x, cfg->dtype, cfg->num_tokens, cfg->hidden_size, noise, xj,
                             stream));
      xr = xj;
    }
    float *lg = logits ? logits : fwd_ws_logits(cfg, workspace);
    if (cfg->dtype == MOE_BF16) {
      // the tensor-core gate kernel for the logits; its routing outputs are
      // rewritten by the routing kernels below
      RouteArgs a{};
      a.S = cfg->num_tokens; a.E = cfg->num_experts; a.k = cfg->k;
      route_carve_workspace(a, workspace);
      GateTcArgs g{};
      g.x = xr; g.w_gate = w_gate; g.S = cfg->num_tokens; g.d = cfg->hidden_size;
      g.E = cfg->num_experts; g.k = cfg->k; g.logit_bias = logit_bias; g.logits = lg;
      g.bias_ld = cfg->logit_bias_per_token ? cfg->num_experts : 0;
      g.inv_temp = inv_temperature(cfg);
      g.probs = nullptr; g.idx = topk_idx; g.w = topk_w; g.rank = slot; g.hist = a.hist;
      g.psum = a.psum; g.err = device_error_ptr();
      MOE_CUDA(launch_gate_tc(g, stream));
    } else {
      MOE_TRY(gate_gemm(cfg, xr, w_gate, logit_bias, lg, stream));
    }
    return route(cfg, lg, probs, topk_idx, topk_w, slot, routed_cnt, kept_cnt, expert_offsets,
                 row_src, l_aux, workspace, stream);
  }
  if (cfg->dtype == MOE_BF16) {
    // one launch: tensor-core gate, routing and slot assignment
    GateRouteArgs ga{};
    ga.x = x; ga.w_gate = w_gate; ga.S = cfg->num_tokens; ga.d = cfg->hidden_size;
    ga.E = cfg->num_experts; ga.k = cfg->k; ga.cap = capacity_of(cfg);
    ga.rows_alloc = max_rows_of(cfg);
    ga.logit_bias = logit_bias; ga.bias_ld = cfg->logit_bias_per_token ? cfg->num_experts : 0;
    ga.inv_temp = inv_temperature(cfg); ga.aux_type = cfg->aux_loss_type;
    ga.logits = logits; ga.probs = probs; ga.idx = topk_idx; ga.w = topk_w; ga.slot = slot;
    ga.routed = routed_cnt; ga.kept = kept_cnt; ga.offsets = expert_offsets; ga.row_src = row_src;
    ga.l_aux = l_aux; ga.ws = workspace; ga.ws_bytes = workspace_bytes; ga.err = device_error_ptr();
    const cudaError_t ge = launch_gate_route(ga, stream);
    if (ge != cudaErrorNotSupported) return cuda_status(ge);
    // larger batches: fused tensor-core gate, then the shared scan / assignment
    RouteArgs a{};
    a.S = cfg->num_tokens; a.E = cfg->num_experts; a.k = cfg->k; a.cap = capacity_of(cfg);
    a.inv_temp = inv_temperature(cfg);
    a.aux_type = cfg->aux_loss_type;
    a.probs = probs; a.idx = topk_idx; a.w = topk_w; a.slot = slot; a.routed = routed_cnt;
    a.kept = kept_cnt; a.offsets = expert_offsets; a.row_src = row_src; a.l_aux = l_aux;
    route_carve_workspace(a, workspace);
    GateTcArgs g{};
    g.x = x; g.w_gate = w_gate; g.S = cfg->num_tokens; g.d = cfg->hidden_size;
    g.E = cfg->num_experts; g.k = cfg->k; g.logit_bias = logit_bias; g.logits = logits;
    g.bias_ld = cfg->logit_bias_per_token ? cfg->num_experts : 0;
    g.inv_temp = inv_temperature(cfg);
    g.probs = probs; g.idx = topk_idx; g.w = topk_w; g.rank = slot; g.hist = a.hist;
    g.psum = a.psum; g.err = device_error_ptr();
    MOE_CUDA(launch_gate_tc(g, stream));
    return cuda_status(launch_route_finish(a, stream));
  }
  float *lg = logits ? logits : fwd_ws_logits(cfg, workspace);
  MOE_TRY(gate_gemm(cfg, x, w_gate, logit_bias, lg, stream));
  return route(cfg, lg, probs, topk_idx, topk_w, slot, routed_cnt, kept_cnt, expert_offsets,
               row_src, l_aux, workspace, stream);
}

moe_status moe_dispatch(const moe_config *cfg, const void *x, const int32_t *topk_idx,
                        const int32_t *slot, const int32_t *expert_offsets, void *x_disp,
                        moe_stream_t stream) {
  MOE_TRY(check_config(cfg));
  if (!ok_ptr(x) || !ok_ptr(topk_idx) || !ok_ptr(slot) || !ok_ptr(expert_offsets) ||
      !ok_ptr(x_disp))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_dispatch(x, cfg->dtype, cfg->num_tokens, cfg->hidden_size, cfg->k,
                                     topk_idx, slot, expert_offsets, x_disp, stream));
}

moe_status moe_expert_ffn(const moe_config *cfg, const void *x_disp,
                          const int32_t *expert_offsets, const void *w1, const void *b1,
                          const void *w2, const void *b2, void *h_pre, void *h, void *out_disp,
                          moe_stream_t stream) {
  MOE_TRY(check_config(cfg));
  if (!ok_ptr(x_disp) || !ok_ptr(expert_offsets) || !ok_ptr(w1) || !ok_ptr(b1) || !ok_ptr(w2) ||
      !ok_ptr(b2) || !ok_opt(h_pre) || !ok_ptr(h) || !ok_ptr(out_disp))
    return MOE_ERR_INVALID_ARG;
  return expert_ffn(cfg, x_disp, expert_offsets, w1, b1, w2, b2, h_pre, h, out_disp, stream);
}

moe_status moe_expert_ffn_gather(const moe_config *cfg, const void *x, const int32_t *row_src,
                                 const int32_t *expert_offsets, const void *w1, const void *b1,
                                 const void *w2, const void *b2, void *h_pre, void *h,
                                 void *out_disp, moe_stream_t stream) {
  MOE_TRY(check_config(cfg));
  if (!ok_ptr(x) || !ok_ptr(row_src) || !ok_ptr(expert_offsets) || !ok_ptr(w1) || !ok_ptr(b1) ||
      !ok_ptr(w2) || !ok_ptr(b2) || !ok_opt(h_pre) || !ok_ptr(h) || !ok_ptr(out_disp))
    return MOE_ERR_INVALID_ARG;
  return expert_ffn_gather(cfg, x, row_src, expert_offsets, w1, b1, w2, b2, h_pre, h, out_disp,
                           stream);
}

moe_status moe_combine(const moe_config *cfg, const void *out_disp, const int32_t *topk_idx,
                       const int32_t *slot, const int32_t *expert_offsets, const float *topk_w,
                       void *y, moe_stream_t stream) {
  MOE_TRY(check_config(cfg));
  if (!ok_ptr(out_disp) || !ok_ptr(topk_idx) || !ok_ptr(slot) || !ok_ptr(expert_offsets) ||
      !ok_ptr(topk_w) || !ok_ptr(y))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_combine(out_disp, cfg->dtype, cfg->num_tokens, cfg->hidden_size,
                                    cfg->k, topk_idx, slot, expert_offsets, topk_w, y, stream));
}

moe_status moe_forward(const moe_config *cfg, const void *x, const void *w_gate,
                       const float *logit_bias, const void *w1, const void *b1, const void *w2,
                       const void *b2, void *y, const moe_buffers *buf, void *workspace,
                       size_t workspace_bytes, moe_stream_t stream) {
  MOE_TRY(check_config(cfg));
  if (!buf || !ok_ptr(y) || !ok_opt(buf->x_disp) || !ok_ptr(buf->h) || !ok_ptr(buf->out_disp) ||
      !ok_opt(buf->h_pre) || !ok_ptr(w1) || !ok_ptr(b1) || !ok_ptr(w2) || !ok_ptr(b2))
    return MOE_ERR_INVALID_ARG;
  if (!buf->x_disp && cfg->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  MOE_TRY(moe_gate_topk(cfg, x, w_gate, logit_bias, buf->logits, buf->probs, buf->topk_idx,
                        buf->topk_w, buf->slot, buf->routed_cnt, buf->kept_cnt,
                        buf->expert_offsets, buf->row_src, buf->l_aux, workspace, workspace_bytes,
                        stream));
  MOE_TRY(dispatch_and_ffn(cfg, x, buf, w1, b1, w2, b2, stream));
  return cuda_status(launch_combine(buf->out_disp, cfg->dtype, cfg->num_tokens, cfg->hidden_size,
                                    cfg->k, buf->topk_idx, buf->slot, buf->expert_offsets,
                                    buf->topk_w, y, stream));
}

moe_status moe_forward_residual(const moe_config *cfg, const void *x, const void *w_gate,
                                const float *logit_bias, const void *w1, const void *b1,
                                const void *w2, const void *b2, const void *rw1, const void *rb1,
                                const void *rw2, const void *rb2, const void *mix_w,
                                const void *mix_b, float *mix, void *y, const moe_buffers *buf,
                                void *res_h, void *res_out, void *workspace,
                                size_t workspace_bytes, moe_stream_t stream) {
  MOE_TRY(check_config(cfg));
  if (!buf || !ok_ptr(y) || !ok_opt(buf->x_disp) || !ok_ptr(buf->h) || !ok_ptr(buf->out_disp) ||
      !ok_opt(buf->h_pre) || !ok_ptr(w1) || !ok_ptr(b1) || !ok_ptr(w2) || !ok_ptr(b2) ||
      !ok_ptr(rw1) || !ok_ptr(rb1) || !ok_ptr(rw2) || !ok_ptr(rb2) || !ok_ptr(res_h) ||
      !ok_ptr(res_out) || !ok_opt(mix_w))
    return MOE_ERR_INVALID_ARG;
  if (!buf->x_disp && cfg->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  // the learned mix takes all three of its arguments, the sum none of them
  if (mix_w ? (!ok_ptr(mix_b) || !ok_ptr(mix)) : (mix_b != nullptr || mix != nullptr))
    return MOE_ERR_INVALID_ARG;
  if (mix_w)
    MOE_CUDA(launch_residual_mix(x, cfg->dtype, cfg->num_tokens, cfg->hidden_size, mix_w, mix_b,
                                 mix, stream));
  MOE_TRY(moe_gate_topk(cfg, x, w_gate, logit_bias, buf->logits, buf->probs, buf->topk_idx,
                        buf->topk_w, buf->slot, buf->routed_cnt, buf->kept_cnt,
                        buf->expert_offsets, buf->row_src, buf->l_aux, workspace, workspace_bytes,
                        stream));
  MOE_TRY(dispatch_and_ffn(cfg, x, buf, w1, b1, w2, b2, stream));
  MOE_TRY(dense_mlp(cfg, x, rw1, rb1, rw2, rb2, res_h, res_out, stream));
  return cuda_status(launch_combine(buf->out_disp, cfg->dtype, cfg->num_tokens, cfg->hidden_size,
                                    cfg->k, buf->topk_idx, buf->slot, buf->expert_offsets,
                                    buf->topk_w, y, stream, res_out, mix));
}

moe_status moe_backward(const moe_config *cfg, const void *x, const void *w_gate, const void *w1,
                        const void *w2, const moe_buffers *sv, const void *dy, void *dx,
                        void *dw_gate, void *dw1, void *db1, void *dw2, void *db2,
                        void *workspace, size_t workspace_bytes, moe_stream_t stream) {
  MOE_TRY(check_config(cfg));
  if (!sv || !ok_ptr(x) || !ok_ptr(w_gate) || !ok_ptr(w1) || !ok_ptr(w2) || !ok_ptr(dy) ||
      !ok_ptr(dx) || !ok_ptr(dw_gate) || !ok_ptr(dw1) || !ok_ptr(db1) || !ok_ptr(dw2) ||
      !ok_ptr(db2) || !ok_ptr(sv->probs) || !ok_ptr(sv->topk_idx) || !ok_ptr(sv->topk_w) ||
      !ok_ptr(sv->slot) || !ok_ptr(sv->expert_offsets) || !ok_ptr(sv->x_disp) ||
      !ok_ptr(sv->h_pre) || !ok_ptr(sv->h) || !ok_ptr(sv->out_disp) || !ok_ptr(workspace))
    return MOE_ERR_INVALID_ARG;
  BwdWs w;
  if (workspace_bytes < bwd_ws_carve(cfg, workspace, &w)) return MOE_ERR_WORKSPACE;
  const int64_t S = cfg->num_tokens, R = max_rows_of(cfg);
  const int d = cfg->hidden_size, f = cfg->ffn_size, E = cfg->num_experts, k = cfg->k;
  const int dt = cfg->dtype;
  cudaStream_t st = stream;

  // 1. dO = w * dY per kept row; dw = <dY, out>
  MOE_CUDA(launch_combine_bwd(dy, sv->out_disp, dt, S, d, k, sv->topk_idx, sv->slot,
                              sv->expert_offsets, sv->topk_w, w.d_out, w.dw, st, w.rows));
  // 2. dW2_e = dO_e^T h_e ; db2 = column sums of dO (in the same kernel
  //    when the CTA-pair weight-gradient GEMM runs)
  bool db2_done = false;
  if (dt == MOE_BF16) {
    TcWgrad g{};
    g.A = w.d_out; g.B = sv->h; g.rows_alloc = R > 0 ? R : 1; g.C = dw2;
    g.M = d; g.N = f; g.G = E; g.offsets = sv->expert_offsets; g.err = device_error_ptr();
    // the bias gradient by a column-sum kernel: in the GEMM it would send
    // the first-N tiles' stages through the relay warps
    g.colsum = nullptr;
    g.group_maps = w.maps;
    cudaError_t e = launch_tc_wgrad(g, st);
    db2_done = e == cudaSuccess && g.colsum != nullptr;
    if (e == cudaErrorNotSupported) {
      g.colsum = nullptr;
      e = launch_tc_wgrad(g, st);
    }
    MOE_CUDA(e);
  } else {
    SimtGemm g{};
    g.a_dtype = g.b_dtype = g.c_dtype = dt;
    g.A = w.d_out; g.a_m = 1; g.a_k = d;
    g.B = sv->h; g.b_n = 1; g.b_k = f;
    g.C = dw2; g.c_m = f; g.c_n = 1; g.c_g = int64_t(d) * f;
    g.M = d; g.N = f; g.K = 0; g.mode = 2; g.offsets = sv->expert_offsets; g.G = E;
    g.act = -1;
    MOE_CUDA(launch_simt_gemm(g, st));
  }
  if (!db2_done) MOE_CUDA(launch_group_colsum(w.d_out, dt, d, E, sv->expert_offsets, db2, st));
  // 3. dh_pre = (dO W2_e) * act'(h_pre)
  if (R > 0) {
    if (dt == MOE_BF16) {
      TcGemm g{};
      g.A = w.d_out; g.rows_alloc = R; g.B = w2; g.b_kmajor = false; g.C = w.dh_pre;
      g.N = f; g.K = d; g.G = E; g.offsets = sv->expert_offsets; g.bias = nullptr; g.act = -1;
      g.pre = nullptr; g.grad_src = sv->h_pre; g.dact = cfg->act; g.err = device_error_ptr();
      g.col_part = w.colpart;  // db1's partial sums, from the values it stores
      MOE_CUDA(launch_tc_gemm(g, st));
    } else {
      SimtGemm g{};
      g.a_dtype = g.b_dtype = g.c_dtype = dt;
      g.A = w.d_out; g.a_m = d; g.a_k = 1;
      g.B = w2; g.b_n = 1; g.b_k = f; g.b_g = int64_t(d) * f;
      g.C = w.dh_pre; g.c_m = f; g.c_n = 1;
      g.N = f; g.K = d; g.mode = 1; g.offsets = sv->expert_offsets; g.G = E; g.max_rows = R;
      g.act = -1; g.grad_src = sv->h_pre; g.dact = cfg->act;
      MOE_CUDA(launch_simt_gemm(g, st));
    }
  }
  // 4. dW1_e = dh_pre_e^T x_disp_e ; db1 = column sums of dh_pre (bf16: the
  //    data-gradient epilogue's partial sums, added here in a fixed order)
  bool db1_done = false;
  if (dt == MOE_BF16) {
    MOE_CUDA(launch_bias_grad_reduce(w.colpart, sv->expert_offsets, E, f, db1, st));
    db1_done = true;
  }
  if (dt == MOE_BF16) {
    TcWgrad g{};
    g.A = w.dh_pre; g.B = sv->x_disp; g.rows_alloc = R > 0 ? R : 1; g.C = dw1;
    g.M = f; g.N = d; g.G = E; g.offsets = sv->expert_offsets; g.err = device_error_ptr();
    g.colsum = nullptr;
    // its own maps: the dW2 launch may still be reading the first half
    g.group_maps = w.maps ? static_cast<char *>(w.maps) + 2 * size_t(E) * kTensorMapBytes
                          : nullptr;
    cudaError_t e = launch_tc_wgrad(g, st);
    db1_done = db1_done || (e == cudaSuccess && g.colsum != nullptr);
    if (e == cudaErrorNotSupported) {
      g.colsum = nullptr;
      e = launch_tc_wgrad(g, st);
    }
    MOE_CUDA(e);
  } else {
    SimtGemm g{};
    g.a_dtype = g.b_dtype = g.c_dtype = dt;
    g.A = w.dh_pre; g.a_m = 1; g.a_k = f;
    g.B = sv->x_disp; g.b_n = 1; g.b_k = d;
    g.C = dw1; g.c_m = d; g.c_n = 1; g.c_g = int64_t(f) * d;
    g.M = f; g.N = d; g.K = 0; g.mode = 2; g.offsets = sv->expert_offsets; g.G = E;
    g.act = -1;
    MOE_CUDA(launch_simt_gemm(g, st));
  }
  if (!db1_done) MOE_CUDA(launch_group_colsum(w.dh_pre, dt, f, E, sv->expert_offsets, db1, st));
  // 5. dx_disp = dh_pre W1_e
  if (R > 0) {
    if (dt == MOE_BF16) {
      TcGemm g{};
      g.A = w.dh_pre; g.rows_alloc = R; g.B = w1; g.b_kmajor = false; g.C = w.dx_disp;
      g.N = d; g.K = f; g.G = E; g.offsets = sv->expert_offsets; g.bias = nullptr; g.act = -1;
      g.pre = nullptr; g.grad_src = nullptr; g.dact = 0; g.err = device_error_ptr();
      MOE_CUDA(launch_tc_gemm(g, st));
    } else {
      SimtGemm g{};
      g.a_dtype = g.b_dtype = g.c_dtype = dt;
      g.A = w.dh_pre; g.a_m = f; g.a_k = 1;
      g.B = w1; g.b_n = 1; g.b_k = d; g.b_g = int64_t(f) * d;
      g.C = w.dx_disp; g.c_m = d; g.c_n = 1;
      g.N = d; g.K = f; g.mode = 1; g.offsets = sv->expert_offsets; g.G = E; g.max_rows = R;
      g.act = -1;
      MOE_CUDA(launch_simt_gemm(g, st));
    }
  }
  // 6. router: dlogits, dW_g = dlogits^T x (the router saw x * f under jitter)
  MOE_CUDA(launch_aux_coef(sv->topk_idx, sv->probs, S, k, E, cfg->aux_loss_type, w.aux_coef,
                           st));
  const bool tc = dt == MOE_BF16;
  void *dl2 = tc ? static_cast<void *>(w.dlogits) : nullptr;
  MOE_CUDA(launch_gate_bwd(sv->probs, sv->topk_idx, w.dw, w.aux_coef, S, E, k,
                           cfg->aux_loss_weight, inv_temperature(cfg), tc ? nullptr : w.dlogits,
                           dl2, router_pad(E), st));
  const RouteNoise noise = noise_of(cfg);
  const RouteNoise *jit = noise.policy == MOE_NOISE_JITTER ? &noise : nullptr;
  const void *xr = x;
  if (jit) {
    MOE_CUDA(launch_jitter(x, dt, S, d, noise, w.xj, st));
    xr = w.xj;
  }
  if (tc) {
    // on the tensor cores: dW_g from x^T [hi | lo]; dX from [hi | lo] [W_g; W_g]
    // with the experts' rows added in the GEMM's epilogue
    MOE_CUDA(launch_gate_wgrad_tc(xr, dl2, S, d, E, w.gate_partial, dw_gate,
                                  device_error_ptr(), st));
    return cuda_status(launch_dx_router_tc(dl2, w_gate, w.dx_disp, S, d, E, k, w.rows,
                                           static_cast<float *>(w.d_out), dx, jit,
                                           device_error_ptr(), st));
  }
  MOE_CUDA(launch_gate_wgrad(w.dlogits, xr, dt, S, d, E, w.gate_partial, dw_gate, st));
  // 7. dX = sum_j dx_disp[row] + (dlogits W_g) (* f under jitter)
  return cuda_status(launch_dx_combine(w.dx_disp, w.dlogits, w_gate, dt, S, d, E, k,
                                       sv->topk_idx, sv->slot, sv->expert_offsets, dx, st, jit));
}

moe_status moe_debug_set_wait_limit(uint64_t ns) {
  return cuda_status(set_gate_wait_limit(ns));
}

moe_status moe_get_device_error(uint32_t *code) {
  if (!code) return MOE_ERR_INVALID_ARG;
  unsigned int *p = device_error_ptr();
  if (!p) return MOE_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpy(&v, p, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
  const unsigned int zero = 0;
  if (cudaMemcpy(p, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess)
    return MOE_ERR_CUDA;
  *code = v;
  return v ? MOE_ERR_DEVICE : MOE_OK;
}

}  // extern "C"
