// Router-side backward kernels: the gate weight gradient and the input
// gradient that gathers the experts' dX rows.
//
// DeepSeek-MoE page (lnwmold.com/news/1162317) §3.1 TopKRouter: the
// gradient flows back only through the selected experts' weights; here
// dlogits (computed by gate_bwd_kernel) already holds it, so
//   dW_g = dlogits^T x                 (E x d, reduction over the S tokens)
//   dX[s] = sum_j dx_disp[row(s,j)] + dlogits[s] . W_g
// dW_g is split over token chunks (fp32 partial sums) and the partials are
// added in a fixed order, so the result is the same on every run.
#include "common.cuh"
#include "kernels.h"
#include "rng.cuh"

namespace moe {
namespace {

// ---------------------------------------------------------------- dW_g
// partial[split][e][c] = sum over the split's tokens s of dl[s,e] * x[s,c].
// CTA tile: 32 experts x 128 columns; tokens staged 64 at a time in shared
// memory (both operands, loaded cooperatively and coalesced); each of the
// 128 threads accumulates an 8 (experts) x 4 (columns) register tile.
constexpr int kGwE = 32, kGwC = 128, kGwK = 64, kGwThreads = 128;

template <typename T>
__global__ void __launch_bounds__(kGwThreads)
gate_wgrad_partial_kernel(const float *__restrict__ dl, const T *__restrict__ x, int64_t S,
                          int d, int E, int64_t tok_per_split, float *__restrict__ partial) {
  griddep_begin();
  __shared__ __align__(16) float s_dl[kGwK][kGwE];
  __shared__ __align__(16) float s_x[kGwK][kGwC];
  const int tid = threadIdx.x, ty = tid >> 5, tx = tid & 31;
  const int c0 = blockIdx.x * kGwC;
  const int e0 = blockIdx.z * kGwE;
  const int64_t s0 = int64_t(blockIdx.y) * tok_per_split;
  const int64_t s1 = min(S, s0 + tok_per_split);
  constexpr int V = 16 / sizeof(T);
  float acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
  for (int64_t sb = s0; sb < s1; sb += kGwK) {
    const int nt = int(min((int64_t)kGwK, s1 - sb));
    __syncthreads();
    for (int i = tid; i < kGwK * kGwE; i += kGwThreads) {
      const int t = i / kGwE, e = i % kGwE;
      s_dl[t][e] = (t < nt && e0 + e < E) ? dl[(sb + t) * E + e0 + e] : 0.0f;
    }
    for (int i = tid; i < kGwK * (kGwC / V); i += kGwThreads) {
      const int t = i / (kGwC / V), cv = (i % (kGwC / V)) * V;
      float v[V];
      if (t < nt && c0 + cv < d) {
        Vec<T>::to_f32(*reinterpret_cast<const uint4 *>(x + (sb + t) * d + c0 + cv), v);
      } else {
#pragma unroll
        for (int j = 0; j < V; ++j) v[j] = 0.0f;
      }
#pragma unroll
      for (int j = 0; j < V; ++j) s_x[t][cv + j] = v[j];
    }
    __syncthreads();
#pragma unroll 4
    for (int t = 0; t < kGwK; ++t) {
      const float4 a0 = *reinterpret_cast<const float4 *>(&s_dl[t][ty * 8]);
      const float4 a1 = *reinterpret_cast<const float4 *>(&s_dl[t][ty * 8 + 4]);
      const float4 b = *reinterpret_cast<const float4 *>(&s_x[t][tx * 4]);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float bb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], bb[j], acc[i][j]);
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = e0 + ty * 8 + i;
    if (e >= E) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int c = c0 + tx * 4 + j;
      if (c < d) partial[(int64_t(blockIdx.y) * E + e) * d + c] = acc[i][j];
    }
  }
}

// dW_g[e,c] = sum over splits, in split order
__global__ void gate_wgrad_reduce_kernel(const float *__restrict__ partial, int nsplit, int E,
                                         int d, int dtype, void *__restrict__ dw_gate) {
  griddep_begin();
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= int64_t(E) * d) return;
  float acc = 0.0f;
  for (int sp = 0; sp < nsplit; ++sp) acc += partial[int64_t(sp) * E * d + i];
  store_elem(dw_gate, dtype, i, acc);
}

// ------------------------------------------------------------------ dX
// dx[s, c] = sum_e dl[s,e] * W_g[e,c] + sum_j dx_disp[row(s,j), c].
// CTA tile: 64 tokens x 128 columns; experts staged 32 at a time in shared
// memory; each of the 256 threads accumulates 8 (tokens) x 4 (columns).
constexpr int kDxT = 64, kDxC = 128, kDxE = 32, kDxThreads = 256;

template <typename T>
__global__ void __launch_bounds__(kDxThreads)
dx_combine_tile_kernel(const T *__restrict__ dx_disp, const float *__restrict__ dlogits,
                       const T *__restrict__ w_gate, int64_t S, int d, int E, int k,
                       const int32_t *__restrict__ idx, const int32_t *__restrict__ slot,
                       const int32_t *__restrict__ offsets, T *__restrict__ dx, int jitter,
                       RouteNoise noise) {
  griddep_begin();
  __shared__ __align__(16) float s_dlT[kDxE][kDxT];
  __shared__ __align__(16) float s_w[kDxE][kDxC];
  __shared__ int64_t s_row[kDxT][2];
  const int tid = threadIdx.x, ty = tid >> 5, tx = tid & 31;
  const int64_t t0 = int64_t(blockIdx.y) * kDxT;
  const int c0 = blockIdx.x * kDxC;
  const int nt = int(min((int64_t)kDxT, S - t0));
  constexpr int V = 16 / sizeof(T);
  if (tid < kDxT * 2) {
    const int t = tid >> 1, j = tid & 1;
    int64_t r = -1;
    if (t < nt && j < k) {
      const int sl = slot[(t0 + t) * k + j];
      if (sl >= 0) r = int64_t(offsets[idx[(t0 + t) * k + j]]) + sl;
    }
    s_row[t][j] = r;
  }
  float acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;
  for (int e0 = 0; e0 < E; e0 += kDxE) {
    __syncthreads();
    for (int i = tid; i < kDxT * kDxE; i += kDxThreads) {
      const int t = i / kDxE, e = i % kDxE;
      s_dlT[e][t] = (t < nt && e0 + e < E) ? dlogits[(t0 + t) * E + e0 + e] : 0.0f;
    }
    for (int i = tid; i < kDxE * (kDxC / V); i += kDxThreads) {
      const int e = i / (kDxC / V), cv = (i % (kDxC / V)) * V;
      float v[V];
      if (e0 + e < E && c0 + cv < d) {
        Vec<T>::to_f32(*reinterpret_cast<const uint4 *>(w_gate + int64_t(e0 + e) * d + c0 + cv),
                       v);
      } else {
#pragma unroll
        for (int j = 0; j < V; ++j) v[j] = 0.0f;
      }
#pragma unroll
      for (int j = 0; j < V; ++j) s_w[e][cv + j] = v[j];
    }
    __syncthreads();
#pragma unroll 4
    for (int e = 0; e < kDxE; ++e) {
      const float4 a0 = *reinterpret_cast<const float4 *>(&s_dlT[e][ty * 8]);
      const float4 a1 = *reinterpret_cast<const float4 *>(&s_dlT[e][ty * 8 + 4]);
      const float4 b = *reinterpret_cast<const float4 *>(&s_w[e][tx * 4]);
      const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float bb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], bb[j], acc[i][j]);
    }
  }
  const int c = c0 + tx * 4;
  if (c >= d) return;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int t = ty * 8 + i;
    if (t >= nt) break;
    float v[4] = {acc[i][0], acc[i][1], acc[i][2], acc[i][3]};
    if (jitter) {
      // the router's input was x * f: its gradient is the router term * f
      const uint4 w4 = rng::block(rng::make_key(noise.seed, noise.offset), rng::kPurposeJitter,
                                  uint32_t(t0 + t), uint32_t(c >> 2));
      const float eps = noise.jitter_eps > 0.0f ? noise.jitter_eps : 0.01f;
#pragma unroll
      for (int q = 0; q < 4; ++q) v[q] *= rng::jitter(rng::uniform(rng::word(w4, q)), eps);
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int64_t r = s_row[t][j];
      if (r < 0) continue;
      const T *src = dx_disp + r * d + c;
#pragma unroll
      for (int q = 0; q < 4; ++q) v[q] += float(src[q]);
    }
    T *dst = dx + (t0 + t) * d + c;
#pragma unroll
    for (int q = 0; q < 4; ++q) dst[q] = T(v[q]);
  }
}

// ------------------------------------------- dW_g from tensor-core partials
// dW_g[e, c] = sum over chunks g of (part[g, c, e] + part[g, c, P + e]): the
// hi and lo halves of each chunk's x^T [hi | lo], added in chunk order.
// CTA: 8 columns c (one per warp) x 32 experts e (one per lane), every
// chunk's loads in flight together; written along c through shared memory.
__global__ void __launch_bounds__(256)
gate_wgrad_tc_reduce_kernel(const float *__restrict__ part, int nchunk, int d, int E, int P,
                            int dtype, void *__restrict__ dw_gate) {
  griddep_begin();
  __shared__ float tile[32][9];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int c = blockIdx.x * 8 + w, e = blockIdx.y * 32 + lane;
  float acc = 0.0f;
  if (c < d && e < E) {
    const float *p = part + int64_t(c) * (2 * P) + e;
    const int64_t step = int64_t(d) * (2 * P);
#pragma unroll 8
    for (int g = 0; g < nchunk; ++g) acc += __ldcs(p + g * step) + __ldcs(p + g * step + P);
  }
  tile[lane][w] = acc;
  __syncthreads();
  // thread t writes expert e0 + t / 8, column c0 + t % 8
  const int eo = blockIdx.y * 32 + (threadIdx.x >> 3), co = blockIdx.x * 8 + (threadIdx.x & 7);
  if (eo < E && co < d)
    store_elem(dw_gate, dtype, int64_t(eo) * d + co, tile[threadIdx.x >> 3][threadIdx.x & 7]);
}

// ------------------------------------------------- dX from the router term
// dX[s] = r[s] * f(s, .) + sum_j dx_disp[rows[s, j]]; one warp per token,
// lanes over 8-feature vectors (16 bytes of bf16, 32 of fp32).
constexpr int kDxrWarps = 8;

__global__ void __launch_bounds__(kDxrWarps * 32)
dx_router_combine_kernel(const float *__restrict__ rterm, const uint4 *__restrict__ dx_disp,
                         const int32_t *__restrict__ rows, int64_t S, int nvec, int k,
                         uint4 *__restrict__ dx, int jitter, RouteNoise noise) {
  griddep_begin();
  const int lane = threadIdx.x & 31;
  const int64_t s = int64_t(blockIdx.x) * kDxrWarps + (threadIdx.x >> 5);
  if (s >= S) return;
  const int r0 = rows[s * k], r1 = k == 2 ? rows[s * k + 1] : -1;
  const float4 *rt = reinterpret_cast<const float4 *>(rterm) + s * nvec * 2;
  const rng::Key key = rng::make_key(noise.seed, noise.offset);
  const float eps = noise.jitter_eps > 0.0f ? noise.jitter_eps : 0.01f;
  for (int c = lane; c < nvec; c += 32) {
    const float4 a = __ldcs(rt + 2 * c), b = __ldcs(rt + 2 * c + 1);
    float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    if (jitter) {
      // the router's input was x * f: its gradient is the router term * f
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint4 w4 = rng::block(key, rng::kPurposeJitter, uint32_t(s), uint32_t(2 * c + h));
#pragma unroll
        for (int q = 0; q < 4; ++q) v[4 * h + q] *= rng::jitter(rng::uniform(rng::word(w4, q)), eps);
      }
    }
    float g[8];
    if (r0 >= 0) {
      Vec<__nv_bfloat16>::to_f32(dx_disp[int64_t(r0) * nvec + c], g);
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] += g[i];
    }
    if (r1 >= 0) {
      Vec<__nv_bfloat16>::to_f32(dx_disp[int64_t(r1) * nvec + c], g);
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] += g[i];
    }
    dx[s * nvec + c] = Vec<__nv_bfloat16>::from_f32(v);
  }
}

}  // namespace

// token chunks of the dW_g product: as many (chunk, 128-column) tiles as
// fit in one wave over the SMs, chunks a multiple of the 64-row K block
static int gate_wgrad_tc_chunk_rows(int64_t S, int d) {
  const int ctiles = (d + 127) / 128;
  int64_t want = num_sms() / ctiles;
  if (want < 1) want = 1;
  const int64_t per = (S + want - 1) / want;
  return int(per < 64 ? 64 : (per + 63) / 64 * 64);
}

int gate_wgrad_tc_chunks(int64_t S, int d) {
  const int64_t rows = gate_wgrad_tc_chunk_rows(S, d);
  const int64_t n = (S + rows - 1) / rows;
  return int(n < 1 ? 1 : n);
}

size_t gate_wgrad_tc_partial_bytes(int64_t S, int E, int d) {
  return size_t(gate_wgrad_tc_chunks(S, d)) * d * 2 * router_pad(E) * 4;
}

cudaError_t launch_gate_wgrad_tc(const void *x, const void *dl2, int64_t S, int d, int E,
                                 float *partial, void *dw_gate, unsigned int *err,
                                 cudaStream_t st) {
  const int P = router_pad(E);
  const dim3 grid(unsigned((d + 7) / 8), unsigned((E + 31) / 32));
  if (S <= 0)  // no tokens: dW_g = 0
    return launch_k(gate_wgrad_tc_reduce_kernel, grid, 256, 0, st,
                    static_cast<const float *>(partial), 0, d, E, P, int(MOE_BF16), dw_gate);
  const int nch = gate_wgrad_tc_chunks(S, d);
  TcWgrad g{};
  g.A = x; g.B = dl2; g.rows_alloc = S;
  g.M = d; g.N = 2 * P; g.G = nch;
  g.offsets = nullptr; g.chunk_rows = gate_wgrad_tc_chunk_rows(S, d);
  g.Cf = partial; g.single = true; g.err = err;
  if (const cudaError_t e = launch_tc_wgrad(g, st); e != cudaSuccess) return e;
  return launch_k(gate_wgrad_tc_reduce_kernel, grid, 256, 0, st,
                  static_cast<const float *>(partial), nch, d, E, P, int(MOE_BF16), dw_gate);
}

cudaError_t launch_dx_router_tc(const void *dl2, const void *w_gate, const void *dx_disp,
                                int64_t S, int d, int E, int k, const int32_t *rows,
                                float *rterm, void *dx, const RouteNoise *jitter,
                                unsigned int *err, cudaStream_t st) {
  if (S <= 0) return cudaSuccess;
  const int P = router_pad(E);
  TcGemm g{};
  g.A = dl2; g.rows_alloc = S; g.B = w_gate; g.b_kmajor = false; g.C = nullptr;
  g.N = d; g.K = 2 * P; g.G = 1; g.offsets = nullptr; g.bias = nullptr; g.act = -1;
  g.pre = nullptr; g.grad_src = nullptr; g.dact = 0; g.err = err;
  g.b_wrap = P; g.b_rows = E; g.c_f32 = rterm;
  if (const cudaError_t e = launch_tc_gemm(g, st); e != cudaSuccess) return e;
  const RouteNoise nz = jitter ? *jitter : RouteNoise{};
  return launch_k(dx_router_combine_kernel, unsigned((S + kDxrWarps - 1) / kDxrWarps),
                  kDxrWarps * 32, 0, st, static_cast<const float *>(rterm),
                  static_cast<const uint4 *>(dx_disp), rows, S, d / 8, k,
                  static_cast<uint4 *>(dx), jitter ? 1 : 0, nz);
}

int64_t gate_wgrad_splits(int64_t S) {
  int64_t n = (S + 255) / 256;
  if (n > 32) n = 32;
  return n < 1 ? 1 : n;
}

size_t gate_wgrad_partial_bytes(int64_t S, int E, int d) {
  return size_t(gate_wgrad_splits(S)) * E * d * 4;
}

cudaError_t launch_gate_wgrad(const float *dlogits, const void *x, int dtype, int64_t S, int d,
                              int E, float *partial, void *dw_gate, cudaStream_t st) {
  const int64_t nsplit = gate_wgrad_splits(S);
  int64_t per = (S + nsplit - 1) / nsplit;
  if (per < 1) per = 1;
  dim3 grid((d + kGwC - 1) / kGwC, unsigned(nsplit), (E + kGwE - 1) / kGwE);
  const cudaError_t e =
      dtype == MOE_F32
          ? launch_k(gate_wgrad_partial_kernel<float>, grid, kGwThreads, 0, st, dlogits,
                     static_cast<const float *>(x), S, d, E, per, partial)
          : launch_k(gate_wgrad_partial_kernel<__nv_bfloat16>, grid, kGwThreads, 0, st, dlogits,
                     static_cast<const __nv_bfloat16 *>(x), S, d, E, per, partial);
  if (e != cudaSuccess) return e;
  const int64_t n = int64_t(E) * d;
  return launch_k(gate_wgrad_reduce_kernel, unsigned((n + 255) / 256), 256, 0, st, partial,
                  int(nsplit), E, d, dtype, dw_gate);
}

cudaError_t launch_dx_combine(const void *dx_disp, const float *dlogits, const void *w_gate,
                              int dtype, int64_t S, int d, int E, int k, const int32_t *idx,
                              const int32_t *slot, const int32_t *offsets, void *dx,
                              cudaStream_t st, const RouteNoise *jitter) {
  if (S == 0) return cudaSuccess;
  const dim3 grid((d + kDxC - 1) / kDxC, unsigned((S + kDxT - 1) / kDxT));
  const RouteNoise nz = jitter ? *jitter : RouteNoise{};
  const int jit = jitter ? 1 : 0;
  if (dtype == MOE_F32)
    return launch_k(dx_combine_tile_kernel<float>, grid, kDxThreads, 0, st,
                    static_cast<const float *>(dx_disp), dlogits, static_cast<const float *>(w_gate),
                    S, d, E, k, idx, slot, offsets, static_cast<float *>(dx), jit, nz);
  return launch_k(dx_combine_tile_kernel<__nv_bfloat16>, grid, kDxThreads, 0, st,
                  static_cast<const __nv_bfloat16 *>(dx_disp), dlogits,
                  static_cast<const __nv_bfloat16 *>(w_gate), S, d, E, k, idx, slot, offsets,
                  static_cast<__nv_bfloat16 *>(dx), jit, nz);
}

}  // namespace moe
