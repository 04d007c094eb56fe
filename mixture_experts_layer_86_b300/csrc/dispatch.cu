// Dispatch, combine and the token-major backward helpers.
//
// Dispatch (MoE explainer, lpnh.cn/news/725941, §3.1 Step 3 "flatten &
// scatter") and combine (§3.1 Step 5 "gather weighted sum"; deepspeed.moe
// overview §3.1 item 4) are HBM-bound row copies: one warp per token, rows
// moved in 16-byte vectors, each x row read once whatever k is, each y row
// written once (a deterministic gather, no atomics).
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int kWarpsPerCta = 8;

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}

__device__ __forceinline__ int64_t row_of(const int32_t *idx, const int32_t *slot,
                                          const int32_t *offsets, int64_t i) {
  const int sl = slot[i];
  return sl < 0 ? -1 : int64_t(offsets[idx[i]]) + sl;
}

// x_disp[row(s,j)] = x[s]
__global__ void __launch_bounds__(kWarpsPerCta * 32)
dispatch_kernel(const uint4 *__restrict__ x, int64_t S, int nvec, int k,
                const int32_t *__restrict__ idx, const int32_t *__restrict__ slot,
                const int32_t *__restrict__ offsets, uint4 *__restrict__ x_disp) {
  griddep_begin();
  const int lane = threadIdx.x & 31;
  const int64_t s = int64_t(blockIdx.x) * kWarpsPerCta + (threadIdx.x >> 5);
  if (s >= S) return;
  const int64_t r0 = row_of(idx, slot, offsets, s * k);
  const int64_t r1 = k == 2 ? row_of(idx, slot, offsets, s * k + 1) : -1;
  if (r0 < 0 && r1 < 0) return;
  const uint4 *src = x + s * nvec;
  uint4 *d0 = r0 >= 0 ? x_disp + r0 * nvec : nullptr;
  uint4 *d1 = r1 >= 0 ? x_disp + r1 * nvec : nullptr;
  for (int c = lane; c < nvec; c += 32) {
    const uint4 v = ld_stream(src + c);
    if (d0) d0[c] = v;
    if (d1) d1[c] = v;
  }
}

// y[s] = res[s] (if res is set) + sum_j w[s,j] * out[row(s,j)]; with the
// per-token mixing weights mix[s] = (c0, c1) set:
// y[s] = c1 * res[s] + c0 * sum_j w[s,j] * out[row(s,j)]
template <typename T>
__global__ void __launch_bounds__(kWarpsPerCta * 32)
combine_kernel(const uint4 *__restrict__ out, int64_t S, int nvec, int k,
               const int32_t *__restrict__ idx, const int32_t *__restrict__ slot,
               const int32_t *__restrict__ offsets, const float *__restrict__ w,
               const uint4 *__restrict__ res, const float2 *__restrict__ mix,
               uint4 *__restrict__ y) {
  griddep_begin();
  using V = Vec<T>;
  const int lane = threadIdx.x & 31;
  const int64_t s = int64_t(blockIdx.x) * kWarpsPerCta + (threadIdx.x >> 5);
  if (s >= S) return;
  const int64_t r0 = row_of(idx, slot, offsets, s * k);
  const int64_t r1 = k == 2 ? row_of(idx, slot, offsets, s * k + 1) : -1;
  const float2 cm = mix ? mix[s] : make_float2(1.0f, 1.0f);
  const float w0 = cm.x * w[s * k];
  const float w1 = k == 2 ? cm.x * w[s * k + 1] : 0.0f;
  for (int c = lane; c < nvec; c += 32) {
    float acc[V::kN], t[V::kN];
    if (res) {
      V::to_f32(ld_stream(res + s * nvec + c), acc);
      if (mix) {
#pragma unroll
        for (int i = 0; i < V::kN; ++i) acc[i] *= cm.y;
      }
    } else {
#pragma unroll
      for (int i = 0; i < V::kN; ++i) acc[i] = 0.0f;
    }
    if (r0 >= 0) {
      V::to_f32(ld_stream(out + r0 * nvec + c), t);
#pragma unroll
      for (int i = 0; i < V::kN; ++i) acc[i] = fmaf(w0, t[i], acc[i]);
    }
    if (r1 >= 0) {
      V::to_f32(ld_stream(out + r1 * nvec + c), t);
#pragma unroll
      for (int i = 0; i < V::kN; ++i) acc[i] = fmaf(w1, t[i], acc[i]);
    }
    y[s * nvec + c] = V::from_f32(acc);
  }
}

// PR-MoE's learned mixing weights: mix[s] = softmax over two of
// (x[s] . cw[j] + cb[j]), j = 0 (the experts) and 1 (the dense MLP); one
// warp per token, x and cw read in 16-byte vectors, fp32 dot products.
template <typename T>
__global__ void __launch_bounds__(kWarpsPerCta * 32)
residual_mix_kernel(const uint4 *__restrict__ x, int64_t S, int nvec,
                    const uint4 *__restrict__ cw, const T *__restrict__ cb,
                    float2 *__restrict__ mix) {
  griddep_begin();
  using V = Vec<T>;
  const int lane = threadIdx.x & 31;
  const int64_t s = int64_t(blockIdx.x) * kWarpsPerCta + (threadIdx.x >> 5);
  if (s >= S) return;
  float z0 = 0.0f, z1 = 0.0f;
  for (int c = lane; c < nvec; c += 32) {
    float xv[V::kN], a[V::kN], b[V::kN];
    V::to_f32(ld_stream(x + s * nvec + c), xv);
    V::to_f32(cw[c], a);
    V::to_f32(cw[nvec + c], b);
#pragma unroll
    for (int i = 0; i < V::kN; ++i) {
      z0 = fmaf(xv[i], a[i], z0);
      z1 = fmaf(xv[i], b[i], z1);
    }
  }
  z0 = warp_sum(z0) + float(cb[0]);
  z1 = warp_sum(z1) + float(cb[1]);
  if (lane == 0) {
    const float m = fmaxf(z0, z1);
    const float e0 = expf(z0 - m), e1 = expf(z1 - m);
    const float inv = 1.0f / (e0 + e1);
    mix[s] = make_float2(e0 * inv, e1 * inv);
  }
}

// dO[row] = w * dY[s]; dw[s,j] = <dY[s], out[row]>
template <typename T>
__global__ void __launch_bounds__(kWarpsPerCta * 32)
combine_bwd_kernel(const uint4 *__restrict__ dy, const uint4 *__restrict__ out,
                   int64_t S, int nvec, int k, const int32_t *__restrict__ idx,
                   const int32_t *__restrict__ slot, const int32_t *__restrict__ offsets,
                   const float *__restrict__ w, uint4 *__restrict__ d_out,
                   float *__restrict__ dw, int32_t *__restrict__ rows) {
  griddep_begin();
  using V = Vec<T>;
  const int lane = threadIdx.x & 31;
  const int64_t s = int64_t(blockIdx.x) * kWarpsPerCta + (threadIdx.x >> 5);
  if (s >= S) return;
  for (int j = 0; j < k; ++j) {
    const int64_t r = row_of(idx, slot, offsets, s * k + j);
    if (rows && lane == 0) rows[s * k + j] = int32_t(r);
    if (r < 0) {
      if (lane == 0) dw[s * k + j] = 0.0f;
      continue;
    }
    const float wj = w[s * k + j];
    float dot = 0.0f;
    for (int c = lane; c < nvec; c += 32) {
      float g[V::kN], o[V::kN];
      V::to_f32(dy[s * nvec + c], g);
      V::to_f32(out[r * nvec + c], o);
#pragma unroll
      for (int i = 0; i < V::kN; ++i) {
        dot = fmaf(g[i], o[i], dot);
        g[i] *= wj;
      }
      d_out[r * nvec + c] = V::from_f32(g);
    }
    dot = warp_sum(dot);
    if (lane == 0) dw[s * k + j] = dot;
  }
}

// bf16 form: a CTA takes 64 columns of one group (a 128-byte segment of
// each row), 8 threads across them (8 columns, 16 bytes each) and 32 row
// groups down the group's rows (every 32nd row); the row groups are then
// added in a fixed order.
constexpr int kColsumCols = 64, kColsumRowGroups = 32;
constexpr int kColsumThreads = (kColsumCols / 8) * kColsumRowGroups;

__global__ void __launch_bounds__(kColsumThreads)
group_colsum_bf16_kernel(const uint4 *__restrict__ M, int nvec,
                         const int32_t *__restrict__ offsets, uint4 *__restrict__ db) {
  griddep_begin();
  __shared__ float part[kColsumRowGroups][kColsumCols + 1];
  __shared__ float tot[kColsumCols];
  const int g = blockIdx.y;
  const int cv = threadIdx.x & 7, rg = threadIdx.x >> 3;
  const int v = blockIdx.x * (kColsumCols / 8) + cv;  // this thread's 16-byte column vector
  const int64_t r0 = offsets[g], r1 = offsets[g + 1];
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  if (v < nvec) {
#pragma unroll 4
    for (int64_t r = r0 + rg; r < r1; r += kColsumRowGroups) {
      float x[8];
      Vec<__nv_bfloat16>::to_f32(__ldcs(M + r * nvec + v), x);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += x[i];
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) part[rg][cv * 8 + i] = acc[i];
  __syncthreads();
  if (threadIdx.x < kColsumCols) {
    float t = 0.0f;
    for (int j = 0; j < kColsumRowGroups; ++j) t += part[j][threadIdx.x];
    tot[threadIdx.x] = t;
  }
  __syncthreads();
  if (threadIdx.x < kColsumCols / 8) {
    const int vo = blockIdx.x * (kColsumCols / 8) + threadIdx.x;
    if (vo < nvec) db[int64_t(g) * nvec + vo] = Vec<__nv_bfloat16>::from_f32(&tot[threadIdx.x * 8]);
  }
}

// db[g, n] = sum over rows of group g of M[r, n]; blockDim (32, 8)
__global__ void group_colsum_kernel(const void *__restrict__ M, int dtype, int N,
                                    const int32_t *__restrict__ offsets,
                                    void *__restrict__ db) {
  griddep_begin();
  __shared__ float part[8][33];
  const int g = blockIdx.y;
  const int n = blockIdx.x * 32 + threadIdx.x;
  const int64_t r0 = offsets[g], r1 = offsets[g + 1];
  float acc = 0.0f;
  if (n < N)
    for (int64_t r = r0 + threadIdx.y; r < r1; r += 8) acc += load_elem(M, dtype, r * N + n);
  part[threadIdx.y][threadIdx.x] = acc;
  __syncthreads();
  if (threadIdx.y == 0 && n < N) {
    float t = 0.0f;
    for (int i = 0; i < 8; ++i) t += part[i][threadIdx.x];
    store_elem(db, dtype, int64_t(g) * N + n, t);
  }
}

// d l_aux / d p[s,e], the same for every token (one CTA):
//   MOE_AUX_LOAD: E * first[e] / S^2   (first[e] = tokens whose first choice is e)
//   MOE_AUX_STD:  (u_e - mean u) / (E * S * std u),  u_e = mean_s p[s,e],
//                 population std; 0 when std u = 0
__global__ void aux_coef_kernel(const int32_t *__restrict__ idx, const float *__restrict__ probs,
                                int64_t S, int k, int E, int aux_type, float *__restrict__ coef) {
  griddep_begin();
  // column sums of p in units of 2^-30: exact integer sums (no FP64; the
  // order of addition does not matter)
  __shared__ long long s_col[kMaxExperts];
  __shared__ long long s_part[1024];
  __shared__ int32_t cnt[kMaxExperts];
  __shared__ float s_std;
  __shared__ long long s_sum;
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    cnt[e] = 0;
    s_col[e] = 0;
  }
  __syncthreads();
  if (aux_type == MOE_AUX_STD) {
    // G token groups per column (consecutive threads on consecutive columns)
    const int G = int(blockDim.x) / E;
    const int e = threadIdx.x % E, grp = threadIdx.x / E;
    if (grp < G) {
      long long acc = 0;
      // p <= 1, so p * 2^30 fits a 32-bit integer
      for (int64_t s = grp; s < S; s += G) acc += __float2int_rn(probs[s * E + e] * kFix30);
      s_part[grp * E + e] = acc;
    }
    __syncthreads();
    for (int c = threadIdx.x; c < E; c += blockDim.x) {
      long long acc = 0;
      for (int g = 0; g < G; ++g) acc += s_part[g * E + c];
      s_col[c] = acc;
    }
  } else {
    for (int64_t s = threadIdx.x; s < S; s += blockDim.x) atomicAdd(&cnt[idx[s * k]], 1);
  }
  __syncthreads();
  if (threadIdx.x < 32 && aux_type == MOE_AUX_STD) {
    // population std of u_e = sum_s p[s,e] / S over the experts
    const int lane = threadIdx.x;
    long long sa = 0;
    for (int e = lane; e < E; e += 32) sa += s_col[e];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sa += __shfl_xor_sync(kFullMask, sa, o);
    float sq = 0.0f;
    if (S > 0)
      for (int e = lane; e < E; e += 32) {
        const float dv = usage_deviation(s_col[e], sa, E, S);
        sq = fmaf(dv, dv, sq);
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(kFullMask, sq, o);
    if (lane == 0) {
      s_std = sqrtf(sq / float(E));
      s_sum = sa;
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    float c;
    if (aux_type == MOE_AUX_STD)
      c = s_std > 0.0f ? usage_deviation(s_col[e], s_sum, E, S) /
                             (float(E) * float(S) * s_std)
                       : 0.0f;
    else
      c = float(E) * float(cnt[e]) / float(S) / float(S);
    coef[e] = c;
  }
}

// One warp per token; lanes over experts.
__global__ void __launch_bounds__(kWarpsPerCta * 32)
gate_bwd_kernel(const float *__restrict__ probs, const int32_t *__restrict__ idx,
                const float *__restrict__ dw, const float *__restrict__ coef,
                int64_t S, int E, int k, float aux_w, float inv_temp,
                float *__restrict__ dlogits, __nv_bfloat16 *__restrict__ dl2, int P) {
  griddep_begin();
  const int lane = threadIdx.x & 31;
  const int64_t s = int64_t(blockIdx.x) * kWarpsPerCta + (threadIdx.x >> 5);
  if (s >= S) return;
  const float *p = probs + s * E;
  const int i1 = idx[s * k];
  const int i2 = k == 2 ? idx[s * k + 1] : -1;
  float g1, g2 = 0.0f;
  if (k == 1) {
    g1 = dw[s];
  } else {
    // w_j = p_j / (p_1 + p_2)
    const float p1 = p[i1], p2 = p[i2];
    const float P = p1 + p2;
    const float inv = 1.0f / (P * P);
    const float d = dw[s * 2] - dw[s * 2 + 1];
    g1 = p2 * d * inv;
    g2 = -p1 * d * inv;
  }
  float dot = 0.0f;
  for (int e = lane; e < E; e += 32) {
    float dp = aux_w * coef[e];
    if (e == i1) dp += g1;
    if (e == i2) dp += g2;
    dot = fmaf(dp, p[e], dot);
  }
  dot = warp_sum(dot);
  for (int e = lane; e < E; e += 32) {
    float dp = aux_w * coef[e];
    if (e == i1) dp += g1;
    if (e == i2) dp += g2;
    const float dl = inv_temp * p[e] * (dp - dot);  // the softmax saw logits / T
    if (dlogits) dlogits[s * E + e] = dl;
    if (dl2) {
      const __nv_bfloat16 hi = __float2bfloat16_rn(dl);
      dl2[s * 2 * P + e] = hi;
      dl2[s * 2 * P + P + e] = __float2bfloat16_rn(dl - __bfloat162float(hi));
    }
  }
  if (dl2)  // the padding columns of both halves
    for (int e = E + lane; e < P; e += 32) {
      dl2[s * 2 * P + e] = __float2bfloat16_rn(0.0f);
      dl2[s * 2 * P + P + e] = __float2bfloat16_rn(0.0f);
    }
}

inline unsigned token_blocks(int64_t S) { return unsigned((S + kWarpsPerCta - 1) / kWarpsPerCta); }

}  // namespace

cudaError_t launch_dispatch(const void *x, int dtype, int64_t S, int d, int k,
                            const int32_t *idx, const int32_t *slot, const int32_t *offsets,
                            void *x_disp, cudaStream_t st) {
  if (S == 0) return cudaSuccess;
  const int nvec = d * elem_bytes(dtype) / 16;
  return launch_k(dispatch_kernel, token_blocks(S), kWarpsPerCta * 32, 0, st,
                  static_cast<const uint4 *>(x), S, nvec, k, idx, slot, offsets,
                  static_cast<uint4 *>(x_disp));
}

cudaError_t launch_combine(const void *out_disp, int dtype, int64_t S, int d, int k,
                           const int32_t *idx, const int32_t *slot, const int32_t *offsets,
                           const float *w, void *y, cudaStream_t st, const void *res,
                           const float *mix) {
  if (S == 0) return cudaSuccess;
  const int nvec = d * elem_bytes(dtype) / 16;
  auto *m2 = reinterpret_cast<const float2 *>(mix);
  if (dtype == MOE_F32)
    return launch_k(combine_kernel<float>, token_blocks(S), kWarpsPerCta * 32, 0, st,
                    static_cast<const uint4 *>(out_disp), S, nvec, k, idx, slot, offsets, w,
                    static_cast<const uint4 *>(res), m2, static_cast<uint4 *>(y));
  return launch_k(combine_kernel<__nv_bfloat16>, token_blocks(S), kWarpsPerCta * 32, 0, st,
                  static_cast<const uint4 *>(out_disp), S, nvec, k, idx, slot, offsets, w,
                  static_cast<const uint4 *>(res), m2, static_cast<uint4 *>(y));
}

cudaError_t launch_residual_mix(const void *x, int dtype, int64_t S, int d, const void *cw,
                                const void *cb, float *mix, cudaStream_t st) {
  if (S == 0) return cudaSuccess;
  const int nvec = d * elem_bytes(dtype) / 16;
  auto *m2 = reinterpret_cast<float2 *>(mix);
  if (dtype == MOE_F32)
    return launch_k(residual_mix_kernel<float>, token_blocks(S), kWarpsPerCta * 32, 0, st,
                    static_cast<const uint4 *>(x), S, nvec, static_cast<const uint4 *>(cw),
                    static_cast<const float *>(cb), m2);
  return launch_k(residual_mix_kernel<__nv_bfloat16>, token_blocks(S), kWarpsPerCta * 32, 0, st,
                  static_cast<const uint4 *>(x), S, nvec, static_cast<const uint4 *>(cw),
                  static_cast<const __nv_bfloat16 *>(cb), m2);
}

cudaError_t launch_combine_bwd(const void *dy, const void *out_disp, int dtype, int64_t S,
                               int d, int k, const int32_t *idx, const int32_t *slot,
                               const int32_t *offsets, const float *w, void *d_out, float *dw,
                               cudaStream_t st, int32_t *rows) {
  if (S == 0) return cudaSuccess;
  const int nvec = d * elem_bytes(dtype) / 16;
  auto *dy4 = static_cast<const uint4 *>(dy);
  auto *o4 = static_cast<const uint4 *>(out_disp);
  auto *do4 = static_cast<uint4 *>(d_out);
  if (dtype == MOE_F32)
    return launch_k(combine_bwd_kernel<float>, token_blocks(S), kWarpsPerCta * 32, 0, st, dy4, o4, S,
                    nvec, k, idx, slot, offsets, w, do4, dw, rows);
  return launch_k(combine_bwd_kernel<__nv_bfloat16>, token_blocks(S), kWarpsPerCta * 32, 0, st, dy4,
                  o4, S, nvec, k, idx, slot, offsets, w, do4, dw, rows);
}

cudaError_t launch_group_colsum(const void *M, int dtype, int N, int G,
                                const int32_t *offsets, void *db, cudaStream_t st) {
  if (dtype == MOE_BF16 && N % 8 == 0) {
    dim3 grid((N + kColsumCols - 1) / kColsumCols, G);
    return launch_k(group_colsum_bf16_kernel, grid, kColsumThreads, 0, st,
                    static_cast<const uint4 *>(M), N / 8, offsets,
                    static_cast<uint4 *>(db));
  }
  dim3 grid((N + 31) / 32, G);
  return launch_k(group_colsum_kernel, grid, dim3(32, 8), 0, st, M, dtype, N, offsets, db);
}

cudaError_t launch_aux_coef(const int32_t *idx, const float *probs, int64_t S, int k, int E,
                            int aux_type, float *coef, cudaStream_t st) {
  if (S == 0) return cudaMemsetAsync(coef, 0, sizeof(float) * E, st);
  return launch_k(aux_coef_kernel, 1, 1024, 0, st, idx, probs, S, k, E, aux_type, coef);
}

cudaError_t launch_gate_bwd(const float *probs, const int32_t *idx, const float *dw,
                            const float *coef, int64_t S, int E, int k, float aux_w,
                            float inv_temp, float *dlogits, void *dl2, int P,
                            cudaStream_t st) {
  if (S == 0) return cudaSuccess;
  return launch_k(gate_bwd_kernel, token_blocks(S), kWarpsPerCta * 32, 0, st, probs, idx, dw,
                  coef, S, E, k, aux_w, inv_temp, dlogits,
                  static_cast<__nv_bfloat16 *>(dl2), P);
}

}  // namespace moe
