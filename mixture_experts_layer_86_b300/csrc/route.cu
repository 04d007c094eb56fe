// Routing: softmax, top-k, combine weights, capacity-limited slot
// assignment in priority order, counts, offsets and l_aux.
//
// MoE explainer (lpnh.cn/news/725941) §3.1 Step 2 (top-k, softmax over the
// selected logits), DeepSeek-MoE page (lnwmold.com/news/1162317) ch.1
// (softmax -> top-2, capacity = ceil(S*2/E*cf)), deepspeed.moe overview
// (adg.csdn.net/694deb285b9f5f31781ae763) §2.1 (min_capacity, drop_tokens,
// gate_loss, expert_count).
//
// Three steps, no atomics (the result is the same on every run):
//  1. per CTA of 128 tokens: softmax, top-k with ties to the lower expert
//     index, weights; the count of each (choice j, expert e) pair in the
//     CTA, the rank of each token among the CTA's tokens with the same
//     (j, e) (kept in `slot` for now), and the CTA's per-expert sum of
//     probabilities.  Done by route_topk (fp32 logits in memory) or by the
//     fused tensor-core gate (gate_tc.cu).  Counts are stored CTA-major,
//     hist[(cta*k + j)*E + e], so a CTA writes one contiguous row and the
//     scan reads rows with consecutive threads on consecutive columns.
//  2. route_scan (one CTA): exclusive scan of every column over CTAs, in
//     place; totals; routed / kept counts; offsets; l_aux.
//  3. route_assign: slot = (first-choice total of e if j == 1) + scanned
//     base + CTA rank.  Every first choice therefore precedes every second
//     choice, each in token order.  slot >= C -> -1; row_src of kept rows.
// The randomised gate options (rng.cuh) enter here: step 1 chooses on the
// logits plus Gumbel noise (rsample, second-choice sampling), and under
// random token selection the CTAs take the tokens in the order of a keyed
// permutation, so every "token order" above becomes that queue order.
#include "common.cuh"
#include "kernels.h"
#include "rng.cuh"

namespace moe {
namespace {

constexpr int kTB = kRouteTokensPerCta;  // tokens per CTA
constexpr int kWarps = kTB / 32;         // warps per CTA (one lane per token in phase 2)
constexpr int kMaxPerLane = kMaxExperts / 32;

inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Reductions within aligned segments of w lanes (w a power of two <= 32; all
// 32 lanes call them).  Over the lanes that hold values, with the others at
// the neutral element, each gives the full-warp tree's result bit for bit:
// the tree only drops additions of zero (maxima of -inf).
__device__ __forceinline__ float seg_sum(float v, int w) {
  for (int o = w >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(kFullMask, v, o);
  return v;
}
__device__ __forceinline__ float seg_max(float v, int w) {
  for (int o = w >> 1; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFullMask, v, o));
  return v;
}
__device__ __forceinline__ void seg_argmax(float &v, int &idx, int w) {
  for (int o = w >> 1; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(kFullMask, v, o);
    const int oi = __shfl_xor_sync(kFullMask, idx, o);
    const bool take = (oi >= 0) && (idx < 0 || ov > v || (ov == v && oi < idx));
    if (take) {
      v = ov;
      idx = oi;
    }
  }
}

// Under random token selection (noise.rts) CTA b works on the tokens at
// queue positions b*kTB ... b*kTB + kTB - 1 instead of those token indices,
// so counts and ranks come out in queue order; every per-token output is
// still written at the token's own index.
__global__ void __launch_bounds__(kTB)
route_topk_kernel(const float *__restrict__ logits, int64_t S, int E, int k, float inv_temp,
                  float *__restrict__ probs, int32_t *__restrict__ idx_out,
                  float *__restrict__ w_out, int32_t *__restrict__ rank_out,
                  int32_t *__restrict__ hist, float *__restrict__ psum, RouteNoise noise) {
  griddep_begin();
  __shared__ int32_t s_choice[2][kTB];
  __shared__ int32_t s_wcnt[kWarps][kMaxExperts];
  __shared__ float s_psum[kWarps][kMaxExperts];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t tok0 = int64_t(blockIdx.x) * kTB;
  const int nq = (E + 31) >> 5;
  const rng::Key key = rng::make_key(noise.seed, noise.offset);
  const rng::Perm perm = rng::make_perm(key, uint32_t(S));
  const bool use_gumbel = noise.gumbel(k);
  const bool sample_all = noise.policy == MOE_NOISE_RSAMPLE;

  float pacc[kMaxPerLane];
#pragma unroll
  for (int q = 0; q < kMaxPerLane; ++q) pacc[q] = 0.0f;

  // ---- phase 1: a segment of W lanes per token (W = E rounded up to a power
  // of two, at most 32), lanes over experts; a warp takes 32 / W tokens per
  // pass, so small expert counts do not leave a warp's tokens in one long
  // dependent chain.  Every reduction gives the full-warp result bit for bit.
  const int W = E > 16 ? 32 : E > 8 ? 16 : E > 4 ? 8 : E > 2 ? 4 : E > 1 ? 2 : 1;
  const int tpp = 32 / W;
  const int sub = lane / W, sl = lane % W;
  // each iteration loads the token rows (logits) of the next pass, then
  // works on the current one (the first iteration only loads)
  const int step = kWarps * tpp;
  float vn[kMaxPerLane], v[kMaxPerLane];
  int64_t s_cur = -1;
  for (int t0 = warp * tpp - step; t0 < kTB; t0 += step) {
    int64_t s_nx = -1;
    if (t0 + step < kTB) {
      s_nx = tok0 + t0 + step + sub;
      if (s_nx >= S) s_nx = -1;
      else if (noise.rts) s_nx = int64_t(rng::token_at(perm, uint32_t(s_nx)));
    }
#pragma unroll
    for (int q = 0; q < kMaxPerLane; ++q) {
      const int e = sl + 32 * q;
      vn[q] = (s_nx >= 0 && q < nq && e < E) ? __ldg(logits + s_nx * E + e) : -INFINITY;
    }
    if (t0 < 0) {
#pragma unroll
      for (int q = 0; q < kMaxPerLane; ++q) v[q] = vn[q];
      s_cur = s_nx;
      continue;
    }
    const int t = t0 + sub;
    const bool live = s_cur >= 0;
    const int64_t s = live ? s_cur : 0;
    float key_v[kMaxPerLane];
    float m = -INFINITY;
#pragma unroll
    for (int q = 0; q < kMaxPerLane; ++q) {
      const int e = sl + 32 * q;
      const bool has = live && q < nq && e < E;
      m = fmaxf(m, v[q]);
      key_v[q] = v[q];
      if (use_gumbel && has) {
        // the selection key: logit + Gumbel noise, one float32 addition
        const uint4 w4 = rng::block(key, rng::kPurposeGateNoise, uint32_t(s), uint32_t(e >> 2));
        key_v[q] = __fadd_rn(v[q], rng::gumbel(rng::uniform(rng::word(w4, e & 3))));
      }
    }
    m = seg_max(m, W);
    float ex[kMaxPerLane];
    float z = 0.0f;
#pragma unroll
    for (int q = 0; q < kMaxPerLane; ++q) {
      const int e = sl + 32 * q;
      ex[q] = (live && q < nq && e < E) ? expf((v[q] - m) * inv_temp) : 0.0f;
      z += ex[q];
    }
    z = seg_sum(z, W);
    const float inv_z = 1.0f / z;
    // top-1 (ties -> lower index), on the noisy keys under rsample
    float b1 = -INFINITY;
    int i1 = -1;
#pragma unroll
    for (int q = 0; q < kMaxPerLane; ++q) {
      const int e = sl + 32 * q;
      const float c = sample_all ? key_v[q] : v[q];
      if (live && q < nq && e < E && (i1 < 0 || c > b1)) {
        b1 = c;
        i1 = e;
      }
    }
    seg_argmax(b1, i1, W);
    int i2 = -1;
    if (k == 2) {
      // the second choice: on the noisy keys under rsample or second-choice
      // sampling
      float b2 = -INFINITY;
#pragma unroll
      for (int q = 0; q < kMaxPerLane; ++q) {
        const int e = sl + 32 * q;
        const float c = use_gumbel ? key_v[q] : v[q];
        if (live && q < nq && e < E && e != i1 && (i2 < 0 || c > b2)) {
          b2 = c;
          i2 = e;
        }
      }
      seg_argmax(b2, i2, W);
    }
#pragma unroll
    for (int q = 0; q < kMaxPerLane; ++q) {
      const int e = sl + 32 * q;
      if (live && q < nq && e < E) {
        const float p = ex[q] * inv_z;
        pacc[q] += p;
        if (probs) probs[s * E + e] = p;
      }
    }
    // exp(l - max) of the chosen experts, from the segment lanes holding them
    float x1 = 0.0f, x2 = 0.0f;
#pragma unroll
    for (int q = 0; q < kMaxPerLane; ++q) {
      const float a = __shfl_sync(kFullMask, ex[q], i1 & 31, W);
      if (i1 >= 0 && (i1 >> 5) == q) x1 = a;
      if (k == 2) {
        const float b = __shfl_sync(kFullMask, ex[q], i2 & 31, W);
        if (i2 >= 0 && (i2 >> 5) == q) x2 = b;
      }
    }
    if (sl == 0) {
      if (!live) {
        s_choice[0][t] = -1;
        s_choice[1][t] = -1;
      } else {
        s_choice[0][t] = i1;
        idx_out[s * k] = i1;
        if (k == 1) {
          w_out[s] = x1 * inv_z;
          s_choice[1][t] = -1;
        } else {
          const float den = x1 + x2;
          w_out[s * 2] = x1 / den;
          w_out[s * 2 + 1] = x2 / den;
          idx_out[s * 2 + 1] = i2;
          s_choice[1][t] = i2;
        }
      }
    }
#pragma unroll
    for (int q = 0; q < kMaxPerLane; ++q) v[q] = vn[q];
    s_cur = s_nx;
  }
  // the segments of a warp hold partial sums of the same experts: add them
  // (lanes of equal sl, in a fixed order)
#pragma unroll
  for (int q = 0; q < kMaxPerLane; ++q)
    for (int o = W; o < 32; o <<= 1) pacc[q] += __shfl_xor_sync(kFullMask, pacc[q], o);
#pragma unroll
  for (int q = 0; q < kMaxPerLane; ++q) {
    const int e = sl + 32 * q;
    if (sub == 0 && q < nq && e < E) s_psum[warp][e] = pacc[q];
  }
  block_sync();
  for (int e = threadIdx.x; e < E; e += kTB) {
    float acc = 0.0f;
    for (int w = 0; w < kWarps; ++w) acc += s_psum[w][e];
    psum[int64_t(blockIdx.x) * E + e] = acc;
  }

  // ---- phase 2: one lane per token; rank among equal (j, e) in queue order
  const int t = threadIdx.x;
  const int64_t s = (noise.rts && tok0 + t < S) ? int64_t(rng::token_at(perm, uint32_t(tok0 + t)))
                                                 : tok0 + t;
  for (int j = 0; j < k; ++j) {
    for (int i = threadIdx.x; i < kWarps * kMaxExperts; i += kTB) (&s_wcnt[0][0])[i] = 0;
    block_sync();
    const int e = s_choice[j][t];
    const unsigned peers = __match_any_sync(kFullMask, e);
    const int rank = __popc(peers & lanemask_lt());
    if (e >= 0 && rank == 0) s_wcnt[warp][e] = __popc(peers);
    block_sync();
    for (int ee = threadIdx.x; ee < E; ee += kTB) {
      int run = 0;
      for (int w = 0; w < kWarps; ++w) {
        const int c = s_wcnt[w][ee];
        s_wcnt[w][ee] = run;
        run += c;
      }
      hist[(int64_t(blockIdx.x) * k + j) * E + ee] = run;
    }
    block_sync();
    if (e >= 0 && s < S) rank_out[s * k + j] = s_wcnt[warp][e] + rank;
    block_sync();
  }
}

constexpr int kScanThreads = 1024;
constexpr int kScanMaxGroups = 32;

// One CTA.  The per-CTA counts form an nblk x (k*E) row-major matrix; thread
// t works on column t % ncol for a contiguous range of rows (group t / ncol),
// so at every step consecutive threads touch consecutive words.  Group sums
// go through shared memory, each group rewrites its rows with exclusive
// prefixes, and the column totals give routed / kept counts, the expert
// offsets (a warp scan) and l_aux.  Probability sums are added as 2^-30
// fixed-point integers: exact, independent of the order, and clear of
// B300's slow float64 pipe (a partial is at most the CTA's token count, so
// S < 2^31 keeps every total below 2^61).
__global__ void __launch_bounds__(kScanThreads)
route_scan_kernel(int64_t nblk, int64_t S, int E, int k, int64_t cap, int aux_type,
                  int32_t *__restrict__ hist, const float *__restrict__ psum,
                  int32_t *__restrict__ first_cnt, int32_t *__restrict__ routed,
                  int32_t *__restrict__ kept, int32_t *__restrict__ offsets,
                  float *__restrict__ l_aux) {
  griddep_begin();
  __shared__ int32_t s_grp[kScanThreads];
  __shared__ long long s_pgrp[kScanThreads];
  __shared__ int32_t s_tot[2][kMaxExperts];
  __shared__ long long s_aux[kMaxExperts];  // sum_s p[s,e] in units of 2^-30
  const int lane = threadIdx.x & 31;

  // ---- count columns: exclusive scan over CTAs, in place
  {
    const int ncol = k * E;
    const int G = min(kScanMaxGroups, kScanThreads / ncol);
    const int col = threadIdx.x % ncol, g = threadIdx.x / ncol;
    const bool act = g < G;
    const int64_t per = (nblk + G - 1) / G;
    const int64_t b0 = act ? min(nblk, g * per) : 0;
    const int64_t b1 = act ? min(nblk, b0 + per) : 0;
    int sum = 0;
#pragma unroll 4
    for (int64_t b = b0; b < b1; ++b) sum += hist[b * ncol + col];
    if (act) s_grp[g * ncol + col] = sum;
    block_sync();
    if (act) {
      int run = 0;
      for (int gg = 0; gg < g; ++gg) run += s_grp[gg * ncol + col];
#pragma unroll 4
      for (int64_t b = b0; b < b1; ++b) {
        const int v = hist[b * ncol + col];
        hist[b * ncol + col] = run;
        run += v;
      }
    }
    if (threadIdx.x < ncol) {
      int tot = 0;
      for (int gg = 0; gg < G; ++gg) tot += s_grp[gg * ncol + threadIdx.x];
      s_tot[threadIdx.x / E][threadIdx.x % E] = tot;
    }
  }
  // ---- probability sums per expert
  {
    const int G = min(kScanMaxGroups, kScanThreads / E);
    const int e = threadIdx.x % E, g = threadIdx.x / E;
    const bool act = g < G;
    const int64_t per = (nblk + G - 1) / G;
    const int64_t b0 = act ? min(nblk, g * per) : 0;
    const int64_t b1 = act ? min(nblk, b0 + per) : 0;
    long long ps = 0;
#pragma unroll 4
    for (int64_t b = b0; b < b1; ++b) ps += fix30_tile(psum[b * E + e]);
    if (act) s_pgrp[g * E + e] = ps;
    block_sync();
    if (threadIdx.x < E) {
      long long tot = 0;
      for (int gg = 0; gg < G; ++gg) tot += s_pgrp[gg * E + threadIdx.x];
      s_aux[threadIdx.x] = tot;
    }
  }
  block_sync();

  // ---- counts, offsets and l_aux: warp 0, lane l owns experts [l*per, ...)
  if (threadIdx.x < 32) {
    const int per = (E + 31) / 32;
    const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
    int local = 0;
    float aux = 0.0f;
    for (int e = e0; e < e1; ++e) {
      const int r = s_tot[0][e] + (k == 2 ? s_tot[1][e] : 0);
      const int kp = (cap < 0 || r < cap) ? r : int(cap);
      routed[e] = r;
      kept[e] = kp;
      first_cnt[e] = s_tot[0][e];
      local += kp;
      aux = fmaf(float(s_aux[e]) * kInvFix30, float(s_tot[0][e]), aux);
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(kFullMask, incl, o);
      if (lane >= o) incl += t;
    }
    int run = incl - local;
    for (int e = e0; e < e1; ++e) {
      offsets[e] = run;
      const int r = s_tot[0][e] + (k == 2 ? s_tot[1][e] : 0);
      run += (cap < 0 || r < cap) ? r : int(cap);
    }
    if (lane == 31) offsets[E] = incl;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) aux += __shfl_xor_sync(kFullMask, aux, o);
    if (aux_type == MOE_AUX_STD) {
      // l_aux = std_e(u_e) + 1e-6, u_e = sum_s p[s,e] / S (population std);
      // fp32 from the exact integer sums (no FP64)
      long long sa = 0;
      for (int e = e0; e < e1; ++e) sa += s_aux[e];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sa += __shfl_xor_sync(kFullMask, sa, o);
      float sq = 0.0f;
      if (S > 0)
        for (int e = e0; e < e1; ++e) {
          const float dv = usage_deviation(s_aux[e], sa, E, S);
          sq = fmaf(dv, dv, sq);
        }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(kFullMask, sq, o);
      if (lane == 0) *l_aux = sqrtf(sq / float(E)) + 1e-6f;
    } else {
      // l_aux = E * sum_e (sum_s p[s,e] / S) * (first[e] / S)
      if (lane == 0) *l_aux = S > 0 ? float(E) * aux / float(S) / float(S) : 0.0f;
    }
  }
}

__global__ void route_assign_kernel(int64_t S, int E, int k, int64_t cap, int64_t nblk,
                                    const int32_t *__restrict__ idx,
                                    const int32_t *__restrict__ hist,
                                    const int32_t *__restrict__ first_cnt,
                                    const int32_t *__restrict__ offsets,
                                    int32_t *__restrict__ slot,
                                    int32_t *__restrict__ row_src, RouteNoise noise) {
  griddep_begin();
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= S * k) return;
  const int64_t s = i / k;
  const int j = int(i - s * k);
  const int e = idx[i];
  // the CTA that ranked this token: by token index, or by queue position
  const int64_t b =
      (noise.rts ? int64_t(rng::position_of(
                       rng::make_perm(rng::make_key(noise.seed, noise.offset), uint32_t(S)),
                       uint32_t(s)))
                 : s) /
      kTB;
  const int pos = hist[(b * k + j) * E + e] + (j == 1 ? first_cnt[e] : 0) + slot[i];
  if (cap < 0 || pos < cap) {
    slot[i] = pos;
    row_src[offsets[e] + pos] = int32_t(i);
  } else {
    slot[i] = -1;
  }
}

}  // namespace

size_t route_workspace_bytes(int64_t S, int E, int k) {
  const int64_t nblk = (S + kTB - 1) / kTB;
  return align256(size_t(nblk) * k * E * 4) + align256(size_t(nblk) * E * 4) +
         align256(size_t(E) * 4);
}

void route_carve_workspace(RouteArgs &a, void *ws) {
  const int64_t nblk = (a.S + kTB - 1) / kTB;
  char *p = static_cast<char *>(ws);
  a.hist = reinterpret_cast<int32_t *>(p);
  p += align256(size_t(nblk) * a.k * a.E * 4);
  a.psum = reinterpret_cast<float *>(p);
  p += align256(size_t(nblk) * a.E * 4);
  a.first_cnt = reinterpret_cast<int32_t *>(p);
}

cudaError_t launch_route_finish(const RouteArgs &a, cudaStream_t st) {
  const int64_t nblk = (a.S + kTB - 1) / kTB;
  if (const cudaError_t e = launch_k(route_scan_kernel, 1, kScanThreads, 0, st, nblk, a.S, a.E, a.k,
                                     a.cap, a.aux_type, a.hist, a.psum, a.first_cnt, a.routed,
                                     a.kept, a.offsets, a.l_aux); e != cudaSuccess)
    return e;
  const int64_t n = a.S * a.k;
  if (n > 0) {
    if (const cudaError_t e = launch_k(route_assign_kernel, unsigned((n + 255) / 256), 256, 0, st,
                                       a.S, a.E, a.k, a.cap, nblk, a.idx, a.hist, a.first_cnt,
                                       a.offsets, a.slot, a.row_src, a.noise); e != cudaSuccess)
      return e;
  }
  return cudaGetLastError();
}

namespace {

// one thread per token: uniforms / Gumbel noise of its experts and its
// queue position
__global__ void gate_noise_kernel(int64_t S, int E, RouteNoise noise, float *__restrict__ uniform,
                                  float *__restrict__ gumbel, int32_t *__restrict__ position) {
  griddep_begin();
  const int64_t s = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (s >= S) return;
  const rng::Key key = rng::make_key(noise.seed, noise.offset);
  if (position) position[s] = int32_t(rng::position_of(rng::make_perm(key, uint32_t(S)), uint32_t(s)));
  for (int e4 = 0; e4 < E; e4 += 4) {
    const uint4 w4 = rng::block(key, rng::kPurposeGateNoise, uint32_t(s), uint32_t(e4 >> 2));
    for (int i = 0; i < 4 && e4 + i < E; ++i) {
      const float u = rng::uniform(rng::word(w4, i));
      if (uniform) uniform[s * E + e4 + i] = u;
      if (gumbel) gumbel[s * E + e4 + i] = rng::gumbel(u);
    }
  }
}

// xj[s, c] = x[s, c] * f[s, c], eight elements per thread (two Philox blocks)
template <typename T>
__global__ void jitter_kernel(const T *__restrict__ x, int64_t S, int d, RouteNoise noise,
                              T *__restrict__ xj) {
  griddep_begin();
  const int n8 = d / 8;
  const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= S * n8) return;
  const int64_t s = i / n8;
  const int c0 = int(i - s * n8) * 8;
  const rng::Key key = rng::make_key(noise.seed, noise.offset);
  const float eps = noise.jitter_eps > 0.0f ? noise.jitter_eps : 0.01f;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const uint4 w4 = rng::block(key, rng::kPurposeJitter, uint32_t(s), uint32_t((c0 >> 2) + h));
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int64_t o = s * d + c0 + h * 4 + q;
      const float f = rng::jitter(rng::uniform(rng::word(w4, q)), eps);
      xj[o] = T(__fmul_rn(float(x[o]), f));
    }
  }
}

}  // namespace

cudaError_t launch_gate_noise(int64_t S, int E, const RouteNoise &n, float *uniform,
                              float *gumbel, int32_t *position, cudaStream_t st) {
  if (S == 0) return cudaSuccess;
  return launch_k(gate_noise_kernel, unsigned((S + 127) / 128), 128, 0, st, S, E, n, uniform,
                  gumbel, position);
}

cudaError_t launch_jitter(const void *x, int dtype, int64_t S, int d, const RouteNoise &n,
                          void *xj, cudaStream_t st) {
  const int64_t total = S * (d / 8);
  if (total == 0) return cudaSuccess;
  const unsigned grid = unsigned((total + 255) / 256);
  if (dtype == MOE_F32)
    return launch_k(jitter_kernel<float>, grid, 256, 0, st, static_cast<const float *>(x), S, d,
                    n, static_cast<float *>(xj));
  return launch_k(jitter_kernel<__nv_bfloat16>, grid, 256, 0, st,
                  static_cast<const __nv_bfloat16 *>(x), S, d, n,
                  static_cast<__nv_bfloat16 *>(xj));
}

cudaError_t launch_route(const RouteArgs &a, cudaStream_t st) {
  const int64_t nblk = (a.S + kTB - 1) / kTB;
  if (nblk > 0) {
    if (const cudaError_t e = launch_k(route_topk_kernel, unsigned(nblk), kTB, 0, st, a.logits, a.S,
                                       a.E, a.k, a.inv_temp, a.probs, a.idx, a.w, a.slot,
                                       a.hist, a.psum, a.noise); e != cudaSuccess)
      return e;
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_route_finish(a, st);
}

}  // namespace moe
