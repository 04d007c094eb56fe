// Fused gate for bf16 layers: router GEMM on the tensor cores + softmax +
// top-k + combine weights + per-CTA routing histograms, one pass over x.
//
// MoE explainer (lpnh.cn/news/725941) §3.1 Steps 1-2 (router linear layer,
// top-k, softmax over the selected logits); DeepSeek-MoE page
// (lnwmold.com/news/1162317) ch.1 (softmax -> top-2).  The router GEMM is
// small (N = E <= 256) and the stage is bound by reading x once from HBM,
// so the kernel streams x through a TMA pipeline into tcgen05.mma
// (M = 128 tokens, N = E rounded up to 16, K = d).  The routing math that
// follows is latency-bound, so it is spread over all 16 warps of the CTA:
//   warp 0      TMA producer (x tile 128 x 64, W_g tile E x 64 per stage)
//   warp 1      TMEM allocator + MMA issuer
//   warps 4..7  copy the 128 x E fp32 logits (+ the per-expert or
//               per-token logit bias) from TMEM into a
//               shared-memory tile (the ring buffers are idle by then)
//   all warps   4 lanes per token, each over a quarter of the experts:
//               top-2 with ties to the lower index, softmax of logits / T
//               (the gate temperature), weights;
//               coalesced row copies of logits / probabilities; per-expert
//               probability sums over the CTA's tokens
//   warps 4..7  the CTA's count and rank of every (choice, expert) pair in
//               token order (deterministic, no atomics).
// The slot scan and assignment that follow are the same kernels as for the
// fp32 layer (route.cu).
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int GBM = 128, GBK = 64, kMaxGateStages = 8;
// the routing scan reads the per-CTA histogram rows this kernel writes
static_assert(GBM == kRouteTokensPerCta, "gate tile and routing CTA must cover the same tokens");
constexpr int kGateThreads = 512;  // 16 warps
constexpr uint32_t kGateABytes = GBM * GBK * 2;  // 16 KB
constexpr uint64_t kGateWaitNs = 2000000000ull;

struct __align__(8) GateCtl {
  uint64_t full[kMaxGateStages];
  uint64_t empty[kMaxGateStages];
  uint64_t done;
  uint32_t tmem_base;
  int abort;
  int32_t wcnt[4][kMaxExperts];     // per token-quadrant counts, then prefixes
  int32_t choice[2][GBM];
};

// A (logit, expert) candidate of the top-2 search; i < 0 is "none".
struct Cand {
  float v;
  int i;
};
// a ranks before b: larger logit, ties to the lower expert index.
__device__ __forceinline__ bool cand_before(const Cand &a, const Cand &b) {
  return a.i >= 0 && (b.i < 0 || a.v > b.v || (a.v == b.v && a.i < b.i));
}
__device__ __forceinline__ void cand_push(Cand &t1, Cand &t2, const Cand &x) {
  if (cand_before(x, t1)) {
    t2 = t1;
    t1 = x;
  } else if (cand_before(x, t2)) {
    t2 = x;
  }
}
// (t1, t2) <- top-2 of the union of two top-2 lists.
__device__ __forceinline__ void cand_merge(Cand &t1, Cand &t2, const Cand &u1, const Cand &u2) {
  if (cand_before(u1, t1)) {
    t2 = cand_before(t1, u2) ? t1 : u2;
    t1 = u1;
  } else if (cand_before(u1, t2)) {
    t2 = u1;
  }
}

__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

__global__ void __launch_bounds__(kGateThreads, 1)
gate_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
               int64_t S, int d, int E, int E_pad, int k, uint32_t idesc, uint32_t tmem_cols,
               int nstages, uint32_t ring_bytes, const float *__restrict__ logit_bias,
               int bias_ld, float inv_temp, float *__restrict__ logits_out,
               float *__restrict__ probs_out, int32_t *__restrict__ idx_out,
               float *__restrict__ w_out, int32_t *__restrict__ rank_out,
               int32_t *__restrict__ hist, float *__restrict__ psum_out, int64_t nblk,
               unsigned int *err) {
  griddep_begin();
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const uint32_t b_bytes = uint32_t(E_pad) * GBK * 2;
  const uint32_t stage_bytes = kGateABytes + b_bytes;  // multiple of 1024
  GateCtl &ctl = *reinterpret_cast<GateCtl *>(smem + ring_bytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = (d + GBK - 1) / GBK;
  const int64_t tok0 = int64_t(blockIdx.x) * GBM;
  // 128 x E logits, then probabilities, row pitch E + 1 floats; it overlays
  // the ring, which is idle once every MMA has completed
  float *tile = reinterpret_cast<float *>(smem);
  const int ldt = E + 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < nstages; ++s) {
      ptx::mbar_init(ptx::smem_addr(&ctl.full[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl.empty[s]), 1);
    }
    ptx::mbar_init(ptx::smem_addr(&ctl.done), 1);
    ctl.abort = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(&ctl.tmem_base), tmem_cols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  block_sync();
  ptx::tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  volatile int *abort = &ctl.abort;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t armed = 0, armed_phase = 0;
      bool ok = true;
      for (int kb = 0; kb < nk; ++kb) {
        const int stage = kb % nstages;
        const uint32_t phase = (kb / nstages) & 1;
        if (!ptx::mbar_wait(ptx::smem_addr(&ctl.empty[stage]), phase ^ 1u, abort, kGateWaitNs)) {
          record_error(err, kErrGateProducer | uint32_t(blockIdx.x & 0xffffff));
          *abort = 1;
          ok = false;
          break;
        }
        const uint32_t fb = ptx::smem_addr(&ctl.full[stage]);
        uint8_t *st = smem + stage * stage_bytes;
        ptx::mbar_arrive_expect_tx(fb, stage_bytes);
        ptx::tma_load_2d(ptx::smem_addr(st), &tmX, fb, kb * GBK, int32_t(tok0));
        ptx::tma_load_2d(ptx::smem_addr(st + kGateABytes), &tmW, fb, kb * GBK, 0);
        armed |= 1u << stage;
        armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
      }
      if (!ok)
        for (int s = 0; s < nstages; ++s)
          if (armed & (1u << s))
            ptx::mbar_wait(ptx::smem_addr(&ctl.full[s]), (armed_phase >> s) & 1u, nullptr,
                           kGateWaitNs / 4);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint64_t desc0 = ptx::sdesc_sw128(ptx::smem_addr(smem), 16, 1024);
      bool ok = true;
      for (int kb = 0; kb < nk; ++kb) {
        const int stage = kb % nstages;
        const uint32_t phase = (kb / nstages) & 1;
        if (!ptx::mbar_wait(ptx::smem_addr(&ctl.full[stage]), phase, abort, kGateWaitNs)) {
          record_error(err, kErrGateMma | uint32_t(blockIdx.x & 0xffffff));
          *abort = 1;
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint64_t ast = ptx::sdesc_add(desc0, stage * stage_bytes);
        const uint64_t bst = ptx::sdesc_add(ast, kGateABytes);
#pragma unroll
        for (int kk = 0; kk < GBK / 16; ++kk)
          ptx::mma_bf16(tmem, ptx::sdesc_add(ast, kk * 32), ptx::sdesc_add(bst, kk * 32), idesc,
                        (kb | kk) != 0 ? 1u : 0u);
        ptx::mma_commit(ptx::smem_addr(&ctl.empty[stage]));
      }
      ptx::mma_commit(ptx::smem_addr(&ctl.done));
      // after a give-up, the MMAs already issued finish before TMEM is freed
      if (!ok) ptx::mbar_wait(ptx::smem_addr(&ctl.done), 0, nullptr, kGateWaitNs / 4);
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------- TMEM -> shared-memory logits tile
    const int q = warp & 3;  // TMEM lane quadrant this warp may access
    const int r = q * 32 + lane;
    if (!ptx::mbar_wait(ptx::smem_addr(&ctl.done), 0, abort, kGateWaitNs)) {
      record_error(err, kErrGateEpilogue | uint32_t(blockIdx.x & 0xffffff));
      *abort = 1;
    }
    ptx::tc_fence_after();
    const uint32_t trow = tmem + (uint32_t(q * 32) << 16);
    float *row = tile + r * ldt;
    // the logit bias of this token: one row for all tokens, or its own row
    const float *bias_row =
        logit_bias == nullptr || (bias_ld != 0 && tok0 + r >= S)
            ? nullptr
            : logit_bias + (bias_ld != 0 ? (tok0 + r) * bias_ld : 0);
    for (int c = 0; c < (E + 31) / 32; ++c) {
      uint32_t raw[32];
      ptx::tmem_ld32(trow + uint32_t(c * 32), raw);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        const int e = c * 32 + t;
        if (e < E) row[e] = __uint_as_float(raw[t]) + (bias_row ? bias_row[e] : 0.0f);
      }
    }
    ptx::tc_fence_before();
  }
  block_sync();  // the logits tile is complete

  // ---- logits out: one token row (E floats) per warp step, coalesced
  if (logits_out)
    for (int rr = warp; rr < GBM; rr += kGateThreads / 32)
      if (tok0 + rr < S)
        for (int e = lane; e < E; e += 32) logits_out[(tok0 + rr) * E + e] = tile[rr * ldt + e];

  // ---- per token: 4 lanes, each over a contiguous quarter of the experts
  const int tk = threadIdx.x >> 2, seg = threadIdx.x & 3;
  const int64_t s = tok0 + tk;
  const bool valid = s < S;
  const int cs = (E + 3) >> 2;
  const int c0 = min(E, seg * cs), c1 = min(E, c0 + cs);
  float *trow_s = tile + tk * ldt;
  Cand best1{-INFINITY, -1}, best2{-INFINITY, -1};
  for (int e = c0; e < c1; ++e) cand_push(best1, best2, Cand{trow_s[e], e});
#pragma unroll
  for (int o = 1; o <= 2; o <<= 1) {
    Cand u1, u2;
    u1.v = __shfl_xor_sync(kFullMask, best1.v, o);
    u1.i = __shfl_xor_sync(kFullMask, best1.i, o);
    u2.v = __shfl_xor_sync(kFullMask, best2.v, o);
    u2.i = __shfl_xor_sync(kFullMask, best2.i, o);
    cand_merge(best1, best2, u1, u2);
  }
  const float m = best1.v;  // the top-1 logit is the softmax shift
  float za = 0.0f, zb = 0.0f;
  int ez = c0;
  for (; ez + 1 < c1; ez += 2) {
    za += expf((trow_s[ez] - m) * inv_temp);
    zb += expf((trow_s[ez + 1] - m) * inv_temp);
  }
  if (ez < c1) za += expf((trow_s[ez] - m) * inv_temp);
  float z = za + zb;
  z += __shfl_xor_sync(kFullMask, z, 1);
  z += __shfl_xor_sync(kFullMask, z, 2);
  const float inv_z = 1.0f / z;
  block_sync();  // every read of the logits tile is done

  // probabilities replace the logits in the tile (0 for tokens >= S)
  for (int e = c0; e < c1; ++e) trow_s[e] = valid ? expf((trow_s[e] - m) * inv_temp) * inv_z : 0.0f;
  if (seg == 0) {
    const int i1 = best1.i, i2 = best2.i;
    if (valid) {
      idx_out[s * k] = i1;
      if (k == 1) {
        w_out[s] = inv_z;  // exp(l1 - max) = 1
      } else {
        const float x2 = expf((best2.v - m) * inv_temp);
        const float den = 1.0f + x2;
        w_out[s * 2] = 1.0f / den;
        w_out[s * 2 + 1] = x2 / den;
        idx_out[s * 2 + 1] = i2;
      }
    }
    ctl.choice[0][tk] = valid ? i1 : -1;
    ctl.choice[1][tk] = (valid && k == 2) ? i2 : -1;
  }
  block_sync();  // probabilities and choices are complete

  if (probs_out)
    for (int rr = warp; rr < GBM; rr += kGateThreads / 32)
      if (tok0 + rr < S)
        for (int e = lane; e < E; e += 32) probs_out[(tok0 + rr) * E + e] = tile[rr * ldt + e];
  {
    // CTA sums of each expert's probabilities: tpc lanes per expert, each
    // over a fixed stride of tokens, then a butterfly (fixed order)
    int tpc = 1;
    while (tpc < 32 && 2 * tpc * E <= kGateThreads) tpc <<= 1;
    const int e = threadIdx.x / tpc, part = threadIdx.x % tpc;
    float ps = 0.0f;
    if (e < E)
      for (int rr = part; rr < GBM; rr += tpc) ps += tile[rr * ldt + e];
    for (int o = tpc >> 1; o > 0; o >>= 1) ps += __shfl_xor_sync(kFullMask, ps, o, tpc);
    if (e < E && part == 0) psum_out[int64_t(blockIdx.x) * E + e] = ps;
  }

  if (warp >= 4 && warp < 8) {
    // per-CTA histogram and in-order ranks of every (choice j, expert e)
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const int64_t sr = tok0 + r;
    const int et = threadIdx.x - 128;  // 0..127 over warps 4..7
    for (int j = 0; j < k; ++j) {
      for (int i = et; i < 4 * kMaxExperts; i += 128) (&ctl.wcnt[0][0])[i] = 0;
      epi_sync();
      const int e = ctl.choice[j][r];
      const unsigned peers = __match_any_sync(kFullMask, e);
      const int rank = __popc(peers & lanemask_lt());
      if (e >= 0 && rank == 0) ctl.wcnt[q][e] = __popc(peers);
      epi_sync();
      for (int ee = et; ee < E; ee += 128) {
        int run = 0;
        for (int w = 0; w < 4; ++w) {
          const int cnt = ctl.wcnt[w][ee];
          ctl.wcnt[w][ee] = run;
          run += cnt;
        }
        hist[(int64_t(blockIdx.x) * k + j) * E + ee] = run;
      }
      epi_sync();
      if (e >= 0) rank_out[sr * k + j] = ctl.wcnt[q][e] + rank;
      epi_sync();
    }
  }

  ptx::tc_fence_before();
  block_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, tmem_cols);
  }
}

}  // namespace

cudaError_t launch_gate_tc(const GateTcArgs &a, cudaStream_t st) {
  const int64_t nblk = (a.S + GBM - 1) / GBM;
  if (nblk == 0) return cudaSuccess;
  const int E_pad = (a.E + 15) / 16 * 16;
  uint32_t cols = 32;
  while (int(cols) < E_pad) cols <<= 1;
  CUtensorMap tx, tw;
  if (!make_bf16_map(&tx, a.x, uint64_t(a.d), uint64_t(a.S), GBK, GBM)) return cudaErrorInvalidValue;
  if (!make_bf16_map(&tw, a.w_gate, uint64_t(a.d), uint64_t(a.E), GBK, uint32_t(E_pad)))
    return cudaErrorInvalidValue;
  // As many ring stages as fit (at most kMaxGateStages, at most one per K
  // block): the stage is one CTA per SM, so the bytes it keeps in flight
  // decide how close the x stream gets to HBM bandwidth.
  constexpr size_t kSmemLimit = 232448;
  const size_t stage_bytes = kGateABytes + size_t(E_pad) * GBK * 2;
  const size_t tile_bytes = (size_t(GBM) * (a.E + 1) * 4 + 1023) & ~size_t(1023);
  const size_t fixed = 1024 + sizeof(GateCtl);
  const int nk = (a.d + GBK - 1) / GBK;
  int nstages = int((kSmemLimit - fixed) / stage_bytes);
  if (nstages > kMaxGateStages) nstages = kMaxGateStages;
  if (nstages > nk) nstages = nk;
  if (nstages < 1) return cudaErrorInvalidValue;
  size_t ring = size_t(nstages) * stage_bytes;
  if (ring < tile_bytes) ring = tile_bytes;
  const size_t smem = fixed + ring;
  if (smem > kSmemLimit) return cudaErrorInvalidValue;
  static PerDevice<int> smem_raised;
  int unused = 0;
  if (const cudaError_t e = smem_raised.get(&unused, [&](int &) {
        return cudaFuncSetAttribute(gate_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    int(kSmemLimit));
      }); e != cudaSuccess)
    return e;
  const uint32_t idesc = ptx::idesc_bf16(GBM, E_pad, 0, 0);
  return launch_k(gate_tc_kernel, unsigned(nblk), kGateThreads, smem, st, tx, tw, a.S, a.d, a.E,
                  E_pad, a.k, idesc, cols, nstages, uint32_t(ring), a.logit_bias, a.bias_ld,
                  a.inv_temp, a.logits, a.probs,
                  a.idx, a.w, a.rank, a.hist, a.psum, nblk, a.err);
}

}  // namespace moe
