// Fused gate for bf16 layers: router GEMM on the tensor cores + softmax +
// top-k + combine weights + per-CTA routing histograms, one pass over x.
//
// MoE explainer (lpnh.cn/news/725941) §3.1 Steps 1-2 (router linear layer,
// top-k, softmax over the selected logits); DeepSeek-MoE page
// (lnwmold.com/news/1162317) ch.1 (softmax -> top-2).  The router GEMM is
// small (N = E <= 256) and the stage is bound by reading x once from HBM,
// so the kernel streams x through a TMA pipeline into tcgen05.mma
// (M = 128 tokens, N = E rounded up to 16, K = d) and does all routing math
// on the 128 fp32 logit rows straight out of TMEM, one token per thread:
//   warp 0      TMA producer (x tile 128 x 64, W_g tile E x 64 per stage)
//   warp 1      TMEM allocator + MMA issuer
//   warps 2..5  epilogue: logits (+ bias) -> max, softmax, top-k with ties to
//               the lower index, weights; then the CTA's count and rank of
//               every (choice, expert) pair in token order and the CTA's
//               per-expert probability sums (deterministic, no atomics).
// The slot scan and assignment that follow are the same kernels as for the
// fp32 layer (route.cu).
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int GBM = 128, GBK = 64, GSTAGES = 4;
constexpr int kGateThreads = 192;
constexpr uint32_t kGateABytes = GBM * GBK * 2;  // 16 KB
constexpr uint64_t kGateWaitNs = 2000000000ull;

struct __align__(8) GateCtl {
  uint64_t full[GSTAGES];
  uint64_t empty[GSTAGES];
  uint64_t done;
  uint32_t tmem_base;
  int abort;
  int32_t wcnt[4][kMaxExperts];     // per token-quadrant counts, then prefixes
  float psum[4][kMaxExperts];       // per token-quadrant probability sums
  int32_t choice[2][GBM];
};

__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

__global__ void __launch_bounds__(kGateThreads)
gate_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
               int64_t S, int d, int E, int E_pad, int k, uint32_t idesc, uint32_t tmem_cols,
               const float *__restrict__ logit_bias, float *__restrict__ logits_out,
               float *__restrict__ probs_out, int32_t *__restrict__ idx_out,
               float *__restrict__ w_out, int32_t *__restrict__ rank_out,
               int32_t *__restrict__ hist, float *__restrict__ psum_out, int64_t nblk,
               unsigned int *err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  const uint32_t b_bytes = uint32_t(E_pad) * GBK * 2;
  const uint32_t stage_bytes = kGateABytes + b_bytes;  // multiple of 1024
  GateCtl &ctl = *reinterpret_cast<GateCtl *>(smem + GSTAGES * stage_bytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = (d + GBK - 1) / GBK;
  const int64_t tok0 = int64_t(blockIdx.x) * GBM;

  if (threadIdx.x == 0) {
    for (int s = 0; s < GSTAGES; ++s) {
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
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ctl.tmem_base;
  volatile int *abort = &ctl.abort;

  if (warp == 0) {
    if (lane == 0) {
      uint32_t armed = 0, armed_phase = 0;
      bool ok = true;
      for (int kb = 0; kb < nk; ++kb) {
        const int stage = kb % GSTAGES;
        const uint32_t phase = (kb / GSTAGES) & 1;
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
        for (int s = 0; s < GSTAGES; ++s)
          if (armed & (1u << s))
            ptx::mbar_wait(ptx::smem_addr(&ctl.full[s]), (armed_phase >> s) & 1u, nullptr,
                           kGateWaitNs / 4);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      for (int kb = 0; kb < nk; ++kb) {
        const int stage = kb % GSTAGES;
        const uint32_t phase = (kb / GSTAGES) & 1;
        if (!ptx::mbar_wait(ptx::smem_addr(&ctl.full[stage]), phase, abort, kGateWaitNs)) {
          record_error(err, kErrGateMma | uint32_t(blockIdx.x & 0xffffff));
          *abort = 1;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t a0 = ptx::smem_addr(smem + stage * stage_bytes);
        const uint32_t b0 = a0 + kGateABytes;
#pragma unroll
        for (int kk = 0; kk < GBK / 16; ++kk)
          ptx::mma_bf16(tmem, ptx::sdesc_sw128(a0 + kk * 32, 16, 1024),
                        ptx::sdesc_sw128(b0 + kk * 32, 16, 1024), idesc,
                        (kb | kk) != 0 ? 1u : 0u);
        ptx::mma_commit(ptx::smem_addr(&ctl.empty[stage]));
      }
      ptx::mma_commit(ptx::smem_addr(&ctl.done));
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;            // TMEM lane quadrant = token group
    const int r = q * 32 + lane;       // token row in the tile
    const int64_t s = tok0 + r;
    const bool valid = s < S;
    const bool ok = ptx::mbar_wait(ptx::smem_addr(&ctl.done), 0, abort, kGateWaitNs);
    if (!ok) {
      record_error(err, kErrGateEpilogue | uint32_t(blockIdx.x & 0xffffff));
      *abort = 1;
    }
    ptx::tc_fence_after();
    const uint32_t trow = tmem + (uint32_t(q * 32) << 16);
    const int nchunk = (E + 31) / 32;

    // pass 1: logits (+ bias), max, top-2 (ties -> lower index)
    float m = -INFINITY, b1 = -INFINITY, b2 = -INFINITY;
    int i1 = -1, i2 = -1;
    for (int c = 0; c < nchunk; ++c) {
      uint32_t raw[32];
      ptx::tmem_ld32(trow + uint32_t(c * 32), raw);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        const int e = c * 32 + t;
        if (e >= E) break;
        float v = __uint_as_float(raw[t]);
        if (logit_bias) v += logit_bias[e];
        if (valid && logits_out) logits_out[s * E + e] = v;
        m = fmaxf(m, v);
        if (i1 < 0 || v > b1) {
          b2 = b1; i2 = i1;
          b1 = v; i1 = e;
        } else if (i2 < 0 || v > b2) {
          b2 = v; i2 = e;
        }
      }
    }
    // pass 2: softmax normaliser
    float z = 0.0f;
    for (int c = 0; c < nchunk; ++c) {
      uint32_t raw[32];
      ptx::tmem_ld32(trow + uint32_t(c * 32), raw);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        const int e = c * 32 + t;
        if (e >= E) break;
        float v = __uint_as_float(raw[t]);
        if (logit_bias) v += logit_bias[e];
        z += expf(v - m);
      }
    }
    const float inv_z = 1.0f / z;
    // pass 3: probabilities and the CTA's per-expert sums (tokens < S only)
    for (int c = 0; c < nchunk; ++c) {
      uint32_t raw[32];
      ptx::tmem_ld32(trow + uint32_t(c * 32), raw);
      ptx::tmem_ld_wait();
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        const int e = c * 32 + t;
        if (e >= E) break;  // uniform across the warp
        float v = __uint_as_float(raw[t]);
        if (logit_bias) v += logit_bias[e];
        const float p = valid ? expf(v - m) * inv_z : 0.0f;
        if (valid && probs_out) probs_out[s * E + e] = p;
        const float ps = warp_sum(p);
        if (lane == 0) ctl.psum[q][e] = ps;
      }
    }
    ptx::tc_fence_before();

    if (valid) {
      idx_out[s * k] = i1;
      if (k == 1) {
        w_out[s] = inv_z;  // exp(l1 - max) = 1
      } else {
        const float x2 = expf(b2 - m);
        const float den = 1.0f + x2;
        w_out[s * 2] = 1.0f / den;
        w_out[s * 2 + 1] = x2 / den;
        idx_out[s * 2 + 1] = i2;
      }
    }
    ctl.choice[0][r] = valid ? i1 : -1;
    ctl.choice[1][r] = (valid && k == 2) ? i2 : -1;

    // per-CTA histogram and in-order ranks of every (choice j, expert e)
    const int et = threadIdx.x - 64;  // 0..127 over the epilogue threads
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
        hist[(int64_t(j) * E + ee) * nblk + blockIdx.x] = run;
      }
      epi_sync();
      if (e >= 0) rank_out[s * k + j] = ctl.wcnt[q][e] + rank;
      epi_sync();
    }
    for (int ee = et; ee < E; ee += 128)
      psum_out[int64_t(ee) * nblk + blockIdx.x] =
          ((ctl.psum[0][ee] + ctl.psum[1][ee]) + ctl.psum[2][ee]) + ctl.psum[3][ee];
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, tmem_cols);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn gate_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

bool gate_map(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint32_t box_inner,
              uint32_t box_outer) {
  EncodeTiledFn fn = gate_encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_gate_tc(const GateTcArgs &a, cudaStream_t st) {
  const int64_t nblk = (a.S + GBM - 1) / GBM;
  if (nblk == 0) return cudaSuccess;
  const int E_pad = (a.E + 15) / 16 * 16;
  uint32_t cols = 32;
  while (int(cols) < E_pad) cols <<= 1;
  CUtensorMap tx, tw;
  if (!gate_map(&tx, a.x, uint64_t(a.d), uint64_t(a.S), GBK, GBM)) return cudaErrorInvalidValue;
  if (!gate_map(&tw, a.w_gate, uint64_t(a.d), uint64_t(a.E), GBK, uint32_t(E_pad)))
    return cudaErrorInvalidValue;
  const size_t smem = 1024 + GSTAGES * (kGateABytes + size_t(E_pad) * GBK * 2) + sizeof(GateCtl);
  static size_t attr = 0;
  if (smem > attr) {
    cudaError_t e = cudaFuncSetAttribute(gate_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(232448));
    if (e != cudaSuccess) return e;
    attr = 232448;
  }
  const uint32_t idesc = ptx::idesc_bf16(GBM, E_pad, 0, 0);
  gate_tc_kernel<<<unsigned(nblk), kGateThreads, smem, st>>>(
      tx, tw, a.S, a.d, a.E, E_pad, a.k, idesc, cols, a.logit_bias, a.logits, a.probs, a.idx,
      a.w, a.rank, a.hist, a.psum, nblk, a.err);
  return cudaGetLastError();
}

}  // namespace moe
