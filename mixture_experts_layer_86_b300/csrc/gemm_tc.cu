// Grouped bf16 GEMM on the B300 tensor cores (tcgen05 + TMEM + TMA).
//
// This is the expert FFN of the MoE layer (MoE explainer, lpnh.cn/news/725941,
// §3.1 Step 4: every expert applies Linear -> act -> Linear to the tokens it
// received), run as ONE persistent kernel over all experts: the experts'
// row counts live on the device (expert_offsets), so no host round trip is
// needed between routing and the FFN.
//
// Operand roles are swapped with respect to C = X W^T: the MMA computes
// C^T = W X^T, so the expert's weights fill the 128-row M side and its
// tokens are the N side.  N is a multiple of 16 chosen per tile, so an
// expert's last token tile pads at most 15 rows instead of a 128-row M
// tile's up to 127 -- at ~500 tokens per expert that padding was ~11% of
// the tensor work.
//
// Two kernels share this design.  tc_gemm_pair_kernel (further down) runs
// it on 2-CTA clusters with tcgen05.mma.cta_group::2 and is the one used on
// any device with two or more SMs; tc_gemm_kernel, described here, is the
// single-CTA form of the same tile loop.
//
// Tiling: 128 output features x up to 256 tokens per tile, K in 64-element
// (128 B) slices, 4-stage TMA -> shared memory pipeline with 128-byte
// swizzle, tcgen05.mma (M=128, N=16..256, K=16) accumulating in TMEM, two
// TMEM accumulators (2 x 256 columns) so the epilogue of one tile overlaps
// the MMAs of the next.  Warp roles (192 threads):
//   warp 0      TMA producer (one lane)
//   warp 1      TMEM allocator + MMA issuer (one lane)
//   warps 2..5  epilogue: each owns 32 features (its TMEM lane quadrant);
//               tcgen05.ld -> bias / activation / dact -> bf16, transposed
//               through a 32 x 32 shared-memory stage so that token rows go
//               out as 16-byte vectors, masked to the expert's tokens.
// Tiles run expert by expert, token tile by token tile, feature tile
// fastest, so CTAs running at the same time share the token tile in L2 and
// an expert's weights stay in L2 across its token tiles.
//
// Every mbarrier wait is bounded: a wait that gives up records an error
// code in the device error word, raises a CTA-wide abort flag, and the CTA
// drains its outstanding copies / MMAs (again bounded) before freeing TMEM.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int kThreads = 192;
constexpr int kTmemCols = 2 * BN;  // two accumulators
constexpr uint32_t kABytes = BM * BK * 2;  // 16 KB
constexpr uint32_t kBBytes = BN * BK * 2;  // 32 KB
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr int kMaxGroups = kMaxExperts;
// swapped-operand grouped GEMM: BM output features x up to BN tokens
constexpr int kFeat = BM, kTok = BN;
constexpr uint32_t kStageBytesPerWarp = 32 * 64;  // 32 tokens x 32 bf16 features

struct __align__(8) SmemCtl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int tile_start[kMaxGroups + 1];  // prefix of (token tiles x feature tiles) over groups
  int row_start[kMaxGroups + 1];   // the expert offsets, read once from global memory
};

constexpr size_t kSmemBytes = 1024 /*align slack*/ + STAGES * (kABytes + kBBytes) +
                              4 * kStageBytesPerWarp + sizeof(SmemCtl);

struct TileCoord {
  int g, tt, ft;  // group, token tile, feature tile
  int row0;       // first row of the group
  int ntok;       // valid tokens of this tile (1..kTok)
};

// Tile order: group by group, token tile by token tile, the nf feature
// tiles of each token tile in turn.  Tiles go to the persistent CTAs
// round-robin, so the pairs working at one time share the group's weights
// and token rows in L2 (a group's partial last token tile comes right after
// its whole ones, while its weights are still there).
template <typename Ctl>
__device__ __forceinline__ void tile_plan(Ctl &c, int G, int nf, const int32_t *offsets,
                                          int64_t dense_rows) {
  // without offsets the rows form one group of dense_rows rows
  for (int g = 0; g <= G; ++g)
    c.row_start[g] = offsets ? offsets[g] : (g == 0 ? 0 : int(dense_rows));
  int run = 0;
  for (int g = 0; g < G; ++g) {
    c.tile_start[g] = run;
    run += ((c.row_start[g + 1] - c.row_start[g] + kTok - 1) / kTok) * nf;
  }
  c.tile_start[G] = run;
}

template <typename Ctl>
__device__ __forceinline__ int tile_total(const Ctl &c, int G) {
  return c.tile_start[G];
}

template <typename Ctl>
__device__ __forceinline__ TileCoord tile_coord(const Ctl &c, int G, int nf, int t) {
  int lo = 0, hi = G - 1;  // last g with tile_start[g] <= t (groups without tiles skipped)
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (c.tile_start[mid] <= t) lo = mid; else hi = mid - 1;
  }
  TileCoord tc;
  tc.g = lo;
  tc.row0 = c.row_start[lo];
  const int rows = c.row_start[lo + 1] - tc.row0;
  const int local = t - c.tile_start[lo];
  tc.tt = local / nf;
  tc.ft = local - tc.tt * nf;
  const int left = rows - tc.tt * kTok;
  tc.ntok = left < kTok ? left : kTok;
  return tc;
}

__device__ __forceinline__ void unpack_bf16x8(const uint4 &u, float *o) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    o[2 * i] = __uint_as_float(w[i] << 16);
    o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}
__device__ __forceinline__ uint4 pack_bf16x8(const float *v) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    w[i] = *reinterpret_cast<uint32_t *>(&b);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// C[r, n] = epi( sum_k X[r, k] * W_g(n, k) ) for the rows r of group g.
// kWMN: W_g is stored [K, N] (N contiguous, the dgrad case) instead of
// [N, K].  The bf16 staging area of each epilogue warp is 32 token rows of
// 32 features (64 B per row).
template <bool kWMN>
__global__ void __launch_bounds__(kThreads, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
               const int32_t *__restrict__ offsets, int64_t dense_rows, int G, int N, int K,
               const __nv_bfloat16 *__restrict__ bias, int act,
               __nv_bfloat16 *__restrict__ C, __nv_bfloat16 *__restrict__ pre,
               const __nv_bfloat16 *__restrict__ grad_src, int dact, unsigned int *err) {
  griddep_begin();
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint8_t *sA = smem;                                   // weights, 128 x 64 per stage
  uint8_t *sB = smem + STAGES * kABytes;                // tokens, 256 x 64 per stage
  uint8_t *sStage = smem + STAGES * (kABytes + kBBytes);
  SmemCtl &ctl = *reinterpret_cast<SmemCtl *>(sStage + 4 * kStageBytesPerWarp);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nf = (N + kFeat - 1) / kFeat;
  const int nk = (K + BK - 1) / BK;

  // ---------------------------------------------------------------- setup
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(ptx::smem_addr(&ctl.full[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl.empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(ptx::smem_addr(&ctl.tfull[a]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl.tempty[a]), 128);
    }
    ptx::mbar_init(ptx::smem_addr(&ctl.drain), 1);
    ctl.abort = 0;
    tile_plan(ctl, G, nf, offsets, dense_rows);
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&tmW);
    ptx::tma_prefetch_desc(&tmX);
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(&ctl.tmem_base), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  block_sync();
  ptx::tc_fence_after();
  const uint32_t tmem_base = ctl.tmem_base;
  const int total = tile_total(ctl, G);
  volatile int *abort = &ctl.abort;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t armed = 0;  // stages holding a copy not yet seen complete here
      uint32_t armed_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        const TileCoord tc = tile_coord(ctl, G, nf, t);
        const int xrow = tc.row0 + tc.tt * kTok;
        for (int kb = 0; kb < nk; ++kb) {
          if (!ptx::mbar_wait(ptx::smem_addr(&ctl.empty[stage]), phase ^ 1u, abort, kWaitLimitNs)) {
            record_error(err, kErrGemmProducer | uint32_t(t & 0xffffff));
            *abort = 1;
            ok = false;
            break;
          }
          const uint32_t fb = ptx::smem_addr(&ctl.full[stage]);
          ptx::mbar_arrive_expect_tx(fb, kABytes + kBBytes);
          if (!kWMN) {
            ptx::tma_load_2d(ptx::smem_addr(sA + stage * kABytes), &tmW, fb, kb * BK,
                             tc.g * N + tc.ft * kFeat);
          } else {
            // two 64(n) x 64(k) boxes, 8 KB apart
#pragma unroll
            for (int j = 0; j < kFeat / 64; ++j)
              ptx::tma_load_2d(ptx::smem_addr(sA + stage * kABytes + j * (BK * 128)), &tmW, fb,
                               tc.ft * kFeat + j * 64, tc.g * K + kb * BK);
          }
          ptx::tma_load_2d(ptx::smem_addr(sB + stage * kBBytes), &tmX, fb, kb * BK, xrow);
          armed |= 1u << stage;
          armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // let copies already issued land before the CTA exits
        for (int s = 0; s < STAGES; ++s)
          if (armed & (1u << s))
            ptx::mbar_wait(ptx::smem_addr(&ctl.full[s]), (armed_phase >> s) & 1u, nullptr,
                           kWaitLimitNs / 4);
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint64_t a_desc0 = kWMN ? ptx::sdesc_sw128(ptx::smem_addr(sA), BK * 128, 1024)
                                    : ptx::sdesc_sw128(ptx::smem_addr(sA), 16, 1024);
      const uint64_t b_desc0 = ptx::sdesc_sw128(ptx::smem_addr(sB), 16, 1024);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++it) {
        const TileCoord tc = tile_coord(ctl, G, nf, t);
        const uint32_t idesc = ptx::idesc_bf16(kFeat, (tc.ntok + 15) & ~15, kWMN ? 1 : 0, 0);
        const int acc = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        if (!ptx::mbar_wait(ptx::smem_addr(&ctl.tempty[acc]), acc_phase ^ 1u, abort, kWaitLimitNs)) {
          record_error(err, kErrGemmMma | 0x800000u | uint32_t(t & 0x7fffff));
          *abort = 1;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + uint32_t(acc * kTok);
        for (int kb = 0; kb < nk; ++kb) {
          if (!ptx::mbar_wait(ptx::smem_addr(&ctl.full[stage]), phase, abort, kWaitLimitNs)) {
            record_error(err, kErrGemmMma | uint32_t(t & 0x7fffff));
            *abort = 1;
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint64_t ast = ptx::sdesc_add(a_desc0, stage * kABytes);
          const uint64_t bst = ptx::sdesc_add(b_desc0, stage * kBBytes);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            ptx::mma_bf16(d_tmem, ptx::sdesc_add(ast, kk * (kWMN ? 16 * 128 : 32)),
                          ptx::sdesc_add(bst, kk * 32), idesc, (kb | kk) != 0 ? 1u : 0u);
          ptx::mma_commit(ptx::smem_addr(&ctl.empty[stage]));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) ptx::mma_commit(ptx::smem_addr(&ctl.tfull[acc]));
      }
      // every MMA issued by this thread has finished before TMEM is freed
      ptx::mma_commit(ptx::smem_addr(&ctl.drain));
      if (!ptx::mbar_wait(ptx::smem_addr(&ctl.drain), 0, nullptr, kWaitLimitNs))
        record_error(err, kErrGemmDrain);
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lane quadrant = this warp's 32 features
    uint8_t *stg = sStage + q * kStageBytesPerWarp;
    // the 16-byte piece (row tr, part) this lane moves in step `it` of a
    // row copy: 8 rows of 64 B per step, 4 steps per 32-token chunk
    const int pr = lane >> 2, pp = lane & 3;
    int it = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
      const TileCoord tc = tile_coord(ctl, G, nf, t);
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      if (!ptx::mbar_wait(ptx::smem_addr(&ctl.tfull[acc]), acc_phase, abort, kWaitLimitNs)) {
        record_error(err, kErrGemmEpilogue | uint32_t(t & 0xffffff));
        *abort = 1;
        break;
      }
      ptx::tc_fence_after();
      const int f0 = tc.ft * kFeat + q * 32;  // first feature of this warp
      const int f = f0 + lane;
      float bv = 0.0f;
      if (bias && f < N) bv = __bfloat162float(bias[int64_t(tc.g) * N + f]);
      const int64_t tok0 = int64_t(tc.row0) + int64_t(tc.tt) * kTok;
      const uint32_t tbase = tmem_base + (uint32_t(q * 32) << 16) + uint32_t(acc * kTok);
      const int nchunk = (tc.ntok + 31) >> 5;
#pragma unroll 1
      for (int c = 0; c < nchunk; ++c) {
        uint32_t raw[32];
        ptx::tmem_ld32(tbase + uint32_t(c * 32), raw);
        ptx::tmem_ld_wait();
        const int ntk = tc.ntok - c * 32 < 32 ? tc.ntok - c * 32 : 32;
        const int64_t trow0 = tok0 + c * 32;
        float x[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(raw[i]) + bv;
        if (grad_src) {
          // act'(grad_src) for this warp's 32 x 32 block, rows in through the stage
#pragma unroll
          for (int s4 = 0; s4 < 4; ++s4) {
            const int tr = s4 * 8 + pr, fc = f0 + pp * 8;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (tr < ntk && fc < N)
              v = *reinterpret_cast<const uint4 *>(grad_src + (trow0 + tr) * N + fc);
            *reinterpret_cast<uint4 *>(stg + tr * 64 + pp * 16) = v;
          }
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float z = __bfloat162float(
                *reinterpret_cast<const __nv_bfloat16 *>(stg + i * 64 + lane * 2));
            x[i] *= act_grad_fast(z, dact);
          }
          __syncwarp();
        }
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
          __nv_bfloat16 *dst = pass == 0 ? pre : C;
          if (pass == 1 && act >= 0) {
#pragma unroll
            for (int i = 0; i < 32; ++i) x[i] = act_fwd_fast(x[i], act);
          }
          if (dst == nullptr) continue;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            *reinterpret_cast<__nv_bfloat16 *>(stg + i * 64 + lane * 2) = __float2bfloat16_rn(x[i]);
          __syncwarp();
#pragma unroll
          for (int s4 = 0; s4 < 4; ++s4) {
            const int tr = s4 * 8 + pr, fc = f0 + pp * 8;
            if (tr < ntk && fc < N)
              *reinterpret_cast<uint4 *>(dst + (trow0 + tr) * N + fc) =
                  *reinterpret_cast<const uint4 *>(stg + tr * 64 + pp * 16);
          }
          __syncwarp();
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_addr(&ctl.tempty[acc]));
    }
  }

  // ------------------------------------------------------------- teardown
  ptx::tc_fence_before();
  block_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------ CTA-pair grouped GEMM
// The same GEMM with tcgen05.mma.cta_group::2: a 2-CTA cluster computes a
// 256-feature x (up to) 256-token tile as one M=256 MMA.  Each CTA loads
// its own 128 weight rows and half of the token rows, so per K slice an SM
// takes in 32 KB and its tensor core reads 8 KB of shared memory per MMA
// instead of 12 KB: with one CTA per SM the 128 x 256 tile needs more
// shared-memory bandwidth than the SM has, the pair does not.
//   both CTAs   warp 0: TMA loads of this CTA's halves, completion counted
//               on the even CTA's `full` barrier; warps 2..9: epilogue of
//               this CTA's 128 features (its own TMEM), release of the
//               accumulator on the even CTA's `tempty` barrier
//   even CTA    warp 1: the pair's MMAs; commits are multicast to the
//               `empty` / `tfull` barriers of both CTAs
// TMEM is allocated and freed by warp 1 of both CTAs together.
//
// Gather form (kGather, the W1 GEMM of the forward with the dispatch fused
// in, MoE explainer §3.1: dispatch, compute and combine in one pass without
// the flattened copy): the token operand is not read from an expert-major
// copy x_disp but straight from the token matrix x, row r of the group
// being token row_src[r] / k.  Four more warps per CTA gather this CTA's
// half of the token tile with 16-byte cp.async copies into the same
// 128-byte-swizzled layout the TMA would write (rows past the group are
// zero), wait for them, fence them for the tensor cores and arrive on the
// even CTA's `full` barrier, which then counts the weight bytes of both
// CTAs' TMA loads and the gather warps of both CTAs.
constexpr int kPairKH = 2;                  // 64-wide K halves per stage
constexpr int kPairBK = 64 * kPairKH;       // K per stage
constexpr int kPairStages = 6 / kPairKH;
constexpr uint32_t kHalfBytes = 128 * 64 * 2;           // 128 rows x 64 K, 16 KB
constexpr uint32_t kPairABytes = kPairKH * kHalfBytes;  // this CTA's 128 weight rows
constexpr uint32_t kPairBBytes = kPairKH * kHalfBytes;  // this CTA's half of the tokens
constexpr uint16_t kPairMask = 0x3;

struct __align__(8) PairCtl {
  uint64_t full[kPairStages];
  uint64_t empty[kPairStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int tile_start[kMaxGroups + 1];  // prefix of (token tiles x 256-feature tiles)
  int row_start[kMaxGroups + 1];   // the expert offsets, read once from global memory
};
// 3 warps per TMEM lane quadrant take every third 32-token chunk, so the
// epilogue (bias, activation, one or two stored outputs, or act' for the
// data gradient) keeps up with tiles whose K loop is short (d = 512 or
// 1024); the gather form keeps 2 per quadrant (its gather warps take the
// rest of the register file)
constexpr int kPairGatherWarps = 4;
__host__ __device__ constexpr int pair_epi_warps(bool gather) { return gather ? 8 : 12; }
__host__ __device__ constexpr int pair_threads(bool gather) {
  return 32 * (2 + pair_epi_warps(gather) + (gather ? kPairGatherWarps : 0));
}
constexpr size_t pair_smem_bytes(bool gather) {
  return 1024 + kPairStages * (kPairABytes + kPairBBytes) +
         pair_epi_warps(gather) * kStageBytesPerWarp + sizeof(PairCtl);
}

template <bool kWMN, bool kGather>
__global__ void __launch_bounds__(pair_threads(kGather), 1)
tc_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmW,
                    const __grid_constant__ CUtensorMap tmX,
                    const int32_t *__restrict__ offsets, int64_t dense_rows, int G, int N,
                    int K,
                    const __nv_bfloat16 *__restrict__ bias, int act,
                    __nv_bfloat16 *__restrict__ C, __nv_bfloat16 *__restrict__ pre,
                    const __nv_bfloat16 *__restrict__ grad_src, int dact, unsigned int *err,
                    const __nv_bfloat16 *__restrict__ xg, const int32_t *__restrict__ row_src,
                    int kch, int b_wrap, float *__restrict__ c_f32,
                    float *__restrict__ col_part) {
  griddep_begin();
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint8_t *sA = smem;
  uint8_t *sB = smem + kPairStages * kPairABytes;
  uint8_t *sStage = smem + kPairStages * (kPairABytes + kPairBBytes);
  constexpr int kEpi = pair_epi_warps(kGather), kSub = kEpi / 4;
  PairCtl &ctl = *reinterpret_cast<PairCtl *>(sStage + kEpi * kStageBytesPerWarp);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const int cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;
  const int nf = (N + 2 * kFeat - 1) / (2 * kFeat);
  const int nk = (K + kPairBK - 1) / kPairBK;

  // ---------------------------------------------------------------- setup
  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      // the producer's arrive (+ the gather warps of both CTAs)
      ptx::mbar_init(ptx::smem_addr(&ctl.full[s]), kGather ? 1 + 2 * kPairGatherWarps : 1);
      ptx::mbar_init(ptx::smem_addr(&ctl.empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(ptx::smem_addr(&ctl.tfull[a]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl.tempty[a]), 2 * kEpi);  // both CTAs
    }
    ptx::mbar_init(ptx::smem_addr(&ctl.drain), 1);
    ctl.abort = 0;
    tile_plan(ctl, G, nf, offsets, dense_rows);
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&tmW);
    ptx::tma_prefetch_desc(&tmX);
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_addr(&ctl.tmem_base), kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  block_sync();
  ptx::cluster_sync();  // both CTAs' barriers exist before any cross-CTA signal
  ptx::tc_fence_after();
  const uint32_t tmem_base = ctl.tmem_base;
  const int total = tile_total(ctl, G);
  volatile int *abort = &ctl.abort;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_phase = 0;
      bool ok = true;
      for (int t = cid; t < total && ok; t += ncl) {
        const TileCoord tc = tile_coord(ctl, G, nf, t);
        const int half = ((tc.ntok + 15) & ~15) >> 1;  // token rows per CTA in the MMA
        const int xrow = tc.row0 + tc.tt * kTok + int(rank) * half;
        const int frow = tc.ft * 2 * kFeat + int(rank) * kFeat;
        for (int kb = 0; kb < nk; ++kb) {
          if (!ptx::mbar_wait_cluster(ptx::smem_addr(&ctl.empty[stage]), phase ^ 1u, abort,
                                      kWaitLimitNs)) {
            record_error(err, kErrGemmProducer | uint32_t(t & 0xffffff));
            *abort = 1;
            ok = false;
            break;
          }
          const uint32_t fb_local = ptx::smem_addr(&ctl.full[stage]);
          const uint32_t fb = ptx::mapa_shared(fb_local, 0);
          if (rank == 0)
            ptx::mbar_arrive_expect_tx(fb_local,
                                       kGather ? 2 * kPairABytes : 2 * (kPairABytes + kPairBBytes));
#pragma unroll
          for (int h = 0; h < kPairKH; ++h) {
            const int k0 = kb * kPairBK + h * 64;
            uint8_t *a = sA + stage * kPairABytes + h * kHalfBytes;
            if (!kWMN) {
              ptx::tma_load_2d_pair(ptx::smem_addr(a), &tmW, fb, k0, tc.g * N + frow);
            } else {
              // the router form repeats B's rows every b_wrap (a multiple of 64)
              const int wrow = b_wrap ? k0 % b_wrap : tc.g * K + k0;
#pragma unroll
              for (int j = 0; j < kFeat / 64; ++j)
                ptx::tma_load_2d_pair(ptx::smem_addr(a + j * (64 * 128)), &tmW, fb, frow + j * 64,
                                      wrow);
            }
            if (!kGather)
              ptx::tma_load_2d_pair(ptx::smem_addr(sB + stage * kPairBBytes + h * kHalfBytes),
                                    &tmX, fb, k0, xrow);
          }
          armed |= 1u << stage;
          armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == kPairStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // every stage filled here is released by the pair's MMAs (and their
      // arrivals on this CTA's barriers have landed) before the CTA moves on
      for (int s = 0; s < kPairStages; ++s)
        if (armed & (1u << s))
          ptx::mbar_wait_cluster(ptx::smem_addr(&ctl.empty[s]), (armed_phase >> s) & 1u,
                                 ok ? nullptr : abort, ok ? kWaitLimitNs : kWaitLimitNs / 4);
    }
  } else if (warp == 1) {
    // -------------------------------------------- MMA issuer (even CTA)
    if (lane == 0 && rank == 0) {
      const uint64_t a_desc0 = kWMN ? ptx::sdesc_sw128(ptx::smem_addr(sA), BK * 128, 1024)
                                    : ptx::sdesc_sw128(ptx::smem_addr(sA), 16, 1024);
      const uint64_t b_desc0 = ptx::sdesc_sw128(ptx::smem_addr(sB), 16, 1024);
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int t = cid; t < total && ok; t += ncl, ++it) {
        const TileCoord tc = tile_coord(ctl, G, nf, t);
        const uint32_t idesc =
            ptx::idesc_bf16(2 * kFeat, (tc.ntok + 15) & ~15, kWMN ? 1 : 0, 0);
        const int acc = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        if (!ptx::mbar_wait_cluster(ptx::smem_addr(&ctl.tempty[acc]), acc_phase ^ 1u, abort,
                                    kWaitLimitNs)) {
          record_error(err, kErrGemmMma | 0x800000u | uint32_t(t & 0x7fffff));
          *abort = 1;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + uint32_t(acc * kTok);
        for (int kb = 0; kb < nk; ++kb) {
          if (!ptx::mbar_wait_cluster(ptx::smem_addr(&ctl.full[stage]), phase, abort,
                                      kWaitLimitNs)) {
            record_error(err, kErrGemmMma | uint32_t(t & 0x7fffff));
            *abort = 1;
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint64_t ast = ptx::sdesc_add(a_desc0, stage * kPairABytes);
          const uint64_t bst = ptx::sdesc_add(b_desc0, stage * kPairBBytes);
#pragma unroll
          for (int kk = 0; kk < kPairBK / 16; ++kk) {
            const uint32_t h = uint32_t(kk >> 2) * kHalfBytes, w = uint32_t(kk & 3);
            ptx::mma_bf16_pair(d_tmem, ptx::sdesc_add(ast, h + w * (kWMN ? 16 * 128 : 32)),
                               ptx::sdesc_add(bst, h + w * 32), idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          ptx::mma_commit_pair_mc(ptx::smem_addr(&ctl.empty[stage]), kPairMask);
          if (++stage == kPairStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) ptx::mma_commit_pair_mc(ptx::smem_addr(&ctl.tfull[acc]), kPairMask);
      }
      // every pair MMA has finished before either CTA frees TMEM
      ptx::mma_commit_pair(ptx::smem_addr(&ctl.drain));
      if (!ptx::mbar_wait_cluster(ptx::smem_addr(&ctl.drain), 0, nullptr, kWaitLimitNs))
        record_error(err, kErrGemmDrain);
    }
  } else if (kGather && warp >= 2 + kEpi) {
    // ------------------- token rows gathered from x (the fused dispatch)
    // this warp's 32 rows of the CTA's half of the token tile, 4 rows per
    // pass: 8 lanes x 16 bytes = one 64-wide K half of a row
    const int gw = warp - (2 + kEpi);
    const int c16 = lane & 7, rsub = lane >> 3;
    const uint32_t full_leader = ptx::mapa_shared(ptx::smem_addr(&ctl.full[0]), 0);
    // stages whose copies are in flight, oldest first: up to the whole ring,
    // as many as the TMA producer keeps in flight
    int stage = 0, pend_head = 0, npend = 0;
    int pend_q[kPairStages];
    uint32_t phase = 0;
    bool ok = true;
    for (int t = cid; t < total && ok; t += ncl) {
      const TileCoord tc = tile_coord(ctl, G, nf, t);
      const int half = ((tc.ntok + 15) & ~15) >> 1;   // token rows per CTA in the MMA
      const int first = tc.tt * kTok + int(rank) * half;
      const int nvalid = tc.ntok - int(rank) * half;  // rows of the group in this half
      int64_t src[8];                                  // element offset of each row in x
#pragma unroll
      for (int ps = 0; ps < 8; ++ps) {
        const int r = gw * 32 + ps * 4 + rsub;
        src[ps] = (r < half && r < nvalid) ? int64_t(row_src[tc.row0 + first + r] / kch) * K : -1;
      }
      for (int kb = 0; kb < nk; ++kb) {
        bool got = true;
        if (lane == 0)
          got = ptx::mbar_wait_cluster(ptx::smem_addr(&ctl.empty[stage]), phase ^ 1u, abort,
                                       kWaitLimitNs);
        got = __shfl_sync(kFullMask, got ? 1 : 0, 0) != 0;
        if (!got) {
          if (lane == 0) {
            record_error(err, kErrGemmGather | uint32_t(t & 0xffffff));
            *abort = 1;
          }
          ok = false;
          break;
        }
        uint8_t *sb = sB + stage * kPairBBytes;
#pragma unroll
        for (int ps = 0; ps < 8; ++ps) {
          const int r = gw * 32 + ps * 4 + rsub;
          if (r >= half) continue;  // the MMA reads `half` rows of this CTA
#pragma unroll
          for (int h = 0; h < kPairKH; ++h) {
            const int col = kb * kPairBK + h * 64 + c16 * 8;
            const bool in = src[ps] >= 0 && col < K;
            ptx::cp_async_16(
                ptx::smem_addr(sb + h * kHalfBytes + r * 128 + ((c16 ^ (r & 7)) << 4)),
                in ? static_cast<const void *>(xg + src[ps] + col) : static_cast<const void *>(xg),
                in ? 16u : 0u);
          }
        }
        ptx::cp_async_commit();
        pend_q[(pend_head + npend) % kPairStages] = stage;
        if (++npend == kPairStages) {
          // the oldest stage's copies have landed: hand it to the MMA
          ptx::cp_async_wait<kPairStages - 1>();
          ptx::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) ptx::mbar_arrive_remote(full_leader + uint32_t(pend_q[pend_head]) * 8u);
          pend_head = (pend_head + 1) % kPairStages;
          --npend;
        }
        if (++stage == kPairStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    ptx::cp_async_wait<0>();
    ptx::fence_proxy_async_smem();
    __syncwarp();
    for (; npend > 0; --npend) {
      if (lane == 0) ptx::mbar_arrive_remote(full_leader + uint32_t(pend_q[pend_head]) * 8u);
      pend_head = (pend_head + 1) % kPairStages;
    }
  } else if (warp >= 2) {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;             // TMEM lane quadrant = this warp's 32 features
    const int sub = (warp - 2) >> 2;    // this warp takes 32-token chunks sub, sub + kSub, ...
    uint8_t *stg = sStage + (warp - 2) * kStageBytesPerWarp;
    const int pr = lane >> 2, pp = lane & 3;
    int it = 0;
    for (int t = cid; t < total; t += ncl, ++it) {
      const TileCoord tc = tile_coord(ctl, G, nf, t);
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      if (!ptx::mbar_wait_cluster(ptx::smem_addr(&ctl.tfull[acc]), acc_phase, abort,
                                  kWaitLimitNs)) {
        record_error(err, kErrGemmEpilogue | uint32_t(t & 0xffffff));
        *abort = 1;
        break;
      }
      ptx::tc_fence_after();
      const int f0 = tc.ft * 2 * kFeat + int(rank) * kFeat + q * 32;
      const int f = f0 + lane;
      float bv = 0.0f;
      if (bias && f < N) bv = __bfloat162float(bias[int64_t(tc.g) * N + f]);
      const int64_t tok0 = int64_t(tc.row0) + int64_t(tc.tt) * kTok;
      const uint32_t tbase = tmem_base + (uint32_t(q * 32) << 16) + uint32_t(acc * kTok);
      const int nchunk = (tc.ntok + 31) >> 5;
      float colacc = 0.0f;  // data-gradient form: this warp's sum over its tokens
#pragma unroll 1
      for (int c = sub; c < nchunk; c += kSub) {
        uint32_t raw[32];
        ptx::tmem_ld32(tbase + uint32_t(c * 32), raw);
        ptx::tmem_ld_wait();
        const int ntk = tc.ntok - c * 32 < 32 ? tc.ntok - c * 32 : 32;
        const int64_t trow0 = tok0 + c * 32;
        float x[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = __uint_as_float(raw[i]) + bv;
        if (kWMN && c_f32) {
          // router form: the fp32 accumulator, each store one 128-byte
          // segment of a token row (lane = feature)
          if (f < N) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (i < ntk) c_f32[(trow0 + i) * N + f] = x[i];
          }
          continue;
        }
        if (grad_src) {
#pragma unroll
          for (int s4 = 0; s4 < 4; ++s4) {
            const int tr = s4 * 8 + pr, fc = f0 + pp * 8;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (tr < ntk && fc < N)
              v = *reinterpret_cast<const uint4 *>(grad_src + (trow0 + tr) * N + fc);
            *reinterpret_cast<uint4 *>(stg + tr * 64 + pp * 16) = v;
          }
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float z = __bfloat162float(
                *reinterpret_cast<const __nv_bfloat16 *>(stg + i * 64 + lane * 2));
            x[i] *= act_grad_fast(z, dact);
          }
          __syncwarp();
          if (kWMN && col_part) {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (i < ntk) colacc += x[i];
          }
        }
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
          __nv_bfloat16 *dst = pass == 0 ? pre : C;
          if (pass == 1 && act >= 0) {
#pragma unroll
            for (int i = 0; i < 32; ++i) x[i] = act_fwd_fast(x[i], act);
          }
          if (dst == nullptr) continue;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            *reinterpret_cast<__nv_bfloat16 *>(stg + i * 64 + lane * 2) = __float2bfloat16_rn(x[i]);
          __syncwarp();
#pragma unroll
          for (int s4 = 0; s4 < 4; ++s4) {
            const int tr = s4 * 8 + pr, fc = f0 + pp * 8;
            if (tr < ntk && fc < N)
              *reinterpret_cast<uint4 *>(dst + (trow0 + tr) * N + fc) =
                  *reinterpret_cast<const uint4 *>(stg + tr * 64 + pp * 16);
          }
          __syncwarp();
        }
      }
      if (kWMN && col_part && f < N) {
        // the bias gradient's partial of this token tile and warp: one slot
        // per (token tile of the whole layer, warp class, feature)
        const int tt_all = ctl.tile_start[tc.g] / nf + tc.tt;
        col_part[(int64_t(tt_all) * kSub + sub) * N + f] = colacc;
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_remote(ptx::mapa_shared(ptx::smem_addr(&ctl.tempty[acc]), 0));
    }
  }

  // ------------------------------------------------------------- teardown
  ptx::tc_fence_before();
  block_sync();
  ptx::cluster_sync();  // the pair's MMAs, epilogues and remote arrivals are done
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

// ------------------------------------------------ K-grouped weight gradient
// C_g[m, n] = sum over rows r of group g of A[r, m] * B[r, n]: the expert
// weight gradients dW2_e = dO_e^T h_e and dW1_e = dh_pre_e^T x_disp_e, whose
// reduction runs over the expert's (variable, possibly zero) token rows.
// Both operands are MN-major in shared memory.  The last K block of a group
// may hold rows of the next group (or unwritten rows past the last group):
// a fixup warp zeroes those rows in shared memory before the MMA reads the
// stage (producer -> full -> fixup -> ready -> MMA); whole K blocks go
// producer -> full -> MMA.
// An expert with no rows gets an exact zero tile without touching TMEM.
// warps: 0 TMA producer, 1 MMA issuer, 2..9 epilogue (2 per TMEM lane
// quadrant, alternate 32-column chunks: a tile's K loop is one expert's
// tokens, short enough that 4 epilogue warps fell behind), 10 fixup
constexpr int kWgEpiWarps = 8;
constexpr int kWgFixupWarp = 2 + kWgEpiWarps;
constexpr int kWgThreads = 32 * (kWgFixupWarp + 1);

struct __align__(8) WgCtl {
  uint64_t full[STAGES];
  uint64_t ready[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
constexpr size_t kWgSmemBytes = 1024 + STAGES * (kABytes + kBBytes) + sizeof(WgCtl);

__device__ __forceinline__ void wg_tile(int t, int mt, int nt, int &g, int &m, int &n) {
  const int per = mt * nt;
  g = t / per;
  const int l = t - g * per;
  n = l / mt;
  m = l - n * mt;
}

// rows [r0, r0 + rows) of group g: from the offsets, or uniform chunks of
// `chunk` rows of rows_total when there are none
__device__ __forceinline__ void wg_group(const int32_t *offsets, int chunk, int64_t rows_total,
                                         int g, int &r0, int &rows) {
  if (offsets) {
    r0 = offsets[g];
    rows = offsets[g + 1] - r0;
  } else {
    const int64_t a = min(int64_t(g) * chunk, rows_total);
    const int64_t b = min(a + chunk, rows_total);
    r0 = int(a);
    rows = int(b - a);
  }
}

__global__ void __launch_bounds__(kWgThreads, 1)
tc_wgrad_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const int32_t *__restrict__ offsets, int G, int M, int N,
                __nv_bfloat16 *__restrict__ C, unsigned int *err, int chunk, int64_t rows_total,
                float *__restrict__ Cf) {
  griddep_begin();
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint8_t *sA = smem;
  uint8_t *sB = smem + STAGES * kABytes;
  WgCtl &ctl = *reinterpret_cast<WgCtl *>(smem + STAGES * (kABytes + kBBytes));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = (M + BM - 1) / BM, nt = (N + BN - 1) / BN;
  const int total = G * mt * nt;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(ptx::smem_addr(&ctl.full[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl.ready[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl.empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(ptx::smem_addr(&ctl.tfull[a]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl.tempty[a]), 32 * kWgEpiWarps);
    }
    ptx::mbar_init(ptx::smem_addr(&ctl.drain), 1);
    ctl.abort = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 1) {
    ptx::tmem_alloc(ptx::smem_addr(&ctl.tmem_base), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  block_sync();
  ptx::tc_fence_after();
  const uint32_t tmem_base = ctl.tmem_base;
  volatile int *abort = &ctl.abort;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, armed = 0, armed_phase = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
        int g, m, n;
        wg_tile(t, mt, nt, g, m, n);
        int r0, rows;
        wg_group(offsets, chunk, rows_total, g, r0, rows);
        const int nk = (rows + BK - 1) / BK;
        for (int kb = 0; kb < nk; ++kb) {
          if (!ptx::mbar_wait(ptx::smem_addr(&ctl.empty[stage]), phase ^ 1u, abort, kWaitLimitNs)) {
            record_error(err, kErrWgradProducer | uint32_t(t & 0xffffff));
            *abort = 1;
            ok = false;
            break;
          }
          const uint32_t fb = ptx::smem_addr(&ctl.full[stage]);
          ptx::mbar_arrive_expect_tx(fb, kABytes + kBBytes);
          const int row = r0 + kb * BK;
#pragma unroll
          for (int j = 0; j < BM / 64; ++j)
            ptx::tma_load_2d(ptx::smem_addr(sA + stage * kABytes + j * (BK * 128)), &tmA, fb,
                             m * BM + j * 64, row);
#pragma unroll
          for (int j = 0; j < BN / 64; ++j)
            ptx::tma_load_2d(ptx::smem_addr(sB + stage * kBBytes + j * (BK * 128)), &tmB, fb,
                             n * BN + j * 64, row);
          armed |= 1u << stage;
          armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok)
        for (int s = 0; s < STAGES; ++s)
          if (armed & (1u << s))
            ptx::mbar_wait(ptx::smem_addr(&ctl.full[s]), (armed_phase >> s) & 1u, nullptr,
                           kWaitLimitNs / 4);
    }
  } else if (warp == kWgFixupWarp) {
    // ------------------------------------- fixup: zero rows past the group
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < total && ok; t += gridDim.x) {
      int g, m, n;
      wg_tile(t, mt, nt, g, m, n);
      int r0, rows;
      wg_group(offsets, chunk, rows_total, g, r0, rows);
      const int nk = (rows + BK - 1) / BK;
      for (int kb = 0; kb < nk; ++kb) {
        if (rows - kb * BK >= BK) {  // a whole K block: the MMA takes it directly
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
          continue;
        }
        bool got = true;
        if (lane == 0)
          got = ptx::mbar_wait(ptx::smem_addr(&ctl.full[stage]), phase, abort, kWaitLimitNs);
        got = __shfl_sync(kFullMask, got ? 1 : 0, 0) != 0;
        if (!got) {
          if (lane == 0) {
            record_error(err, kErrWgradFixup | uint32_t(t & 0xffffff));
            *abort = 1;
          }
          ok = false;
          break;
        }
        const int valid = rows - kb * BK;
        if (valid < BK) {
          const int nbytes = (BK - valid) * 128;  // contiguous tail of each 64-row box
          const uint4 z = make_uint4(0, 0, 0, 0);
          for (int box = 0; box < BM / 64 + BN / 64; ++box) {
            uint8_t *base = box < BM / 64
                                ? sA + stage * kABytes + box * (BK * 128)
                                : sB + stage * kBBytes + (box - BM / 64) * (BK * 128);
            for (int i = lane * 16; i < nbytes; i += 32 * 16)
              *reinterpret_cast<uint4 *>(base + valid * 128 + i) = z;
          }
          ptx::fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_addr(&ctl.ready[stage]));
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint64_t a_desc0 = ptx::sdesc_sw128(ptx::smem_addr(sA), BK * 128, 1024);
      const uint64_t b_desc0 = ptx::sdesc_sw128(ptx::smem_addr(sB), BK * 128, 1024);
      int stage = 0, it = 0;
      uint32_t phase = 0, ready_ph = 0;  // ready completes only on the blocks the fixup takes
      bool ok = true;
      for (int t = blockIdx.x; t < total && ok; t += gridDim.x, ++it) {
        int g, m, n;
        wg_tile(t, mt, nt, g, m, n);
        int r0, rows;
        wg_group(offsets, chunk, rows_total, g, r0, rows);
        const int nk = (rows + BK - 1) / BK;
        // N of the MMA: the tile's columns rounded up to a 64-wide swizzle atom
        const int ncols = min(BN, (min(BN, N - n * BN) + 63) & ~63);
        const uint32_t idesc = ptx::idesc_bf16(BM, ncols, 1, 1);
        const int acc = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        if (!ptx::mbar_wait(ptx::smem_addr(&ctl.tempty[acc]), acc_phase ^ 1u, abort, kWaitLimitNs)) {
          record_error(err, kErrWgradMma | 0x800000u | uint32_t(t & 0x7fffff));
          *abort = 1;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + uint32_t(acc * BN);
        for (int kb = 0; kb < nk; ++kb) {
          const bool whole = rows - kb * BK >= BK;
          const uint32_t bar = ptx::smem_addr(whole ? &ctl.full[stage] : &ctl.ready[stage]);
          const uint32_t par = whole ? phase : (ready_ph >> stage) & 1u;
          if (!whole) ready_ph ^= 1u << stage;
          if (!ptx::mbar_wait(bar, par, abort, kWaitLimitNs)) {
            record_error(err, kErrWgradMma | uint32_t(t & 0x7fffff));
            *abort = 1;
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint64_t ast = ptx::sdesc_add(a_desc0, stage * kABytes);
          const uint64_t bst = ptx::sdesc_add(b_desc0, stage * kBBytes);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            ptx::mma_bf16(d_tmem, ptx::sdesc_add(ast, kk * 16 * 128),
                          ptx::sdesc_add(bst, kk * 16 * 128), idesc, (kb | kk) != 0 ? 1u : 0u);
          ptx::mma_commit(ptx::smem_addr(&ctl.empty[stage]));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) ptx::mma_commit(ptx::smem_addr(&ctl.tfull[acc]));
      }
      ptx::mma_commit(ptx::smem_addr(&ctl.drain));
      if (!ptx::mbar_wait(ptx::smem_addr(&ctl.drain), 0, nullptr, kWaitLimitNs))
        record_error(err, kErrGemmDrain);
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;             // TMEM lane quadrant
    const int half = (warp - 2) >> 2;   // which alternate 32-column chunks
    const int r_in_tile = q * 32 + lane;
    int it = 0;
    for (int t = blockIdx.x; t < total; t += gridDim.x, ++it) {
      int g, m, n;
      wg_tile(t, mt, nt, g, m, n);
      int r0, rows;
      wg_group(offsets, chunk, rows_total, g, r0, rows);
      const bool empty_group = rows == 0;
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      if (!ptx::mbar_wait(ptx::smem_addr(&ctl.tfull[acc]), acc_phase, abort, kWaitLimitNs)) {
        record_error(err, kErrWgradEpilogue | uint32_t(t & 0xffffff));
        *abort = 1;
        break;
      }
      ptx::tc_fence_after();
      const int row = m * BM + r_in_tile;
      const bool valid = row < M;
      __nv_bfloat16 *crow = C + (int64_t(g) * M + row) * N;
      float *crow_f = Cf + (int64_t(g) * M + row) * N;
      const uint32_t tbase = tmem_base + (uint32_t(q * 32) << 16) + uint32_t(acc * BN);
#pragma unroll 1
      for (int c = half; c < BN / 32; c += 2) {
        uint32_t raw[32];
        if (!empty_group) {
          ptx::tmem_ld32(tbase + uint32_t(c * 32), raw);
          ptx::tmem_ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) raw[i] = 0u;
        }
        const int n0 = n * BN + c * 32;
        if (!valid || n0 >= N) continue;
#pragma unroll
        for (int v8 = 0; v8 < 4; ++v8) {
          const int col = n0 + v8 * 8;
          if (col >= N) break;
          float x[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) x[i] = __uint_as_float(raw[v8 * 8 + i]);
          if (Cf) {
            *reinterpret_cast<float4 *>(crow_f + col) = make_float4(x[0], x[1], x[2], x[3]);
            *reinterpret_cast<float4 *>(crow_f + col + 4) = make_float4(x[4], x[5], x[6], x[7]);
          } else {
            *reinterpret_cast<uint4 *>(crow + col) = pack_bf16x8(x);
          }
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(ptx::smem_addr(&ctl.tempty[acc]));
    }
  }

  ptx::tc_fence_before();
  block_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, kTmemCols);
  }
}

// --------------------------------------- K-grouped weight gradient, CTA pairs
// The same K-grouped product with tcgen05.mma.cta_group::2: a 2-CTA cluster
// computes a 256 (M) x 256 (N) tile of C_g.  Each CTA loads its own 128
// columns of A (the M half whose rows of D live in its TMEM) and 128 of the
// 256 columns of B (tcgen05 splits B's N between the pair), 128 K rows per
// stage: 64 KB per CTA per stage instead of the 96 KB that a single-CTA
// 128 x 256 tile needs for the same work.
// A stage takes one of two paths:
//   direct  (no column sums): both CTAs' TMA copies complete on the even
//           CTA's `full` barrier, which the MMA waits on -- the forward pair
//           GEMM's path.  A group's last, partial K block is direct too when
//           the launch has per-group tensor maps (the operands' maps cut to
//           the group's end row, written on the device by
//           wgrad_group_maps_kernel): TMA reads the rows past the group as
//           zeros, where they would otherwise hold the next group's rows or
//           unwritten memory;
//   relayed (any K block of a first-N tile, whose A columns also give the
//           bias gradient db_g = sum over rows of A, and without per-group
//           maps the partial last block): each CTA's copies complete on its
//           own `tail` barrier; its 4 relay warps zero the rows past the
//           group unless TMA did (each a quarter of the rows), add A's valid
//           rows column by column (each a quarter of the columns), fence the
//           stage for the tensor cores if they wrote to it, and arrive on
//           the even CTA's `ready` barrier, which the MMA waits on.
// Both CTAs walk the same tiles and K blocks, so every role agrees on each
// stage's path; the phase of each barrier kind is tracked per stage.
//   both CTAs  warp 0: TMA producer; warps 10..13: the relay; warps 2..9:
//              epilogue of this CTA's 128 rows of the tile
//   even CTA   warp 1: the pair MMAs; commits are multicast to both CTAs'
//              `empty` / `tfull` barriers.
constexpr int kWpBK = 128;                   // K rows per stage (two 64-row halves)
constexpr int kWpStages = 3;
constexpr uint32_t kWpBoxBytes = 64 * 64 * 2;               // 64 cols x 64 rows, 8 KB
constexpr uint32_t kWpOpBytes = 4 * kWpBoxBytes;            // one operand half per stage, 32 KB
constexpr int kWpEpiWarps = 8;
constexpr int kWpFixupWarp = 2 + kWpEpiWarps;  // the first relay warp
constexpr int kWpRelayWarps = 4;
constexpr int kWpThreads = 32 * (kWpFixupWarp + kWpRelayWarps);

struct __align__(8) WpCtl {
  uint64_t full[kWpStages];    // even CTA: direct stages, both CTAs' bytes
  uint64_t tail[kWpStages];    // each CTA: relayed stages, its own bytes
  uint64_t ready[kWpStages];   // even CTA: relayed stages, both relays
  uint64_t empty[kWpStages];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
// each epilogue warp's bf16 staging tile: 32 rows x 32 columns, 64 B a row
constexpr uint32_t kWpStgBytes = 32 * 64;
constexpr size_t kWpSmemBytes =
    1024 + kWpStages * 2 * kWpOpBytes + kWpEpiWarps * kWpStgBytes + sizeof(WpCtl);

// whether K block kb of a group with `rows` rows goes through the relay:
// a block of a bias-sum tile, or the group's partial last block when there
// are no per-group tensor maps to zero-fill the rows past the group
__device__ __forceinline__ bool wp_relayed(int rows, int kb, bool sum, bool zero_fill) {
  return sum || (!zero_fill && rows - kb * kWpBK < kWpBK);
}

// Per-group tensor maps of the two operands: the launch's maps with the
// outer extent cut to the group's end row, so that TMA fills the rows past
// the group with zeros.  One warp per group; maps[2g] is A's, maps[2g+1] B's.
__global__ void __launch_bounds__(256)
wgrad_group_maps_kernel(const __grid_constant__ CUtensorMap tmA,
                        const __grid_constant__ CUtensorMap tmB,
                        const int32_t *__restrict__ offsets, int G, CUtensorMap *maps) {
  griddep_begin();
  __shared__ __align__(128) uint4 sm[8][2][8];  // per warp: A's and B's 128 bytes
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = blockIdx.x * 8 + warp;
  if (g >= G) return;  // the whole warp
  if (lane < 16) {
    const CUtensorMap *src = lane < 8 ? &tmA : &tmB;
    sm[warp][lane >> 3][lane & 7] = reinterpret_cast<const uint4 *>(src)[lane & 7];
  }
  __syncwarp();
  if (lane == 0) {
    const int end = offsets[g + 1];
    const uint32_t extent = uint32_t(end > 0 ? end : 1);
    ptx::tensormap_set_dim1(ptx::smem_addr(&sm[warp][0][0]), extent);
    ptx::tensormap_set_dim1(ptx::smem_addr(&sm[warp][1][0]), extent);
  }
  __syncwarp();
  ptx::tensormap_publish(&maps[2 * g], ptx::smem_addr(&sm[warp][0][0]));
  ptx::tensormap_publish(&maps[2 * g + 1], ptx::smem_addr(&sm[warp][1][0]));
}

// Stage layout of one operand half: [k half 0: cols 0-63, cols 64-127]
// [k half 1: cols 0-63, cols 64-127], each box 64 K rows of 128 B
// (MN-major, 128-byte swizzle).
__global__ void __launch_bounds__(kWpThreads, 1)
tc_wgrad_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB,
                     const int32_t *__restrict__ offsets, int G, int M, int N,
                     __nv_bfloat16 *__restrict__ C, __nv_bfloat16 *__restrict__ colsum,
                     unsigned int *err, const CUtensorMap *__restrict__ gmaps) {
  griddep_begin();
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint8_t *sA = smem;
  uint8_t *sB = smem + kWpStages * kWpOpBytes;
  uint8_t *sStg = smem + kWpStages * 2 * kWpOpBytes;
  WpCtl &ctl = *reinterpret_cast<WpCtl *>(sStg + kWpEpiWarps * kWpStgBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const int cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;
  const int mt = (M + 255) / 256, nt = (N + 255) / 256;
  const int total = G * mt * nt;
  const bool with_sum = colsum != nullptr;
  const bool zero_fill = gmaps != nullptr;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kWpStages; ++s) {
      ptx::mbar_init(ptx::smem_addr(&ctl.full[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl.tail[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl.ready[s]), 2 * kWpRelayWarps);  // both CTAs' relays
      ptx::mbar_init(ptx::smem_addr(&ctl.empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(ptx::smem_addr(&ctl.tfull[a]), 1);
      ptx::mbar_init(ptx::smem_addr(&ctl.tempty[a]), 2 * kWpEpiWarps);  // both CTAs
    }
    ptx::mbar_init(ptx::smem_addr(&ctl.drain), 1);
    ctl.abort = 0;
    ptx::fence_mbar_init();
    ptx::fence_proxy_async_smem();
  }
  if (warp == 0 && lane == 0) {
    ptx::tma_prefetch_desc(&tmA);
    ptx::tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(ptx::smem_addr(&ctl.tmem_base), kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  block_sync();
  ptx::cluster_sync();  // both CTAs' barriers exist before any cross-CTA signal
  ptx::tc_fence_after();
  const uint32_t tmem_base = ctl.tmem_base;
  volatile int *abort = &ctl.abort;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      uint32_t tail_armed = 0, tail_ph = 0;  // relayed fills not yet seen land here
      bool ok = true;
      const uint32_t full_leader = ptx::mapa_shared(ptx::smem_addr(&ctl.full[0]), 0);
      for (int t = cid; t < total && ok; t += ncl) {
        int g, m, n;
        wg_tile(t, mt, nt, g, m, n);
        const int r0 = offsets[g], rows = offsets[g + 1] - r0;
        const int nk = (rows + kWpBK - 1) / kWpBK;
        const bool sum = with_sum && n == 0;
        const int acol = m * 256 + int(rank) * 128, bcol = n * 256 + int(rank) * 128;
        for (int kb = 0; kb < nk; ++kb) {
          if (!ptx::mbar_wait_cluster(ptx::smem_addr(&ctl.empty[stage]), phase ^ 1u, abort,
                                      kWaitLimitNs)) {
            record_error(err, kErrWgradProducer | uint32_t(t & 0xffffff));
            *abort = 1;
            ok = false;
            break;
          }
          const int row = r0 + kb * kWpBK;
          // the group's partial last block through the group's own maps
          // (rows past the group read as zero), the others through the launch's
          const bool part = rows - kb * kWpBK < kWpBK;
          const CUtensorMap *ma = &tmA, *mb = &tmB;
          if (zero_fill && part) {
            ma = gmaps + 2 * g;
            mb = ma + 1;
            ptx::tensormap_acquire(ma);
            ptx::tensormap_acquire(mb);
          }
          if (wp_relayed(rows, kb, sum, zero_fill)) {
            const uint32_t tb = ptx::smem_addr(&ctl.tail[stage]);
            ptx::mbar_arrive_expect_tx(tb, 2 * kWpOpBytes);
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                const uint32_t off = stage * kWpOpBytes + (h * 2 + j) * kWpBoxBytes;
                ptx::tma_load_2d(ptx::smem_addr(sA + off), ma, tb, acol + j * 64, row + h * 64);
                ptx::tma_load_2d(ptx::smem_addr(sB + off), mb, tb, bcol + j * 64, row + h * 64);
              }
            tail_armed |= 1u << stage;
            tail_ph ^= 1u << stage;
          } else {
            const uint32_t fb = full_leader + uint32_t(stage) * 8u;
            if (rank == 0) ptx::mbar_arrive_expect_tx(ptx::smem_addr(&ctl.full[stage]),
                                                      4 * kWpOpBytes);
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                const uint32_t off = stage * kWpOpBytes + (h * 2 + j) * kWpBoxBytes;
                ptx::tma_load_2d_pair(ptx::smem_addr(sA + off), ma, fb, acol + j * 64,
                                      row + h * 64);
                ptx::tma_load_2d_pair(ptx::smem_addr(sB + off), mb, fb, bcol + j * 64,
                                      row + h * 64);
              }
          }
          if (++stage == kWpStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // relayed copies issued here land before the CTA moves on
        for (int s = 0; s < kWpStages; ++s)
          if (tail_armed & (1u << s))
            ptx::mbar_wait(ptx::smem_addr(&ctl.tail[s]), ((tail_ph >> s) & 1u) ^ 1u, nullptr,
                           kWaitLimitNs / 4);
      }
      // every stage filled here has been read by the pair's MMAs before the
      // CTA moves on: the next fill of each stage would wait for exactly that
      for (int i = 0; i < kWpStages && ok; ++i) {
        ptx::mbar_wait_cluster(ptx::smem_addr(&ctl.empty[stage]), phase ^ 1u, nullptr,
                               kWaitLimitNs);
        if (++stage == kWpStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else if (warp >= kWpFixupWarp) {
    // ------------------------------ the relay of relayed stages (see above)
    const int rw = warp - kWpFixupWarp;
    int stage = 0;
    uint32_t tail_ph = 0;
    bool ok = true;
    const uint32_t ready_leader = ptx::mapa_shared(ptx::smem_addr(&ctl.ready[0]), 0);
    // zeroing: this warp's 32 rows of the 128, in K half zh
    const int zh = rw >> 1, zr0 = (rw & 1) * 32;
    // column sums: this warp's 32 of the CTA's 128 columns of A (box cj),
    // this lane's 4 of them (16-byte chunk cchunk, byte offset csub) over
    // rows 32 * rg .. 32 * rg + 31 of each stage
    const int quad = lane & 7, rg = lane >> 3;
    const int cj = rw >> 1, cchunk = 4 * (rw & 1) + (quad >> 1), csub = (quad & 1) * 8;
    for (int t = cid; t < total && ok; t += ncl) {
      int g, m, n;
      wg_tile(t, mt, nt, g, m, n);
      const int rows = offsets[g + 1] - offsets[g];
      const int nk = (rows + kWpBK - 1) / kWpBK;
      const bool sum = with_sum && n == 0;
      float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      for (int kb = 0; kb < nk; ++kb) {
        const int st = stage;
        if (++stage == kWpStages) stage = 0;
        if (!wp_relayed(rows, kb, sum, zero_fill)) continue;
        bool got = true;
        if (lane == 0)
          got = ptx::mbar_wait(ptx::smem_addr(&ctl.tail[st]), (tail_ph >> st) & 1u, abort,
                               kWaitLimitNs);
        tail_ph ^= 1u << st;
        got = __shfl_sync(kFullMask, got ? 1 : 0, 0) != 0;
        if (!got) {
          if (lane == 0) {
            record_error(err, kErrWgradFixup | uint32_t(t & 0xffffff));
            *abort = 1;
          }
          ok = false;
          break;
        }
        const int valid = rows - kb * kWpBK;  // rows of this stage inside the group
        // rows [max(valid, 64 zh + zr0), 64 zh + zr0 + 32) of both operands
        const int vr = max(0, min(32, valid - (64 * zh + zr0)));
        // 0: nothing of this warp's to zero (or TMA filled those rows with zeros)
        const int nbytes = zero_fill ? 0 : (32 - vr) * 128;
        if (nbytes > 0) {
          const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const uint32_t off =
                st * kWpOpBytes + (zh * 2 + j) * kWpBoxBytes + (zr0 + vr) * 128;
            for (int i = lane * 16; i < nbytes; i += 32 * 16) {
              *reinterpret_cast<uint4 *>(sA + off + i) = z;
              *reinterpret_cast<uint4 *>(sB + off + i) = z;
            }
          }
        }
        if (sum) {
          // the valid rows only (the others are being zeroed by the warps
          // that own them), in row order
          const int h = rg >> 1, r0 = (rg & 1) * 32;
          const uint8_t *box = sA + st * kWpOpBytes + (h * 2 + cj) * kWpBoxBytes;
          const int nr = max(0, min(32, valid - 32 * rg));
#pragma unroll 4
          for (int i = 0; i < nr; ++i) {
            const int kr = r0 + i;
            const uint2 v = *reinterpret_cast<const uint2 *>(
                box + kr * 128 + ((cchunk ^ (kr & 7)) << 4) + csub);
            acc[0] += __uint_as_float(v.x << 16);
            acc[1] += __uint_as_float(v.x & 0xffff0000u);
            acc[2] += __uint_as_float(v.y << 16);
            acc[3] += __uint_as_float(v.y & 0xffff0000u);
          }
        }
        // this warp's zeroes (if any) are visible to the MMA's reads; the
        // even CTA's warps arrive on their own barrier directly
        if (nbytes > 0) ptx::fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          if (rank == 0)
            ptx::mbar_arrive(ptx::smem_addr(&ctl.ready[st]));
          else
            ptx::mbar_arrive_remote(ready_leader + uint32_t(st) * 8u);
        }
      }
      if (sum && ok) {
        // the 4 row groups' sums, in row-group order (lanes q, q+8, q+16, q+24)
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const float a1 = __shfl_sync(kFullMask, acc[c], quad + 8);
          const float a2 = __shfl_sync(kFullMask, acc[c], quad + 16);
          const float a3 = __shfl_sync(kFullMask, acc[c], quad + 24);
          const float a0 = __shfl_sync(kFullMask, acc[c], quad);
          acc[c] = ((a0 + a1) + a2) + a3;
        }
        const int col = m * 256 + int(rank) * 128 + cj * 64 + cchunk * 8 + (csub >> 1);
        if (rg == 0) {
#pragma unroll
          for (int c = 0; c < 4; ++c)
            if (col + c < M) colsum[int64_t(g) * M + col + c] = __float2bfloat16_rn(acc[c]);
        }
      }
    }
  } else if (warp == 1) {
    // -------------------------------------------- MMA issuer (even CTA)
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = ptx::idesc_bf16(256, 256, 1, 1);
      const uint64_t a_desc0 = ptx::sdesc_sw128(ptx::smem_addr(sA), kWpBoxBytes, 1024);
      const uint64_t b_desc0 = ptx::sdesc_sw128(ptx::smem_addr(sB), kWpBoxBytes, 1024);
      int stage = 0, it = 0;
      uint32_t phase = 0, full_ph = 0, ready_ph = 0;
      bool ok = true;
      for (int t = cid; t < total && ok; t += ncl, ++it) {
        int g, m, n;
        wg_tile(t, mt, nt, g, m, n);
        const int rows = offsets[g + 1] - offsets[g];
        const int nk = (rows + kWpBK - 1) / kWpBK;
        const bool sum = with_sum && n == 0;
        const int acc = it & 1;
        const uint32_t acc_phase = (it >> 1) & 1;
        if (!ptx::mbar_wait_cluster(ptx::smem_addr(&ctl.tempty[acc]), acc_phase ^ 1u, abort,
                                    kWaitLimitNs)) {
          record_error(err, kErrWgradMma | 0x800000u | uint32_t(t & 0x7fffff));
          *abort = 1;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + uint32_t(acc * 256);
        for (int kb = 0; kb < nk; ++kb) {
          const bool relayed = wp_relayed(rows, kb, sum, zero_fill);
          const uint32_t bar =
              ptx::smem_addr(relayed ? &ctl.ready[stage] : &ctl.full[stage]);
          const uint32_t par = ((relayed ? ready_ph : full_ph) >> stage) & 1u;
          if (relayed)
            ready_ph ^= 1u << stage;
          else
            full_ph ^= 1u << stage;
          if (!ptx::mbar_wait_cluster(bar, par, abort, kWaitLimitNs)) {
            record_error(err, kErrWgradMma | uint32_t(t & 0x7fffff));
            *abort = 1;
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t so = stage * kWpOpBytes;
#pragma unroll
          for (int kk = 0; kk < kWpBK / 16; ++kk) {
            const uint32_t off = so + uint32_t(kk >> 2) * (2 * kWpBoxBytes) + uint32_t(kk & 3) * (16 * 128);
            ptx::mma_bf16_pair(d_tmem, ptx::sdesc_add(a_desc0, off), ptx::sdesc_add(b_desc0, off),
                               idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          ptx::mma_commit_pair_mc(ptx::smem_addr(&ctl.empty[stage]), kPairMask);
          if (++stage == kWpStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) ptx::mma_commit_pair_mc(ptx::smem_addr(&ctl.tfull[acc]), kPairMask);
      }
      ptx::mma_commit_pair(ptx::smem_addr(&ctl.drain));
      if (!ptx::mbar_wait_cluster(ptx::smem_addr(&ctl.drain), 0, nullptr, kWaitLimitNs))
        record_error(err, kErrGemmDrain);
      (void)phase;
    }
  } else if (warp >= 2) {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;             // TMEM lane quadrant
    const int half = (warp - 2) >> 2;   // which alternate 32-column chunks
    const uint32_t tempty_leader = ptx::mapa_shared(ptx::smem_addr(&ctl.tempty[0]), 0);
    // the chunk goes through shared memory so that each store writes 8 rows
    // x 64 contiguous bytes; 16-byte pieces are swizzled by row so that
    // neither side of the transpose has bank conflicts
    uint8_t *stg = sStg + (warp - 2) * kWpStgBytes;
    const int pr = lane >> 2, pp = lane & 3;
    int it = 0;
    for (int t = cid; t < total; t += ncl, ++it) {
      int g, m, n;
      wg_tile(t, mt, nt, g, m, n);
      const bool empty_group = offsets[g + 1] == offsets[g];
      const int acc = it & 1;
      const uint32_t acc_phase = (it >> 1) & 1;
      if (!ptx::mbar_wait_cluster(ptx::smem_addr(&ctl.tfull[acc]), acc_phase, abort,
                                  kWaitLimitNs)) {
        record_error(err, kErrWgradEpilogue | uint32_t(t & 0xffffff));
        *abort = 1;
        break;
      }
      ptx::tc_fence_after();
      const int row0 = m * 256 + int(rank) * 128 + q * 32;  // this warp's first row
      const uint32_t tbase = tmem_base + (uint32_t(q * 32) << 16) + uint32_t(acc * 256);
#pragma unroll 1
      for (int c = half; c < 256 / 32; c += 2) {
        const int n0 = n * 256 + c * 32;
        if (n0 >= N) break;
        uint32_t raw[32];
        if (!empty_group) {
          ptx::tmem_ld32(tbase + uint32_t(c * 32), raw);
          ptx::tmem_ld_wait();
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) raw[i] = 0u;
        }
#pragma unroll
        for (int v8 = 0; v8 < 4; ++v8) {
          float x[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) x[i] = __uint_as_float(raw[v8 * 8 + i]);
          *reinterpret_cast<uint4 *>(stg + lane * 64 + ((v8 ^ ((lane >> 1) & 3)) << 4)) =
              pack_bf16x8(x);
        }
        __syncwarp();
#pragma unroll
        for (int s4 = 0; s4 < 4; ++s4) {
          const int tr = s4 * 8 + pr, row = row0 + tr, col = n0 + pp * 8;
          if (row < M && col < N)
            *reinterpret_cast<uint4 *>(C + (int64_t(g) * M + row) * N + col) =
                *reinterpret_cast<const uint4 *>(stg + tr * 64 + ((pp ^ ((tr >> 1) & 3)) << 4));
        }
        __syncwarp();
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_remote(tempty_leader + uint32_t(acc) * 8u);
    }
  }

  // ------------------------------------------------------------- teardown
  ptx::tc_fence_before();
  block_sync();
  ptx::cluster_sync();  // the pair's MMAs, epilogues and remote arrivals are done
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, kTmemCols);
  }
}

// db[g, n] = sum over the token tiles of group g (in order) and the warp
// classes (in order) of the data-gradient epilogue's partials.
__global__ void __launch_bounds__(256)
bias_grad_reduce_kernel(const float *__restrict__ part, const int32_t *__restrict__ offsets,
                        int N, int nsub, __nv_bfloat16 *__restrict__ db) {
  griddep_begin();
  __shared__ int s_base, s_cnt;
  const int g = blockIdx.y;
  if (threadIdx.x < 32) {  // the token tiles of the groups before g, a lane per group
    int base = 0;
    for (int j = threadIdx.x; j < g; j += 32) base += (offsets[j + 1] - offsets[j] + kTok - 1) / kTok;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) base += __shfl_xor_sync(kFullMask, base, o);
    if (threadIdx.x == 0) {
      s_base = base;
      s_cnt = (offsets[g + 1] - offsets[g] + kTok - 1) / kTok;
    }
  }
  __syncthreads();
  const int n = blockIdx.x * 256 + threadIdx.x;
  if (n >= N) return;
  float acc = 0.0f;
  for (int tt = s_base; tt < s_base + s_cnt; ++tt)
    for (int sb = 0; sb < nsub; ++sb) acc += part[(int64_t(tt) * nsub + sb) * N + n];
  db[int64_t(g) * N + n] = __float2bfloat16_rn(acc);
}

// ----------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(p);
    return static_cast<EncodeTiledFn>(nullptr);
  }();
  return fn;
}

}  // namespace

size_t bias_grad_part_bytes(int64_t max_rows, int G, int N) {
  return size_t((max_rows + kTok - 1) / kTok + G) * (pair_epi_warps(false) / 4) * N * 4;
}

cudaError_t launch_bias_grad_reduce(const float *part, const int32_t *offsets, int G, int N,
                                    void *db, cudaStream_t st) {
  const dim3 grid(unsigned((N + 255) / 256), unsigned(G));
  return launch_k(bias_grad_reduce_kernel, grid, 256, 0, st, part, offsets, N,
                  pair_epi_warps(false) / 4, static_cast<__nv_bfloat16 *>(db));
}


bool make_bf16_map(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer,
                   uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_tc_wgrad(const TcWgrad &g, cudaStream_t st) {
  if (g.G <= 0) return cudaErrorInvalidValue;
  CUtensorMap ta, tb;
  if (!make_bf16_map(&ta, g.A, uint64_t(g.M), uint64_t(g.rows_alloc), 64, BK) ||
      !make_bf16_map(&tb, g.B, uint64_t(g.N), uint64_t(g.rows_alloc), 64, BK))
    return cudaErrorInvalidValue;
  const int sms = num_sms();
  if (sms >= 2 && !g.single) {
    if (g.Cf || !g.offsets) return cudaErrorNotSupported;
    // CTA pairs: 256 x 256 tiles, one M half of A and one N half of B per CTA
    cudaLaunchConfig_t lc = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    lc.blockDim = dim3(kWpThreads);
    lc.dynamicSmemBytes = kWpSmemBytes;
    lc.stream = st;
    lc.attrs = attr;
    lc.numAttrs = 1;
    static PerDevice<int> resident_pairs;
    int npairs = 0;
    cudaError_t e = resident_pairs.get(&npairs, [&](int &v) {
      cudaError_t r = cudaFuncSetAttribute(tc_wgrad_pair_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           int(kWpSmemBytes));
      if (r != cudaSuccess) return r;
      lc.gridDim = dim3(sms & ~1);
      int ncl = 0;
      r = cudaOccupancyMaxActiveClusters(&ncl, tc_wgrad_pair_kernel, &lc);
      if (r != cudaSuccess) return r;
      if (ncl < 1) return cudaErrorInvalidConfiguration;
      v = ncl < sms / 2 ? ncl : sms / 2;
      return cudaSuccess;
    });
    if (e != cudaSuccess) return e;
    const int tiles = g.G * ((g.M + 255) / 256) * ((g.N + 255) / 256);
    lc.gridDim = dim3(2 * (tiles < npairs ? tiles : npairs));
    CUtensorMap *gmaps = static_cast<CUtensorMap *>(g.group_maps);
    if (gmaps) {
      const cudaError_t em = launch_k(wgrad_group_maps_kernel, unsigned((g.G + 7) / 8), 256, 0,
                                      st, ta, tb, g.offsets, g.G, gmaps);
      if (em != cudaSuccess) return em;
    }
    return cudaLaunchKernelEx(&lc, tc_wgrad_pair_kernel, ta, tb, g.offsets, g.G, g.M, g.N,
                              static_cast<__nv_bfloat16 *>(g.C),
                              static_cast<__nv_bfloat16 *>(g.colsum), g.err,
                              static_cast<const CUtensorMap *>(gmaps));
  }
  if (g.colsum) return cudaErrorNotSupported;  // the single-CTA kernel has no column sums
  if (!g.offsets && g.chunk_rows <= 0) return cudaErrorInvalidValue;
  static PerDevice<int> smem_raised;
  int unused = 0;
  if (const cudaError_t e = smem_raised.get(&unused, [](int &) {
        return cudaFuncSetAttribute(tc_wgrad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    int(kWgSmemBytes));
      }); e != cudaSuccess)
    return e;
  const int tiles = g.G * ((g.M + BM - 1) / BM) * ((g.N + BN - 1) / BN);
  const int grid = tiles < num_sms() ? tiles : num_sms();
  return launch_k(tc_wgrad_kernel, grid, kWgThreads, kWgSmemBytes, st, ta, tb, g.offsets, g.G, g.M,
                  g.N, static_cast<__nv_bfloat16 *>(g.C), g.err, g.chunk_rows, g.rows_alloc, g.Cf);
}

cudaError_t launch_tc_gemm(const TcGemm &g, cudaStream_t st) {
  if (g.G <= 0 || g.G > kMaxGroups) return cudaErrorInvalidValue;
  CUtensorMap tw, tx;
  if (!make_bf16_map(&tx, g.A, uint64_t(g.K), uint64_t(g.rows_alloc), BK, kTok))
    return cudaErrorInvalidValue;
  bool okw;
  if (g.b_kmajor)
    okw = make_bf16_map(&tw, g.B, uint64_t(g.K), uint64_t(g.G) * g.N, BK, kFeat);
  else
    okw = make_bf16_map(&tw, g.B, uint64_t(g.N),
                        g.b_wrap ? uint64_t(g.b_rows) : uint64_t(g.G) * g.K, 64, BK);
  if (!okw) return cudaErrorInvalidValue;

  const int sms = num_sms();
  if (sms >= 2) {
    // CTA pairs: this CTA's weight rows (128) and half of the token tile
    CUtensorMap txp;
    if (!make_bf16_map(&txp, g.A, uint64_t(g.K), uint64_t(g.rows_alloc), BK, 128))
      return cudaErrorInvalidValue;
    // 0: weights K-major, 1: weights MN-major (data gradient), 2: the gather
    // form (weights K-major, token rows read from x through row_src)
    const bool gather = g.row_src != nullptr;
    if (gather && !g.b_kmajor) return cudaErrorInvalidValue;
    const int which = gather ? 2 : (g.b_kmajor ? 0 : 1);
    auto kern = gather ? tc_gemm_pair_kernel<false, true>
                       : (g.b_kmajor ? tc_gemm_pair_kernel<false, false>
                                     : tc_gemm_pair_kernel<true, false>);
    cudaLaunchConfig_t lc = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    lc.blockDim = dim3(pair_threads(gather));
    lc.dynamicSmemBytes = pair_smem_bytes(gather);
    lc.stream = st;
    lc.attrs = attr;
    lc.numAttrs = 1;
    // persistent grid: as many pairs as can be resident at once (the
    // shared-memory limit is raised and the occupancy asked once per device)
    static PerDevice<int> resident_pairs[3];
    int npairs = 0;
    const cudaError_t e = resident_pairs[which].get(&npairs, [&](int &v) {
      cudaError_t r = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           int(pair_smem_bytes(gather)));
      if (r != cudaSuccess) return r;
      lc.gridDim = dim3(sms & ~1);
      int ncl = 0;
      r = cudaOccupancyMaxActiveClusters(&ncl, kern, &lc);
      if (r != cudaSuccess) return r;
      if (ncl < 1) return cudaErrorInvalidConfiguration;
      v = ncl < sms / 2 ? ncl : sms / 2;
      return cudaSuccess;
    });
    if (e != cudaSuccess) return e;
    lc.gridDim = dim3(2 * npairs);
    return cudaLaunchKernelEx(&lc, kern, tw, txp, g.offsets, g.rows_alloc, g.G, g.N, g.K,
                              static_cast<const __nv_bfloat16 *>(g.bias), g.act,
                              static_cast<__nv_bfloat16 *>(g.C),
                              static_cast<__nv_bfloat16 *>(g.pre),
                              static_cast<const __nv_bfloat16 *>(g.grad_src), g.dact, g.err,
                              static_cast<const __nv_bfloat16 *>(g.A), g.row_src, g.k_choices,
                              g.b_wrap, g.c_f32, g.col_part);
  }
  if (g.row_src || g.b_wrap || g.c_f32 || g.col_part)
    return cudaErrorNotSupported;  // the gather and router forms need CTA pairs
  static PerDevice<int> smem_raised[2];
  const int which = g.b_kmajor ? 0 : 1;
  auto kern = g.b_kmajor ? tc_gemm_kernel<false> : tc_gemm_kernel<true>;
  int unused = 0;
  if (const cudaError_t e = smem_raised[which].get(&unused, [&](int &) {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    int(kSmemBytes));
      }); e != cudaSuccess)
    return e;
  const int grid = sms;
  return launch_k(kern, grid, kThreads, kSmemBytes, st, tw, tx, g.offsets, g.rows_alloc, g.G,
                  g.N, g.K,
                  static_cast<const __nv_bfloat16 *>(g.bias), g.act,
                  static_cast<__nv_bfloat16 *>(g.C), static_cast<__nv_bfloat16 *>(g.pre),
                  static_cast<const __nv_bfloat16 *>(g.grad_src), g.dact, g.err);
}

}  // namespace moe
