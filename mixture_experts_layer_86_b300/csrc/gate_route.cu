// Single-launch gate for bf16 layers: router GEMM on the tensor cores,
// softmax, top-k, combine weights AND the capacity-limited slot assignment,
// counts, offsets and l_aux, in one kernel.
//
// MoE explainer (lpnh.cn/news/725941) §3.1 Steps 1-2 (router linear layer,
// top-k, softmax over the selected logits); DeepSeek-MoE page
// (lnwmold.com/news/1162317) ch.1 (softmax -> top-2, capacity =
// ceil(S*2/E*cf)); deepspeed.moe overview (adg.csdn.net/694deb285b9f5f31781ae763)
// §2.1 (min_capacity, drop_tokens, gate_loss, expert_count).
//
// The stage is bound by reading x once from HBM.  Every CTA but the last
// takes one tile of TM tokens, TM = ceil(S / (#SMs - 1)) rounded up to 8 rows
// (at most 128), so every SM streams its share of x at the same time; the
// kernel is launched cooperatively (all CTAs resident), one CTA per SM.
//
// Phase A, per tile:
//   warp 0     TMA producer: x tile (TM x 64 per box) and W_g tile
//              (E x 64 per box) K-slices into a shared-memory ring; the
//              first pass over the ring is issued during the setup
//   warp 1     TMEM allocator + MMA issuer: tcgen05.mma M = 128 (rows
//              past TM are zero), N = E rounded up to 16, fp32 in TMEM
//   all warps  epilogue: warp w reads TMEM lane quadrant w % 4 (32 tokens)
//              and every other 32-expert chunk; top-2 with ties to the
//              lower expert index, softmax of logits / T, combine weights;
//              the tile's per-expert probability sums (column sums through
//              a shared-memory transpose, fixed order)
//   warps 4-7  per (choice j, expert e) the tile's count and each token's
//              rank among the tile's tokens with the same (j, e), in token
//              order (__match_any_sync within a warp, warp prefixes across)
//   The tile's counts and probability sums go to the workspace.
// Grid barrier (bounded wait), which the last CTA joins straight away.
// Phase B, every tile CTA for its own tile, in parallel: the counts of all
//   tiles give this tile's prefix (the tiles before it) and the totals;
//   slot = prefix[j][e] + (j == 1 ? first-choice total of e : 0) + rank,
//   dropped at >= capacity.  Every first choice therefore precedes every
//   second choice, each in token order (the GShard priority order of the
//   layer's specification).  Meanwhile the last CTA writes the routed /
//   kept counts, the expert offsets (exclusive scan of kept) and l_aux.
// Everything is deterministic: integer counts, probability sums added in
// a fixed order and then as exact 2^-30 fixed-point integers.
#include <cuda.h>

#include <algorithm>
#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace moe {

// Barrier words of the gate's grid-wide barrier: the number of CTAs that
// have arrived and a generation.  Zero when the module loads; the last CTA
// to arrive resets the count before it bumps the generation, so the words
// are (0, g+1) after every launch.  Launches take the slots in turn, so
// gate launches that overlap on the GPU (different streams) use different
// words as long as fewer than kGateBarrierSlots of them overlap.
struct GridBarrierWords {
  unsigned int count;
  unsigned int gen;
};
constexpr int kGateBarrierSlots = 64;
__device__ GridBarrierWords g_gate_barrier[kGateBarrierSlots];

// Time limit of the waits that follow the kernel's progress (for a copy, an
// MMA, the grid barrier).  2 s unless moe_debug_set_wait_limit changed it to
// exercise the give-up path.  The waits that drain this CTA's own copies and
// MMAs before it exits keep their fixed limit, so no copy or MMA is still in
// flight when the CTA leaves.
__device__ unsigned long long g_gate_wait_limit_ns = 2000000000ull;

namespace {

constexpr int kGrThreads = 256;                 // 8 warps
constexpr int kGrMaxStages = 8;
constexpr int kGrMaxTile = 128;
constexpr uint32_t kXBoxBytes = 128 * 128;      // 128 token rows x 64 bf16; TM rows loaded
constexpr uint32_t kStgFloats = 32 * 33;        // one epilogue warp's transpose tile
constexpr uint64_t kGrWaitNs = 2000000000ull;   // 2 s
constexpr int kGrMaxBoxes = 4;                 // 64-wide K boxes per ring stage, at most
// tile elements (TM x d) from which the rehearsal pays: inside a step it
// made the gate 4 us faster at 56 x 1024 (and is needed at 112 x 2048), 4 us
// slower at 32 x 512, where the tiles finish before it does
constexpr int64_t kRehearseMinTile = 32 * 1024;

struct __align__(16) GrCtl {
  uint64_t full[kGrMaxStages];
  uint64_t empty[kGrMaxStages];
  uint64_t done;
  uint32_t tmem_base;
  int abort;
  int barrier_ok;
  float bias[kMaxExperts];          // the [E] logit bias (zero without one)
  float psum_w[4][kMaxExperts];     // per-warp probability sums of the tile
  int32_t cnt[2][kMaxExperts];      // this tile's count per (j, e)
  int32_t pre[2][kMaxExperts];      // counts of the tiles before this one
  int32_t tot[2][kMaxExperts];      // counts of all tiles
  int32_t offs[kMaxExperts + 1];    // expert offsets
  int32_t choice[2][kGrMaxTile];    // chosen expert per (j, token), -1 none
  int32_t rank[2][kGrMaxTile];      // rank among the tile's (j, e) tokens
  float cand_v[2][kGrMaxTile][2];   // each half's top-2 logits per token
  int32_t cand_i[2][kGrMaxTile][2]; // and their experts
  float zpart[2][kGrMaxTile];       // each half's softmax sum per token
  long long aux[kMaxExperts];       // sum over tokens of p[., e], 2^-30 units
};

struct GrParams {
  int64_t S;
  int d, E, E_pad, k, TM, ntiles, nbox, nstages, nk, nk64;
  uint32_t idesc, tmem_cols, stage_bytes;
  int64_t cap;          // -1: no capacity
  int64_t rows_alloc;   // rows of the expert-major buffers
  const float *logit_bias;
  int bias_ld;          // 0: [E] bias; E: [S,E] bias
  float inv_temp;
  int aux_type;
  float *logits, *probs;
  int32_t *idx;
  float *w;
  int32_t *slot;
  int32_t *routed, *kept, *offsets, *row_src;
  float *l_aux;
  int32_t *hist;        // [ntiles][hist_pitch] counts per (j, e)
  float *psum;          // [ntiles][psum_pitch] probability sums per e
  int32_t *scratch;     // [kMaxExperts + 1]: where the last CTA's rehearsal of phase B writes
  int rehearse;         // nonzero: the last CTA rehearses phase B before the grid barrier
  int hist_pitch, psum_pitch;
  int chunks_per_warp;  // 32-expert chunks each epilogue warp keeps in shared memory
  unsigned int *err;
  unsigned int barrier_slot;
};

__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int *p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Grid-wide barrier; thread 0 of every CTA calls it once, after a block
// barrier.  Returns false when it waited longer than limit_ns (the CTA has
// still arrived, so the words stay consistent for the next launch).
__device__ bool grid_barrier(GridBarrierWords *b, unsigned int nblocks, uint64_t limit_ns) {
  __threadfence();  // this CTA's global writes are visible before it arrives
  const unsigned int gen0 = ld_acquire_gpu(&b->gen);
  const unsigned int t = atomicAdd(&b->count, 1u);
  if (t == nblocks - 1) {
    atomicExch(&b->count, 0u);
    __threadfence();
    atomicAdd(&b->gen, 1u);
    return true;
  }
  const uint64_t t0 = ptx::globaltimer();
  while (ld_acquire_gpu(&b->gen) == gen0) {
    __nanosleep(64);
    if (ptx::globaltimer() - t0 > limit_ns) return false;
  }
  return true;
}

__device__ __forceinline__ void epi_sync() {
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

__device__ __forceinline__ int4 add4(int4 a, int4 b) {
  return make_int4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}
__device__ __forceinline__ int comp4(const int4 &v, int c) {
  return c == 0 ? v.x : c == 1 ? v.y : c == 2 ? v.z : v.w;
}

// the copies of ring stage kb % nstages: nbox K boxes of the tile's x rows
// and of W_g, completing on the stage's `full` barrier
__device__ __forceinline__ void issue_stage(const GrParams &p, const CUtensorMap *tmX,
                                            const CUtensorMap *tmW, uint8_t *ring, GrCtl &ctl,
                                            int kb, int64_t tok0) {
  const int stage = kb % p.nstages;
  const uint32_t wbox_bytes = uint32_t(p.E_pad) * 128;
  const int nb = min(p.nbox, p.nk64 - kb * p.nbox);
  const uint32_t fb = ptx::smem_addr(&ctl.full[stage]);
  uint8_t *st = ring + stage * p.stage_bytes;
  ptx::mbar_arrive_expect_tx(fb, uint32_t(nb) * (uint32_t(p.TM) * 128 + wbox_bytes));
  for (int b = 0; b < nb; ++b) {
    const int k0 = (kb * p.nbox + b) * 64;
    ptx::tma_load_2d(ptx::smem_addr(st + b * kXBoxBytes), tmX, fb, k0, int32_t(tok0));
    ptx::tma_load_2d(ptx::smem_addr(st + p.nbox * kXBoxBytes + b * wbox_bytes), tmW, fb, k0, 0);
  }
}

// Phase B of one CTA (see the header): the prefix of all tiles' counts, the
// offsets, this tile's slots and row map; for the last CTA also the routed /
// kept counts, the offsets and l_aux, written through `o`.  Not inlined: the
// last CTA, which has no tile, runs it once with `o` pointing at scratch
// before it joins the grid barrier, so that the code is in its instruction
// cache when the real pass comes (each SM otherwise fetches this one-shot
// code line by line from L2 or DRAM after the barrier).
struct GrOut {
  int32_t *routed, *kept, *offsets;
  float *l_aux;
};

__device__ __noinline__ void gate_phase_b(const GrParams &p, GrCtl &ctl, uint8_t *ring, int tile,
                                          bool okb, const GrOut o) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tid = threadIdx.x;
  const int64_t tok0 = int64_t(tile) * p.TM;
  const int E = p.E, k = p.k;
  // prefix and totals of the per-tile counts, 4 columns per load
  {
    const int nv = p.hist_pitch >> 2;
    const int RG = max(1, kGrThreads / nv);
    const int v = tid % nv, g = tid / nv;
    int4 pre = make_int4(0, 0, 0, 0), tot = make_int4(0, 0, 0, 0);
    const int4 *h4 = reinterpret_cast<const int4 *>(p.hist);
    if (g < RG && okb) {
      // 8 rows per round, every load issued before any is used: the prefix
      // costs a round trip to L2 per 8 * RG tiles.  Wider rounds are faster
      // with the code cached, but this code runs once per launch and is
      // fetched cold inside a step: 24 rows per round (and 16 for the
      // probability sums below) made the launch 3-6 us slower there.
      constexpr int kU = 8;
      for (int t0 = g; t0 < p.ntiles; t0 += kU * RG) {
        int4 a[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int t = t0 + u * RG;
          a[u] = t < p.ntiles ? __ldcg(h4 + int64_t(t) * nv + v) : make_int4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          tot = add4(tot, a[u]);
          if (t0 + u * RG < tile) pre = add4(pre, a[u]);
        }
      }
    }
    int4 *red = reinterpret_cast<int4 *>(ring);  // [2][RG][nv]
    if (g < RG) {
      red[g * nv + v] = pre;
      red[RG * nv + g * nv + v] = tot;
    }
    block_sync();
    for (int i = tid; i < k * E; i += kGrThreads) {
      const int vi = i >> 2, c = i & 3;
      int P = 0, T = 0;
      for (int gg = 0; gg < RG; ++gg) {
        P += comp4(red[gg * nv + vi], c);
        T += comp4(red[RG * nv + gg * nv + vi], c);
      }
      ctl.pre[i / E][i % E] = P;
      ctl.tot[i / E][i % E] = T;
    }
    block_sync();
  }
  // routed / kept counts and the expert offsets (warp 0; lane l owns a
  // contiguous range of experts)
  if (warp == 0) {
    const int per = (E + 31) / 32;
    const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
    int local = 0;
    for (int e = e0; e < e1; ++e) {
      const int rt = ctl.tot[0][e] + (k == 2 ? ctl.tot[1][e] : 0);
      local += (p.cap < 0 || rt < p.cap) ? rt : int(p.cap);
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(kFullMask, incl, o);
      if (lane >= o) incl += t;
    }
    int run = incl - local;
    for (int e = e0; e < e1; ++e) {
      const int rt = ctl.tot[0][e] + (k == 2 ? ctl.tot[1][e] : 0);
      const int kp = (p.cap < 0 || rt < p.cap) ? rt : int(p.cap);
      // offsets never pass the rows the buffers hold (true by construction
      // when every tile's counts arrived)
      ctl.offs[e] = run < p.rows_alloc ? run : int(p.rows_alloc);
      if (tile == p.ntiles) {
        o.routed[e] = rt;
        o.kept[e] = kp;
        o.offsets[e] = ctl.offs[e];
      }
      run += kp;
    }
    if (lane == 31) {
      ctl.offs[E] = incl < p.rows_alloc ? incl : int(p.rows_alloc);
      if (tile == p.ntiles) o.offsets[E] = ctl.offs[E];
    }
  }
  block_sync();
  // final slots and the row map of this tile's choices
  for (int i = tid; i < p.TM * k; i += kGrThreads) {
    const int r = i / k, j = i - r * k;
    const int64_t s = tok0 + r;
    if (s >= p.S) continue;
    const int e = ctl.choice[j][r];
    int pos = -1;
    if (okb && e >= 0) {
      pos = ctl.pre[j][e] + (j == 1 ? ctl.tot[0][e] : 0) + ctl.rank[j][r];
      if (pos >= ctl.offs[e + 1] - ctl.offs[e]) pos = -1;  // beyond the capacity
    }
    p.slot[s * k + j] = pos;
    if (pos >= 0) p.row_src[ctl.offs[e] + pos] = int32_t(s * k + j);
  }
  // l_aux (the last CTA): probability sums over all tiles, as exact fixed-point
  if (tile == p.ntiles) {
    const int nv = p.psum_pitch >> 2;
    const int RG = max(1, kGrThreads / nv);
    const int v = tid % nv, g = tid / nv;
    long long a[4] = {0, 0, 0, 0};
    const float4 *p4 = reinterpret_cast<const float4 *>(p.psum);
    if (g < RG && okb) {
      constexpr int kU = 4;
      for (int t0 = g; t0 < p.ntiles; t0 += kU * RG) {
        float4 f[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const int t = t0 + u * RG;
          f[u] = t < p.ntiles ? __ldcg(p4 + int64_t(t) * nv + v) : make_float4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          a[0] += fix30_tile(f[u].x);
          a[1] += fix30_tile(f[u].y);
          a[2] += fix30_tile(f[u].z);
          a[3] += fix30_tile(f[u].w);
        }
      }
    }
    // the count reduction above is done with the ring: reuse it
    long long *red = reinterpret_cast<long long *>(ring);  // [RG][psum_pitch]
    if (g < RG)
      for (int c = 0; c < 4; ++c) red[g * p.psum_pitch + v * 4 + c] = a[c];
    block_sync();
    for (int e = tid; e < E; e += kGrThreads) {
      long long t = 0;
      for (int gg = 0; gg < RG; ++gg) t += red[gg * p.psum_pitch + e];
      ctl.aux[e] = t;
    }
    block_sync();
    if (warp == 0) {
      // fp32 from the exact integer sums (no FP64): lane l owns a
      // contiguous range of experts, lanes are added in a fixed tree order
      const int per = (E + 31) / 32;
      const int e0 = min(E, lane * per), e1 = min(E, e0 + per);
      const float S = float(p.S);
      if (p.aux_type == MOE_AUX_STD) {
        // l_aux = std_e(u_e) + 1e-6, u_e = sum_s p[s,e] / S (population std)
        long long sa = 0;
        for (int e = e0; e < e1; ++e) sa += ctl.aux[e];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sa += __shfl_xor_sync(kFullMask, sa, o);
        float sq = 0.0f;
        for (int e = e0; e < e1; ++e) {
          const float dv = usage_deviation(ctl.aux[e], sa, E, p.S);
          sq = fmaf(dv, dv, sq);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(kFullMask, sq, o);
        if (lane == 0) *o.l_aux = okb ? sqrtf(sq / float(E)) + 1e-6f : NAN;
      } else {
        // l_aux = E * sum_e (sum_s p[s,e] / S) * (first[e] / S)
        float aux = 0.0f;
        for (int e = e0; e < e1; ++e)
          aux = fmaf(float(ctl.aux[e]) * kInvFix30, float(ctl.tot[0][e]), aux);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) aux += __shfl_xor_sync(kFullMask, aux, o);
        if (lane == 0) *o.l_aux = okb ? float(E) * aux / S / S : NAN;
      }
    }
  }
}

__global__ void __launch_bounds__(kGrThreads, 1)
gate_route_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                  const __grid_constant__ GrParams p) {
  griddep_begin();
  extern __shared__ uint8_t smem_raw[];
  uint8_t *ring = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  GrCtl &ctl = *reinterpret_cast<GrCtl *>(ring + size_t(p.nstages) * p.stage_bytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tid = threadIdx.x;
  const int tile = blockIdx.x;
  const int64_t tok0 = int64_t(tile) * p.TM;
  const int E = p.E, k = p.k;
  const uint32_t wbox_bytes = uint32_t(p.E_pad) * 128;
  const uint64_t lim = g_gate_wait_limit_ns;

  // Phase A for the tiles; the last CTA has no tile: it only meets the
  // others at the grid barrier and then publishes the counts, the offsets
  // and l_aux while they assign their slots.
  if (tile < p.ntiles) {
    // ---------------------------------------------------------------- setup
    if (tid == 0) {
      for (int s = 0; s < p.nstages; ++s) {
        ptx::mbar_init(ptx::smem_addr(&ctl.full[s]), 1);
        ptx::mbar_init(ptx::smem_addr(&ctl.empty[s]), 1);
      }
      ptx::mbar_init(ptx::smem_addr(&ctl.done), 1);
      ctl.abort = 0;
      ptx::tma_prefetch_desc(&tmX);
      ptx::tma_prefetch_desc(&tmW);
      ptx::fence_mbar_init();
      // the first pass over the ring needs no empty slot: its copies start
      // now, while the other warps set up (they write only the bytes past the
      // TM rows of each x box, which the copies never touch)
      for (int kb = 0; kb < p.nstages; ++kb) issue_stage(p, &tmX, &tmW, ring, ctl, kb, tok0);
    }
    if (warp == 1) {
      ptx::tmem_alloc(ptx::smem_addr(&ctl.tmem_base), p.tmem_cols);
      ptx::tmem_relinquish();
    }
    // the [E] bias, and zeros in the x-box rows past TM that the M = 128 MMA
    // reads (written once; the TMA copies never touch them)
    for (int e = tid; e < kMaxExperts; e += kGrThreads)
      ctl.bias[e] = (p.logit_bias != nullptr && p.bias_ld == 0 && e < E) ? p.logit_bias[e] : 0.0f;
    if (p.TM < kGrMaxTile) {
      const uint32_t pad = (kGrMaxTile - p.TM) * 128;  // bytes past the TM rows of one box
      const uint32_t per_box = pad / 16;
      const uint32_t n = uint32_t(p.nstages * p.nbox) * per_box;
      for (uint32_t i = tid; i < n; i += kGrThreads) {
        const uint32_t box = i / per_box, off = (i - box * per_box) * 16;
        const uint32_t st = box / p.nbox, b = box - st * p.nbox;
        *reinterpret_cast<uint4 *>(ring + st * p.stage_bytes + b * kXBoxBytes + p.TM * 128 + off) =
            make_uint4(0, 0, 0, 0);
      }
      ptx::fence_proxy_async_smem();  // visible to the tensor cores' reads
    }
    ptx::tc_fence_before();
    block_sync();
    ptx::tc_fence_after();
    const uint32_t tmem = ctl.tmem_base;
    volatile int *abort = &ctl.abort;

    // ------------------------------------------------------------ phase A
    if (warp == 0) {
      if (lane == 0) {
        // stages 0 .. nstages-1 were issued during the setup (phase 0)
        uint32_t armed = (1u << p.nstages) - 1u, armed_phase = 0;
        bool ok = true;
        for (int kb = p.nstages; kb < p.nk; ++kb) {
          const int stage = kb % p.nstages;
          const uint32_t phase = (kb / p.nstages) & 1;
          if (!ptx::mbar_wait(ptx::smem_addr(&ctl.empty[stage]), phase ^ 1u, abort, lim)) {
            record_error(p.err, kErrGateProducer | uint32_t(tile & 0xffffff));
            *abort = 1;
            ok = false;
            break;
          }
          issue_stage(p, &tmX, &tmW, ring, ctl, kb, tok0);
          armed |= 1u << stage;
          armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
        }
        if (!ok)  // copies already issued land before the ring is reused
          for (int s = 0; s < p.nstages; ++s)
            if (armed & (1u << s))
              ptx::mbar_wait(ptx::smem_addr(&ctl.full[s]), (armed_phase >> s) & 1u, nullptr,
                             kGrWaitNs / 4);
      }
    } else if (warp == 1) {
      if (lane == 0) {
        const uint64_t desc0 = ptx::sdesc_sw128(ptx::smem_addr(ring), 16, 1024);
        bool ok = true;
        for (int kb = 0; kb < p.nk; ++kb) {
          const int stage = kb % p.nstages;
          const uint32_t phase = (kb / p.nstages) & 1;
          if (!ptx::mbar_wait(ptx::smem_addr(&ctl.full[stage]), phase, abort, lim)) {
            record_error(p.err, kErrGateMma | uint32_t(tile & 0xffffff));
            *abort = 1;
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const int nb = min(p.nbox, p.nk64 - kb * p.nbox);
          const uint64_t sdesc = ptx::sdesc_add(desc0, stage * p.stage_bytes);
          for (int b = 0; b < nb; ++b) {
            const uint64_t ad = ptx::sdesc_add(sdesc, b * kXBoxBytes);
            const uint64_t bd = ptx::sdesc_add(sdesc, p.nbox * kXBoxBytes + b * wbox_bytes);
  #pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              ptx::mma_bf16(tmem, ptx::sdesc_add(ad, kk * 32), ptx::sdesc_add(bd, kk * 32), p.idesc,
                            (kb | b | kk) != 0 ? 1u : 0u);
          }
          ptx::mma_commit(ptx::smem_addr(&ctl.empty[stage]));
        }
        ptx::mma_commit(ptx::smem_addr(&ctl.done));
        // after a give-up, the MMAs already issued finish before TMEM is freed
        if (!ok) ptx::mbar_wait(ptx::smem_addr(&ctl.done), 0, nullptr, kGrWaitNs / 4);
      }
    }

    // ---------------------------------------------- epilogue: all 8 warps
    // Warp w reads TMEM lane quadrant q = w % 4 (tokens 32q .. 32q+31 of the
    // tile) and the expert chunks c = h, h + 2, ... (h = w / 4) of 32 experts
    // each.  Per chunk the logits (+ bias) go to a 32 x 33 shared tile, whose
    // rows are tokens and columns experts, so that logits, then exp(l - m),
    // then probabilities live in the same tile; the two warps of a quadrant
    // merge their top-2 candidates, maxima and sums through shared memory in a
    // fixed order.  The ring is idle once every MMA is done.
    __syncwarp();
    {
      const int q = warp & 3, h = warp >> 2;
      const int r = q * 32 + lane;  // token row of the tile
      const int64_t s = tok0 + r;
      const bool valid = r < p.TM && s < p.S;
      if (!ptx::mbar_wait(ptx::smem_addr(&ctl.done), 0, abort, lim)) {
        record_error(p.err, kErrGateEpilogue | uint32_t(tile & 0xffffff));
        *abort = 1;
      }
      ptx::tc_fence_after();
      const uint32_t trow = tmem + (uint32_t(q * 32) << 16);
      const float *brow = (p.logit_bias != nullptr && p.bias_ld != 0 && valid)
                              ? p.logit_bias + s * p.bias_ld
                              : nullptr;
      const int nchunk = (E + 31) >> 5;
      const int my_chunks = (nchunk - h + 1) >> 1;  // chunks h, h+2, ...
      float *stg0 = reinterpret_cast<float *>(ring) + (warp * p.chunks_per_warp) * kStgFloats;
      const int64_t wrow0 = tok0 + q * 32;  // first token of this warp's rows
      int64_t wr = p.S - wrow0;              // valid rows of this warp (<= 0: none)
      if (wr > p.TM - q * 32) wr = p.TM - q * 32;
      const int wrows = wr > 32 ? 32 : int(wr);

      // pass 1: logits (+ bias) into the shared tiles; top-2 candidates
      float b1 = -INFINITY, b2 = -INFINITY;
      int i1 = -1, i2 = -1;
      for (int ci = 0; ci < my_chunks; ++ci) {
        const int c = h + 2 * ci;
        float *stg = stg0 + ci * kStgFloats;
        uint32_t raw[32];
        ptx::tmem_ld32(trow + uint32_t(c * 32), raw);
        ptx::tmem_ld_wait();
  #pragma unroll
        for (int t = 0; t < 32; ++t) {
          const int e = c * 32 + t;
          if (e < E) {
            const float v = __uint_as_float(raw[t]) + (brow ? brow[e] : ctl.bias[e]);
            if (i1 < 0 || v > b1) {
              b2 = b1;
              i2 = i1;
              b1 = v;
              i1 = e;
            } else if (i2 < 0 || v > b2) {
              b2 = v;
              i2 = e;
            }
            stg[lane * 33 + t] = v;
          }
        }
        if (p.logits) {  // coalesced rows of the logits
          __syncwarp();
          const int e = c * 32 + lane;
          for (int rr = 0; rr < wrows; ++rr)
            if (e < E) p.logits[(wrow0 + rr) * E + e] = stg[rr * 33 + lane];
        }
      }
      ptx::tc_fence_before();
      ctl.cand_v[h][r][0] = b1;
      ctl.cand_v[h][r][1] = b2;
      ctl.cand_i[h][r][0] = i1;
      ctl.cand_i[h][r][1] = i2;
      block_sync();
      // the row's top-2 over both halves: ranked by value, ties to the lower
      // expert index (each half's candidates come in that order already)
      {
        const float ov1 = ctl.cand_v[h ^ 1][r][0], ov2 = ctl.cand_v[h ^ 1][r][1];
        const int oi1 = ctl.cand_i[h ^ 1][r][0], oi2 = ctl.cand_i[h ^ 1][r][1];
        auto before = [](float av, int ai, float bv, int bi) {
          return ai >= 0 && (bi < 0 || av > bv || (av == bv && ai < bi));
        };
        if (before(ov1, oi1, b1, i1)) {
          if (before(b1, i1, ov2, oi2)) {
            b2 = b1;
            i2 = i1;
          } else {
            b2 = ov2;
            i2 = oi2;
          }
          b1 = ov1;
          i1 = oi1;
        } else if (before(ov1, oi1, b2, i2)) {
          b2 = ov1;
          i2 = oi1;
        }
      }
      const float m = b1;  // the top-1 logit is the softmax shift
      // pass 2: exp((l - m) / T) in place; this half's sum.  Passes 2 and 3
      // work on shared memory and are only partly unrolled: the epilogue
      // runs once per launch and is fetched cold inside a step, where the
      // smaller code made the launch ~2 us faster
      float z = 0.0f;
      for (int ci = 0; ci < my_chunks; ++ci) {
        const int c = h + 2 * ci;
        float *stg = stg0 + ci * kStgFloats;
  #pragma unroll 4
        for (int t = 0; t < 32; ++t) {
          if (c * 32 + t < E) {
            const float ev = expf((stg[lane * 33 + t] - m) * p.inv_temp);
            stg[lane * 33 + t] = ev;
            z += ev;
          }
        }
      }
      ctl.zpart[h][r] = z;
      block_sync();
      const float inv_z = 1.0f / (ctl.zpart[0][r] + ctl.zpart[1][r]);
      // pass 3: probabilities (0 past the batch), column sums over the tile's
      // rows in a fixed order, the optional probability rows
      for (int ci = 0; ci < my_chunks; ++ci) {
        const int c = h + 2 * ci;
        float *stg = stg0 + ci * kStgFloats;
  #pragma unroll 8
        for (int t = 0; t < 32; ++t)
          if (c * 32 + t < E) stg[lane * 33 + t] = valid ? stg[lane * 33 + t] * inv_z : 0.0f;
        __syncwarp();
        const int e = c * 32 + lane;
        float cs[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // rows rr = 4 i + u, fixed order
  #pragma unroll 2
        for (int rr = 0; rr < 32; rr += 4) {
  #pragma unroll
          for (int u = 0; u < 4; ++u) cs[u] += stg[(rr + u) * 33 + lane];
        }
        if (e < E) ctl.psum_w[q][e] = (cs[0] + cs[1]) + (cs[2] + cs[3]);
        if (p.probs)
          for (int rr = 0; rr < wrows; ++rr)
            if (e < E) p.probs[(wrow0 + rr) * E + e] = stg[rr * 33 + lane];
        __syncwarp();
      }
      if (h == 0) {
        if (valid) {
          p.idx[s * k] = i1;
          if (k == 1) {
            p.w[s] = inv_z;  // exp(l1 - max) = 1
          } else {
            const float x2 = expf((b2 - m) * p.inv_temp);
            const float den = 1.0f + x2;
            p.w[s * 2] = 1.0f / den;
            p.w[s * 2 + 1] = x2 / den;
            p.idx[s * 2 + 1] = i2;
          }
        }
        ctl.choice[0][r] = valid ? i1 : -1;
        ctl.choice[1][r] = (valid && k == 2) ? i2 : -1;
      }
    }
    block_sync();

    if (warp >= 4) {
      // the tile's count and each token's rank per (j, e), in token order:
      // within a warp by __match_any_sync, across the 4 warps by their counts'
      // prefix; both choices at once, the counts in the ring (idle now)
      const int q = warp & 3;
      const int r = q * 32 + lane;
      const int et = tid - 128;  // 0..127 over warps 4..7
      int32_t *wc = reinterpret_cast<int32_t *>(ring);  // [k][4][E]
      for (int i = et; i < k * 4 * E; i += 128) wc[i] = 0;
      epi_sync();
      int ej[2], rk[2];
  #pragma unroll
      for (int j = 0; j < 2; ++j) {
        ej[j] = j < k ? ctl.choice[j][r] : -1;
        const unsigned peers = __match_any_sync(kFullMask, ej[j]);
        rk[j] = __popc(peers & lanemask_lt());
        if (ej[j] >= 0 && rk[j] == 0) wc[(j * 4 + q) * E + ej[j]] = __popc(peers);
      }
      epi_sync();
      for (int i = et; i < k * E; i += 128) {
        const int j = i / E, ee = i - j * E;
        int run = 0;
        for (int w4 = 0; w4 < 4; ++w4) {
          const int cnum = wc[(j * 4 + w4) * E + ee];
          wc[(j * 4 + w4) * E + ee] = run;
          run += cnum;
        }
        ctl.cnt[j][ee] = run;
      }
      epi_sync();
  #pragma unroll
      for (int j = 0; j < 2; ++j)
        if (j < k) ctl.rank[j][r] = ej[j] >= 0 ? wc[(j * 4 + q) * E + ej[j]] + rk[j] : 0;
    } else {
      // publish the tile's probability sums (padding entries 0)
      for (int e = tid; e < p.psum_pitch; e += 128)
        p.psum[int64_t(tile) * p.psum_pitch + e] =
            e < E ? ((ctl.psum_w[0][e] + ctl.psum_w[1][e]) + ctl.psum_w[2][e]) + ctl.psum_w[3][e]
                  : 0.0f;
    }
    block_sync();
    // publish the tile's counts (padding entries 0)
    for (int i = tid; i < p.hist_pitch; i += kGrThreads)
      p.hist[int64_t(tile) * p.hist_pitch + i] = i < k * E ? ctl.cnt[i / E][i % E] : 0;

    ptx::tc_fence_before();
    block_sync();
    if (warp == 1) {
      ptx::tc_fence_after();
      ptx::tmem_dealloc(tmem, p.tmem_cols);
    }
  }

  // the last CTA: phase B once on scratch outputs while the tiles stream
  // (when their stream is long enough to hide it)
  if (tile == p.ntiles && p.rehearse) {
    const GrOut dry{p.scratch, p.scratch, p.scratch, reinterpret_cast<float *>(p.scratch)};
    gate_phase_b(p, ctl, ring, tile, true, dry);
    block_sync();
  }

  // ------------------------------------------------------- grid barrier
  if (tid == 0) {
    const bool ok = grid_barrier(&g_gate_barrier[p.barrier_slot], unsigned(p.ntiles) + 1u, lim);
    if (!ok) record_error(p.err, kErrGateBarrier | uint32_t(tile & 0xffffff));
    ctl.barrier_ok = ok ? 1 : 0;
  }
  block_sync();
  // Without the barrier some tiles' counts may be missing: every choice of
  // this tile is then dropped and the last CTA reports empty experts.
  const bool okb = ctl.barrier_ok != 0;

  // ------------------------------------------------------------ phase B
  gate_phase_b(p, ctl, ring, tile, okb, GrOut{p.routed, p.kept, p.offsets, p.l_aux});
}

unsigned int next_barrier_slot() {
  static std::atomic<unsigned int> n{0};
  return n.fetch_add(1u, std::memory_order_relaxed) % kGateBarrierSlots;
}

}  // namespace

cudaError_t set_gate_wait_limit(uint64_t ns) {
  const unsigned long long v = ns ? ns : 2000000000ull;
  return cudaMemcpyToSymbol(g_gate_wait_limit_ns, &v, sizeof(v));
}

cudaError_t launch_gate_route(const GateRouteArgs &a, cudaStream_t st) {
  if (a.S <= 0) return cudaErrorNotSupported;
  // one tile per SM but one: that SM runs the CTA that publishes the counts
  const int ntile_max = num_sms() - 1;
  if (ntile_max < 1) return cudaErrorNotSupported;
  int64_t tm = (a.S + ntile_max - 1) / ntile_max;
  tm = (tm + 7) & ~int64_t(7);
  if (tm < 16) tm = 16;
  if (tm > kGrMaxTile) return cudaErrorNotSupported;  // more tokens than one wave of tiles
  GrParams p{};
  p.S = a.S; p.d = a.d; p.E = a.E; p.k = a.k;
  p.TM = int(tm);
  p.ntiles = int((a.S + tm - 1) / tm);
  p.E_pad = (a.E + 15) / 16 * 16;
  uint32_t cols = 32;
  while (int(cols) < p.E_pad) cols <<= 1;
  p.tmem_cols = cols;
  // ring stages of nbox 64-wide K boxes: the widest boxes (each tile row
  // read in longer runs) that still leave two stages in flight
  constexpr size_t kSmemLimit = 232448;
  const size_t fixed = 1024 + sizeof(GrCtl);
  p.nk64 = (a.d + 63) / 64;
  int nst = 0;
  for (int nb = kGrMaxBoxes; nb >= 1; nb >>= 1) {
    p.nbox = nb;
    p.nk = (p.nk64 + nb - 1) / nb;
    p.stage_bytes = uint32_t(nb) * (kXBoxBytes + uint32_t(p.E_pad) * 128);
    nst = int((kSmemLimit - fixed) / p.stage_bytes);
    if (nst > kGrMaxStages) nst = kGrMaxStages;
    if (nst > p.nk) nst = p.nk;
    if (nst >= 2 || (nb == 1 && nst >= 1)) break;
  }
  if (nst < 1) return cudaErrorNotSupported;
  p.nstages = nst;
  p.hist_pitch = (a.k * a.E + 3) & ~3;
  p.psum_pitch = (a.E + 3) & ~3;
  // the ring also holds the epilogue's shared tiles (8 warps, each with
  // its half of the 32-expert chunks) and phase B's reduction scratch
  p.chunks_per_warp = ((a.E + 31) / 32 + 1) / 2;
  size_t ring = size_t(nst) * p.stage_bytes;
  const int rg_aux = std::max(1, kGrThreads / (p.psum_pitch >> 2));
  const size_t need =
      std::max({size_t(8) * p.chunks_per_warp * kStgFloats * 4, size_t(2) * kGrThreads * 16,
                size_t(rg_aux) * p.psum_pitch * 8});
  if (ring < need) return cudaErrorNotSupported;
  const size_t smem = fixed + ring;
  if (smem > kSmemLimit) return cudaErrorNotSupported;
  const size_t ws_need =
      size_t(p.ntiles) * (p.hist_pitch + p.psum_pitch) * 4 + (kMaxExperts + 4) * 4;
  if (ws_need > a.ws_bytes) return cudaErrorNotSupported;
  p.hist = static_cast<int32_t *>(a.ws);
  p.psum = reinterpret_cast<float *>(static_cast<char *>(a.ws) +
                                     size_t(p.ntiles) * p.hist_pitch * 4);
  p.scratch = reinterpret_cast<int32_t *>(p.psum + size_t(p.ntiles) * p.psum_pitch);
  // The rehearsal runs while the tiles stream x and run their epilogue; with
  // tiles much smaller than kRehearseMinTile the last CTA would reach the
  // grid barrier after them.
  p.rehearse = int64_t(p.TM) * a.d >= kRehearseMinTile ? 1 : 0;
  p.idesc = ptx::idesc_bf16(128, p.E_pad, 0, 0);
  p.cap = a.cap;
  p.rows_alloc = a.rows_alloc;
  p.logit_bias = a.logit_bias; p.bias_ld = a.bias_ld; p.inv_temp = a.inv_temp;
  p.aux_type = a.aux_type;
  p.logits = a.logits; p.probs = a.probs; p.idx = a.idx; p.w = a.w; p.slot = a.slot;
  p.routed = a.routed; p.kept = a.kept; p.offsets = a.offsets; p.row_src = a.row_src;
  p.l_aux = a.l_aux; p.err = a.err;
  p.barrier_slot = next_barrier_slot();

  CUtensorMap tx, tw;
  if (!make_bf16_map(&tx, a.x, uint64_t(a.d), uint64_t(a.S), 64, uint32_t(p.TM)))
    return cudaErrorInvalidValue;
  if (!make_bf16_map(&tw, a.w_gate, uint64_t(a.d), uint64_t(a.E), 64, uint32_t(p.E_pad)))
    return cudaErrorInvalidValue;
  static PerDevice<int> smem_raised;
  int unused = 0;
  if (const cudaError_t e = smem_raised.get(&unused, [](int &) {
        return cudaFuncSetAttribute(gate_route_kernel,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, int(kSmemLimit));
      }); e != cudaSuccess)
    return e;
  // cooperative: every CTA resident at once (the grid barrier needs it);
  // programmatic serialization: overlaps the launch with the previous kernel
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(unsigned(p.ntiles) + 1u);  // + the CTA that publishes counts and l_aux
  lc.blockDim = dim3(kGrThreads);
  lc.dynamicSmemBytes = smem;
  lc.stream = st;
  lc.attrs = attr;
  lc.numAttrs = 2;
  cudaError_t e = cudaLaunchKernelEx(&lc, gate_route_kernel, tx, tw, p);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();  // a rejected configuration is not sticky
    lc.numAttrs = 1;
    e = cudaLaunchKernelEx(&lc, gate_route_kernel, tx, tw, p);
  }
  return e;
}

}  // namespace moe
