// CUDA-core grouped GEMM with fp32 accumulation and arbitrary element
// strides.  It is the fp32 path of the layer (tensor cores have no exact
// fp32 mode) and serves the small gate-gradient contraction.  64x64 output
// tile per CTA, 16-deep K slices staged in shared memory, 4x4 outputs per
// thread.
#include "common.cuh"
#include "kernels.h"

namespace moe {
namespace {

constexpr int BM = 64, BN = 64, BK = 16;

__global__ void __launch_bounds__(256) simt_gemm_kernel(SimtGemm g) {
  griddep_begin();
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  __shared__ int s_group, s_row0, s_rows;

  const int tid = threadIdx.x;
  const int tx = tid & 15, ty = tid >> 4;
  const int n0 = blockIdx.y * BN;

  int grp = 0;
  int64_t row0 = 0, rows = 0, kbeg = 0, kend = g.K;
  if (g.mode == 1) {
    // map blockIdx.x to (group, m-tile) through the groups' tile counts
    if (tid == 0) {
      int64_t t = blockIdx.x;
      int found = -1;
      for (int e = 0; e < g.G; ++e) {
        const int64_t a = g.offsets[e], b = g.offsets[e + 1];
        const int64_t nt = (b - a + BM - 1) / BM;
        if (t < nt) {
          found = e;
          s_row0 = int(a + t * BM);
          s_rows = int(min((int64_t)BM, b - (a + t * BM)));
          break;
        }
        t -= nt;
      }
      s_group = found;
    }
    __syncthreads();
    grp = s_group;
    if (grp < 0) return;
    row0 = s_row0;
    rows = s_rows;
  } else if (g.mode == 2) {
    grp = blockIdx.z;
    row0 = int64_t(blockIdx.x) * BM;
    rows = min((int64_t)BM, g.M - row0);
    kbeg = g.offsets[grp];
    kend = g.offsets[grp + 1];
  } else {
    row0 = int64_t(blockIdx.x) * BM;
    rows = min((int64_t)BM, g.M - row0);
  }
  if (rows <= 0) return;

  const int64_t b_base = (g.mode == 1) ? int64_t(grp) * g.b_g : 0;

  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.0f;

  for (int64_t k0 = kbeg; k0 < kend; k0 += BK) {
    // each thread stages 4 A and 4 B elements
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = tid + i * 256;       // 0..1023 over a 64x16 tile
      const int mm = e >> 4, kk = e & 15;
      const int64_t kg = k0 + kk;
      float av = 0.0f, bv = 0.0f;
      if (mm < rows && kg < kend) av = load_elem(g.A, g.a_dtype, (row0 + mm) * g.a_m + kg * g.a_k);
      if (n0 + mm < g.N && kg < kend)
        bv = load_elem(g.B, g.b_dtype, b_base + int64_t(n0 + mm) * g.b_n + kg * g.b_k);
      As[kk][mm] = av;
      Bs[kk][mm] = bv;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = As[kk][ty * 4 + i];
        b[i] = Bs[kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }

  const int64_t c_base = (g.mode == 2) ? int64_t(grp) * g.c_g : 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int mm = ty * 4 + i;
    if (mm >= rows) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= g.N) continue;
      float v = acc[i][j];
      if (g.bias) v += load_elem(g.bias, g.b_dtype, int64_t(grp) * g.bias_g + n);
      if (g.bias_f32) v += g.bias_f32[(row0 + mm) * g.bias_f32_ld + n];
      const int64_t ci = c_base + (row0 + mm) * g.c_m + int64_t(n) * g.c_n;
      if (g.pre) store_elem(g.pre, g.c_dtype, ci, v);
      if (g.act >= 0) v = act_fwd(v, g.act);
      if (g.grad_src) v *= act_grad(load_elem(g.grad_src, g.c_dtype, ci), g.dact);
      store_elem(g.C, g.c_dtype, ci, v);
    }
  }
}

}  // namespace

cudaError_t launch_simt_gemm(const SimtGemm &g, cudaStream_t st) {
  dim3 grid;
  grid.y = (g.N + BN - 1) / BN;
  if (g.mode == 1) {
    grid.x = unsigned((g.max_rows + BM - 1) / BM + g.G);
    grid.z = 1;
  } else {
    grid.x = unsigned((g.M + BM - 1) / BM);
    grid.z = g.mode == 2 ? g.G : 1;
  }
  if (grid.x == 0 || grid.y == 0 || grid.z == 0) return cudaSuccess;
  return launch_k(simt_gemm_kernel, grid, 256, 0, st, g);
}

}  // namespace moe
