// Shared device helpers of the MoE layer library (element access,
// activations, warp reductions).  Internal header.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_b300.h"

namespace moe {

constexpr int kMaxExperts = 256;
constexpr unsigned kFullMask = 0xffffffffu;

// Element load/store with the element type chosen at run time
// (MOE_F32 or MOE_BF16).  Used by kernels that serve both types.
__device__ __forceinline__ float load_elem(const void *p, int dtype, int64_t i) {
  if (dtype == MOE_F32) return static_cast<const float *>(p)[i];
  return __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[i]);
}

__device__ __forceinline__ void store_elem(void *p, int dtype, int64_t i, float v) {
  if (dtype == MOE_F32)
    static_cast<float *>(p)[i] = v;
  else
    static_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(v);
}

__host__ __device__ __forceinline__ int elem_bytes(int dtype) {
  return dtype == MOE_F32 ? 4 : 2;
}

// Activations of the expert FFN (MoE explainer §3.1 Step 4: GELU; ReLU for
// the small fp32 layer).  tanhf / erff are CUDA's own functions.
__device__ __forceinline__ float act_fwd(float z, int act) {
  if (act == MOE_ACT_RELU) return fmaxf(z, 0.0f);
  if (act == MOE_ACT_GELU_TANH) {
    const float u = 0.7978845608028654f * (z + 0.044715f * z * z * z);
    return 0.5f * z * (1.0f + tanhf(u));
  }
  return 0.5f * z * (1.0f + erff(z * 0.7071067811865476f));
}

// d act / d z.
__device__ __forceinline__ float act_grad(float z, int act) {
  if (act == MOE_ACT_RELU) return z > 0.0f ? 1.0f : 0.0f;
  if (act == MOE_ACT_GELU_TANH) {
    const float z2 = z * z;
    const float u = 0.7978845608028654f * (z + 0.044715f * z2 * z);
    const float t = tanhf(u);
    const float du = 0.7978845608028654f * (1.0f + 0.134145f * z2);
    return 0.5f * (1.0f + t) + 0.5f * z * (1.0f - t * t) * du;
  }
  const float pdf = 0.3989422804014327f * expf(-0.5f * z * z);
  return 0.5f * (1.0f + erff(z * 0.7071067811865476f)) + z * pdf;
}

// ---- l_aux statistics without FP64 arithmetic (the FP64 rate of this GPU
// is a small fraction of its FP32 rate, and these run on a single warp).
// Inputs: per-expert probability sums A_e in units of 2^-30 (exact integer
// sums, so the order of addition does not matter) and first-choice counts.
constexpr float kFix30 = 1073741824.0f;        // 2^30
constexpr float kInvFix30 = 9.313225746154785e-10f;  // 2^-30

// a probability sum of at most 2^7 tokens in units of 2^-30, converted
// through a 32-bit integer at 2^-23 (64-bit float-to-integer conversions are
// slow on this GPU); the sums stay exact integers
__device__ __forceinline__ long long fix30_tile(float v) {
  return static_cast<long long>(__float2int_rn(v * 8388608.0f)) << 7;
}

// signed 128-bit integer to the nearest-ish float (two roundings)
__device__ __forceinline__ float i128_to_float(__int128 v) {
  const bool neg = v < 0;
  const unsigned __int128 m = neg ? (unsigned __int128)(-v) : (unsigned __int128)v;
  const float f = __ull2float_rn((unsigned long long)(m >> 64)) * 18446744073709551616.0f +
                  __ull2float_rn((unsigned long long)m);
  return neg ? -f : f;
}

// (u_e - mean_e u) for the usage u_e = A_e 2^-30 / S: the deviation is
// formed exactly as A_e E - sum A in 128-bit integers, then scaled once.
__device__ __forceinline__ float usage_deviation(long long A_e, long long sum_A, int E,
                                                 int64_t S) {
  const __int128 dev = (__int128)A_e * E - (__int128)sum_A;  // (u_e - mean) S E 2^30
  return i128_to_float(dev) * kInvFix30 / (float(S) * float(E));
}

// 16-byte vector of row elements and its conversion to / from fp32.
template <typename T> struct Vec;
template <> struct Vec<float> {
  static constexpr int kN = 4;
  __device__ static void to_f32(const uint4 &u, float *o) {
    o[0] = __uint_as_float(u.x); o[1] = __uint_as_float(u.y);
    o[2] = __uint_as_float(u.z); o[3] = __uint_as_float(u.w);
  }
  __device__ static uint4 from_f32(const float *v) {
    return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]),
                      __float_as_uint(v[2]), __float_as_uint(v[3]));
  }
};
template <> struct Vec<__nv_bfloat16> {
  static constexpr int kN = 8;
  __device__ static void to_f32(const uint4 &u, float *o) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      o[2 * i] = __uint_as_float(w[i] << 16);
      o[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
  __device__ static uint4 from_f32(const float *v) {
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 b = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
      w[i] = *reinterpret_cast<uint32_t *>(&b);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
  }
};

// Activation variants for bf16 epilogues: tanh from the hardware
// tanh.approx.f32 instruction (relative error about 2^-11, well below the
// bf16 rounding of the stored result).
__device__ __forceinline__ float tanh_fast(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float act_fwd_fast(float z, int act) {
  if (act == MOE_ACT_GELU_TANH) {
    const float u = 0.7978845608028654f * fmaf(0.044715f * z, z * z, z);
    const float hz = 0.5f * z;
    return fmaf(hz, tanh_fast(u), hz);
  }
  return act_fwd(z, act);
}

__device__ __forceinline__ float act_grad_fast(float z, int act) {
  if (act == MOE_ACT_GELU_TANH) {
    const float z2 = z * z;
    const float u = 0.7978845608028654f * fmaf(0.044715f * z, z2, z);
    const float t = tanh_fast(u);
    const float du = 0.7978845608028654f * fmaf(0.134145f, z2, 1.0f);
    return 0.5f * (1.0f + t) + 0.5f * z * (1.0f - t * t) * du;
  }
  return act_grad(z, act);
}

// Programmatic dependent launch.  Every kernel of the library is launched
// with launch_k (below), so it may be scheduled while the previous kernel in
// the stream is still finishing; it starts with griddep_begin(), which waits
// until that kernel has completed and its writes are visible, and then lets
// the next kernel be scheduled in turn.  The launch latency of each kernel
// thereby overlaps the tail of the one before it.
__device__ __forceinline__ void griddep_begin() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t st, Args &&...args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = block;
  lc.dynamicSmemBytes = smem;
  lc.stream = st;
  lc.attrs = attr;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, kern, static_cast<KArgs>(args)...);
}

// Block barrier for code where lanes of a warp may have diverged (one lane
// issuing TMA copies or MMAs in a loop, one lane polling a flag).
// __syncthreads() is an aligned barrier: a warp counts as arrived as soon as
// its first lanes reach it, so a lane still inside such a loop would be left
// behind.  __syncwarp() waits for every lane of the warp first.
__device__ __forceinline__ void block_sync() {
  __syncwarp();
  __syncthreads();
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFullMask, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFullMask, v, o));
  return v;
}

// Arg-max over the warp with ties to the lower index; idx < 0 marks "none".
__device__ __forceinline__ void warp_argmax(float &v, int &idx) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(kFullMask, v, o);
    const int oi = __shfl_xor_sync(kFullMask, idx, o);
    const bool take = (oi >= 0) && (idx < 0 || ov > v || (ov == v && oi < idx));
    if (take) {
      v = ov;
      idx = oi;
    }
  }
}

__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm volatile("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Error codes a kernel writes into the device error word (first writer
// wins).  High byte: kernel; low bytes: the wait that gave up.
enum : uint32_t {
  kErrGemmProducer = 0x01000000u,
  kErrGemmMma = 0x02000000u,
  kErrGemmEpilogue = 0x03000000u,
  kErrGemmDrain = 0x04000000u,
  kErrGateProducer = 0x05000000u,
  kErrGateMma = 0x06000000u,
  kErrGateEpilogue = 0x07000000u,
  kErrWgradProducer = 0x08000000u,
  kErrWgradMma = 0x09000000u,
  kErrWgradEpilogue = 0x0a000000u,
  kErrWgradFixup = 0x0b000000u,
  kErrGateBarrier = 0x0c000000u,
  kErrGemmGather = 0x0d000000u,
};

__device__ __forceinline__ void record_error(unsigned int *err, uint32_t code) {
  if (err) atomicCAS(err, 0u, code);
}

}  // namespace moe
