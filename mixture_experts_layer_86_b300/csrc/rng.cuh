// Counter-based randomness of the gating variants: Philox4x32-10 and the
// draws built on it.  Internal header.
//
// The deepspeed.moe overview (adg.csdn.net/694deb285b9f5f31781ae763, §2.1)
// names noisy_gate_policy (jitter / rsample), use_rts and
// top2_2nd_expert_sampling without formulas.  The layer draws their
// randomness itself from Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC 2011:
// ten rounds of two 32x32->64-bit multiplies on a 4-word counter, the 2-word
// key advanced by the Weyl constants between rounds), so that a run is
// reproducible from (seed, offset) and checkable word for word:
//   key     = (seed low word, seed high word)
//   counter = (index, purpose << 24 | sub, offset low word, offset high word)
//   purpose 1  gate noise u[s,e]: index s, sub e / 4, output word e % 4
//   purpose 2  jitter u[s,c]:     index s, sub c / 4, output word c % 4
//   purpose 3  round r of the random-token-selection permutation: index =
//              the round's input half, sub r, output word 0
//   u = ((word >> 9) + 0.5) * 2^-23, inside (0, 1) and exact in float32.
#pragma once

#include <stdint.h>

namespace moe {
namespace rng {

constexpr uint32_t kPurposeGateNoise = 1, kPurposeJitter = 2, kPurposeRts = 3;

struct Key {
  uint32_t k0, k1;   // from the seed
  uint32_t o0, o1;   // the offset: counter words 2 and 3
};

__host__ __device__ inline Key make_key(uint64_t seed, uint64_t offset) {
  return Key{uint32_t(seed), uint32_t(seed >> 32), uint32_t(offset), uint32_t(offset >> 32)};
}

__device__ __forceinline__ uint4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2,
                                               uint32_t c3, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t lo0 = 0xD2511F53u * c0, hi0 = __umulhi(0xD2511F53u, c0);
    const uint32_t lo1 = 0xCD9E8D57u * c2, hi1 = __umulhi(0xCD9E8D57u, c2);
    const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return make_uint4(c0, c1, c2, c3);
}

// the 4 words of the block holding element i (of 4 per block) of row `index`
__device__ __forceinline__ uint4 block(const Key &k, uint32_t purpose, uint32_t index,
                                       uint32_t sub) {
  return philox4x32_10(index, (purpose << 24) | sub, k.o0, k.o1, k.k0, k.k1);
}

__device__ __forceinline__ uint32_t word(const uint4 &w, int i) {
  return i == 0 ? w.x : i == 1 ? w.y : i == 2 ? w.z : w.w;
}

// u in (0, 1): the 23 high bits of the word, centred in their interval
__device__ __forceinline__ float uniform(uint32_t w) {
  return (float(w >> 9) + 0.5f) * 1.1920928955078125e-07f;  // 2^-23
}

// standard Gumbel variate -ln(-ln u) (CUDA's logf)
__device__ __forceinline__ float gumbel(float u) { return -logf(-logf(u)); }

// multiplicative jitter 1 + eps * (2u - 1), each step rounded to float32
// (no contraction into fused multiply-adds, so the value is reproducible)
__device__ __forceinline__ float jitter(float u, float eps) {
  return __fadd_rn(1.0f, __fmul_rn(eps, __fsub_rn(__fmul_rn(2.0f, u), 1.0f)));
}

// ---- random token selection: a keyed permutation of [0, n)
// A 4-round Feistel network on b-bit words (b even, the smallest with
// 2^b >= n, halves of b/2 bits), restricted to [0, n) by cycle walking.
struct Perm {
  Key key;
  uint32_t n, half, mask;
};

__host__ __device__ inline Perm make_perm(const Key &k, uint32_t n) {
  uint32_t b = 2;
  while (b < 32 && (uint64_t(1) << b) < n) b += 2;
  return Perm{k, n, b / 2, (1u << (b / 2)) - 1u};
}

__device__ __forceinline__ uint32_t feistel_round(const Perm &p, uint32_t v, uint32_t r) {
  return philox4x32_10(v, (kPurposeRts << 24) | r, p.key.o0, p.key.o1, p.key.k0, p.key.k1).x &
         p.mask;
}

__device__ __forceinline__ uint32_t feistel(const Perm &p, uint32_t x) {
  uint32_t l = x >> p.half, r = x & p.mask;
#pragma unroll
  for (uint32_t i = 0; i < 4; ++i) {
    const uint32_t t = r;
    r = l ^ feistel_round(p, r, i);
    l = t;
  }
  return (l << p.half) | r;
}

__device__ __forceinline__ uint32_t feistel_inv(const Perm &p, uint32_t y) {
  uint32_t l = y >> p.half, r = y & p.mask;
#pragma unroll
  for (int i = 3; i >= 0; --i) {
    const uint32_t t = l;
    l = r ^ feistel_round(p, l, uint32_t(i));
    r = t;
  }
  return (l << p.half) | r;
}

// queue position of token s; the walk stays inside the cycle through s,
// which holds s itself, so it ends after fewer than 2^b steps
__device__ __forceinline__ uint32_t position_of(const Perm &p, uint32_t s) {
  uint32_t y = feistel(p, s);
  while (y >= p.n) y = feistel(p, y);
  return y;
}

// token at queue position q
__device__ __forceinline__ uint32_t token_at(const Perm &p, uint32_t q) {
  uint32_t x = feistel_inv(p, q);
  while (x >= p.n) x = feistel_inv(p, x);
  return x;
}

}  // namespace rng
}  // namespace moe
