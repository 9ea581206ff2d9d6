// device_common.cuh -- device-side building blocks of the 2:4 mask layer.
//
// "MaskLLM: Learnable Semi-Structured Sparsity for Large Language Models",
// Fig. 3: per group of 4 weights a categorical distribution over the six 2:4
// candidates, sampled with the Gumbel softmax and averaged into a soft mask.
// The noise comes from Philox4x32-10 (Salmon et al., "Parallel Random
// Numbers: As Easy as 1, 2, 3", SC'11), regenerated in registers from
// (seed, group index, step, tensor id) -- never stored.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace maskllm {

constexpr int kCand = 6;
constexpr int kTableBits = 14;
constexpr int kTableSize = 1 << kTableBits;
constexpr float kLog2e = 1.44269504088896340736f;  // log2(e)

// Round keys of Philox4x32-10 for one seed: key_i = key_0 + i * (Weyl
// constants), computed on the host and passed by value so that the xor with
// the key reads a kernel-parameter (constant bank) operand.
struct RoundKeys {
  uint32_t k0[10];
  uint32_t k1[10];
};

// Host side: the key schedule of one seed (Weyl increments of the Philox
// key, one pair per round).
inline RoundKeys make_round_keys(uint64_t seed) {
  RoundKeys k;
  uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
  for (int i = 0; i < 10; ++i) {
    k.k0[i] = k0;
    k.k1[i] = k1;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return k;
}

// The Philox4x32 bijection, 10 rounds: each round takes the 64-bit products
// of counter words 0 and 2 with the two Philox multipliers, xors each high
// half with the other pair's odd word and the round key, and moves the low
// halves into the odd words.
__device__ __forceinline__ uint4 philox4x32_10(uint32_t x0, uint32_t x1, uint32_t x2,
                                               uint32_t x3, const RoundKeys& K) {
#pragma unroll
  for (int i = 0; i < 10; ++i) {
    const uint64_t p0 = static_cast<uint64_t>(0xD2511F53u) * x0;
    const uint64_t p1 = static_cast<uint64_t>(0xCD9E8D57u) * x2;
    const uint32_t y0 = static_cast<uint32_t>(p1 >> 32) ^ x1 ^ K.k0[i];
    const uint32_t y2 = static_cast<uint32_t>(p0 >> 32) ^ x3 ^ K.k1[i];
    x1 = static_cast<uint32_t>(p1);
    x3 = static_cast<uint32_t>(p0);
    x0 = y0;
    x2 = y2;
  }
  return make_uint4(x0, x1, x2, x3);
}

// Noise words of group gidx: counter (gidx lo, gidx hi, step, tensor id).
__device__ __forceinline__ uint4 group_words(uint64_t gidx, uint32_t step, uint32_t tensor_id,
                                             const RoundKeys& K) {
  return philox4x32_10(static_cast<uint32_t>(gidx), static_cast<uint32_t>(gidx >> 32), step,
                       tensor_id, K);
}

// Gumbel noise of the six candidates: candidate c reads the 16-bit half
// (c & 1) of word (c >> 1), low half first, and its top 14 bits index the
// quantile table (resident in shared memory).  The byte offset of cell
// (h >> 2) is h & ~3, taken straight from the word.
__device__ __forceinline__ float table_at(const float* tab, uint32_t byte_offset) {
  return *reinterpret_cast<const float*>(reinterpret_cast<const char*>(tab) + byte_offset);
}

__device__ __forceinline__ void gumbel6(const uint4 w, const float* __restrict__ tab,
                                        float g[kCand]) {
  g[0] = table_at(tab, w.x & 0xFFFCu);
  g[1] = table_at(tab, (w.x >> 16) & 0xFFFCu);
  g[2] = table_at(tab, w.y & 0xFFFCu);
  g[3] = table_at(tab, (w.y >> 16) & 0xFFFCu);
  g[4] = table_at(tab, w.z & 0xFFFCu);
  g[5] = table_at(tab, (w.z >> 16) & 0xFFFCu);
}

// 2^x, flushing subnormal results to zero (one MUFU operation).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Exponent offset of the unnormalised softmax terms: e_c = 2^(d_c + 64) with
// d_c = (z_c - max z) log2 e <= ~0, so the largest term is ~2^64 and terms
// down to 2^-190 of it stay normal fp32 numbers when ex2 flushes subnormals.
// Anything smaller cannot reach a bf16 W' (w * M < 2^-190 rounds to zero;
// the smallest bf16 subnormal is 2^-133).  The factor cancels in e_c / sum e.
constexpr float kExpOffset = 64.0f;

// Unnormalised softmax of one group.  The noisy logit
//   z_c = fl(fl(fl(kappa * L_c) + g_c) * rho)
// is formed with explicitly rounded operations (no contraction), so it is
// bit-identical to any other IEEE implementation of the same three steps.
// Then e_c = 2^(z_c log2 e - m log2 e + 64) with m = max z: the shift is
// common to all six terms and cancels in p_c = e_c / sum e.  Also returns the
// four soft-mask numerators n_j = sum of e_c over the candidates keeping j:
// position 0: c0 (0,1) c1 (0,2) c2 (0,3);  position 1: c0, c3 (1,2), c4 (1,3);
// position 2: c1, c3, c5 (2,3);            position 3: c2, c4, c5.
__device__ __forceinline__ void noisy_logits6(const float L[kCand], const float g[kCand],
                                              float kappa, float rho, float y[kCand],
                                              float z[kCand]) {
#pragma unroll
  for (int c = 0; c < kCand; ++c) {
    y[c] = __fmul_rn(kappa, L[c]);
    z[c] = __fmul_rn(__fadd_rn(y[c], g[c]), rho);
  }
}

__device__ __forceinline__ void softmax6_of_z(const float z[kCand], float e[kCand],
                                              float& inv_sum, float num[4]) {
  const float m = fmaxf(fmaxf(fmaxf(z[0], z[1]), fmaxf(z[2], z[3])), fmaxf(z[4], z[5]));
  const float shift = kExpOffset - __fmul_rn(m, kLog2e);
#pragma unroll
  for (int c = 0; c < kCand; ++c) e[c] = ex2_approx(__fmaf_rn(z[c], kLog2e, shift));
  const float e34 = e[3] + e[4];
  const float e35 = e[3] + e[5];
  const float e45 = e[4] + e[5];
  num[0] = (e[0] + e[1]) + e[2];
  num[1] = e[0] + e34;
  num[2] = e[1] + e35;
  num[3] = e[2] + e45;
  inv_sum = rcp_approx(num[0] + e34 + e[5]);
}

__device__ __forceinline__ void softmax6(const float L[kCand], const float g[kCand], float kappa,
                                         float rho, float e[kCand], float& inv_sum,
                                         float num[4]) {
  float y[kCand], z[kCand];
  noisy_logits6(L, g, kappa, rho, y, z);
  softmax6_of_z(z, e, inv_sum, num);
}

// Soft mask M_j = sum of p_c over the candidates keeping position j.
__device__ __forceinline__ void soft_mask4(const float num[4], float inv_sum, float M[4]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) M[j] = num[j] * inv_sum;
}

// bf16 pairs packed in a 32-bit word: element 0 in the low half.
__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Copy the Gumbel quantile table from global into shared memory (one CTA).
__device__ __forceinline__ void load_table(float* __restrict__ smem_tab,
                                           const float* __restrict__ gtab) {
  const float4* src = reinterpret_cast<const float4*>(gtab);
  float4* dst = reinterpret_cast<float4*>(smem_tab);
  for (int i = threadIdx.x; i < kTableSize / 4; i += blockDim.x) dst[i] = __ldg(src + i);
}

}  // namespace maskllm
