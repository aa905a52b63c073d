// dequant.cuh — Q1 / INT4-affine dequantisers shared by the GEMM (which stores their
// output into tensor memory as the MMA's A operand) and the stand-alone dequantisation
// kernel used by the bit-exact unpacking test, so that test exercises the very code the
// GEMM runs. Each turns 32 consecutive weights of one row into 16 f16x2 words (k order,
// low half = even k).
#pragma once
#include <cuda_fp16.h>
#include <cstdint>

#include "pf_internal.h"

namespace pf {

// Q1: one 32-bit word of negative flags (pair i at bits 15-i / 31-i, see pf_internal.h)
// and the f16 scale replicated in both halves of s2 -> +-scale.
__device__ __forceinline__ void dq_q1_32(uint32_t Z, uint32_t s2, uint32_t (&w)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) w[i] = ((Z << i) & 0x80008000u) ^ s2;
}

// INT4 pair p of a nibble word -> f16x2 of f16(f16(q - z) * s).
__device__ __forceinline__ uint32_t int4_pair(uint32_t word, int p, __half2 s2, __half2 z2) {
  const uint32_t v = ((word >> (4 * p)) & 0x000F000Fu) | 0x64006400u;  // 1024 + q, exact
  __half2 h = *reinterpret_cast<const __half2*>(&v);
  h = __hsub2(h, __half2half2(__ushort_as_half(0x6400)));  // q, exact
  h = __hmul2(__hsub2(h, z2), s2);                          // f16(f16(q - z) * s)
  return *reinterpret_cast<uint32_t*>(&h);
}

// INT4: four nibble words (32 weights) -> 16 f16x2 words.
__device__ __forceinline__ void dq_i4_32(uint4 q, __half2 s2, __half2 z2, uint32_t (&w)[16]) {
  const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int j = 0; j < 4; ++j)
#pragma unroll
    for (int p = 0; p < 4; ++p) w[4 * j + p] = int4_pair(words[j], p, s2, z2);
}

}  // namespace pf
