// dequant.cuh — Q1 / INT4-affine dequantisers shared by the GEMM (which writes the
// UMMA B operand) and the stand-alone dequantisation kernel used by the bit-exact
// unpacking test, so that test exercises the very code the GEMM runs.
#pragma once
#include <cuda_fp16.h>
#include <cstdint>

#include "pf_internal.h"

namespace pf {

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// Q1: one row's 64 weights of a stage -> 8 swizzled 16-B chunks of f16.
__device__ __forceinline__ void dequant_row_q1(const uint8_t* p, int r, uint32_t b_tile) {
  const uint2 z = *reinterpret_cast<const uint2*>(p + r * 8);
  const uint32_t s16 = reinterpret_cast<const uint16_t*>(p + Q1_HALF_BYTES)[r];
  const uint32_t s2 = s16 | (s16 << 16);
  const uint32_t row_base = b_tile + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint32_t Z = (c < 4) ? z.x : z.y;
    const int i0 = 4 * (c & 3);
    const uint32_t w0 = ((Z << (i0 + 0)) & 0x80008000u) ^ s2;
    const uint32_t w1 = ((Z << (i0 + 1)) & 0x80008000u) ^ s2;
    const uint32_t w2 = ((Z << (i0 + 2)) & 0x80008000u) ^ s2;
    const uint32_t w3 = ((Z << (i0 + 3)) & 0x80008000u) ^ s2;
    st_shared_v4(row_base + ((c ^ (r & 7)) << 4), w0, w1, w2, w3);
  }
}

__device__ __forceinline__ uint32_t int4_pair(uint32_t word, int p, __half2 s2, __half2 z2) {
  const uint32_t v = ((word >> (4 * p)) & 0x000F000Fu) | 0x64006400u;  // 1024 + q, exact
  __half2 h = *reinterpret_cast<const __half2*>(&v);
  h = __hsub2(h, __half2half2(__ushort_as_half(0x6400)));  // q, exact
  h = __hmul2(__hsub2(h, z2), s2);                          // f16(f16(q - z) * s)
  return *reinterpret_cast<uint32_t*>(&h);
}

// INT4-affine: one row's 64 weights of a stage -> 8 swizzled 16-B chunks of f16.
__device__ __forceinline__ void dequant_row_int4(const uint8_t* p, int r, uint32_t b_tile) {
  const uint4 q0 = *reinterpret_cast<const uint4*>(p + r * 32);
  const uint4 q1 = *reinterpret_cast<const uint4*>(p + r * 32 + 16);
  const uint16_t s16 = reinterpret_cast<const uint16_t*>(p + I4_HALF_BYTES)[r];
  const uint16_t z16 = reinterpret_cast<const uint16_t*>(p + I4_HALF_BYTES + TILE_N * 2)[r];
  const __half2 s2 = __half2half2(__ushort_as_half(s16));
  const __half2 z2 = __half2half2(__ushort_as_half(z16));
  const uint32_t row_base = b_tile + (r >> 3) * 1024 + (r & 7) * 128;
  const uint32_t words[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    st_shared_v4(row_base + ((c ^ (r & 7)) << 4), int4_pair(words[c], 0, s2, z2),
                 int4_pair(words[c], 1, s2, z2), int4_pair(words[c], 2, s2, z2),
                 int4_pair(words[c], 3, s2, z2));
  }
}


}  // namespace pf
