// gemv.cu — the quantised projections for chunks of at most 8 tokens: the GEMV end of the
// small-M crossover (oxibonsai-kernels metal_full_layer.rs `encode_layer_into`, the decode
// layer, whose projections are one pass over the weights per token). At M <= 8 streaming the
// packed weights from HBM is the whole cost; the tcgen05 path reads its A operand (the
// weights) from tensor memory at a fixed ~22 weights per clock per SM whatever the token
// count, so here the weights go from registers straight into warp-level MMAs.
//
// A warp owns 16 weight rows and computes out^T[16 rows, 8 tokens] with
// mma.sync m16n8k16 (f16 operands, f32 accumulation): the dequantised codes are the A
// fragment, the activations (tokens >= M zero) the B fragment. The reduction order inside a
// 16-wide k-step is free, so each thread's four A columns are taken from the packed word it
// loaded itself (k permuted identically in A and B): lane (g, c) = (lane / 4, lane % 4) reads,
// per 64-wide half of a group, 8 bytes (INT4: codes 16c .. 16c+15 of the half) or one sign
// word (Q1: elements 32 (c / 2) .. +31) of rows g and g + 8, and the 16 activations
// 16c .. 16c+15 of the half for token g. Per group the accumulator is scaled by the row's
// scale (INT4: the codes enter as the f16 value q - z, rounded like the tcgen05 path's
// dequantiser rounds it) and added to the row's total in f32.
//
// A CTA is 8 warps = one 128-row block (half a packed 256-row tile: for SwiGLU its 64 gate
// rows and their 64 up rows). The (row block, group) units are shared out in equal contiguous
// ranges, one per CTA (SwiGLU: one whole row block per CTA, so gate and up meet in one CTA).
// Residual form: each range's share is added into out (an f32 atomic add where other CTAs
// share the row block); store form: out is zeroed first and added to the same way.
#include <cuda_fp16.h>

#include <algorithm>

#include "pf_internal.h"
#include "ptx.cuh"

namespace pf {
namespace {

constexpr int RB = 128;              // weight rows per CTA (row block)
constexpr int THREADS_V = 256;       // 8 warps x 16 rows
constexpr int D_PREFETCH = 4;        // groups of packed weights in flight per thread

__device__ __forceinline__ uint2 ld_stream8(const void* p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld_stream4(const void* p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld_stream2(const void* p) {
  uint16_t v;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}
// Activations are written by the previous kernel: a coherent load, kept after
// griddepcontrol.wait by being volatile (an invariant load could be hoisted above it).
__device__ __forceinline__ uint4 ld_act16(const void* p) {
  uint4 v;
  asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

__device__ __forceinline__ void mma16816(const uint32_t (&a)[4], uint32_t b0, uint32_t b1, float (&d)[4]) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2*>(&u); }
__device__ __forceinline__ float h2f(uint32_t bits) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(bits)));
}

// One thread's packed weights of one group: rows g and g + 8 of the warp, both halves.
template <int WFMT>
struct WU;
template <>
struct WU<PF_W_Q1_G128> {
  uint32_t z[2][2];  // [half][row]: sign word c / 2 of the half-row
  uint32_t s[2];
  __device__ __forceinline__ void load(const uint8_t* ch, int row2, int c) {
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int i = 0; i < 2; ++i) z[h][i] = ld_stream4(ch + h * Q1_HALF_BYTES + (row2 + 8 * i) * 8 + (c >> 1) * 4);
#pragma unroll
    for (int i = 0; i < 2; ++i) s[i] = ld_stream2(ch + Q1_SCALE_OFF + (row2 + 8 * i) * 2);
  }
  // A fragment of k-step ks of half h: +-1.0 for pairs i0, i0 + 1 of the word (the word's
  // pair i keeps its negative flags at bits 15 - i / 31 - i)
  __device__ __forceinline__ void frag(int h, int ks, int c, uint32_t (&a)[4]) const {
    const int i0 = 8 * (c & 1) + 2 * ks;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      a[i] = ((z[h][i] << i0) & 0x80008000u) | 0x3C003C00u;
      a[2 + i] = ((z[h][i] << (i0 + 1)) & 0x80008000u) | 0x3C003C00u;
    }
  }
};
template <>
struct WU<PF_W_INT4_AFFINE_G128> {
  uint2 q[2][2];  // [half][row]: nibble words 2c, 2c + 1 of the half-row
  uint32_t s[2], zp[2];
  __device__ __forceinline__ void load(const uint8_t* ch, int row2, int c) {
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int i = 0; i < 2; ++i) q[h][i] = ld_stream8(ch + h * I4_HALF_BYTES + (row2 + 8 * i) * 32 + c * 8);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      s[i] = ld_stream2(ch + I4_SCALE_OFF + (row2 + 8 * i) * 2);
      zp[i] = ld_stream2(ch + I4_ZERO_OFF + (row2 + 8 * i) * 2);
    }
  }
  // A fragment of k-step ks: pairs 2 (ks % 2), 2 (ks % 2) + 1 of word 2c + ks / 2, as the f16
  // values q - z ((1024 + q) and (1024 + 16 q) are exact f16 bit patterns)
  __device__ __forceinline__ void frag(int h, int ks, int c, uint32_t (&a)[4]) const {
    const __half2 k1024 = u2h(0x64006400u), k16th = u2h(0x2C002C00u), km64 = u2h(0xD400D400u);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      uint32_t W = (ks >> 1) ? q[h][i].y : q[h][i].x;
      if (ks & 1) W >>= 8;
      const __half2 z2 = u2h(zp[i] | (zp[i] << 16));
      a[i] = h2u(__hsub2(__hsub2(u2h((W & 0x000F000Fu) | 0x64006400u), k1024), z2));
      a[2 + i] = h2u(__hsub2(__hfma2(u2h((W & 0x00F000F0u) | 0x64006400u), k16th, km64), z2));
    }
  }
};

__device__ __forceinline__ float silu_mul_v(float g, float u) { return g / (1.0f + __expf(-g)) * u; }

template <int WFMT, int EPI>
__global__ void __launch_bounds__(THREADS_V, 2)
    gemv_kernel(const __half* a, const uint8_t* __restrict__ wpk, int M, int N, int K,
                void* __restrict__ out, long long units, int ctas) {
  constexpr size_t P = WFMT == PF_W_Q1_G128 ? Q1_CHUNK_BYTES : I4_CHUNK_BYTES;
  __shared__ float xch[RB / 2][8];  // SwiGLU: up rows' totals handed to the gate rows
  griddep_launch_dependents();
  const int G = K / GROUP;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, c = lane & 3;
  const int r0 = 16 * warp + gq;  // rows r0 and r0 + 8 of the row block
  const bool tok = gq < M;        // this lane's B column (token gq) exists
  const long long u0 = units * blockIdx.x / ctas, u1 = units * (blockIdx.x + 1) / ctas;
  bool waited = false;
  for (long long u = u0; u < u1;) {
    // ---- one segment: groups [g0, g1) of row block rb
    const int rb = static_cast<int>(u / G);
    const int g0 = static_cast<int>(u - static_cast<long long>(rb) * G);
    const int g1 = static_cast<int>(std::min<long long>(G, g0 + (u1 - u)));
    const bool whole = g0 == 0 && g1 == G;
    u += g1 - g0;
    const int n = g1 - g0;
    const int row2 = (rb & 1) * RB + r0;  // row within the 256-row packed tile
    const uint8_t* tile = wpk + static_cast<size_t>(rb >> 1) * G * P + static_cast<size_t>(g0) * P;
    const __half* xrow = a + static_cast<size_t>(tok ? gq : 0) * K + g0 * GROUP + 16 * c;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};  // (r0, 2c), (r0, 2c+1), (r0+8, 2c), (r0+8, 2c+1)
    WU<WFMT> un[D_PREFETCH];
#pragma unroll
    for (int d = 0; d < D_PREFETCH; ++d)
      if (d < n) un[d].load(tile + d * P, row2, c);
    if (!waited) {  // the weights never depend on the previous kernel; the activations do
      griddep_wait();
      waited = true;
    }
    for (int j0 = 0; j0 < n; j0 += D_PREFETCH) {
#pragma unroll
      for (int d = 0; d < D_PREFETCH; ++d) {
        const int j = j0 + d;
        if (j < n) {
          uint4 xb[2][2];  // [half][8 of the 16 activations]
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int e = 0; e < 2; ++e)
              xb[h][e] = tok ? ld_act16(xrow + j * GROUP + 64 * h + 8 * e) : make_uint4(0u, 0u, 0u, 0u);
          float dd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              uint32_t af[4];
              un[d].frag(h, ks, c, af);
              const uint4& xv = xb[h][ks >> 1];
              mma16816(af, (ks & 1) ? xv.z : xv.x, (ks & 1) ? xv.w : xv.y, dd);
            }
          }
          const float s0 = h2f(un[d].s[0]), s1 = h2f(un[d].s[1]);
          acc[0] = fmaf(s0, dd[0], acc[0]);
          acc[1] = fmaf(s0, dd[1], acc[1]);
          acc[2] = fmaf(s1, dd[2], acc[2]);
          acc[3] = fmaf(s1, dd[3], acc[3]);
          if (j + D_PREFETCH < n) un[d].load(tile + static_cast<size_t>(j + D_PREFETCH) * P, row2, c);
        }
      }
    }
    // ---- the segment's share: acc[2i + t] is row r0 + 8i, token 2c + t
    if (EPI == EPI_SWIGLU) {
      // every SwiGLU range is one whole row block: rows 0..63 gate, 64..127 the matching up
      if (warp >= 4) {
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
          for (int t = 0; t < 2; ++t) xch[r0 + 8 * i - RB / 2][2 * c + t] = acc[2 * i + t];
      }
      __syncthreads();
      if (warp < 4) {
        __half* o = reinterpret_cast<__half*>(out);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const int col = rb * (RB / 2) + r0 + 8 * i;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int m = 2 * c + t;
            if (m < M && col < (N >> 1))
              o[static_cast<size_t>(m) * (N >> 1) + col] =
                  __float2half_rn(silu_mul_v(acc[2 * i + t], xch[r0 + 8 * i][m]));
          }
        }
      }
      __syncthreads();  // xch is free for the next segment
    } else {
      float* o = reinterpret_cast<float*>(out);
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int row = rb * RB + r0 + 8 * i;
        if (row >= N) continue;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int m = 2 * c + t;
          if (m >= M) continue;
          float* p = o + static_cast<size_t>(m) * N + row;
          if (whole) *p += acc[2 * i + t];  // no other CTA has this row block
          else atomicAdd(p, acc[2 * i + t]);
        }
      }
    }
  }
  if (!waited) griddep_wait();
}

template <int WFMT, int EPI>
cudaError_t launch_v(const GemmArgs& g, cudaStream_t stream) {
  static const int ctas_max = [] {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemv_kernel<WFMT, EPI>, THREADS_V, 0) != cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
    return per_sm * device_sm_count();
  }();
  const int G = g.K / GROUP;
  const long long nrb = padded_rows(g.N) / RB;
  const long long units = nrb * G;
  // SwiGLU: one whole row block per CTA (gate and up rows meet in it); otherwise equal ranges
  const int ctas = EPI == EPI_SWIGLU ? static_cast<int>(nrb) : static_cast<int>(std::min<long long>(units, ctas_max));
  return launch_pdl(gemv_kernel<WFMT, EPI>, dim3(ctas), dim3(THREADS_V), 0, stream,
                    reinterpret_cast<const __half*>(g.a), g.w, g.M, g.N, g.K, g.out, units, ctas);
}

template <int WFMT>
cudaError_t launch_fmt_v(const GemmArgs& g, cudaStream_t stream) {
  if (g.epilogue == EPI_SWIGLU) return launch_v<WFMT, EPI_SWIGLU>(g, stream);
  return launch_v<WFMT, EPI_RESID_ADD>(g, stream);
}

}  // namespace

int gemv_max_m(int wfmt) { return wfmt == PF_W_Q1_G128 ? GEMV_M_MAX_Q1 : GEMV_M_MAX_I4; }

cudaError_t launch_gemv(const GemmArgs& g, cudaStream_t stream) {
  if (g.M < 1 || g.M > 8 || g.K % GROUP) return cudaErrorInvalidValue;
  if (g.epilogue == EPI_STORE_F32) {
    // zero the M x N output and add every range's share, as the residual form does
    cudaError_t e = cudaMemsetAsync(g.out, 0, static_cast<size_t>(g.M) * g.N * sizeof(float), stream);
    if (e != cudaSuccess) return e;
  }
  if (g.wfmt == PF_W_Q1_G128) return launch_fmt_v<PF_W_Q1_G128>(g, stream);
  return launch_fmt_v<PF_W_INT4_AFFINE_G128>(g, stream);
}

}  // namespace pf
