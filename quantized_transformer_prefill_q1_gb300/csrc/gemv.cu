// gemv.cu — the quantised projections for chunks of at most 16 tokens: the GEMV end of the
// small-M crossover (oxibonsai-kernels metal_full_layer.rs `encode_layer_into`, the decode
// layer, whose projections are one pass over the weights per token). At M <= 16 streaming
// the packed weights from HBM and dequantising them is the whole cost; the tcgen05 path reads
// its A operand (the weights) from tensor memory at a fixed ~22 weights per clock per SM
// whatever the token count, so here the weights go from shared memory through registers into
// warp-level MMAs.
//
// A warp owns 16 weight rows (for SwiGLU 8 gate rows and their 8 up rows) and computes
// out^T[16 rows, 8 tokens] with mma.sync m16n8k16 (f16 operands, f32 accumulation) per block
// of 8 tokens (one block for M <= 8, two for M <= 16, each dequantised A fragment feeding
// both): the dequantised codes are the A fragment, the activations (tokens >= M zero) the B
// fragment.
// The (16-row tile, group) units are shared out in equal contiguous ranges, one per warp,
// and warps never wait for one another; only SwiGLU pairs two warps of a CTA on one tile
// (even and odd groups), which meet in shared memory to form silu(gate) * up. A warp streams its rows' slice of each packed chunk (16 rows x 128 weights: 1024 B of
// INT4 codes + scales and zeros, or 256 B of Q1 signs + scales) into a ring of stages in
// shared memory with cp.async, many groups ahead, so that enough bytes are in flight per SM
// to keep HBM busy without holding them in registers.
//
// The reduction order inside a 16-wide k-step is free, so each thread's four A columns are
// taken from the packed word it reads (k permuted identically in A and B): lane (g, c) =
// (lane / 4, lane % 4) reads, per 64-wide half of a group, 8 bytes (INT4: codes
// 16c .. 16c+15 of the half) or one sign word (Q1: elements 32 (c / 2) .. +31) of MMA rows g
// and g + 8, and the 16 activations 16c .. 16c+15 of the half for token g (+ 8 b). Per group the
// accumulator is scaled by the row's scale (INT4: the codes enter as f16(q s - f16(z s)), whose
// error against (q - z) s is of the order of the tcgen05 path's f16(f16(q - z) s): half an
// ulp of z s against half an ulp of q - z, times s) and added to the row's total in f32.
// Residual form: each range's share is added into out (an f32 atomic add where another warp
// shares the tile); store form: out is zeroed first and added to the same way.
#include <cuda_fp16.h>

#include <algorithm>

#include "pf_internal.h"
#include "ptx.cuh"

namespace pf {
namespace {

constexpr int WARPS_V = 4;
constexpr int THREADS_V = 32 * WARPS_V;

// One warp's stage: its 16 rows of one packed chunk. MMA rows 0-7 come from source rows
// roA .. roA+7 of the 256-row tile, MMA rows 8-15 from roB .. roB+7.
template <int WFMT>
struct ST;
template <>
struct ST<PF_W_Q1_G128> {
  static constexpr int SC = 2 * 16 * 8;  // [half][row][2 sign words], then scales [16]
  static constexpr int BYTES = SC + 32;  // 288
  static constexpr int DS = 24;          // stages in flight per warp
};
template <>
struct ST<PF_W_INT4_AFFINE_G128> {
  static constexpr int SC = 2 * 16 * 32;  // [half][row][8 nibble words], then scales, zeros
  static constexpr int ZP = SC + 32;
  static constexpr int BYTES = ZP + 32;   // 1088
  static constexpr int DS = 8;
};

__device__ __forceinline__ void cp16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
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
__device__ __forceinline__ uint32_t lds32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t a) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t lds16(uint32_t a) {
  uint16_t v;
  asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a) : "memory");
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

// Copies one warp's stage (chunk `ch`, source rows roA.., roB..) into shared memory at `st`.
__device__ __forceinline__ void issue_q1(uint32_t st, const uint8_t* ch, int roA, int roB, int lane) {
  if (lane < 16) {  // signs: [half h][block b][4 x 16 B]
    const int h = lane >> 3, b = (lane >> 2) & 1, p = lane & 3;
    cp16(st + h * 128 + b * 64 + 16 * p, ch + h * Q1_HALF_BYTES + (b ? roB : roA) * 8 + 16 * p);
  } else if (lane < 18) {
    const int b = lane - 16;
    cp16(st + ST<PF_W_Q1_G128>::SC + 16 * b, ch + Q1_SCALE_OFF + (b ? roB : roA) * 2);
  }
}
__device__ __forceinline__ void issue_i4(uint32_t st, const uint8_t* ch, int roA, int roB, int lane) {
  const int b = (lane >> 4) & 1, p = lane & 15;  // codes: [half][block b][16 x 16 B]
#pragma unroll
  for (int h = 0; h < 2; ++h)
    cp16(st + h * 512 + b * 256 + 16 * p, ch + h * I4_HALF_BYTES + (b ? roB : roA) * 32 + 16 * p);
  if (lane < 4) {
    const int bb = lane & 1;
    const bool zero = lane >= 2;
    cp16(st + (zero ? ST<PF_W_INT4_AFFINE_G128>::ZP : ST<PF_W_INT4_AFFINE_G128>::SC) + 16 * bb,
         ch + (zero ? I4_ZERO_OFF : I4_SCALE_OFF) + (bb ? roB : roA) * 2);
  }
}

// A fragment of k-step ks of half h from the stage at `st` (lane g = gq, c):
// Q1: +-1.0 for pairs i0, i0 + 1 of sign word c / 2 (pair i keeps its negative flags at bits
//     15 - i / 31 - i);
// INT4: pairs 2 (ks % 2), 2 (ks % 2) + 1 of nibble word 2c + ks / 2, dequantised to f16
//     ((1024 + q) and (1024 + 16 q) are exact f16 bit patterns).
template <int WFMT>
struct Frag;
template <>
struct Frag<PF_W_Q1_G128> {
  uint32_t z[2][2];  // [half][row g, g + 8]
  uint32_t s2[2];    // the rows' f16 scales in both halves
  // With one token block the sign words are shifted once by this lane's 8 (c & 1), so that
  // the per-k-step shifts below are constants (fewer variable shifts: decode 1.70 -> 1.65 ms
  // per token); with two blocks the per-step form measured faster.
  template <int NB>
  __device__ __forceinline__ void read(uint32_t st, int gq, int c) {
    const int sh = NB == 1 ? 8 * (c & 1) : 0;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int i = 0; i < 2; ++i) z[h][i] = lds32(st + h * 128 + i * 64 + gq * 8 + (c >> 1) * 4) << sh;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint32_t b = lds16(st + ST<PF_W_Q1_G128>::SC + i * 16 + gq * 2);
      s2[i] = b | (b << 16);
    }
  }
  // +-scale, as the tensor-core path's dequantiser forms it
  template <int NB>
  __device__ __forceinline__ void a(int h, int ks, int c, uint32_t (&f)[4]) const {
    const int i0 = (NB == 1 ? 0 : 8 * (c & 1)) + 2 * ks;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      f[i] = ((z[h][i] << i0) & 0x80008000u) ^ s2[i];
      f[2 + i] = ((z[h][i] << (i0 + 1)) & 0x80008000u) ^ s2[i];
    }
  }
};
template <>
struct Frag<PF_W_INT4_AFFINE_G128> {
  uint2 q[2][2];
  __half2 s2[2], nzs2[2];  // the rows' scale and -f16(z s), in both halves
  template <int NB>
  __device__ __forceinline__ void read(uint32_t st, int gq, int c) {
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int i = 0; i < 2; ++i) q[h][i] = lds64(st + h * 512 + i * 256 + gq * 32 + c * 8);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint32_t sb = lds16(st + ST<PF_W_INT4_AFFINE_G128>::SC + i * 16 + gq * 2);
      const uint32_t zb = lds16(st + ST<PF_W_INT4_AFFINE_G128>::ZP + i * 16 + gq * 2);
      s2[i] = u2h(sb | (sb << 16));
      nzs2[i] = __hneg2(__hmul2(u2h(zb | (zb << 16)), s2[i]));
    }
  }
  // f16(q s - f16(z s)): the code q comes out exact ((1024 + q) and (1024 + 16 q) are f16
  // bit patterns), then one fused multiply-add per weight pair: two f16 operations per pair
  // instead of the three of f16(f16(q - z) s)
  template <int NB>
  __device__ __forceinline__ void a(int h, int ks, int c, uint32_t (&f)[4]) const {
    const __half2 k1024 = u2h(0x64006400u), k16th = u2h(0x2C002C00u), km64 = u2h(0xD400D400u);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      uint32_t W = (ks >> 1) ? q[h][i].y : q[h][i].x;
      if (ks & 1) W >>= 8;
      f[i] = h2u(__hfma2(__hsub2(u2h((W & 0x000F000Fu) | 0x64006400u), k1024), s2[i], nzs2[i]));
      f[2 + i] = h2u(__hfma2(__hfma2(u2h((W & 0x00F000F0u) | 0x64006400u), k16th, km64), s2[i], nzs2[i]));
    }
  }
};

// silu(g) * u = g / (1 + e^-g) * u. The exponent is capped at 80 so the denominator stays
// below 2^126, where the fast division is within 2 ulp; for g < -80 the result is ~1e-33 * u.
__device__ __forceinline__ float silu_mul_v(float g, float u) {
  return __fdividef(g, 1.0f + __expf(fminf(-g, 80.0f))) * u;
}

// Unit u = (16-row tile t, group g). Tile t covers, for SwiGLU, gate rows 8q .. 8q+7 and the
// matching up rows of 128-row packed group b = t / 8 (q = t % 8: source rows 128 (b % 2) + 8q
// and + 64 of the 256-row tile b / 2); otherwise rows 16t .. 16t+15.
template <int EPI>
__device__ __forceinline__ void tile_rows(int t, int& tile256, int& roA, int& roB) {
  if (EPI == EPI_SWIGLU) {
    const int b = t >> 3;
    tile256 = b >> 1;
    roA = (b & 1) * 128 + 8 * (t & 7);
    roB = roA + 64;
  } else {
    tile256 = t >> 4;
    roA = (t & 15) * 16;
    roB = roA + 8;
  }
}

template <int WFMT, int EPI, int GS, int NB>
__global__ void __launch_bounds__(THREADS_V)
    gemv_kernel(const __half* a, const uint8_t* __restrict__ wpk, int M, int N, int K,
                void* __restrict__ out, long long units, int warps) {
  PF_TIMELINE(TL_GEMV + EPI);
  // NB blocks of 8 token columns (M <= 8 NB): each dequantised A fragment feeds NB MMAs
  using S = ST<WFMT>;
  constexpr int DS = S::DS / GS;     // stages in flight per warp
  constexpr int SB = GS * S::BYTES;  // a stage: GS consecutive groups of one 16-row tile
  constexpr size_t P = WFMT == PF_W_Q1_G128 ? Q1_CHUNK_BYTES : I4_CHUNK_BYTES;
  static_assert(DS >= 2, "ring depth");
  extern __shared__ __align__(16) uint8_t gv_smem[];
  __shared__ float part[WARPS_V / 2][32][4 * NB];  // SwiGLU: the odd-stage half of a tile's sums
  griddep_launch_dependents();
  const int G = K / GROUP;
  const int GG = G / GS;  // stages per tile
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gq = lane >> 2, c = lane & 3;

  const int gw = blockIdx.x * WARPS_V + warp;
  // This warp's units (tile, stage) as a cursor (t, g) stepping by `gs`: SwiGLU tiles are
  // split between two warps of the CTA by stage parity (warp 2i + p takes stages p, p + 2, ...
  // of tile 2 blockIdx + i); otherwise an equal contiguous range of units.
  int t0, g0, gs, n;
  if (EPI == EPI_SWIGLU) {
    t0 = gw >> 1;
    g0 = gw & 1;
    gs = 2;
    n = t0 < warps ? (GG - g0 + 1) >> 1 : 0;
  } else {
    const long long u0 = gw < warps ? units * gw / warps : 0;
    const long long u1 = gw < warps ? units * (gw + 1) / warps : 0;
    t0 = static_cast<int>(u0 / GG);
    g0 = static_cast<int>(u0 - static_cast<long long>(t0) * GG);
    gs = 1;
    n = static_cast<int>(u1 - u0);
  }
  const uint32_t ring = smem_u32(gv_smem) + static_cast<uint32_t>(warp * DS * SB);

  int ti = t0, gi = g0, si = 0;  // issue cursor and its stage
  auto issue_next = [&]() {
    int tile256, roA, roB;
    tile_rows<EPI>(ti, tile256, roA, roB);
    const uint8_t* ch = wpk + (static_cast<size_t>(tile256) * G + gi * GS) * P;
    const uint32_t st = ring + static_cast<uint32_t>(si * SB);
#pragma unroll
    for (int q = 0; q < GS; ++q) {
      if (WFMT == PF_W_Q1_G128) issue_q1(st + q * S::BYTES, ch + q * P, roA, roB, lane);
      else issue_i4(st + q * S::BYTES, ch + q * P, roA, roB, lane);
    }
    gi += gs;
    if (gi >= GG) {
      gi -= GG;
      ++ti;
    }
    si = si + 1 == DS ? 0 : si + 1;
  };
  // the weights never depend on the previous kernel: start streaming them before the wait
#pragma unroll 1
  for (int j = 0; j < DS - 1; ++j) {
    if (j < n) issue_next();
    cp_commit();
  }
  griddep_wait();  // the activations and the output do

  int tc = t0, gc = g0, sc = 0;  // compute cursor
  // this lane's B columns: tokens gq + 8 b of the NB blocks (zero past M)
  bool tok[NB];
  const __half* xbase[NB];
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    tok[b] = gq + 8 * b < M;
    xbase[b] = a + static_cast<size_t>(tok[b] ? gq + 8 * b : 0) * K + 16 * c;
  }
  uint4 xn[NB][4] = {};  // the next group's 16 activations of each half, per token block
  auto load_x = [&](int g, uint4 (&x)[NB][4]) {
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        x[b][e] = tok[b] ? ld_act16(xbase[b] + g * GROUP + 64 * (e >> 1) + 8 * (e & 1)) : make_uint4(0u, 0u, 0u, 0u);
  };
  if (n > 0) load_x(gc * GS, xn);
  // four independent MMA chains per token block (half, k-step parity), accumulated over a
  // segment's groups (the scales are inside the A fragments): (row g, token 2c), (g, 2c+1),
  // (g+8, 2c), (g+8, 2c+1), tokens offset by 8 b
  float d[NB][4][4] = {};
  bool seg_first = true;
  int seg_g0 = 0;
#pragma unroll 1
  for (int j = 0; j < n; ++j) {
    if (j + DS - 1 < n) issue_next();
    cp_commit();
    int tn = tc, gn = gc + gs;
    if (gn >= GG) {
      gn -= GG;
      ++tn;
    }
    cp_wait<DS - 1>();  // this lane's copies of stage j have landed
    __syncwarp();       // and every other lane's
    if (seg_first) {
      seg_g0 = gc;
      seg_first = false;
    }
#pragma unroll
    for (int q = 0; q < GS; ++q) {
      uint4 xc[NB][4];
#pragma unroll
      for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int e = 0; e < 4; ++e) xc[b][e] = xn[b][e];
      // the next group's activations: the next in this stage, else the next stage's first
      if (q + 1 < GS) load_x(gc * GS + q + 1, xn);
      else if (j + 1 < n) load_x(gn * GS, xn);
      Frag<WFMT> fr;
      fr.template read<NB>(ring + static_cast<uint32_t>(sc * SB + q * S::BYTES), gq, c);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          uint32_t af[4];
          fr.template a<NB>(h, ks, c, af);
#pragma unroll
          for (int b = 0; b < NB; ++b) {
            const uint4& xv = xc[b][2 * h + (ks >> 1)];
            mma16816(af, (ks & 1) ? xv.z : xv.x, (ks & 1) ? xv.w : xv.y, d[b][2 * h + (ks & 1)]);
          }
        }
      }
    }
    __syncwarp();  // the stage is read: it may be refilled
    const bool tile_end = EPI == EPI_SWIGLU ? j == n - 1 : (gc == GG - 1 || j == n - 1);
    const int t = tc;
    const int g = gc;
    tc = tn;
    gc = gn;
    sc = sc + 1 == DS ? 0 : sc + 1;
    if (!tile_end || EPI == EPI_SWIGLU) continue;
    // ---- end of a segment of tile t: its share (MMA row g + 8i, token 8b + 2c + e)
    const bool whole = seg_g0 == 0 && g == GG - 1;
    float* o = reinterpret_cast<float*>(out);
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int row = 16 * t + gq + 8 * i;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int m = 8 * b + 2 * c + e;
          const float v = (d[b][0][2 * i + e] + d[b][1][2 * i + e]) + (d[b][2][2 * i + e] + d[b][3][2 * i + e]);
          if (row >= N || m >= M) continue;
          float* p = o + static_cast<size_t>(m) * N + row;
          if (whole) *p += v;  // no other warp has this tile
          else atomicAdd(p, v);
        }
      }
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) d[b][x][y] = 0.f;
    seg_first = true;
  }
  if (EPI == EPI_SWIGLU) {
    // the odd-stage warp hands its sums to the even-stage warp of the same tile, which forms
    // silu(gate) * up: MMA rows g are gate rows, g + 8 their up rows
    float acc[NB][4];
#pragma unroll
    for (int b = 0; b < NB; ++b)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[b][i] = (d[b][0][i] + d[b][1][i]) + (d[b][2][i] + d[b][3][i]);
    const int pair = warp >> 1;
    if (warp & 1) {
#pragma unroll
      for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int i = 0; i < 4; ++i) part[pair][lane][4 * b + i] = acc[b][i];
    }
    __syncthreads();
    if (!(warp & 1) && n > 0) {
      if (GG > 1) {
#pragma unroll
        for (int b = 0; b < NB; ++b)
#pragma unroll
          for (int i = 0; i < 4; ++i) acc[b][i] += part[pair][lane][4 * b + i];
      }
      const int col = 8 * t0 + gq;
      __half* o = reinterpret_cast<__half*>(out);
#pragma unroll
      for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int m = 8 * b + 2 * c + e;
          if (m < M && col < (N >> 1))
            o[static_cast<size_t>(m) * (N >> 1) + col] = __float2half_rn(silu_mul_v(acc[b][e], acc[b][2 + e]));
        }
    }
  }
  cp_wait<0>();
}

template <int WFMT, int EPI, int GS, int NB>
cudaError_t launch_vg(const GemmArgs& g, cudaStream_t stream) {
  constexpr int smem = WARPS_V * (ST<WFMT>::DS / GS) * GS * ST<WFMT>::BYTES;
  static_assert(smem <= 48 * 1024, "GEMV stages");
  static const int warps_max = [] {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemv_kernel<WFMT, EPI, GS, NB>, THREADS_V, smem) !=
            cudaSuccess ||
        per_sm < 1)
      per_sm = 1;
    return per_sm * device_sm_count() * WARPS_V;
  }();
  const int G = g.K / GROUP;
  const long long tiles = EPI == EPI_SWIGLU ? g.N / 16 : padded_rows(g.N) / 16;
  const long long units = tiles * (G / GS);
  // SwiGLU: two warps per tile (gate and up rows meet in the CTA); `warps` counts tiles there.
  // Otherwise equal ranges of units, one per warp.
  int warps, ctas;
  if (EPI == EPI_SWIGLU) {
    warps = static_cast<int>(tiles);
    ctas = static_cast<int>((2 * tiles + WARPS_V - 1) / WARPS_V);
  } else {
    warps = static_cast<int>(std::min<long long>(units, warps_max));
    ctas = (warps + WARPS_V - 1) / WARPS_V;
  }
  return launch_pdl(gemv_kernel<WFMT, EPI, GS, NB>, dim3(ctas), dim3(THREADS_V), smem, stream,
                    reinterpret_cast<const __half*>(g.a), g.w, g.M, g.N, g.K, g.out, units, warps);
}

// Groups per stage: 4 when the 128-wide groups of a row divide by 4, else 2, else 1.
template <int WFMT, int EPI>
cudaError_t launch_v(const GemmArgs& g, cudaStream_t stream) {
  const int G = g.K / GROUP;
  if (g.M > 8) {  // two 8-token column blocks
    if (G % 4 == 0) return launch_vg<WFMT, EPI, 4, 2>(g, stream);
    if (G % 2 == 0) return launch_vg<WFMT, EPI, 2, 2>(g, stream);
    return launch_vg<WFMT, EPI, 1, 2>(g, stream);
  }
  if (G % 4 == 0) return launch_vg<WFMT, EPI, 4, 1>(g, stream);
  if (G % 2 == 0) return launch_vg<WFMT, EPI, 2, 1>(g, stream);
  return launch_vg<WFMT, EPI, 1, 1>(g, stream);
}

template <int WFMT>
cudaError_t launch_fmt_v(const GemmArgs& g, cudaStream_t stream) {
  if (g.epilogue == EPI_SWIGLU) return launch_v<WFMT, EPI_SWIGLU>(g, stream);
  return launch_v<WFMT, EPI_RESID_ADD>(g, stream);
}

}  // namespace

int gemv_max_m(int wfmt) { return wfmt == PF_W_Q1_G128 ? GEMV_M_MAX_Q1 : GEMV_M_MAX_I4; }

cudaError_t launch_gemv(const GemmArgs& g, cudaStream_t stream) {
  if (g.M < 1 || g.M > 16 || g.K % GROUP) return cudaErrorInvalidValue;
  if (g.epilogue == EPI_SWIGLU && g.N % 256) return cudaErrorInvalidValue;
  if (g.epilogue == EPI_STORE_F32 && !g.out_zeroed) {
    // zero the M x N output (unless the caller has) and add every range's share, as the
    // residual form does
    cudaError_t e = cudaMemsetAsync(g.out, 0, static_cast<size_t>(g.M) * g.N * sizeof(float), stream);
    if (e != cudaSuccess) return e;
  }
  if (g.wfmt == PF_W_Q1_G128) return launch_fmt_v<PF_W_Q1_G128>(g, stream);
  return launch_fmt_v<PF_W_INT4_AFFINE_G128>(g, stream);
}

}  // namespace pf

PF_TIMELINE_SETTER(gemv)
