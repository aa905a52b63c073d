// kernels.cu — the HBM-bound steps of the prefill path: RMSNorm, fused QK-norm + RoPE +
// KV-store, embedding gather, the final-norm + LM-head GEMV, a split-K SwiGLU, and the
// stand-alone dequantiser used to check unpacking bit-exactly.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "dequant.cuh"
#include "ptx.cuh"

#include <algorithm>
#include <climits>

namespace pf {
namespace {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Sum over the block; every thread gets the result. `red` holds >= 32 floats.
__device__ __forceinline__ float block_sum(float v, float* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) red[warp] = v;
  __syncthreads();
  const int nw = (blockDim.x + 31) >> 5;
  float t = lane < nw ? red[lane] : 0.f;
  return warp_sum(t);
}

// Row `row` of an optional f32 buffer [rows, 4 zero4] set to zero (a store-form GEMM that
// follows accumulates its output there by reduce-add): issued with the norm, so the GEMM needs
// no memset of its own between the two kernels.
__device__ __forceinline__ void zero_row(float4* __restrict__ zero, int zero4, int row) {
  if (zero == nullptr) return;
  float4* z = zero + static_cast<size_t>(row) * zero4;
  for (int i = threadIdx.x; i < zero4; i += blockDim.x) __stcg(z + i, make_float4(0.f, 0.f, 0.f, 0.f));
}

// ------------------------------------------------------------------ RMSNorm
// oxibonsai-kernels metal_prefill.rs `encode_layer_prefill` sections 1 and 5
// (`dispatch_batched_rmsnorm`): y[m, :] = x[m, :] * w / sqrt(mean(x[m, :]^2) + eps),
// f32 in, f16 out (the next GEMM's operand). One CTA per row, 128-bit loads.
__global__ void __launch_bounds__(256) rmsnorm_kernel(const float* __restrict__ x,
                                                      const float* __restrict__ w, float eps,
                                                      int H, __half* __restrict__ y,
                                                      float4* __restrict__ zero, int zero4) {
  PF_TIMELINE(TL_RMSNORM);
  __shared__ float red[32];
  griddep_launch_dependents();
  griddep_wait();
  const int row = blockIdx.x;
  zero_row(zero, zero4, row);
  const float4* xr = reinterpret_cast<const float4*>(x + static_cast<size_t>(row) * H);
  const float4* w4 = reinterpret_cast<const float4*>(w);
  __half2* yr = reinterpret_cast<__half2*>(y + static_cast<size_t>(row) * H);
  const int n4 = H >> 2;
  float ss = 0.f;
  for (int i = threadIdx.x; i < n4; i += blockDim.x) {
    const float4 v = xr[i];
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  ss = block_sum(ss, red);
  const float r = rsqrtf(ss / static_cast<float>(H) + eps);
  for (int i = threadIdx.x; i < n4; i += blockDim.x) {
    const float4 v = xr[i];
    const float4 g = w4[i];
    yr[2 * i] = __floats2half2_rn(v.x * r * g.x, v.y * r * g.y);
    yr[2 * i + 1] = __floats2half2_rn(v.z * r * g.z, v.w * r * g.w);
  }
}

// Same, for H = 512 * NV: 128 threads per row, each holding NV float4 of the row in
// registers, so the row is read from global memory once; one barrier for the reduction.
template <int NV>
__global__ void __launch_bounds__(128) rmsnorm_reg_kernel(const float* __restrict__ x,
                                                          const float* __restrict__ w, float eps,
                                                          int H, __half* __restrict__ y,
                                                          float4* __restrict__ zero, int zero4) {
  PF_TIMELINE(TL_RMSNORM_REG);
  __shared__ float red[4];
  griddep_launch_dependents();
  // the norm weights never depend on the previous kernel: load them while it finishes
  const float4* w4 = reinterpret_cast<const float4*>(w);
  float4 g[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) g[i] = w4[threadIdx.x + 128 * i];
  griddep_wait();
  const int row = blockIdx.x;
  const float4* xr = reinterpret_cast<const float4*>(x + static_cast<size_t>(row) * H);
  float4 v[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) v[i] = xr[threadIdx.x + 128 * i];
  zero_row(zero, zero4, row);
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i) ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  ss = red[0] + red[1] + red[2] + red[3];
  const float r = rsqrtf(ss / static_cast<float>(H) + eps);
  uint2* yr = reinterpret_cast<uint2*>(y + static_cast<size_t>(row) * H);
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int idx = threadIdx.x + 128 * i;
    const __half2 a = __floats2half2_rn(v[i].x * r * g[i].x, v[i].y * r * g[i].y);
    const __half2 b = __floats2half2_rn(v[i].z * r * g[i].z, v[i].w * r * g[i].w);
    yr[idx] = make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
  }
}

// ------------------------------------------------------------------ QK-norm + RoPE + KV
constexpr int QK_SLOTS = 4;  // head groups per warp in qk_norm_rope_kv_kernel
template <typename T>
__device__ __forceinline__ T to_elem(float v);
template <>
__device__ __forceinline__ float to_elem<float>(float v) { return v; }
template <>
__device__ __forceinline__ __half to_elem<__half>(float v) { return __float2half_rn(v); }
template <>
__device__ __forceinline__ __nv_bfloat16 to_elem<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

template <typename T>
__device__ __forceinline__ void store4(T* dst, float a, float b, float c, float d);
template <>
__device__ __forceinline__ void store4<float>(float* dst, float a, float b, float c, float d) {
  *reinterpret_cast<float4*>(dst) = make_float4(a, b, c, d);
}
template <>
__device__ __forceinline__ void store4<__half>(__half* dst, float a, float b, float c, float d) {
  const __half2 x = __floats2half2_rn(a, b), y = __floats2half2_rn(c, d);
  *reinterpret_cast<uint2*>(dst) =
      make_uint2(*reinterpret_cast<const uint32_t*>(&x), *reinterpret_cast<const uint32_t*>(&y));
}
template <>
__device__ __forceinline__ void store4<__nv_bfloat16>(__nv_bfloat16* dst, float a, float b, float c,
                                                      float d) {
  const __nv_bfloat162 x = __floats2bfloat162_rn(a, b), y = __floats2bfloat162_rn(c, d);
  *reinterpret_cast<uint2*>(dst) =
      make_uint2(*reinterpret_cast<const uint32_t*>(&x), *reinterpret_cast<const uint32_t*>(&y));
}

// One group of HD/8 lanes per (token, head) of the fused QKV output, heads ordered
// Q | K | V; lane l holds elements 4l..4l+3 of each half of the head (128-bit loads).
// metal_prefill.rs `encode_layer_prefill` section 3 (fused_qk_norm, fused_qk_rope,
// fused_kv_store) and metal_full_layer.rs `dispatch_fused_qk_norm_rope`, batched over the
// chunk: Q and K heads get an RMSNorm over head_dim (weights w_q / w_k, the layer eps)
// when enabled, then rotate-half RoPE at position start + t from the (cos, sin) table;
// Q goes to q_out [M, nq, hd], K to the cache slot [layer, kvh, pos, :], and V is copied
// unchanged to its slot. Cache layout of metal_full_layer.rs `GpuKvCache`:
// [n_layers][nkv][max_seq][hd]: K/V row (kv_layer * nkv + kvh) * kv_rows + start + t
// (kv_by_pos = 1); a ring cache's chunk buffers take row kvh * kv_rows + t (kv_layer = 0,
// kv_by_pos = 0) and the ring slots are filled after the attention (ring_store_kernel).
template <int HD, typename QT, typename KT>
__global__ void __launch_bounds__(256, 3) qk_norm_rope_kv_kernel(
    const float* __restrict__ qkv, const float* __restrict__ qn, const float* __restrict__ kn,
    const float* __restrict__ rope, int M, int nq, int nkv, int kv_rows, int kv_layer, int kv_by_pos,
    const int* __restrict__ start_dev, int start_host, float eps, int qk_norm,
    QT* __restrict__ q_out, KT* __restrict__ kc, KT* __restrict__ vc, const int* __restrict__ blocks) {
  PF_TIMELINE(TL_QK_ROPE_KV);
  constexpr int HALF = HD / 2;
  constexpr int LPH = HALF / 4;   // lanes per head
  constexpr int HPW = 32 / LPH;   // heads per warp and slot
  griddep_launch_dependents();
  const int heads = nq + 2 * nkv;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int l = lane % LPH;
  griddep_wait();
  const int start = start_dev ? *start_dev : start_host;
  // QK_SLOTS groups of HPW (token, head) pairs per warp: every slot's head values are loaded
  // before any is used, so a launch is one round trip per thread and fits the GPU in one wave
  // (the (cos, sin) rows and norm weights, shared by the heads of a token / kind, come after)
  float4 A[QK_SLOTS], B[QK_SLOTS];
#pragma unroll
  for (int s = 0; s < QK_SLOTS; ++s) {
    const int gh = (gw * QK_SLOTS + s) * HPW + lane / LPH;  // (token, head) index
    const int t = gh / heads, j = gh - t * heads;
    A[s] = B[s] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (t < M) {
      const float4* src = reinterpret_cast<const float4*>(qkv + (static_cast<size_t>(t) * heads + j) * HD);
      A[s] = src[l];
      B[s] = src[LPH + l];
    }
  }
#pragma unroll
  for (int s = 0; s < QK_SLOTS; ++s) {
    const int gh = (gw * QK_SLOTS + s) * HPW + lane / LPH;
    const int t = gh / heads, j = gh - t * heads;
    const bool is_q = j < nq, is_v = j >= nq + nkv;
    float4 a = A[s], b = B[s];
    // per-head sum of squares over the LPH lanes of the group (every lane takes part)
    float ss = a.x * a.x + a.y * a.y + a.z * a.z + a.w * a.w + b.x * b.x + b.y * b.y + b.z * b.z + b.w * b.w;
#pragma unroll
    for (int o = LPH / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (t >= M) continue;
    const int pos = start + t;
    // cache slot of the position; a paged cache goes through the block table
    const int kv_row = !kv_by_pos ? t : (blocks ? blocks[pos / PF_KV_BLOCK] * PF_KV_BLOCK + pos % PF_KV_BLOCK : pos);
    if (is_v) {  // V head: straight to the cache
      KT* dst = vc + ((static_cast<size_t>(kv_layer) * nkv + (j - nq - nkv)) * kv_rows + kv_row) * HD;
      store4<KT>(dst + 4 * l, a.x, a.y, a.z, a.w);
      store4<KT>(dst + HALF + 4 * l, b.x, b.y, b.z, b.w);
      continue;
    }
    const float4* cs = reinterpret_cast<const float4*>(rope + (static_cast<size_t>(pos) * HALF + 4 * l) * 2);
    const float4 c01 = __ldg(cs), c23 = __ldg(cs + 1);
    if (qk_norm) {  // the norm weights (the same for every head of a kind) come from L1
      const float r = rsqrtf(ss / static_cast<float>(HD) + eps);
      const float4* w4 = reinterpret_cast<const float4*>(is_q ? qn : kn);
      const float4 wa = __ldg(w4 + l), wb = __ldg(w4 + LPH + l);
      a = make_float4(a.x * r * wa.x, a.y * r * wa.y, a.z * r * wa.z, a.w * r * wa.w);
      b = make_float4(b.x * r * wb.x, b.y * r * wb.y, b.z * r * wb.z, b.w * r * wb.w);
    }
    const float ra0 = a.x * c01.x - b.x * c01.y, rb0 = b.x * c01.x + a.x * c01.y;
    const float ra1 = a.y * c01.z - b.y * c01.w, rb1 = b.y * c01.z + a.y * c01.w;
    const float ra2 = a.z * c23.x - b.z * c23.y, rb2 = b.z * c23.x + a.z * c23.y;
    const float ra3 = a.w * c23.z - b.w * c23.w, rb3 = b.w * c23.z + a.w * c23.w;
    if (is_q) {
      QT* dst = q_out + (static_cast<size_t>(t) * nq + j) * HD;
      store4<QT>(dst + 4 * l, ra0, ra1, ra2, ra3);
      store4<QT>(dst + HALF + 4 * l, rb0, rb1, rb2, rb3);
    } else {
      KT* dst = kc + ((static_cast<size_t>(kv_layer) * nkv + (j - nq)) * kv_rows + kv_row) * HD;
      store4<KT>(dst + 4 * l, ra0, ra1, ra2, ra3);
      store4<KT>(dst + HALF + 4 * l, rb0, rb1, rb2, rb3);
    }
  }
}

// ------------------------------------------------------------------ ring / sink KV store
// The ring cache of the batch-attention contract (turbospark-runtime prefill.rs:
// ring_capacity R, sink_count S): position p keeps slot p when p < S, otherwise slot
// S + (p - S) mod (R - S). After the chunk's attention (which read the chunk's own keys from
// the chunk buffers), the rows a ring keeps are copied in: the sinks among the chunk's
// positions and its last R - S positions (earlier ones would be overwritten within the chunk
// anyway, so no two copies hit one slot). One warp per (token, kv head), `words` 32-bit words
// per row.
__global__ void __launch_bounds__(256) ring_store_kernel(
    const uint32_t* __restrict__ kb, const uint32_t* __restrict__ vb, int chunk_rows, int M,
    int nkv, int words, int layer, int R, int S, const int* __restrict__ start_dev, int start_host,
    uint32_t* __restrict__ kc, uint32_t* __restrict__ vc) {
  PF_TIMELINE(TL_RING_STORE);
  griddep_launch_dependents();
  griddep_wait();
  const int item = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (item >= M * nkv) return;
  const int t = item / nkv, kvh = item - (item / nkv) * nkv;
  const int start = start_dev ? *start_dev : start_host;
  const int p = start + t;
  const int W = R - S;
  if (p >= S && p < start + M - W) return;  // overwritten by a later position of this chunk
  const int slot = p < S ? p : S + (p - S) % W;
  const size_t src = (static_cast<size_t>(kvh) * chunk_rows + t) * words;
  const size_t dst = ((static_cast<size_t>(layer) * nkv + kvh) * R + slot) * words;
  for (int w = lane; w < words; w += 32) {
    kc[dst + w] = kb[src + w];
    vc[dst + w] = vb[src + w];
  }
}

// ------------------------------------------------------------------ embedding
// turbospark-runtime prefill.rs (`encode_embed_any` per token, scale 1.0): x[t] = E[id].
// An id outside [0, vocab) gets a zero row and records PF_ERR_TOKEN_OUT_OF_VOCAB.
__global__ void __launch_bounds__(256) embed_kernel(const float* __restrict__ E,
                                                    const int* __restrict__ tokens, int H,
                                                    int vocab, float* __restrict__ x,
                                                    int* __restrict__ status) {
  PF_TIMELINE(TL_EMBED);
  griddep_launch_dependents();
  griddep_wait();
  const int t = blockIdx.x;
  const int id = tokens[t];
  float4* dst = reinterpret_cast<float4*>(x + static_cast<size_t>(t) * H);
  if (id < 0 || id >= vocab) {
    for (int i = threadIdx.x; i < (H >> 2); i += blockDim.x) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (threadIdx.x == 0 && status) atomicCAS(status, 0, PF_ERR_TOKEN_OUT_OF_VOCAB);
    return;
  }
  const float4* src = reinterpret_cast<const float4*>(E + static_cast<size_t>(id) * H);
  for (int i = threadIdx.x; i < (H >> 2); i += blockDim.x) dst[i] = src[i];
}

// ------------------------------------------------------------------ tail: norm + LM head
// metal_prefill.rs `encode_full_forward_prefill` tail: `rmsnorm_weighted_v2` on the last
// row, then `dispatch_gemv_q1`. Each CTA recomputes the (one-row) norm into shared memory
// and produces the logits of one 256-row weight tile; thread r owns row r of the tile,
// so each group's 16 B of sign bits per row are read fully coalesced.
template <int WFMT>
__global__ void __launch_bounds__(256) lm_head_kernel(const float* __restrict__ x_row,
                                                      const float* __restrict__ nw, float eps,
                                                      const uint8_t* __restrict__ W, int vocab,
                                                      int H, float* __restrict__ logits) {
  PF_TIMELINE(TL_LM_HEAD);
  extern __shared__ float ys[];  // [H] normalised row, then [H/128] group sums
  __shared__ float red[32];
  griddep_launch_dependents();
  griddep_wait();
  float ss = 0.f;
  for (int i = threadIdx.x; i < H; i += blockDim.x) {
    const float v = x_row[i];
    ss += v * v;
  }
  ss = block_sum(ss, red);
  const float r = rsqrtf(ss / static_cast<float>(H) + eps);
  for (int i = threadIdx.x; i < H; i += blockDim.x) ys[i] = x_row[i] * r * nw[i];
  __syncthreads();
  const int G = H / GROUP;
  float* gsum = ys + H;
  if (WFMT == PF_W_INT4_AFFINE_G128) {
    for (int g = threadIdx.x; g < G; g += blockDim.x) {
      float s = 0.f;
      for (int k = 0; k < GROUP; ++k) s += ys[g * GROUP + k];
      gsum[g] = s;
    }
    __syncthreads();
  }
  const int tile = blockIdx.x;
  const int rr = threadIdx.x;
  const int row = tile * TILE_N + rr;
  float acc = 0.f;
  for (int g = 0; g < G; ++g) {
    const float* yg = ys + g * GROUP;
    if (WFMT == PF_W_Q1_G128) {
      const uint8_t* ch = W + (static_cast<size_t>(tile) * G + g) * Q1_CHUNK_BYTES;
      const uint2 h0 = *reinterpret_cast<const uint2*>(ch + rr * 8);
      const uint2 h1 = *reinterpret_cast<const uint2*>(ch + Q1_HALF_BYTES + rr * 8);
      const float s = __half2float(reinterpret_cast<const __half*>(ch + Q1_SCALE_OFF)[rr]);
      const uint32_t words[4] = {h0.x, h0.y, h1.x, h1.y};
      float part = 0.f;
#pragma unroll
      for (int wi = 0; wi < 4; ++wi) {
        const uint32_t Z = words[wi];
        const float* yb = yg + 32 * wi;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          // even element's negative flag sits at bit 15-i, the odd one's at bit 31-i
          part += __uint_as_float(__float_as_uint(yb[2 * i]) ^ ((Z << (16 + i)) & 0x80000000u));
          part += __uint_as_float(__float_as_uint(yb[2 * i + 1]) ^ ((Z << i) & 0x80000000u));
        }
      }
      acc += s * part;
    } else {
      const uint8_t* ch = W + (static_cast<size_t>(tile) * G + g) * I4_CHUNK_BYTES;
      const float s = __half2float(reinterpret_cast<const __half*>(ch + I4_SCALE_OFF)[rr]);
      const float z = __half2float(reinterpret_cast<const __half*>(ch + I4_ZERO_OFF)[rr]);
      float part = 0.f;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const uint4* cw = reinterpret_cast<const uint4*>(ch + h * I4_HALF_BYTES + rr * 32);
        const uint4 q0 = cw[0], q1 = cw[1];
        const uint32_t words[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
        for (int wi = 0; wi < 8; ++wi) {
          const float* yb = yg + 64 * h + 8 * wi;
#pragma unroll
          for (int p = 0; p < 4; ++p) {
            const float qe = static_cast<float>((words[wi] >> (4 * p)) & 15u);
            const float qo = static_cast<float>((words[wi] >> (16 + 4 * p)) & 15u);
            part += qe * yb[2 * p] + qo * yb[2 * p + 1];
          }
        }
      }
      acc += s * (part - z * gsum[g]);
    }
  }
  if (row < vocab) logits[row] = acc;
}

// ------------------------------------------------------------------ dequant (test)
// Runs the GEMM's own dequantisers (dq_q1_32 / dq_i4_32) on every 32-weight run of the
// packed tensor and writes w [N, K] f16 row-major. One thread per (row, 32-k run).
template <int WFMT>
__global__ void __launch_bounds__(256) dequant_kernel(const uint8_t* __restrict__ W, int64_t N,
                                                      int64_t K, __half* __restrict__ w) {
  PF_TIMELINE(TL_DEQUANT);
  const int G = static_cast<int>(K / GROUP);
  const int64_t n = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x;  // packed row
  const int run = blockIdx.y;                                             // 32-k run
  if (n >= N) return;
  const int t = static_cast<int>(n / TILE_N), r = static_cast<int>(n % TILE_N);
  const int g = run >> 2, h = (run >> 1) & 1, half32 = run & 1;
  const uint8_t* ch = W + (static_cast<size_t>(t) * G + g) * chunk_bytes(WFMT);
  uint32_t v[16];
  if (WFMT == PF_W_Q1_G128) {
    const uint32_t Z = reinterpret_cast<const uint32_t*>(ch + h * Q1_HALF_BYTES + r * 8)[half32];
    const uint32_t s16 = reinterpret_cast<const uint16_t*>(ch + Q1_SCALE_OFF)[r];
    dq_q1_32(Z, s16 | (s16 << 16), v);
  } else {
    const uint4 q = reinterpret_cast<const uint4*>(ch + h * I4_HALF_BYTES + r * 32)[half32];
    const uint16_t s16 = reinterpret_cast<const uint16_t*>(ch + I4_SCALE_OFF)[r];
    const uint16_t z16 = reinterpret_cast<const uint16_t*>(ch + I4_ZERO_OFF)[r];
    dq_i4_32(q, __half2half2(__ushort_as_half(s16)), __half2half2(__ushort_as_half(z16)), v);
  }
  uint4* dst = reinterpret_cast<uint4*>(w + n * K + static_cast<int64_t>(run) * 32);
#pragma unroll
  for (int j = 0; j < 4; ++j) dst[j] = make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
}

__global__ void set_int_kernel(int* dst, int v) {
  PF_TIMELINE(TL_SET_INT);
  griddep_launch_dependents();
  griddep_wait(); *dst = v; }

// ------------------------------------------------------------------ greedy argmax
// oxibonsai-kernels metal_prefill.rs `dispatch_argmax` (greedy decoding on the GPU; the
// verify tail dispatches it once per position with 1024 threads): one CTA of 1024 threads
// per row. The largest value wins; ties go to the lowest index (the pages do not print the
// kernel); NaN never wins, and a row with no number gives 0.
__device__ __forceinline__ void argmax_take(float v, int i, float& best, int& bi) {
  if (v > best || (v == best && i < bi)) {
    best = v;
    bi = i;
  }
}
__global__ void __launch_bounds__(1024) argmax_rows_kernel(const float* __restrict__ x, int n,
                                                           long long ld, int* __restrict__ out) {
  PF_TIMELINE(TL_ARGMAX);
  __shared__ float wb[32];
  __shared__ int wi[32];
  griddep_launch_dependents();
  griddep_wait();
  const float* row = x + static_cast<long long>(blockIdx.x) * ld;
  float best = -INFINITY;
  int bi = INT_MAX;
  for (int i = threadIdx.x; i < n; i += blockDim.x) argmax_take(row[i], i, best, bi);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ob = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    argmax_take(ob, oi, best, bi);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) {
    wb[warp] = best;
    wi[warp] = bi;
  }
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    best = lane < nw ? wb[lane] : -INFINITY;
    bi = lane < nw ? wi[lane] : INT_MAX;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      argmax_take(ob, oi, best, bi);
    }
    if (lane == 0) out[blockIdx.x] = bi == INT_MAX ? 0 : bi;
  }
}

// Exercises the bounded wait every pipelined kernel uses: one mbarrier expecting one
// arrival; with `arrive` set a thread provides it, otherwise nothing ever does and the
// wait must give up after limit_ns and record PF_ERR_DEVICE_TIMEOUT.
__global__ void wait_selftest_kernel(int* status, long long limit_ns, int arrive) {
  PF_TIMELINE(TL_WAIT_SELFTEST);
  griddep_launch_dependents();
  griddep_wait();
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 1 && arrive) mbar_arrive(b);
  if (threadIdx.x == 0) {
    const bool ok = mbar_wait(b, 0, &abort_flag, static_cast<uint64_t>(limit_ns));
    if (!ok && status) atomicCAS(status, 0, PF_ERR_DEVICE_TIMEOUT);
  }
}

}  // namespace

cudaError_t launch_rmsnorm(const float* x, const float* w, float eps, int M, int H, void* y,
                           cudaStream_t stream, float* zero, int zero_cols) {
  __half* yh = reinterpret_cast<__half*>(y);
  if (zero != nullptr && (zero_cols % 4 != 0 || reinterpret_cast<uintptr_t>(zero) % 16 != 0))
    return cudaErrorInvalidValue;
  float4* z4 = reinterpret_cast<float4*>(zero);
  const int zero4 = zero_cols / 4;
  auto reg = [&](auto kernel) {
    return launch_pdl(kernel, dim3(M), dim3(128), 0, stream, x, w, eps, H, yh, z4, zero4);
  };
  if (H % 512 == 0) {
    switch (H / 512) {
      case 1: return reg(rmsnorm_reg_kernel<1>);
      case 2: return reg(rmsnorm_reg_kernel<2>);
      case 4: return reg(rmsnorm_reg_kernel<4>);
      case 8: return reg(rmsnorm_reg_kernel<8>);
      case 16: return reg(rmsnorm_reg_kernel<16>);
      default: break;
    }
  }
  const int threads = H / 4 >= 256 ? 256 : ((H / 4 + 31) / 32) * 32;
  return launch_pdl(rmsnorm_kernel, dim3(M), dim3(threads), 0, stream, x, w, eps, H, yh, z4, zero4);
}

struct QkDst {
  int kv_layer, kv_rows, kv_by_pos;
  const int* blocks;  // paged cache: block table, else NULL
};

template <int HD, typename QT, typename KT>
static void qk_launch(const pf_config& c, const float* qkv, const float* qn, const float* kn,
                      const float* rope, QkDst d, const int* start_dev, int start_host, int M,
                      void* q, void* kc, void* vc, cudaStream_t stream) {
  const int heads = c.n_q_heads + 2 * c.n_kv_heads;
  constexpr int HPW = 32 / (HD / 8);
  const long long warps = (static_cast<long long>(M) * heads + HPW * QK_SLOTS - 1) / (HPW * QK_SLOTS);
  const int blocks = static_cast<int>((warps * 32 + 255) / 256);
  launch_pdl(qk_norm_rope_kv_kernel<HD, QT, KT>, dim3(blocks), dim3(256), 0, stream, qkv, qn, kn,
             rope, M, c.n_q_heads, c.n_kv_heads, d.kv_rows, d.kv_layer, d.kv_by_pos, start_dev,
             start_host, c.eps, c.qk_norm, reinterpret_cast<QT*>(q), reinterpret_cast<KT*>(kc),
             reinterpret_cast<KT*>(vc), d.blocks);
}

template <int HD>
static void qk_dispatch_kv(const pf_config& c, const float* qkv, const float* qn, const float* kn,
                           const float* rope, QkDst d, const int* sd, int sh, int M, void* q,
                           void* kc, void* vc, cudaStream_t st) {
  switch (c.kv_dtype) {
    case PF_KV_BF16:
      qk_launch<HD, __nv_bfloat16, __nv_bfloat16>(c, qkv, qn, kn, rope, d, sd, sh, M, q, kc, vc, st);
      break;
    case PF_KV_F16:
      qk_launch<HD, __half, __half>(c, qkv, qn, kn, rope, d, sd, sh, M, q, kc, vc, st);
      break;
    default:
      qk_launch<HD, __half, float>(c, qkv, qn, kn, rope, d, sd, sh, M, q, kc, vc, st);
      break;
  }
}

cudaError_t launch_qk_norm_rope_kv(const pf_config& c, const float* qkv, const float* q_norm,
                                   const float* k_norm, const float* rope, int kv_layer, int kv_rows,
                                   int kv_by_pos, const int* start_dev, int start_host, int M,
                                   void* q_out, void* k_dst, void* v_dst, cudaStream_t stream,
                                   const int* blocks) {
  const QkDst d{kv_layer, kv_rows, kv_by_pos, blocks};
  if (c.head_dim == 128)
    qk_dispatch_kv<128>(c, qkv, q_norm, k_norm, rope, d, start_dev, start_host, M, q_out, k_dst,
                        v_dst, stream);
  else
    qk_dispatch_kv<64>(c, qkv, q_norm, k_norm, rope, d, start_dev, start_host, M, q_out, k_dst,
                       v_dst, stream);
  return cudaGetLastError();
}

cudaError_t launch_ring_store(const pf_config& c, const void* k_chunk, const void* v_chunk,
                              int chunk_rows, int layer, const int* start_dev, int start_host, int M,
                              void* k_cache, void* v_cache, cudaStream_t stream) {
  const int words = c.head_dim * (c.kv_dtype == PF_KV_F32 ? 4 : 2) / 4;
  const int rows = M * c.n_kv_heads;
  return launch_pdl(ring_store_kernel, dim3((rows + 7) / 8), dim3(256), 0, stream,
                    static_cast<const uint32_t*>(k_chunk), static_cast<const uint32_t*>(v_chunk),
                    chunk_rows, M, c.n_kv_heads, words, layer, c.ring_capacity, c.sink_count,
                    start_dev, start_host, static_cast<uint32_t*>(k_cache),
                    static_cast<uint32_t*>(v_cache));
}

cudaError_t launch_embed(const float* E, const int* tokens, int M, int H, int vocab, float* x,
                         int* status, cudaStream_t stream) {
  return launch_pdl(embed_kernel, dim3(M), dim3(256), 0, stream, E, tokens, H, vocab, x, status);
}

// Q1 LM head (P1 section "LM-head GEMV"): logits[n] = sum_g s[n,g] sum_{k in g} (+-y_k) with
// y = RMSNorm(x_row). Each 32-bit sign word holds 8 nibbles; nibble n of word u covers four
// elements of one parity (even for n < 4, odd for n >= 4, see the packed layout), so the 16
// signed sums of those four y values are tabulated once per CTA (64 KB for H = 4096) and
// every nibble of every row costs one table lookup and one add. A warp's 32 rows read the
// same nibble table: at most 16 distinct words in distinct banks, no conflicts.
__device__ __forceinline__ int q1_nibble_elem(int n, int b) {  // element of bit b of nibble n
  return n < 4 ? 30 - 8 * n - 2 * b : 31 - 8 * (n - 4) - 2 * b;
}

// Table value for nibble N of sign word Z, the word's table at shared address `base`
// (512-B aligned): one shift, one LOP3 merging (nibble * 4) into the address, one load with
// the nibble's 64-B slot as immediate offset.
template <int N>
__device__ __forceinline__ float q1_lut_ld(uint32_t Z, uint32_t base) {
  const uint32_t sh = N == 0 ? (Z << 2) : (Z >> (4 * N - 2));
  uint32_t a;
  asm("lop3.b32 %0, %1, 0x3C, %2, 0xEA;" : "=r"(a) : "r"(sh), "r"(base));
  float t;
  // volatile: the table is written before a barrier; the load must stay after it
  asm volatile("ld.shared.f32 %0, [%1+%2];" : "=f"(t) : "r"(a), "n"(64 * N));
  return t;
}

__global__ void __launch_bounds__(512) lm_head_q1_kernel(const float* __restrict__ x_row,
                                                         const float* __restrict__ nw, float eps,
                                                         const uint8_t* __restrict__ W, int vocab,
                                                         int H, float* __restrict__ logits) {
  PF_TIMELINE(TL_LM_HEAD_Q1);
  // [H/32 words][8 nibbles][16 values] (each word's table 512-B aligned), then y [H], then [256]
  extern __shared__ __align__(1024) float lut[];
  __shared__ float red[32];
  float* ys = lut + (H / 32) * 8 * 16;
  float* half_sum = ys + H;
  const uint32_t lut_s = smem_u32(lut);
  griddep_launch_dependents();
  griddep_wait();
  float ss = 0.f;
  for (int i = threadIdx.x; i < H; i += blockDim.x) {
    const float v = x_row[i];
    ss += v * v;
  }
  ss = block_sum(ss, red);
  const float r = rsqrtf(ss / static_cast<float>(H) + eps);
  for (int i = threadIdx.x; i < H; i += blockDim.x) ys[i] = x_row[i] * r * nw[i];
  __syncthreads();
  // table entry (u, n, v): sum over the nibble's four elements, negated where v's bit is set.
  // One thread fills one nibble's 16 entries: the signed sums of its elements (0, 1) and
  // (2, 3) for the four sign patterns of each pair, then every entry is one pair sum plus
  // the other.
  for (int t = threadIdx.x; t < (H / 32) * 8; t += blockDim.x) {
    const int n = t & 7;
    const float* yu = ys + 32 * (t >> 3);
    const float y0 = yu[q1_nibble_elem(n, 0)], y1 = yu[q1_nibble_elem(n, 1)];
    const float y2 = yu[q1_nibble_elem(n, 2)], y3 = yu[q1_nibble_elem(n, 3)];
    const float lo[4] = {y0 + y1, y1 - y0, y0 - y1, -y0 - y1};  // bits 0, 1 of v
    const float hi[4] = {y2 + y3, y3 - y2, y2 - y3, -y2 - y3};  // bits 2, 3 of v
    float4* dst = reinterpret_cast<float4*>(lut + 16 * t);
#pragma unroll
    for (int q = 0; q < 4; ++q) dst[q] = make_float4(lo[0] + hi[q], lo[1] + hi[q], lo[2] + hi[q], lo[3] + hi[q]);
  }
  __syncthreads();
  // two threads per weight row, each over half of the groups (more loads in flight per SM)
  const int G = H / GROUP;
  const int tiles = (vocab + TILE_N - 1) / TILE_N;
  const int rr = threadIdx.x & (TILE_N - 1);
  const int part = threadIdx.x >> 8;
  const int g0 = part * (G / 2), g1 = part ? G : G / 2;
  // one group's packed weights of this thread's row: two sign-word pairs and the scale
  struct GroupW {
    uint2 h0, h1;
    unsigned short s;
  };
  for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x) {
    const uint8_t* tw = W + static_cast<size_t>(tile) * G * Q1_CHUNK_BYTES;
    auto load = [&](int g, GroupW& d) {
      const uint8_t* ch = tw + static_cast<size_t>(g) * Q1_CHUNK_BYTES;
      d.h0 = __ldg(reinterpret_cast<const uint2*>(ch + rr * 8));
      d.h1 = __ldg(reinterpret_cast<const uint2*>(ch + Q1_HALF_BYTES + rr * 8));
      d.s = __ldg(reinterpret_cast<const unsigned short*>(ch + Q1_SCALE_OFF) + rr);
    };
    float acc = 0.f;
    auto add = [&](int g, const GroupW& d) {
      const uint32_t words[4] = {d.h0.x, d.h0.y, d.h1.x, d.h1.y};
      float p[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        // word w's table starts 512-B aligned, so (nibble * 4) merges into the address with
        // one LOP3 and the nibble's 64-B slot is the load's immediate offset
        const uint32_t base = lut_s + (4 * g + w) * 512;
        const uint32_t Z = words[w];
        p[0] += q1_lut_ld<0>(Z, base);
        p[1] += q1_lut_ld<1>(Z, base);
        p[2] += q1_lut_ld<2>(Z, base);
        p[3] += q1_lut_ld<3>(Z, base);
        p[0] += q1_lut_ld<4>(Z, base);
        p[1] += q1_lut_ld<5>(Z, base);
        p[2] += q1_lut_ld<6>(Z, base);
        p[3] += q1_lut_ld<7>(Z, base);
      }
      acc = fmaf(__half2float(__ushort_as_half(d.s)), (p[0] + p[1]) + (p[2] + p[3]), acc);
    };
    // four groups in flight while the previous four are added
    GroupW cur[4], nxt[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      if (g0 + i < g1) load(g0 + i, cur[i]);
    for (int g = g0; g < g1; g += 4) {
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (g + 4 + i < g1) load(g + 4 + i, nxt[i]);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        if (g + i < g1) add(g + i, cur[i]);
#pragma unroll
      for (int i = 0; i < 4; ++i) cur[i] = nxt[i];
    }
    if (part) half_sum[rr] = acc;
    __syncthreads();
    const int row = tile * TILE_N + rr;
    if (!part && row < vocab) logits[row] = acc + half_sum[rr];
    __syncthreads();
  }
}

cudaError_t launch_lm_head(int wfmt, const float* x_row, const float* norm_w, float eps,
                           const uint8_t* packed, int vocab, int H, float* logits,
                           cudaStream_t stream) {
  const int tiles = static_cast<int>(padded_rows(vocab) / TILE_N);
  const size_t smem = (static_cast<size_t>(H) + H / GROUP) * sizeof(float);
  // H % 32 == 0 (H % 128 is checked); table + y row: 68 KB at H = 4096, two CTAs per SM
  const size_t smem_q1 = (static_cast<size_t>(H / 32) * 8 * 16 + H + TILE_N) * sizeof(float);
  if (wfmt == PF_W_Q1_G128 && smem_q1 <= 227 * 1024) {
    if (smem_q1 > 48 * 1024)
      cudaFuncSetAttribute(lm_head_q1_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem_q1));
    const int ctas = std::min(tiles, 2 * device_sm_count());
    launch_pdl(lm_head_q1_kernel, dim3(ctas), dim3(512), smem_q1, stream, x_row, norm_w, eps, packed,
               vocab, H, logits);
  } else if (wfmt == PF_W_Q1_G128) {  // rows too wide for the table: one row per thread
    if (smem > 48 * 1024)
      cudaFuncSetAttribute(lm_head_kernel<PF_W_Q1_G128>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    launch_pdl(lm_head_kernel<PF_W_Q1_G128>, dim3(tiles), dim3(256), smem, stream, x_row, norm_w,
               eps, packed, vocab, H, logits);
  } else {
    if (smem > 48 * 1024)
      cudaFuncSetAttribute(lm_head_kernel<PF_W_INT4_AFFINE_G128>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    launch_pdl(lm_head_kernel<PF_W_INT4_AFFINE_G128>, dim3(tiles), dim3(256), smem, stream, x_row,
               norm_w, eps, packed, vocab, H, logits);
  }
  return cudaGetLastError();
}

cudaError_t launch_dequant(int wfmt, const uint8_t* packed, int64_t N, int64_t K, void* w,
                           cudaStream_t stream) {
  dim3 grid(static_cast<unsigned>((N + 255) / 256), static_cast<unsigned>(K / 32));
  if (wfmt == PF_W_Q1_G128)
    dequant_kernel<PF_W_Q1_G128><<<grid, 256, 0, stream>>>(packed, N, K,
                                                           reinterpret_cast<__half*>(w));
  else
    dequant_kernel<PF_W_INT4_AFFINE_G128><<<grid, 256, 0, stream>>>(packed, N, K,
                                                                    reinterpret_cast<__half*>(w));
  return cudaGetLastError();
}

cudaError_t launch_argmax_rows(const float* x, int rows, int n, long long ld, int* out, cudaStream_t stream) {
  if (rows <= 0 || n <= 0 || ld < n) return cudaErrorInvalidValue;
  return launch_pdl(argmax_rows_kernel, dim3(rows), dim3(1024), 0, stream, x, n, ld, out);
}

cudaError_t launch_set_int(int* dst, int value, cudaStream_t stream) {
  return launch_pdl(set_int_kernel, dim3(1), dim3(1), 0, stream, dst, value);
}

cudaError_t launch_wait_selftest(int* status, long long limit_ns, int arrive, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(status, limit_ns, arrive);
  return cudaGetLastError();
}

}  // namespace pf

PF_TIMELINE_SETTER(kernels)
