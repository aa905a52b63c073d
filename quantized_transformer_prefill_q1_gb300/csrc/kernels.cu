// kernels.cu — the HBM-bound steps of the prefill path: RMSNorm, fused QK-norm + RoPE +
// KV-store, embedding gather, the final-norm + LM-head GEMV, a split-K SwiGLU, and the
// stand-alone dequantiser used to check unpacking bit-exactly.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "dequant.cuh"
#include "ptx.cuh"

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

// ------------------------------------------------------------------ RMSNorm
// oxibonsai-kernels metal_prefill.rs `encode_layer_prefill` sections 1 and 5
// (`dispatch_batched_rmsnorm`): y[m, :] = x[m, :] * w / sqrt(mean(x[m, :]^2) + eps),
// f32 in, f16 out (the next GEMM's operand). One CTA per row, 128-bit loads.
__global__ void __launch_bounds__(256) rmsnorm_kernel(const float* __restrict__ x,
                                                      const float* __restrict__ w, float eps,
                                                      int H, __half* __restrict__ y) {
  __shared__ float red[32];
  const int row = blockIdx.x;
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

// ------------------------------------------------------------------ QK-norm + RoPE + KV
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

// One warp per (token, head) of the fused QKV output, heads ordered Q | K | V.
// metal_prefill.rs `encode_layer_prefill` section 3 (fused_qk_norm, fused_qk_rope,
// fused_kv_store) and metal_full_layer.rs `dispatch_fused_qk_norm_rope`, batched over the
// chunk: Q and K heads get an RMSNorm over head_dim (weights w_q / w_k, the layer eps)
// when enabled, then rotate-half RoPE at position start + t from the (cos, sin) table;
// Q goes to q_out [M, nq, hd], K to the cache slot [layer, kvh, pos, :], and V is copied
// unchanged to its slot. Cache layout of metal_full_layer.rs `GpuKvCache`:
// [n_layers][nkv][max_seq][hd].
template <int HD, typename QT, typename KT>
__global__ void __launch_bounds__(256) qk_norm_rope_kv_kernel(
    const float* __restrict__ qkv, const float* __restrict__ qn, const float* __restrict__ kn,
    const float* __restrict__ rope, int M, int nq, int nkv, int max_seq, int layer,
    const int* __restrict__ start_dev, int start_host, float eps, int qk_norm,
    QT* __restrict__ q_out, KT* __restrict__ kc, KT* __restrict__ vc) {
  constexpr int HALF = HD / 2;
  constexpr int E = HALF / 32;  // elements per lane in each half
  const int heads = nq + 2 * nkv;
  const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  const int t = gw / heads;
  const int j = gw - t * heads;
  if (t >= M) return;
  const int start = start_dev ? *start_dev : start_host;
  const int pos = start + t;
  const float* src = qkv + (static_cast<size_t>(t) * heads + j) * HD;
  float a[E], b[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    a[e] = src[lane * E + e];
    b[e] = src[HALF + lane * E + e];
  }
  if (j >= nq + nkv) {  // V head: straight to the cache
    const int kvh = j - nq - nkv;
    KT* dst = vc + ((static_cast<size_t>(layer) * nkv + kvh) * max_seq + pos) * HD;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      dst[lane * E + e] = to_elem<KT>(a[e]);
      dst[HALF + lane * E + e] = to_elem<KT>(b[e]);
    }
    return;
  }
  const bool is_q = j < nq;
  if (qk_norm) {
    float ss = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) ss += a[e] * a[e] + b[e] * b[e];
    ss = warp_sum(ss);
    const float r = rsqrtf(ss / static_cast<float>(HD) + eps);
    const float* w = is_q ? qn : kn;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      a[e] = a[e] * r * w[lane * E + e];
      b[e] = b[e] * r * w[HALF + lane * E + e];
    }
  }
  const float2* cs = reinterpret_cast<const float2*>(rope) + static_cast<size_t>(pos) * HALF;
  float ra[E], rb[E];
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const float2 c = cs[lane * E + e];  // (cos, sin)
    ra[e] = a[e] * c.x - b[e] * c.y;
    rb[e] = b[e] * c.x + a[e] * c.y;
  }
  if (is_q) {
    QT* dst = q_out + (static_cast<size_t>(t) * nq + j) * HD;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      dst[lane * E + e] = to_elem<QT>(ra[e]);
      dst[HALF + lane * E + e] = to_elem<QT>(rb[e]);
    }
  } else {
    const int kvh = j - nq;
    KT* dst = kc + ((static_cast<size_t>(layer) * nkv + kvh) * max_seq + pos) * HD;
#pragma unroll
    for (int e = 0; e < E; ++e) {
      dst[lane * E + e] = to_elem<KT>(ra[e]);
      dst[HALF + lane * E + e] = to_elem<KT>(rb[e]);
    }
  }
}

// ------------------------------------------------------------------ embedding
// turbospark-runtime prefill.rs (`encode_embed_any` per token, scale 1.0): x[t] = E[id].
// An id outside [0, vocab) gets a zero row and records PF_ERR_TOKEN_OUT_OF_VOCAB.
__global__ void __launch_bounds__(256) embed_kernel(const float* __restrict__ E,
                                                    const int* __restrict__ tokens, int H,
                                                    int vocab, float* __restrict__ x,
                                                    int* __restrict__ status) {
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
  extern __shared__ float ys[];  // [H] normalised row, then [H/128] group sums
  __shared__ float red[32];
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

// ------------------------------------------------------------------ split-K SwiGLU
// Used when the gate_up GEMM is split along K (small chunks): gu holds the f32 GEMM
// output in packed-row order, where each 128-column tile is 64 gate columns then the 64
// matching up columns. out[m, f] = silu(gate) * up, f16.
__global__ void swiglu_f32_kernel(const float* __restrict__ gu, int M, int I,
                                  __half* __restrict__ out) {
  const size_t idx = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<size_t>(M) * I) return;
  const int m = static_cast<int>(idx / I);
  const int f = static_cast<int>(idx - static_cast<size_t>(m) * I);
  const int t = f >> 6, r = f & 63;
  const size_t ld = 2 * static_cast<size_t>(I);
  const float g = gu[m * ld + t * 128 + r];
  const float u = gu[m * ld + t * 128 + 64 + r];
  out[idx] = __float2half_rn(g / (1.0f + __expf(-g)) * u);
}

// ------------------------------------------------------------------ dequant (test)
// Runs the GEMM's own dequantisers (dq_q1_32 / dq_i4_32) on every 32-weight run of the
// packed tensor and writes w [N, K] f16 row-major. One thread per (row, 32-k run).
template <int WFMT>
__global__ void __launch_bounds__(256) dequant_kernel(const uint8_t* __restrict__ W, int64_t N,
                                                      int64_t K, __half* __restrict__ w) {
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

__global__ void set_int_kernel(int* dst, int v) { *dst = v; }

// Exercises the bounded wait every pipelined kernel uses: one mbarrier expecting one
// arrival; with `arrive` set a thread provides it, otherwise nothing ever does and the
// wait must give up after limit_ns and record PF_ERR_DEVICE_TIMEOUT.
__global__ void wait_selftest_kernel(int* status, long long limit_ns, int arrive) {
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
                           cudaStream_t stream) {
  const int threads = H / 4 >= 256 ? 256 : ((H / 4 + 31) / 32) * 32;
  rmsnorm_kernel<<<M, threads, 0, stream>>>(x, w, eps, H, reinterpret_cast<__half*>(y));
  return cudaGetLastError();
}

template <int HD, typename QT, typename KT>
static void qk_launch(const pf_config& c, const float* qkv, const float* qn, const float* kn,
                      const float* rope, int layer, const int* start_dev, int start_host, int M,
                      void* q, void* kc, void* vc, cudaStream_t stream) {
  const int heads = c.n_q_heads + 2 * c.n_kv_heads;
  const long long warps = static_cast<long long>(M) * heads;
  const int blocks = static_cast<int>((warps * 32 + 255) / 256);
  qk_norm_rope_kv_kernel<HD, QT, KT><<<blocks, 256, 0, stream>>>(
      qkv, qn, kn, rope, M, c.n_q_heads, c.n_kv_heads, c.max_seq, layer, start_dev, start_host,
      c.eps, c.qk_norm, reinterpret_cast<QT*>(q), reinterpret_cast<KT*>(kc),
      reinterpret_cast<KT*>(vc));
}

template <int HD>
static void qk_dispatch_kv(const pf_config& c, const float* qkv, const float* qn, const float* kn,
                           const float* rope, int layer, const int* sd, int sh, int M, void* q,
                           void* kc, void* vc, cudaStream_t st) {
  switch (c.kv_dtype) {
    case PF_KV_BF16:
      qk_launch<HD, __nv_bfloat16, __nv_bfloat16>(c, qkv, qn, kn, rope, layer, sd, sh, M, q, kc, vc, st);
      break;
    case PF_KV_F16:
      qk_launch<HD, __half, __half>(c, qkv, qn, kn, rope, layer, sd, sh, M, q, kc, vc, st);
      break;
    default:
      qk_launch<HD, __half, float>(c, qkv, qn, kn, rope, layer, sd, sh, M, q, kc, vc, st);
      break;
  }
}

cudaError_t launch_qk_norm_rope_kv(const pf_config& c, const float* qkv, const float* q_norm,
                                   const float* k_norm, const float* rope, int layer,
                                   const int* start_dev, int start_host, int M, void* q_out,
                                   void* k_cache, void* v_cache, cudaStream_t stream) {
  if (c.head_dim == 128)
    qk_dispatch_kv<128>(c, qkv, q_norm, k_norm, rope, layer, start_dev, start_host, M, q_out,
                        k_cache, v_cache, stream);
  else
    qk_dispatch_kv<64>(c, qkv, q_norm, k_norm, rope, layer, start_dev, start_host, M, q_out,
                       k_cache, v_cache, stream);
  return cudaGetLastError();
}

cudaError_t launch_embed(const float* E, const int* tokens, int M, int H, int vocab, float* x,
                         int* status, cudaStream_t stream) {
  embed_kernel<<<M, 256, 0, stream>>>(E, tokens, H, vocab, x, status);
  return cudaGetLastError();
}

cudaError_t launch_lm_head(int wfmt, const float* x_row, const float* norm_w, float eps,
                           const uint8_t* packed, int vocab, int H, float* logits,
                           cudaStream_t stream) {
  const int tiles = static_cast<int>(padded_rows(vocab) / TILE_N);
  const size_t smem = (static_cast<size_t>(H) + H / GROUP) * sizeof(float);
  if (wfmt == PF_W_Q1_G128) {
    if (smem > 48 * 1024)
      cudaFuncSetAttribute(lm_head_kernel<PF_W_Q1_G128>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    lm_head_kernel<PF_W_Q1_G128><<<tiles, 256, smem, stream>>>(x_row, norm_w, eps, packed, vocab,
                                                              H, logits);
  } else {
    if (smem > 48 * 1024)
      cudaFuncSetAttribute(lm_head_kernel<PF_W_INT4_AFFINE_G128>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    lm_head_kernel<PF_W_INT4_AFFINE_G128><<<tiles, 256, smem, stream>>>(x_row, norm_w, eps,
                                                                       packed, vocab, H, logits);
  }
  return cudaGetLastError();
}

cudaError_t launch_swiglu_f32(const float* gu, int M, int I, void* out, cudaStream_t stream) {
  const size_t n = static_cast<size_t>(M) * I;
  swiglu_f32_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, stream>>>(
      gu, M, I, reinterpret_cast<__half*>(out));
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

cudaError_t launch_set_int(int* dst, int value, cudaStream_t stream) {
  set_int_kernel<<<1, 1, 0, stream>>>(dst, value);
  return cudaGetLastError();
}

cudaError_t launch_wait_selftest(int* status, long long limit_ns, int arrive, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(status, limit_ns, arrive);
  return cudaGetLastError();
}

}  // namespace pf
