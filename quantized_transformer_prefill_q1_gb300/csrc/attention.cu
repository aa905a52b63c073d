// attention.cu — causal GQA attention for a chunk of query rows over the KV cache.
//
// The pages compute attention one token at a time (oxibonsai-kernels metal_prefill.rs
// `encode_layer_prefill` section 3: scores over seq_len = pos + 1 cache entries scaled by
// inv_sqrt_hd, softmax, weighted sum of V; q head h reads kv head h / heads_per_group) and
// turbospark-runtime prefill.rs batches the query rows of a chunk in one
// `encode_attention_decode_batch`. Here one CTA takes the query rows of one kv head's
// group for a run of consecutive tokens (row = token * G + head-in-group, so every row of
// the CTA shares the K/V tiles), streams 64-key tiles of the cache through shared memory
// with an online (running max / running sum) softmax, and masks keys beyond each row's
// own position. Tensor-core MMAs are m16n8k16 with f32 accumulation.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace pf {
namespace {

constexpr int BR = 64;  // query rows per CTA (4 warps x 16)
constexpr int BC = 64;  // keys per tile
constexpr int THREADS = 128;

template <typename T>
struct MmaName;
template <>
struct MmaName<__nv_bfloat16> {
  static constexpr bool bf16 = true;
};
template <>
struct MmaName<__half> {
  static constexpr bool bf16 = false;
};

template <typename T>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  if constexpr (MmaName<T>::bf16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

template <typename T>
__device__ __forceinline__ uint32_t pack2(float a, float b);
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Byte offset of 16-B chunk c of row r in a [rows][HD] 16-bit tile (XOR swizzle on the
// low three chunk bits, so the 8 rows an ldmatrix reads hit 8 different bank groups).
template <int HD>
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return static_cast<uint32_t>(r * (HD * 2) + ((c ^ (r & 7)) << 4));
}

// Loads rows [j0, j0 + BC) of one kv head's cache into a swizzled tile; rows at or past
// kv_len are zero (their V must not meet a zero probability as NaN in the MMA).
template <int HD, typename T, typename KT>
__device__ __forceinline__ void load_kv_tile(uint8_t* tile, const KT* __restrict__ src, int j0,
                                             int kv_len) {
  constexpr int CH = HD / 8;  // 16-B chunks (of T) per row
  for (int i = threadIdx.x; i < BC * CH; i += THREADS) {
    const int r = i / CH, c = i - (i / CH) * CH;
    const int j = j0 + r;
    uint8_t* dst = tile + swz<HD>(r, c);
    if (j >= kv_len) {
      *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
    } else if constexpr (sizeof(KT) == 2) {
      cp_async16(smem_addr(dst), src + static_cast<size_t>(j) * HD + c * 8);
    } else {
      const float4* s4 = reinterpret_cast<const float4*>(src + static_cast<size_t>(j) * HD + c * 8);
      const float4 a = s4[0], b = s4[1];
      *reinterpret_cast<uint4*>(dst) =
          make_uint4(pack2<T>(a.x, a.y), pack2<T>(a.z, a.w), pack2<T>(b.x, b.y), pack2<T>(b.z, b.w));
    }
  }
}

template <int HD, typename T, typename KT>
__global__ void __launch_bounds__(THREADS) attention_kernel(
    const T* __restrict__ q, const KT* __restrict__ kc, const KT* __restrict__ vc, int M, int nq,
    int nkv, int max_seq, int layer, const int* __restrict__ start_dev, int start_host,
    float scale_log2, __half* __restrict__ out) {
  PF_TIMELINE(TL_ATTENTION_F32);
  extern __shared__ __align__(128) uint8_t sm[];
  uint8_t* Qs = sm;
  uint8_t* Ks = Qs + BR * HD * 2;
  uint8_t* Vs = Ks + 2 * BC * HD * 2;
  constexpr int TILE = BC * HD * 2;
  constexpr int CH = HD / 8;

  griddep_launch_dependents();
  griddep_wait();
  const int G = nq / nkv;
  const int BT = BR / G;  // tokens per CTA
  const int n_ttiles = (M + BT - 1) / BT;
  const int tt = n_ttiles - 1 - static_cast<int>(blockIdx.x);  // longest rows first
  const int kvh = blockIdx.y;
  const int t0 = tt * BT;
  const int start = start_dev ? *start_dev : start_host;
  const int kv_len = start + min(t0 + BT, M);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const KT* kbase = kc + (static_cast<size_t>(layer) * nkv + kvh) * max_seq * HD;
  const KT* vbase = vc + (static_cast<size_t>(layer) * nkv + kvh) * max_seq * HD;

  // Q tile: row r = token (t0 + r / G), head kvh * G + r % G
  for (int i = threadIdx.x; i < BR * CH; i += THREADS) {
    const int r = i / CH, c = i - (i / CH) * CH;
    const int t = t0 + r / G;
    const int h = kvh * G + r % G;
    uint8_t* dst = Qs + swz<HD>(r, c);
    if (t < M)
      cp_async16(smem_addr(dst), q + (static_cast<size_t>(t) * nq + h) * HD + c * 8);
    else
      *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
  }
  load_kv_tile<HD, T, KT>(Ks, kbase, 0, kv_len);
  load_kv_tile<HD, T, KT>(Vs, vbase, 0, kv_len);
  cp_async_commit();
  cp_async_wait_all();
  __syncthreads();

  // Q fragments for this warp's 16 rows
  uint32_t qa[HD / 16][4];
  {
    const int r = warp * 16 + (lane & 15);
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) ldsm_x4(smem_addr(Qs + swz<HD>(r, 2 * kk + (lane >> 4))), qa[kk]);
  }

  // positions of the two rows this thread accumulates (rows g and g + 8 of the warp)
  const int g = lane >> 2, tq = lane & 3;
  const int pos0 = start + t0 + (warp * 16 + g) / G;
  const int pos1 = start + t0 + (warp * 16 + g + 8) / G;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

  const int n_tiles = (kv_len + BC - 1) / BC;
  for (int it = 0; it < n_tiles; ++it) {
    const int buf = it & 1;
    if (it + 1 < n_tiles) {  // prefetch the next tile into the other buffer
      load_kv_tile<HD, T, KT>(Ks + (buf ^ 1) * TILE, kbase, (it + 1) * BC, kv_len);
      load_kv_tile<HD, T, KT>(Vs + (buf ^ 1) * TILE, vbase, (it + 1) * BC, kv_len);
      cp_async_commit();
    }
    const uint8_t* Kt = Ks + buf * TILE;
    const uint8_t* Vt = Vs + buf * TILE;
    const int j0 = it * BC;

    float s[BC / 8][4];
#pragma unroll
    for (int i = 0; i < BC / 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < HD / 16; ++kk) {
#pragma unroll
      for (int nb2 = 0; nb2 < BC / 16; ++nb2) {
        uint32_t b[4];
        const int key = nb2 * 16 + (lane & 7) + ((lane >> 4) << 3);
        ldsm_x4(smem_addr(Kt + swz<HD>(key, 2 * kk + ((lane >> 3) & 1))), b);
        mma16816<T>(s[2 * nb2], qa[kk], b[0], b[1]);
        mma16816<T>(s[2 * nb2 + 1], qa[kk], b[2], b[3]);
      }
    }
    // scale (log2 domain) and causal mask
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nb = 0; nb < BC / 8; ++nb) {
      const int kj = j0 + nb * 8 + 2 * tq;
      s[nb][0] = (kj <= pos0) ? s[nb][0] * scale_log2 : -INFINITY;
      s[nb][1] = (kj + 1 <= pos0) ? s[nb][1] * scale_log2 : -INFINITY;
      s[nb][2] = (kj <= pos1) ? s[nb][2] * scale_log2 : -INFINITY;
      s[nb][3] = (kj + 1 <= pos1) ? s[nb][3] * scale_log2 : -INFINITY;
      mx0 = fmaxf(mx0, fmaxf(s[nb][0], s[nb][1]));
      mx1 = fmaxf(mx1, fmaxf(s[nb][2], s[nb][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float al0 = exp2f(m0 - mn0), al1 = exp2f(m1 - mn1);
    m0 = mn0;
    m1 = mn1;
    float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
    for (int nb = 0; nb < BC / 8; ++nb) {
      s[nb][0] = exp2f(s[nb][0] - mn0);
      s[nb][1] = exp2f(s[nb][1] - mn0);
      s[nb][2] = exp2f(s[nb][2] - mn1);
      s[nb][3] = exp2f(s[nb][3] - mn1);
      rs0 += s[nb][0] + s[nb][1];
      rs1 += s[nb][2] + s[nb][3];
    }
    l0 = l0 * al0 + rs0;
    l1 = l1 * al1 + rs1;
#pragma unroll
    for (int i = 0; i < HD / 8; ++i) {
      o[i][0] *= al0;
      o[i][1] *= al0;
      o[i][2] *= al1;
      o[i][3] *= al1;
    }
    // O += P V
#pragma unroll
    for (int kk = 0; kk < BC / 16; ++kk) {
      uint32_t a[4];
      a[0] = pack2<T>(s[2 * kk][0], s[2 * kk][1]);
      a[1] = pack2<T>(s[2 * kk][2], s[2 * kk][3]);
      a[2] = pack2<T>(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      a[3] = pack2<T>(s[2 * kk + 1][2], s[2 * kk + 1][3]);
      const int key = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
      for (int db2 = 0; db2 < HD / 16; ++db2) {
        uint32_t b[4];
        ldsm_x4_t(smem_addr(Vt + swz<HD>(key, 2 * db2 + (lane >> 4))), b);
        mma16816<T>(o[2 * db2], a, b[0], b[1]);
        mma16816<T>(o[2 * db2 + 1], a, b[2], b[3]);
      }
    }
    cp_async_wait_all();
    __syncthreads();
  }

  // quad-reduce the row sums (each thread holds a partial over its columns)
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const float inv0 = 1.f / l0, inv1 = 1.f / l1;
  const int r0 = warp * 16 + g, r1 = r0 + 8;
  const int ta = t0 + r0 / G, tb = t0 + r1 / G;
  const int ha = kvh * G + r0 % G, hb = kvh * G + r1 % G;
#pragma unroll
  for (int db = 0; db < HD / 8; ++db) {
    const int d = db * 8 + 2 * tq;
    if (ta < M)
      *reinterpret_cast<__half2*>(out + (static_cast<size_t>(ta) * nq + ha) * HD + d) =
          __floats2half2_rn(o[db][0] * inv0, o[db][1] * inv0);
    if (tb < M)
      *reinterpret_cast<__half2*>(out + (static_cast<size_t>(tb) * nq + hb) * HD + d) =
          __floats2half2_rn(o[db][2] * inv1, o[db][3] * inv1);
  }
}

template <int HD, typename T, typename KT>
cudaError_t launch_t(const pf_config& c, const void* q, const void* kc, const void* vc, int layer,
                     const int* start_dev, int start_host, int M, void* out, cudaStream_t st) {
  const int G = c.n_q_heads / c.n_kv_heads;
  const int BT = BR / G;
  const int smem = (BR + 4 * BC) * HD * 2;
  auto kern = attention_kernel<HD, T, KT>;
  dim3 grid((M + BT - 1) / BT, c.n_kv_heads);
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(HD));
  return launch_pdl(kern, grid, dim3(THREADS), static_cast<size_t>(smem), st,
                    reinterpret_cast<const T*>(q), reinterpret_cast<const KT*>(kc),
                    reinterpret_cast<const KT*>(vc), M, c.n_q_heads, c.n_kv_heads, c.max_seq, layer,
                    start_dev, start_host, scale_log2, reinterpret_cast<__half*>(out));
}

template <int HD>
cudaError_t dispatch_kv(const pf_config& c, const void* q, const void* kc, const void* vc,
                        int layer, const int* sd, int sh, int M, void* out, cudaStream_t st) {
  switch (c.kv_dtype) {
    case PF_KV_BF16:
      return launch_t<HD, __nv_bfloat16, __nv_bfloat16>(c, q, kc, vc, layer, sd, sh, M, out, st);
    case PF_KV_F16:
      return launch_t<HD, __half, __half>(c, q, kc, vc, layer, sd, sh, M, out, st);
    default:
      return launch_t<HD, __half, float>(c, q, kc, vc, layer, sd, sh, M, out, st);
  }
}

}  // namespace

template <int HD, typename T, typename KT>
cudaError_t set_attr() {
  return cudaFuncSetAttribute(attention_kernel<HD, T, KT>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, (BR + 4 * BC) * HD * 2);
}

cudaError_t prepare_attention_kernels() {
  cudaError_t e = cudaSuccess, r;
  if ((r = set_attr<128, __nv_bfloat16, __nv_bfloat16>()) != cudaSuccess) e = r;
  if ((r = set_attr<128, __half, __half>()) != cudaSuccess) e = r;
  if ((r = set_attr<128, __half, float>()) != cudaSuccess) e = r;
  if ((r = set_attr<64, __nv_bfloat16, __nv_bfloat16>()) != cudaSuccess) e = r;
  if ((r = set_attr<64, __half, __half>()) != cudaSuccess) e = r;
  if ((r = set_attr<64, __half, float>()) != cudaSuccess) e = r;
  return e;
}

// Routes 16-bit caches to the tcgen05 kernel (attention_tc.cu); f32 caches stage K/V
// through registers into the m16n8k16 kernel above.
cudaError_t launch_attention(const AttnArgs& a, cudaStream_t stream) {
  const pf_config& c = *a.c;
  if (attention_tc_supported(c)) return launch_attention_tc(a, stream);
  if (c.ring_capacity > 0 || a.n_split > 1) return cudaErrorInvalidValue;  // tensor-core kernel only
  if (c.head_dim == 128)
    return dispatch_kv<128>(c, a.q, a.k_cache, a.v_cache, a.layer, a.start_dev, a.start_host, a.M,
                            a.out, stream);
  return dispatch_kv<64>(c, a.q, a.k_cache, a.v_cache, a.layer, a.start_dev, a.start_host, a.M, a.out,
                         stream);
}

}  // namespace pf

PF_TIMELINE_SETTER(attention)
