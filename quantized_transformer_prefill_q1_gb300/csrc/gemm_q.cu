// gemm_q.cu — quantised GEMM on the 5th-generation tensor cores (tcgen05 / TMEM).
//
// out[m, n] (+)= sum_k a[m, k] * w[n, k] with a = f16 activations [M, K] (the RMSNorm /
// SwiGLU / attention outputs) and w a packed Q1 or INT4-affine weight [N, K]. This is
// the batched projection of oxibonsai-kernels metal_prefill.rs `encode_layer_prefill`:
// section 2 (QKV GEMM, plain store), sections 4 and 7 (O / down GEMM with the residual
// add fused, `dispatch_gemm_q1_v7_residual`) and section 6 (gate+up GEMM with SwiGLU
// fused, `dispatch_fused_gate_up_swiglu_gemm`).
//
// One CTA computes a 128 (tokens) x 256 (weight rows) tile over a K range:
//   warp 0      TMA producer: activation tile (128 x 64, 128-B swizzle) + the packed
//               weight block of the stage (bulk copy), one mbarrier per stage;
//   warps 2..5  dequantise the packed block into a 256 x 64 f16 K-major tile in the
//               same swizzled layout (the UMMA B operand), then run the epilogue;
//   warp 1      allocates TMEM (256 columns = the 128 x 256 f32 accumulator) and one
//               elected lane issues tcgen05.mma (M=128, N=256, K=16) x 4 per stage,
//               committing each stage back to the producer.
// Q1 weights are +-scale exactly in f16, so the f16 tensor-core operand loses nothing.
#include <cuda_fp16.h>

#include "dequant.cuh"
#include "ptx.cuh"

namespace pf {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int NUM_THREADS = 192;
constexpr int A_STAGE = BM * BK * 2;  // 16 KB
constexpr int B_STAGE = BN * BK * 2;  // 32 KB
constexpr int TMEM_COLS = 256;

template <int WFMT>
struct Fmt;
template <>
struct Fmt<PF_W_Q1_G128> {
  static constexpr int CHUNK = Q1_CHUNK_BYTES;
  static constexpr int HALF = Q1_HALF_BYTES;
  static constexpr int META_OFF = Q1_SCALE_OFF;
  static constexpr int META = TILE_N * 2;
  static constexpr int P_STAGE = HALF + META;  // 2560
  static constexpr int STAGES = 4;
};
template <>
struct Fmt<PF_W_INT4_AFFINE_G128> {
  static constexpr int CHUNK = I4_CHUNK_BYTES;
  static constexpr int HALF = I4_HALF_BYTES;
  static constexpr int META_OFF = I4_SCALE_OFF;
  static constexpr int META = TILE_N * 4;  // scales then zeros
  static constexpr int P_STAGE = HALF + META;  // 9216
  static constexpr int STAGES = 3;
};

template <int WFMT>
constexpr int smem_bytes() {
  return 1024 /*alignment slack*/ + Fmt<WFMT>::STAGES * (A_STAGE + B_STAGE + Fmt<WFMT>::P_STAGE) +
         256 /*barriers and flags*/;
}

// Bounded wait that ignores the abort flag (used while draining after an abort).
__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > PF_WAIT_LIMIT_NS) return;
  }
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + __expf(-g)) * u; }

template <int WFMT, int EPI>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_q_kernel(const __grid_constant__ CUtensorMap tmap_a, const uint8_t* __restrict__ wpk,
                  int M, int N, int K, void* __restrict__ out, int kb_per_split,
                  int* __restrict__ status) {
  using F = Fmt<WFMT>;
  constexpr int S = F::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t a_st = base;
  const uint32_t b_st = a_st + S * A_STAGE;
  const uint32_t p_st = b_st + S * B_STAGE;
  uint8_t* p_gen = gbase + (p_st - base);
  const uint32_t bar0 = p_st + S * F::P_STAGE;
  // barriers: full[S], bfull[S], empty[S], accum, drain; then flags
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto bfull = [&](int s) { return bar0 + 8u * (S + s); };
  auto empty = [&](int s) { return bar0 + 8u * (2 * S + s); };
  const uint32_t accum_bar = bar0 + 8u * (3 * S);
  const uint32_t drain_bar = accum_bar + 8u;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + (drain_bar + 8u - base));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + (drain_bar + 16u - base));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nt = blockIdx.x;
  const int m0 = blockIdx.y * BM;
  const int nkb_total = K / BK;
  const int kb0 = blockIdx.z * kb_per_split;
  const int kb1 = min(nkb_total, kb0 + kb_per_split);
  const int nkb = kb1 - kb0;
  if (nkb <= 0) return;  // uniform across the CTA: nothing allocated yet

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 1);
      mbar_init(bfull(s), 128);
      mbar_init(empty(s), 1);
    }
    mbar_init(accum_bar, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_d = *tmem_slot;

  const int G = K / GROUP;
  if (warp == 0) {
    if (lane == 0) {
      int issued = 0;
      for (int i = 0; i < nkb; ++i) {
        const int s = i % S;
        const uint32_t ph = (i / S) & 1;
        if (!mbar_wait(empty(s), ph ^ 1, abort_flag)) break;
        const int kb = kb0 + i;
        const uint8_t* chunk =
            wpk + (static_cast<size_t>(nt) * G + (kb >> 1)) * static_cast<size_t>(F::CHUNK);
        mbar_arrive_expect_tx(full(s), A_STAGE + F::P_STAGE);
        tma_load_2d(a_st + s * A_STAGE, &tmap_a, kb * BK, m0, full(s));
        bulk_load(p_st + s * F::P_STAGE, chunk + (kb & 1) * F::HALF, F::HALF, full(s));
        bulk_load(p_st + s * F::P_STAGE + F::HALF, chunk + F::META_OFF, F::META, full(s));
        ++issued;
      }
      if (*abort_flag) {
        // let copies already in flight land before the CTA's shared memory is released
        for (int i = max(0, issued - S); i < issued; ++i)
          mbar_wait_drain(full(i % S), (i / S) & 1);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16(BM, BN, 0);
      bool ok = true;
      for (int i = 0; i < nkb && ok; ++i) {
        const int s = i % S;
        const uint32_t ph = (i / S) & 1;
        ok = mbar_wait(bfull(s), ph, abort_flag) && mbar_wait(full(s), ph, abort_flag);
        if (!ok) break;
        tc_fence_after();
        const uint64_t ad = sdesc_kmajor_sw128(a_st + s * A_STAGE);
        const uint64_t bd = sdesc_kmajor_sw128(b_st + s * B_STAGE);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          umma_f16_ss(tmem_d, ad + 2 * kk, bd + 2 * kk, idesc, (i | kk) != 0);
        umma_commit(empty(s));
      }
      if (ok) {
        umma_commit(accum_bar);
      } else {
        umma_commit(drain_bar);  // wait for any MMA still reading shared memory / TMEM
        mbar_wait_drain(drain_bar, 0);
      }
    }
  } else {
    // warps 2..5: dequantise, then epilogue
    const int d = threadIdx.x - 64;  // 0..127
    for (int i = 0; i < nkb; ++i) {
      const int s = i % S;
      const uint32_t ph = (i / S) & 1;
      if (!mbar_wait(full(s), ph, abort_flag)) break;
      const uint8_t* p = p_gen + s * F::P_STAGE;
      const uint32_t bt = b_st + s * B_STAGE;
      if (WFMT == PF_W_Q1_G128) {
        dequant_row_q1(p, d, bt);
        dequant_row_q1(p, d + 128, bt);
      } else {
        dequant_row_int4(p, d, bt);
        dequant_row_int4(p, d + 128, bt);
      }
      fence_proxy_async_smem();
      mbar_arrive(bfull(s));
    }

    const bool ok = mbar_wait(accum_bar, 0, abort_flag);
    tc_fence_after();
    if (ok) {
      const int q = warp & 3;  // TMEM lane quarter this warp may read
      const int row = m0 + 32 * q + lane;
      const uint32_t tb = tmem_d + (static_cast<uint32_t>(32 * q) << 16);
      if (EPI == EPI_SWIGLU) {
        const int NO = N >> 1;
        __half* o = reinterpret_cast<__half*>(out);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t g[32], u[32];
          tmem_ld_32x32b_x32(tb + 32 * c, g);
          tmem_ld_32x32b_x32(tb + 128 + 32 * c, u);
          tmem_ld_wait();
          const int col = nt * 128 + 32 * c;
          if (row < M && col < NO) {
            uint4* dst = reinterpret_cast<uint4*>(o + static_cast<size_t>(row) * NO + col);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint32_t pk[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int x = 8 * j + 2 * e;
                const __half2 h = __floats2half2_rn(
                    silu_mul(__uint_as_float(g[x]), __uint_as_float(u[x])),
                    silu_mul(__uint_as_float(g[x + 1]), __uint_as_float(u[x + 1])));
                pk[e] = *reinterpret_cast<const uint32_t*>(&h);
              }
              dst[j] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
          }
        }
      } else {
        float* o = reinterpret_cast<float*>(out);
        const bool atomic = gridDim.z > 1;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tb + 32 * c, v);
          tmem_ld_wait();
          const int col = nt * BN + 32 * c;
          if (row < M) {
            float4* dst = reinterpret_cast<float4*>(o + static_cast<size_t>(row) * N + col);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              if (col + 4 * j >= N) break;
              const float4 val = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                             __uint_as_float(v[4 * j + 2]),
                                             __uint_as_float(v[4 * j + 3]));
              if (EPI == EPI_RESID_ADD || atomic) {
                if (atomic) {
                  atomicAdd(dst + j, val);
                } else {
                  float4 x = dst[j];
                  x.x += val.x; x.y += val.y; x.z += val.z; x.w += val.w;
                  dst[j] = x;
                }
              } else {
                dst[j] = val;
              }
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_d, TMEM_COLS);
  }
  if (threadIdx.x == 0 && *abort_flag && status != nullptr) atomicCAS(status, 0, PF_ERR_DEVICE_TIMEOUT);
}

template <int WFMT, int EPI>
cudaError_t launch_t(const GemmArgs& g, const CUtensorMap& tm, cudaStream_t stream) {
  auto kern = gemm_q_kernel<WFMT, EPI>;
  constexpr int smem = smem_bytes<WFMT>();
  const int nkb = g.K / BK;
  const int split = EPI == EPI_SWIGLU ? 1 : max(1, min(g.split_k, nkb));
  const int per = (nkb + split - 1) / split;
  const int splits = (nkb + per - 1) / per;
  dim3 grid(static_cast<unsigned>(padded_rows(g.N) / TILE_N), (g.M + BM - 1) / BM, splits);
  kern<<<grid, NUM_THREADS, smem, stream>>>(tm, g.w, g.M, g.N, g.K, g.out, per, g.status);
  return cudaGetLastError();
}

}  // namespace

bool encode_tmap_f16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                        uint32_t box_inner, uint32_t box_outer);

int choose_split_k(int M, int N, int K, int epilogue, int num_sms) {
  if (epilogue == EPI_SWIGLU) return 1;
  const int tiles = static_cast<int>(padded_rows(N) / TILE_N) * ((M + BM - 1) / BM);
  const int nkb = K / BK;
  int best = 1;
  double best_cost = 1e30;
  for (int s = 1; s <= 16 && s <= nkb / 4; ++s) {
    const int per = (nkb + s - 1) / s;
    const int splits = (nkb + per - 1) / per;
    const int waves = (tiles * splits + num_sms - 1) / num_sms;
    const double cost = waves * (per + 4.0) + (s > 1 ? 1.0 : 0.0);
    if (cost < best_cost - 1e-9) {
      best_cost = cost;
      best = s;
    }
  }
  return best;
}

template <int WFMT, int EPI>
cudaError_t set_smem_attr() {
  return cudaFuncSetAttribute(gemm_q_kernel<WFMT, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              smem_bytes<WFMT>());
}

cudaError_t prepare_gemm_kernels() {
  cudaError_t e = cudaSuccess;
  cudaError_t r;
  if ((r = set_smem_attr<PF_W_Q1_G128, EPI_STORE_F32>()) != cudaSuccess) e = r;
  if ((r = set_smem_attr<PF_W_Q1_G128, EPI_RESID_ADD>()) != cudaSuccess) e = r;
  if ((r = set_smem_attr<PF_W_Q1_G128, EPI_SWIGLU>()) != cudaSuccess) e = r;
  if ((r = set_smem_attr<PF_W_INT4_AFFINE_G128, EPI_STORE_F32>()) != cudaSuccess) e = r;
  if ((r = set_smem_attr<PF_W_INT4_AFFINE_G128, EPI_RESID_ADD>()) != cudaSuccess) e = r;
  if ((r = set_smem_attr<PF_W_INT4_AFFINE_G128, EPI_SWIGLU>()) != cudaSuccess) e = r;
  return e;
}

cudaError_t launch_gemm(const GemmArgs& g, cudaStream_t stream) {
  CUtensorMap tm;
  if (!encode_tmap_f16_2d(&tm, g.a, static_cast<uint64_t>(g.K), static_cast<uint64_t>(g.M), BK, BM))
    return cudaErrorInvalidValue;
  if (g.wfmt == PF_W_Q1_G128) {
    switch (g.epilogue) {
      case EPI_STORE_F32: return launch_t<PF_W_Q1_G128, EPI_STORE_F32>(g, tm, stream);
      case EPI_RESID_ADD: return launch_t<PF_W_Q1_G128, EPI_RESID_ADD>(g, tm, stream);
      case EPI_SWIGLU: return launch_t<PF_W_Q1_G128, EPI_SWIGLU>(g, tm, stream);
    }
  } else {
    switch (g.epilogue) {
      case EPI_STORE_F32: return launch_t<PF_W_INT4_AFFINE_G128, EPI_STORE_F32>(g, tm, stream);
      case EPI_RESID_ADD: return launch_t<PF_W_INT4_AFFINE_G128, EPI_RESID_ADD>(g, tm, stream);
      case EPI_SWIGLU: return launch_t<PF_W_INT4_AFFINE_G128, EPI_SWIGLU>(g, tm, stream);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace pf
