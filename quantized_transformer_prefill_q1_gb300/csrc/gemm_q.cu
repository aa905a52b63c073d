// gemm_q.cu — quantised GEMM on the 5th-generation tensor cores (tcgen05 / TMEM).
//
// out[m, n] (+)= sum_k a[m, k] * w[n, k] with a = f16 activations [M, K] (the RMSNorm /
// SwiGLU / attention outputs) and w a packed Q1 or INT4-affine weight [N, K]. This is
// the batched projection of oxibonsai-kernels metal_prefill.rs `encode_layer_prefill`:
// section 2 (QKV GEMM, plain store), sections 4 and 7 (O / down GEMM with the residual
// add fused, `dispatch_gemm_q1_v7_residual`) and section 6 (gate+up GEMM with SwiGLU
// fused, `dispatch_fused_gate_up_swiglu_gemm`).
//
// Persistent CTAs (one per SM) walk a list of work units = (128-token tile, 256-row
// weight tile, K split). Warp roles:
//   warp 0       TMA producer: activation tile (128 x 64 f16, 128-B swizzle) and the
//                stage's packed weight block (bulk copy) into a ring of stages;
//   warps 6..13  dequantise the packed block (one weight row per thread) into a 256 x 64
//                f16 K-major tile in the same swizzled layout: the UMMA B operand;
//   warp 1       allocates 512 TMEM columns (two 128 x 256 f32 accumulators) and one lane
//                issues tcgen05.mma (M=128, N=256, K=16) x 4 per stage, committing each
//                stage back to the ring and each finished unit to the epilogue;
//   warps 2..5   epilogue: tcgen05.ld of the finished accumulator (f32 store / residual
//                add / SwiGLU), overlapping the next unit's main loop in the other buffer.
// Q1 weights are +-scale, exact in f16, so the f16 tensor-core operand loses nothing.
#include <cuda_fp16.h>

#include "dequant.cuh"
#include "ptx.cuh"

namespace pf {
namespace {

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int NUM_EPI_WARPS = 4;
constexpr int NUM_DQ_WARPS = 8;
constexpr int DQ_THREADS = NUM_DQ_WARPS * 32;  // == BN: one weight row per thread
constexpr int EPI_THREADS = NUM_EPI_WARPS * 32;
constexpr int NUM_THREADS = 32 * (2 + NUM_EPI_WARPS + NUM_DQ_WARPS);  // 448
constexpr int FIRST_DQ_WARP = 2 + NUM_EPI_WARPS;
constexpr int A_STAGE = BM * BK * 2;  // 16 KB
constexpr int B_STAGE = BN * BK * 2;  // 32 KB
constexpr int TMEM_COLS = 512;        // two accumulators of 256 f32 columns
static_assert(DQ_THREADS == BN, "one dequantising thread per weight row");

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

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// One weight row's 64 weights of a stage (packed block p) -> 8 16-B chunks of f16 in the
// 128-B swizzle K-major layout of the UMMA B tile: row r at (r / 8) * 1024 + (r % 8) * 128,
// chunk c (k 8c .. 8c+7) at chunk position c ^ (r % 8).
template <int WFMT>
__device__ __forceinline__ void dequant_row_smem(const uint8_t* p, int r, uint32_t b_tile) {
  const uint32_t row_base = b_tile + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
  for (int half = 0; half < 2; ++half) {  // k 0..31, 32..63
    uint32_t w[16];
    if (WFMT == PF_W_Q1_G128) {
      const uint32_t Z = reinterpret_cast<const uint32_t*>(p + r * 8)[half];
      const uint32_t s16 = reinterpret_cast<const uint16_t*>(p + Q1_HALF_BYTES)[r];
      dq_q1_32(Z, s16 | (s16 << 16), w);
    } else {
      const uint4 q = reinterpret_cast<const uint4*>(p + r * 32)[half];
      const uint16_t s16 = reinterpret_cast<const uint16_t*>(p + I4_HALF_BYTES)[r];
      const uint16_t z16 = reinterpret_cast<const uint16_t*>(p + I4_HALF_BYTES + TILE_N * 2)[r];
      dq_i4_32(q, __half2half2(__ushort_as_half(s16)), __half2half2(__ushort_as_half(z16)), w);
    }
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {
      const int c = 4 * half + c4;
      st_shared_v4(row_base + ((c ^ (r & 7)) << 4), w[4 * c4], w[4 * c4 + 1], w[4 * c4 + 2],
                   w[4 * c4 + 3]);
    }
  }
}

struct Units {
  int n_mt, n_nt, per_split, nkb_total;
  __device__ __forceinline__ void decode(int u, int& mt, int& nt, int& kb0, int& nkb) const {
    const int tiles = n_mt * n_nt;
    const int split = u / tiles;
    const int r = u - split * tiles;
    nt = r / n_mt;
    mt = r - nt * n_mt;  // token tiles fastest: neighbouring CTAs share a weight tile
    kb0 = split * per_split;
    nkb = min(nkb_total, kb0 + per_split) - kb0;
  }
};

template <int WFMT, int EPI>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_q_kernel(const __grid_constant__ CUtensorMap tmap_a, const uint8_t* __restrict__ wpk,
                  int M, int N, int K, void* __restrict__ out, Units units, int n_units,
                  int atomic_out, int* __restrict__ status) {
  using F = Fmt<WFMT>;
  constexpr int S = F::STAGES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t a_st = base;
  const uint32_t b_st = a_st + S * A_STAGE;
  const uint32_t p_st = b_st + S * B_STAGE;
  const uint8_t* p_gen = gbase + (p_st - base);
  const uint32_t bar0 = p_st + S * F::P_STAGE;
  // barriers: full[S], bfull[S], empty[S], acc_full[2], acc_empty[2], drain; then flags
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto bfull = [&](int s) { return bar0 + 8u * (S + s); };
  auto empty = [&](int s) { return bar0 + 8u * (2 * S + s); };
  auto acc_full = [&](int b) { return bar0 + 8u * (3 * S + b); };
  auto acc_empty = [&](int b) { return bar0 + 8u * (3 * S + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (3 * S + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + (drain_bar + 8u - base));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + (drain_bar + 16u - base));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  griddep_launch_dependents();

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 1);
      mbar_init(bfull(s), DQ_THREADS);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full(b), 1);
      mbar_init(acc_empty(b), EPI_THREADS);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  griddep_wait();  // inputs come from the previous kernel in the stream
  const int G = K / GROUP;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        int mt, nt, kb0, nkb;
        units.decode(u, mt, nt, kb0, nkb);
        for (int i = 0; i < nkb; ++i, ++it) {
          const int s = it % S;
          const uint32_t ph = (it / S) & 1;
          if (!mbar_wait(empty(s), ph ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          const int kb = kb0 + i;
          const uint8_t* chunk =
              wpk + (static_cast<size_t>(nt) * G + (kb >> 1)) * static_cast<size_t>(F::CHUNK);
          mbar_arrive_expect_tx(full(s), A_STAGE + F::P_STAGE);
          tma_load_2d(a_st + s * A_STAGE, &tmap_a, kb * BK, mt * BM, full(s));
          bulk_load(p_st + s * F::P_STAGE, chunk + (kb & 1) * F::HALF, F::HALF, full(s));
          bulk_load(p_st + s * F::P_STAGE + F::HALF, chunk + F::META_OFF, F::META, full(s));
        }
      }
      if (!ok) {  // let copies already in flight land before shared memory is released
        for (int j = max(0, it - S); j < it; ++j) mbar_wait_drain(full(j % S), (j / S) & 1);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16(BM, BN, 0);
      int it = 0, local = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++local) {
        int mt, nt, kb0, nkb;
        units.decode(u, mt, nt, kb0, nkb);
        const int b = local & 1;
        const uint32_t use = static_cast<uint32_t>(local >> 1);
        if (!mbar_wait(acc_empty(b), (use & 1) ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + b * BN;
        for (int i = 0; i < nkb; ++i, ++it) {
          const int s = it % S;
          const uint32_t ph = (it / S) & 1;
          if (!(mbar_wait(bfull(s), ph, abort_flag) && mbar_wait(full(s), ph, abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sdesc_kmajor_sw128(a_st + s * A_STAGE);
          const uint64_t bd = sdesc_kmajor_sw128(b_st + s * B_STAGE);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            umma_f16_ss(d_tmem, ad + 2 * kk, bd + 2 * kk, idesc, (i | kk) != 0);
          umma_commit(empty(s));
        }
        if (ok) umma_commit(acc_full(b));
      }
      if (!ok) {
        umma_commit(drain_bar);  // wait for any MMA still reading shared memory / TMEM
        mbar_wait_drain(drain_bar, 0);
      }
    }
  } else if (warp >= FIRST_DQ_WARP) {
    // ---------------------------------------------------------------- dequantisers
    const int d = threadIdx.x - FIRST_DQ_WARP * 32;  // weight row of the tile
    int it = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      int mt, nt, kb0, nkb;
      units.decode(u, mt, nt, kb0, nkb);
      for (int i = 0; i < nkb; ++i, ++it) {
        const int s = it % S;
        const uint32_t ph = (it / S) & 1;
        if (!mbar_wait(full(s), ph, abort_flag)) {
          ok = false;
          break;
        }
        const uint8_t* p = p_gen + s * F::P_STAGE;
        const uint32_t bt = b_st + s * B_STAGE;
        dequant_row_smem<WFMT>(p, d, bt);
        fence_proxy_async_smem();
        mbar_arrive(bfull(s));
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue (warps 2..5)
    const int q = warp & 3;  // TMEM lane quarter this warp may read
    int local = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++local) {
      int mt, nt, kb0, nkb;
      units.decode(u, mt, nt, kb0, nkb);
      const int b = local & 1;
      const uint32_t use = static_cast<uint32_t>(local >> 1);
      // warp-uniform: the tcgen05.ld below is warp-collective
      if (!__all_sync(0xffffffffu, mbar_wait(acc_full(b), use & 1, abort_flag))) break;
      tc_fence_after();
      const int row = mt * BM + 32 * q + lane;
      const uint32_t tb = tmem_base + b * BN + (static_cast<uint32_t>(32 * q) << 16);
      if (EPI == EPI_SWIGLU) {
        // each 128 columns of the tile: 64 gate columns, then the 64 matching up columns
        const int NO = N >> 1;
        __half* o = reinterpret_cast<__half*>(out);
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          const int h = c >> 1, q2 = c & 1;  // 128-column half, 32-column quarter of its gates
          uint32_t g[32], v[32];
          tmem_ld_32x32b_x32(tb + 128 * h + 32 * q2, g);
          tmem_ld_32x32b_x32(tb + 128 * h + 64 + 32 * q2, v);
          tmem_ld_wait();
          const int col = nt * 128 + 64 * h + 32 * q2;
          if (row < M && col < NO) {
            uint4* dst = reinterpret_cast<uint4*>(o + static_cast<size_t>(row) * NO + col);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              uint32_t pk[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int x = 8 * j + 2 * e;
                const __half2 hv = __floats2half2_rn(
                    silu_mul(__uint_as_float(g[x]), __uint_as_float(v[x])),
                    silu_mul(__uint_as_float(g[x + 1]), __uint_as_float(v[x + 1])));
                pk[e] = *reinterpret_cast<const uint32_t*>(&hv);
              }
              dst[j] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
          }
        }
      } else {
        float* o = reinterpret_cast<float*>(out);
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
              if (atomic_out) {
                atomicAdd(dst + j, val);
              } else if (EPI == EPI_RESID_ADD) {
                float4 x = dst[j];
                x.x += val.x;
                x.y += val.y;
                x.z += val.z;
                x.w += val.w;
                dst[j] = x;
              } else {
                dst[j] = val;
              }
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(acc_empty(b));
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    __syncwarp();  // lane 0 ran the MMA loop: reconverge before the collective dealloc
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
  if (threadIdx.x == 0 && *abort_flag && status != nullptr) atomicCAS(status, 0, PF_ERR_DEVICE_TIMEOUT);
}

template <int WFMT, int EPI>
cudaError_t launch_t(const GemmArgs& g, const CUtensorMap& tm, int num_sms, cudaStream_t stream) {
  constexpr int smem = smem_bytes<WFMT>();
  const int nkb = g.K / BK;
  const int split = EPI == EPI_SWIGLU ? 1 : max(1, min(g.split_k, nkb));
  Units u;
  u.per_split = (nkb + split - 1) / split;
  const int splits = (nkb + u.per_split - 1) / u.per_split;
  u.n_mt = (g.M + BM - 1) / BM;
  u.n_nt = static_cast<int>(padded_rows(g.N) / TILE_N);
  u.nkb_total = nkb;
  const int n_units = u.n_mt * u.n_nt * splits;
  const int grid = min(n_units, num_sms);
  return launch_pdl(gemm_q_kernel<WFMT, EPI>, dim3(grid), dim3(NUM_THREADS), smem, stream, tm, g.w,
                    g.M, g.N, g.K, g.out, u, n_units, splits > 1 ? 1 : 0, g.status);
}

}  // namespace

bool encode_tmap_f16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                        uint32_t box_inner, uint32_t box_outer);

// Split along K when that shortens the critical path: cost = rounds of units per SM x
// k-blocks per unit (+ a fixed per-unit overhead), with persistent CTAs.
int choose_split_k(int M, int N, int K, int epilogue, int num_sms) {
  if (epilogue == EPI_SWIGLU) return 1;
  const int tiles = static_cast<int>(padded_rows(N) / TILE_N) * ((M + BM - 1) / BM);
  const int nkb = K / BK;
  int best = 1;
  double best_cost = 1e30;
  for (int s = 1; s <= 16 && s <= nkb / 4; ++s) {
    const int per = (nkb + s - 1) / s;
    const int splits = (nkb + per - 1) / per;
    const int rounds = (tiles * splits + num_sms - 1) / num_sms;
    // each extra split adds an f32 atomic reduction of the M x N output; measured on
    // GB300 at ~1.6e-6 k-block-times per output byte and split
    const double atomics = splits > 1 ? splits * static_cast<double>(M) * N * 1.6e-6 : 0.0;
    const double cost = rounds * (per + 3.0) + atomics;
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
  static int sms = device_sm_count();
  if (g.wfmt == PF_W_Q1_G128) {
    switch (g.epilogue) {
      case EPI_STORE_F32: return launch_t<PF_W_Q1_G128, EPI_STORE_F32>(g, tm, sms, stream);
      case EPI_RESID_ADD: return launch_t<PF_W_Q1_G128, EPI_RESID_ADD>(g, tm, sms, stream);
      case EPI_SWIGLU: return launch_t<PF_W_Q1_G128, EPI_SWIGLU>(g, tm, sms, stream);
    }
  } else {
    switch (g.epilogue) {
      case EPI_STORE_F32: return launch_t<PF_W_INT4_AFFINE_G128, EPI_STORE_F32>(g, tm, sms, stream);
      case EPI_RESID_ADD: return launch_t<PF_W_INT4_AFFINE_G128, EPI_RESID_ADD>(g, tm, sms, stream);
      case EPI_SWIGLU: return launch_t<PF_W_INT4_AFFINE_G128, EPI_SWIGLU>(g, tm, sms, stream);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace pf
