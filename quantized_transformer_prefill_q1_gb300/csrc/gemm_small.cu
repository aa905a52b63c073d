// gemm_small.cu — the quantised GEMM for chunks of a few tokens (16 < M <= 64): the weight side
// of a layer's projections (oxibonsai-kernels metal_prefill.rs `encode_layer_prefill`
// sections 2, 4, 6 and 7) when the chunk is so short that streaming the packed weights from
// HBM is the whole cost (the GEMV end of the small-M crossover).
//
// The MMA is turned around: weight rows are its M side (two MMAs of 128 rows cover one
// 256-row packed tile) and the chunk's tokens (padded to NT = 32 or 64) its N side,
// out^T[n, m] = sum_k w[n, k] a[m, k]. The dequantised f16 weights go from registers
// straight into tensor memory (tcgen05.st) as the A operand, so shared memory carries only
// the packed chunks and the small activation tiles. One stage is one 128-wide group: the
// tile's whole packed chunk (one bulk copy) and the activation tile of both 64-wide halves
// (one 3-D TMA load), so few, large copies keep the weight stream HBM-bound.
//   warp 0      TMA producer, a ring of S group stages;
//   warp 1      (whole warp, one elected lane issues) tcgen05.mma M=128, N=NT, K=16: 8 per
//               128-row half and group, A from tensor memory, B the activation tile;
//   warps 2..17 one (weight row, 64-wide half of the group) per thread (warp w: lane
//               quarter w % 4, row half ((w - 2) / 4) % 2, k half (w - 2) / 8): dequantise
//               64 weights into one of 3 A stages in tensor memory (four warps per scheduler
//               keep the INT4 dequantisation arithmetic busy); at the end of a segment read
//               the accumulator (row x tokens, the k half picking the token half) and apply
//               the epilogue.
// The groups of all 256-row tiles are shared out by the same stream-K partition as the large
// GEMM: the residual form adds every CTA's share into out with f32 reductions; the store and
// SwiGLU forms pass split tiles' partials through scratch + per-tile arrival counters.
#include <cuda_fp16.h>

#include <algorithm>

#include "dequant.cuh"
#include "ptx.cuh"
#include "streamk.cuh"

namespace pf {
namespace {
using sk::Plan;
using sk::Range;
using sk::Segment;

constexpr int TR = 128;             // weight rows per MMA (M)
constexpr int TT = 256;             // weight rows per tile (one packed tile)
constexpr int THREADS_S = 576;      // warp 0 TMA, warp 1 MMA, warps 2..17 dequant + epilogue
constexpr int EPI_T = 512;
constexpr int SA = 3;               // A stages in tensor memory: 128 columns each (2 halves x 64)
constexpr uint32_t COL_D = SA * 128;  // accumulators of the two row halves: [384, 384 + 2 NT)
constexpr size_t SLOT = static_cast<size_t>(128) * 256;  // floats per scratch slot
constexpr int SMEM_LIMIT = 232448;

template <int WFMT>
struct SF {
  static constexpr int P = WFMT == PF_W_Q1_G128 ? Q1_CHUNK_BYTES : I4_CHUNK_BYTES;  // one chunk
};

template <int WFMT, int NT>
struct SL {
  static constexpr int B = 2 * NT * 128;             // activation tile: two halves of NT x 64 f16
  static constexpr int XCH = 128 * NT * 4;           // SwiGLU: up rows handed to gate rows
  static constexpr int FIXED = 1024 + XCH + 1024;    // alignment, exchange, barriers
  static constexpr int S0 = (SMEM_LIMIT - FIXED) / (B + SF<WFMT>::P);
  static constexpr int S = S0 > 24 ? 24 : S0;
  static constexpr int BYTES = FIXED + S * (B + SF<WFMT>::P);
  static_assert(S >= 3 && BYTES <= SMEM_LIMIT, "small-M GEMM shared memory");
  static_assert(SA * 128 + 2 * NT <= 512, "small-M GEMM tensor memory");
};

__device__ __forceinline__ void mbar_wait_drain_s(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > PF_WAIT_LIMIT_NS) return;
  }
}
__device__ __forceinline__ void bar_sync_s(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}
__device__ __forceinline__ bool bar_and_s(int id, int threads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, %2, %3, p;\n"
      " selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(threads)
      : "memory");
  return r != 0;
}
// silu(g) * u = g / (1 + e^-g) * u. The exponent is capped at 80 so the denominator stays
// below 2^126, where the fast division is within 2 ulp; for g < -80 the result is ~1e-33 * u.
__device__ __forceinline__ float silu_mul_s(float g, float u) {
  return __fdividef(g, 1.0f + __expf(fminf(-g, 80.0f))) * u;
}

template <int WFMT, int EPI, int NT>
__global__ void __launch_bounds__(THREADS_S, 1)
    gemm_small_kernel(const __grid_constant__ CUtensorMap tmap_x, const uint8_t* __restrict__ wpk,
                      int M, int N, int K, void* __restrict__ out, Plan plan,
                      float* __restrict__ scratch, int* __restrict__ counters,
                      int* __restrict__ status) {
  PF_TIMELINE(TL_GEMM_SMALL + EPI);
  using F = SF<WFMT>;
  using L = SL<WFMT, NT>;
  constexpr int S = L::S;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t b_st = base;                  // S activation tiles (1024-B multiples)
  const uint32_t p_st = b_st + S * L::B;       // S packed chunks
  const uint32_t x_st = p_st + S * F::P;       // SwiGLU exchange
  const uint32_t bar0 = (x_st + L::XCH + 7u) & ~7u;
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto empty = [&](int s) { return bar0 + 8u * (S + s); };
  auto a_full = [&](int a) { return bar0 + 8u * (2 * S + a); };
  auto a_empty = [&](int a) { return bar0 + 8u * (2 * S + SA + a); };
  const uint32_t acc_full = bar0 + 8u * (2 * S + 2 * SA);
  const uint32_t acc_empty = acc_full + 8u;
  const uint32_t drain_bar = acc_full + 16u;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + (drain_bar + 8u - base));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + (drain_bar + 16u - base));
  volatile int* flags = reinterpret_cast<volatile int*>(gbase + (drain_bar + 24u - base));  // [4]
  const uint8_t* p_gen = gbase + (p_st - base);
  float* xch = reinterpret_cast<float*>(gbase + (x_st - base));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  griddep_launch_dependents();
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int a = 0; a < SA; ++a) {
      mbar_init(a_full(a), EPI_T);
      mbar_init(a_empty(a), 1);
    }
    mbar_init(acc_full, 1);
    mbar_init(acc_empty, EPI_T);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    __syncwarp();
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Only the activation tiles and the epilogue's global accesses depend on the previous
  // kernel (griddep_wait below); the producer issues the first stages' weight chunks first.
  const int G = K / GROUP;
  const Range rg(plan, blockIdx.x);

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      int pre = 0;  // stages whose weight chunk is issued before the wait
      for (int k = 0; k < rg.n && pre < S; ++k) {
        const Segment sg = rg.at(plan, k);
        for (int i = 0; i < sg.nkb && pre < S; ++i, ++pre) {
          mbar_arrive_expect_tx(full(pre), L::B + F::P);
          bulk_load(p_st + pre * F::P, wpk + (static_cast<size_t>(sg.nt) * G + sg.kb0 + i) * F::P, F::P,
                    full(pre));
        }
      }
      griddep_wait();  // the activations come from the previous kernel
      for (int k = 0, j = 0; k < rg.n && j < pre; ++k) {
        const Segment sg = rg.at(plan, k);
        for (int i = 0; i < sg.nkb && j < pre; ++i, ++j)
          tma_load_3d(b_st + j * L::B, &tmap_x, 0, 0, 2 * (sg.kb0 + i), full(j));
      }
      int it = 0;
      bool ok = true;
      for (int k = 0; k < rg.n && ok; ++k) {
        const Segment sg = rg.at(plan, k);
        for (int i = 0; i < sg.nkb; ++i, ++it) {
          if (it < pre) continue;  // issued above
          const int s = it % S;
          if (!mbar_wait(empty(s), ((it / S) & 1) ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          const int g = sg.kb0 + i;  // group
          mbar_arrive_expect_tx(full(s), L::B + F::P);
          // activation k-blocks 2g, 2g+1 of rows 0..NT-1: smem [2][NT][64] (rows >= M zero)
          tma_load_3d(b_st + s * L::B, &tmap_x, 0, 0, 2 * g, full(s));
          bulk_load(p_st + s * F::P, wpk + (static_cast<size_t>(sg.nt) * G + g) * F::P, F::P, full(s));
        }
      }
      if (!ok) {  // let copies already in flight land before shared memory is released
        for (int j = max(0, it - S); j < it; ++j) mbar_wait_drain_s(full(j % S), (j / S) & 1);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    constexpr uint32_t idesc = idesc_f16(TR, NT, 0);
    int it = 0;
    bool ok = true;
    for (int k = 0; k < rg.n && ok; ++k) {
      const Segment sg = rg.at(plan, k);
      if (!__all_sync(0xffffffffu, mbar_wait(acc_empty, (k & 1) ^ 1, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      for (int i = 0; i < sg.nkb; ++i, ++it) {
        const int s = it % S, a = it % SA;
        ok = __all_sync(0xffffffffu, mbar_wait(a_full(a), (it / SA) & 1, abort_flag) &&
                                         mbar_wait(full(s), (it / S) & 1, abort_flag));
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
          for (int kk = 0; kk < GROUP / 16; ++kk) {
            const uint64_t bd = sdesc_kmajor_sw128(b_st + s * L::B + (kk >> 2) * (NT * 128)) + 2 * (kk & 3);
            umma_f16_ts_warp(tmem + COL_D + h * NT, tmem + a * 128 + h * 64 + 8 * kk, bd, idesc,
                             (i | kk) != 0);
          }
        }
        umma_commit_warp(empty(s));
        umma_commit_warp(a_empty(a));
      }
      if (ok) umma_commit_warp(acc_full);
    }
    if (!ok) {
      umma_commit_warp(drain_bar);
      mbar_wait_drain_s(drain_bar, 0);
    }
  } else {
    // ---------------------------------------------------------------- dequant + epilogue
    griddep_wait();  // out / scratch / counters are shared with the previous kernels
    const int dw = warp - 2;
    const int q = warp & 3;
    const int hh = (dw >> 2) & 1;       // 128-row half of the tile
    const int jj = dw >> 3;             // 64-wide half of the group (and token half)
    const int rl = 32 * q + lane;       // TMEM lane
    const int r = 128 * hh + rl;        // weight row within the 256-row tile
    const int et = threadIdx.x - 64;
    const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;
    constexpr int MH = NT / 2;          // tokens per thread in the epilogue
    const int m0 = jj * MH;
    int it = 0;
    bool ok = true;
    for (int k = 0; k < rg.n && ok; ++k) {
      const Segment sg = rg.at(plan, k);
      for (int i = 0; i < sg.nkb; ++i, ++it) {
        const int s = it % S, a = it % SA;
        if (!__all_sync(0xffffffffu, mbar_wait(full(s), (it / S) & 1, abort_flag) &&
                                         mbar_wait(a_empty(a), ((it / SA) & 1) ^ 1, abort_flag))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint8_t* p = p_gen + s * F::P;
        uint32_t w[32];
        if (WFMT == PF_W_Q1_G128) {
          const uint2 Z = reinterpret_cast<const uint2*>(p + jj * Q1_HALF_BYTES)[r];
          const uint32_t s16 = reinterpret_cast<const uint16_t*>(p + Q1_SCALE_OFF)[r];
          dq_q1_32(Z.x, s16 | (s16 << 16), *reinterpret_cast<uint32_t(*)[16]>(w));
          dq_q1_32(Z.y, s16 | (s16 << 16), *reinterpret_cast<uint32_t(*)[16]>(w + 16));
        } else {
          const uint4* qw = reinterpret_cast<const uint4*>(p + jj * I4_HALF_BYTES + r * 32);
          const __half2 s2 = __half2half2(reinterpret_cast<const __half*>(p + I4_SCALE_OFF)[r]);
          const __half2 z2 = __half2half2(reinterpret_cast<const __half*>(p + I4_ZERO_OFF)[r]);
          dq_i4_32(qw[0], s2, z2, *reinterpret_cast<uint32_t(*)[16]>(w));
          dq_i4_32(qw[1], s2, z2, *reinterpret_cast<uint32_t(*)[16]>(w + 16));
        }
        tmem_st_32x32b_x32(tmem + a * 128 + hh * 64 + jj * 32 + lane_off, w);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(a_full(a));
      }
      // ---- end of segment: the accumulator (row r x tokens m0 .. m0+MH-1) and the epilogue
      const bool got = ok && mbar_wait(acc_full, k & 1, abort_flag);
      if (!bar_and_s(1, EPI_T, got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float v[32];
      {
        uint32_t u[32];
        tmem_ld_32x32b_x32(tmem + COL_D + hh * NT + m0 + lane_off, u);
        tmem_ld_wait();
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(u[j]);
      }
      tc_fence_before();
      mbar_arrive(acc_empty);  // the accumulator is in registers: the next segment may start
      if (EPI == EPI_RESID_ADD) {
        // residual: every segment, whole or split, adds its share into out (f32 reductions)
        const int row = sg.nt * TT + r;
        if (row < N) {
          float* o = reinterpret_cast<float*>(out) + row;
#pragma unroll
          for (int m = 0; m < MH; ++m)
            if (m0 + m < M) atomicAdd(o + static_cast<size_t>(m0 + m) * N, v[m]);
        }
        continue;
      }
      bool finish = sg.whole;
      int c_lo = 0, c_hi = -1;
      if (!sg.whole) {
        // partial [token][row] in this CTA's slot; the last contributor finishes the tile
        c_lo = plan.owner(static_cast<long long>(sg.tile) * plan.kbt);
        c_hi = plan.owner(static_cast<long long>(sg.tile + 1) * plan.kbt - 1);
        const int others = c_hi - c_lo;
        const int slot = plan.slot(blockIdx.x, sg.tile);
        volatile int* flag = flags + 2 * slot;
        if (et == 0) flag[0] = ld_acquire_gpu(counters + sg.tile) == others ? 1 : 0;
        bar_sync_s(1, EPI_T);
        finish = flag[0] != 0;
        if (!finish) {
          float* mine = scratch + (static_cast<size_t>(blockIdx.x) * 2 + slot) * SLOT;
#pragma unroll
          for (int m = 0; m < MH; ++m)
            if (m0 + m < M) __stcg(mine + (m0 + m) * TT + r, v[m]);
          __threadfence();
          bar_sync_s(1, EPI_T);
          if (et == 0) flag[1] = atomicAdd(counters + sg.tile, 1) == others ? 1 : 0;
          bar_sync_s(1, EPI_T);
          finish = flag[1] != 0;
        }
        if (finish) {
          if (et == 0) counters[sg.tile] = 0;  // every contributor is in: ready for reuse
          __threadfence();
          for (int c = c_lo; c <= c_hi; ++c) {
            if (c == static_cast<int>(blockIdx.x)) continue;
            const float* src = scratch + (static_cast<size_t>(c) * 2 + plan.slot(c, sg.tile)) * SLOT;
#pragma unroll
            for (int m = 0; m < MH; ++m)
              if (m0 + m < M) v[m] += __ldcg(src + (m0 + m) * TT + r);
          }
        }
      }
      if (finish) {
        if (EPI == EPI_SWIGLU) {
          // rows 128h .. 128h+63 are gate rows, 128h+64 .. 128h+127 the matching up rows
          if (rl >= 64) {
#pragma unroll
            for (int m = 0; m < MH; ++m) xch[(64 * hh + rl - 64) * NT + m0 + m] = v[m];
          }
          bar_sync_s(1, EPI_T);
          const int col = sg.nt * 128 + 64 * hh + rl;  // output column of gate row r
          if (rl < 64 && col < (N >> 1)) {
            __half* o = reinterpret_cast<__half*>(out);
#pragma unroll
            for (int m = 0; m < MH; ++m)
              if (m0 + m < M)
                o[static_cast<size_t>(m0 + m) * (N >> 1) + col] =
                    __float2half_rn(silu_mul_s(v[m], xch[(64 * hh + rl) * NT + m0 + m]));
          }
          bar_sync_s(1, EPI_T);  // the exchange area is free again
        } else {
          const int row = sg.nt * TT + r;
          if (row < N) {
            float* o = reinterpret_cast<float*>(out) + row;
#pragma unroll
            for (int m = 0; m < MH; ++m)
              if (m0 + m < M) o[static_cast<size_t>(m0 + m) * N] = v[m];
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    __syncwarp();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && *abort_flag && status != nullptr) atomicCAS(status, 0, PF_ERR_DEVICE_TIMEOUT);
}

template <int WFMT, int EPI, int NT>
cudaError_t launch_s(const GemmArgs& g, int num_sms, cudaStream_t stream) {
  // activations as [K/64][M][64]: box {64, NT, 2} = k-blocks 2g, 2g+1 of rows 0..NT-1
  CUtensorMap tx;
  const uint64_t dims[3] = {64, static_cast<uint64_t>(g.M), static_cast<uint64_t>(g.K / 64)};
  const uint64_t strides[2] = {static_cast<uint64_t>(g.K) * 2, 128};
  const uint32_t box[3] = {64, static_cast<uint32_t>(NT), 2};
  if (!encode_tmap_16(&tx, 0, 3, g.a, dims, strides, box)) return cudaErrorInvalidValue;
  Plan p{};
  p.n_mt = 1;
  p.n_nt = static_cast<int>(padded_rows(g.N) / TT);
  p.kbt = g.K / GROUP;
  p.total = static_cast<long long>(p.n_nt) * p.kbt;
  p.ctas = static_cast<int>(std::min<long long>(std::min(g.max_ctas, num_sms), p.total));
  // store / SwiGLU: a tile split between CTAs costs a partial hand-off, so when the tiles
  // alone fill at least half of the CTAs, run whole tiles (the residual form adds shares)
  if (EPI != EPI_RESID_ADD && p.n_nt < p.ctas && 2 * p.n_nt >= p.ctas) p.ctas = p.n_nt;
  p.late0 = p.ctas;  // no skew
  p.dk = 0;
  float* scratch = reinterpret_cast<float*>(g.scratch);
  int* counters = reinterpret_cast<int*>(scratch + static_cast<size_t>(2) * g.max_ctas * SLOT);
  return launch_pdl(gemm_small_kernel<WFMT, EPI, NT>, dim3(p.ctas), dim3(THREADS_S), SL<WFMT, NT>::BYTES,
                    stream, tx, g.w, g.M, g.N, g.K, g.out, p, scratch, counters, g.status);
}

template <int WFMT, int NT>
cudaError_t launch_fmt(const GemmArgs& g, int sms, cudaStream_t stream) {
  switch (g.epilogue) {
    case EPI_STORE_F32: return launch_s<WFMT, EPI_STORE_F32, NT>(g, sms, stream);
    case EPI_RESID_ADD: return launch_s<WFMT, EPI_RESID_ADD, NT>(g, sms, stream);
    case EPI_SWIGLU: return launch_s<WFMT, EPI_SWIGLU, NT>(g, sms, stream);
  }
  return cudaErrorInvalidValue;
}

template <int WFMT, int EPI, int NT>
cudaError_t attr_s() {
  return cudaFuncSetAttribute(gemm_small_kernel<WFMT, EPI, NT>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, SL<WFMT, NT>::BYTES);
}
template <int WFMT, int NT>
cudaError_t attr_fmt() {
  cudaError_t e = cudaSuccess, r;
  if ((r = attr_s<WFMT, EPI_STORE_F32, NT>()) != cudaSuccess) e = r;
  if ((r = attr_s<WFMT, EPI_RESID_ADD, NT>()) != cudaSuccess) e = r;
  if ((r = attr_s<WFMT, EPI_SWIGLU, NT>()) != cudaSuccess) e = r;
  return e;
}

}  // namespace

cudaError_t prepare_gemm_small_kernels() {
  cudaError_t e = cudaSuccess, r;
  if ((r = attr_fmt<PF_W_Q1_G128, 32>()) != cudaSuccess) e = r;
  if ((r = attr_fmt<PF_W_Q1_G128, 64>()) != cudaSuccess) e = r;
  if ((r = attr_fmt<PF_W_INT4_AFFINE_G128, 32>()) != cudaSuccess) e = r;
  if ((r = attr_fmt<PF_W_INT4_AFFINE_G128, 64>()) != cudaSuccess) e = r;
  return e;
}

cudaError_t launch_gemm_small(const GemmArgs& g, cudaStream_t stream) {
  static int sms = device_sm_count();
  if (g.epilogue == EPI_STORE_F32) {
    // the output is small (M x N f32, M <= 64): zero it (unless the caller has) and accumulate
    // every CTA's share like the residual form, instead of passing split tiles through scratch
    if (!g.out_zeroed) {
      cudaError_t e = cudaMemsetAsync(g.out, 0, static_cast<size_t>(g.M) * g.N * sizeof(float), stream);
      if (e != cudaSuccess) return e;
    }
    GemmArgs r = g;
    r.epilogue = EPI_RESID_ADD;
    return launch_gemm_small(r, stream);
  }
  // chunks of at most 16 tokens go to the GEMV (launch_gemm routes them there)
  if (g.M <= GEMV_M_MAX_Q1 && g.M <= GEMV_M_MAX_I4) return cudaErrorInvalidValue;
  const int nt = g.M <= 32 ? 32 : 64;
  if (g.wfmt == PF_W_Q1_G128) {
    if (nt == 32) return launch_fmt<PF_W_Q1_G128, 32>(g, sms, stream);
    return launch_fmt<PF_W_Q1_G128, 64>(g, sms, stream);
  }
  if (nt == 32) return launch_fmt<PF_W_INT4_AFFINE_G128, 32>(g, sms, stream);
  return launch_fmt<PF_W_INT4_AFFINE_G128, 64>(g, sms, stream);
}

}  // namespace pf

PF_TIMELINE_SETTER(gemm_small)
