// gemm_q.cu — quantised GEMM on the 5th-generation tensor cores (tcgen05 / TMEM).
//
// out[m, n] (+)= sum_k a[m, k] * w[n, k] with a = f16 activations [M, K] (the RMSNorm /
// SwiGLU / attention outputs) and w a packed Q1 or INT4-affine weight [N, K]. This is
// the batched projection of oxibonsai-kernels metal_prefill.rs `encode_layer_prefill`:
// section 2 (QKV GEMM), sections 4 and 7 (O / down GEMM with the residual add fused,
// `dispatch_gemm_q1_v7_residual`) and section 6 (gate+up GEMM with SwiGLU fused,
// `dispatch_fused_gate_up_swiglu_gemm`).
//
// Tiles are 128 tokens x 256 weight rows. The k-blocks (64 wide) of all tiles form one
// list cut into equal contiguous ranges, one per persistent CTA ("stream-K"), so that no
// SM idles while others finish a last round of tiles. The part of a tile inside one
// CTA's range is a segment; a CTA runs its (at most two) partial segments first and its
// whole tiles after them, so that split tiles complete early.
//   * residual epilogue: every segment adds its accumulator into out with a TMA
//     reduce-add (out += partial), whole or not; the order of the f32 additions varies.
//   * store / SwiGLU epilogues: a whole tile is stored directly. A split tile is finished
//     by the contributor that arrives last: the others store their partial accumulators
//     in scratch and bump the tile's arrival counter; the last one adds them to its own,
//     applies the epilogue and resets the counter. No CTA ever waits for another.
//
// Warp roles:
//   warp 0      TMA producer: activation tile (128 x 64 f16, 128-B swizzle) and the
//               stage's packed weight block (bulk copy) into a ring of stages;
//   warps 6..13 dequantise the packed block (one weight row per thread) into a 256 x 64
//               f16 K-major tile in the same swizzled layout: the UMMA B operand;
//   warp 1      allocates 512 TMEM columns (two 128 x 256 f32 accumulators) and one lane
//               issues tcgen05.mma (M=128, N=256, K=16) x 4 per stage, committing each
//               stage back to the ring and each finished segment to the epilogue;
//   warps 2..5  epilogue: tcgen05.ld of 32 rows x 32 columns at a time into registers,
//               then through a per-warp shared staging tile to global memory by TMA
//               (coalesced whole lines), overlapping the next segment's main loop.
// Q1 weights are +-scale, exact in f16, so the f16 tensor-core operand loses nothing.
#include <cuda_fp16.h>

#include <algorithm>
#include <cstdlib>

#include "dequant.cuh"
#include "ptx.cuh"
#include "streamk.cuh"

namespace pf {

void streamk_skew(sk::Plan& p, int late_units, int late_kb) {
  p.late0 = p.ctas;
  p.dk = 0;
  // (the late units are a minority of the units on the GPU the values were measured on; with
  // fewer SMs the pattern is not known, and the plan stays even)
  if (late_units > 0 && late_kb > 0 && 2 * late_units <= p.ctas) {
    p.late0 = p.ctas - late_units;
    p.dk = static_cast<int>(std::min<long long>(late_kb, std::max<long long>(0, p.total / p.ctas - 1)));
  }
}

namespace {
using sk::Plan;
using sk::Range;
using sk::Segment;

constexpr int BM = 128;
constexpr int BN = 256;
constexpr int BK = 64;
constexpr int NUM_EPI_WARPS = 4;
constexpr int NUM_DQ_WARPS = 8;
constexpr int DQ_THREADS = NUM_DQ_WARPS * 32;  // == BN: one weight row per thread
constexpr int EPI_THREADS = NUM_EPI_WARPS * 32;
constexpr int NUM_THREADS = 32 * (2 + NUM_EPI_WARPS + NUM_DQ_WARPS);  // 448
constexpr int FIRST_DQ_WARP = 2 + NUM_EPI_WARPS;
constexpr int LAST_THREADS = EPI_THREADS + DQ_THREADS;  // barrier 3: the last residual epilogue
constexpr int A_STAGE = BM * BK * 2;  // 16 KB
constexpr int STG_BYTES = 32 * 32 * 4;  // per epilogue warp: 32 rows x 32 f32
constexpr int TMEM_COLS = 512;          // two accumulators of 256 f32 columns
constexpr size_t SLOT_FLOATS = static_cast<size_t>(BM) * BN;  // one partial tile
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

// One CTA per tile (PAIR = false): 128 tokens x 256 weight rows, the CTA dequantises all
// 256 rows. A CTA pair (PAIR = true, cta_group::2): 256 tokens x 256 weight rows per pair,
// each CTA loads 128 token rows and dequantises 128 weight rows (its half of B), so a CTA
// moves about two thirds of the shared-memory bytes per k-block (A 16 KB + B half 16 KB read
// by the MMA, 16 KB of dequantised B written, instead of 16 + 32 + 32 KB), and the smaller
// stages allow a deeper ring.
template <int WFMT, bool PAIR>
struct Cfg {
  using F = Fmt<WFMT>;
  static constexpr int B_ROWS = PAIR ? BN / 2 : BN;  // weight rows dequantised per CTA
  static constexpr int TILE_M = PAIR ? 2 * BM : BM;  // tokens per tile
  static constexpr int B_STAGE = B_ROWS * BK * 2;
  // packed bytes per stage: the rows' codes of one 64-wide k-block, then their scales
  // (and zeros)
  static constexpr int P_STAGE = PAIR ? B_ROWS * (WFMT == PF_W_Q1_G128 ? 8 + 2 : 32 + 4) : F::P_STAGE;
  static constexpr int STAGES = PAIR ? (WFMT == PF_W_Q1_G128 ? 6 : 5) : F::STAGES;
  static constexpr int RING = STAGES * (A_STAGE + B_STAGE + P_STAGE);
  static constexpr int SMEM = 1024 /*alignment*/ + (RING + 1023) / 1024 * 1024 + NUM_EPI_WARPS * STG_BYTES +
                              256 /*barriers and flags*/;
  static_assert(SMEM <= 232448, "GEMM shared memory");
  static_assert(RING >= NUM_EPI_WARPS * (BN / 32) * STG_BYTES,
                "the last segment's epilogue stages every chunk in the operand ring");
  static_assert(P_STAGE % 16 == 0 && B_STAGE % 1024 == 0, "stage alignment");
};

// Bounded wait that ignores the abort flag (used while draining after an abort).
__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > PF_WAIT_LIMIT_NS) return;
  }
}

// silu(g) * u = g / (1 + e^-g) * u. The exponent is capped at 80 so the denominator stays
// below 2^126, where the fast division is within 2 ulp; for g < -80 the result is ~1e-33 * u.
__device__ __forceinline__ float silu_mul(float g, float u) {
  return __fdividef(g, 1.0f + __expf(fminf(-g, 80.0f))) * u;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Barrier over `threads` threads that returns whether `pred` held in all of them.
__device__ __forceinline__ bool named_bar_and(int id, int threads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, %2, %3, p;\n"
      " selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(threads)
      : "memory");
  return r != 0;
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

// Pair form: thread (row r of the CTA's 128 weight rows, k half h) -> 4 16-B chunks of the
// 128 x 64 B half tile (same swizzled layout). Stage layout: codes [128 rows][8 (Q1) or 32
// (INT4) bytes], then scales [128] (and INT4 zeros [128]) as f16.
template <int WFMT>
__device__ __forceinline__ void dequant_half_row_pair(const uint8_t* p, int r, int h, uint32_t b_tile) {
  const uint32_t row_base = b_tile + (r >> 3) * 1024 + (r & 7) * 128;
  uint32_t w[16];
  if (WFMT == PF_W_Q1_G128) {
    const uint32_t Z = reinterpret_cast<const uint32_t*>(p + r * 8)[h];
    const uint32_t s16 = reinterpret_cast<const uint16_t*>(p + (BN / 2) * 8)[r];
    dq_q1_32(Z, s16 | (s16 << 16), w);
  } else {
    const uint4 q = reinterpret_cast<const uint4*>(p + r * 32)[h];
    const uint16_t s16 = reinterpret_cast<const uint16_t*>(p + (BN / 2) * 32)[r];
    const uint16_t z16 = reinterpret_cast<const uint16_t*>(p + (BN / 2) * 34)[r];
    dq_i4_32(q, __half2half2(__ushort_as_half(s16)), __half2half2(__ushort_as_half(z16)), w);
  }
#pragma unroll
  for (int c4 = 0; c4 < 4; ++c4) {
    const int c = 4 * h + c4;
    st_shared_v4(row_base + ((c ^ (r & 7)) << 4), w[4 * c4], w[4 * c4 + 1], w[4 * c4 + 2], w[4 * c4 + 3]);
  }
}

// Staging tile of one epilogue warp, f32 32 x 32 in the TMA 128-B swizzle: row r at
// r * 128, 16-B unit j at (j ^ (r % 8)) * 16 (a warp's store of unit j hits all banks).
__device__ __forceinline__ void stage_f32(uint32_t stg, int r, const uint32_t (&v)[32]) {
#pragma unroll
  for (int j = 0; j < 8; ++j)
    st_shared_v4(stg + r * 128 + ((j ^ (r & 7)) << 4), v[4 * j], v[4 * j + 1], v[4 * j + 2],
                 v[4 * j + 3]);
}

// SwiGLU chunk of one epilogue warp: silu(g) * u of 32 rows x 32 columns, f16 in the 64-B
// swizzle of the output box (row r at r * 64, unit j at (j ^ ((r / 2) % 4)) * 16).
__device__ __forceinline__ void stage_swiglu(uint32_t buf, int r, const uint32_t (&g)[32],
                                             const uint32_t (&u)[32]) {
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t pk[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int x = 8 * j + 2 * e;
      const __half2 hv =
          __floats2half2_rn(silu_mul(__uint_as_float(g[x]), __uint_as_float(u[x])),
                            silu_mul(__uint_as_float(g[x + 1]), __uint_as_float(u[x + 1])));
      pk[e] = *reinterpret_cast<const uint32_t*>(&hv);
    }
    st_shared_v4(buf + r * 64 + ((j ^ ((r >> 1) & 3)) << 4), pk[0], pk[1], pk[2], pk[3]);
  }
}

template <int WFMT, int EPI, bool PAIR>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gemm_q_kernel(const __grid_constant__ CUtensorMap tmap_a,
                  const __grid_constant__ CUtensorMap tmap_out, const uint8_t* __restrict__ wpk,
                  int M, int N, int K, Plan plan, float* __restrict__ scratch,
                  int* __restrict__ counters, int* __restrict__ status,
                  float4* __restrict__ side_zero, long long side_zero4) {
  PF_TIMELINE(TL_GEMM + EPI + (PAIR ? 3 : 0));
  using F = Fmt<WFMT>;
  using C = Cfg<WFMT, PAIR>;
  constexpr int S = C::STAGES;
  constexpr int B_STAGE = C::B_STAGE;
  constexpr int P_STAGE = C::P_STAGE;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t a_st = base;
  const uint32_t b_st = a_st + S * A_STAGE;
  const uint32_t p_st = b_st + S * B_STAGE;
  const uint8_t* p_gen = gbase + (p_st - base);
  const uint32_t stg0 = base + (C::RING + 1023) / 1024 * 1024;
  const uint32_t bar0 = stg0 + NUM_EPI_WARPS * STG_BYTES;
  // barriers: full[S], bfull[S], empty[S], acc_full[2], acc_empty[2], drain; then flags
  auto full = [&](int s) { return bar0 + 8u * s; };
  auto bfull = [&](int s) { return bar0 + 8u * (S + s); };
  auto empty = [&](int s) { return bar0 + 8u * (2 * S + s); };
  auto acc_full = [&](int b) { return bar0 + 8u * (3 * S + b); };
  auto acc_empty = [&](int b) { return bar0 + 8u * (3 * S + 2 + b); };
  const uint32_t drain_bar = bar0 + 8u * (3 * S + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + (drain_bar + 8u - base));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + (drain_bar + 16u - base));
  volatile int* flags = reinterpret_cast<volatile int*>(gbase + (drain_bar + 24u - base));  // [4]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // pair form: `rank` 0 issues the MMAs; the plan's unit is the pair
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const int unit = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  griddep_launch_dependents();

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full(s), 1);
      // pair: one arrival per dequantising warp of both CTAs, on the even CTA's barrier
      mbar_init(bfull(s), PAIR ? 2 * NUM_DQ_WARPS : DQ_THREADS);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full(b), 1);
      mbar_init(acc_empty(b), PAIR ? 2 * NUM_EPI_WARPS : EPI_THREADS);
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  // Only the activation tiles and the epilogue's global accesses depend on the previous
  // kernel in the stream (griddep_wait below); the packed weights do not, so the producer
  // issues the first stages' weight copies right after its own barriers exist, before the
  // TMEM allocation, the pair's cluster barrier and the wait.
  const int G = K / GROUP;
  const Range rg(plan, unit);
  const int a_row = static_cast<int>(rank) * BM;  // this CTA's first token row of a tile
  // the stage's packed copies: pair CTAs take their 128 weight rows' codes and scales (zeros)
  auto load_packed = [&](int s, const uint8_t* chunk, int kb) {
    const uint32_t dst = p_st + s * P_STAGE;
    if (!PAIR) {
      bulk_load(dst, chunk + (kb & 1) * F::HALF, F::HALF, full(s));
      bulk_load(dst + F::HALF, chunk + F::META_OFF, F::META, full(s));
    } else {
      constexpr int CODE = WFMT == PF_W_Q1_G128 ? 8 : 32;  // bytes per row and k-block
      const uint8_t* half = chunk + (kb & 1) * F::HALF;
      bulk_load(dst, half + rank * (BN / 2) * CODE, (BN / 2) * CODE, full(s));
      bulk_load(dst + (BN / 2) * CODE, chunk + F::META_OFF + rank * BN, BN, full(s));
      if (WFMT != PF_W_Q1_G128)
        bulk_load(dst + (BN / 2) * (CODE + 2), chunk + F::META_OFF + 2 * BN + rank * BN, BN, full(s));
    }
  };
  __syncthreads();  // this CTA's barriers are initialised
  // Pair: the cluster barrier is split. Each thread arrives once its part of the set-up that
  // the other CTA relies on is done (barriers above; warp 1: this CTA's share of the pair's
  // TMEM) and waits only before its first access to the other CTA (dequantisers, MMA and
  // epilogue warps before their loops; the producer, which never touches it, at the end).
  if (PAIR && warp != 1) cluster_arrive_relaxed();
  int pre = 0;      // (producer thread) stages whose weight copies are issued before the wait
  if (threadIdx.x == 0) {
    for (int k = 0; k < rg.n && pre < S; ++k) {
      const Segment sg = rg.at(plan, k);
      for (int i = 0; i < sg.nkb && pre < S; ++i, ++pre) {
        const int kb = sg.kb0 + i;
        const uint8_t* chunk =
            wpk + (static_cast<size_t>(sg.nt) * G + (kb >> 1)) * static_cast<size_t>(F::CHUNK);
        mbar_arrive_expect_tx(full(pre), A_STAGE + P_STAGE);
        load_packed(pre, chunk, kb);
      }
    }
  }
  if (warp == 1) {
    __syncwarp();
    if (PAIR) {
      tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
      tmem_relinquish_pair();
      tc_fence_before();
      cluster_arrive_release();
    } else {
      tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
      tmem_relinquish();
    }
  }
  // the TMEM address, for every warp but the producer (the dequantisers share the residual
  // form's last epilogue)
  uint32_t tmem_base = 0;
  if (warp >= 1) {
    tc_fence_before();
    named_bar_sync(2, NUM_THREADS - 32);
    tc_fence_after();
    tmem_base = *tmem_slot;
  }
  // Residual form, last segment: its 8 chunks of 32 columns per TMEM lane quarter are drained
  // by the quarter's epilogue warp (share 0) and its two dequantising warps (shares 1, 2),
  // chunks share, share + 3, ... each into a 4 KB buffer of its own in the idle operand ring.
  auto last_resid_chunks = [&](const Segment& sg, uint32_t tb, int row0, int share) {
    const int q = warp & 3;
#pragma unroll 1
    for (int c = share; c < BN / 32; c += 3) {
      uint32_t v[32];
      tmem_ld_32x32b_x32(tb + 32 * c, v);
      tmem_ld_wait();
      const uint32_t buf = a_st + static_cast<uint32_t>(q * (BN / 32) + c) * STG_BYTES;
      stage_f32(buf, lane, v);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_reduce_add_2d(&tmap_out, buf, sg.nt * BN + 32 * c, row0);
        bulk_commit();
      }
    }
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      griddep_wait();  // the activations come from the previous kernel
      for (int k = 0, j = 0; k < rg.n && j < pre; ++k) {
        const Segment sg = rg.at(plan, k);
        for (int i = 0; i < sg.nkb && j < pre; ++i, ++j)
          tma_load_2d(a_st + j * A_STAGE, &tmap_a, (sg.kb0 + i) * BK, sg.mt * C::TILE_M + a_row, full(j));
      }
      int it = 0;
      bool ok = true;
      for (int k = 0; k < rg.n && ok; ++k) {
        const Segment sg = rg.at(plan, k);
        for (int i = 0; i < sg.nkb; ++i, ++it) {
          if (it < pre) continue;  // issued above
          const int s = it % S;
          const uint32_t ph = (it / S) & 1;
          if (!mbar_wait(empty(s), ph ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          const int kb = sg.kb0 + i;
          const uint8_t* chunk =
              wpk + (static_cast<size_t>(sg.nt) * G + (kb >> 1)) * static_cast<size_t>(F::CHUNK);
          mbar_arrive_expect_tx(full(s), A_STAGE + P_STAGE);
          tma_load_2d(a_st + s * A_STAGE, &tmap_a, kb * BK, sg.mt * C::TILE_M + a_row, full(s));
          load_packed(s, chunk, kb);
        }
      }
      if (!ok) {  // let copies already in flight land before shared memory is released
        for (int j = max(0, it - S); j < it; ++j) mbar_wait_drain(full(j % S), (j / S) & 1);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    // The whole warp runs the loop (uniform control flow and operands); one elected lane
    // issues each MMA / commit. Wait outcomes are made warp-uniform by vote. In a pair only
    // the even CTA issues: its bfull / acc_empty barriers count both CTAs' arrivals, and
    // its commits arrive on the same barrier in both CTAs.
    constexpr uint32_t idesc = idesc_f16(C::TILE_M, BN, 0);
    auto mma = [&](uint32_t d, uint64_t ad, uint64_t bd, uint32_t acc) {
      if (PAIR)
        umma_pair_f16_ss_warp(d, ad, bd, idesc, acc);
      else
        umma_f16_ss_warp(d, ad, bd, idesc, acc);
    };
    auto commit = [&](uint32_t bar) {
      if (PAIR)
        umma_pair_commit_warp(bar, 3);
      else
        umma_commit_warp(bar);
    };
    if (PAIR) cluster_wait();  // the other CTA's barriers and TMEM share exist
    int it = 0;
    bool ok = true;
    for (int k = 0; k < (PAIR && rank != 0 ? 0 : rg.n) && ok; ++k) {
      const Segment sg = rg.at(plan, k);
      const int b = k & 1;
      const uint32_t use = static_cast<uint32_t>(k >> 1);
      if (!__all_sync(0xffffffffu, mbar_wait(acc_empty(b), (use & 1) ^ 1, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + b * BN;
      for (int i = 0; i < sg.nkb; ++i, ++it) {
        const int s = it % S;
        const uint32_t ph = (it / S) & 1;
        // (the dequantisers arrive on bfull after their own stage's copies landed)
        ok = __all_sync(0xffffffffu,
                        mbar_wait(bfull(s), ph, abort_flag) && mbar_wait(full(s), ph, abort_flag));
        if (!ok) break;
        tc_fence_after();
        const uint64_t ad = sdesc_kmajor_sw128(a_st + s * A_STAGE);
        const uint64_t bd = sdesc_kmajor_sw128(b_st + s * B_STAGE);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) mma(d_tmem, ad + 2 * kk, bd + 2 * kk, (i | kk) != 0);
        commit(empty(s));
      }
      if (ok) commit(acc_full(b));
    }
    if (!ok) {
      commit(drain_bar);  // wait for any MMA still reading shared memory / TMEM
      mbar_wait_drain(drain_bar, 0);
    }
  } else if (warp >= FIRST_DQ_WARP) {
    // ---------------------------------------------------------------- dequantisers
    const int d = threadIdx.x - FIRST_DQ_WARP * 32;  // weight row of the tile (pair: row + 128 half)
    if (PAIR) cluster_wait();  // before the first arrival on the even CTA's barriers
    int it = 0;
    bool ok = true;
    for (int k = 0; k < rg.n && ok; ++k) {
      const Segment sg = rg.at(plan, k);
      for (int i = 0; i < sg.nkb; ++i, ++it) {
        const int s = it % S;
        const uint32_t ph = (it / S) & 1;
        if (!mbar_wait(full(s), ph, abort_flag)) {
          ok = false;
          break;
        }
        if (PAIR) {
          dequant_half_row_pair<WFMT>(p_gen + s * P_STAGE, d & (BN / 2 - 1), d / (BN / 2), b_st + s * B_STAGE);
          fence_proxy_async_smem();  // this CTA's shared memory, read by the pair's MMA
          __syncwarp();
          if (lane == 0) {
            if (rank == 0)
              mbar_arrive(bfull(s));
            else
              mbar_arrive_cta(bfull(s), 0);
          }
        } else {
          dequant_row_smem<WFMT>(p_gen + s * P_STAGE, d, b_st + s * B_STAGE);
          fence_proxy_async_smem();
          mbar_arrive(bfull(s));
        }
      }
    }
    if (EPI == EPI_RESID_ADD && rg.n > 0) {
      // the epilogue warps meet these warps on barrier 3 once the last accumulator is ready
      if (named_bar_and(3, LAST_THREADS, ok)) {
        tc_fence_after();
        const int k = rg.n - 1;
        const Segment sg = rg.at(plan, k);
        const int q = warp & 3;
        const int row0 = sg.mt * C::TILE_M + a_row + 32 * q;
        last_resid_chunks(sg, tmem_base + (k & 1) * BN + (static_cast<uint32_t>(32 * q) << 16), row0,
                          warp < FIRST_DQ_WARP + 4 ? 1 : 2);
      }
      tc_fence_before();
      if (lane == 0) bulk_wait0();
      __syncwarp();
    }
  } else {
    // ---------------------------------------------------------------- epilogue (warps 2..5)
    griddep_wait();  // out / scratch / counters are shared with the previous kernels
    const int q = warp & 3;           // TMEM lane quarter this warp may read
    const int et = threadIdx.x - 64;  // 0..127
    if (side_zero != nullptr) {
      // idle until the first accumulator is ready: clear this CTA's share of the buffer a
      // later kernel accumulates into
      const long long per = (side_zero4 + gridDim.x - 1) / gridDim.x;
      const long long z1 = min(side_zero4, per * (blockIdx.x + 1));
      for (long long i = per * blockIdx.x + et; i < z1; i += EPI_THREADS)
        __stcg(side_zero + i, make_float4(0.f, 0.f, 0.f, 0.f));
    }
    if (PAIR) cluster_wait();
    const uint32_t stg = stg0 + q * STG_BYTES;
    // hands a staging tile (after its 32 x 32 values were written) to TMA
    auto stage_out = [&](uint32_t buf, int x, int y) {
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        if (EPI == EPI_RESID_ADD)
          tma_reduce_add_2d(&tmap_out, buf, x, y);
        else
          tma_store_2d(&tmap_out, buf, x, y);
        bulk_commit();
      }
    };
    bool met_last = false;  // residual form: barrier 3 with the dequantising warps passed
    for (int k = 0; k < rg.n; ++k) {
      // The last segment's epilogue runs after the main loop has ended, when the operand ring
      // is idle (its last MMA has completed): each 32-column chunk then gets a 4 KB buffer of
      // its own there, so no chunk waits for the TMA read of the one before. Earlier segments
      // share this warp's staging tile and wait for it.
      const bool last = k == rg.n - 1;
      auto stage_buf = [&](int c) {
        if (last) return a_st + static_cast<uint32_t>(q * (BN / 32) + c) * STG_BYTES;
        if (lane == 0) bulk_wait_read0();  // the previous TMA store has read the tile
        __syncwarp();
        return stg;
      };
      const Segment sg = rg.at(plan, k);
      const int b = k & 1;
      const uint32_t use = static_cast<uint32_t>(k >> 1);
      // uniform over the four epilogue warps: tcgen05.ld is warp-collective and the partial
      // hand-off synchronises the four warps
      const bool got = mbar_wait(acc_full(b), use & 1, abort_flag);
      if (!named_bar_and(1, EPI_THREADS, got)) break;
      tc_fence_after();
      const int row0 = sg.mt * C::TILE_M + a_row + 32 * q;  // first row of this warp's quarter
      const int lrow = 32 * q + lane;        // row within the tile
      const bool valid = row0 + lane < M;
      const uint32_t tb = tmem_base + b * BN + (static_cast<uint32_t>(32 * q) << 16);

      if (EPI == EPI_RESID_ADD && last) {
        // out += the last segment's partial sum (whole tile or not): this warp's share, after
        // handing the rest to the dequantising warps
        met_last = true;
        named_bar_and(3, LAST_THREADS, true);
        last_resid_chunks(sg, tb, row0, 0);
      } else if (EPI == EPI_RESID_ADD) {
        // out += this segment's partial sum, through the warp's staging tile
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tb + 32 * c, v);
          tmem_ld_wait();
          const uint32_t buf = stage_buf(c);
          stage_f32(buf, lane, v);
          stage_out(buf, sg.nt * BN + 32 * c, row0);
        }
      } else {
        // ---- a tile split across CTAs: hand the partial off, or finish the tile if last.
        // Partials are float4 [chunk 0..7][j 0..7][tile row 0..127]: a warp's store or load
        // of one (chunk, j) covers 512 contiguous bytes.
        bool finish = sg.whole;
        int c_lo = 0, c_hi = -1;
        if (!sg.whole) {
          c_lo = plan.owner(static_cast<long long>(sg.tile) * plan.kbt);
          c_hi = plan.owner(static_cast<long long>(sg.tile + 1) * plan.kbt - 1);
          const int others = c_hi - c_lo;  // contributors besides this CTA
          const int slot = plan.slot(unit, sg.tile);
          // a pair tile's two row halves are finished independently, one counter each
          int* ctr = counters + (PAIR ? 2 * sg.tile + static_cast<int>(rank) : sg.tile);
          volatile int* flag = flags + 2 * slot;  // each slot serves one segment only
          // if every other contributor has arrived already, finish without storing
          if (et == 0) flag[0] = ld_acquire_gpu(ctr) == others ? 1 : 0;
          named_bar_sync(1, EPI_THREADS);
          finish = flag[0] != 0;
          if (!finish) {
            float4* mine = reinterpret_cast<float4*>(scratch) +
                           (static_cast<size_t>(blockIdx.x) * 2 + slot) * (SLOT_FLOATS / 4) + lrow;
#pragma unroll 1
            for (int c = 0; c < BN / 32; ++c) {
              uint32_t v[32];
              tmem_ld_32x32b_x32(tb + 32 * c, v);
              tmem_ld_wait();
              if (valid) {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                  __stcg(mine + (c * 8 + j) * BM,
                         make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                     __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3])));
              }
            }
            __threadfence();
            named_bar_sync(1, EPI_THREADS);
            if (et == 0) flag[1] = atomicAdd(ctr, 1) == others ? 1 : 0;
            named_bar_sync(1, EPI_THREADS);
            finish = flag[1] != 0;
          }
          if (finish) {
            if (et == 0) *ctr = 0;  // every contributor is in: ready for reuse
            __threadfence();
          }
        }
        // adds the other contributors' partials of 32-column chunk `chunk` of this row to v
        auto add_partials = [&](uint32_t (&v)[32], int chunk) {
          for (int c = c_lo; c <= c_hi; ++c) {
            if (c == unit) continue;
            const int cta = PAIR ? 2 * c + static_cast<int>(rank) : c;  // same row half
            const float4* src = reinterpret_cast<const float4*>(scratch) +
                                (static_cast<size_t>(cta) * 2 + plan.slot(c, sg.tile)) * (SLOT_FLOATS / 4) +
                                lrow;
            float4 x[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) x[j] = __ldcg(src + (chunk * 8 + j) * BM);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
              v[4 * j] = __float_as_uint(__uint_as_float(v[4 * j]) + x[j].x);
              v[4 * j + 1] = __float_as_uint(__uint_as_float(v[4 * j + 1]) + x[j].y);
              v[4 * j + 2] = __float_as_uint(__uint_as_float(v[4 * j + 2]) + x[j].z);
              v[4 * j + 3] = __float_as_uint(__uint_as_float(v[4 * j + 3]) + x[j].w);
            }
          }
        };

        if (finish && EPI == EPI_SWIGLU) {
          // each 128 columns of the tile: 64 gate columns, then the 64 matching up columns
#pragma unroll 1
          for (int c = 0; c < 4; ++c) {
            const int h = c >> 1, q2 = c & 1;
            uint32_t g[32], u[32];
            tmem_ld_32x32b_x32(tb + 128 * h + 32 * q2, g);
            tmem_ld_32x32b_x32(tb + 128 * h + 64 + 32 * q2, u);
            tmem_ld_wait();
            if (!sg.whole && valid) {
              add_partials(g, 4 * h + q2);
              add_partials(u, 4 * h + 2 + q2);
            }
            const uint32_t buf = stage_buf(c);
            stage_swiglu(buf, lane, g, u);
            stage_out(buf, sg.nt * 128 + 64 * h + 32 * q2, row0);
          }
        } else if (finish) {
#pragma unroll 1
          for (int c = 0; c < BN / 32; ++c) {
            uint32_t v[32];
            tmem_ld_32x32b_x32(tb + 32 * c, v);
            tmem_ld_wait();
            if (!sg.whole && valid) add_partials(v, c);
            const uint32_t buf = stage_buf(c);
            stage_f32(buf, lane, v);
            stage_out(buf, sg.nt * BN + 32 * c, row0);
          }
        }
      }
      tc_fence_before();
      if (PAIR) {
        __syncwarp();
        if (lane == 0) {
          if (rank == 0)
            mbar_arrive(acc_empty(b));
          else
            mbar_arrive_cta(acc_empty(b), 0);
        }
      } else {
        mbar_arrive(acc_empty(b));
      }
    }
    if (EPI == EPI_RESID_ADD && rg.n > 0 && !met_last) named_bar_and(3, LAST_THREADS, false);
    // this CTA's TMEM reads and arrivals on the other CTA are done: arrive on the end barrier
    // before the last TMA writes drain
    tc_fence_before();
    if (PAIR) cluster_arrive_release();
    if (lane == 0) bulk_wait0();  // TMA writes complete before the CTA retires
    __syncwarp();
  }

  if (PAIR && warp == 0) cluster_wait();  // the producer's wait of the split start-up barrier
  // A pair's CTAs stay until both are done with each other: the even CTA's MMAs read the odd
  // one's shared memory and write its TMEM, the odd one arrives on the even one's barriers.
  // The end barrier is split as well (the epilogue warps arrived above).
  tc_fence_before();
  __syncwarp();
  if (PAIR) {
    if (warp < 2 || warp >= FIRST_DQ_WARP) cluster_arrive_release();
    cluster_wait();
  } else {
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    __syncwarp();  // reconverge before the collective dealloc
    if (PAIR)
      tmem_dealloc_pair(tmem_base, TMEM_COLS);
    else
      tmem_dealloc(tmem_base, TMEM_COLS);
  }
  if (threadIdx.x == 0 && *abort_flag && status != nullptr) atomicCAS(status, 0, PF_ERR_DEVICE_TIMEOUT);
}

template <int WFMT, int EPI, bool PAIR>
cudaError_t launch_t(const GemmArgs& g, const CUtensorMap& ta, const CUtensorMap& to, int num_sms,
                     cudaStream_t stream) {
  using C = Cfg<WFMT, PAIR>;
  Plan p{};
  p.n_mt = (g.M + C::TILE_M - 1) / C::TILE_M;
  p.n_nt = static_cast<int>(padded_rows(g.N) / TILE_N);
  p.kbt = g.K / BK;
  p.total = static_cast<long long>(p.n_mt) * p.n_nt * p.kbt;
  // the plan's units: CTAs, or CTA pairs (no more pairs than can be resident at once)
  int units = std::min(g.max_ctas, num_sms) / (PAIR ? 2 : 1);
  if (PAIR) {
    static const int resident = [] {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2);
      cfg.blockDim = dim3(NUM_THREADS);
      cfg.dynamicSmemBytes = C::SMEM;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, gemm_q_kernel<WFMT, EPI, true>, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
      }
      return n;
    }();
    if (resident > 0) units = std::min(units, resident);
  }
  p.ctas = static_cast<int>(std::min<long long>(units, p.total));
  // store / SwiGLU epilogues: a tile split between units costs a partial hand-off, so when
  // the tiles alone fill at least half of the units, run one whole tile per unit instead
  const int tiles = p.n_mt * p.n_nt;
  if (EPI != EPI_RESID_ADD && tiles < p.ctas && 2 * tiles >= p.ctas) p.ctas = tiles;
  streamk_skew(p, PAIR ? g.late_units : 0, g.late_kb);
  float* scratch = reinterpret_cast<float*>(g.scratch);
  int* counters =
      scratch ? reinterpret_cast<int*>(scratch + static_cast<size_t>(2) * g.max_ctas * SLOT_FLOATS) : nullptr;
  float4* zero = reinterpret_cast<float4*>(g.side_zero);
  const long long zero4 = static_cast<long long>(g.side_zero_bytes / 16);
  if (PAIR)
    return launch_pdl_pairs(gemm_q_kernel<WFMT, EPI, true>, dim3(2 * p.ctas), dim3(NUM_THREADS), C::SMEM,
                            stream, ta, to, g.w, g.M, g.N, g.K, p, scratch, counters, g.status, zero, zero4);
  return launch_pdl(gemm_q_kernel<WFMT, EPI, false>, dim3(p.ctas), dim3(NUM_THREADS), C::SMEM, stream, ta,
                    to, g.w, g.M, g.N, g.K, p, scratch, counters, g.status, zero, zero4);
}

// CTA pairs for more than one 128-token block (PF_GEMM_PAIRS=0 in the environment turns
// them off, to compare the two forms).
bool use_pairs(const GemmArgs& g, int sms) {
  static const bool enabled = [] {
    const char* e = getenv("PF_GEMM_PAIRS");
    return e == nullptr || atoi(e) != 0;
  }();
  return enabled && g.M > BM && std::min(g.max_ctas, sms) >= 2;
}

}  // namespace


// Scratch of a launch with at most max_ctas CTAs: two partial tiles per CTA (a CTA's range
// begins and ends inside at most two tiles), then one arrival counter per output tile, which
// must be zero before the first launch (every launch that completes leaves them zero).
size_t gemm_scratch_bytes(int M, int N, int max_ctas) {
  // one counter per 128 x 256 tile, or two per 256 x 256 pair tile (one per row half); the
  // small-M kernel's 256-row tiles are fewer
  const size_t nt = static_cast<size_t>(padded_rows(N) / TILE_N);
  const size_t tiles = std::max<size_t>((M + BM - 1) / BM, 2 * ((M + 2 * BM - 1) / (2 * BM))) * nt;
  return static_cast<size_t>(2) * max_ctas * SLOT_FLOATS * sizeof(float) + tiles * sizeof(int);
}

template <int WFMT, int EPI, bool PAIR>
cudaError_t set_smem_attr() {
  return cudaFuncSetAttribute(gemm_q_kernel<WFMT, EPI, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              Cfg<WFMT, PAIR>::SMEM);
}

cudaError_t prepare_gemm_kernels() {
  cudaError_t e = cudaSuccess;
  cudaError_t r;
  if ((r = set_smem_attr<PF_W_Q1_G128, EPI_RESID_ADD, false>()) != cudaSuccess) e = r;
  if ((r = set_smem_attr<PF_W_Q1_G128, EPI_SWIGLU, false>()) != cudaSuccess) e = r;
  if ((r = set_smem_attr<PF_W_INT4_AFFINE_G128, EPI_RESID_ADD, false>()) != cudaSuccess) e = r;
  if ((r = set_smem_attr<PF_W_INT4_AFFINE_G128, EPI_SWIGLU, false>()) != cudaSuccess) e = r;
  if ((r = set_smem_attr<PF_W_Q1_G128, EPI_RESID_ADD, true>()) != cudaSuccess) e = r;
  if ((r = set_smem_attr<PF_W_Q1_G128, EPI_SWIGLU, true>()) != cudaSuccess) e = r;
  if ((r = set_smem_attr<PF_W_INT4_AFFINE_G128, EPI_RESID_ADD, true>()) != cudaSuccess) e = r;
  if ((r = set_smem_attr<PF_W_INT4_AFFINE_G128, EPI_SWIGLU, true>()) != cudaSuccess) e = r;
  return e;
}

bool gemm_side_zero_supported(int wfmt, int M) { return M > gemv_max_m(wfmt) && M > SMALL_M_MAX; }

cudaError_t launch_gemm(const GemmArgs& g, cudaStream_t stream) {
  if (g.side_zero != nullptr && (g.M <= SMALL_M_MAX || g.M <= gemv_max_m(g.wfmt) ||
                                 g.side_zero_bytes % 16 != 0 ||
                                 reinterpret_cast<uintptr_t>(g.side_zero) % 16 != 0))
    return cudaErrorInvalidValue;
  if (g.M <= gemv_max_m(g.wfmt)) return launch_gemv(g, stream);
  if (g.M <= SMALL_M_MAX) return launch_gemm_small(g, stream);
  if (g.epilogue == EPI_STORE_F32) {
    // accumulate every CTA's share into a zeroed output by TMA reduce-add (no partial
    // hand-off, all SMs busy), as the residual form does
    if (!g.out_zeroed) {
      cudaError_t e = cudaMemsetAsync(g.out, 0, static_cast<size_t>(g.M) * g.N * sizeof(float), stream);
      if (e != cudaSuccess) return e;
    }
    GemmArgs r = g;
    r.epilogue = EPI_RESID_ADD;
    return launch_gemm(r, stream);
  }
  CUtensorMap ta, to;
  if (!encode_tmap_f16_2d(&ta, g.a, static_cast<uint64_t>(g.K), static_cast<uint64_t>(g.M), BK, BM))
    return cudaErrorInvalidValue;
  const bool swiglu = g.epilogue == EPI_SWIGLU;
  // 32 x 32 output boxes: f32 rows of 128 B (128-B swizzle) or f16 rows of 64 B (64-B swizzle)
  if (!encode_tmap_out_2d(&to, !swiglu, g.out, static_cast<uint64_t>(swiglu ? g.N / 2 : g.N),
                          static_cast<uint64_t>(g.M), 32, 32, swiglu ? 64 : 128))
    return cudaErrorInvalidValue;
  static int sms = device_sm_count();
  const bool pair = use_pairs(g, sms);
  const bool q1 = g.wfmt == PF_W_Q1_G128;
  constexpr int Q1 = PF_W_Q1_G128, I4 = PF_W_INT4_AFFINE_G128;
  if (swiglu) {
    if (q1) return pair ? launch_t<Q1, EPI_SWIGLU, true>(g, ta, to, sms, stream)
                        : launch_t<Q1, EPI_SWIGLU, false>(g, ta, to, sms, stream);
    return pair ? launch_t<I4, EPI_SWIGLU, true>(g, ta, to, sms, stream)
                : launch_t<I4, EPI_SWIGLU, false>(g, ta, to, sms, stream);
  }
  if (g.epilogue != EPI_RESID_ADD) return cudaErrorInvalidValue;
  if (q1) return pair ? launch_t<Q1, EPI_RESID_ADD, true>(g, ta, to, sms, stream)
                      : launch_t<Q1, EPI_RESID_ADD, false>(g, ta, to, sms, stream);
  return pair ? launch_t<I4, EPI_RESID_ADD, true>(g, ta, to, sms, stream)
              : launch_t<I4, EPI_RESID_ADD, false>(g, ta, to, sms, stream);
}

}  // namespace pf

PF_TIMELINE_SETTER(gemm_q)
