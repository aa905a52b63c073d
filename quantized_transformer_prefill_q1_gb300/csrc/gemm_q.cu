// gemm_q.cu — quantised GEMM on the 5th-generation tensor cores (tcgen05 / TMEM).
//
// out[m, n] (+)= sum_k a[m, k] * w[n, k] with a = f16 activations [M, K] (the RMSNorm /
// SwiGLU / attention outputs) and w a packed Q1 or INT4-affine weight [N, K]. This is
// the batched projection of oxibonsai-kernels metal_prefill.rs `encode_layer_prefill`:
// section 2 (QKV GEMM, plain store), sections 4 and 7 (O / down GEMM with the residual
// add fused, `dispatch_gemm_q1_v7_residual`) and section 6 (gate+up GEMM with SwiGLU
// fused, `dispatch_fused_gate_up_swiglu_gemm`).
//
// The dequantised weights never touch shared memory: they are written with tcgen05.st
// straight into tensor memory and used as the MMA's A operand (D[weight row][token] =
// W_tile x A_tokens^T), so shared memory only carries the activation tile (TMA in, MMA
// out) and the small packed-weight stream. Persistent CTAs (one per SM) walk work units
// = (128-row weight tile, 128-token tile, K split). Warp roles:
//   warp 0       TMA producer of the activation ring (128 tokens x 128 k per stage, as
//                two 64-k atoms in the 128-B swizzle layout);
//   warp 22      bulk-copy producer of the packed-weight ring (128 rows x one 128-weight
//                scale group per stage);
//   warps 6..21  dequantisers: warp w owns TMEM lane quarter w % 4 (32 weight rows) and
//                one 32-wide quarter of the stage's 128 k; each thread turns its row's sign
//                bits (or nibbles) into 16 f16x2 words and stores them with one tcgen05.st
//                into the stage's A slot (64 TMEM columns per 128 k);
//   warp 1       allocates all 512 TMEM columns (two 128 x 128 f32 accumulators + four A
//                slots) and one lane issues tcgen05.mma (A from TMEM, B = activations
//                from shared memory; M=128, N=128, K=16) x 8 per stage;
//   warps 2..5   epilogue: tcgen05.ld of a finished accumulator (thread = weight row,
//                registers = 32 tokens), f32 store / residual add / SwiGLU, overlapping
//                the next unit's main loop in the other accumulator.
// Q1 weights are +-scale, exact in f16, so the f16 tensor-core operand loses nothing.
#include <cuda_fp16.h>

#include "dequant.cuh"
#include "ptx.cuh"

namespace pf {
namespace {

constexpr int BW = 128;  // weight rows per unit (MMA M, TMEM lanes)
constexpr int BT = 128;  // tokens per unit (MMA N)
constexpr int BK = 128;  // k per stage (one scale group)
constexpr int NUM_EPI_WARPS = 4;
constexpr int NUM_DQ_WARPS = 16;  // 4 per TMEM lane quarter, one 32-k quarter each
constexpr int FIRST_DQ_WARP = 2 + NUM_EPI_WARPS;
constexpr int PK_WARP = FIRST_DQ_WARP + NUM_DQ_WARPS;
constexpr int NUM_THREADS = 32 * (PK_WARP + 1);  // 736
constexpr int DQ_THREADS = NUM_DQ_WARPS * 32;
constexpr int EPI_THREADS = NUM_EPI_WARPS * 32;
constexpr int B_STAGE = BT * BK * 2;  // 32 KB activation tile (two 64-k swizzle atoms)
constexpr int B_ATOM = BT * 128;      // one 64-k atom: 128 tokens x 128 B
constexpr int SB = 4;                 // activation ring depth
constexpr int SA = 4;                 // A slots in TMEM (64 columns each)
constexpr int A_SLOT_COLS = BK / 2;   // f16 pairs per row
constexpr int ACC_COLS = BT;          // one accumulator: 128 f32 columns
constexpr int A_COL0 = 2 * ACC_COLS;  // A slots after the two accumulators
constexpr int TMEM_COLS = 512;
constexpr int STAGE_BYTES = 64 * 32 * 4;  // SwiGLU epilogue staging: 64 rows x 32 tokens f32
static_assert(A_COL0 + SA * A_SLOT_COLS == TMEM_COLS, "TMEM budget");

template <int WFMT>
struct Fmt;
template <>
struct Fmt<PF_W_Q1_G128> {
  static constexpr int CHUNK = Q1_CHUNK_BYTES;
  static constexpr int HALF = Q1_HALF_BYTES;  // 256 rows x 8 B for one 64-k half of a chunk
  static constexpr int ROWB = 8;              // bytes per row per 64-k half
  static constexpr int META_OFF = Q1_SCALE_OFF;
  static constexpr int NMETA = 1;             // scales
  static constexpr int P_STAGE = 2 * BW * ROWB + BW * 2 * NMETA;  // 2304
  static constexpr int SP = 12;
};
template <>
struct Fmt<PF_W_INT4_AFFINE_G128> {
  static constexpr int CHUNK = I4_CHUNK_BYTES;
  static constexpr int HALF = I4_HALF_BYTES;
  static constexpr int ROWB = 32;
  static constexpr int META_OFF = I4_SCALE_OFF;
  static constexpr int NMETA = 2;             // scales, zeros
  static constexpr int P_STAGE = 2 * BW * ROWB + BW * 2 * NMETA;  // 8704
  static constexpr int SP = 6;
};

template <int WFMT>
constexpr int smem_bytes() {
  using F = Fmt<WFMT>;
  return 1024 /*alignment slack*/ + SB * B_STAGE + F::SP * F::P_STAGE + STAGE_BYTES +
         512 /*barriers and flags*/;
}

// Bounded wait that ignores the abort flag (used while draining after an abort).
__device__ __forceinline__ void mbar_wait_drain(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > PF_WAIT_LIMIT_NS) return;
  }
}

__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.0f + __expf(-g)) * u; }

// D[tmem] (+)= A[tmem] * B[smem]^T, kind::f16.
__device__ __forceinline__ void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tmem_st_x16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

struct Units {
  int n_tt, n_wt, per_split, nkb_total;
  __device__ __forceinline__ void decode(int u, int& tt, int& wt, int& kb0, int& nkb) const {
    const int tiles = n_tt * n_wt;
    const int split = u / tiles;
    const int r = u - split * tiles;
    wt = r / n_tt;
    tt = r - wt * n_tt;  // token tiles fastest: neighbouring CTAs share a weight tile
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
  constexpr int SP = F::SP;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t b_st = base;
  const uint32_t p_st = b_st + SB * B_STAGE;
  const uint8_t* p_gen = gbase + (p_st - base);
  const uint32_t stg = p_st + SP * F::P_STAGE;
  float* stage_f = reinterpret_cast<float*>(gbase + (stg - base));
  const uint32_t bar0 = stg + STAGE_BYTES;
  // barriers: fullB/emptyB [SB], fullA/emptyA [SA], fullP/emptyP [SP], acc_full/acc_empty
  // [2], drain; then the abort flag and the TMEM address slot
  auto full_b = [&](int s) { return bar0 + 8u * s; };
  auto empty_b = [&](int s) { return bar0 + 8u * (SB + s); };
  auto full_a = [&](int s) { return bar0 + 8u * (2 * SB + s); };
  auto empty_a = [&](int s) { return bar0 + 8u * (2 * SB + SA + s); };
  auto full_p = [&](int s) { return bar0 + 8u * (2 * SB + 2 * SA + s); };
  auto empty_p = [&](int s) { return bar0 + 8u * (2 * SB + 2 * SA + SP + s); };
  const uint32_t acc0 = bar0 + 8u * (2 * SB + 2 * SA + 2 * SP);
  auto acc_full = [&](int b) { return acc0 + 8u * b; };
  auto acc_empty = [&](int b) { return acc0 + 8u * (2 + b); };
  const uint32_t drain_bar = acc0 + 8u * 4;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + (drain_bar + 8u - base));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + (drain_bar + 16u - base));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < SB; ++s) {
      mbar_init(full_b(s), 1);
      mbar_init(empty_b(s), 1);
    }
    for (int s = 0; s < SA; ++s) {
      mbar_init(full_a(s), DQ_THREADS);
      mbar_init(empty_a(s), 1);
    }
    for (int s = 0; s < SP; ++s) {
      mbar_init(full_p(s), 1);
      mbar_init(empty_p(s), DQ_THREADS);
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
  const int G = K / GROUP;

  if (warp == 0 || warp == PK_WARP) {
    // ---------------------------------------------------------------- producers
    if (lane == 0) {
      const bool act = warp == 0;  // activation ring, else packed-weight ring
      const int S = act ? SB : SP;
      int it = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
        int tt, wt, kb0, nkb;
        units.decode(u, tt, wt, kb0, nkb);
        for (int i = 0; i < nkb; ++i, ++it) {
          const int s = it % S;
          const uint32_t ph = (it / S) & 1;
          if (!mbar_wait(act ? empty_b(s) : empty_p(s), ph ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          const int kb = kb0 + i;
          if (act) {
            mbar_arrive_expect_tx(full_b(s), B_STAGE);
            tma_load_2d(b_st + s * B_STAGE, &tmap_a, kb * BK, tt * BT, full_b(s));
            tma_load_2d(b_st + s * B_STAGE + B_ATOM, &tmap_a, kb * BK + 64, tt * BT, full_b(s));
          } else {
            // 128-row half (wt & 1) of the 256-row chunk (wt >> 1, group kb): both 64-k
            // halves of the rows' codes, then their scales (and zeros)
            const uint8_t* chunk =
                wpk + (static_cast<size_t>(wt >> 1) * G + kb) * static_cast<size_t>(F::CHUNK);
            const int r0 = (wt & 1) * BW;
            const uint32_t dst = p_st + s * F::P_STAGE;
            mbar_arrive_expect_tx(full_p(s), F::P_STAGE);
            bulk_load(dst, chunk + r0 * F::ROWB, BW * F::ROWB, full_p(s));
            bulk_load(dst + BW * F::ROWB, chunk + F::HALF + r0 * F::ROWB, BW * F::ROWB, full_p(s));
            bulk_load(dst + 2 * BW * F::ROWB, chunk + F::META_OFF + r0 * 2, BW * 2, full_p(s));
            if (F::NMETA == 2)
              bulk_load(dst + 2 * BW * F::ROWB + BW * 2, chunk + F::META_OFF + TILE_N * 2 + r0 * 2,
                        BW * 2, full_p(s));
          }
        }
      }
      if (!ok) {  // let copies already in flight land before shared memory is released
        for (int j = max(0, it - S); j < it; ++j)
          mbar_wait_drain(act ? full_b(j % S) : full_p(j % S), (j / S) & 1);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16(BW, BT, 0);
      int it = 0, local = 0;
      bool ok = true;
      for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++local) {
        int tt, wt, kb0, nkb;
        units.decode(u, tt, wt, kb0, nkb);
        const int b = local & 1;
        const uint32_t use = static_cast<uint32_t>(local >> 1);
        if (!mbar_wait(acc_empty(b), (use & 1) ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + b * ACC_COLS;
        for (int i = 0; i < nkb; ++i, ++it) {
          const int sa = it % SA, sb = it % SB;
          if (!(mbar_wait(full_a(sa), (it / SA) & 1, abort_flag) &&
                mbar_wait(full_b(sb), (it / SB) & 1, abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_tmem = tmem_base + A_COL0 + sa * A_SLOT_COLS;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t bd = sdesc_kmajor_sw128(b_st + sb * B_STAGE + (kk >> 2) * B_ATOM) + 2 * (kk & 3);
            umma_f16_ts(d_tmem, a_tmem + 8 * kk, bd, idesc, (i | kk) != 0);
          }
          umma_commit(empty_a(sa));
          umma_commit(empty_b(sb));
        }
        if (ok) umma_commit(acc_full(b));
      }
      if (!ok) {
        umma_commit(drain_bar);  // wait for any MMA still reading shared / tensor memory
        mbar_wait_drain(drain_bar, 0);
      }
    }
  } else if (warp >= FIRST_DQ_WARP) {
    // ---------------------------------------------------------------- dequantisers
    const int quarter = warp & 3;
    const int kq = (warp - FIRST_DQ_WARP) >> 2;     // which 32 of the stage's 128 k
    const int khalf = kq >> 1, kword = kq & 1;
    const int r = 32 * quarter + lane;              // weight row of the tile
    const uint32_t lane_off = static_cast<uint32_t>(32 * quarter) << 16;
    int it = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
      int tt, wt, kb0, nkb;
      units.decode(u, tt, wt, kb0, nkb);
      for (int i = 0; i < nkb; ++i, ++it) {
        const int sp = it % SP, sa = it % SA;
        // warp-uniform outcome: tcgen05.st below is warp-collective
        if (!__all_sync(0xffffffffu, mbar_wait(full_p(sp), (it / SP) & 1, abort_flag) &&
                                         mbar_wait(empty_a(sa), ((it / SA) & 1) ^ 1, abort_flag))) {
          ok = false;
          break;
        }
        const uint8_t* p = p_gen + sp * F::P_STAGE;
        uint32_t w[16];
        if (WFMT == PF_W_Q1_G128) {
          const uint32_t Z = reinterpret_cast<const uint32_t*>(p + khalf * (BW * 8) + r * 8)[kword];
          const uint32_t s16 = reinterpret_cast<const uint16_t*>(p + 2 * BW * 8)[r];
          dq_q1_32(Z, s16 | (s16 << 16), w);
        } else {
          const uint4 q = reinterpret_cast<const uint4*>(p + khalf * (BW * 32) + r * 32)[kword];
          const uint16_t s16 = reinterpret_cast<const uint16_t*>(p + 2 * BW * 32)[r];
          const uint16_t z16 = reinterpret_cast<const uint16_t*>(p + 2 * BW * 32 + BW * 2)[r];
          dq_i4_32(q, __half2half2(__ushort_as_half(s16)), __half2half2(__ushort_as_half(z16)), w);
        }
        tmem_st_x16(tmem_base + lane_off + A_COL0 + sa * A_SLOT_COLS + 16 * kq, w);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(full_a(sa));
        mbar_arrive(empty_p(sp));
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue (warps 2..5)
    const int quarter = warp & 3;  // TMEM lane quarter this warp may read
    const int et = threadIdx.x - 64;  // 0..127
    int local = 0;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++local) {
      int tt, wt, kb0, nkb;
      units.decode(u, tt, wt, kb0, nkb);
      const int b = local & 1;
      const uint32_t use = static_cast<uint32_t>(local >> 1);
      // warp-uniform: the tcgen05.ld below is warp-collective
      if (!__all_sync(0xffffffffu, mbar_wait(acc_full(b), use & 1, abort_flag))) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + b * ACC_COLS + (static_cast<uint32_t>(32 * quarter) << 16);
      const int t0 = tt * BT;
      if (EPI == EPI_SWIGLU) {
        // tile rows 0..63 are gate rows of features wt*64 + 0..63, rows 64..127 the
        // matching up rows: up warps stage their values, gate warps combine and store
        const int NO = N >> 1;
        __half* o = reinterpret_cast<__half*>(out);
        const bool up = quarter >= 2;
        const int frow = 32 * (quarter & 1) + lane;  // 0..63
        const int f = wt * 64 + frow;
#pragma unroll 1
        for (int c = 0; c < BT / 32; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tb + 32 * c, v);
          tmem_ld_wait();
          if (up) {
#pragma unroll
            for (int e = 0; e < 32; ++e) stage_f[e * 64 + frow] = __uint_as_float(v[e]);
          }
          named_bar_sync(1, EPI_THREADS);
          if (!up && f < NO) {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int t = t0 + 32 * c + e;
              if (t < M)
                o[static_cast<size_t>(t) * NO + f] =
                    __float2half_rn(silu_mul(__uint_as_float(v[e]), stage_f[e * 64 + frow]));
            }
          }
          named_bar_sync(1, EPI_THREADS);
        }
      } else {
        float* o = reinterpret_cast<float*>(out);
        const int n = wt * BW + 32 * quarter + lane;
#pragma unroll 1
        for (int c = 0; c < BT / 32; ++c) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tb + 32 * c, v);
          tmem_ld_wait();
          if (n < N) {
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              const int t = t0 + 32 * c + e;
              if (t < M) {
                float* dst = o + static_cast<size_t>(t) * N + n;
                const float val = __uint_as_float(v[e]);
                if (atomic_out)
                  atomicAdd(dst, val);
                else if (EPI == EPI_RESID_ADD)
                  *dst += val;
                else
                  *dst = val;
              }
            }
          }
        }
      }
      (void)et;
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
  u.n_tt = (g.M + BT - 1) / BT;
  u.n_wt = static_cast<int>(padded_rows(g.N) / BW);
  u.nkb_total = nkb;
  const int n_units = u.n_tt * u.n_wt * splits;
  const int grid = min(n_units, num_sms);
  gemm_q_kernel<WFMT, EPI><<<grid, NUM_THREADS, smem, stream>>>(tm, g.w, g.M, g.N, g.K, g.out, u,
                                                              n_units, splits > 1 ? 1 : 0, g.status);
  return cudaGetLastError();
}

}  // namespace

bool encode_tmap_f16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                        uint32_t box_inner, uint32_t box_outer);

// Split along K when that shortens the critical path: cost = rounds of units per SM x
// k-blocks per unit (+ a fixed per-unit overhead), with persistent CTAs.
int choose_split_k(int M, int N, int K, int epilogue, int num_sms) {
  if (epilogue == EPI_SWIGLU) return 1;
  const int tiles = static_cast<int>(padded_rows(N) / BW) * ((M + BT - 1) / BT);
  const int nkb = K / BK;
  int best = 1;
  double best_cost = 1e30;
  for (int s = 1; s <= 16 && s <= nkb / 4; ++s) {
    const int per = (nkb + s - 1) / s;
    const int splits = (nkb + per - 1) / per;
    const int rounds = (tiles * splits + num_sms - 1) / num_sms;
    const double cost = rounds * (per + 3.0) + (s > 1 ? 2.0 : 0.0);
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
  // 64-wide boxes (128 B, the swizzle span); each stage loads two of them
  if (!encode_tmap_f16_2d(&tm, g.a, static_cast<uint64_t>(g.K), static_cast<uint64_t>(g.M), 64, BT))
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
