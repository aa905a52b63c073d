// attention_tc.cu — causal GQA attention of a chunk of query rows over the KV cache on
// the 5th-generation tensor cores (tcgen05 / TMEM), for 16-bit caches.
//
// The method: oxibonsai-kernels metal_prefill.rs `encode_layer_prefill` section 3 (for
// each query position, scores q.k_j * inv_sqrt_hd over the seq_len = pos + 1 cached keys
// of its kv head h / heads_per_group, softmax, weighted sum of V), batched over the chunk
// as in turbospark-runtime prefill.rs `encode_attention_decode_batch`.
//
// One CTA = one kv head and 128 query rows (128/G tokens x the G query heads that share
// the kv head; row = token * G + head-in-group), so every row reads the same K/V tiles:
//   warp 0      TMA: the Q tile once (3-D map over q[M][nq][hd]), then 128-key K and V
//               tiles straight from the cache [layer][kvh][pos][hd] into two 2-stage rings;
//               a K stage is free again once its QK^T is done, so K runs a tile ahead of V;
//   warp 1      TMEM (512 columns: two S buffers of 128 + the O accumulator) and the MMAs:
//               S_j = Q K_j^T (K-major operands), then O += P_{j-1} V_{j-1} (V used
//               MN-major, as it lies in the cache), so QK^T of tile j overlaps the softmax
//               of tile j-1;
//   warps 2..9  softmax, two threads per query row: warp w reads TMEM lane quarter w % 4
//               and takes key columns [0, 64) (warps 2..5) or [64, 128) (warps 6..9) of
//               each tile, so two warps per scheduler hide each other's latency. Read
//               S_j from TMEM, causal mask (key > pos: -inf), row max combined with the
//               partner thread through shared memory, online softmax in the exp2 domain,
//               P_j (bf16/f16) into shared memory; the running max is raised only when a
//               tile's max exceeds it by more than 2^8 (then O is rescaled in TMEM), so
//               probabilities stay <= 256 and f32 accumulation is exact enough; final
//               O / l to f16.
// Every wait is bounded; a timeout aborts the CTA and records PF_ERR_DEVICE_TIMEOUT.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace pf {
namespace {

constexpr int TQ = 128;       // query rows per CTA (MMA M)
constexpr int TK = 128;       // keys per tile
constexpr int THREADS = 320;  // warp 0 TMA, warp 1 MMA, warps 2..9 softmax
constexpr int SM_THREADS = 256;  // softmax threads: two per query row
constexpr int HK = TK / 2;       // keys per softmax thread and tile
constexpr float RESCALE_LOG2 = 8.0f;

template <int HD>
struct ASmem {
  static constexpr int Q = TQ * HD * 2;
  static constexpr int KV = TK * HD * 2;  // one of K or V
  static constexpr int P = TQ * TK * 2;
  static constexpr int RED = 2 * TQ * 4;  // partner exchange: [half][row] f32
  static constexpr int BYTES = 1024 + Q + 2 * 2 * KV + 2 * P + RED + 256;
  static_assert(BYTES <= 232448, "attention shared memory");
};

__device__ __forceinline__ void mbar_wait_drain_a(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > PF_WAIT_LIMIT_NS) return;
  }
}

__device__ __forceinline__ void named_bar_sync_a(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Barrier over `threads` threads that returns whether `pred` held in all of them.
__device__ __forceinline__ bool named_bar_and_a(int id, int threads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, %2, %3, p;\n"
      " selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(threads)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ void st_shared_v4a(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                              uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// 2^x with the hardware approximation (relative error ~2^-22; subnormal results flush to
// zero, which for probabilities below 2^-126 is immaterial).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int BF16>
__device__ __forceinline__ uint32_t pack_pair(float a, float b) {
  if (BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

template <int HD, int BF16>
__global__ void __launch_bounds__(THREADS, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, int M, int nq, int nkv, int max_seq,
                   int layer, const int* __restrict__ start_dev, int start_host, float scale_log2,
                   __half* __restrict__ out, int* __restrict__ status) {
  using L = ASmem<HD>;
  constexpr int NH = HD / 64;  // 64-wide (128-B) swizzle regions along head_dim
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t q_s = base;
  const uint32_t kv_s = q_s + L::Q;  // stage s: K at kv_s + 2s*KV, V at kv_s + (2s+1)*KV
  const uint32_t p_s = kv_s + 4 * L::KV;
  const uint32_t red_s = p_s + 2 * L::P;
  const uint32_t bar0 = red_s + L::RED;
  const uint32_t q_full = bar0;
  auto k_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto k_empty = [&](int s) { return bar0 + 8u * (3 + s); };
  auto v_full = [&](int s) { return bar0 + 8u * (5 + s); };
  auto v_empty = [&](int s) { return bar0 + 8u * (7 + s); };
  auto s_full = [&](int s) { return bar0 + 8u * (9 + s); };
  auto s_empty = [&](int s) { return bar0 + 8u * (11 + s); };
  auto p_full = [&](int s) { return bar0 + 8u * (13 + s); };
  auto p_empty = [&](int s) { return bar0 + 8u * (15 + s); };
  const uint32_t o_done = bar0 + 8u * 17;
  const uint32_t o_final = bar0 + 8u * 18;
  const uint32_t drain_bar = bar0 + 8u * 19;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + (bar0 + 160u - base));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + (bar0 + 168u - base));
  auto k_tile = [&](int s) { return kv_s + (2 * s) * L::KV; };
  auto v_tile = [&](int s) { return kv_s + (2 * s + 1) * L::KV; };

  griddep_launch_dependents();
  griddep_wait();  // the start position and q / cache come from earlier kernels
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = nq / nkv;
  const int BT = TQ / G;  // tokens per CTA
  const int n_tt = (M + BT - 1) / BT;
  const int tt = n_tt - 1 - static_cast<int>(blockIdx.x);  // longest rows first
  const int kvh = blockIdx.y;
  const int t0 = tt * BT;
  const int start = start_dev ? *start_dev : start_host;
  const int kv_len = start + min(t0 + BT, M);
  const int n_tiles = (kv_len + TK - 1) / TK;
  const int row0 = (layer * nkv + kvh) * max_seq;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), 1);
      mbar_init(s_full(s), 1);
      mbar_init(s_empty(s), SM_THREADS);
      mbar_init(p_full(s), SM_THREADS);
      mbar_init(p_empty(s), 1);
    }
    mbar_init(o_done, 1);
    mbar_init(o_final, 1);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_o = tmem + 256;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, L::Q);
      for (int h = 0; h < NH; ++h)
        tma_load_3d(q_s + h * (TQ * 128), &tm_q, h * 64, kvh * G, t0, q_full);
      // K_i, then V_{i-1}: K runs one tile ahead of V
      int k_issued = 0, v_issued = 0;
      bool ok = true;
      for (int i = 0; i <= n_tiles && ok; ++i) {
        if (i < n_tiles) {
          const int s = i & 1;
          if (!mbar_wait(k_empty(s), ((i >> 1) & 1) ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(k_full(s), L::KV);
          for (int h = 0; h < NH; ++h)
            tma_load_2d(k_tile(s) + h * (TK * 128), &tm_k, h * 64, row0 + i * TK, k_full(s));
          ++k_issued;
        }
        if (i >= 1) {
          const int jv = i - 1, s = jv & 1;
          if (!mbar_wait(v_empty(s), ((jv >> 1) & 1) ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(v_full(s), L::KV);
          for (int h = 0; h < NH; ++h)
            tma_load_2d(v_tile(s) + h * (TK * 128), &tm_v, h * 64, row0 + jv * TK, v_full(s));
          ++v_issued;
        }
      }
      if (*abort_flag) {
        mbar_wait_drain_a(q_full, 0);
        for (int j = max(0, k_issued - 2); j < k_issued; ++j) mbar_wait_drain_a(k_full(j & 1), (j >> 1) & 1);
        for (int j = max(0, v_issued - 2); j < v_issued; ++j) mbar_wait_drain_a(v_full(j & 1), (j >> 1) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_f16(TQ, TK, BF16, 0);
      constexpr uint32_t idesc_o = idesc_f16(TQ, HD, BF16, 1);
      bool ok = mbar_wait(q_full, 0, abort_flag);
      for (int j = 0; j <= n_tiles && ok; ++j) {
        if (j < n_tiles) {  // S_j = Q K_j^T
          const int s = j & 1;
          if (!(mbar_wait(k_full(s), (j >> 1) & 1, abort_flag) &&
                mbar_wait(s_empty(s), ((j >> 1) & 1) ^ 1, abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kc = 0; kc < HD / 16; ++kc) {
            const uint32_t off = (kc >> 2) * (TQ * 128) + (kc & 3) * 32;
            const uint32_t offk = (kc >> 2) * (TK * 128) + (kc & 3) * 32;
            umma_f16_ss(tmem + s * TK, sdesc_kmajor_sw128(q_s + off),
                        sdesc_kmajor_sw128(k_tile(s) + offk), idesc_s, kc > 0);
          }
          umma_commit(s_full(s));
          umma_commit(k_empty(s));  // K_j is free once QK^T is done
        }
        if (j >= 1) {  // O += P_{j-1} V_{j-1}
          const int i = j - 1, s = i & 1;
          if (!(mbar_wait(p_full(s), (i >> 1) & 1, abort_flag) &&
                mbar_wait(v_full(s), (i >> 1) & 1, abort_flag))) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kc = 0; kc < TK / 16; ++kc) {
            const uint32_t offp = s * L::P + (kc >> 2) * (TQ * 128) + (kc & 3) * 32;
            umma_f16_ss(tmem_o, sdesc_kmajor_sw128(p_s + offp),
                        sdesc_mnmajor_sw128(v_tile(s) + kc * 2048, TK * 128), idesc_o,
                        (i > 0 || kc > 0));
          }
          umma_commit(p_empty(s));
          umma_commit(v_empty(s));
          umma_commit(o_done);
        }
      }
      if (ok) {
        umma_commit(o_final);
      } else {
        umma_commit(drain_bar);
        mbar_wait_drain_a(drain_bar, 0);
      }
    }
  } else {
    // ------------------------------------------------------------------ softmax rows
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;  // key columns [64 half, 64 half + 64) of each tile
    const int r = 32 * quarter + lane;
    const uint32_t lane_off = static_cast<uint32_t>(32 * quarter) << 16;
    const int t_loc = r / G, h_loc = r - (r / G) * G;
    const int pos = start + t0 + t_loc;
    volatile float* red = reinterpret_cast<volatile float*>(gbase + (red_s - base));  // [2][TQ]
    float m = -INFINITY, l = 0.f;
    bool ok = true, failed = false;
    // tcgen05.ld / tcgen05.st are warp-collective: every branch around them is warp-uniform.
    // The 256 softmax threads meet at named barrier 1 twice per tile; a failed wait is
    // carried to the next barrier-and, where all of them stop together.
    for (int j = 0; j < n_tiles; ++j) {
      const int s = j & 1;
      const bool got = mbar_wait(s_full(s), (j >> 1) & 1, abort_flag);
      if (!named_bar_and_a(1, SM_THREADS, got && !failed)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t sbuf = tmem + lane_off + s * TK + half * HK;
      const int kbase = j * TK + half * HK;  // first key of this thread's columns
      uint32_t v[HK];
#pragma unroll
      for (int c = 0; c < HK / 32; ++c)
        tmem_ld_32x32b_x32(sbuf + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(v + 32 * c));
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(s_empty(s));  // S_j is in registers: the MMA may reuse its columns
      // a tile wholly at or below the CTA's first position needs no causal mask
      const bool diag = j * TK + TK - 1 > start + t0;
      float mp[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mp[i] = -INFINITY;
      if (diag) {
#pragma unroll
        for (int e = 0; e < HK; ++e)
          if (kbase + e <= pos) mp[e & 7] = fmaxf(mp[e & 7], __uint_as_float(v[e]));
      } else {
#pragma unroll
        for (int e = 0; e < HK; ++e) mp[e & 7] = fmaxf(mp[e & 7], __uint_as_float(v[e]));
      }
      float mraw = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                         fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
      red[half * TQ + r] = mraw;
      named_bar_sync_a(1, SM_THREADS);
      mraw = fmaxf(mraw, red[(1 - half) * TQ + r]);  // the row's max over all 128 keys
      const float mx = mraw * scale_log2;  // scale > 0 keeps the order
      const bool need = j > 0 && mx > m + RESCALE_LOG2;
      if (j == 0) {
        m = mx;  // key 0 is visible to every row, so this is finite
      } else if (__any_sync(0xffffffffu, need)) {
        // some row of this warp raises its max: the warp rescales its half of those O rows,
        // the rows that keep their max with alpha = 1 (the partner warp decides the same)
        const float alpha = need ? exp2f(m - mx) : 1.0f;
        l *= alpha;
        // O holds P_0..P_{j-1} V: wait for PV_{j-1}, then scale it in place
        if (__all_sync(0xffffffffu, mbar_wait(o_done, (j - 1) & 1, abort_flag))) {
          tc_fence_after();
#pragma unroll 1
          for (int c = half * (HD / 64); c < (half + 1) * (HD / 64); ++c) {
            uint32_t o[32];
            tmem_ld_32x32b_x32(tmem_o + lane_off + 32 * c, o);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st_32x32b_x32(tmem_o + lane_off + 32 * c, o);
          }
          tmem_st_wait();
        } else {
          failed = true;
        }
        if (need) m = mx;
      }
      if (!failed && !mbar_wait(p_empty(s), ((j >> 1) & 1) ^ 1, abort_flag)) failed = true;
      const uint32_t pbuf = p_s + s * L::P;
      const float neg_m = -m;
      float rsp[4] = {0.f, 0.f, 0.f, 0.f};  // independent partial row sums
      if (!failed) {
        // keys 8ch .. 8ch+7 of this thread: K-atom `half`, chunk ch within it
        const uint32_t row_base = pbuf + half * (TQ * 128) + r * 128;
#pragma unroll
        for (int ch = 0; ch < HK / 8; ++ch) {
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const int x = 8 * ch + e;
            float p0 = ex2_approx(fmaf(__uint_as_float(v[x]), scale_log2, neg_m));
            float p1 = ex2_approx(fmaf(__uint_as_float(v[x + 1]), scale_log2, neg_m));
            if (diag) {
              p0 = (kbase + x <= pos) ? p0 : 0.f;
              p1 = (kbase + x + 1 <= pos) ? p1 : 0.f;
            }
            rsp[e >> 1] += p0 + p1;
            pk[e >> 1] = pack_pair<BF16>(p0, p1);
          }
          st_shared_v4a(row_base + ((ch ^ (r & 7)) << 4), pk[0], pk[1], pk[2], pk[3]);
        }
        l += (rsp[0] + rsp[1]) + (rsp[2] + rsp[3]);
        if (j == n_tiles - 1 && j * TK + r >= kv_len) {
          // key row r of this tile lies past the cache's filled range: zero its V row (once
          // the tile has landed) so a zero probability never meets a stale NaN / Inf in the
          // PV product
          if (!mbar_wait(v_full(s), (j >> 1) & 1, abort_flag)) failed = true;
          for (int h = half; h < NH; h += 2)
            for (int ch = 0; ch < 8; ++ch) st_shared_v4a(v_tile(s) + h * (TK * 128) + r * 128 + ch * 16, 0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(p_full(s));
    }
    // ------------------------------------------------------------------ epilogue
    const bool fin = ok && !failed && mbar_wait(o_final, 0, abort_flag);
    const bool all_ok = named_bar_and_a(1, SM_THREADS, fin);  // partners are done with red
    red[half * TQ + r] = l;
    named_bar_sync_a(1, SM_THREADS);
    if (all_ok) {
      tc_fence_after();
      const float inv = 1.f / (l + red[(1 - half) * TQ + r]);
      const int t = t0 + t_loc;
      const int h = kvh * G + h_loc;
#pragma unroll 1
      for (int c = half * (HD / 64); c < (half + 1) * (HD / 64); ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem_o + lane_off + 32 * c, v);
        tmem_ld_wait();
        if (t < M) {
          uint4* dst = reinterpret_cast<uint4*>(out + (static_cast<size_t>(t) * nq + h) * HD + 32 * c);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __half2 hv = __floats2half2_rn(__uint_as_float(v[8 * q4 + 2 * e]) * inv,
                                                   __uint_as_float(v[8 * q4 + 2 * e + 1]) * inv);
              w[e] = *reinterpret_cast<const uint32_t*>(&hv);
            }
            dst[q4] = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    __syncwarp();  // lane 0 ran the MMA loop: reconverge before the collective dealloc
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && *abort_flag && status != nullptr) atomicCAS(status, 0, PF_ERR_DEVICE_TIMEOUT);
}

template <int HD, int BF16>
cudaError_t launch_tc(const pf_config& c, const void* q, const void* kc, const void* vc, int layer,
                      const int* start_dev, int start_host, int M, void* out, int* status,
                      cudaStream_t st) {
  const int G = c.n_q_heads / c.n_kv_heads;
  const int BT = TQ / G;
  const uint64_t rows = static_cast<uint64_t>(c.n_layers) * c.n_kv_heads * c.max_seq;
  CUtensorMap tq, tk, tv;
  const uint64_t qd[3] = {static_cast<uint64_t>(HD), static_cast<uint64_t>(c.n_q_heads),
                          static_cast<uint64_t>(M)};
  const uint64_t qs[2] = {static_cast<uint64_t>(HD) * 2, static_cast<uint64_t>(c.n_q_heads) * HD * 2};
  const uint32_t qb[3] = {64, static_cast<uint32_t>(G), static_cast<uint32_t>(BT)};
  const uint64_t kd[2] = {static_cast<uint64_t>(HD), rows};
  const uint64_t ks[1] = {static_cast<uint64_t>(HD) * 2};
  const uint32_t kb[2] = {64, static_cast<uint32_t>(TK)};
  if (!encode_tmap_16(&tq, BF16, 3, q, qd, qs, qb) || !encode_tmap_16(&tk, BF16, 2, kc, kd, ks, kb) ||
      !encode_tmap_16(&tv, BF16, 2, vc, kd, ks, kb))
    return cudaErrorInvalidValue;
  dim3 grid((M + BT - 1) / BT, c.n_kv_heads);
  const float scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(HD));
  return launch_pdl(attn_tc_kernel<HD, BF16>, grid, dim3(THREADS), ASmem<HD>::BYTES, st, tq, tk, tv,
                    M, c.n_q_heads, c.n_kv_heads, c.max_seq, layer, start_dev, start_host, scale_log2,
                    reinterpret_cast<__half*>(out), status);
}

template <int HD, int BF16>
cudaError_t set_attr_tc() {
  return cudaFuncSetAttribute(attn_tc_kernel<HD, BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              ASmem<HD>::BYTES);
}

}  // namespace

bool attention_tc_supported(const pf_config& c) {
  const int G = c.n_q_heads / c.n_kv_heads;
  return (c.kv_dtype == PF_KV_BF16 || c.kv_dtype == PF_KV_F16) &&
         (c.head_dim == 128 || c.head_dim == 64) && G >= 1 && TQ % G == 0;
}

cudaError_t prepare_attention_tc_kernels() {
  cudaError_t e = cudaSuccess, r;
  if ((r = set_attr_tc<128, 1>()) != cudaSuccess) e = r;
  if ((r = set_attr_tc<128, 0>()) != cudaSuccess) e = r;
  if ((r = set_attr_tc<64, 1>()) != cudaSuccess) e = r;
  if ((r = set_attr_tc<64, 0>()) != cudaSuccess) e = r;
  return e;
}

cudaError_t launch_attention_tc(const pf_config& c, const void* q, const void* k_cache,
                                const void* v_cache, int layer, const int* start_dev, int start_host,
                                int M, void* out, int* status, cudaStream_t stream) {
  const bool bf = c.kv_dtype == PF_KV_BF16;
  if (c.head_dim == 128)
    return bf ? launch_tc<128, 1>(c, q, k_cache, v_cache, layer, start_dev, start_host, M, out, status, stream)
              : launch_tc<128, 0>(c, q, k_cache, v_cache, layer, start_dev, start_host, M, out, status, stream);
  return bf ? launch_tc<64, 1>(c, q, k_cache, v_cache, layer, start_dev, start_host, M, out, status, stream)
            : launch_tc<64, 0>(c, q, k_cache, v_cache, layer, start_dev, start_host, M, out, status, stream);
}

}  // namespace pf
