// attention_tc.cu — causal GQA attention of a chunk of query rows over the KV cache on
// the 5th-generation tensor cores (tcgen05 / TMEM), for 16-bit caches.
//
// The method: oxibonsai-kernels metal_prefill.rs `encode_layer_prefill` section 3 (for
// each query position, scores q.k_j * inv_sqrt_hd over the seq_len = pos + 1 cached keys
// of its kv head h / heads_per_group, softmax, weighted sum of V), batched over the chunk
// as in turbospark-runtime prefill.rs `encode_attention_decode_batch`.
//
// One CTA = one kv head and 128 query rows (128/G tokens x the G query heads that share
// the kv head; row = token * G + head-in-group), so every row reads the same K/V tiles.
// The probabilities P stay in tensor memory as the A operand of the PV product:
//   warp 0      TMA: the Q tile once (3-D map over q[M][nq][hd]), then 128-key K and V tiles
//               straight from the cache [layer][kvh][pos][hd] into two 3-stage rings; a K
//               stage is free again once its QK^T is done, so K runs a tile ahead of V;
//   warp 1      TMEM (512 columns: three S buffers of 128 and O) and the MMAs, issued by
//               the whole warp with one elected lane: S_0, S_1, then per tile
//               O += P_j V_j (P from TMEM over S_j's columns, V used MN-major as it lies in
//               the cache) followed by S_{j+2} = Q K_{j+2}^T, so the scores of the next
//               tile are ready before the softmax reaches it;
//   warps 2..9  softmax, two threads per query row: warp w reads TMEM lane quarter w % 4
//               and takes key columns [0, 64) (warps 2..5) or [64, 128) (warps 6..9) of
//               each tile. Per tile: read S_j,
//               causal mask (key > pos: -inf), row max combined with the partner thread
//               through shared memory, online softmax in the exp2 domain, P_j (bf16/f16)
//               back into TMEM; the running max is raised only when a tile's max exceeds it
//               by more than 2^8 (then O is rescaled in TMEM), so probabilities stay <= 256
//               and f32 accumulation is exact enough; final O / l to f16.
// Every wait is bounded; a timeout aborts the CTA and records PF_ERR_DEVICE_TIMEOUT.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace pf {
namespace {

constexpr int TQ = 128;          // query rows per CTA (MMA M)
constexpr int TK = 128;          // keys per tile
constexpr int KS = 3;            // K and V ring stages
constexpr int THREADS = 320;     // warp 0 TMA, warp 1 MMA, warps 2..9 softmax
constexpr int SM_THREADS = 256;  // softmax threads: two per query row
constexpr int HK = TK / 2;       // keys per softmax thread and tile
constexpr int NSB = 3;           // S / P buffers in TMEM
constexpr float RESCALE_LOG2 = 8.0f;
// TMEM columns: S buffers b at b TK (P_j over the first TK/2 columns of its buffer), O at 3 TK
constexpr uint32_t COL_O = NSB * TK;

template <int HD>
struct ASmem {
  static constexpr int Q = TQ * HD * 2;
  static constexpr int KV = TK * HD * 2;  // one K or V tile
  static constexpr int RED = 2 * TQ * 4;  // partner exchange: [half][row] f32
  static constexpr int BYTES = 1024 + Q + 2 * KS * KV + RED + 256;
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
                   const __grid_constant__ CUtensorMap tm_v, int M, int nq, int nkv, int max_seq, int layer,
                   const int* __restrict__ start_dev, int start_host, float scale_log2,
                   __half* __restrict__ out, int* __restrict__ status) {
  using L = ASmem<HD>;
  constexpr int NH = HD / 64;  // 64-wide (128-B) swizzle regions along head_dim
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t q_s = base;
  const uint32_t k_s = q_s + L::Q;          // K stage s at k_s + s * KV
  const uint32_t v_s = k_s + KS * L::KV;    // V stage s at v_s + s * KV
  const uint32_t red_s = v_s + KS * L::KV;
  const uint32_t bar0 = red_s + L::RED;
  auto k_full = [&](int s) { return bar0 + 8u * s; };
  auto k_empty = [&](int s) { return bar0 + 8u * (KS + s); };
  auto v_full = [&](int s) { return bar0 + 8u * (2 * KS + s); };
  auto v_empty = [&](int s) { return bar0 + 8u * (3 * KS + s); };
  auto s_full = [&](int b) { return bar0 + 8u * (4 * KS + b); };
  auto s_empty = [&](int b) { return bar0 + 8u * (4 * KS + NSB + b); };
  auto p_full = [&](int b) { return bar0 + 8u * (4 * KS + 2 * NSB + b); };
  constexpr int NB = 4 * KS + 3 * NSB;  // barriers so far
  const uint32_t q_full = bar0 + 8u * NB;
  const uint32_t o_done = bar0 + 8u * (NB + 1);
  const uint32_t o_final = bar0 + 8u * (NB + 2);
  const uint32_t drain_bar = bar0 + 8u * (NB + 3);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + (bar0 + 8u * (NB + 4) - base));
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + (bar0 + 8u * (NB + 5) - base));
  static_assert(8 * (NB + 6) <= 256, "barrier area");
  auto k_tile = [&](int s) { return k_s + s * L::KV; };
  auto v_tile = [&](int s) { return v_s + s * L::KV; };

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
    for (int s = 0; s < KS; ++s) {
      mbar_init(k_full(s), 1);
      mbar_init(k_empty(s), 1);
      mbar_init(v_full(s), 1);
      mbar_init(v_empty(s), 1);
    }
    for (int b = 0; b < NSB; ++b) {
      mbar_init(s_full(b), 1);
      mbar_init(s_empty(b), 1);
      mbar_init(p_full(b), SM_THREADS);
    }
    mbar_init(q_full, 1);
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
  const uint32_t tmem_o = tmem + COL_O;

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
          const int s = i % KS;
          if (!mbar_wait(k_empty(s), ((i / KS) & 1) ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(k_full(s), L::KV);
          for (int h = 0; h < NH; ++h)
            tma_load_2d(k_tile(s) + h * (TK * 128), &tm_k, h * 64, row0 + i * TK, k_full(s));
          ++k_issued;
        }
        if (i >= 1) {
          const int jv = i - 1, s = jv % KS;
          if (!mbar_wait(v_empty(s), ((jv / KS) & 1) ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(v_full(s), L::KV);
          for (int h = 0; h < NH; ++h)
            tma_load_2d(v_tile(s) + h * (TK * 128), &tm_v, h * 64, row0 + jv * TK, v_full(s));
          ++v_issued;
        }
      }
      if (*abort_flag) {  // let copies already in flight land before shared memory is released
        mbar_wait_drain_a(q_full, 0);
        for (int j = max(0, k_issued - KS); j < k_issued; ++j) mbar_wait_drain_a(k_full(j % KS), (j / KS) & 1);
        for (int j = max(0, v_issued - KS); j < v_issued; ++j) mbar_wait_drain_a(v_full(j % KS), (j / KS) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop (uniform control flow and operands); one elected lane
    // issues each MMA / commit. Wait outcomes are made warp-uniform by vote.
    constexpr uint32_t idesc_s = idesc_f16(TQ, TK, BF16, 0);
    constexpr uint32_t idesc_o = idesc_f16(TQ, HD, BF16, 1);
    // S_j = Q K_j^T into S buffer j % 3
    auto issue_s = [&](int j) -> bool {
      const int sb = j % NSB, ks = j % KS;
      if (!__all_sync(0xffffffffu, mbar_wait(k_full(ks), (j / KS) & 1, abort_flag) &&
                                       mbar_wait(s_empty(sb), ((j / NSB) & 1) ^ 1, abort_flag)))
        return false;
      tc_fence_after();
#pragma unroll
      for (int kc = 0; kc < HD / 16; ++kc) {
        const uint32_t off = (kc >> 2) * (TQ * 128) + (kc & 3) * 32;
        const uint32_t offk = (kc >> 2) * (TK * 128) + (kc & 3) * 32;
        umma_f16_ss_warp(tmem + sb * TK, sdesc_kmajor_sw128(q_s + off),
                         sdesc_kmajor_sw128(k_tile(ks) + offk), idesc_s, kc > 0);
      }
      umma_commit_warp(s_full(sb));
      umma_commit_warp(k_empty(ks));  // K_j is free once QK^T is done
      return true;
    };
    bool ok = __all_sync(0xffffffffu, mbar_wait(q_full, 0, abort_flag));
    if (ok) ok = issue_s(0);
    if (ok && n_tiles > 1) ok = issue_s(1);
    for (int j = 0; j < n_tiles && ok; ++j) {
      // O += P_j V_j, P from TMEM over S_j's columns
      const int sb = j % NSB, vs = j % KS;
      if (!__all_sync(0xffffffffu, mbar_wait(p_full(sb), (j / NSB) & 1, abort_flag) &&
                                       mbar_wait(v_full(vs), (j / KS) & 1, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int kc = 0; kc < TK / 16; ++kc)
        umma_f16_ts_warp(tmem_o, tmem + sb * TK + 8 * kc,
                         sdesc_mnmajor_sw128(v_tile(vs) + kc * 2048, TK * 128), idesc_o,
                         (j > 0 || kc > 0));
      umma_commit_warp(s_empty(sb));  // P_j consumed: S buffer reusable
      umma_commit_warp(v_empty(vs));
      umma_commit_warp(o_done);
      if (j + 2 < n_tiles) ok = issue_s(j + 2);
    }
    if (ok) {
      umma_commit_warp(o_final);
    } else {
      umma_commit_warp(drain_bar);
      mbar_wait_drain_a(drain_bar, 0);
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
      const int s = j % NSB;
      const bool got = mbar_wait(s_full(s), (j / NSB) & 1, abort_flag);
      if (!named_bar_and_a(1, SM_THREADS, got && !failed)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t sbuf = tmem + lane_off + s * TK;
      const int kbase = j * TK + half * HK;  // first key of this thread's columns
      uint32_t v[HK];
#pragma unroll
      for (int c = 0; c < HK / 32; ++c)
        tmem_ld_32x32b_x32(sbuf + half * HK + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(v + 32 * c));
      tmem_ld_wait();
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
      // both partners have read their S columns before either writes P over them
      tc_fence_before();
      named_bar_sync_a(1, SM_THREADS);
      tc_fence_after();
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
      const float neg_m = -m;
      float rsp[4] = {0.f, 0.f, 0.f, 0.f};  // independent partial row sums
      uint32_t pk[HK / 2];                  // this thread's 64 probabilities, packed in pairs
#pragma unroll
      for (int x = 0; x < HK; x += 2) {
        float p0 = ex2_approx(fmaf(__uint_as_float(v[x]), scale_log2, neg_m));
        float p1 = ex2_approx(fmaf(__uint_as_float(v[x + 1]), scale_log2, neg_m));
        if (diag) {
          p0 = (kbase + x <= pos) ? p0 : 0.f;
          p1 = (kbase + x + 1 <= pos) ? p1 : 0.f;
        }
        rsp[(x >> 1) & 3] += p0 + p1;
        pk[x >> 1] = pack_pair<BF16>(p0, p1);
      }
      l += (rsp[0] + rsp[1]) + (rsp[2] + rsp[3]);
      // P_j over the first TK/2 columns of S buffer s: keys 2c, 2c+1 in column c
      tmem_st_32x32b_x32(sbuf + half * (HK / 2), pk);
      if (j == n_tiles - 1 && j * TK + r >= kv_len) {
        // key row r of this tile lies past the cache's filled range: zero its V row (once
        // the tile has landed) so a zero probability never meets a stale NaN / Inf in the
        // PV product
        const int vs = j % KS;
        if (!mbar_wait(v_full(vs), (j / KS) & 1, abort_flag)) failed = true;
        for (int h = half; h < NH; h += 2)
          for (int ch = 0; ch < 8; ++ch) st_shared_v4a(v_tile(vs) + h * (TK * 128) + r * 128 + ch * 16, 0, 0, 0, 0);
        fence_proxy_async_smem();
      }
      tmem_st_wait();
      tc_fence_before();
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
                    M, c.n_q_heads, c.n_kv_heads, c.max_seq, layer, start_dev, start_host,
                    scale_log2, reinterpret_cast<__half*>(out), status);
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
