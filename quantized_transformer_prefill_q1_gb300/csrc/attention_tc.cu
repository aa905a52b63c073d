// attention_tc.cu — causal GQA attention of a chunk of query rows over the KV cache on
// the 5th-generation tensor cores (tcgen05 / TMEM), for 16-bit caches.
//
// The method: oxibonsai-kernels metal_prefill.rs `encode_layer_prefill` section 3 (for
// each query position, scores q.k_j * inv_sqrt_hd over the seq_len = pos + 1 cached keys
// of its kv head h / heads_per_group, softmax, weighted sum of V), batched over the chunk
// as in turbospark-runtime prefill.rs `encode_attention_decode_batch`. With a ring cache
// (the batch-attention contract's ring_capacity R and sink_count S on the same page) the
// query at position p sees the S sink positions and the R - S most recent positions up to p.
//
// One CTA = one kv head and 128 query rows (128/G tokens x the G query heads that share
// the kv head; row = token * G + head-in-group), so every row reads the same K/V tiles.
// The keys the CTA's rows may see form a list of 128-key tiles (KeyTiles below): a linear
// cache gives one run of positions 0 .. last; a ring cache gives the history sinks, the
// history window (in ring slots, wrapping once) and the chunk's own keys (read from the chunk
// buffers the QK-norm / RoPE kernel wrote, since the chunk's later tokens may overwrite ring
// slots its earlier tokens still need). With n_split > 1 the tile list is cut into n_split
// contiguous parts, one CTA each (split-KV, for chunks too small to fill the GPU); each part
// writes its unnormalised O, running max and sum, and attn_combine_kernel merges them.
//
// Warp roles:
//   warp 0      TMA: the Q tile once (3-D map over q[M][nq][hd]), then the K and V tiles
//               into two 3-stage rings; a K stage is free again once its QK^T is done, so
//               K runs a tile ahead of V;
//   warp 1      TMEM (512 columns: three S buffers of 128 and O) and the MMAs, issued by
//               the whole warp with one elected lane: S_0, S_1, then per tile
//               O += P_j V_j (P from TMEM over S_j's columns, V used MN-major as it lies in
//               the cache) followed by S_{j+2} = Q K_{j+2}^T;
//   warps 2..9  softmax, two threads per query row: warp w reads TMEM lane quarter w % 4
//               and takes key columns [0, 64) (warps 2..5) or [64, 128) (warps 6..9) of
//               each tile. Per tile: read S_j, mask keys the row may not see, row max
//               combined with the partner thread through shared memory, online softmax in
//               the exp2 domain, P_j (bf16/f16) back into TMEM; the running max is raised
//               only when a tile's max exceeds it by more than 2^8 (then O is rescaled in
//               TMEM), so probabilities stay <= 256; final O / l to f16 (or the partials).
// Every wait is bounded; a timeout aborts the CTA and records PF_ERR_DEVICE_TIMEOUT.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <type_traits>

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
constexpr int MAX_SPLIT = 64;
// split-KV chunks of at most 2 tokens merge inside the kernel: at most 8 rows per kv head
// (G <= 4), one per softmax warp; more rows per warp lost to the separate merge kernel
constexpr int MERGE_M_MAX = 2;
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

// One run of consecutive key positions held in consecutive rows of one tensor.
struct KeyRange {
  int src;   // 0: the cache, 1: the chunk buffers
  int row0;  // first row (slot / chunk row) of the run within its (layer, kv head)
  int pos0;  // position of row0
  int len;   // keys in the run
};

struct KeyTile {
  int src, row, pos0, nvalid;
};

// The 128-key tiles a CTA's query rows (tokens t0 .. t1-1 of the chunk at `start`) may see.
struct KeyTiles {
  KeyRange r[4];
  int nt[4];
  int total;

  __device__ __forceinline__ void finish() {
    total = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      nt[i] = r[i].len > 0 ? (r[i].len + TK - 1) / TK : 0;
      total += nt[i];
    }
  }
  // linear cache: positions 0 .. start + t1 - 1 at rows = positions
  __device__ __forceinline__ void init_linear(int start, int t1) {
    r[0] = {0, 0, 0, start + t1};
    r[1] = r[2] = r[3] = {0, 0, 0, 0};
    finish();
  }
  // ring cache of R slots, S sinks, window W = R - S
  __device__ __forceinline__ void init_ring(int start, int t0, int t1, int S, int W, int R) {
    r[0] = {0, 0, 0, min(S, start)};  // history sinks: slot = position
    const int wa = max(S, start + t0 - W + 1);  // oldest history key in any row's window
    const int wlen = max(0, start - wa);
    const int slot = wlen > 0 ? S + (wa - S) % W : S;
    const int l1 = min(wlen, R - slot);  // up to the ring's end, then from slot S on
    r[1] = {0, slot, wa, l1};
    r[2] = {0, S, wa + l1, wlen - l1};
    const int c0 = start < S ? 0 : max(0, t0 - W + 1);  // the chunk's own keys
    r[3] = {1, c0, start + c0, t1 - c0};
    finish();
  }
  // tile j of the list (selects with constant indices keep the ranges in registers)
  __device__ __forceinline__ KeyTile at(int j) const {
    KeyRange x = r[0];
    if (j >= nt[0]) {
      j -= nt[0];
      x = r[1];
      if (j >= nt[1]) {
        j -= nt[1];
        x = r[2];
        if (j >= nt[2]) {
          j -= nt[2];
          x = r[3];
        }
      }
    }
    KeyTile t;
    t.src = x.src;
    t.row = x.row0 + j * TK;
    t.pos0 = x.pos0 + j * TK;
    t.nvalid = min(TK, x.len - j * TK);
    return t;
  }
};

struct AttnKParams {
  int M, nq, nkv, layer;
  int cache_rows;  // rows per (layer, kv head) in the cache: max_seq, or R for a ring
  int chunk_rows;  // rows per kv head in the chunk buffers (ring mode)
  int ring_R, ring_S;
  const int* start_dev;
  int start_host;
  float scale_log2;
  int n_split;
  int merge;  // split-KV with few rows (M <= MERGE_M_MAX): the last part to finish merges them
  __half* out;
  float* partial;
  int* counters;  // merge: one arrival counter per kv head (such a chunk is one query tile)
  int* status;
  const int* blocks;  // paged cache: block table (position block -> physical block), else NULL
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

// Bits [0, n) set (n clamped to [0, 64]).
__device__ __forceinline__ uint64_t low_bits(int n) {
  return n <= 0 ? 0ull : (n >= 64 ? ~0ull : (1ull << n) - 1ull);
}

// Visibility of one thread's 64 key columns to its query row: column e is visible when
// e < nvalid (inside the tile's run), e < lim (at or before the row's position), and not in
// [a, b) (a ring's keys older than the row's window that are not sinks).
__device__ __forceinline__ uint64_t visible_cols(int nvalid, int lim, int a, int b) {
  return low_bits(min(nvalid, lim)) & ~(low_bits(b) & ~low_bits(a));
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

// Merges the n_split partial results of (token, head) row `row` (of `rows` per part): with
// m* the largest of the parts' running maxima, O = sum_s 2^(m_s - m*) O_s / sum_s 2^(m_s - m*)
// l_s (the parts keep O_s and l_s relative to their own m_s, in the exp2 domain). Parts that
// saw no key of the row (m_s = -inf) wrote no O and are skipped. One warp per row: lane s
// reads part s's (m, l) (and s + 32), the warp reduces m* and the weighted sum of l, then each
// lane accumulates its HD / 32 columns over the parts with the weights broadcast from their
// lanes, eight parts' loads in flight while the previous eight are added (through L2: other
// CTAs of the same kernel may have written them).
template <int HD>
__device__ __forceinline__ void merge_row(const float* part, int rows, int n_split, int row, int lane,
                                          __half* out) {
  constexpr int PER = HD / 32;
  // each lane's PER columns as one vector load per part (float4 for HD 128, float2 for 64)
  using V = typename std::conditional<PER == 4, float4, float2>::type;
  static_assert(PER == 4 || PER == 2, "head_dim 64 or 128");
  const float* ml = part + static_cast<size_t>(n_split) * rows * HD;
  const V* o0 = reinterpret_cast<const V*>(part + static_cast<size_t>(row) * HD + lane * PER);
  const size_t stride = static_cast<size_t>(rows) * HD / PER;  // between parts, in vectors
  // parts s0 .. s0 + 7 of this lane's columns (zero past n_split)
  auto load8 = [&](int s0, V (&x)[8]) {
#pragma unroll
    for (int u = 0; u < 8; ++u) x[u] = s0 + u < n_split ? __ldcg(o0 + (s0 + u) * stride) : V{};
  };
  // the parts' (m, l) and the first eight parts' rows are requested together: one round trip
  float m0 = -INFINITY, l0 = 0.f, m1 = -INFINITY, l1 = 0.f;  // parts lane and lane + 32
  if (lane < n_split) {
    const size_t sr = static_cast<size_t>(lane) * rows + row;
    m0 = __ldcg(ml + 2 * sr);
    l0 = __ldcg(ml + 2 * sr + 1);
  }
  if (lane + 32 < n_split) {
    const size_t sr = static_cast<size_t>(lane + 32) * rows + row;
    m1 = __ldcg(ml + 2 * sr);
    l1 = __ldcg(ml + 2 * sr + 1);
  }
  V xa[8], xb[8];
  load8(0, xa);
  float mstar = fmaxf(m0, m1);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mstar = fmaxf(mstar, __shfl_xor_sync(0xffffffffu, mstar, o));
  const float w0 = m0 == -INFINITY ? 0.f : exp2f(m0 - mstar);
  const float w1 = m1 == -INFINITY ? 0.f : exp2f(m1 - mstar);
  float lsum = w0 * l0 + w1 * l1;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
  float acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  auto add8 = [&](int s0, const V (&x)[8]) {
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int s = s0 + u;
      const float w = __shfl_sync(0xffffffffu, s < 32 ? w0 : w1, s & 31);
      if (w == 0.f) continue;  // a part that saw no key of the row wrote no O (warp-uniform)
      const float* xv = reinterpret_cast<const float*>(&x[u]);
#pragma unroll
      for (int i = 0; i < PER; ++i) acc[i] = fmaf(w, xv[i], acc[i]);
    }
  };
  // two batches of eight parts in flight: the next batch's loads go out before this one adds
  for (int s0 = 0; s0 < n_split; s0 += 16) {
    if (s0 + 8 < n_split) load8(s0 + 8, xb);
    add8(s0, xa);
    if (s0 + 16 < n_split) load8(s0 + 16, xa);
    if (s0 + 8 < n_split) add8(s0 + 8, xb);
  }
  const float inv = 1.f / lsum;
  __half* dst = out + static_cast<size_t>(row) * HD + lane * PER;
#pragma unroll
  for (int i = 0; i < PER; i += 2) *reinterpret_cast<__half2*>(dst + i) = __floats2half2_rn(acc[i] * inv, acc[i + 1] * inv);
}

template <int HD, int BF16>
__global__ void __launch_bounds__(THREADS, 1)
    attn_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_kc,
                   const __grid_constant__ CUtensorMap tm_vc, const __grid_constant__ CUtensorMap tm_o,
                   const AttnKParams P) {
  PF_TIMELINE(TL_ATTENTION_TC);
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
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // barriers and the TMEM allocation need nothing from earlier kernels: set them up while the
  // previous kernel finishes
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
  griddep_wait();  // the start position and q / cache come from earlier kernels
  const int M = P.M, nq = P.nq;
  const int G = nq / P.nkv;
  const int BT = TQ / G;  // tokens per CTA
  const int n_tt = (M + BT - 1) / BT;
  const int tt = n_tt - 1 - static_cast<int>(blockIdx.x);  // longest rows first
  const int kvh = blockIdx.y;
  const int split = blockIdx.z;
  const int t0 = tt * BT;
  const int t1 = min(t0 + BT, M);
  const int start = P.start_dev ? *P.start_dev : P.start_host;
  const bool ring = P.ring_R > 0;
  const int S = P.ring_S, W = P.ring_R - P.ring_S;
  KeyTiles kt;
  if (ring)
    kt.init_ring(start, t0, t1, S, W, P.ring_R);
  else
    kt.init_linear(start, t1);
  // this CTA's part of the tile list
  const int jb = static_cast<int>(static_cast<long long>(kt.total) * split / P.n_split);
  const int nt = static_cast<int>(static_cast<long long>(kt.total) * (split + 1) / P.n_split) - jb;
  const int crow0 = (P.layer * P.nkv + kvh) * P.cache_rows;  // (layer, kv head) in the cache
  const int brow0 = kvh * P.chunk_rows;                      // kv head in the chunk buffers
  const int first_pos = start + t0, last_pos = start + t1 - 1;
  // whether some key of tile `t` is hidden from some query row of the CTA
  auto needs_mask = [&](const KeyTile& t) {
    if (t.nvalid < TK || t.pos0 + TK - 1 > first_pos) return true;
    return ring && t.pos0 + TK - 1 >= S && t.pos0 <= last_pos - W;
  };


  // Split-KV with few rows: every part's softmax threads (two per query row, the mapping of
  // the softmax warps) count the part in once its partial rows are written; the part that
  // completes the count merges all parts' rows of its (query tile, kv head) into the output
  // and resets the counter (what attn_combine_kernel does otherwise, without its launch).
  __shared__ int merge_last;
  auto merge_tail = [&](bool wrote) {
    int* ctr = P.counters + kvh;
    __threadfence();  // this thread's partial rows are visible GPU-wide before the count
    named_bar_sync_a(1, SM_THREADS);
    if (threadIdx.x == 64) merge_last = (wrote && atomicAdd(ctr, 1) == P.n_split - 1) ? 1 : 0;
    named_bar_sync_a(1, SM_THREADS);
    if (!merge_last) return;
    __threadfence();
    // one softmax warp per row of this CTA that exists (t < M)
    const int rows_cta = (t1 - t0) * G;
    for (int rr = warp - 2; rr < rows_cta; rr += SM_THREADS / 32) {
      const int t = t0 + rr / G, h = kvh * G + rr % G;
      merge_row<HD>(P.partial, M * nq, P.n_split, t * nq + h, lane, P.out);
    }
    if (threadIdx.x == 64) *ctr = 0;  // every part is in: ready for the next launch
  };

  if (nt == 0) {
    // an empty part of a split list: its rows contribute nothing (max -inf, sum 0)
    if (warp >= 2) {
      const int quarter = warp & 3, half = (warp - 2) >> 2;
      const int r = 32 * quarter + lane;
      const int t = t0 + r / G;
      if (half == 0 && t < M) {
        float* ml = P.partial + static_cast<size_t>(P.n_split) * M * nq * HD;
        const size_t row = (static_cast<size_t>(split) * M + t) * nq + kvh * G + r % G;
        ml[2 * row] = -INFINITY;
        ml[2 * row + 1] = 0.f;
      }
      if (P.merge) merge_tail(true);
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, L::Q);
      for (int h = 0; h < NH; ++h)
        tma_load_3d(q_s + h * (TQ * 128), &tm_q, h * 64, kvh * G, t0, q_full);
      // K_i, then V_{i-1}: K runs one tile ahead of V. A paged cache's tiles are whole blocks
      // (tile j of the list = position block j): its row comes from the block table, read a
      // tile ahead so the load's latency hides behind the stage waits.
      const bool paged = P.blocks != nullptr;
      auto cache_row = [&](const KeyTile& t, int blk) {
        return t.src ? brow0 + t.row : crow0 + (paged ? blk * TK : t.row);
      };
      int blk_cur = paged && nt > 0 ? P.blocks[kt.at(jb).pos0 / TK] : 0, blk_prev = 0;
      int k_issued = 0, v_issued = 0;
      bool ok = true;
      for (int i = 0; i <= nt && ok; ++i) {
        const int blk_next = paged && i + 1 < nt ? P.blocks[kt.at(jb + i + 1).pos0 / TK] : 0;
        if (i < nt) {
          const int s = i % KS;
          if (!mbar_wait(k_empty(s), ((i / KS) & 1) ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          const KeyTile kt_i = kt.at(jb + i);
          const CUtensorMap* mk = kt_i.src ? &tm_kc : &tm_k;
          const int row = cache_row(kt_i, blk_cur);
          mbar_arrive_expect_tx(k_full(s), L::KV);
          for (int h = 0; h < NH; ++h) tma_load_2d(k_tile(s) + h * (TK * 128), mk, h * 64, row, k_full(s));
          ++k_issued;
        }
        if (i >= 1) {
          const int jv = i - 1, s = jv % KS;
          if (!mbar_wait(v_empty(s), ((jv / KS) & 1) ^ 1, abort_flag)) {
            ok = false;
            break;
          }
          const KeyTile kt_v = kt.at(jb + jv);
          const CUtensorMap* mv = kt_v.src ? &tm_vc : &tm_v;
          const int row = cache_row(kt_v, blk_prev);
          mbar_arrive_expect_tx(v_full(s), L::KV);
          for (int h = 0; h < NH; ++h) tma_load_2d(v_tile(s) + h * (TK * 128), mv, h * 64, row, v_full(s));
          ++v_issued;
        }
        blk_prev = blk_cur;
        blk_cur = blk_next;
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
    if (ok && nt > 1) ok = issue_s(1);
    for (int j = 0; j < nt && ok; ++j) {
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
      if (j + 2 < nt) ok = issue_s(j + 2);
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
    for (int j = 0; j < nt; ++j) {
      const int s = j % NSB;
      const KeyTile tl = kt.at(jb + j);
      const bool got = mbar_wait(s_full(s), (j / NSB) & 1, abort_flag);
      if (!named_bar_and_a(1, SM_THREADS, got && !failed)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t sbuf = tmem + lane_off + s * TK;
      uint32_t v[HK];
#pragma unroll
      for (int c = 0; c < HK / 32; ++c)
        tmem_ld_32x32b_x32(sbuf + half * HK + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(v + 32 * c));
      tmem_ld_wait();
      // key column e of this thread holds position kp0 + e; keys this row may not see (outside the tile's run, after the row's position, or, in
      // a ring, older than its window and not a sink) become -inf scores in place, so one
      // code path follows: they add nothing to the max and get probability ex2(-inf) = 0
      if (needs_mask(tl)) {
        const int kp0 = tl.pos0 + half * HK;  // position of this thread's first key column
        const uint64_t vis = visible_cols(tl.nvalid - half * HK, pos - kp0 + 1,
                                          ring ? S - kp0 : 0, ring ? pos - W + 1 - kp0 : 0);
        const uint32_t lo = static_cast<uint32_t>(vis), hi = static_cast<uint32_t>(vis >> 32);
#pragma unroll
        for (int e = 0; e < HK; ++e)
          if (!(((e < 32 ? lo : hi) >> (e & 31)) & 1u)) v[e] = 0xff800000u;  // -inf
      }
      float mp[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mp[i] = -INFINITY;
#pragma unroll
      for (int e = 0; e < HK; ++e) mp[e & 7] = fmaxf(mp[e & 7], __uint_as_float(v[e]));
      float mraw = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                         fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
      red[half * TQ + r] = mraw;
      // both partners have read their S columns before either writes P over them
      tc_fence_before();
      named_bar_sync_a(1, SM_THREADS);
      tc_fence_after();
      mraw = fmaxf(mraw, red[(1 - half) * TQ + r]);  // the row's max over all 128 keys
      const float mx = mraw * P.scale_log2;  // scale > 0 keeps the order; -inf stays
      const bool need = j > 0 && mx > m + RESCALE_LOG2;
      if (j == 0) {
        m = mx;  // -inf when no key of the first tile is visible to the row
      } else if (__any_sync(0xffffffffu, need)) {
        // some row of this warp raises its max: the warp rescales its half of those O rows,
        // the rows that keep their max with alpha = 1 (the partner warp decides the same);
        // a row whose max was -inf has O = 0 and l = 0, and alpha = 0 keeps them so
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
      // a row that has seen no key yet (max -inf) has only -inf scores: any finite offset
      // keeps ex2 at 0 (-inf - -inf would be NaN)
      const float neg_m = m == -INFINITY ? 0.f : -m;
      const float sl2 = P.scale_log2;
      float rsp[4] = {0.f, 0.f, 0.f, 0.f};  // independent partial row sums
      uint32_t pk[HK / 2];                  // this thread's 64 probabilities, packed in pairs
#pragma unroll
      for (int x = 0; x < HK; x += 2) {
        const float p0 = ex2_approx(fmaf(__uint_as_float(v[x]), sl2, neg_m));
        const float p1 = ex2_approx(fmaf(__uint_as_float(v[x + 1]), sl2, neg_m));
        rsp[(x >> 1) & 3] += p0 + p1;
        pk[x >> 1] = pack_pair<BF16>(p0, p1);
      }
      l += (rsp[0] + rsp[1]) + (rsp[2] + rsp[3]);
      // P_j over the first TK/2 columns of S buffer s: keys 2c, 2c+1 in column c
      tmem_st_32x32b_x32(sbuf + half * (HK / 2), pk);
      if (r >= tl.nvalid) {
        // key row r of this tile lies outside its run (another head's slots, a stale or
        // unwritten row, or past the tensor): zero its V row once the tile has landed, so a
        // zero probability never meets a NaN / Inf in the PV product
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
      const float l_row = l + red[(1 - half) * TQ + r];
      const int t = t0 + t_loc;
      const int h = kvh * G + h_loc;
      const bool partial = P.n_split > 1;
      const float inv = partial ? 1.f : 1.f / l_row;
      if (partial && half == 0 && t < M) {
        float* ml = P.partial + static_cast<size_t>(P.n_split) * M * nq * HD;
        const size_t row = (static_cast<size_t>(split) * M + t) * nq + h;
        ml[2 * row] = m;
        ml[2 * row + 1] = l_row;
      }
#pragma unroll 1
      for (int c = half * (HD / 64); c < (half + 1) * (HD / 64); ++c) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem_o + lane_off + 32 * c, v);
        tmem_ld_wait();
        if (t < M) {
          if (partial) {
            float4* dst = reinterpret_cast<float4*>(
                P.partial + ((static_cast<size_t>(split) * M + t) * nq + h) * HD + 32 * c);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
              dst[q4] = make_float4(__uint_as_float(v[4 * q4]), __uint_as_float(v[4 * q4 + 1]),
                                    __uint_as_float(v[4 * q4 + 2]), __uint_as_float(v[4 * q4 + 3]));
          }
        }
        if (!partial) {
          // O / l as f16 into the idle K ring, in the layout of the output's TMA box: box
          // b = c / 2 (64 head-dim columns) at k_s + b * 16 KB, row r at r * 128 B, 16-B unit
          // j at (j ^ (r % 8)) * 16 (128-B swizzle); rows past M are clipped by the store
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __half2 hv = __floats2half2_rn(__uint_as_float(v[8 * q4 + 2 * e]) * inv,
                                                   __uint_as_float(v[8 * q4 + 2 * e + 1]) * inv);
              w[e] = *reinterpret_cast<const uint32_t*>(&hv);
            }
            const int j = (c & 1) * 4 + q4;
            st_shared_v4a(k_s + (c >> 1) * (TQ * 128) + r * 128 + ((j ^ (r & 7)) << 4), w[0], w[1], w[2], w[3]);
          }
        }
      }
      if (!partial) {
        fence_proxy_async_smem();
        named_bar_sync_a(1, SM_THREADS);
        if (threadIdx.x == 64) {  // one thread stores the tile: NH boxes of 64 x G x BT
          for (int b = 0; b < NH; ++b) tma_store_3d(&tm_o, k_s + b * (TQ * 128), 64 * b, kvh * G, t0);
          bulk_commit();
          bulk_wait0();  // complete before the CTA retires
        }
      }
    }
    if (P.merge) merge_tail(all_ok);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    __syncwarp();  // lane 0 ran the MMA loop: reconverge before the collective dealloc
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0 && *abort_flag && P.status != nullptr) atomicCAS(P.status, 0, PF_ERR_DEVICE_TIMEOUT);
}

// The merge of split-KV parts as its own kernel (chunks of more than 2 tokens): one warp per
// (token, head) row.
template <int HD>
__global__ void __launch_bounds__(256) attn_combine_kernel(const float* __restrict__ part, int rows,
                                                           int n_split, __half* __restrict__ out) {
  PF_TIMELINE(TL_ATTN_COMBINE);
  griddep_launch_dependents();
  griddep_wait();
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= rows) return;
  merge_row<HD>(part, rows, n_split, row, threadIdx.x & 31, out);
}

template <int HD, int BF16>
cudaError_t launch_tc(const AttnArgs& a, cudaStream_t st) {
  const pf_config& c = *a.c;
  const int G = c.n_q_heads / c.n_kv_heads;
  const int BT = TQ / G;
  const bool ring = c.ring_capacity > 0;
  const int cache_rows = cache_slots(c);
  const uint64_t rows = static_cast<uint64_t>(c.n_layers) * c.n_kv_heads * cache_rows;
  CUtensorMap tq, tk, tv, tkc, tvc;
  const uint64_t qd[3] = {static_cast<uint64_t>(HD), static_cast<uint64_t>(c.n_q_heads),
                          static_cast<uint64_t>(a.M)};
  const uint64_t qs[2] = {static_cast<uint64_t>(HD) * 2, static_cast<uint64_t>(c.n_q_heads) * HD * 2};
  const uint32_t qb[3] = {64, static_cast<uint32_t>(G), static_cast<uint32_t>(BT)};
  const uint64_t kd[2] = {static_cast<uint64_t>(HD), rows};
  const uint64_t ks[1] = {static_cast<uint64_t>(HD) * 2};
  const uint32_t kb[2] = {64, static_cast<uint32_t>(TK)};
  CUtensorMap to;  // the f16 output [M][nq][hd], boxes like Q's
  if (!encode_tmap_16(&to, 0, 3, a.out, qd, qs, qb)) return cudaErrorInvalidValue;
  if (!encode_tmap_16(&tq, BF16, 3, a.q, qd, qs, qb) || !encode_tmap_16(&tk, BF16, 2, a.k_cache, kd, ks, kb) ||
      !encode_tmap_16(&tv, BF16, 2, a.v_cache, kd, ks, kb))
    return cudaErrorInvalidValue;
  if (ring) {
    const uint64_t cd[2] = {static_cast<uint64_t>(HD), static_cast<uint64_t>(c.n_kv_heads) * a.chunk_rows};
    if (!a.k_chunk || !a.v_chunk || !encode_tmap_16(&tkc, BF16, 2, a.k_chunk, cd, ks, kb) ||
        !encode_tmap_16(&tvc, BF16, 2, a.v_chunk, cd, ks, kb))
      return cudaErrorInvalidValue;
  } else {
    tkc = tk;
    tvc = tv;
  }
  const int n_split = std::max(1, std::min(a.n_split, MAX_SPLIT));
  if (n_split > 1 && !a.partial) return cudaErrorInvalidValue;
  AttnKParams p;
  p.M = a.M;
  p.nq = c.n_q_heads;
  p.nkv = c.n_kv_heads;
  p.layer = a.layer;
  p.cache_rows = cache_rows;
  p.chunk_rows = a.chunk_rows;
  p.ring_R = ring ? c.ring_capacity : 0;
  p.ring_S = ring ? c.sink_count : 0;
  p.start_dev = a.start_dev;
  p.start_host = a.start_host;
  p.scale_log2 = 1.4426950408889634f / sqrtf(static_cast<float>(HD));
  p.n_split = n_split;
  p.merge = n_split > 1 && a.M <= MERGE_M_MAX && a.M * G <= SM_THREADS / 32;
  p.out = reinterpret_cast<__half*>(a.out);
  // the buffer: the arrival counters, then the partial O sums and (max, sum) per row
  p.counters = reinterpret_cast<int*>(a.partial);
  p.partial = a.partial ? a.partial + attention_counter_bytes(c) / sizeof(float) : nullptr;
  p.status = a.status;
  p.blocks = a.blocks;
  dim3 grid((a.M + BT - 1) / BT, c.n_kv_heads, n_split);
  cudaError_t e = launch_pdl(attn_tc_kernel<HD, BF16>, grid, dim3(THREADS), ASmem<HD>::BYTES, st, tq, tk,
                             tv, tkc, tvc, to, p);
  if (e != cudaSuccess || n_split == 1 || p.merge) return e;
  const int rows_out = a.M * c.n_q_heads;
  return launch_pdl(attn_combine_kernel<HD>, dim3((rows_out + 7) / 8), dim3(256), 0, st,
                    static_cast<const float*>(p.partial), rows_out, n_split,
                    reinterpret_cast<__half*>(a.out));
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

int attention_splits(const pf_config& c, int M, int sms) {
  if (!attention_tc_supported(c) || M <= 0) return 1;
  const int BT = TQ / (c.n_q_heads / c.n_kv_heads);
  const int ctas = (M + BT - 1) / BT * c.n_kv_heads;
  if (2 * ctas > sms) return 1;  // at least half of the SMs busy without splitting
  return std::max(1, std::min(MAX_SPLIT, sms / ctas));
}

size_t attention_counter_bytes(const pf_config& c) {
  return (static_cast<size_t>(c.n_kv_heads) * sizeof(int) + 15) / 16 * 16;
}

size_t attention_partial_bytes(const pf_config& c, int M, int n_split) {
  if (n_split <= 1) return 0;
  // the arrival counters, then the partial O sums and (max, sum) per row
  return attention_counter_bytes(c) + static_cast<size_t>(n_split) * M * c.n_q_heads * (c.head_dim + 2) * sizeof(float);
}

size_t attention_partial_bytes_max(const pf_config& c, int max_sms) {
  if (!attention_tc_supported(c)) return 0;
  const int BT = TQ / (c.n_q_heads / c.n_kv_heads);
  size_t best = 0;
  for (int nqt = 1; nqt <= (c.max_chunk + BT - 1) / BT; ++nqt) {
    const int M = std::min(nqt * BT, c.max_chunk);
    int worst = 1;
    for (int sms = 1; sms <= max_sms; ++sms) worst = std::max(worst, attention_splits(c, M, sms));
    best = std::max(best, attention_partial_bytes(c, M, worst));
    if (2 * nqt * c.n_kv_heads > max_sms) break;  // no split at this size or beyond
  }
  return best;
}

cudaError_t prepare_attention_tc_kernels() {
  cudaError_t e = cudaSuccess, r;
  if ((r = set_attr_tc<128, 1>()) != cudaSuccess) e = r;
  if ((r = set_attr_tc<128, 0>()) != cudaSuccess) e = r;
  if ((r = set_attr_tc<64, 1>()) != cudaSuccess) e = r;
  if ((r = set_attr_tc<64, 0>()) != cudaSuccess) e = r;
  return e;
}

cudaError_t launch_attention_tc(const AttnArgs& a, cudaStream_t stream) {
  const pf_config& c = *a.c;
  const bool bf = c.kv_dtype == PF_KV_BF16;
  if (c.head_dim == 128) return bf ? launch_tc<128, 1>(a, stream) : launch_tc<128, 0>(a, stream);
  return bf ? launch_tc<64, 1>(a, stream) : launch_tc<64, 0>(a, stream);
}

}  // namespace pf

PF_TIMELINE_SETTER(attention_tc)
