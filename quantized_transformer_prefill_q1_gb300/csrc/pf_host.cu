// pf_host.cu — libpf's C ABI: argument validation, the host-side weight packer, the
// RoPE table, workspace layout, sessions, and the layer / chunk driver that enqueues the
// kernels on one stream (optionally recorded once per shape as a CUDA graph and
// replayed).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <tuple>
#include <vector>

#include "pf_internal.h"
#include "streamk.cuh"

namespace pf {
namespace {

thread_local std::string g_err = "";

pf_status fail(pf_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return st;
}

pf_status cuda_fail(cudaError_t e, const char* what) {
  return fail(PF_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

#define PF_CUDA(call, what)                        \
  do {                                             \
    cudaError_t e_ = (call);                       \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

size_t kv_elem_bytes(int kv_dtype) { return kv_dtype == PF_KV_F32 ? 4 : 2; }

// ------------------------------------------------------------------ workspace layout
struct WsLayout {
  size_t status, params, tokens, x, y, qkv, q, attn, act, logits, gemm, gemm_bytes, rope;
  size_t kchunk, vchunk;          // ring mode: the chunk's K / V rows [nkv][max_chunk][hd]
  size_t attn_part, attn_part_bytes;  // split-KV partial results
  size_t blocks;                      // paged cache: block table [block_table_entries] int32
  size_t total;
};

WsLayout ws_layout(const pf_config& c) {
  WsLayout L{};
  const size_t C = static_cast<size_t>(c.max_chunk);
  const size_t H = c.hidden, I = c.intermediate, hd = c.head_dim;
  const size_t qkv_rows = static_cast<size_t>(c.n_q_heads + 2 * c.n_kv_heads) * hd;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes, 256);
    return at;
  };
  L.status = take(STATUS_WORDS * sizeof(int));
  L.params = take(4 * sizeof(int));
  L.tokens = take(C * sizeof(int));
  L.x = take(C * H * 4);
  L.y = take(C * H * 2);
  L.qkv = take(C * qkv_rows * 4);
  L.q = take(C * c.n_q_heads * hd * 2);
  L.attn = take(C * c.n_q_heads * hd * 2);
  L.act = take(C * I * 2);
  L.logits = take(static_cast<size_t>(c.vocab > 0 ? c.vocab : 1) * 4);
  // GEMM scratch sized for the widest projection of a full chunk
  const int widest = static_cast<int>(std::max<size_t>({qkv_rows, H, 2 * I}));
  L.gemm_bytes = gemm_scratch_bytes(c.max_chunk, widest, GEMM_MAX_CTAS);
  L.gemm = take(L.gemm_bytes);
  L.rope = take(static_cast<size_t>(c.max_seq) * (hd / 2) * 2 * 4);
  const size_t chunk_kv = c.ring_capacity > 0 ? C * c.n_kv_heads * hd * kv_elem_bytes(c.kv_dtype) : 0;
  L.kchunk = take(chunk_kv);
  L.vchunk = take(chunk_kv);
  L.attn_part_bytes = attention_partial_bytes_max(c, GEMM_MAX_CTAS);
  L.attn_part = take(L.attn_part_bytes);
  L.blocks = take(c.kv_block_pool > 0 ? block_table_entries(c) * sizeof(int) : 0);
  L.total = o;
  return L;
}

// ------------------------------------------------------------------ tensor maps
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace

bool encode_tmap_f16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                        uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tmap_16(CUtensorMap* map, int bf16, int rank, const void* base, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn || rank < 2 || rank > 5) return false;
  cuuint64_t d[5], s[4];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
    if (i + 1 < rank) s[i] = strides_bytes[i];
  }
  return fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
            static_cast<cuuint32_t>(rank), const_cast<void*>(base), d, s, b, e,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_tmap_out_2d(CUtensorMap* map, bool f32, const void* base, uint64_t inner, uint64_t outer,
                        uint32_t box_inner, uint32_t box_outer, int swizzle_bytes) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  const uint64_t esz = f32 ? 4 : 2;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * esz};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle sw = swizzle_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                      : CU_TENSOR_MAP_SWIZZLE_NONE;
  return fn(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
            const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int device_sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
  return n;
}

}  // namespace pf

using namespace pf;

// ====================================================================== sessions
struct GraphKey {
  int M;
  const void* x;
  const void* tokens;
  const void* logits;
  int layer;  // -1: whole stack
  bool operator<(const GraphKey& o) const {
    return std::tie(M, x, tokens, logits, layer) < std::tie(o.M, o.x, o.tokens, o.logits, o.layer);
  }
};

struct GraphExec {
  cudaGraphExec_t exec;
  int64_t kernels;  // libpf kernels recorded in it
};

struct ProfRecord {
  int cls;
  cudaEvent_t e0, e1;
};

struct pf_session {
  pf_model model;
  std::vector<pf_layer_weights> layers;
  void* k = nullptr;
  void* v = nullptr;
  uint8_t* ws = nullptr;
  size_t ws_bytes = 0;
  WsLayout L{};
  int position = 0;
  bool graphs = true;
  bool profile = false;
  int sms = 148;
  int64_t launches = 0;
  std::map<GraphKey, GraphExec> execs;
  std::vector<ProfRecord> prof;
  std::vector<cudaEvent_t> event_pool;
  cudaStream_t capture_stream = nullptr;
  std::vector<int32_t> blocks;  // paged cache: host copy of the block table (-1 = unassigned)
};

namespace {

template <typename T>
T* wsp(pf_session* s, size_t off) {
  return reinterpret_cast<T*>(s->ws + off);
}

pf_status check_cfg(const pf_config* c) {
  if (!c) return fail(PF_ERR_INVALID_ARG, "config is NULL");
  if (c->hidden <= 0 || c->hidden % 128) return fail(PF_ERR_SHAPE, "hidden %d: need a positive multiple of 128", c->hidden);
  if (c->intermediate <= 0 || c->intermediate % 128)
    return fail(PF_ERR_SHAPE, "intermediate %d: need a positive multiple of 128", c->intermediate);
  if (c->head_dim != 64 && c->head_dim != 128) return fail(PF_ERR_SHAPE, "head_dim %d: 64 or 128", c->head_dim);
  if (c->n_q_heads <= 0 || c->n_kv_heads <= 0 || c->n_q_heads % c->n_kv_heads)
    return fail(PF_ERR_SHAPE, "heads %d/%d: nkv must divide nq", c->n_q_heads, c->n_kv_heads);
  const int G = c->n_q_heads / c->n_kv_heads;
  if (64 % G) return fail(PF_ERR_SHAPE, "GQA group %d must divide 64", G);
  if ((c->n_q_heads * c->head_dim) % 128)
    return fail(PF_ERR_SHAPE, "nq*hd %d: need a multiple of 128", c->n_q_heads * c->head_dim);
  if (c->n_layers <= 0) return fail(PF_ERR_SHAPE, "n_layers %d", c->n_layers);
  if (c->vocab < 0) return fail(PF_ERR_SHAPE, "vocab %d", c->vocab);
  if (c->wfmt != PF_W_Q1_G128 && c->wfmt != PF_W_INT4_AFFINE_G128)
    return fail(PF_ERR_INVALID_ARG, "weight format %d", c->wfmt);
  if (c->kv_dtype != PF_KV_F32 && c->kv_dtype != PF_KV_BF16 && c->kv_dtype != PF_KV_F16)
    return fail(PF_ERR_INVALID_ARG, "kv dtype %d", c->kv_dtype);
  if (c->max_seq <= 0) return fail(PF_ERR_SHAPE, "max_seq %d", c->max_seq);
  if (c->max_chunk <= 0 || c->max_chunk > 8192) return fail(PF_ERR_SHAPE, "max_chunk %d: 1..8192", c->max_chunk);
  if (!(c->eps >= 0.f) || !(c->final_eps >= 0.f) || !(c->rope_theta > 0.f))
    return fail(PF_ERR_INVALID_ARG, "eps / rope_theta");
  if (c->ring_capacity < 0) return fail(PF_ERR_SHAPE, "ring_capacity %d", c->ring_capacity);
  if (c->ring_capacity > 0) {
    if (c->sink_count < 0 || c->sink_count >= c->ring_capacity)
      return fail(PF_ERR_SHAPE, "ring cache: need 0 <= sink_count (%d) < ring_capacity (%d)", c->sink_count,
                  c->ring_capacity);
    if (!attention_tc_supported(*c))
      return fail(PF_ERR_UNSUPPORTED, "ring cache: needs a 16-bit cache (bf16 / f16) and a GQA group dividing 128");
  } else if (c->sink_count != 0) {
    return fail(PF_ERR_SHAPE, "sink_count %d without a ring cache", c->sink_count);
  }
  if (c->kv_block_pool < 0) return fail(PF_ERR_SHAPE, "kv_block_pool %d", c->kv_block_pool);
  if (c->kv_block_pool > 0) {
    if (c->ring_capacity > 0) return fail(PF_ERR_SHAPE, "a paged cache cannot also be a ring");
    if (!attention_tc_supported(*c))
      return fail(PF_ERR_UNSUPPORTED, "paged cache: needs a 16-bit cache (bf16 / f16) and a GQA group dividing 128");
    if (static_cast<int64_t>(c->kv_block_pool) * PF_KV_BLOCK > (int64_t{1} << 30))
      return fail(PF_ERR_SHAPE, "kv_block_pool %d too large", c->kv_block_pool);
  }
  return PF_OK;
}

// Paged caches: every position block of [0, end) has a physical block.
pf_status check_blocks(const pf_session* s, int64_t end) {
  if (s->model.cfg.kv_block_pool <= 0) return PF_OK;
  for (int64_t b = 0; b * PF_KV_BLOCK < end; ++b)
    if (b >= static_cast<int64_t>(s->blocks.size()) || s->blocks[b] < 0)
      return fail(PF_ERR_KV_CAPACITY, "paged cache: position block %lld (positions %lld..) has no physical block",
                  static_cast<long long>(b), static_cast<long long>(b * PF_KV_BLOCK));
  return PF_OK;
}

cudaEvent_t take_event(pf_session* s) {
  if (!s->event_pool.empty()) {
    cudaEvent_t e = s->event_pool.back();
    s->event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Enqueues one libpf kernel through `call`, counting it and, in profile mode, bracketing
// it with CUDA events on its stream.
template <typename Call>
pf_status launch_k(pf_session* s, int cls, cudaStream_t st, const char* what, Call call) {
  cudaEvent_t e0 = nullptr;
  if (s->profile) {
    e0 = take_event(s);
    PF_CUDA(cudaEventRecord(e0, st), "event record");
  }
  PF_CUDA(call(), what);
  if (s->profile) {
    cudaEvent_t e1 = take_event(s);
    PF_CUDA(cudaEventRecord(e1, st), "event record");
    s->prof.push_back({cls, e0, e1});
  }
  ++s->launches;
  return PF_OK;
}

#define PF_TRY(expr)                \
  do {                              \
    pf_status r_ = (expr);          \
    if (r_ != PF_OK) return r_;     \
  } while (0)

pf_status enqueue_gemm(pf_session* s, int cls, int wfmt, int epi, const void* a, const void* w,
                       int M, int N, int K, void* out, cudaStream_t st, bool out_zeroed = false,
                       void* side_zero = nullptr, size_t side_zero_bytes = 0) {
  GemmArgs g{};
  g.out_zeroed = out_zeroed;
  g.side_zero = side_zero;
  g.side_zero_bytes = side_zero_bytes;
  g.wfmt = wfmt;
  g.epilogue = epi;
  g.a = a;
  g.w = reinterpret_cast<const uint8_t*>(w);
  g.M = M;
  g.N = N;
  g.K = K;
  g.out = out;
  g.max_ctas = GEMM_MAX_CTAS;
  g.scratch = wsp<void>(s, s->L.gemm);
  g.status = wsp<int>(s, s->L.status);
  // Stream-K skew of the layer GEMMs at full chunks: the CTAs launched last start on SMs that
  // the previous kernel still holds, 1-2 us after the others (per-CTA timeline, 512-token
  // chunks on GB300: the last ~26 of 76 pairs after an RMSNorm, a ramp over the last ~36 after
  // attention, the last ~20 after gate_up), so those units take a few k-blocks fewer.
  if (M >= 384) {
    switch (cls) {
      case PF_K_GEMM_QKV: g.late_units = 26; g.late_kb = 5; break;
      case PF_K_GEMM_GATE_UP: g.late_units = 26; g.late_kb = 3; break;
      case PF_K_GEMM_O: g.late_units = 36; g.late_kb = 3; break;
      case PF_K_GEMM_DOWN: g.late_units = 20; g.late_kb = 4; break;
      default: break;
    }
  }
  return launch_k(s, cls, st, "gemm launch", [&] { return launch_gemm(g, st); });
}

// metal_prefill.rs encode_layer_prefill, sections 1-7, on x [M, H] (in place). Where the
// QKV GEMM accumulates into a zeroed qkv buffer (gemm_side_zero_supported), `qkv_zeroed` says
// an earlier kernel has zeroed it already, and `zero_next_qkv` has this layer's gate_up GEMM
// zero it for the next layer (its epilogue warps are idle during the main loop).
pf_status enqueue_layer(pf_session* s, int l, float* x, int M, cudaStream_t st, bool qkv_zeroed,
                        bool zero_next_qkv) {
  const pf_config& c = s->model.cfg;
  const pf_layer_weights& w = s->layers[l];
  const int H = c.hidden, I = c.intermediate, hd = c.head_dim;
  const int qkv_rows = (c.n_q_heads + 2 * c.n_kv_heads) * hd;
  const int* start_dev = wsp<int>(s, s->L.params);
  void* y = wsp<void>(s, s->L.y);
  float* qkv = wsp<float>(s, s->L.qkv);
  void* q = wsp<void>(s, s->L.q);
  void* attn = wsp<void>(s, s->L.attn);
  void* act = wsp<void>(s, s->L.act);
  // 1. pre-attention RMSNorm; where the QKV GEMM accumulates into a zeroed output, the norm's
  //    CTAs zero it (one qkv row each), so no memset breaks the launch chain
  //    Every GEMM path accumulates the QKV projection into a zeroed qkv: the previous layer's
  //    gate_up GEMM zeroes it where it can (M > 64), this norm's CTAs otherwise
  const bool side = gemm_side_zero_supported(c.wfmt, M);
  const bool zero_qkv = !(qkv_zeroed && side);
  PF_TRY(launch_k(s, PF_K_RMSNORM, st, "rmsnorm", [&] {
    return launch_rmsnorm(x, w.attn_norm, c.eps, M, H, y, st, zero_qkv ? qkv : nullptr, qkv_rows);
  }));
  // 2. fused QKV projection
  PF_TRY(enqueue_gemm(s, PF_K_GEMM_QKV, c.wfmt, EPI_STORE_F32, y, w.qkv, M, qkv_rows, H, qkv, st, true));
  // 3. QK-norm + RoPE + KV store, then causal GQA attention over cache + chunk. A ring cache
  //    takes the chunk's K / V in the chunk buffers first (its later tokens may overwrite
  //    slots its earlier tokens still see) and into the ring after the attention.
  const bool ring = c.ring_capacity > 0;
  const int* blocks = c.kv_block_pool > 0 ? wsp<int>(s, s->L.blocks) : nullptr;
  void* kc = ring ? wsp<void>(s, s->L.kchunk) : s->k;
  void* vc = ring ? wsp<void>(s, s->L.vchunk) : s->v;
  PF_TRY(launch_k(s, PF_K_QK_ROPE_KV, st, "qk_norm_rope_kv", [&] {
    return launch_qk_norm_rope_kv(c, qkv, w.q_norm, w.k_norm, wsp<float>(s, s->L.rope), ring ? 0 : l,
                                  ring ? c.max_chunk : cache_slots(c), ring ? 0 : 1, start_dev, 0, M, q, kc,
                                  vc, st, blocks);
  }));
  AttnArgs aa{};
  aa.c = &c;
  aa.q = q;
  aa.k_cache = s->k;
  aa.v_cache = s->v;
  aa.k_chunk = ring ? kc : nullptr;
  aa.v_chunk = ring ? vc : nullptr;
  aa.chunk_rows = c.max_chunk;
  aa.layer = l;
  aa.start_dev = start_dev;
  aa.M = M;
  aa.out = attn;
  aa.n_split = attention_splits(c, M, std::min(s->sms, GEMM_MAX_CTAS));
  aa.partial = wsp<float>(s, s->L.attn_part);
  aa.status = wsp<int>(s, s->L.status);
  aa.blocks = blocks;
  PF_TRY(launch_k(s, PF_K_ATTENTION, st, "attention", [&] { return launch_attention(aa, st); }));
  if (ring)
    PF_TRY(launch_k(s, PF_K_QK_ROPE_KV, st, "ring store", [&] {
      return launch_ring_store(c, kc, vc, c.max_chunk, l, start_dev, 0, M, s->k, s->v, st);
    }));
  // 4. O projection + residual
  PF_TRY(enqueue_gemm(s, PF_K_GEMM_O, c.wfmt, EPI_RESID_ADD, attn, w.o_proj, M, H,
                      c.n_q_heads * hd, x, st));
  // 5. FFN RMSNorm
  PF_TRY(launch_k(s, PF_K_RMSNORM, st, "rmsnorm",
                  [&] { return launch_rmsnorm(x, w.ffn_norm, c.eps, M, H, y, st); }));
  // 6. gate_up + SwiGLU
  const bool zero_next = side && zero_next_qkv;
  PF_TRY(enqueue_gemm(s, PF_K_GEMM_GATE_UP, c.wfmt, EPI_SWIGLU, y, w.gate_up, M, 2 * I, H, act, st,
                      false, zero_next ? qkv : nullptr,
                      zero_next ? static_cast<size_t>(M) * qkv_rows * sizeof(float) : 0));
  // 7. down projection + residual
  PF_TRY(enqueue_gemm(s, PF_K_GEMM_DOWN, c.wfmt, EPI_RESID_ADD, act, w.down, M, H, I, x, st));
  return PF_OK;
}

// One micro-batch: [embed] -> every layer -> [final norm + LM head on the last row].
pf_status enqueue_chunk(pf_session* s, float* x, int M, const int* tokens_dev, float* logits,
                        cudaStream_t st) {
  const pf_config& c = s->model.cfg;
  if (tokens_dev)
    PF_TRY(launch_k(s, PF_K_EMBED, st, "embed", [&] {
      return launch_embed(s->model.embed, tokens_dev, M, c.hidden, c.vocab, x,
                          wsp<int>(s, s->L.status), st);
    }));
  for (int l = 0; l < c.n_layers; ++l) PF_TRY(enqueue_layer(s, l, x, M, st, l > 0, l + 1 < c.n_layers));
  if (logits)
    PF_TRY(launch_k(s, PF_K_LM_HEAD, st, "lm_head", [&] {
      return launch_lm_head(c.wfmt, x + static_cast<size_t>(M - 1) * c.hidden, s->model.final_norm,
                            c.final_eps, reinterpret_cast<const uint8_t*>(s->model.lm_head), c.vocab,
                            c.hidden, logits, st);
    }));
  return PF_OK;
}

// Runs body(stream) directly on `st`, or as a CUDA graph recorded on first use for `key`
// and replayed on `st` (never while profiling: the per-launch events need the launches
// themselves). Recording uses the session's own non-blocking stream, since the caller's
// stream may be the legacy default stream, on which capture is not permitted; recording
// executes nothing.
template <typename Body>
pf_status run_maybe_graph(pf_session* s, const GraphKey& key, cudaStream_t st, Body body) {
  if (!s->graphs || s->profile) return body(st);
  auto it = s->execs.find(key);
  if (it == s->execs.end()) {
    if (!s->capture_stream)
      PF_CUDA(cudaStreamCreateWithFlags(&s->capture_stream, cudaStreamNonBlocking), "capture stream");
    cudaStream_t cs = s->capture_stream;
    const int64_t before = s->launches;
    PF_CUDA(cudaStreamBeginCapture(cs, cudaStreamCaptureModeThreadLocal), "begin capture");
    pf_status r = body(cs);
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaStreamEndCapture(cs, &graph);
    const int64_t recorded = s->launches - before;
    s->launches = before;  // counted when the graph runs
    if (r != PF_OK) {
      if (graph) cudaGraphDestroy(graph);
      return r;
    }
    if (e != cudaSuccess) return cuda_fail(e, "end capture");
    cudaGraphExec_t exec = nullptr;
    e = cudaGraphInstantiate(&exec, graph, 0);
    cudaGraphDestroy(graph);
    if (e != cudaSuccess) return cuda_fail(e, "graph instantiate");
    if (s->execs.size() >= 64) {
      cudaGraphExecDestroy(s->execs.begin()->second.exec);
      s->execs.erase(s->execs.begin());
    }
    it = s->execs.emplace(key, GraphExec{exec, recorded}).first;
  }
  PF_CUDA(cudaGraphLaunch(it->second.exec, st), "graph launch");
  s->launches += it->second.kernels;
  return PF_OK;
}

pf_status set_start(pf_session* s, int start, cudaStream_t st) {
  return launch_k(s, PF_K_OTHER, st, "set start",
                  [&] { return launch_set_int(wsp<int>(s, s->L.params), start, st); });
}

// Raises the dynamic shared-memory limit of the big kernels once, outside any capture.
void prepare_all() {
  static std::once_flag once;
  std::call_once(once, [] {
    prepare_gemm_kernels();
    prepare_gemm_small_kernels();
    prepare_attention_kernels();
    prepare_attention_tc_kernels();
  });
}

}  // namespace

// ====================================================================== C ABI
extern "C" {

const char* pf_last_error(void) { return g_err.c_str(); }

const char* pf_status_name(int st) {
  switch (st) {
    case PF_OK: return "PF_OK";
    case PF_ERR_INVALID_ARG: return "PF_ERR_INVALID_ARG";
    case PF_ERR_SHAPE: return "PF_ERR_SHAPE";
    case PF_ERR_EMPTY_CHUNK: return "PF_ERR_EMPTY_CHUNK";
    case PF_ERR_NONSEQUENTIAL_START: return "PF_ERR_NONSEQUENTIAL_START";
    case PF_ERR_TOKEN_OUT_OF_VOCAB: return "PF_ERR_TOKEN_OUT_OF_VOCAB";
    case PF_ERR_KV_CAPACITY: return "PF_ERR_KV_CAPACITY";
    case PF_ERR_LOGITS: return "PF_ERR_LOGITS";
    case PF_ERR_UNSUPPORTED: return "PF_ERR_UNSUPPORTED";
    case PF_ERR_CUDA: return "PF_ERR_CUDA";
    case PF_ERR_DEVICE_TIMEOUT: return "PF_ERR_DEVICE_TIMEOUT";
    case PF_ERR_WORKSPACE: return "PF_ERR_WORKSPACE";
    default: return "PF_ERR_UNKNOWN";
  }
}

int32_t pf_abi_version(void) { return 4; }

size_t pf_packed_bytes(int32_t wfmt, int64_t N, int64_t K) {
  if ((wfmt != PF_W_Q1_G128 && wfmt != PF_W_INT4_AFFINE_G128) || N <= 0 || K <= 0 || K % GROUP)
    return 0;
  return static_cast<size_t>(padded_rows(N) / TILE_N) * static_cast<size_t>(K / GROUP) *
         chunk_bytes(wfmt);
}

pf_status pf_pack_weights_host(int32_t wfmt, const uint8_t* codes, const uint16_t* scales,
                               const uint16_t* zeros, int64_t N, int64_t K,
                               int32_t interleave_gate_up, void* dst, size_t dst_bytes) {
  const size_t need = pf_packed_bytes(wfmt, N, K);
  if (need == 0) return fail(PF_ERR_SHAPE, "pack: format %d, N %lld, K %lld (K %% 128 == 0)", wfmt, (long long)N, (long long)K);
  if (!codes || !scales || !dst) return fail(PF_ERR_INVALID_ARG, "pack: NULL pointer");
  if (wfmt == PF_W_INT4_AFFINE_G128 && !zeros) return fail(PF_ERR_INVALID_ARG, "pack: INT4 needs zeros");
  if (dst_bytes < need) return fail(PF_ERR_INVALID_ARG, "pack: dst holds %zu bytes, need %zu", dst_bytes, need);
  if (interleave_gate_up && (N % 256)) return fail(PF_ERR_SHAPE, "pack: interleaved gate_up needs N = 2I, I %% 128 == 0");
  uint8_t* out = static_cast<uint8_t*>(dst);
  std::memset(out, 0, need);
  const int64_t G = K / GROUP, Np = padded_rows(N), I = N / 2;
  const size_t cb = chunk_bytes(wfmt);
  // even / odd bit compaction of one byte: low nibble = bits 0,2,4,6; high = bits 1,3,5,7
  static uint8_t eo[256];
  static std::once_flag once;
  std::call_once(once, [] {
    for (int b = 0; b < 256; ++b) {
      int e = 0, o = 0;
      for (int i = 0; i < 4; ++i) {
        e |= ((b >> (2 * i)) & 1) << i;
        o |= ((b >> (2 * i + 1)) & 1) << i;
      }
      eo[b] = static_cast<uint8_t>(e | (o << 4));
    }
  });
  auto rev16 = [](uint32_t v) {
    v = ((v & 0x5555u) << 1) | ((v >> 1) & 0x5555u);
    v = ((v & 0x3333u) << 2) | ((v >> 2) & 0x3333u);
    v = ((v & 0x0F0Fu) << 4) | ((v >> 4) & 0x0F0Fu);
    v = ((v & 0x00FFu) << 8) | ((v >> 8) & 0x00FFu);
    return v & 0xFFFFu;
  };
  for (int64_t p = 0; p < Np; ++p) {
    int64_t src;
    if (interleave_gate_up) {
      // every 128 packed rows: 64 gate rows, then the 64 matching up rows
      const int64_t t = p / 128, r = p % 128;
      src = r < 64 ? t * 64 + r : I + t * 64 + (r - 64);
    } else {
      src = p < N ? p : -1;
    }
    if (src < 0) continue;  // padding row: zero scale (and zero codes)
    const int64_t t = p / TILE_N, r = p % TILE_N;
    for (int64_t g = 0; g < G; ++g) {
      uint8_t* ch = out + (t * G + g) * cb;
      const uint16_t sc = scales[src * G + g];
      if (wfmt == PF_W_Q1_G128) {
        const uint8_t* row = codes + src * (K / 8) + g * 16;
        for (int h = 0; h < 2; ++h)
          for (int b = 0; b < 2; ++b) {
            const uint8_t* w4 = row + h * 8 + b * 4;  // 32 weights, LSB-first
            uint32_t E = 0, O = 0;
            for (int j = 0; j < 4; ++j) {
              E |= static_cast<uint32_t>(eo[w4[j]] & 15) << (4 * j);
              O |= static_cast<uint32_t>(eo[w4[j]] >> 4) << (4 * j);
            }
            // bit i of E/O = sign bit of element 2i / 2i+1; store NEGATIVE flags at 15-i / 31-i
            const uint32_t Z = rev16(~E & 0xFFFFu) | (rev16(~O & 0xFFFFu) << 16);
            std::memcpy(ch + h * Q1_HALF_BYTES + r * 8 + b * 4, &Z, 4);
          }
        std::memcpy(ch + Q1_SCALE_OFF + r * 2, &sc, 2);
      } else {
        const uint8_t* row = codes + src * (K / 2) + g * 64;
        for (int h = 0; h < 2; ++h)
          for (int w = 0; w < 8; ++w) {
            const uint8_t* b = row + h * 32 + w * 4;  // 8 weights: byte j = (k 2j, k 2j+1)
            uint32_t lo = 0, hi = 0;
            for (int j = 0; j < 4; ++j) {
              lo |= static_cast<uint32_t>(b[j] & 15) << (4 * j);
              hi |= static_cast<uint32_t>(b[j] >> 4) << (4 * j);
            }
            const uint32_t word = lo | (hi << 16);
            std::memcpy(ch + h * I4_HALF_BYTES + r * 32 + w * 4, &word, 4);
          }
        const uint16_t z = zeros[src * G + g];
        std::memcpy(ch + I4_SCALE_OFF + r * 2, &sc, 2);
        std::memcpy(ch + I4_ZERO_OFF + r * 2, &z, 2);
      }
    }
  }
  return PF_OK;
}

size_t pf_kv_bytes(const pf_config* c) {
  if (check_cfg(c) != PF_OK) return 0;
  const int slots = cache_slots(*c);
  return static_cast<size_t>(c->n_layers) * c->n_kv_heads * slots * c->head_dim *
         kv_elem_bytes(c->kv_dtype);
}

size_t pf_workspace_bytes(const pf_config* c) {
  if (check_cfg(c) != PF_OK) return 0;
  return ws_layout(*c).total;
}

pf_status pf_config_check(const pf_config* c) { return check_cfg(c); }

pf_status pf_validate_chunk(const pf_config* c, int32_t kv_position, const int32_t* tokens,
                            int32_t M, int32_t start, int32_t want_logits, int32_t has_head) {
  pf_status r = check_cfg(c);
  if (r != PF_OK) return r;
  if (M <= 0) return fail(PF_ERR_EMPTY_CHUNK, "prefill called with an empty chunk (M = %d)", M);
  if (start != kv_position)
    return fail(PF_ERR_NONSEQUENTIAL_START, "non-sequential chunk start %d; KV cache is at %d", start, kv_position);
  if (tokens) {
    for (int i = 0; i < M; ++i)
      if (tokens[i] < 0 || tokens[i] >= c->vocab)
        return fail(PF_ERR_TOKEN_OUT_OF_VOCAB, "token id %d outside vocab %d", tokens[i], c->vocab);
  }
  if (static_cast<int64_t>(start) + M > c->max_seq)
    return fail(PF_ERR_KV_CAPACITY, "chunk [%d, %d) exceeds KV capacity %d", start, start + M, c->max_seq);
  if (want_logits && !has_head)
    return fail(PF_ERR_LOGITS, "logits requested but the model has no final norm / LM head");
  return PF_OK;
}

pf_status pf_rope_table_host(float theta, int32_t hd, int32_t max_seq, float* dst) {
  if (!dst || hd <= 0 || hd % 2 || max_seq <= 0 || !(theta > 0.f))
    return fail(PF_ERR_INVALID_ARG, "rope table arguments");
  const int half = hd / 2;
  for (int i = 0; i < half; ++i) {
    const double inv = std::pow(static_cast<double>(theta), -2.0 * i / hd);
    for (int p = 0; p < max_seq; ++p) {
      const double a = p * inv;
      dst[(static_cast<size_t>(p) * half + i) * 2 + 0] = static_cast<float>(std::cos(a));
      dst[(static_cast<size_t>(p) * half + i) * 2 + 1] = static_cast<float>(std::sin(a));
    }
  }
  return PF_OK;
}

pf_status pf_session_create(const pf_model* model, void* k, void* v, void* ws, size_t ws_bytes,
                            void* stream, pf_session** out) {
  if (!out) return fail(PF_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!model) return fail(PF_ERR_INVALID_ARG, "model is NULL");
  pf_status r = check_cfg(&model->cfg);
  if (r != PF_OK) return r;
  const pf_config& c = model->cfg;
  if (!model->layers || !k || !v || !ws) return fail(PF_ERR_INVALID_ARG, "layers / k / v / workspace is NULL");
  for (int l = 0; l < c.n_layers; ++l) {
    const pf_layer_weights& w = model->layers[l];
    if (!w.attn_norm || !w.qkv || !w.o_proj || !w.ffn_norm || !w.gate_up || !w.down)
      return fail(PF_ERR_INVALID_ARG, "layer %d: a weight pointer is NULL", l);
    if (c.qk_norm && (!w.q_norm || !w.k_norm))
      return fail(PF_ERR_INVALID_ARG, "layer %d: qk_norm set but q_norm / k_norm NULL", l);
  }
  const WsLayout L = ws_layout(c);
  if (ws_bytes < L.total) return fail(PF_ERR_WORKSPACE, "workspace %zu bytes, need %zu", ws_bytes, L.total);
  if ((reinterpret_cast<uintptr_t>(ws) & 255) || (reinterpret_cast<uintptr_t>(k) & 15) ||
      (reinterpret_cast<uintptr_t>(v) & 15))
    return fail(PF_ERR_INVALID_ARG, "workspace must be 256-B aligned, caches 16-B aligned");
  auto* s = new pf_session();
  s->model = *model;
  s->layers.assign(model->layers, model->layers + c.n_layers);
  s->model.layers = s->layers.data();
  s->k = k;
  s->v = v;
  s->ws = static_cast<uint8_t*>(ws);
  s->ws_bytes = ws_bytes;
  s->L = L;
  s->sms = device_sm_count();
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  std::vector<float> rope(static_cast<size_t>(c.max_seq) * (c.head_dim / 2) * 2);
  pf_rope_table_host(c.rope_theta, c.head_dim, c.max_seq, rope.data());
  cudaError_t e = cudaMemcpyAsync(s->ws + L.rope, rope.data(), rope.size() * 4, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(s->ws + L.status, 0, STATUS_WORDS * 4, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(s->ws + L.gemm, 0, L.gemm_bytes, st);  // tile counters
  if (e == cudaSuccess && L.attn_part_bytes)  // split-KV arrival counters
    e = cudaMemsetAsync(s->ws + L.attn_part, 0, attention_counter_bytes(c), st);
  if (c.kv_block_pool > 0) {  // every position block unassigned (-1)
    s->blocks.assign(block_table_entries(c), -1);
    if (e == cudaSuccess) e = cudaMemsetAsync(s->ws + L.blocks, 0xff, s->blocks.size() * sizeof(int), st);
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) {
    delete s;
    return cuda_fail(e, "session init");
  }
  prepare_all();
  *out = s;
  return PF_OK;
}

pf_status pf_session_destroy(pf_session* s) {
  if (!s) return fail(PF_ERR_INVALID_ARG, "session is NULL");
  for (auto& kv : s->execs) cudaGraphExecDestroy(kv.second.exec);
  for (auto& r : s->prof) {
    cudaEventDestroy(r.e0);
    cudaEventDestroy(r.e1);
  }
  for (auto e : s->event_pool) cudaEventDestroy(e);
  if (s->capture_stream) cudaStreamDestroy(s->capture_stream);
  delete s;
  return PF_OK;
}

int32_t pf_session_position(const pf_session* s) { return s ? s->position : -1; }

pf_status pf_session_set_position(pf_session* s, int32_t position) {
  if (!s) return fail(PF_ERR_INVALID_ARG, "session is NULL");
  if (position < 0 || position > s->model.cfg.max_seq)
    return fail(PF_ERR_KV_CAPACITY, "position %d outside [0, %d]", position, s->model.cfg.max_seq);
  s->position = position;
  return PF_OK;
}

pf_status pf_session_set_block_table(pf_session* s, const int32_t* table, int32_t n) {
  if (!s) return fail(PF_ERR_INVALID_ARG, "session is NULL");
  const pf_config& c = s->model.cfg;
  if (c.kv_block_pool <= 0) return fail(PF_ERR_UNSUPPORTED, "not a paged cache (kv_block_pool 0)");
  if (!table) return fail(PF_ERR_INVALID_ARG, "table is NULL");
  if (n != block_table_entries(c))
    return fail(PF_ERR_SHAPE, "block table of %d entries; this configuration has %d", n, block_table_entries(c));
  std::vector<char> used(c.kv_block_pool, 0);
  for (int i = 0; i < n; ++i) {
    if (table[i] == -1) continue;
    if (table[i] < 0 || table[i] >= c.kv_block_pool)
      return fail(PF_ERR_SHAPE, "block table entry %d = %d outside [0, %d) (or -1)", i, table[i], c.kv_block_pool);
    if (used[table[i]]) return fail(PF_ERR_SHAPE, "block table entry %d repeats physical block %d", i, table[i]);
    used[table[i]] = 1;
  }
  PF_CUDA(cudaMemcpy(s->ws + s->L.blocks, table, static_cast<size_t>(n) * sizeof(int), cudaMemcpyHostToDevice),
          "block table upload");
  s->blocks.assign(table, table + n);
  return PF_OK;
}

pf_status pf_session_set_graphs(pf_session* s, int32_t enable) {
  if (!s) return fail(PF_ERR_INVALID_ARG, "session is NULL");
  s->graphs = enable != 0;
  return PF_OK;
}

pf_status pf_session_set_profile(pf_session* s, int32_t enable) {
  if (!s) return fail(PF_ERR_INVALID_ARG, "session is NULL");
  s->profile = enable != 0;
  return PF_OK;
}

pf_status pf_timeline_set(uint64_t* buffer, int64_t capacity) {
  if (buffer != nullptr && capacity <= 0) return fail(PF_ERR_INVALID_ARG, "timeline capacity %lld", (long long)capacity);
  unsigned long long* b = reinterpret_cast<unsigned long long*>(buffer);
  if (b != nullptr) {
    const unsigned long long hdr[4] = {0ull, static_cast<unsigned long long>(capacity), 0ull, 0ull};
    PF_CUDA(cudaMemcpy(b, hdr, sizeof(hdr), cudaMemcpyHostToDevice), "timeline header");
  }
  PF_CUDA(timeline_set_kernels(b), "timeline");
  PF_CUDA(timeline_set_gemm_q(b), "timeline");
  PF_CUDA(timeline_set_gemm_small(b), "timeline");
  PF_CUDA(timeline_set_gemv(b), "timeline");
  PF_CUDA(timeline_set_attention(b), "timeline");
  PF_CUDA(timeline_set_attention_tc(b), "timeline");
  return PF_OK;
}

const char* pf_timeline_kernel_name(int32_t id) {
  static const std::vector<std::string> names = [] {
    std::vector<std::string> n(64);
    const char* fixed[15] = {"", "rmsnorm", "rmsnorm_reg", "qk_norm_rope_kv", "ring_store", "embed",
                             "lm_head", "dequant", "set_int", "argmax_rows", "wait_selftest", "lm_head_q1",
                             "attention_f32", "attention_tc", "attn_combine"};
    for (int i = 1; i < 15; ++i) n[i] = fixed[i];
    const char* epi[3] = {"store", "resid", "swiglu"};
    for (int e = 0; e < 3; ++e) {
      n[TL_GEMM + e] = std::string("gemm_") + epi[e];
      n[TL_GEMM + 3 + e] = std::string("gemm_pair_") + epi[e];
      n[TL_GEMM_SMALL + e] = std::string("gemm_small_") + epi[e];
      n[TL_GEMV + e] = std::string("gemv_") + epi[e];
    }
    return n;
  }();
  if (id < 1 || id >= 64 || names[id].empty()) return nullptr;
  return names[id].c_str();
}

pf_status pf_session_profile_read(pf_session* s, void* stream, double* ms_out, int64_t* launches_out) {
  if (!s || !ms_out || !launches_out) return fail(PF_ERR_INVALID_ARG, "NULL pointer");
  PF_CUDA(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)), "stream sync");
  for (int i = 0; i < PF_K_COUNT; ++i) {
    ms_out[i] = 0.0;
    launches_out[i] = 0;
  }
  for (auto& r : s->prof) {
    float ms = 0.f;
    PF_CUDA(cudaEventElapsedTime(&ms, r.e0, r.e1), "event elapsed");
    ms_out[r.cls] += ms;
    launches_out[r.cls] += 1;
    s->event_pool.push_back(r.e0);
    s->event_pool.push_back(r.e1);
  }
  s->prof.clear();
  return PF_OK;
}

int64_t pf_session_kernel_launches(const pf_session* s) { return s ? s->launches : -1; }

pf_status pf_session_sync(pf_session* s, void* stream) {
  if (!s) return fail(PF_ERR_INVALID_ARG, "session is NULL");
  return pf_status_read(wsp<int>(s, s->L.status), stream);
}

pf_status pf_selftest_bounded_wait(int32_t* status_dev, int64_t limit_ns, int32_t arrive,
                                   void* stream) {
  if (!status_dev) return fail(PF_ERR_INVALID_ARG, "status pointer is NULL");
  if (limit_ns < 1000 || limit_ns > 10000000000LL) return fail(PF_ERR_INVALID_ARG, "limit_ns %lld", (long long)limit_ns);
  PF_CUDA(launch_wait_selftest(status_dev, limit_ns, arrive, static_cast<cudaStream_t>(stream)),
          "wait selftest");
  return PF_OK;
}

pf_status pf_status_read(int32_t* status_dev, void* stream) {
  if (!status_dev) return fail(PF_ERR_INVALID_ARG, "status pointer is NULL");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int32_t h = 0;
  PF_CUDA(cudaStreamSynchronize(st), "stream sync");
  PF_CUDA(cudaMemcpy(&h, status_dev, 4, cudaMemcpyDeviceToHost), "status read");
  if (h != 0) {
    PF_CUDA(cudaMemset(status_dev, 0, 4), "status clear");
    return fail(static_cast<pf_status>(h), "device status %d (%s) recorded by a kernel", h, pf_status_name(h));
  }
  return PF_OK;
}

// tokens: host ids (checked here, copied per micro-batch) or, with tokens_on_device, device
// ids (checked by the embedding kernel); x: hidden rows when tokens is NULL.
static pf_status prefill_common(pf_session* s, const int32_t* tokens, bool tokens_on_device,
                                float* x, int32_t M, int32_t start, float* logits, void* stream) {
  if (!s) return fail(PF_ERR_INVALID_ARG, "session is NULL");
  const pf_config& c = s->model.cfg;
  if (M > 0 && tokens == nullptr && x == nullptr) return fail(PF_ERR_INVALID_ARG, "input is NULL");
  if (tokens && (!s->model.embed || c.vocab <= 0)) return fail(PF_ERR_INVALID_ARG, "model has no embedding table");
  const int has_head = s->model.lm_head && s->model.final_norm && c.vocab > 0;
  pf_status v = pf_validate_chunk(&c, s->position, tokens_on_device ? nullptr : tokens, M, start,
                                  logits != nullptr, has_head);
  if (v != PF_OK) return v;
  v = check_blocks(s, static_cast<int64_t>(start) + M);
  if (v != PF_OK) return v;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int off = 0;
  while (off < M) {  // micro-batches of at most max_chunk rows; head on the last only
    const int m = std::min(M - off, c.max_chunk);
    const bool last = off + m == M;
    float* xc;
    const int* tok_dev = nullptr;
    if (tokens) {
      xc = wsp<float>(s, s->L.x);
      if (tokens_on_device) {
        tok_dev = tokens + off;
      } else {
        tok_dev = wsp<int>(s, s->L.tokens);
        PF_CUDA(cudaMemcpyAsync(wsp<int>(s, s->L.tokens), tokens + off, static_cast<size_t>(m) * 4,
                                cudaMemcpyHostToDevice, st),
                "tokens upload");
      }
    } else {
      xc = x + static_cast<size_t>(off) * c.hidden;
    }
    PF_TRY(set_start(s, start + off, st));
    float* lg = last ? logits : nullptr;
    GraphKey key{m, xc, tok_dev, lg, -1};
    PF_TRY(run_maybe_graph(s, key, st,
                           [&](cudaStream_t rs) { return enqueue_chunk(s, xc, m, tok_dev, lg, rs); }));
    s->position = start + off + m;  // turbospark prefill.rs: kv.advance_by(m)
    off += m;
  }
  return PF_OK;
}

pf_status pf_prefill_chunk(pf_session* s, const int32_t* tokens_host, int32_t M, int32_t start_pos,
                           float* logits_dev, void* stream) {
  if (s && M > 0 && !tokens_host) return fail(PF_ERR_INVALID_ARG, "tokens is NULL");
  return prefill_common(s, tokens_host, false, nullptr, M, start_pos, logits_dev, stream);
}

pf_status pf_prefill_chunk_dev(pf_session* s, const int32_t* tokens_dev, int32_t M, int32_t start_pos,
                               float* logits_dev, void* stream) {
  if (s && M > 0 && !tokens_dev) return fail(PF_ERR_INVALID_ARG, "tokens is NULL");
  return prefill_common(s, tokens_dev, true, nullptr, M, start_pos, logits_dev, stream);
}

pf_status pf_decode_step(pf_session* s, const int32_t* token_dev, float* logits_dev, void* stream) {
  if (!s) return fail(PF_ERR_INVALID_ARG, "session is NULL");
  if (!token_dev) return fail(PF_ERR_INVALID_ARG, "token is NULL");
  if (!logits_dev) return fail(PF_ERR_LOGITS, "decode needs logits");
  return prefill_common(s, token_dev, true, nullptr, 1, s->position, logits_dev, stream);
}

pf_status pf_decode_step_greedy(pf_session* s, const int32_t* token_in_dev, int32_t* token_out_dev,
                                float* logits_dev, void* stream) {
  if (!s) return fail(PF_ERR_INVALID_ARG, "session is NULL");
  if (!token_in_dev || !token_out_dev) return fail(PF_ERR_INVALID_ARG, "token is NULL");
  if (!logits_dev) return fail(PF_ERR_LOGITS, "decode needs logits");
  pf_status r = prefill_common(s, token_in_dev, true, nullptr, 1, s->position, logits_dev, stream);
  if (r != PF_OK) return r;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int vocab = s->model.cfg.vocab;
  return launch_k(s, PF_K_OTHER, st, "argmax",
                  [&] { return launch_argmax_rows(logits_dev, 1, vocab, vocab, token_out_dev, st); });
}

// P1 encode_full_forward_prefill_verify: the layer loop of one micro-batch, then the
// batched final RMSNorm on all positions, the LM-head GEMM on all positions and one argmax
// per position.
pf_status pf_prefill_verify(pf_session* s, const int32_t* tokens_dev, int32_t M, int32_t start_pos,
                            float* logits_all_dev, int32_t* ids_dev, void* stream) {
  if (!s) return fail(PF_ERR_INVALID_ARG, "session is NULL");
  const pf_config& c = s->model.cfg;
  if (!tokens_dev || !logits_all_dev || !ids_dev) return fail(PF_ERR_INVALID_ARG, "NULL pointer");
  if (!s->model.lm_head || !s->model.final_norm || c.vocab <= 0)
    return fail(PF_ERR_LOGITS, "verify needs the final norm and LM head");
  if (M > c.max_chunk) return fail(PF_ERR_SHAPE, "verify chunk M %d exceeds max_chunk %d", M, c.max_chunk);
  if (c.vocab % 8) return fail(PF_ERR_SHAPE, "verify needs vocab %% 8 == 0 (vocab %d)", c.vocab);
  if (reinterpret_cast<uintptr_t>(logits_all_dev) & 15) return fail(PF_ERR_INVALID_ARG, "logits must be 16-B aligned");
  pf_status r = prefill_common(s, tokens_dev, true, nullptr, M, start_pos, nullptr, stream);
  if (r != PF_OK) return r;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const float* x = wsp<float>(s, s->L.x);  // the final hidden rows of the micro-batch
  void* y = wsp<void>(s, s->L.y);
  PF_TRY(launch_k(s, PF_K_RMSNORM, st, "final rmsnorm", [&] {
    return launch_rmsnorm(x, s->model.final_norm, c.final_eps, M, c.hidden, y, st);
  }));
  PF_TRY(enqueue_gemm(s, PF_K_LM_HEAD, c.wfmt, EPI_STORE_F32, y, s->model.lm_head, M, c.vocab, c.hidden,
                      logits_all_dev, st));
  return launch_k(s, PF_K_OTHER, st, "argmax", [&] {
    return launch_argmax_rows(logits_all_dev, M, c.vocab, c.vocab, ids_dev, st);
  });
}

pf_status pf_prefill_hidden(pf_session* s, float* x_dev, int32_t M, int32_t start_pos,
                            float* logits_dev, void* stream) {
  if (s && M > 0 && !x_dev) return fail(PF_ERR_INVALID_ARG, "x is NULL");
  return prefill_common(s, nullptr, false, x_dev, M, start_pos, logits_dev, stream);
}

pf_status pf_layer_forward(pf_session* s, int32_t layer, float* x_dev, int32_t M, int32_t start_pos,
                           void* stream) {
  if (!s) return fail(PF_ERR_INVALID_ARG, "session is NULL");
  const pf_config& c = s->model.cfg;
  if (layer < 0 || layer >= c.n_layers) return fail(PF_ERR_INVALID_ARG, "layer %d of %d", layer, c.n_layers);
  if (M <= 0) return fail(PF_ERR_EMPTY_CHUNK, "empty chunk (M = %d)", M);
  if (M > c.max_chunk) return fail(PF_ERR_SHAPE, "M %d exceeds max_chunk %d", M, c.max_chunk);
  if (!x_dev) return fail(PF_ERR_INVALID_ARG, "x is NULL");
  if (start_pos < 0 || static_cast<int64_t>(start_pos) + M > c.max_seq)
    return fail(PF_ERR_KV_CAPACITY, "chunk [%d, %d) exceeds KV capacity %d", start_pos, start_pos + M, c.max_seq);
  pf_status r = check_blocks(s, static_cast<int64_t>(start_pos) + M);
  if (r != PF_OK) return r;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  r = set_start(s, start_pos, st);
  if (r != PF_OK) return r;
  GraphKey key{M, x_dev, nullptr, nullptr, layer};
  return run_maybe_graph(s, key, st,
                         [&](cudaStream_t rs) { return enqueue_layer(s, layer, x_dev, M, rs, false, false); });
}

pf_status pf_prefill_tokens_host(pf_session* s, const int32_t* tokens_host, int32_t M, int32_t start_pos,
                                 float* logits_host, void* stream) {
  if (!s) return fail(PF_ERR_INVALID_ARG, "session is NULL");
  const pf_config& c = s->model.cfg;
  float* lg_dev = nullptr;
  if (logits_host) {
    if (!s->model.lm_head || c.vocab <= 0) return fail(PF_ERR_LOGITS, "no LM head");
    lg_dev = wsp<float>(s, s->L.logits);  // device copy of the logits before the download
  }
  pf_status r = pf_prefill_chunk(s, tokens_host, M, start_pos, lg_dev, stream);
  if (r != PF_OK) return r;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (logits_host)
    PF_CUDA(cudaMemcpyAsync(logits_host, lg_dev, static_cast<size_t>(c.vocab) * 4,
                            cudaMemcpyDeviceToHost, st),
            "logits download");
  PF_CUDA(cudaStreamSynchronize(st), "sync");
  return PF_OK;
}

// ---------------------------------------------------------------------- single steps
pf_status pf_op_rmsnorm(const float* x, const float* w, float eps, int32_t M, int32_t H,
                        uint16_t* y, void* stream) {
  if (!x || !w || !y) return fail(PF_ERR_INVALID_ARG, "NULL pointer");
  if (M <= 0 || H <= 0 || H % 4) return fail(PF_ERR_SHAPE, "M %d, H %d", M, H);
  PF_CUDA(launch_rmsnorm(x, w, eps, M, H, y, static_cast<cudaStream_t>(stream)), "rmsnorm");
  return PF_OK;
}

pf_status pf_op_dequant(int32_t wfmt, const void* packed, int64_t N, int64_t K, uint16_t* w,
                        void* stream) {
  if (pf_packed_bytes(wfmt, N, K) == 0) return fail(PF_ERR_SHAPE, "dequant shape");
  if (!packed || !w) return fail(PF_ERR_INVALID_ARG, "NULL pointer");
  PF_CUDA(launch_dequant(wfmt, static_cast<const uint8_t*>(packed), N, K, w,
                         static_cast<cudaStream_t>(stream)),
          "dequant");
  return PF_OK;
}

size_t pf_gemm_scratch_bytes(int32_t M, int32_t N, int32_t max_ctas) {
  if (M <= 0 || N <= 0 || max_ctas < 0 || max_ctas > GEMM_MAX_CTAS) return 0;
  return gemm_scratch_bytes(M, N, max_ctas == 0 ? GEMM_MAX_CTAS : max_ctas);
}

pf_status pf_op_gemm(int32_t wfmt, int32_t epi, const uint16_t* a, const void* packed, int32_t M,
                     int32_t N, int32_t K, void* out, int32_t max_ctas, void* scratch,
                     size_t scratch_bytes, int32_t* status, void* stream) {
  if (!a || !packed || !out) return fail(PF_ERR_INVALID_ARG, "NULL pointer");
  if (wfmt != PF_W_Q1_G128 && wfmt != PF_W_INT4_AFFINE_G128) return fail(PF_ERR_INVALID_ARG, "format");
  if (epi < EPI_STORE_F32 || epi > EPI_SWIGLU) return fail(PF_ERR_INVALID_ARG, "epilogue %d", epi);
  if (M <= 0 || N <= 0 || K <= 0 || K % 128 || N % 8) return fail(PF_ERR_SHAPE, "M %d N %d K %d", M, N, K);
  if (epi == EPI_SWIGLU && N % 256) return fail(PF_ERR_SHAPE, "SwiGLU needs N = 2I with I %% 128 == 0");
  if ((reinterpret_cast<uintptr_t>(a) & 15) || (reinterpret_cast<uintptr_t>(out) & 15))
    return fail(PF_ERR_INVALID_ARG, "a and out must be 16-B aligned");
  if (max_ctas < 0 || max_ctas > GEMM_MAX_CTAS)
    return fail(PF_ERR_INVALID_ARG, "max_ctas %d outside [0, %d]", max_ctas, GEMM_MAX_CTAS);
  if (max_ctas == 0) max_ctas = GEMM_MAX_CTAS;
  const size_t need = gemm_scratch_bytes(M, N, max_ctas);
  if (!scratch || scratch_bytes < need)
    return fail(PF_ERR_WORKSPACE, "GEMM scratch %zu bytes, need %zu", scratch_bytes, need);
  if (reinterpret_cast<uintptr_t>(scratch) & 15) return fail(PF_ERR_INVALID_ARG, "scratch must be 16-B aligned");
  prepare_all();
  GemmArgs g{};
  g.wfmt = wfmt;
  g.epilogue = epi;
  g.a = a;
  g.w = static_cast<const uint8_t*>(packed);
  g.M = M;
  g.N = N;
  g.K = K;
  g.out = out;
  g.max_ctas = max_ctas;
  g.scratch = scratch;
  g.status = status;
  PF_CUDA(launch_gemm(g, static_cast<cudaStream_t>(stream)), "gemm");
  return PF_OK;
}

// ---------------------------------------------------------------------- GEMM without allocation
// For callers that may not allocate device memory: a plug-in whose host owns every device
// allocation through its own pool, or a latency-bound service that cannot afford the device
// synchronisation cudaMalloc / cudaFree may cause once it runs. The GEMM's scratch then lives
// in this fixed array, which every GPU that loads the library keeps until the process exits.
namespace {
constexpr int STATIC_GEMM_CTAS = 16;          // partial tiles for at most 16 CTAs: 4 MiB
constexpr size_t STATIC_GEMM_TILES = 16384;   // arrival counters: 64 KiB
constexpr size_t STATIC_GEMM_BYTES =
    static_cast<size_t>(2) * STATIC_GEMM_CTAS * 128 * 256 * sizeof(float) + STATIC_GEMM_TILES * sizeof(int);
static __device__ __align__(256) unsigned char g_static_gemm_scratch[STATIC_GEMM_BYTES];

// Device address of the array on the current device (host code cannot use the symbol
// itself: on the host it names a stand-in, not device memory). Looked up on every call:
// the lookup is cheap once the module is loaded, and an address kept from an earlier call
// could be stale after cudaDeviceReset or a new primary context reloads the module.
pf_status static_gemm_scratch(void** out) {
  void* p = nullptr;
  PF_CUDA(cudaGetSymbolAddress(&p, g_static_gemm_scratch), "cudaGetSymbolAddress");
  *out = p;
  return PF_OK;
}
}  // namespace

pf_status pf_op_gemm_static_scratch(int32_t wfmt, int32_t epi, const uint16_t* a, const void* packed,
                                    int32_t M, int32_t N, int32_t K, void* out, int32_t* status,
                                    void* stream) {
  if (!a || !packed || !out) return fail(PF_ERR_INVALID_ARG, "NULL pointer");
  if (wfmt != PF_W_Q1_G128 && wfmt != PF_W_INT4_AFFINE_G128) return fail(PF_ERR_INVALID_ARG, "format");
  if (epi < EPI_STORE_F32 || epi > EPI_SWIGLU) return fail(PF_ERR_INVALID_ARG, "epilogue %d", epi);
  if (M <= 0 || N <= 0 || K <= 0 || K % 128 || N % 8) return fail(PF_ERR_SHAPE, "M %d N %d K %d", M, N, K);
  if (epi == EPI_SWIGLU && N % 256) return fail(PF_ERR_SHAPE, "SwiGLU needs N = 2I with I %% 128 == 0");
  if ((reinterpret_cast<uintptr_t>(a) & 15) || (reinterpret_cast<uintptr_t>(out) & 15))
    return fail(PF_ERR_INVALID_ARG, "a and out must be 16-B aligned");
  // arrival counters: one per 128 x 256 tile, or two per 256 x 256 tile of a CTA pair
  const size_t tiles = std::max<size_t>((M + 127) / 128, 2 * ((M + 255) / 256)) *
                       static_cast<size_t>((N + 255) / 256);
  if (tiles > STATIC_GEMM_TILES)
    return fail(PF_ERR_SHAPE,
                "M %d x N %d is %zu output tiles of 128 x 256; the static GEMM scratch holds at most %zu",
                M, N, tiles, STATIC_GEMM_TILES);
  if (gemm_scratch_bytes(M, N, STATIC_GEMM_CTAS) > STATIC_GEMM_BYTES)
    return fail(PF_ERR_SHAPE, "M %d x N %d needs more than the static GEMM scratch", M, N);
  void* scratch = nullptr;
  pf_status r = static_gemm_scratch(&scratch);
  if (r != PF_OK) return r;
  prepare_all();
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // the arrival counters must start at zero; a call that completes leaves them zero, one that
  // timed out may not, so clear the ones this call uses
  void* counters = static_cast<unsigned char*>(scratch) + (STATIC_GEMM_BYTES - STATIC_GEMM_TILES * sizeof(int));
  PF_CUDA(cudaMemsetAsync(counters, 0, tiles * sizeof(int), st), "clear GEMM counters");
  GemmArgs g{};
  g.wfmt = wfmt;
  g.epilogue = epi;
  g.a = a;
  g.w = static_cast<const uint8_t*>(packed);
  g.M = M;
  g.N = N;
  g.K = K;
  g.out = out;
  g.max_ctas = STATIC_GEMM_CTAS;
  g.scratch = scratch;
  g.status = status;
  PF_CUDA(launch_gemm(g, st), "gemm");
  return PF_OK;
}

pf_status pf_op_qk_norm_rope_kv(const pf_config* cfg, const float* qkv, const float* qn,
                                const float* kn, const float* rope, int32_t layer, int32_t start,
                                int32_t M, void* q, void* kc, void* vc, void* stream) {
  pf_status r = check_cfg(cfg);
  if (r != PF_OK) return r;
  if (cfg->ring_capacity > 0 || cfg->kv_block_pool > 0)
    return fail(PF_ERR_UNSUPPORTED, "single-step KV store: linear caches only");
  if (!qkv || !rope || !q || !kc || !vc || (cfg->qk_norm && (!qn || !kn)))
    return fail(PF_ERR_INVALID_ARG, "NULL pointer");
  if (M <= 0 || layer < 0 || layer >= cfg->n_layers || start < 0 ||
      static_cast<int64_t>(start) + M > cfg->max_seq)
    return fail(PF_ERR_SHAPE, "M %d layer %d start %d", M, layer, start);
  PF_CUDA(launch_qk_norm_rope_kv(*cfg, qkv, qn, kn, rope, layer, cfg->max_seq, 1, nullptr, start, M, q,
                                 kc, vc, static_cast<cudaStream_t>(stream)),
          "qk_norm_rope_kv");
  return PF_OK;
}

static pf_status attention_op(const pf_config* cfg, const void* q, const void* kc, const void* vc,
                              int32_t layer, int32_t start, int32_t M, int32_t n_split, void* scratch,
                              size_t scratch_bytes, uint16_t* out, void* stream) {
  pf_status r = check_cfg(cfg);
  if (r != PF_OK) return r;
  if (cfg->ring_capacity > 0 || cfg->kv_block_pool > 0)
    return fail(PF_ERR_UNSUPPORTED, "single-step attention: linear caches only");
  if (!q || !kc || !vc || !out) return fail(PF_ERR_INVALID_ARG, "NULL pointer");
  if (M <= 0 || layer < 0 || layer >= cfg->n_layers || start < 0 ||
      static_cast<int64_t>(start) + M > cfg->max_seq)
    return fail(PF_ERR_SHAPE, "M %d layer %d start %d", M, layer, start);
  if (n_split > 1) {
    if (!attention_tc_supported(*cfg)) return fail(PF_ERR_UNSUPPORTED, "split-KV attention needs a 16-bit cache");
    if (n_split > 64) return fail(PF_ERR_INVALID_ARG, "n_split %d outside 1..64", n_split);
    const size_t need = attention_partial_bytes(*cfg, M, n_split);
    if (!scratch || scratch_bytes < need)
      return fail(PF_ERR_WORKSPACE, "attention scratch %zu bytes, need %zu", scratch_bytes, need);
    if (reinterpret_cast<uintptr_t>(scratch) & 15) return fail(PF_ERR_INVALID_ARG, "scratch must be 16-B aligned");
  }
  prepare_all();
  AttnArgs a{};
  a.c = cfg;
  a.q = q;
  a.k_cache = kc;
  a.v_cache = vc;
  a.layer = layer;
  a.start_host = start;
  a.M = M;
  a.out = out;
  a.n_split = n_split < 1 ? 1 : n_split;
  a.partial = static_cast<float*>(scratch);
  if (n_split > 1)  // the caller's scratch: its arrival counters start at zero
    PF_CUDA(cudaMemsetAsync(scratch, 0, attention_counter_bytes(*cfg), static_cast<cudaStream_t>(stream)),
            "attention counters");
  PF_CUDA(launch_attention(a, static_cast<cudaStream_t>(stream)), "attention");
  return PF_OK;
}

pf_status pf_op_attention(const pf_config* cfg, const void* q, const void* kc, const void* vc,
                          int32_t layer, int32_t start, int32_t M, uint16_t* out, void* stream) {
  return attention_op(cfg, q, kc, vc, layer, start, M, 1, nullptr, 0, out, stream);
}

size_t pf_attention_scratch_bytes(const pf_config* cfg, int32_t M, int32_t n_split) {
  if (check_cfg(cfg) != PF_OK || M <= 0 || n_split < 1 || n_split > 64) return 0;
  return attention_partial_bytes(*cfg, M, n_split);
}

pf_status pf_op_attention_split(const pf_config* cfg, const void* q, const void* kc, const void* vc,
                                int32_t layer, int32_t start, int32_t M, int32_t n_split, void* scratch,
                                size_t scratch_bytes, uint16_t* out, void* stream) {
  if (n_split < 1) return fail(PF_ERR_INVALID_ARG, "n_split %d outside 1..64", n_split);
  return attention_op(cfg, q, kc, vc, layer, start, M, n_split, scratch, scratch_bytes, out, stream);
}

pf_status pf_op_embed(const float* E, const int32_t* tokens, int32_t M, int32_t H, int32_t vocab,
                      float* x, int32_t* status, void* stream) {
  if (!E || !tokens || !x) return fail(PF_ERR_INVALID_ARG, "NULL pointer");
  if (M <= 0 || H <= 0 || H % 4 || vocab <= 0) return fail(PF_ERR_SHAPE, "M %d H %d vocab %d", M, H, vocab);
  PF_CUDA(launch_embed(E, tokens, M, H, vocab, x, status, static_cast<cudaStream_t>(stream)), "embed");
  return PF_OK;
}

pf_status pf_op_lm_head(int32_t wfmt, const float* x_row, const float* nw, float eps,
                        const void* packed, int32_t vocab, int32_t H, float* logits, void* stream) {
  if (!x_row || !nw || !packed || !logits) return fail(PF_ERR_INVALID_ARG, "NULL pointer");
  if (pf_packed_bytes(wfmt, vocab, H) == 0) return fail(PF_ERR_SHAPE, "vocab %d H %d", vocab, H);
  PF_CUDA(launch_lm_head(wfmt, x_row, nw, eps, static_cast<const uint8_t*>(packed), vocab, H,
                         logits, static_cast<cudaStream_t>(stream)),
          "lm_head");
  return PF_OK;
}

pf_status pf_op_argmax(const float* x, int32_t rows, int32_t n, int64_t ld, int32_t* out, void* stream) {
  if (!x || !out) return fail(PF_ERR_INVALID_ARG, "NULL pointer");
  if (rows <= 0 || n <= 0 || ld < n) return fail(PF_ERR_SHAPE, "rows %d n %d ld %lld", rows, n, (long long)ld);
  PF_CUDA(launch_argmax_rows(x, rows, n, ld, out, static_cast<cudaStream_t>(stream)), "argmax");
  return PF_OK;
}

}  // extern "C"

pf_status pf_streamk_plan_host(int32_t n_mt, int32_t n_nt, int32_t kbt, int32_t ctas, int32_t late_units,
                               int32_t late_kb, int64_t* begins, int32_t* segs, int32_t max_segs,
                               const int64_t* w_query, int32_t n_query, int32_t* owners) {
  using namespace pf;
  if (!begins || !segs) return fail(PF_ERR_INVALID_ARG, "NULL pointer");
  if (n_mt < 1 || n_nt < 1 || kbt < 1 || ctas < 1 || max_segs < 1 || late_units < 0 || late_kb < 0)
    return fail(PF_ERR_SHAPE, "plan sizes");
  sk::Plan p{};
  p.n_mt = n_mt;
  p.n_nt = n_nt;
  p.kbt = kbt;
  p.total = static_cast<long long>(n_mt) * n_nt * kbt;
  if (ctas > p.total) return fail(PF_ERR_SHAPE, "ctas %d > %lld k-blocks", ctas, p.total);
  p.ctas = ctas;
  streamk_skew(p, late_units, late_kb);
  for (int c = 0; c <= ctas; ++c) begins[c] = p.begin(c);
  for (int c = 0; c < ctas; ++c) {
    const sk::Range rg(p, c);
    if (rg.n > max_segs) return fail(PF_ERR_SHAPE, "unit %d has %d segments", c, rg.n);
    for (int k = 0; k < max_segs; ++k) {
      int32_t* o = segs + (static_cast<size_t>(c) * max_segs + k) * 4;
      if (k >= rg.n) {
        o[0] = -1;
        o[1] = o[2] = o[3] = 0;
        continue;
      }
      const sk::Segment sg = rg.at(p, k);
      o[0] = sg.tile;
      o[1] = sg.kb0;
      o[2] = sg.nkb;
      o[3] = sg.whole ? -1 : p.slot(c, sg.tile);
    }
  }
  if (owners && w_query)
    for (int i = 0; i < n_query; ++i) owners[i] = p.owner(w_query[i]);
  return PF_OK;
}
