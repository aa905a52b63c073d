// pf_internal.h — definitions shared by libpf's translation units (not installed).
#pragma once
#include <cstddef>
#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/pf.h"

// A bounded device-side wait gives up after this long (ns) and reports
// PF_ERR_DEVICE_TIMEOUT; healthy waits last microseconds.
#ifndef PF_WAIT_LIMIT_NS
#define PF_WAIT_LIMIT_NS 1000000000ull
#endif

namespace pf {

// ------------------------------------------------------------------ packed weight layout
// Cache slots per (layer, kv head): ring slots, paged blocks x PF_KV_BLOCK, or max_seq.
inline int cache_slots(const pf_config& c) {
  return c.ring_capacity > 0 ? c.ring_capacity : (c.kv_block_pool > 0 ? c.kv_block_pool * PF_KV_BLOCK : c.max_seq);
}
// Entries of a paged session's block table.
inline int block_table_entries(const pf_config& c) { return (c.max_seq + PF_KV_BLOCK - 1) / PF_KV_BLOCK; }

// Tiles of TILE_N = 256 rows x GROUP = 128 weights ("chunks"), chunk (t, g) at byte
// offset (t * K/128 + g) * chunk_bytes. Inside a chunk, each half h (k in
// [128g + 64h, 128g + 64h + 64)) of every row is contiguous so that one GEMM stage
// (64 k x 256 rows) is one contiguous block, followed by the 256 scales (and zeros).
//
// Q1 half-row (8 B): two 32-bit words Z0 (k 0..31 of the half), Z1 (k 32..63). In a
// word, element pair i (elements 2i, 2i+1) keeps the NEGATIVE flag of element 2i at
// bit 15-i and of element 2i+1 at bit 31-i, so ((Z << i) & 0x80008000) is directly the
// f16x2 sign mask of pair i.
// INT4 half-row (32 B): eight 32-bit words, word w = k 8w..8w+7; pair p of the word
// (elements 8w+2p, 8w+2p+1) keeps the even code at bits [4p, 4p+4) and the odd code at
// bits [16+4p, 16+4p+4), so ((word >> 4p) & 0x000F000F) are both codes of pair p.
constexpr int TILE_N = 256;
constexpr int GROUP = 128;
constexpr int Q1_HALF_BYTES = TILE_N * 8;            // 2048
constexpr int Q1_SCALE_OFF = 2 * Q1_HALF_BYTES;       // 4096
constexpr int Q1_CHUNK_BYTES = Q1_SCALE_OFF + TILE_N * 2;  // 4608
constexpr int I4_HALF_BYTES = TILE_N * 32;           // 8192
constexpr int I4_SCALE_OFF = 2 * I4_HALF_BYTES;       // 16384
constexpr int I4_ZERO_OFF = I4_SCALE_OFF + TILE_N * 2; // 16896
constexpr int I4_CHUNK_BYTES = I4_ZERO_OFF + TILE_N * 2;  // 17408

__host__ __device__ inline int64_t padded_rows(int64_t N) { return (N + TILE_N - 1) / TILE_N * TILE_N; }
__host__ __device__ inline size_t chunk_bytes(int wfmt) {
  return wfmt == PF_W_Q1_G128 ? Q1_CHUNK_BYTES : I4_CHUNK_BYTES;
}

enum Epilogue : int { EPI_STORE_F32 = 0, EPI_RESID_ADD = 1, EPI_SWIGLU = 2 };

// ------------------------------------------------------------------ status words
// int32 [4] in device memory: [0] = first error code recorded by a kernel.
constexpr int STATUS_WORDS = 4;

// ------------------------------------------------------------------ launchers
// Each returns cudaGetLastError() after enqueueing on `stream`.
struct GemmArgs {
  int wfmt;
  int epilogue;
  const void* a;        // f16 [M, K] row-major
  const uint8_t* w;     // packed
  int M, N, K;
  void* out;            // f32 [M, N] or f16 [M, N/2], 16-B aligned
  int max_ctas;         // 1..GEMM_MAX_CTAS; the scratch layout depends on it
  void* scratch;        // gemm_scratch_bytes(M, N, max_ctas); its counters zero before the launch
  int* status;          // may be NULL
  bool out_zeroed;      // store form: the caller has set out to zero (every path accumulates
                        // the store form into a zeroed output; without this flag it zeroes
                        // it itself first)
  // optional (M > SMALL_M_MAX only): a buffer that the CTAs' epilogue warps set to zero while
  // the main loop runs (the accumulator of a later store-form GEMM); 16-B aligned and sized
  void* side_zero;
  size_t side_zero_bytes;
  // optional stream-K skew (CTA-pair form): the last `late_units` units take `late_kb`
  // k-blocks fewer each, for CTAs that start late on SMs the previous kernel still holds
  int late_units;
  int late_kb;
};
cudaError_t launch_gemm(const GemmArgs& g, cudaStream_t stream);
namespace sk {
struct Plan;
}
// Applies a stream-K skew (GemmArgs::late_units / late_kb) to a plan whose tiles and units
// are set: units [ctas - late_units, ctas) take up to late_kb k-blocks fewer each.
void streamk_skew(sk::Plan& p, int late_units, int late_kb);
// Whether GemmArgs::side_zero is available at this M (the persistent tcgen05 GEMM).
bool gemm_side_zero_supported(int wfmt, int M);
// M <= SMALL_M_MAX: the weight rows are the MMA's M side (gemm_small.cu); launch_gemm routes
cudaError_t launch_gemm_small(const GemmArgs& g, cudaStream_t stream);
cudaError_t prepare_gemm_small_kernels();
constexpr int SMALL_M_MAX = 64;
// M <= gemv_max_m(wfmt): the warp-MMA GEMV (gemv.cu), which needs no scratch; launch_gemm
// routes there first
constexpr int GEMV_M_MAX_Q1 = 16;
constexpr int GEMV_M_MAX_I4 = 16;
int gemv_max_m(int wfmt);
cudaError_t launch_gemv(const GemmArgs& g, cudaStream_t stream);
bool encode_tmap_f16_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer,
                        uint32_t box_inner, uint32_t box_outer);
// The GEMM runs at most min(max_ctas, SMs) persistent CTAs; its scratch holds two f32
// 128 x 256 partial tiles per CTA and one arrival counter per output tile.
constexpr int GEMM_MAX_CTAS = 160;
size_t gemm_scratch_bytes(int M, int N, int max_ctas);

// y_f16 [M, H] = RMSNorm of x [M, H]; with `zero` (16-B aligned, zero_cols % 4 == 0) each
// row's CTA also sets row m of the f32 buffer zero [M, zero_cols] to 0.
cudaError_t launch_rmsnorm(const float* x, const float* w, float eps, int M, int H, void* y_f16,
                           cudaStream_t stream, float* zero = nullptr, int zero_cols = 0);
cudaError_t launch_dequant(int wfmt, const uint8_t* packed, int64_t N, int64_t K, void* w_f16,
                           cudaStream_t stream);
// K and V go to row (kv_layer * nkv + kvh) * kv_rows + (kv_by_pos ? slot(start + t) : t) of
// k_dst / v_dst: the cache slot of position p = start + t (kv_layer = layer, kv_rows = cache
// slots, kv_by_pos = 1; slot(p) = p, or with a block table blocks[p / PF_KV_BLOCK] *
// PF_KV_BLOCK + p % PF_KV_BLOCK) or row t of the ring mode's chunk buffers (0, chunk rows, 0).
cudaError_t launch_qk_norm_rope_kv(const pf_config& c, const float* qkv, const float* q_norm,
                                   const float* k_norm, const float* rope, int kv_layer, int kv_rows,
                                   int kv_by_pos, const int* start_dev, int start_host, int M,
                                   void* q_out, void* k_dst, void* v_dst, cudaStream_t stream,
                                   const int* blocks = nullptr);
// Keys an attention launch reads. A linear cache holds position p of (layer, kv head) at row
// (layer * nkv + kvh) * max_seq + p. A ring cache (ring_capacity R > 0, sink_count S) holds
// position p at slot p (p < S) or S + (p - S) mod (R - S), row (layer * nkv + kvh) * R + slot;
// the chunk's own keys are then read from the chunk buffers [nkv][chunk_rows][hd] that the
// QK-norm / RoPE kernel wrote, and stored into the ring after the attention (launch_ring_store).
struct AttnArgs {
  const pf_config* c;
  const void* q;        // [M][nq][hd] (bf16 for a bf16 cache, else f16)
  const void* k_cache;
  const void* v_cache;
  const void* k_chunk;  // ring mode only
  const void* v_chunk;
  int chunk_rows;
  int layer;
  const int* start_dev;  // start position in device memory, or NULL to use start_host
  int start_host;
  int M;
  void* out;            // f16 [M][nq * hd]
  int n_split;          // key-tile parts (split-KV); 1 = none
  float* partial;       // n_split > 1: attention_partial_bytes(c, M, n_split) bytes
  int* status;
  const int* blocks;    // paged cache: the block table (device), else NULL
};
cudaError_t launch_attention(const AttnArgs& a, cudaStream_t stream);
// Split-KV parts for a chunk of M rows on `sms` SMs (1 unless the chunk's CTAs fill less
// than half of the SMs; only the tensor-core kernel splits).
int attention_splits(const pf_config& c, int M, int sms);
size_t attention_partial_bytes(const pf_config& c, int M, int n_split);
// the largest partial buffer any M <= max_chunk needs on a GPU of at most max_sms SMs
size_t attention_partial_bytes_max(const pf_config& c, int max_sms);
// the arrival counters at the start of the partial buffer (one int per kv head, used when a
// split chunk of at most 2 tokens merges its parts in the kernel); they must be zero before
// the first launch, and every launch that completes leaves them zero
size_t attention_counter_bytes(const pf_config& c);
// Ring cache: stores the chunk's K/V rows (chunk buffers) into the ring slots of `layer`
// that the chunk's positions keep (sinks, and the last R - S positions).
cudaError_t launch_ring_store(const pf_config& c, const void* k_chunk, const void* v_chunk,
                              int chunk_rows, int layer, const int* start_dev, int start_host, int M,
                              void* k_cache, void* v_cache, cudaStream_t stream);
cudaError_t launch_embed(const float* E, const int* tokens, int M, int H, int vocab, float* x,
                         int* status, cudaStream_t stream);
cudaError_t launch_lm_head(int wfmt, const float* x_row, const float* norm_w, float eps,
                           const uint8_t* packed, int vocab, int H, float* logits,
                           cudaStream_t stream);
cudaError_t launch_set_int(int* dst, int value, cudaStream_t stream);
// out[r] = index of the largest of x[r * ld + 0 .. n-1] (lowest index on ties, NaN never wins)
cudaError_t launch_argmax_rows(const float* x, int rows, int n, long long ld, int* out, cudaStream_t stream);
cudaError_t launch_wait_selftest(int* status, long long limit_ns, int arrive, cudaStream_t stream);

// Launches `kern` with programmatic stream serialisation (see griddep_wait in ptx.cuh).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Same, in clusters of two CTAs along x (the grid's x extent even).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_pairs(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                    cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Kernel timeline ids (timeline.cuh); names in pf_timeline_kernel_name.
enum TimelineId : int {
  TL_RMSNORM = 1, TL_RMSNORM_REG = 2, TL_QK_ROPE_KV = 3, TL_RING_STORE = 4, TL_EMBED = 5,
  TL_LM_HEAD = 6, TL_DEQUANT = 7, TL_SET_INT = 8, TL_ARGMAX = 9, TL_WAIT_SELFTEST = 10,
  TL_LM_HEAD_Q1 = 11, TL_ATTENTION_F32 = 12, TL_ATTENTION_TC = 13, TL_ATTN_COMBINE = 14,
  TL_GEMM = 20,        // + epilogue (0 store, 1 residual, 2 SwiGLU) + 3 for the CTA-pair form
  TL_GEMM_SMALL = 30,  // + epilogue
  TL_GEMV = 40         // + epilogue
};
// Per translation unit: points its kernels' timeline buffer at `buf` (NULL: off).
cudaError_t timeline_set_kernels(unsigned long long* buf);
cudaError_t timeline_set_gemm_q(unsigned long long* buf);
cudaError_t timeline_set_gemm_small(unsigned long long* buf);
cudaError_t timeline_set_gemv(unsigned long long* buf);
cudaError_t timeline_set_attention(unsigned long long* buf);
cudaError_t timeline_set_attention_tc(unsigned long long* buf);

int device_sm_count();
// Tiled tensor map over a 16-bit (bf16 if `bf16`, else f16) array of `rank` dims
// (innermost first), 128-B swizzle, zero fill out of bounds.
bool encode_tmap_16(CUtensorMap* map, int bf16, int rank, const void* base, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box);
// Tiled 2-D tensor map over a row-major f32 (or f16) [outer, inner] array for TMA stores,
// swizzle 128 or 64 bytes (or 0 = none).
bool encode_tmap_out_2d(CUtensorMap* map, bool f32, const void* base, uint64_t inner, uint64_t outer,
                        uint32_t box_inner, uint32_t box_outer, int swizzle_bytes);
bool attention_tc_supported(const pf_config& c);
cudaError_t prepare_attention_tc_kernels();
cudaError_t launch_attention_tc(const AttnArgs& a, cudaStream_t stream);
cudaError_t prepare_gemm_kernels();
cudaError_t prepare_attention_kernels();

}  // namespace pf
