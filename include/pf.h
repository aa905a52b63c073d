/*
 * pf.h — C ABI of libpf: batched / chunked prefill through a dense Qwen3/Llama-style
 * decoder stack whose linear weights are 1-bit sign + f16 group scale ("Q1") or
 * INT4-affine, on one sm_103a GPU.
 *
 * The operation follows three pages:
 *   [P1] oxibonsai-kernels 0.1.1, src/gpu_backend/metal_prefill.rs
 *        (encode_layer_prefill: sections 1-7; encode_full_forward_prefill: tail)
 *   [P2] oxibonsai-kernels 0.1.0, src/gpu_backend/metal_full_layer.rs
 *        (GpuKvCache layout; encode_layer_into: the per-token twin)
 *   [P3] turbospark-runtime 0.3.0, src/families/llama/prefill.rs
 *        (prefill_chunk_real_llama_dense: chunk contract, micro-batching, checks)
 *
 * Conventions for every entry point:
 *  - Memory. The caller owns every buffer (packed weights, norm weights, KV cache,
 *    workspace, inputs, outputs); libpf keeps non-owning pointers only and performs
 *    no device allocation. "_dev" pointers are device memory of the current CUDA
 *    device, "_host" pointers host memory.
 *  - Errors. Arguments are validated before anything is launched; on failure the
 *    call returns a pf_status other than PF_OK, pf_last_error() describes it, and no
 *    state (KV position, buffers) has changed. CUDA launch errors return PF_ERR_CUDA.
 *  - Asynchrony. GPU work is enqueued on the given stream (a cudaStream_t passed as
 *    void*, NULL = legacy default stream) and is not waited for, except where a call
 *    says it synchronises. Kernels whose internal waits time out (a bounded wait on
 *    a barrier that never completed) record PF_ERR_DEVICE_TIMEOUT in a device status
 *    word; pf_session_sync() / pf_status_read() report it.
 *  - Constant operands. Packed weights and norm weights are read as constants: a
 *    kernel launched as a programmatic dependent of the previous kernel on the stream
 *    may read them before that kernel has finished. Write them with a copy (or with a
 *    kernel followed by a stream or event synchronisation), not with a kernel enqueued
 *    directly before the call that reads them. Activations, caches and positions are
 *    read only after every earlier kernel on the stream has completed.
 *  - Thread safety. Calls on distinct sessions may run concurrently; one session is
 *    used by one host thread at a time. pf_last_error() is thread-local.
 */
#ifndef PF_H_
#define PF_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------ status codes */
/* Mirrors the error cases of [P1] encode_full_forward_prefill (short buffers, layer
 * count) and [P3] prefill_chunk_real_llama_dense (empty chunk, non-sequential start,
 * token outside vocab, logits length). */
typedef enum {
  PF_OK = 0,
  PF_ERR_INVALID_ARG = 1,        /* NULL pointer, negative size, bad enum value */
  PF_ERR_SHAPE = 2,              /* dimensions the kernels do not support */
  PF_ERR_EMPTY_CHUNK = 3,        /* M == 0 ([P3] "empty chunk") */
  PF_ERR_NONSEQUENTIAL_START = 4,/* start_pos != KV position ([P3]) */
  PF_ERR_TOKEN_OUT_OF_VOCAB = 5, /* token < 0 or >= vocab ([P3]) */
  PF_ERR_KV_CAPACITY = 6,        /* start_pos + M > max_seq, or a paged block unassigned */
  PF_ERR_LOGITS = 7,             /* logits requested but no LM head / buffer */
  PF_ERR_UNSUPPORTED = 8,        /* a mode the library does not implement */
  PF_ERR_CUDA = 9,               /* a CUDA runtime call failed */
  PF_ERR_DEVICE_TIMEOUT = 10,    /* a kernel's bounded wait expired (see status word) */
  PF_ERR_WORKSPACE = 11          /* workspace too small / not initialised */
} pf_status;

typedef enum { PF_W_Q1_G128 = 0, PF_W_INT4_AFFINE_G128 = 1 } pf_wformat;
typedef enum { PF_KV_F32 = 0, PF_KV_BF16 = 1, PF_KV_F16 = 2 } pf_kvdtype;

/* Model configuration ([P1] LayerConfig + the tail's final_norm_eps / vocab). */
typedef struct {
  int32_t hidden;        /* H; multiple of 128 */
  int32_t intermediate;  /* I; multiple of 128 */
  int32_t n_q_heads;     /* nq */
  int32_t n_kv_heads;    /* nkv; divides nq */
  int32_t head_dim;      /* hd; 64 or 128 */
  int32_t n_layers;
  int32_t vocab;         /* 0 when the model has no embedding / LM head */
  float rope_theta;
  float eps;             /* RMSNorm eps of the layers (also the QK-norm eps) */
  float final_eps;       /* eps of the final norm */
  int32_t qk_norm;       /* 1: per-head RMSNorm of Q and K before RoPE */
  int32_t wfmt;          /* pf_wformat */
  int32_t kv_dtype;      /* pf_kvdtype */
  int32_t max_seq;       /* largest position + 1 (RoPE table); the linear cache's capacity */
  int32_t max_chunk;     /* largest micro-batch the workspace is sized for (<= 8192) */
  /* Ring / sink KV cache ([P3] batch-attention contract fields ring_capacity, sink_count):
   * 0 = linear cache of max_seq slots. R > 0 = a cache of R slots per (layer, kv head):
   * positions 0 .. S-1 (S = sink_count, 0 <= S < R) keep slots 0 .. S-1, a later position p
   * goes to slot S + (p - S) mod (R - S), and the query at p attends to the S sinks and the
   * R - S most recent positions up to p (RoPE stays at absolute positions). Needs a 16-bit
   * cache. */
  int32_t ring_capacity;
  int32_t sink_count;
  /* Paged KV cache (the "paged" KV layout the target names beside the contiguous one): 0 =
   * off. P > 0 = K and V each hold P blocks of PF_KV_BLOCK positions per (layer, kv head),
   * slots = PF_KV_BLOCK * P, and the session's block table (pf_session_set_block_table) maps
   * position block b = p / PF_KV_BLOCK to the physical block holding positions
   * b * PF_KV_BLOCK .. +PF_KV_BLOCK-1 (same block for every layer and head). Sessions given
   * the same K / V buffers and disjoint tables share one pool. Needs a 16-bit cache and no
   * ring. */
  int32_t kv_block_pool;
} pf_config;

#define PF_KV_BLOCK 128 /* positions per paged KV block: one attention key tile */

/* One layer's weights ([P1] LayerWeightRefs), all device pointers. Packed tensors
 * come from pf_pack_weights_host (gate_up with interleave_gate_up = 1). */
typedef struct {
  const float* attn_norm; /* [H] f32 */
  const void* qkv;        /* packed, N = (nq + 2 nkv) hd rows (Q|K|V, head-major), K = H */
  const float* q_norm;    /* [hd] f32, NULL when qk_norm == 0 */
  const float* k_norm;    /* [hd] f32, NULL when qk_norm == 0 */
  const void* o_proj;     /* packed, N = H, K = nq hd */
  const float* ffn_norm;  /* [H] f32 */
  const void* gate_up;    /* packed + interleaved, N = 2 I (gate rows then up rows), K = H */
  const void* down;       /* packed, N = H, K = I */
} pf_layer_weights;

/* Whole model. `layers` is a HOST array of n_layers entries. */
typedef struct {
  pf_config cfg;
  const pf_layer_weights* layers;
  const float* embed;      /* [vocab, H] f32 device, or NULL (hidden-input use only) */
  const float* final_norm; /* [H] f32 device, or NULL */
  const void* lm_head;     /* packed, N = vocab, K = H, or NULL */
} pf_model;

typedef struct pf_session pf_session; /* opaque */

/* ------------------------------------------------------------------ misc */
const char* pf_last_error(void);      /* thread-local, never NULL */
const char* pf_status_name(int status);
int32_t pf_abi_version(void);         /* bumps on any ABI change (2: ring fields, 3: kv_block_pool,
                                        4: split-KV counters in the attention scratch,
                                        pf_streamk_plan_host) */

/* ------------------------------------------------------------------ packing
 * Canonical host formats (the pages name "Q1 block bytes" and an "AoS -> SoA"
 * conversion at upload, [P2] build_cached_weights, without the block layout):
 *  Q1:   codes = sign bits uint8 [N, K/8]; bit j (LSB first) of byte b of row n is
 *        weight k = 8b + j; a set bit means +scale. scales = f16 bits [N, K/128].
 *  INT4: codes uint8 [N, K/2]; low nibble of byte b is k = 2b, high nibble k = 2b+1;
 *        w = scale * (q - zero); scales, zeros = f16 bits [N, K/128].
 * The device layout (tiles of 256 rows x 128 weights, scales beside their bits, sign
 * bits / nibbles permuted for the dequantiser) is private to libpf; only its size
 * is public. With interleave_gate_up = 1 (N = 2I, I % 128 == 0), each 128-row tile
 * holds 64 gate rows followed by the 64 matching up rows, so one GEMM tile sees
 * both inputs of SwiGLU. Rows are padded to a multiple of 256 with zero scale.
 * Pure host code; safe without a GPU.
 */
size_t pf_packed_bytes(int32_t wfmt, int64_t N, int64_t K);
pf_status pf_pack_weights_host(int32_t wfmt, const uint8_t* codes_host,
                               const uint16_t* scales_f16_host,
                               const uint16_t* zeros_f16_host /* NULL for Q1 */,
                               int64_t N, int64_t K, int32_t interleave_gate_up,
                               void* dst_host, size_t dst_bytes);

/* ------------------------------------------------------------------ sizes */
size_t pf_kv_bytes(const pf_config* cfg);        /* bytes of ONE of K / V:
                                                    n_layers*nkv*slots*hd*elem, slots =
                                                    ring_capacity (ring), PF_KV_BLOCK *
                                                    kv_block_pool (paged) or max_seq */
size_t pf_workspace_bytes(const pf_config* cfg); /* activations for max_chunk rows,
                                                    RoPE table, status words */
/* Validates a configuration; PF_OK or the reason it is not supported. Host only. */
pf_status pf_config_check(const pf_config* cfg);
/* The argument checks pf_prefill_chunk / pf_prefill_hidden run before any launch, in
 * the order of [P3] prefill_chunk_real_llama_dense (empty chunk, sequential start,
 * vocabulary), then KV capacity and the head: tokens_host may be NULL (hidden input);
 * kv_position is the session's current position; want_logits / has_head say whether
 * logits are requested and whether the model has a final norm + LM head. Host only. */
pf_status pf_validate_chunk(const pf_config* cfg, int32_t kv_position,
                            const int32_t* tokens_host, int32_t M, int32_t start_pos,
                            int32_t want_logits, int32_t has_head);

/* ------------------------------------------------------------------ sessions
 * A session binds a model, a KV cache (K and V buffers of pf_kv_bytes each, layout
 * [n_layers][nkv][slots][hd] of the cache element type, [P2] GpuKvCache; slots = max_seq
 * positions, or ring_capacity ring slots) and a workspace. Creation computes the RoPE table cos/sin(p * theta^(-2i/hd)) on the
 * host in double precision ([P1] PrefillBuffers cos_buf/sin_buf are host-made too),
 * copies it into the workspace and clears the status words; it synchronises the
 * stream. The KV position starts at 0. The model struct and its layer array are
 * copied; the device buffers they point to must outlive the session.
 */
pf_status pf_session_create(const pf_model* model, void* k_cache_dev, void* v_cache_dev,
                            void* workspace_dev, size_t workspace_bytes, void* stream,
                            pf_session** out);
pf_status pf_session_destroy(pf_session* s);
int32_t pf_session_position(const pf_session* s); /* -1 for NULL */
/* Sets the KV position (e.g. 0 to reuse the cache for a new prompt, or the length of a
 * cache the caller filled itself). Slots at or beyond the new position are stale. */
pf_status pf_session_set_position(pf_session* s, int32_t position);
/* 1: record each chunk's launches once per (M, buffers) as a CUDA graph and replay it
 * (default); 0: launch kernels directly. */
pf_status pf_session_set_graphs(pf_session* s, int32_t enable);
/* Synchronises the stream, then reads and clears the session's device status word. */
pf_status pf_session_sync(pf_session* s, void* stream);

/* Per-kernel timing, the CUDA analogue of the pages' per-layer / per-phase profiling
 * ([P2] OXIBONSAI_PROFILE, [P3] phase counters). While enabled, chunks run without graph
 * replay and every kernel launch is bracketed by CUDA events on its stream;
 * pf_session_profile_read synchronises the stream and returns, per kernel class, the
 * summed device milliseconds and the launch count since the previous read (arrays of
 * PF_K_COUNT entries), then clears them. */
typedef enum {
  PF_K_RMSNORM = 0, PF_K_GEMM_QKV = 1, PF_K_QK_ROPE_KV = 2, PF_K_ATTENTION = 3,
  PF_K_GEMM_O = 4, PF_K_GEMM_GATE_UP = 5, PF_K_GEMM_DOWN = 6, PF_K_EMBED = 7,
  PF_K_LM_HEAD = 8, PF_K_OTHER = 9, PF_K_COUNT = 10
} pf_kernel_class;
pf_status pf_session_set_profile(pf_session* s, int32_t enable);
pf_status pf_session_profile_read(pf_session* s, void* stream, double* ms_out,
                                  int64_t* launches_out);
/* Paged caches: sets the session's block table from a HOST array of
 * ceil(max_seq / PF_KV_BLOCK) entries; entry b is the physical block (0 .. kv_block_pool-1)
 * of positions b * PF_KV_BLOCK .. +PF_KV_BLOCK-1, or -1 while unassigned. Assigned entries
 * must be distinct. A chunk whose positions reach an unassigned block is refused
 * (PF_ERR_KV_CAPACITY) before any launch. Copied to the workspace synchronously: call with
 * none of the session's work in flight. New sessions start with every entry unassigned.
 * Errors: PF_ERR_UNSUPPORTED (not a paged configuration), PF_ERR_SHAPE (wrong count, entry
 * out of range, repeated block), PF_ERR_CUDA. */
pf_status pf_session_set_block_table(pf_session* s, const int32_t* table_host, int32_t n_entries);

/* Number of libpf kernels enqueued by this session so far (graph replays count every
 * kernel node they run). */
int64_t pf_session_kernel_launches(const pf_session* s);

/* Kernel timeline, per CTA: the CUDA analogue of the GPU start / end stamps the pages take
 * per command buffer ([P2] OXIBONSAI_PROFILE_GPU, GPUStartTime / GPUEndTime). While a buffer
 * is set, each CTA of every libpf kernel (graph replays included, any session or op) appends
 * one record when its first thread leaves the kernel:
 *   buffer[0]              records appended so far (may exceed `capacity`: those are dropped)
 *   buffer[1]              capacity (written here)
 *   buffer[4 + 4 i + 0]    %globaltimer (ns) when the CTA's first thread started
 *   buffer[4 + 4 i + 1]    %globaltimer (ns) when it left the kernel
 *   buffer[4 + 4 i + 2]    kernel id << 48 | SM id << 32 | linear CTA index (low 32 bits)
 * `buffer`: DEVICE memory of 4 + 4 * capacity uint64 words, owned by the caller; its first
 * word is zeroed here. NULL stops recording. Synchronous: call with no libpf work in flight.
 * Errors: PF_ERR_INVALID_ARG (capacity <= 0 with a buffer), PF_ERR_CUDA. */
pf_status pf_timeline_set(uint64_t* buffer, int64_t capacity);
/* Name of a timeline kernel id ("gemm_pair_swiglu", "attention_tc", ...); NULL if unknown. */
const char* pf_timeline_kernel_name(int32_t id);

/* ------------------------------------------------------------------ the path
 * pf_prefill_chunk — [P3] prefill_chunk(tokens, start_position, logits): embeds M
 * token ids (HOST array, checked against vocab on the host before any launch), runs
 * them through every layer at positions start_pos .. start_pos+M-1 in micro-batches
 * of at most max_chunk rows ([P3] MAX_PREFILL_BATCH), and, if logits_dev != NULL,
 * writes the f32 logits [vocab] of the LAST position ([P1] tail: final RMSNorm of the
 * last row + LM head). Requires start_pos == pf_session_position ([P3] sequential
 * start) and start_pos + M <= max_seq. On success the KV position advances by M.
 */
pf_status pf_prefill_chunk(pf_session* s, const int32_t* tokens_host, int32_t M,
                           int32_t start_pos, float* logits_dev, void* stream);

/* Same, from f32 hidden rows x_dev [M, H] (updated in place to the last layer's
 * output, [P1] hidden_buf is updated in place by the residual GEMMs). M may exceed
 * max_chunk; rows are processed in micro-batches. */
pf_status pf_prefill_hidden(pf_session* s, float* x_dev, int32_t M, int32_t start_pos,
                            float* logits_dev, void* stream);

/* One layer ([P1] encode_layer_prefill, sections 1-7) on x_dev [M, H] (in place),
 * writing the layer's KV slots start_pos .. start_pos+M-1. Does NOT check or move the
 * session's KV position (the caller sequences layers); M <= max_chunk. */
pf_status pf_layer_forward(pf_session* s, int32_t layer, float* x_dev, int32_t M,
                           int32_t start_pos, void* stream);

/* Same as pf_prefill_chunk with the token ids already in device memory (int32 [M]).
 * Every host-side check runs except the vocabulary check, which the embedding kernel
 * performs instead: an id outside [0, vocab) gets a zero row and records
 * PF_ERR_TOKEN_OUT_OF_VOCAB in the session status word (read by pf_session_sync); the
 * KV position still advances by M in that case. */
pf_status pf_prefill_chunk_dev(pf_session* s, const int32_t* tokens_dev, int32_t M,
                               int32_t start_pos, float* logits_dev, void* stream);

/* One decode step ([P2] encode_layer_into for every layer, then the decode tail: final
 * norm + LM head): the token at *token_dev (device int32, e.g. the previous step's argmax)
 * at the session's KV position, which advances by one; logits_dev [vocab] f32 receives its
 * logits. Same kernels as a one-token chunk (the projections on the GEMV path); the recorded
 * graph of M = 1 is reused from step to step. Errors as pf_prefill_chunk_dev (PF_ERR_LOGITS when the
 * model has no LM head or logits_dev is NULL). */
pf_status pf_decode_step(pf_session* s, const int32_t* token_dev, float* logits_dev, void* stream);

/* Greedy decode step ([P1] encode_full_forward_prefill, greedy decoding: the argmax of the
 * logits taken on the GPU so that one token id, not the logits, is the step's result):
 * pf_decode_step on *token_in_dev, then the index of the largest logit (lowest index on
 * ties) written to *token_out_dev (device int32; may be token_in_dev). Consecutive calls
 * can chain tokens without a host round trip. Errors as pf_decode_step. */
pf_status pf_decode_step_greedy(pf_session* s, const int32_t* token_in_dev, int32_t* token_out_dev,
                                float* logits_dev, void* stream);

/* Speculative-verify prefill ([P1] encode_full_forward_prefill_verify): the M device token
 * ids at start_pos through every layer as one micro-batch (1 <= M <= max_chunk), then the
 * final RMSNorm and the LM head on EVERY position and the argmax of each position's logits.
 * logits_all_dev: f32 [M][vocab] (row t = logits after token t); ids_dev: int32 [M], the
 * greedy next token after each position (lowest index on ties). The KV position advances
 * by M. Needs an LM head and vocab % 8 == 0; PF_ERR_SHAPE for M > max_chunk. */
pf_status pf_prefill_verify(pf_session* s, const int32_t* tokens_dev, int32_t M, int32_t start_pos,
                            float* logits_all_dev, int32_t* ids_dev, void* stream);

/* End to end from host memory: copies tokens_host to the device, runs
 * pf_prefill_chunk, copies the last position's logits into logits_host [vocab]
 * (may be NULL) and synchronises the stream. */
pf_status pf_prefill_tokens_host(pf_session* s, const int32_t* tokens_host, int32_t M,
                                 int32_t start_pos, float* logits_host, void* stream);

/* ------------------------------------------------------------------ single steps
 * Each step of the path as its own call, for step-level parity checks. They launch
 * the same kernels the session uses. status_dev (int32, device) receives
 * PF_ERR_DEVICE_TIMEOUT if a bounded wait expires; it may be NULL for kernels
 * without waits. None of them synchronises.
 */
/* RMSNorm rows ([P1] dispatch_batched_rmsnorm): y = x * w / sqrt(mean(x^2) + eps),
 * x f32 [M, H] -> y f16 [M, H] (the GEMM operand type). */
pf_status pf_op_rmsnorm(const float* x_dev, const float* w_dev, float eps, int32_t M,
                        int32_t H, uint16_t* y_f16_dev, void* stream);
/* Dequantise a packed tensor to f16 [N, K] row-major (bit-exact check of unpacking):
 * Q1 -> +-scale; INT4 -> f16(f16(q - z) * s) evaluated in f16 arithmetic. */
pf_status pf_op_dequant(int32_t wfmt, const void* packed_dev, int64_t N, int64_t K,
                        uint16_t* w_f16_dev, void* stream);
/* Quantised GEMM out[m, n] (+)= sum_k a[m, k] w[n, k] on the tensor cores.
 * a: f16 [M, K] row-major; out 16-B aligned; epilogue: 0 = store f32 out[M, N] (ld = N),
 * 1 = residual add into f32 out[M, N] (out += a W^T), 2 = SwiGLU of an interleaved
 * gate_up weight: out f16 [M, N/2] = silu(gate) * up (N = 2I, I % 128 == 0).
 * The 128 x 256 output tiles' k-blocks are shared out evenly over at most max_ctas
 * persistent CTAs (0 = 160; never more than the SM count; 1..160 accepted). With
 * epilogue 1 every CTA adds its share of a tile into out; with epilogues 0 and 2 a tile
 * split between CTAs is summed through scratch_dev (device, 16-B aligned, at least
 * pf_gemm_scratch_bytes(M, N, max_ctas) bytes, owned by the caller, required for every
 * epilogue): its trailing per-tile counters must be zero before the first call, and each
 * call that completes leaves them zero; after PF_ERR_DEVICE_TIMEOUT zero them again.
 * Calls sharing one scratch must not overlap in time (same stream, or ordered).
 * The kernel depends on M: M > 64 the persistent tcgen05 GEMM described above; 16 < M <= 64
 * the same partition with the weight rows as the MMA's M side; M <= 16 a warp-level MMA
 * GEMV that ignores max_ctas and the scratch (residual and store forms add with f32
 * atomics, the store form after zeroing out). The results agree to the GEMM tolerances:
 * all three use f16 operands with f32 accumulation. */
size_t pf_gemm_scratch_bytes(int32_t M, int32_t N, int32_t max_ctas);
pf_status pf_op_gemm(int32_t wfmt, int32_t epilogue, const uint16_t* a_f16_dev,
                     const void* packed_dev, int32_t M, int32_t N, int32_t K, void* out_dev,
                     int32_t max_ctas, void* scratch_dev, size_t scratch_bytes,
                     int32_t* status_dev, void* stream);
/* The same GEMM for callers that may not allocate device memory (a plug-in whose host
 * owns all device memory, or a service that cannot risk the device synchronisation an
 * allocation may cause): no scratch argument; the split-tile partials and counters live in
 * one fixed 4 MiB + 64 KiB array inside the library, which every GPU that loads the library
 * keeps until the process exits. The pages have no counterpart of this call. It runs at
 * most 16 CTAs (slower than pf_op_gemm on large shapes) and rejects with PF_ERR_SHAPE an
 * output of more than 16384 tiles of 128 x 256. Each call looks the array's device address
 * up (cudaGetSymbolAddress) on the current device; the first call on a device may load the
 * library's device code and should come before any stream capture. Each call clears the
 * tile counters it uses on `stream`. Every call on a device
 * shares the array: calls that overlap on the GPU (other streams, other threads) race and
 * corrupt each other's results. Allocates nothing; arguments otherwise as pf_op_gemm. */
pf_status pf_op_gemm_static_scratch(int32_t wfmt, int32_t epilogue, const uint16_t* a_f16_dev,
                                    const void* packed_dev, int32_t M, int32_t N, int32_t K,
                                    void* out_dev, int32_t* status_dev, void* stream);
/* Host view of the stream-K partition the quantised GEMMs run (for tests and tools; no GPU
 * work): n_mt x n_nt output tiles of kbt k-blocks cut into `ctas` contiguous ranges, the last
 * late_units of them late_kb k-blocks shorter (0, 0: even ranges; the GEMM's own launches
 * set these for the layer projections on CTA pairs). Fills begins[0 .. ctas] (k-block where
 * each unit's range starts, begins[ctas] = the total) and, per unit, up to max_segs segments
 * in the order the unit runs them as (tile, first k-block within the tile, k-blocks, scratch
 * slot) in segs[unit][max_segs][4] (tile = -1 past the unit's last segment); when owners is
 * not NULL, owners[i] = the unit whose range holds k-block w_query[i]. Returns PF_ERR_SHAPE
 * for sizes out of range (any count < 1, ctas > the total, a unit with more than max_segs
 * segments). */
pf_status pf_streamk_plan_host(int32_t n_mt, int32_t n_nt, int32_t kbt, int32_t ctas, int32_t late_units,
                               int32_t late_kb, int64_t* begins, int32_t* segs, int32_t max_segs,
                               const int64_t* w_query, int32_t n_query, int32_t* owners);
/* Fused per-head QK RMSNorm + RoPE + KV store ([P1] section 3 fused_qk_norm /
 * fused_qk_rope / fused_kv_store; [P2] dispatch_fused_qk_norm_rope): from qkv f32
 * [M, (nq+2nkv) hd], writes q_dev [M, nq, hd] (bf16 when kv_dtype is bf16, else f16)
 * and the K (post-RoPE) / V slots of `layer` at positions start_pos.. in the caches.
 * rope_dev: table from pf_rope_table_host ([max_seq][hd/2] of (cos, sin) f32). Linear
 * caches only (PF_ERR_UNSUPPORTED for a ring configuration). */
pf_status pf_op_qk_norm_rope_kv(const pf_config* cfg, const float* qkv_dev,
                                const float* q_norm_dev, const float* k_norm_dev,
                                const float* rope_dev, int32_t layer, int32_t start_pos,
                                int32_t M, void* q_dev, void* k_cache_dev,
                                void* v_cache_dev, void* stream);
/* Causal GQA attention ([P1] section 3 scores/softmax/weighted sum, batched; [P3]
 * encode_attention_decode_batch): query rows at positions start_pos.., keys 0..pos of
 * `layer`'s cache; out f16 [M, nq hd]. Linear caches only (a ring configuration returns
 * PF_ERR_UNSUPPORTED: its keys come from the session's chunk buffers). */
pf_status pf_op_attention(const pf_config* cfg, const void* q_dev, const void* k_cache_dev,
                          const void* v_cache_dev, int32_t layer, int32_t start_pos,
                          int32_t M, uint16_t* out_f16_dev, void* stream);
/* The same with the keys cut into n_split contiguous parts (1..64), one CTA each, whose
 * unnormalised partial results (O sums, running max and sum per row) go to scratch_dev
 * (device, 16-B aligned, caller-owned, at least pf_attention_scratch_bytes(cfg, M, n_split)
 * bytes: a counter per kv head, which the call zeroes first, then the partials) and are
 * merged by a second kernel, or for M <= 2 by the part that completes each kv head's count:
 * the split-KV form the sessions use when a chunk's CTAs fill less than half of the GPU
 * (decode, small chunks). 16-bit linear caches only; the same result as pf_op_attention up
 * to the order of the f32 additions. */
size_t pf_attention_scratch_bytes(const pf_config* cfg, int32_t M, int32_t n_split);
pf_status pf_op_attention_split(const pf_config* cfg, const void* q_dev, const void* k_cache_dev,
                                const void* v_cache_dev, int32_t layer, int32_t start_pos,
                                int32_t M, int32_t n_split, void* scratch_dev, size_t scratch_bytes,
                                uint16_t* out_f16_dev, void* stream);
/* Embedding rows ([P3] encode_embed_any, scale 1.0): x[t] = E[tokens[t]] (device ids).
 * An id outside [0, vocab) yields a zero row and PF_ERR_TOKEN_OUT_OF_VOCAB in
 * *status_dev (if not NULL). */
pf_status pf_op_embed(const float* embed_dev, const int32_t* tokens_dev, int32_t M,
                      int32_t H, int32_t vocab, float* x_dev, int32_t* status_dev,
                      void* stream);
/* Tail ([P1] rmsnorm_weighted_v2 + dispatch_gemv_q1): logits[v] = W_lm . rmsnorm(x_row)
 * for one f32 row x_row_dev [H]; logits f32 [vocab]. */
pf_status pf_op_lm_head(int32_t wfmt, const float* x_row_dev, const float* norm_w_dev,
                        float eps, const void* packed_dev, int32_t vocab, int32_t H,
                        float* logits_dev, void* stream);
/* Greedy argmax of each row ([P1] dispatch_argmax, one 1024-thread group per row):
 * out_dev[r] = index of the largest of x_dev[r * ld .. r * ld + n - 1] (f32), lowest index
 * on ties, NaN never chosen (a row without a number gives 0). rows >= 1, n >= 1, ld >= n. */
pf_status pf_op_argmax(const float* x_dev, int32_t rows, int32_t n, int64_t ld, int32_t* out_dev,
                       void* stream);
/* Host RoPE table [max_seq][hd/2][2] = (cos, sin)(p * theta^(-2i/hd)), computed in
 * double and rounded to f32. */
pf_status pf_rope_table_host(float theta, int32_t head_dim, int32_t max_seq, float* dst_host);
/* Reads (and clears) a device status word written by the single-step kernels;
 * synchronises the stream. */
pf_status pf_status_read(int32_t* status_dev, void* stream);
/* Failure-detection self-test: one CTA waits, bounded by limit_ns (1 us .. 10 s), on an
 * mbarrier that gets its single arrival only if `arrive` is non-zero. Without it the wait
 * gives up and records PF_ERR_DEVICE_TIMEOUT in *status_dev — the path every pipelined
 * kernel takes when a stage never completes. Nothing faults or hangs. */
pf_status pf_selftest_bounded_wait(int32_t* status_dev, int64_t limit_ns, int32_t arrive,
                                   void* stream);

#ifdef __cplusplus
}
#endif
#endif /* PF_H_ */
