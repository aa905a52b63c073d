"""CPU oracle for batched / chunked prefill through a dense Q1 / INT4-affine stack.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this module: only
``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg may.
It shares no code with the CUDA library (no kernels, headers, tables or helpers);
the only thing both sides use is the seeded input generator
(``quantized_transformer_prefill_q1_gb300.synth``), which draws numbers and does
none of the method's arithmetic.

Precision: activations are stored as float32 between steps (the pages keep every
batched buffer in f32: oxibonsai-kernels metal_prefill.rs, ``PrefillBuffers``);
every step is evaluated in float64 (dot products, means, softmax sums). The KV
cache stores values rounded to the cache's element type (f32, bf16 or f16) —
storing into a typed cache is part of the method (the pages' cache is f16:
metal_full_layer.rs, ``GpuKvCache``; the workloads here use f32 and bf16).

The method, as the pages state it: a decoder layer of seven steps (pre-attention RMSNorm,
fused QKV projection, per-head QK-norm + RoPE + KV store and causal GQA attention, O
projection with the residual add, FFN RMSNorm, gate+up with SwiGLU, down projection with
the residual add; oxibonsai-kernels 0.1.1 metal_prefill.rs, the prefill layer encoder,
sections 1-7), a tail of final RMSNorm and LM head on the last position (the same page's
full-forward prefill), and chunks of a prompt at consecutive start positions over one KV
cache (turbospark-runtime 0.3.0 families/llama/prefill.rs, the dense chunk function). The
per-token form below is the decode layer of oxibonsai-kernels 0.1.0 metal_full_layer.rs,
written independently of the batched form.

Where the pages are silent, each function states in words the reading it takes.

Parity status: every function below is pinned by ``tests/test_oracle_pins.py``
except the composition of a full stack's logits, which has no worked example on
the pages ("parity unpinned" beyond the invariants one-shot = chunked = decode,
causality and per-step pins).
"""
from __future__ import annotations

import math
from typing import Dict, List, Optional, Sequence

import numpy as np

GROUP = 128

# --------------------------------------------------------------------------------------
# dequantisation
# --------------------------------------------------------------------------------------


def dequant_q1(bits: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """Q1 weight -> float64 [N, K].

    Reading taken (the pages name "Q1 block bytes" only — metal_full_layer.rs,
    ``FullForwardLayerParams``): bit j (LSB first) of byte b of row n is k = 8b+j;
    a set bit means +s, a clear bit -s; s is the f16 scale of group k // 128.
    """
    n = bits.shape[0]
    signs = np.unpackbits(bits, axis=1, bitorder="little").astype(np.float64) * 2.0 - 1.0
    k = signs.shape[1]
    s = np.repeat(scales.astype(np.float64), GROUP, axis=1)
    assert s.shape == (n, k)
    return signs * s


def dequant_int4(codes: np.ndarray, scales: np.ndarray, zeros: np.ndarray) -> np.ndarray:
    """INT4-affine weight -> float64 [N, K]: w = s * (q - z) per 128-group.

    Reading taken (turbospark-runtime prefill.rs only names an "INT4-affine" M-row
    GEMM): q is the uint4 code (low nibble = even k), s and z the group's f16
    scale and zero point. Evaluated exactly in float64.
    """
    n, half = codes.shape
    q = np.empty((n, 2 * half), dtype=np.float64)
    q[:, 0::2] = codes & 0x0F
    q[:, 1::2] = codes >> 4
    s = np.repeat(scales.astype(np.float64), GROUP, axis=1)
    z = np.repeat(zeros.astype(np.float64), GROUP, axis=1)
    return s * (q - z)


def dequant(w: Dict) -> np.ndarray:
    if w["fmt"] == "q1":
        return dequant_q1(w["bits"], w["scales"])
    return dequant_int4(w["codes"], w["scales"], w["zeros"])


# --------------------------------------------------------------------------------------
# element steps
# --------------------------------------------------------------------------------------


def rmsnorm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """y_i = w_i * x_i / sqrt(mean_j(x_j^2) + eps) over the last axis, in float64.

    Reading taken (the kernel bodies behind ``dispatch_batched_rmsnorm`` /
    ``rmsnorm_weighted_v2`` in metal_prefill.rs are not printed): the weight
    multiplies as-is (no implicit 1 + w).
    """
    x64 = np.asarray(x, dtype=np.float64)
    ms = np.mean(x64 * x64, axis=-1, keepdims=True)
    return x64 / np.sqrt(ms + eps) * np.asarray(w, dtype=np.float64)


def rope_inv_freq(head_dim: int, theta: float) -> np.ndarray:
    """inv_freq_i = theta^(-2i/head_dim), i = 0 .. head_dim/2 - 1 (the standard RoPE ladder;
    the pages only build per-position cos / sin tables)."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * i / head_dim)


def rope_angles(positions: np.ndarray, head_dim: int, theta: float) -> np.ndarray:
    """angle[p, i] = p * inv_freq_i, float64 [len(positions), head_dim/2]."""
    return np.asarray(positions, dtype=np.float64)[:, None] * rope_inv_freq(head_dim, theta)[None, :]


def apply_rope(v: np.ndarray, angles: np.ndarray) -> np.ndarray:
    """Rotate-half RoPE (the pages do not state the pairing; reading: pair i is (i, i + hd/2)).

    v: [..., T, heads, hd]; angles: [T, hd/2]. out_a = a cos - b sin,
    out_b = b cos + a sin, where a = v[..., :hd/2], b = v[..., hd/2:].
    The pages precompute cos/sin per position on the host (metal_prefill.rs,
    ``PrefillBuffers`` cos_buf / sin_buf) and apply them per token
    (``fused_qk_rope`` in ``encode_layer_prefill`` section 3).
    """
    v64 = np.asarray(v, dtype=np.float64)
    half = v64.shape[-1] // 2
    c = np.cos(angles)[:, None, :]
    s = np.sin(angles)[:, None, :]
    a, b = v64[..., :half], v64[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def silu(g: np.ndarray) -> np.ndarray:
    g64 = np.asarray(g, dtype=np.float64)
    return g64 / (1.0 + np.exp(-g64))


def round_to_cache(x: np.ndarray, kv_dtype: str) -> np.ndarray:
    """Value stored in a KV cache of element type kv_dtype, returned as float32.

    Round-to-nearest-even from float32 (the storing rule is not printed; reading: IEEE
    round to nearest even). bf16 keeps the top 16 bits
    of the float32 pattern after adding the RNE rounding bias.
    """
    x32 = np.asarray(x, dtype=np.float32)
    if kv_dtype == "f32":
        return x32.copy()
    if kv_dtype == "f16":
        return x32.astype(np.float16).astype(np.float32)
    if kv_dtype == "bf16":
        u = x32.view(np.uint32).astype(np.uint64)
        lsb = (u >> 16) & 1
        r = ((u + 0x7FFF + lsb) >> 16) & 0xFFFF
        return (r.astype(np.uint32) << 16).view(np.float32)
    raise ValueError(kv_dtype)


def causal_gqa_attention(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                         start: int, window: Optional[int] = None, sinks: int = 0) -> np.ndarray:
    """Causal GQA attention for query rows at positions start .. start+T-1.

    q: [T, nq, hd] (float64 or float32); k_cache, v_cache: [nkv, >=start+T, hd] holding
    the cache for this layer by absolute position. Query at position p sees keys 0..p
    inclusive (``seq_len = pos + 1`` in metal_prefill.rs
    ``encode_layer_prefill`` section 3). Scores use 1/sqrt(hd) (``inv_sqrt_hd``); q head h
    reads kv head h // (nq/nkv) (``heads_per_group``: consecutive q heads share a kv head).
    Softmax subtracts the
    row max and is evaluated in float64. Returns float64 [T, nq, hd].

    With a ring cache (turbospark-runtime prefill.rs ``BatchAttentionInputContract``:
    ``ring_capacity``, ``sink_count``; the contract only names them, and the reading taken
    is the usual sliding window with attention sinks) the query at p sees only the first
    ``sinks`` positions and the ``window`` most recent positions up to p.
    """
    T, nq, hd = q.shape
    nkv = k_cache.shape[0]
    G = nq // nkv
    L = start + T
    out = np.empty((T, nq, hd), dtype=np.float64)
    key_pos = np.arange(L)
    qry_pos = start + np.arange(T)
    mask = key_pos[None, :] > qry_pos[:, None]  # True where the key is in the future
    if window is not None:  # older than the window and not a sink
        mask |= (key_pos[None, :] <= qry_pos[:, None] - window) & (key_pos[None, :] >= sinks)
    scale = 1.0 / math.sqrt(hd)
    for h in range(nq):
        kvh = h // G
        K = k_cache[kvh, :L].astype(np.float64)
        V = v_cache[kvh, :L].astype(np.float64)
        s = (q[:, h, :].astype(np.float64) @ K.T) * scale
        s[mask] = -np.inf
        s -= s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=1, keepdims=True)
        out[:, h, :] = p @ V
    return out


# --------------------------------------------------------------------------------------
# model state
# --------------------------------------------------------------------------------------


class OracleModel:
    """Dequantised float64 weights of a stack plus an f32-valued KV cache.

    ``layers`` holds, per layer, the canonical tensors from the input generator.
    The cache is [n_layers, nkv, max_seq, hd] per K and V (metal_full_layer.rs
    ``GpuKvCache``: layer-major, then kv head, then position, then head dim),
    holding values already rounded to the cache's element type.
    """

    def __init__(self, shape, layers: Sequence[Dict], extra: Optional[Dict] = None,
                 cache_dequant: bool = True, ring_capacity: Optional[int] = None,
                 sink_count: int = 0):
        if ring_capacity is not None and not 0 <= sink_count < ring_capacity:
            raise ValueError("ring cache: need 0 <= sink_count < ring_capacity")
        self.ring_capacity = ring_capacity
        self.sink_count = sink_count
        self.shape = shape
        self.raw_layers = list(layers)
        self.cache_dequant = cache_dequant
        self._dq: Dict[int, Dict] = {}
        self.extra = extra or {}
        self._lm_w = None
        s = shape
        self.k_cache = np.full((s.n_layers, s.n_kv_heads, s.max_seq, s.head_dim), np.nan, np.float32)
        self.v_cache = np.full_like(self.k_cache, np.nan)
        if ring_capacity is not None:  # the physical ring the per-token restatement uses
            self.ring_k = np.full((s.n_layers, s.n_kv_heads, ring_capacity, s.head_dim), np.nan, np.float32)
            self.ring_v = np.full_like(self.ring_k, np.nan)
            self.ring_pos = np.full((s.n_layers, ring_capacity), -1, np.int64)
        self.position = 0

    @property
    def layers(self):
        return _LayerView(self)

    def layer(self, l: int) -> Dict:
        """Canonical tensors of layer l plus their float64 dequantisation."""
        if l in self._dq:
            return self._dq[l]
        w = self.raw_layers[l]
        d = dict(w)
        for name in ("qkv", "o", "gate_up", "down"):
            d[name + "_w"] = dequant(w[name])
        if self.cache_dequant:
            self._dq[l] = d
        return d

    @property
    def lm_w(self):
        if self._lm_w is None:
            self._lm_w = dequant(self.extra["lm_head"])
        return self._lm_w

    def reset(self):
        self.k_cache[:] = np.nan
        self.v_cache[:] = np.nan
        if self.ring_capacity is not None:
            self.ring_k[:] = np.nan
            self.ring_v[:] = np.nan
            self.ring_pos[:] = -1
        self.position = 0

    # ---- one layer, a chunk of T rows (metal_prefill.rs encode_layer_prefill) --------
    def layer_forward(self, l: int, x: np.ndarray, start: int) -> np.ndarray:
        s = self.shape
        w = self.layer(l)
        T = x.shape[0]
        nq, nkv, hd = s.n_q_heads, s.n_kv_heads, s.head_dim
        x = np.asarray(x, dtype=np.float32)
        if start + T > s.max_seq:
            raise ValueError("chunk exceeds KV capacity")
        # 1. pre-attention RMSNorm
        y = rmsnorm(x, w["attn_norm"], s.eps).astype(np.float32)
        # 2. fused QKV projection: rows Q | K | V, head-major (the offsets the page uses)
        qkv = (y.astype(np.float64) @ w["qkv_w"].T).astype(np.float32)
        q = qkv[:, : nq * hd].reshape(T, nq, hd)
        k = qkv[:, nq * hd: (nq + nkv) * hd].reshape(T, nkv, hd)
        v = qkv[:, (nq + nkv) * hd:].reshape(T, nkv, hd)
        # 3a. per-head QK RMSNorm over head_dim, same eps as the layer (the page passes the
        #     layer eps to its fused QK-norm)
        if s.qk_norm:
            q = rmsnorm(q, w["q_norm"], s.eps).astype(np.float32)
            k = rmsnorm(k, w["k_norm"], s.eps).astype(np.float32)
        # 3b. RoPE at absolute positions start .. start+T-1
        ang = rope_angles(np.arange(start, start + T), hd, s.rope_theta)
        q = apply_rope(q, ang).astype(np.float32)
        k = apply_rope(k, ang).astype(np.float32)
        # 3c. KV store at [l, kvh, pos, :] — K after RoPE, V as projected
        self.k_cache[l, :, start:start + T, :] = round_to_cache(k, s.kv_dtype).transpose(1, 0, 2)
        self.v_cache[l, :, start:start + T, :] = round_to_cache(v, s.kv_dtype).transpose(1, 0, 2)
        # 3d. causal GQA attention over cache positions 0 .. pos (a ring cache: the sinks and
        #     the last ring_capacity - sink_count positions)
        window = None if self.ring_capacity is None else self.ring_capacity - self.sink_count
        o = causal_gqa_attention(q, self.k_cache[l], self.v_cache[l], start, window,
                                 self.sink_count).astype(np.float32)
        # 4. O projection + residual
        x = (x.astype(np.float64) + o.reshape(T, nq * hd).astype(np.float64) @ w["o_w"].T).astype(np.float32)
        # 5. FFN RMSNorm
        y = rmsnorm(x, w["ffn_norm"], s.eps).astype(np.float32)
        # 6. gate_up (gate rows first, then up rows) + SwiGLU = silu(gate) * up
        gu = y.astype(np.float64) @ w["gate_up_w"].T
        I = s.intermediate
        act = (silu(gu[:, :I]) * gu[:, I:]).astype(np.float32)
        # 7. down projection + residual
        x = (x.astype(np.float64) + act.astype(np.float64) @ w["down_w"].T).astype(np.float32)
        return x

    # ---- the ring cache's slots (sinks first, then a cycle over the remaining slots) -----
    def ring_slot(self, p: int) -> int:
        """Slot of absolute position p in a ring cache of ring_capacity slots: the first
        sink_count positions keep slots 0 .. sink_count-1; later positions cycle through
        the remaining ring_capacity - sink_count slots."""
        R, S = self.ring_capacity, self.sink_count
        return p if p < S else S + (p - S) % (R - S)

    def ring_cache(self, l: int):
        """Layer l's K and V as a ring cache of ring_capacity slots would hold them after
        positions 0 .. position-1 were stored in order (a slot keeps the last position
        stored into it; slots never written keep NaN). Returns ([nkv, R, hd], [nkv, R, hd])."""
        R = self.ring_capacity
        s = self.shape
        k = np.full((s.n_kv_heads, R, s.head_dim), np.nan, np.float32)
        v = np.full_like(k, np.nan)
        for p in range(self.position):
            k[:, self.ring_slot(p)] = self.k_cache[l, :, p]
            v[:, self.ring_slot(p)] = self.v_cache[l, :, p]
        return k, v

    # ---- tail: final norm on the last row + LM head (encode_full_forward_prefill) -------
    def head(self, x_last: np.ndarray) -> np.ndarray:
        y = rmsnorm(x_last, self.extra["final_norm"], self.shape.final_eps).astype(np.float32)
        return (self.lm_w @ y.astype(np.float64)).astype(np.float32)

    def head_all(self, x_rows: np.ndarray) -> np.ndarray:
        """The verify tail (oxibonsai-kernels metal_prefill.rs
        ``encode_full_forward_prefill_verify``): final norm and LM head on every row, the
        same per-row arithmetic as ``head``. Returns f32 logits [rows, vocab]."""
        return np.stack([self.head(r) for r in np.asarray(x_rows, dtype=np.float32)])

    def prefill_verify(self, tokens: np.ndarray):
        """One chunk of token ids through every layer, then the logits of every position
        and each position's greedy next token."""
        x, _ = self.forward_chunk(self.embed(tokens), self.position, False)
        logits = self.head_all(x)
        return logits, argmax_first(logits)

    def embed(self, tokens: np.ndarray) -> np.ndarray:
        """x[t] = E[token_t] with no sqrt(hidden) scale (turbospark-runtime
        prefill.rs embeds each token at scale 1.0)."""
        tokens = np.asarray(tokens)
        if tokens.size and (tokens.min() < 0 or tokens.max() >= self.shape.vocab):
            raise ValueError("token outside vocab")
        return self.extra["embed"][tokens].astype(np.float32)

    # ---- one micro-batch through every layer -------------------------------------------
    def forward_chunk(self, x: np.ndarray, start: int, want_logits: bool):
        if x.shape[0] == 0:
            raise ValueError("empty chunk")
        if start != self.position:
            raise ValueError("non-sequential chunk start")
        for l in range(self.shape.n_layers):
            x = self.layer_forward(l, x, start)
        self.position = start + x.shape[0]
        logits = self.head(x[-1]) if want_logits else None
        return x, logits

    def prefill(self, x_or_tokens: np.ndarray, chunk_sizes: Sequence[int], from_tokens: bool,
                want_logits: bool):
        """Run a prompt as consecutive chunks (turbospark-runtime prefill.rs: micro-batches
        at consecutive start positions, logits only after the last). Returns the final
        hidden rows of every position (stacked) and the last position's logits."""
        assert sum(chunk_sizes) == len(x_or_tokens)
        outs = []
        logits = None
        off = 0
        for i, m in enumerate(chunk_sizes):
            piece = x_or_tokens[off: off + m]
            x = self.embed(piece) if from_tokens else np.asarray(piece, dtype=np.float32)
            last = i == len(chunk_sizes) - 1
            xo, lg = self.forward_chunk(x, self.position, want_logits and last)
            outs.append(xo)
            logits = lg if lg is not None else logits
            off += m
        return np.concatenate(outs, axis=0), logits


    def prefill_layer_major(self, x_or_tokens: np.ndarray, chunk_sizes: Sequence[int],
                            from_tokens: bool, want_logits: bool):
        """Same result as ``prefill`` with the loops swapped: every chunk passes layer l
        before any chunk enters layer l+1. Chunk c's layer-l step reads only the layer-l
        cache written by chunks <= c, so the arithmetic is identical; each layer's
        weights are dequantised once (used for the 36-layer stack)."""
        assert sum(chunk_sizes) == len(x_or_tokens)
        if self.position != 0:
            raise ValueError("layer-major prefill starts from an empty cache")
        starts = np.concatenate([[0], np.cumsum(chunk_sizes)[:-1]]).astype(int)
        xs = []
        for st, m in zip(starts, chunk_sizes):
            piece = x_or_tokens[st: st + m]
            xs.append(self.embed(piece) if from_tokens else np.asarray(piece, dtype=np.float32))
        for l in range(self.shape.n_layers):
            for c, st in enumerate(starts):
                xs[c] = self.layer_forward(l, xs[c], int(st))
            self._dq.pop(l, None)
        self.position = int(sum(chunk_sizes))
        x = np.concatenate(xs, axis=0)
        return x, (self.head(x[-1]) if want_logits else None)


class _LayerView:
    def __init__(self, model: "OracleModel"):
        self._m = model

    def __getitem__(self, l: int) -> Dict:
        return self._m.layer(l)

    def __len__(self) -> int:
        return len(self._m.raw_layers)


# --------------------------------------------------------------------------------------
# per-token decode restatement (metal_full_layer.rs encode_layer_into): one token at a
# time, per-head loops, explicit score vector — written independently of the batched
# form above so that "one-shot = chunked = token-by-token" checks two formulations.
# --------------------------------------------------------------------------------------


def decode_token(model: OracleModel, l: int, x_row: np.ndarray, pos: int) -> np.ndarray:
    s = model.shape
    w = model.layers[l]
    nq, nkv, hd = s.n_q_heads, s.n_kv_heads, s.head_dim
    G = nq // nkv
    half = hd // 2
    x_row = np.asarray(x_row, dtype=np.float32)
    y = rmsnorm(x_row, w["attn_norm"], s.eps).astype(np.float32)
    qkv = (w["qkv_w"] @ y.astype(np.float64)).astype(np.float32)
    heads = [qkv[i * hd:(i + 1) * hd] for i in range(nq + 2 * nkv)]
    inv = [float(s.rope_theta) ** (-2.0 * i / hd) for i in range(half)]
    rotated = []
    for j in range(nq + nkv):  # q heads then k heads
        hv = heads[j]
        if s.qk_norm:
            hv = rmsnorm(hv, w["q_norm"] if j < nq else w["k_norm"], s.eps).astype(np.float32)
        hv = hv.astype(np.float64)
        r = np.empty(hd)
        for i in range(half):
            c, sn = math.cos(pos * inv[i]), math.sin(pos * inv[i])
            r[i] = hv[i] * c - hv[i + half] * sn
            r[i + half] = hv[i + half] * c + hv[i] * sn
        rotated.append(r.astype(np.float32))
    for g in range(nkv):
        model.k_cache[l, g, pos] = round_to_cache(rotated[nq + g], s.kv_dtype)
        model.v_cache[l, g, pos] = round_to_cache(heads[nq + nkv + g], s.kv_dtype)
    if model.ring_capacity is None:
        keys = [(model.k_cache[l, g_], model.v_cache[l, g_]) for g_ in range(nkv)]
        n_keys = pos + 1
    else:
        # a physical ring of ring_capacity slots: store at the position's slot, then attend
        # over every slot in use (the sinks and the most recent positions)
        slot = model.ring_slot(pos)
        for g in range(nkv):
            model.ring_k[l, g, slot] = model.k_cache[l, g, pos]
            model.ring_v[l, g, slot] = model.v_cache[l, g, pos]
        model.ring_pos[l, slot] = pos
        used = np.flatnonzero(model.ring_pos[l] >= 0)
        keys = [(model.ring_k[l, g_, used], model.ring_v[l, g_, used]) for g_ in range(nkv)]
        n_keys = used.size
    o = np.empty(nq * hd, dtype=np.float32)
    for h in range(nq):
        g = h // G
        kh, vh = keys[g]
        qh = rotated[h].astype(np.float64)
        sc = np.array([float(qh @ kh[j].astype(np.float64)) / math.sqrt(hd) for j in range(n_keys)])
        e = np.exp(sc - sc.max())
        p = e / e.sum()
        acc = np.zeros(hd)
        for j in range(n_keys):
            acc += p[j] * vh[j].astype(np.float64)
        o[h * hd:(h + 1) * hd] = acc.astype(np.float32)
    x_row = (x_row.astype(np.float64) + w["o_w"] @ o.astype(np.float64)).astype(np.float32)
    y = rmsnorm(x_row, w["ffn_norm"], s.eps).astype(np.float32)
    I = s.intermediate
    g_ = w["gate_up_w"][:I] @ y.astype(np.float64)
    u_ = w["gate_up_w"][I:] @ y.astype(np.float64)
    act = (g_ / (1.0 + np.exp(-g_)) * u_).astype(np.float32)
    return (x_row.astype(np.float64) + w["down_w"] @ act.astype(np.float64)).astype(np.float32)


def decode_prompt(model: OracleModel, x: np.ndarray, start: int = 0) -> np.ndarray:
    """Token-by-token pass over hidden rows x at positions start.. (all layers)."""
    outs = []
    for t in range(x.shape[0]):
        r = np.asarray(x[t], dtype=np.float32)
        for l in range(model.shape.n_layers):
            r = decode_token(model, l, r, start + t)
        outs.append(r)
    model.position = start + x.shape[0]
    return np.stack(outs)


def argmax_first(logits: np.ndarray) -> np.ndarray:
    """Greedy selection (oxibonsai-kernels metal_prefill.rs: the argmax of the logits on
    the GPU, one token id per position). Per row of the last axis: the index of the largest
    value; ties go to the lowest index (the pages do not print the kernel; reading: the
    first maximum);
    NaN is never chosen and a row without a number gives 0. Written out row by row."""
    x = np.asarray(logits, dtype=np.float64)
    rows = x.reshape(-1, x.shape[-1])
    out = np.zeros(rows.shape[0], dtype=np.int64)
    for i, r in enumerate(rows):
        best, idx = -math.inf, -1
        for j, v in enumerate(r):
            if v > best or (v == best and idx < 0):
                best, idx = v, j
        out[i] = max(idx, 0)
    return out.reshape(x.shape[:-1])


def rel_l2(a: np.ndarray, b: np.ndarray) -> float:
    a64 = np.asarray(a, dtype=np.float64)
    b64 = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a64 - b64) / max(np.linalg.norm(b64), 1e-300))
