"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the CPU oracle.

This module only DRAWS numbers. It holds none of the method's arithmetic (no
dequantisation, no normalisation, no attention): both the oracle and the GPU
path consume exactly these arrays, in the canonical host formats the C ABI's
packer accepts (`include/pf.h`, `pf_pack_weights_host`).

Canonical formats (the reading of the pages' "Q1 block bytes" / "AoS->SoA"
weight upload in oxibonsai-kernels metal_full_layer.rs, `FullForwardLayerParams`
and `build_cached_weights`, which do not print the block layout):

* Q1 (1-bit sign + f16 scale per 128-weight group): ``bits`` uint8 [N, K/8],
  bit j (LSB first) of byte b of row n is weight k = 8*b + j; a set bit is the
  positive sign. ``scales`` float16 [N, K/128]; group g covers k in [128g, 128g+128).
* INT4-affine: ``codes`` uint8 [N, K/2]; the low nibble of byte b is weight
  k = 2b, the high nibble k = 2b+1. ``scales`` and ``zeros`` float16 [N, K/128].

Every tensor is drawn from its own PCG64 stream keyed by (seed, tensor id), so a
single layer of a 36-layer stack can be regenerated without drawing the others.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional

import numpy as np

GROUP = 128  # weights per scale group (all K in the workloads are multiples of it)

Q1 = "q1"
INT4 = "int4"

KV_F32 = "f32"
KV_BF16 = "bf16"
KV_F16 = "f16"


@dataclasses.dataclass(frozen=True)
class ModelShape:
    """Shape and hyper-parameters of a dense Qwen3/Llama-style decoder stack."""

    hidden: int
    intermediate: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    n_layers: int
    vocab: int
    rope_theta: float
    eps: float
    final_eps: float
    qk_norm: bool
    wfmt: str
    kv_dtype: str
    max_seq: int

    @property
    def qkv_rows(self) -> int:
        return (self.n_q_heads + 2 * self.n_kv_heads) * self.head_dim


# Workloads: the five configurations' sizes and value distributions.
TINY = ModelShape(hidden=256, intermediate=768, n_q_heads=4, n_kv_heads=2, head_dim=64,
                  n_layers=1, vocab=0, rope_theta=1e6, eps=1e-6, final_eps=1e-6,
                  qk_norm=True, wfmt=Q1, kv_dtype=KV_F32, max_seq=64)
QWEN3_8B_LAYER = ModelShape(hidden=4096, intermediate=12288, n_q_heads=32, n_kv_heads=8,
                            head_dim=128, n_layers=1, vocab=0, rope_theta=1e6, eps=1e-6,
                            final_eps=1e-6, qk_norm=True, wfmt=Q1, kv_dtype=KV_BF16,
                            max_seq=4096)
QWEN3_8B_LAYER_LONG = dataclasses.replace(QWEN3_8B_LAYER, max_seq=8192)
QWEN3_8B_STACK = dataclasses.replace(QWEN3_8B_LAYER, n_layers=36, vocab=151936, max_seq=2048)
LLAMA3_8B_INT4_LAYER = ModelShape(hidden=4096, intermediate=14336, n_q_heads=32, n_kv_heads=8,
                                  head_dim=128, n_layers=1, vocab=0, rope_theta=5e5, eps=1e-5,
                                  final_eps=1e-5, qk_norm=False, wfmt=INT4, kv_dtype=KV_BF16,
                                  max_seq=8704)

# tensor ids for the per-tensor streams
_T_HIDDEN, _T_TOKENS, _T_EMBED, _T_FINAL_NORM, _T_LM_HEAD, _T_KV = 1, 2, 3, 4, 5, 6
_T_LAYER_BASE = 100
_LAYER_TENSORS = ("attn_norm", "q_norm", "k_norm", "ffn_norm", "qkv", "o", "gate_up", "down")


def rng_for(seed: int, *key: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64([seed, *key]))


def q1_weight(rng: np.random.Generator, n: int, k: int) -> Dict[str, np.ndarray]:
    """Sign bits Bernoulli(0.5); f16 scales |N(0, 0.02)| per 128-group."""
    assert k % GROUP == 0
    bits = rng.integers(0, 256, size=(n, k // 8), dtype=np.uint8)
    scales = np.abs(rng.normal(0.0, 0.02, size=(n, k // GROUP))).astype(np.float16)
    return {"fmt": Q1, "n": n, "k": k, "bits": bits, "scales": scales}


def int4_weight(rng: np.random.Generator, n: int, k: int) -> Dict[str, np.ndarray]:
    """uint4 codes uniform 0..15; f16 scale |N(0, 0.01)|; f16 zero-point U(0, 15)."""
    assert k % GROUP == 0
    codes = rng.integers(0, 256, size=(n, k // 2), dtype=np.uint8)  # two uniform nibbles
    scales = np.abs(rng.normal(0.0, 0.01, size=(n, k // GROUP))).astype(np.float16)
    zeros = rng.uniform(0.0, 15.0, size=(n, k // GROUP)).astype(np.float16)
    return {"fmt": INT4, "n": n, "k": k, "codes": codes, "scales": scales, "zeros": zeros}


def quant_weight(fmt: str, rng: np.random.Generator, n: int, k: int) -> Dict[str, np.ndarray]:
    return q1_weight(rng, n, k) if fmt == Q1 else int4_weight(rng, n, k)


def norm_weight(rng: np.random.Generator, n: int) -> np.ndarray:
    """Norm weights 1 + N(0, 0.1), f32."""
    return (1.0 + rng.normal(0.0, 0.1, size=n)).astype(np.float32)


def layer_weights(shape: ModelShape, layer: int, seed: int = 0) -> Dict[str, object]:
    """All tensors of one decoder layer in canonical host formats.

    ``gate_up`` is one quantised tensor of 2*I rows: the I gate rows first, then
    the I up rows (the concatenation order of the pages' fused gate+up upload).
    """
    H, I, hd = shape.hidden, shape.intermediate, shape.head_dim
    base = _T_LAYER_BASE + 16 * layer
    r = {name: rng_for(seed, base + i) for i, name in enumerate(_LAYER_TENSORS)}
    w: Dict[str, object] = {
        "attn_norm": norm_weight(r["attn_norm"], H),
        "ffn_norm": norm_weight(r["ffn_norm"], H),
        "q_norm": norm_weight(r["q_norm"], hd) if shape.qk_norm else None,
        "k_norm": norm_weight(r["k_norm"], hd) if shape.qk_norm else None,
        "qkv": quant_weight(shape.wfmt, r["qkv"], shape.qkv_rows, H),
        "o": quant_weight(shape.wfmt, r["o"], H, shape.n_q_heads * hd),
        "gate_up": quant_weight(shape.wfmt, r["gate_up"], 2 * I, H),
        "down": quant_weight(shape.wfmt, r["down"], H, I),
    }
    return w


def hidden_input(m: int, hidden: int, seed: int = 0, stream: int = 0) -> np.ndarray:
    """Input hidden rows f32 N(0, 1)."""
    return rng_for(seed, _T_HIDDEN, stream).standard_normal((m, hidden), dtype=np.float32)


def tokens(m: int, vocab: int, seed: int = 0, stream: int = 0) -> np.ndarray:
    """Token ids uniform over [0, vocab), int32."""
    return rng_for(seed, _T_TOKENS, stream).integers(0, vocab, size=m, dtype=np.int32)


def embedding(shape: ModelShape, seed: int = 0) -> np.ndarray:
    """Embedding table f32 [vocab, hidden] ~ N(0, 0.02)."""
    g = rng_for(seed, _T_EMBED)
    e = g.standard_normal((shape.vocab, shape.hidden), dtype=np.float32)
    e *= np.float32(0.02)
    return e


def final_norm(shape: ModelShape, seed: int = 0) -> np.ndarray:
    return norm_weight(rng_for(seed, _T_FINAL_NORM), shape.hidden)


def lm_head(shape: ModelShape, seed: int = 0) -> Dict[str, np.ndarray]:
    return quant_weight(shape.wfmt, rng_for(seed, _T_LM_HEAD), shape.vocab, shape.hidden)


def kv_prefill_bf16_bits(n_layers: int, n_kv: int, positions: int, head_dim: int,
                         seed: int = 0) -> Dict[str, np.ndarray]:
    """K and V for already-filled cache positions: N(0, 1) values given as bf16 bit
    patterns (uint16) [n_layers, n_kv, positions, head_dim]. The bf16 values are
    the top 16 bits of f32 normal draws (truncation is part of the draw; the
    values are then exact bf16)."""
    g = rng_for(seed, _T_KV)
    out = {}
    for name in ("k", "v"):
        f = g.standard_normal((n_layers, n_kv, positions, head_dim), dtype=np.float32)
        out[name] = (f.view(np.uint32) >> 16).astype(np.uint16)
    return out


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def model_inputs(shape: ModelShape, seed: int = 0, with_head: Optional[bool] = None):
    """Everything a stack needs: per-layer weights, and (when the shape has a vocab)
    the embedding, final norm and LM head."""
    with_head = shape.vocab > 0 if with_head is None else with_head
    layers = [layer_weights(shape, l, seed) for l in range(shape.n_layers)]
    extra = {}
    if with_head:
        extra["embed"] = embedding(shape, seed)
        extra["final_norm"] = final_norm(shape, seed)
        extra["lm_head"] = lm_head(shape, seed)
    return layers, extra
