"""ctypes binding of libpf (include/pf.h): the same entry-point names, argument
marshalling only. Every step of the path runs in libpf's CUDA kernels; torch is used
for device memory and streams. If libpf.so is missing, importing the library raises —
there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
from typing import Dict, List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpf.so")

PF_OK = 0
STATUS = {
    0: "PF_OK", 1: "PF_ERR_INVALID_ARG", 2: "PF_ERR_SHAPE", 3: "PF_ERR_EMPTY_CHUNK",
    4: "PF_ERR_NONSEQUENTIAL_START", 5: "PF_ERR_TOKEN_OUT_OF_VOCAB", 6: "PF_ERR_KV_CAPACITY",
    7: "PF_ERR_LOGITS", 8: "PF_ERR_UNSUPPORTED", 9: "PF_ERR_CUDA", 10: "PF_ERR_DEVICE_TIMEOUT",
    11: "PF_ERR_WORKSPACE",
}
W_Q1, W_INT4 = 0, 1
KV_F32, KV_BF16, KV_F16 = 0, 1, 2
EPI_STORE_F32, EPI_RESID_ADD, EPI_SWIGLU = 0, 1, 2
KERNEL_CLASSES = ("rmsnorm", "gemm_qkv", "qk_rope_kv", "attention", "gemm_o", "gemm_gate_up",
                  "gemm_down", "embed", "lm_head", "other")
_WFMT = {"q1": W_Q1, "int4": W_INT4}
_KVDT = {"f32": KV_F32, "bf16": KV_BF16, "f16": KV_F16}


class PfError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"{STATUS.get(status, status)}: {msg}")
        self.status = status


class pf_config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("intermediate", ctypes.c_int32),
                ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("n_layers", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("rope_theta", ctypes.c_float),
                ("eps", ctypes.c_float), ("final_eps", ctypes.c_float),
                ("qk_norm", ctypes.c_int32), ("wfmt", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("max_seq", ctypes.c_int32),
                ("max_chunk", ctypes.c_int32), ("ring_capacity", ctypes.c_int32),
                ("sink_count", ctypes.c_int32), ("kv_block_pool", ctypes.c_int32)]

KV_BLOCK = 128  # PF_KV_BLOCK: positions per paged KV block


class pf_layer_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in
                ("attn_norm", "qkv", "q_norm", "k_norm", "o_proj", "ffn_norm", "gate_up", "down")]


class pf_model(ctypes.Structure):
    _fields_ = [("cfg", pf_config), ("layers", ctypes.POINTER(pf_layer_weights)),
                ("embed", ctypes.c_void_p), ("final_norm", ctypes.c_void_p),
                ("lm_head", ctypes.c_void_p)]


_VP, _I32, _I64, _SZ, _F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_float
_SIGS = {
    "pf_last_error": ([], ctypes.c_char_p),
    "pf_status_name": ([ctypes.c_int], ctypes.c_char_p),
    "pf_abi_version": ([], _I32),
    "pf_packed_bytes": ([_I32, _I64, _I64], _SZ),
    "pf_pack_weights_host": ([_I32, _VP, _VP, _VP, _I64, _I64, _I32, _VP, _SZ], _I32),
    "pf_kv_bytes": ([ctypes.POINTER(pf_config)], _SZ),
    "pf_workspace_bytes": ([ctypes.POINTER(pf_config)], _SZ),
    "pf_config_check": ([ctypes.POINTER(pf_config)], _I32),
    "pf_validate_chunk": ([ctypes.POINTER(pf_config), _I32, _VP, _I32, _I32, _I32, _I32], _I32),
    "pf_session_create": ([ctypes.POINTER(pf_model), _VP, _VP, _VP, _SZ, _VP,
                           ctypes.POINTER(_VP)], _I32),
    "pf_session_destroy": ([_VP], _I32),
    "pf_session_position": ([_VP], _I32),
    "pf_session_set_position": ([_VP, _I32], _I32),
    "pf_session_set_graphs": ([_VP, _I32], _I32),
    "pf_session_set_block_table": ([_VP, _VP, _I32], _I32),
    "pf_session_sync": ([_VP, _VP], _I32),
    "pf_prefill_chunk": ([_VP, _VP, _I32, _I32, _VP, _VP], _I32),
    "pf_prefill_chunk_dev": ([_VP, _VP, _I32, _I32, _VP, _VP], _I32),
    "pf_decode_step": ([_VP, _VP, _VP, _VP], _I32),
    "pf_decode_step_greedy": ([_VP, _VP, _VP, _VP, _VP], _I32),
    "pf_prefill_verify": ([_VP, _VP, _I32, _I32, _VP, _VP, _VP], _I32),
    "pf_session_set_profile": ([_VP, _I32], _I32),
    "pf_session_profile_read": ([_VP, _VP, ctypes.POINTER(ctypes.c_double),
                                 ctypes.POINTER(ctypes.c_int64)], _I32),
    "pf_session_kernel_launches": ([_VP], ctypes.c_int64),
    "pf_timeline_set": ([_VP, ctypes.c_int64], _I32),
    "pf_timeline_kernel_name": ([_I32], ctypes.c_char_p),
    "pf_prefill_hidden": ([_VP, _VP, _I32, _I32, _VP, _VP], _I32),
    "pf_layer_forward": ([_VP, _I32, _VP, _I32, _I32, _VP], _I32),
    "pf_prefill_tokens_host": ([_VP, _VP, _I32, _I32, _VP, _VP], _I32),
    "pf_op_rmsnorm": ([_VP, _VP, _F, _I32, _I32, _VP, _VP], _I32),
    "pf_op_dequant": ([_I32, _VP, _I64, _I64, _VP, _VP], _I32),
    "pf_op_gemm": ([_I32, _I32, _VP, _VP, _I32, _I32, _I32, _VP, _I32, _VP, _SZ, _VP, _VP], _I32),
    "pf_gemm_scratch_bytes": ([_I32, _I32, _I32], _SZ),
    "pf_op_gemm_static_scratch": ([_I32, _I32, _VP, _VP, _I32, _I32, _I32, _VP, _VP, _VP], _I32),
    "pf_streamk_plan_host": ([_I32, _I32, _I32, _I32, _I32, _I32, _VP, _VP, _I32, _VP, _I32, _VP], _I32),
    "pf_op_qk_norm_rope_kv": ([ctypes.POINTER(pf_config), _VP, _VP, _VP, _VP, _I32, _I32, _I32,
                               _VP, _VP, _VP, _VP], _I32),
    "pf_op_attention": ([ctypes.POINTER(pf_config), _VP, _VP, _VP, _I32, _I32, _I32, _VP, _VP], _I32),
    "pf_attention_scratch_bytes": ([ctypes.POINTER(pf_config), _I32, _I32], _SZ),
    "pf_op_attention_split": ([ctypes.POINTER(pf_config), _VP, _VP, _VP, _I32, _I32, _I32, _I32, _VP, _SZ,
                               _VP, _VP], _I32),
    "pf_op_embed": ([_VP, _VP, _I32, _I32, _I32, _VP, _VP, _VP], _I32),
    "pf_op_lm_head": ([_I32, _VP, _VP, _F, _VP, _I32, _I32, _VP, _VP], _I32),
    "pf_op_argmax": ([_VP, _I32, _I32, _I64, _VP, _VP], _I32),
    "pf_rope_table_host": ([_F, _I32, _I32, _VP], _I32),
    "pf_status_read": ([_VP, _VP], _I32),
    "pf_selftest_bounded_wait": ([_VP, _I64, _I32, _VP], _I32),
}

_lib = None


def lib() -> ctypes.CDLL:
    """Loads libpf.so (built by ``build.py``); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libpf.so not built ({LIB_PATH}); run __graft_entry__.build()")
        l = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGS.items():
            f = getattr(l, name)
            f.argtypes = args
            f.restype = res
        _lib = l
    return _lib


def header_symbols() -> List[str]:
    return list(_SIGS)


def check(status: int) -> None:
    if status != PF_OK:
        raise PfError(status, lib().pf_last_error().decode())


def _ptr(t) -> Optional[int]:
    """Device / host address of a torch tensor or numpy array (None passes NULL)."""
    if t is None:
        return None
    if isinstance(t, np.ndarray):
        assert t.flags["C_CONTIGUOUS"]
        return t.ctypes.data
    return t.data_ptr()


def _stream(stream=None) -> Optional[int]:
    if stream is not None:
        return stream
    import torch
    return torch.cuda.current_stream().cuda_stream


# ------------------------------------------------------------------ host-side calls
def make_config(shape, max_chunk: int, n_layers: Optional[int] = None, max_seq: Optional[int] = None,
                vocab: Optional[int] = None, ring_capacity: int = 0, sink_count: int = 0,
                kv_block_pool: int = 0) -> pf_config:
    return pf_config(hidden=shape.hidden, intermediate=shape.intermediate,
                     n_q_heads=shape.n_q_heads, n_kv_heads=shape.n_kv_heads,
                     head_dim=shape.head_dim,
                     n_layers=shape.n_layers if n_layers is None else n_layers,
                     vocab=shape.vocab if vocab is None else vocab,
                     rope_theta=shape.rope_theta, eps=shape.eps, final_eps=shape.final_eps,
                     qk_norm=int(shape.qk_norm), wfmt=_WFMT[shape.wfmt],
                     kv_dtype=_KVDT[shape.kv_dtype],
                     max_seq=shape.max_seq if max_seq is None else max_seq, max_chunk=max_chunk,
                     ring_capacity=ring_capacity, sink_count=sink_count, kv_block_pool=kv_block_pool)


def pf_packed_bytes(wfmt: int, n: int, k: int) -> int:
    return lib().pf_packed_bytes(wfmt, n, k)


def pf_pack_weights_host(w: Dict, interleave_gate_up: bool = False) -> np.ndarray:
    """Packs one canonical quantised tensor (see ``synth``) into libpf's device layout."""
    wfmt = _WFMT[w["fmt"]]
    n, k = w["n"], w["k"]
    nbytes = pf_packed_bytes(wfmt, n, k)
    out = np.empty(nbytes, np.uint8)
    codes = np.ascontiguousarray(w["bits"] if wfmt == W_Q1 else w["codes"])
    scales = np.ascontiguousarray(w["scales"]).view(np.uint16)
    zeros = None if wfmt == W_Q1 else np.ascontiguousarray(w["zeros"]).view(np.uint16)
    check(lib().pf_pack_weights_host(wfmt, _ptr(codes), _ptr(scales), _ptr(zeros), n, k,
                                     int(interleave_gate_up), _ptr(out), nbytes))
    return out


def pf_validate_chunk(cfg: pf_config, kv_position: int, tokens: Optional[np.ndarray], m: int,
                      start: int, want_logits: bool, has_head: bool) -> int:
    t = None if tokens is None else np.ascontiguousarray(tokens, dtype=np.int32)
    return lib().pf_validate_chunk(ctypes.byref(cfg), kv_position, _ptr(t), m, start,
                                   int(want_logits), int(has_head))


def pf_rope_table_host(theta: float, head_dim: int, max_seq: int) -> np.ndarray:
    out = np.empty((max_seq, head_dim // 2, 2), np.float32)
    check(lib().pf_rope_table_host(theta, head_dim, max_seq, _ptr(out)))
    return out


# ------------------------------------------------------------------ single steps (GPU)
def pf_op_rmsnorm(x, w, eps, y, stream=None):
    m, h = x.shape
    check(lib().pf_op_rmsnorm(_ptr(x), _ptr(w), eps, m, h, _ptr(y), _stream(stream)))


def pf_op_dequant(wfmt, packed, n, k, out, stream=None):
    check(lib().pf_op_dequant(wfmt, _ptr(packed), n, k, _ptr(out), _stream(stream)))


def pf_gemm_scratch_bytes(m, n, max_ctas=0):
    return lib().pf_gemm_scratch_bytes(m, n, max_ctas)


def gemm_scratch(m, n, max_ctas=0, device="cuda"):
    """Zeroed scratch (uint8 tensor) for pf_op_gemm on an M x N output."""
    import torch
    return torch.zeros(pf_gemm_scratch_bytes(m, n, max_ctas), dtype=torch.uint8, device=device)


def pf_op_gemm(wfmt, epilogue, a, packed, m, n, k, out, scratch, max_ctas=0, status=None,
               stream=None):
    check(lib().pf_op_gemm(wfmt, epilogue, _ptr(a), _ptr(packed), m, n, k, _ptr(out), max_ctas,
                           _ptr(scratch), scratch.numel() * scratch.element_size(), _ptr(status),
                           _stream(stream)))


def pf_op_gemm_static_scratch(wfmt, epilogue, a, packed, m, n, k, out, status=None, stream=None):
    """pf_op_gemm with the library's fixed scratch: for callers that may not allocate."""
    check(lib().pf_op_gemm_static_scratch(wfmt, epilogue, _ptr(a), _ptr(packed), m, n, k, _ptr(out),
                                          _ptr(status), _stream(stream)))


def pf_streamk_plan_host(n_mt, n_nt, kbt, ctas, late_units=0, late_kb=0, max_segs=8, w_query=None):
    """The GEMMs' stream-K partition on the host: (begins [ctas + 1], segments [ctas, max_segs, 4]
    as (tile, kb0, nkb, slot; -1 slot for a whole tile; tile -1 past the last), owners of
    w_query or None)."""
    begins = np.zeros(ctas + 1, np.int64)
    segs = np.zeros((ctas, max_segs, 4), np.int32)
    wq = None if w_query is None else np.ascontiguousarray(w_query, np.int64)
    owners = None if wq is None else np.zeros(len(wq), np.int32)
    check(lib().pf_streamk_plan_host(n_mt, n_nt, kbt, ctas, late_units, late_kb, _ptr(begins), _ptr(segs),
                                     max_segs, _ptr(wq), 0 if wq is None else len(wq), _ptr(owners)))
    return begins, segs, owners


def pf_op_qk_norm_rope_kv(cfg, qkv, qn, kn, rope, layer, start, m, q, kc, vc, stream=None):
    check(lib().pf_op_qk_norm_rope_kv(ctypes.byref(cfg), _ptr(qkv), _ptr(qn), _ptr(kn), _ptr(rope),
                                      layer, start, m, _ptr(q), _ptr(kc), _ptr(vc), _stream(stream)))


def pf_op_attention(cfg, q, kc, vc, layer, start, m, out, stream=None):
    check(lib().pf_op_attention(ctypes.byref(cfg), _ptr(q), _ptr(kc), _ptr(vc), layer, start, m,
                                _ptr(out), _stream(stream)))


def pf_attention_scratch_bytes(cfg, m, n_split):
    return lib().pf_attention_scratch_bytes(ctypes.byref(cfg), m, n_split)


def pf_op_attention_split(cfg, q, kc, vc, layer, start, m, n_split, scratch, out, stream=None):
    check(lib().pf_op_attention_split(ctypes.byref(cfg), _ptr(q), _ptr(kc), _ptr(vc), layer, start, m,
                                      n_split, _ptr(scratch), scratch.numel() * scratch.element_size(),
                                      _ptr(out), _stream(stream)))


def pf_op_argmax(x, rows, n, ld, out, stream=None):
    check(lib().pf_op_argmax(_ptr(x), rows, n, ld, _ptr(out), _stream(stream)))


def pf_op_embed(e, tokens, m, h, vocab, x, status=None, stream=None):
    check(lib().pf_op_embed(_ptr(e), _ptr(tokens), m, h, vocab, _ptr(x), _ptr(status),
                            _stream(stream)))


def pf_op_lm_head(wfmt, x_row, norm_w, eps, packed, vocab, h, logits, stream=None):
    check(lib().pf_op_lm_head(wfmt, _ptr(x_row), _ptr(norm_w), eps, _ptr(packed), vocab, h,
                              _ptr(logits), _stream(stream)))


def pf_status_read(status, stream=None):
    check(lib().pf_status_read(_ptr(status), _stream(stream)))


def pf_selftest_bounded_wait(status, limit_ns: int, arrive: bool, stream=None):
    check(lib().pf_selftest_bounded_wait(_ptr(status), limit_ns, int(arrive), _stream(stream)))


# ------------------------------------------------------------------ model + session
def pf_timeline_set(buffer, capacity: int) -> None:
    """Point every libpf kernel's per-CTA timeline at `buffer` (device int64/uint64 tensor
    of 4 + 4 * capacity words), or stop recording with None."""
    check(lib().pf_timeline_set(_ptr(buffer), int(capacity) if buffer is not None else 0))


def pf_timeline_kernel_name(kernel_id: int) -> Optional[str]:
    n = lib().pf_timeline_kernel_name(int(kernel_id))
    return n.decode() if n is not None else None


def timeline_records(buffer) -> np.ndarray:
    """The records of a timeline buffer as a structured array (start_ns, end_ns, kernel,
    sm, cta), sorted by start; records past the capacity were dropped by the device."""
    b = buffer.cpu().numpy().view(np.uint64)
    n = int(min(b[0], b[1]))
    r = b[4:4 + 4 * n].reshape(n, 4)
    out = np.zeros(n, dtype=[("start_ns", np.int64), ("end_ns", np.int64), ("kernel", np.int32),
                             ("sm", np.int32), ("cta", np.int64)])
    out["start_ns"] = r[:, 0].astype(np.int64)
    out["end_ns"] = r[:, 1].astype(np.int64)
    out["kernel"] = (r[:, 2] >> np.uint64(48)).astype(np.int32)
    out["sm"] = ((r[:, 2] >> np.uint64(32)) & np.uint64(0xffff)).astype(np.int32)
    out["cta"] = (r[:, 2] & np.uint64(0xffffffff)).astype(np.int64)
    return np.sort(out, order="start_ns", kind="stable")


class DeviceModel:
    """Uploads a stack's weights (packed once, on the host) into device memory owned by
    torch tensors and fills a ``pf_model`` pointing at them."""

    def __init__(self, shape, layers: Sequence[Dict], extra: Optional[Dict] = None,
                 max_chunk: int = 512, device: str = "cuda", max_seq: Optional[int] = None,
                 ring_capacity: int = 0, sink_count: int = 0, kv_block_pool: int = 0):
        import torch
        self.shape = shape
        self.keep: List = []
        extra = extra or {}

        def dev(a: np.ndarray):
            t = torch.from_numpy(np.ascontiguousarray(a)).to(device)
            self.keep.append(t)
            return t

        def packed(w, inter=False):
            return dev(pf_pack_weights_host(w, inter))

        n = len(layers)
        self.cfg = make_config(shape, max_chunk, n_layers=n, max_seq=max_seq,
                               vocab=shape.vocab if "lm_head" in extra else 0,
                               ring_capacity=ring_capacity, sink_count=sink_count,
                               kv_block_pool=kv_block_pool)
        self.layer_arr = (pf_layer_weights * n)()
        for i, w in enumerate(layers):
            lw = self.layer_arr[i]
            lw.attn_norm = _ptr(dev(w["attn_norm"]))
            lw.ffn_norm = _ptr(dev(w["ffn_norm"]))
            lw.q_norm = _ptr(dev(w["q_norm"])) if w["q_norm"] is not None else None
            lw.k_norm = _ptr(dev(w["k_norm"])) if w["k_norm"] is not None else None
            lw.qkv = _ptr(packed(w["qkv"]))
            lw.o_proj = _ptr(packed(w["o"]))
            lw.gate_up = _ptr(packed(w["gate_up"], True))
            lw.down = _ptr(packed(w["down"]))
        self.model = pf_model(cfg=self.cfg, layers=self.layer_arr)
        if "embed" in extra:
            self.model.embed = _ptr(dev(extra["embed"]))
        if "lm_head" in extra:
            self.model.final_norm = _ptr(dev(extra["final_norm"]))
            self.model.lm_head = _ptr(packed(extra["lm_head"]))


_KV_TORCH = {KV_F32: "float32", KV_BF16: "bfloat16", KV_F16: "float16"}


class Session:
    """A pf_session with its KV cache and workspace allocated by torch (caller-owned)."""

    def __init__(self, dm: DeviceModel, stream=None, kv_fill_bits: Optional[int] = None,
                 graphs: bool = True, kv=None, block_table: Optional[Sequence[int]] = None):
        """`kv`: an existing (k, v) pair to share (paged caches: one pool, disjoint block
        tables); `block_table`: a paged session's table (default: position block b in
        physical block b, when the pool has enough blocks)."""
        import torch
        self.dm = dm
        c = dm.cfg
        dt = getattr(torch, _KV_TORCH[c.kv_dtype])
        slots = c.ring_capacity if c.ring_capacity > 0 else (
            c.kv_block_pool * KV_BLOCK if c.kv_block_pool > 0 else c.max_seq)
        shape = (c.n_layers, c.n_kv_heads, slots, c.head_dim)
        if kv is not None:
            self.k, self.v = kv
        else:
            self.k = torch.empty(shape, dtype=dt, device="cuda")
            self.v = torch.empty(shape, dtype=dt, device="cuda")
        if kv_fill_bits is not None:  # sentinel bit pattern in every slot
            ib = torch.int32 if c.kv_dtype == KV_F32 else torch.int16
            self.k.view(ib).fill_(kv_fill_bits)
            self.v.view(ib).fill_(kv_fill_bits)
        check(lib().pf_config_check(ctypes.byref(c)))
        wsb = lib().pf_workspace_bytes(ctypes.byref(c))
        if wsb == 0:
            raise PfError(2, lib().pf_last_error().decode())
        self.ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
        h = ctypes.c_void_p()
        check(lib().pf_session_create(ctypes.byref(dm.model), _ptr(self.k), _ptr(self.v),
                                      _ptr(self.ws), wsb, _stream(stream), ctypes.byref(h)))
        self.h = h
        check(lib().pf_session_set_graphs(self.h, int(graphs)))
        if c.kv_block_pool > 0:
            n = -(-c.max_seq // KV_BLOCK)
            if block_table is None and c.kv_block_pool >= n:
                block_table = range(n)
            if block_table is not None:
                self.set_block_table(block_table)

    def set_block_table(self, table: Sequence[int]) -> None:
        t = np.ascontiguousarray(np.asarray(table, dtype=np.int32))
        check(lib().pf_session_set_block_table(self.h, _ptr(t), len(t)))

    @property
    def position(self) -> int:
        return lib().pf_session_position(self.h)

    def set_position(self, p: int) -> None:
        check(lib().pf_session_set_position(self.h, p))

    def set_graphs(self, on: bool) -> None:
        check(lib().pf_session_set_graphs(self.h, int(on)))

    def prefill_chunk(self, tokens: np.ndarray, start: int, logits=None, stream=None) -> None:
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        check(lib().pf_prefill_chunk(self.h, _ptr(t), len(t), start, _ptr(logits), _stream(stream)))

    def prefill_chunk_dev(self, tokens_dev, start: int, logits=None, stream=None) -> None:
        check(lib().pf_prefill_chunk_dev(self.h, _ptr(tokens_dev), tokens_dev.shape[0], start,
                                         _ptr(logits), _stream(stream)))

    def decode_step(self, token_dev, logits, stream=None) -> None:
        """One decode step: the token at token_dev (device int32) at the current position."""
        check(lib().pf_decode_step(self.h, _ptr(token_dev), _ptr(logits), _stream(stream)))

    def decode_step_greedy(self, token_in_dev, token_out_dev, logits, stream=None) -> None:
        """A decode step whose logits' argmax (device int32) is written to token_out_dev."""
        check(lib().pf_decode_step_greedy(self.h, _ptr(token_in_dev), _ptr(token_out_dev), _ptr(logits),
                                          _stream(stream)))

    def prefill_verify(self, tokens_dev, start: int, logits_all, ids, stream=None) -> None:
        """Prefill of tokens_dev, then logits [M, vocab] and their argmax [M] at every position."""
        check(lib().pf_prefill_verify(self.h, _ptr(tokens_dev), tokens_dev.shape[0], start, _ptr(logits_all),
                                      _ptr(ids), _stream(stream)))

    def set_profile(self, on: bool) -> None:
        check(lib().pf_session_set_profile(self.h, int(on)))

    def profile_read(self, stream=None) -> Dict[str, tuple]:
        """{kernel class: (summed ms, launches)} since the previous read."""
        ms = (ctypes.c_double * len(KERNEL_CLASSES))()
        n = (ctypes.c_int64 * len(KERNEL_CLASSES))()
        check(lib().pf_session_profile_read(self.h, _stream(stream), ms, n))
        return {name: (ms[i], n[i]) for i, name in enumerate(KERNEL_CLASSES)}

    @property
    def kernel_launches(self) -> int:
        return lib().pf_session_kernel_launches(self.h)

    def prefill_hidden(self, x, start: int, logits=None, stream=None) -> None:
        check(lib().pf_prefill_hidden(self.h, _ptr(x), x.shape[0], start, _ptr(logits),
                                      _stream(stream)))

    def layer_forward(self, layer: int, x, start: int, stream=None) -> None:
        check(lib().pf_layer_forward(self.h, layer, _ptr(x), x.shape[0], start, _stream(stream)))

    def prefill_tokens_host(self, tokens: np.ndarray, start: int, logits_host: Optional[np.ndarray],
                            stream=None) -> None:
        t = np.ascontiguousarray(tokens, dtype=np.int32)
        check(lib().pf_prefill_tokens_host(self.h, _ptr(t), len(t), start, _ptr(logits_host),
                                           _stream(stream)))

    def sync(self, stream=None) -> None:
        check(lib().pf_session_sync(self.h, _stream(stream)))

    def close(self) -> None:
        if getattr(self, "h", None):
            lib().pf_session_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
