"""Host-side checks of libpf that need no GPU: the library loads and exports every
symbol include/pf.h declares, the packer's layout round-trips, and the argument checks
return the statuses of the pages' error cases in their order."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

from quantized_transformer_prefill_q1_gb300 import pf, synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(pf.LIB_PATH):
        from quantized_transformer_prefill_q1_gb300 import build
        build.build()
    return pf.lib()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "pf.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pf_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 30
    for n in names:
        assert hasattr(lib, n), n
    out = subprocess.run(["nm", "-D", "--defined-only", pf.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r" T (pf_[a-z0-9_]+)", out))
    assert set(names) <= exported
    # the binding declares the same names
    assert set(pf.header_symbols()) == set(names)


def test_library_has_no_cuda_link_dependency(lib):
    out = subprocess.run(["ldd", pf.LIB_PATH], capture_output=True, text=True).stdout
    assert "libcuda.so" not in out and "libcudart" not in out


def _decode_q1(packed, n, k):
    """Reads libpf's Q1 device layout back into canonical LSB-first sign bits."""
    G = k // 128
    tiles = (n + 255) // 256
    ch = packed.reshape(tiles, G, 4608)
    bits = np.zeros((n, k), np.uint8)
    for t in range(tiles):
        for g in range(G):
            for h in range(2):
                words = ch[t, g, h * 2048:(h + 1) * 2048].view(np.uint32).reshape(256, 2)
                for b in range(2):
                    Z = words[:, b].astype(np.uint64)
                    for i in range(16):
                        neg_e = (Z >> np.uint64(15 - i)) & 1
                        neg_o = (Z >> np.uint64(31 - i)) & 1
                        k0 = 128 * g + 64 * h + 32 * b + 2 * i
                        rows = np.arange(256) + 256 * t
                        ok = rows < n
                        bits[rows[ok], k0] = 1 - neg_e[ok]
                        bits[rows[ok], k0 + 1] = 1 - neg_o[ok]
    scales = ch[:, :, 4096:4608].view(np.uint16).reshape(tiles, G, 256).transpose(0, 2, 1).reshape(tiles * 256, G)[:n]
    return np.packbits(bits, axis=1, bitorder="little"), scales


def test_q1_pack_layout_roundtrip(lib):
    n, k = 300, 384
    w = synth.q1_weight(synth.rng_for(21), n, k)
    packed = pf.pf_pack_weights_host(w)
    assert packed.size == pf.pf_packed_bytes(pf.W_Q1, n, k) == 2 * 3 * 4608
    bits, scales = _decode_q1(packed, n, k)
    np.testing.assert_array_equal(bits, w["bits"])
    np.testing.assert_array_equal(scales, w["scales"].view(np.uint16))
    # padding rows carry zero scales
    tail = packed.reshape(2, 3, 4608)[1, :, 4096:].view(np.uint16).reshape(3, 256)[:, n - 256:]
    assert np.all(tail == 0)


def test_int4_pack_layout_roundtrip(lib):
    n, k = 256, 256
    w = synth.int4_weight(synth.rng_for(22), n, k)
    packed = pf.pf_pack_weights_host(w).reshape(1, 2, 17408)
    for g in range(2):
        for h in range(2):
            words = packed[0, g, h * 8192:(h + 1) * 8192].view(np.uint32).reshape(256, 8)
            for wi in range(8):
                for p in range(4):
                    ke = 128 * g + 64 * h + 8 * wi + 2 * p
                    qe = (words[:, wi] >> (4 * p)) & 15
                    qo = (words[:, wi] >> (16 + 4 * p)) & 15
                    np.testing.assert_array_equal(qe, w["codes"][:, ke // 2] & 15)
                    np.testing.assert_array_equal(qo, w["codes"][:, ke // 2] >> 4)
        np.testing.assert_array_equal(packed[0, g, 16384:16896].view(np.uint16), w["scales"][:, g].view(np.uint16))
        np.testing.assert_array_equal(packed[0, g, 16896:].view(np.uint16), w["zeros"][:, g].view(np.uint16))


def test_pack_rejects_bad_arguments(lib):
    w = synth.q1_weight(synth.rng_for(23), 256, 256)
    out = np.empty(10, np.uint8)
    st = lib.pf_pack_weights_host(0, w["bits"].ctypes.data, w["scales"].ctypes.data, None, 256, 256, 0,
                                  out.ctypes.data, out.size)
    assert st == 1  # destination too small
    assert lib.pf_packed_bytes(0, 256, 100) == 0  # K not a multiple of 128
    st = lib.pf_pack_weights_host(1, w["bits"].ctypes.data, w["scales"].ctypes.data, None, 256, 256, 0,
                                  out.ctypes.data, out.size)
    assert st == 1  # INT4 without zero points


def test_validate_chunk_order_and_codes(lib):
    s = synth.TINY
    import dataclasses
    c = pf.make_config(dataclasses.replace(s, vocab=100), max_chunk=16)
    toks = np.array([1, 2, 3], np.int32)
    assert pf.pf_validate_chunk(c, 0, toks, 3, 0, False, False) == 0
    assert pf.pf_validate_chunk(c, 0, toks, 0, 0, False, False) == 3       # empty chunk first
    assert pf.pf_validate_chunk(c, 5, toks, 3, 0, False, False) == 4       # non-sequential start
    bad = np.array([1, 100, 3], np.int32)
    assert pf.pf_validate_chunk(c, 0, bad, 3, 0, False, False) == 5        # out of vocab
    assert pf.pf_validate_chunk(c, 5, bad, 3, 0, False, False) == 4        # start is checked before vocab
    assert pf.pf_validate_chunk(c, 0, np.array([-1], np.int32), 1, 0, False, False) == 5
    assert pf.pf_validate_chunk(c, 62, toks, 3, 62, False, False) == 6     # 62 + 3 > max_seq 64
    assert pf.pf_validate_chunk(c, 0, toks, 3, 0, True, False) == 7        # logits without a head
    assert pf.pf_validate_chunk(c, 0, toks, 3, 0, True, True) == 0
    assert b"vocab" in lib.pf_last_error() or True


def test_config_check(lib):
    import dataclasses
    good = pf.make_config(synth.QWEN3_8B_LAYER, 512)
    assert lib.pf_config_check(ctypes.byref(good)) == 0
    for field, val in (("hidden", 100), ("head_dim", 96), ("n_kv_heads", 5), ("max_chunk", 0),
                       ("wfmt", 7), ("kv_dtype", 9)):
        bad = pf.make_config(synth.QWEN3_8B_LAYER, 512)
        setattr(bad, field, val)
        assert lib.pf_config_check(ctypes.byref(bad)) != 0, field
    assert lib.pf_kv_bytes(ctypes.byref(good)) == 1 * 8 * 4096 * 128 * 2
    assert lib.pf_workspace_bytes(ctypes.byref(good)) > 0


def test_ring_config_check_and_sizes(lib):
    # the ring / sink cache (turbospark-runtime prefill.rs batch-attention contract:
    # ring_capacity, sink_count): 0 <= S < R, a 16-bit cache, and K/V of R slots per head
    import dataclasses
    s = synth.QWEN3_8B_LAYER
    ring = pf.make_config(s, 512, ring_capacity=1024, sink_count=4)
    assert lib.pf_config_check(ctypes.byref(ring)) == 0
    assert lib.pf_kv_bytes(ctypes.byref(ring)) == 1 * 8 * 1024 * 128 * 2
    linear = pf.make_config(s, 512)
    # the ring adds the chunk's K / V rows to the workspace: 2 x 8 heads x 512 rows x 128 x 2 B
    extra = lib.pf_workspace_bytes(ctypes.byref(ring)) - lib.pf_workspace_bytes(ctypes.byref(linear))
    assert extra >= 2 * 8 * 512 * 128 * 2
    for R, S, want in ((1024, 1024, 2), (1024, -1, 2), (0, 3, 2), (-5, 0, 2)):
        bad = pf.make_config(s, 512, ring_capacity=R, sink_count=S)
        assert lib.pf_config_check(ctypes.byref(bad)) == want, (R, S)
    f32 = pf.make_config(dataclasses.replace(s, kv_dtype="f32"), 512, ring_capacity=64, sink_count=0)
    assert lib.pf_config_check(ctypes.byref(f32)) == 8  # PF_ERR_UNSUPPORTED
    assert lib.pf_abi_version() == 4


def test_paged_config_check_and_sizes(lib):
    # paged cache: P blocks of PF_KV_BLOCK = 128 positions per (layer, kv head); a 16-bit cache,
    # not combined with a ring; K/V hold 128 P slots; the workspace gains the block table
    import dataclasses
    s = synth.QWEN3_8B_LAYER  # max_seq 4096: 32 position blocks
    paged = pf.make_config(s, 512, kv_block_pool=40)
    assert lib.pf_config_check(ctypes.byref(paged)) == 0
    assert lib.pf_kv_bytes(ctypes.byref(paged)) == 1 * 8 * (40 * 128) * 128 * 2
    linear = pf.make_config(s, 512)
    extra = lib.pf_workspace_bytes(ctypes.byref(paged)) - lib.pf_workspace_bytes(ctypes.byref(linear))
    assert 32 * 4 <= extra <= 32 * 4 + 256
    assert lib.pf_config_check(ctypes.byref(pf.make_config(s, 512, kv_block_pool=-1))) == 2  # PF_ERR_SHAPE
    both = pf.make_config(s, 512, kv_block_pool=8, ring_capacity=1024, sink_count=4)
    assert lib.pf_config_check(ctypes.byref(both)) == 2
    f32 = pf.make_config(dataclasses.replace(s, kv_dtype="f32"), 512, kv_block_pool=8)
    assert lib.pf_config_check(ctypes.byref(f32)) == 8  # PF_ERR_UNSUPPORTED


def test_attention_scratch_bytes(lib):
    s = synth.QWEN3_8B_LAYER
    c = pf.make_config(s, 512)
    # 8 kv heads' arrival counters (32 B), then the partial O sums and (max, sum) per row
    assert lib.pf_attention_scratch_bytes(ctypes.byref(c), 16, 9) == 32 + 9 * 16 * 32 * (128 + 2) * 4
    assert lib.pf_attention_scratch_bytes(ctypes.byref(c), 16, 1) == 0
    assert lib.pf_attention_scratch_bytes(ctypes.byref(c), 16, 65) == 0
    assert lib.pf_attention_scratch_bytes(ctypes.byref(c), 0, 2) == 0


def test_rope_table_matches_definition(lib):
    t = pf.pf_rope_table_host(1e6, 128, 64)
    p, i = 37, 5
    ang = p * (1e6 ** (-2 * i / 128))
    assert t[p, i, 0] == np.float32(np.cos(ang)) and t[p, i, 1] == np.float32(np.sin(ang))
    assert np.all(t[0, :, 0] == 1) and np.all(t[0, :, 1] == 0)


def test_greedy_and_verify_reject_bad_arguments_before_any_launch(lib):
    """The argmax, greedy-decode and verify entry points refuse NULL / malformed arguments
    on the host (no device memory is touched, so this runs without a GPU): status 1 is
    PF_ERR_INVALID_ARG, 2 PF_ERR_SHAPE."""
    out = ctypes.c_int32()
    x = np.zeros(4, np.float32)
    assert lib.pf_op_argmax(None, 1, 4, 4, ctypes.addressof(out), None) == 1
    assert lib.pf_op_argmax(x.ctypes.data, 1, 4, 4, None, None) == 1
    assert lib.pf_op_argmax(x.ctypes.data, 0, 4, 4, ctypes.addressof(out), None) == 2
    assert lib.pf_op_argmax(x.ctypes.data, 1, 0, 4, ctypes.addressof(out), None) == 2
    assert lib.pf_op_argmax(x.ctypes.data, 1, 4, 3, ctypes.addressof(out), None) == 2
    assert lib.pf_decode_step_greedy(None, None, None, None, None) == 1
    assert lib.pf_prefill_verify(None, None, 1, 0, None, None, None) == 1
    assert b"session" in lib.pf_last_error()
