"""Pins for the CPU oracle: each check ties an oracle function to something other
than itself — a closed form, an invariant, a special case with a known answer, a
library routine evaluated by a different route, or brute force on tiny inputs.

Each test names the mistake it is meant to catch.
"""
import math

import numpy as np
import pytest
import torch

from oracle import prefill_oracle as O
from quantized_transformer_prefill_q1_gb300 import synth

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ----------------------------------------------------------------------------- dequant
def test_q1_bit_order_and_sign_special_case():
    # one row, K = 256 (two groups). Byte 0 = 0x01: only k = 0 set (LSB first);
    # byte 1 = 0x80: only k = 15 set. Group 0 scale 0.5, group 1 scale 0.25.
    # Catches: MSB-first bit order, inverted sign convention, scale on the wrong axis.
    bits = np.zeros((1, 32), np.uint8)
    bits[0, 0] = 0x01
    bits[0, 1] = 0x80
    bits[0, 16] = 0xFF  # k = 128..135 all positive (group 1)
    scales = np.array([[0.5, 0.25]], np.float16)
    w = O.dequant_q1(bits, scales)
    assert w.shape == (1, 256)
    assert w[0, 0] == 0.5 and w[0, 1] == -0.5 and w[0, 7] == -0.5
    assert w[0, 8] == -0.5 and w[0, 15] == 0.5
    assert w[0, 127] == -0.5
    assert np.all(w[0, 128:136] == 0.25) and w[0, 136] == -0.25


def test_q1_closed_form_row_sums_via_popcount():
    # sum_k w[n, k] over group g = s * (2 * popcount(bits of group) - 128), with
    # popcount taken by Python's int.bit_count (a different route than unpackbits).
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 256, size=(5, 48), dtype=np.uint8)  # K = 384, 3 groups
    scales = rng.uniform(0.01, 0.1, size=(5, 3)).astype(np.float16)
    w = O.dequant_q1(bits, scales)
    for n in range(5):
        for g in range(3):
            pc = sum(int(b).bit_count() for b in bits[n, 16 * g: 16 * (g + 1)])
            expect = float(scales[n, g]) * (2 * pc - 128)
            assert w[n, 128 * g: 128 * (g + 1)].sum() == pytest.approx(expect, abs=1e-12)


def test_q1_all_ones_gemv_closed_form():
    # all bits set, one scale s  =>  W x = s * sum(x) for every row.
    bits = np.full((3, 64), 0xFF, np.uint8)
    scales = np.full((3, 4), 0.0625, np.float16)
    x = np.random.default_rng(2).standard_normal(512)
    np.testing.assert_allclose(O.dequant_q1(bits, scales) @ x, 0.0625 * x.sum() * np.ones(3),
                               rtol=1e-12)


def test_int4_nibble_order_and_affine_special_case():
    # byte 0x21: low nibble 1 -> k = 0, high nibble 2 -> k = 1. s = 2, z = 0.5
    # => w = [1, 3]. Catches nibble swap and w = s*q - z style mistakes.
    codes = np.zeros((1, 64), np.uint8)
    codes[0, 0] = 0x21
    codes[0, 1] = 0xF0  # k = 2 -> 0, k = 3 -> 15
    scales = np.array([[2.0]], np.float16)
    zeros = np.array([[0.5]], np.float16)
    w = O.dequant_int4(codes, scales, zeros)
    assert w[0, 0] == 1.0 and w[0, 1] == 3.0 and w[0, 2] == -1.0 and w[0, 3] == 29.0
    assert w[0, 4] == -1.0


def test_gemm_bruteforce_tiny():
    # y @ W^T against a pure-Python loop that extracts each bit with integer ops and
    # sums with math.fsum (independent of unpackbits / BLAS).
    rng = np.random.default_rng(3)
    N, K, M = 3, 256, 2
    bits = rng.integers(0, 256, size=(N, K // 8), dtype=np.uint8)
    scales = rng.uniform(0.01, 0.05, size=(N, K // 128)).astype(np.float16)
    y = rng.standard_normal((M, K))
    got = y @ O.dequant_q1(bits, scales).T
    for m in range(M):
        for n in range(N):
            terms = []
            for k in range(K):
                bit = (int(bits[n, k // 8]) >> (k % 8)) & 1
                s = float(scales[n, k // 128])
                terms.append((s if bit else -s) * float(y[m, k]))
            assert got[m, n] == pytest.approx(math.fsum(terms), rel=1e-12, abs=1e-12)


# ----------------------------------------------------------------------------- rmsnorm
def test_rmsnorm_constant_row_closed_form():
    c, eps = 0.75, 1e-6
    w = np.linspace(0.5, 1.5, 64)
    y = O.rmsnorm(np.full(64, c), w, eps)
    np.testing.assert_allclose(y, w * c / math.sqrt(c * c + eps), rtol=1e-15)


def test_rmsnorm_scale_invariance_and_library():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((5, 96))
    w = 1 + 0.1 * rng.standard_normal(96)
    np.testing.assert_allclose(O.rmsnorm(7.0 * x, w, 0.0), O.rmsnorm(x, w, 0.0), rtol=1e-13)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (96,), torch.from_numpy(w), eps=1e-6)
    np.testing.assert_allclose(O.rmsnorm(x, w, 1e-6), ref.numpy(), rtol=1e-12)


# ----------------------------------------------------------------------------- RoPE
def test_rope_matches_complex_multiplication():
    # RoFormer's definition: the pair (a_i, b_i) as a + i b is multiplied by e^{i*angle}.
    rng = np.random.default_rng(5)
    T, H, hd = 7, 3, 64
    v = rng.standard_normal((T, H, hd))
    ang = O.rope_angles(np.arange(100, 100 + T), hd, 1e6)
    out = O.apply_rope(v, ang)
    z = (v[..., : hd // 2] + 1j * v[..., hd // 2:]) * np.exp(1j * ang)[:, None, :]
    np.testing.assert_allclose(out[..., : hd // 2], z.real, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(out[..., hd // 2:], z.imag, rtol=1e-12, atol=1e-12)


def test_rope_invariants():
    rng = np.random.default_rng(6)
    hd = 128
    q = rng.standard_normal((1, 1, hd))
    k = rng.standard_normal((1, 1, hd))
    # position 0 is the identity
    np.testing.assert_array_equal(O.apply_rope(q, O.rope_angles([0], hd, 1e6)), q)
    # each pair's norm is preserved
    r = O.apply_rope(q, O.rope_angles([4095], hd, 1e6))
    n0 = q[..., :64] ** 2 + q[..., 64:] ** 2
    n1 = r[..., :64] ** 2 + r[..., 64:] ** 2
    np.testing.assert_allclose(n1, n0, rtol=1e-12)

    # <R_p q, R_p' k> depends only on p - p'
    def dot(p, pp):
        return float(np.sum(O.apply_rope(q, O.rope_angles([p], hd, 5e5)) *
                            O.apply_rope(k, O.rope_angles([pp], hd, 5e5))))
    assert dot(10, 3) == pytest.approx(dot(1007, 1000), rel=1e-9)
    assert dot(10, 3) != pytest.approx(dot(10, 4), rel=1e-6)


def test_rope_frequency_ladder():
    # pair 0 turns by exactly p radians; consecutive pairs' rates form a geometric
    # ladder with ratio theta^(-2/hd) (catches theta^(-i/hd) or reversed order).
    hd, theta = 128, 1e6
    inv = O.rope_inv_freq(hd, theta)
    assert inv[0] == 1.0
    np.testing.assert_allclose(inv[1:] / inv[:-1], theta ** (-2.0 / hd), rtol=1e-12)
    assert inv[-1] == pytest.approx(theta ** (-(hd - 2) / hd), rel=1e-12)


# ----------------------------------------------------------------------------- attention
def _sdpa_reference(q, kc, vc, start):
    T, nq, hd = q.shape
    nkv = kc.shape[0]
    L = start + T
    K = torch.from_numpy(kc[:, :L].astype(np.float64)).repeat_interleave(nq // nkv, dim=0)
    V = torch.from_numpy(vc[:, :L].astype(np.float64)).repeat_interleave(nq // nkv, dim=0)
    Q = torch.from_numpy(q.astype(np.float64)).transpose(0, 1)  # [nq, T, hd]
    mask = torch.arange(L)[None, :] <= (start + torch.arange(T))[:, None]
    o = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask)
    return o.transpose(0, 1).numpy()


@pytest.mark.parametrize("nq,nkv,start,T", [(4, 2, 0, 9), (8, 2, 13, 5), (4, 4, 3, 6)])
def test_attention_vs_torch_sdpa(nq, nkv, start, T):
    rng = np.random.default_rng(7)
    hd = 32
    q = rng.standard_normal((T, nq, hd))
    kc = rng.standard_normal((nkv, start + T + 4, hd)).astype(np.float32)
    vc = rng.standard_normal((nkv, start + T + 4, hd)).astype(np.float32)
    kc[:, start + T:] = np.nan  # never read beyond the last query position
    vc[:, start + T:] = np.nan
    got = O.causal_gqa_attention(q, kc, vc, start)
    np.testing.assert_allclose(got, _sdpa_reference(q, kc, vc, start), rtol=1e-10, atol=1e-12)


def test_attention_weights_sum_to_one_and_single_key():
    rng = np.random.default_rng(8)
    q = rng.standard_normal((5, 4, 16)) * 10
    kc = rng.standard_normal((2, 5, 16)).astype(np.float32)
    ones = np.ones((2, 5, 16), np.float32)
    np.testing.assert_allclose(O.causal_gqa_attention(q, kc, ones, 0), 1.0, rtol=0, atol=1e-12)
    # the first position sees only itself: output = v_0 of its kv head
    vc = rng.standard_normal((2, 5, 16)).astype(np.float32)
    o = O.causal_gqa_attention(q, kc, vc, 0)
    for h in range(4):
        np.testing.assert_allclose(o[0, h], vc[h // 2, 0], rtol=1e-12)


# ----------------------------------------------------------------------------- misc steps
def test_silu_matches_torch():
    g = np.linspace(-30, 30, 1001)
    np.testing.assert_allclose(O.silu(g), torch.nn.functional.silu(torch.from_numpy(g)).numpy(),
                               rtol=1e-13, atol=1e-300)


@pytest.mark.parametrize("dt,tdt", [("bf16", torch.bfloat16), ("f16", torch.float16)])
def test_cache_rounding_matches_torch(dt, tdt):
    rng = np.random.default_rng(9)
    x = (rng.standard_normal(100000) * np.exp(rng.uniform(-8, 8, 100000))).astype(np.float32)
    ref = torch.from_numpy(x).to(tdt).to(torch.float32).numpy()
    np.testing.assert_array_equal(O.round_to_cache(x, dt), ref)


# ----------------------------------------------------------------------------- layer / stack
def _tiny(**kw):
    return __import__("dataclasses").replace(synth.TINY, **kw)


def test_kv_slots_written_exactly_in_range():
    s = _tiny(max_seq=40)
    layers, _ = synth.model_inputs(s)
    m = O.OracleModel(s, layers)
    x = synth.hidden_input(20, s.hidden)
    m.prefill(x[:12], [12], False, False)
    k_before = m.k_cache.copy()
    m.forward_chunk(x[12:20], 12, False)
    # positions 0..11 untouched, 12..19 written, 20.. still the NaN sentinel
    np.testing.assert_array_equal(m.k_cache[:, :, :12], k_before[:, :, :12])
    assert np.all(np.isfinite(m.k_cache[:, :, 12:20]))
    assert np.all(np.isnan(m.k_cache[:, :, 20:])) and np.all(np.isnan(m.v_cache[:, :, 20:]))


@pytest.mark.parametrize("shape_kw", [{}, {"kv_dtype": "bf16"}, {"qk_norm": False, "wfmt": "int4"}])
def test_one_shot_equals_chunked_equals_decode(shape_kw):
    s = _tiny(**shape_kw)
    layers, _ = synth.model_inputs(s)
    x = synth.hidden_input(16, s.hidden)
    m = O.OracleModel(s, layers)
    one, _ = m.prefill(x, [16], False, False)
    m.reset()
    chunked, _ = m.prefill(x, [5, 1, 7, 3], False, False)
    m.reset()
    dec = O.decode_prompt(m, x)
    assert O.rel_l2(chunked, one) <= 1e-6
    assert O.rel_l2(dec, one) <= 1e-6


def test_layer_major_equals_chunk_major_with_head():
    s = _tiny(n_layers=3, vocab=1000, max_seq=64)
    layers, extra = synth.model_inputs(s)
    toks = synth.tokens(24, s.vocab)
    a = O.OracleModel(s, layers, extra)
    xa, la = a.prefill(toks, [8, 8, 8], True, True)
    b = O.OracleModel(s, layers, extra)
    xb, lb = b.prefill_layer_major(toks, [8, 8, 8], True, True)
    assert O.rel_l2(xb, xa) <= 1e-6 and O.rel_l2(lb, la) <= 1e-6
    np.testing.assert_array_equal(a.k_cache[:, :, :24].shape, b.k_cache[:, :, :24].shape)


def test_causality():
    s = _tiny(n_layers=2)
    layers, _ = synth.model_inputs(s)
    x = synth.hidden_input(12, s.hidden)
    x2 = x.copy()
    x2[7:] = synth.hidden_input(5, s.hidden, stream=9)
    a, _ = O.OracleModel(s, layers).prefill(x, [12], False, False)
    b, _ = O.OracleModel(s, layers).prefill(x2, [12], False, False)
    np.testing.assert_array_equal(a[:7], b[:7])
    assert not np.array_equal(a[7:], b[7:])


def test_validation_errors():
    s = _tiny(vocab=100, max_seq=16)
    layers, extra = synth.model_inputs(s)
    m = O.OracleModel(s, layers, extra)
    with pytest.raises(ValueError):
        m.forward_chunk(np.zeros((0, s.hidden), np.float32), 0, False)
    with pytest.raises(ValueError):
        m.forward_chunk(np.zeros((2, s.hidden), np.float32), 3, False)
    with pytest.raises(ValueError):
        m.embed(np.array([5, 100]))
    with pytest.raises(ValueError):
        m.forward_chunk(np.zeros((17, s.hidden), np.float32), 0, False)


# ----------------------------------------------------------------------------- embedding / head
def test_embed_rows_exact_without_scale():
    # The embedding is a plain row gather at scale 1.0 (turbospark-runtime 0.3.0
    # families/llama/prefill.rs, the chunk function's embedding step; no sqrt(hidden)
    # factor). Rows planted with known values (each row's entries encode its own id) come
    # back bit for bit, first and last id included, repeated ids included, in token order.
    # Catches: a sqrt(H) scale, an off-by-one id, a transposed table, an f16 round trip.
    H, V = 256, 37
    s = _tiny(vocab=V)
    table = (np.arange(V, dtype=np.float32)[:, None] * np.float32(1000.0)
             + np.arange(H, dtype=np.float32)[None, :] * np.float32(0.125))
    table[V - 1] = np.float32(1.0) + np.float32(2.0 ** -20)  # not representable in f16
    m = O.OracleModel(s, synth.model_inputs(s)[0], {"embed": table})
    toks = np.array([0, V - 1, 5, 5, 36, 1], np.int32)
    got = m.embed(toks)
    assert got.dtype == np.float32 and got.shape == (6, H)
    for i, t in enumerate(toks):
        np.testing.assert_array_equal(got[i], table[t])
    assert got[0, 1] == np.float32(0.125) and got[2, 0] == np.float32(5000.0)
    assert got[1, 0] == np.float32(1.0) + np.float32(2.0 ** -20)


def test_head_uses_the_final_eps():
    # The tail normalises the last row with the final norm's own eps (metal_prefill.rs,
    # encode_full_forward_prefill: final_norm_eps, separate from the layers' eps), then
    # applies the LM head. A row of small magnitude makes the two eps values give clearly
    # different results; the expected logits are formed in pure Python (bit extraction,
    # math.fsum), a different route from the oracle's numpy code.
    # Catches: the layer eps used in the tail, the norm weight skipped, the wrong row.
    H, V = 256, 5
    s = _tiny(vocab=V, eps=1e-6, final_eps=1e-2)
    rng = np.random.default_rng(11)
    lm = synth.q1_weight(rng, V, H)
    fn = (1.0 + 0.1 * rng.standard_normal(H)).astype(np.float32)
    x = (0.05 * rng.standard_normal(H)).astype(np.float32)
    m = O.OracleModel(s, synth.model_inputs(s)[0], {"final_norm": fn, "lm_head": lm})
    got = m.head(x)

    def expect(eps):
        ms = math.fsum(float(v) * float(v) for v in x) / H
        y = [np.float32(float(x[k]) / math.sqrt(ms + eps) * float(fn[k])) for k in range(H)]
        out = []
        for n in range(V):
            terms = []
            for k in range(H):
                bit = (int(lm["bits"][n, k // 8]) >> (k % 8)) & 1
                sc = float(lm["scales"][n, k // 128])
                terms.append((sc if bit else -sc) * float(y[k]))
            out.append(math.fsum(terms))
        return np.array(out)

    np.testing.assert_allclose(got, expect(1e-2), rtol=1e-6, atol=1e-7)
    wrong = expect(1e-6)
    assert np.max(np.abs(wrong - expect(1e-2))) > 100 * np.max(np.abs(got - expect(1e-2))) + 1e-3


# ----------------------------------------------------------------------------- greedy tail
def test_argmax_first_special_cases_and_library():
    # Catches: the last (not first) of equal maxima, NaN winning or poisoning the row, an
    # all -inf or all-NaN row giving -1, and an off-by-one on the row axis.
    rows = np.array([[1.0, 5.0, 5.0, 2.0],
                     [np.nan, 1.0, np.nan, 3.0],
                     [np.nan, np.nan, np.nan, np.nan],
                     [-np.inf, -np.inf, -np.inf, -np.inf],
                     [0.0, -0.0, 0.0, -1.0]], np.float32)
    np.testing.assert_array_equal(O.argmax_first(rows), [1, 3, 0, 0, 0])
    assert int(O.argmax_first(np.array([7.0], np.float32))) == 0
    # without NaNs, numpy's argmax (which also returns the first maximum) agrees, ties
    # planted at random places included
    rng = np.random.default_rng(5)
    x = rng.standard_normal((40, 257)).astype(np.float32)
    x[::3, 200] = x[::3].max(axis=1)  # a tie with an earlier maximum in every third row
    np.testing.assert_array_equal(O.argmax_first(x), np.argmax(x, axis=1))


def test_verify_tail_is_the_head_at_every_position():
    # The verify tail scores every position: row t must be the single-token tail of the
    # prefix that ends at t. Catches: the norm or head applied to the wrong row, a shifted
    # row order, and the ids not being the rows' argmax.
    s = _tiny(n_layers=2, vocab=257, max_seq=32)
    layers, extra = synth.model_inputs(s)
    toks = synth.tokens(6, s.vocab)
    lg, ids = O.OracleModel(s, layers, extra).prefill_verify(toks)
    assert lg.shape == (6, s.vocab) and ids.shape == (6,)
    np.testing.assert_array_equal(ids, O.argmax_first(lg))
    for t in range(6):
        _, ref = O.OracleModel(s, layers, extra).prefill(toks[:t + 1], [t + 1], True, True)
        assert O.rel_l2(lg[t], ref) <= 1e-12


# ----------------------------------------------------------------------------- ring / sink KV
def test_ring_attention_brute_force():
    # Windowed attention with sinks against an explicit gather of the keys each query may
    # see, in pure Python loops. Catches: a window off by one, sinks that let a query see
    # the future, a mask of the wrong sign, the kv-head mapping lost in the windowed path.
    rng = np.random.default_rng(11)
    nq, nkv, hd, L, start, T, window, sinks = 4, 2, 16, 20, 12, 8, 5, 2
    q = rng.standard_normal((T, nq, hd))
    k = rng.standard_normal((nkv, L, hd)).astype(np.float32)
    v = rng.standard_normal((nkv, L, hd)).astype(np.float32)
    out = O.causal_gqa_attention(q, k, v, start, window, sinks)
    for t in range(T):
        p = start + t
        vis = [j for j in range(p + 1) if j < sinks or j > p - window]
        assert len(vis) == sinks + window
        for h in range(nq):
            g = h // (nq // nkv)
            sc = [math.fsum(q[t, h, d] * float(k[g, j, d]) for d in range(hd)) / math.sqrt(hd) for j in vis]
            mx = max(sc)
            e = [math.exp(x - mx) for x in sc]
            z = math.fsum(e)
            ref = [math.fsum(e[i] / z * float(v[g, j, d]) for i, j in enumerate(vis)) for d in range(hd)]
            np.testing.assert_allclose(out[t, h], ref, rtol=1e-12, atol=1e-12)


def test_ring_window_of_one_is_the_token_itself():
    # closed form: a window of one position and no sinks gives o = v of the query's own position
    rng = np.random.default_rng(12)
    q = rng.standard_normal((5, 4, 8))
    k = rng.standard_normal((2, 9, 8)).astype(np.float32)
    v = rng.standard_normal((2, 9, 8)).astype(np.float32)
    out = O.causal_gqa_attention(q, k, v, 4, window=1, sinks=0)
    for t in range(5):
        for h in range(4):
            np.testing.assert_array_equal(out[t, h], v[h // 2, 4 + t].astype(np.float64))


def test_ring_slot_mapping():
    # sinks keep their slots, later positions cycle through the rest
    s = _tiny(max_seq=32)
    layers, _ = synth.model_inputs(s)
    m = O.OracleModel(s, layers, ring_capacity=6, sink_count=2)
    assert [m.ring_slot(p) for p in range(12)] == [0, 1, 2, 3, 4, 5, 2, 3, 4, 5, 2, 3]
    with pytest.raises(ValueError):
        O.OracleModel(s, layers, ring_capacity=4, sink_count=4)


def test_ring_wide_enough_equals_linear():
    # a ring that never wraps changes nothing (bit-identical)
    s = _tiny(max_seq=40)
    layers, _ = synth.model_inputs(s)
    x = synth.hidden_input(16, s.hidden)
    lin, _ = O.OracleModel(s, layers).prefill(x, [16], False, False)
    for R, S in ((16, 0), (20, 3)):
        ring, _ = O.OracleModel(s, layers, ring_capacity=R, sink_count=S).prefill(x, [16], False, False)
        np.testing.assert_array_equal(ring, lin)


def test_ring_one_shot_equals_chunked_equals_physical_ring_decode():
    # The batched form masks a linear history; the per-token form reads a physical ring of
    # ring_capacity slots. Both must agree, chunked or not, and the ring must matter.
    s = _tiny(max_seq=48)
    layers, _ = synth.model_inputs(s)
    x = synth.hidden_input(24, s.hidden)
    kw = dict(ring_capacity=10, sink_count=2)
    a = O.OracleModel(s, layers, **kw)
    one, _ = a.prefill(x, [24], False, False)
    chunked, _ = O.OracleModel(s, layers, **kw).prefill(x, [5, 7, 12], False, False)
    d = O.OracleModel(s, layers, **kw)
    dec = O.decode_prompt(d, x)
    assert O.rel_l2(chunked, one) <= 1e-6
    assert O.rel_l2(dec, one) <= 1e-6
    lin, _ = O.OracleModel(s, layers).prefill(x, [24], False, False)
    assert O.rel_l2(one, lin) > 1e-3
    for l in range(s.n_layers):  # what the batched model's history implies for the ring slots
        k, v = a.ring_cache(l)
        np.testing.assert_allclose(k, d.ring_k[l], rtol=1e-5, atol=1e-6)
        np.testing.assert_allclose(v, d.ring_v[l], rtol=1e-5, atol=1e-6)
