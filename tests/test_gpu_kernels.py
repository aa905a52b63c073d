"""Step-level parity: each libpf kernel (through the C ABI) against the CPU oracle on the
same seeded inputs. Integer / byte / index work is compared bit-exactly; floating point
within the tolerance stated (and derived) at each test."""
import dataclasses

import numpy as np
import pytest

from oracle import prefill_oracle as O
from quantized_transformer_prefill_q1_gb300 import pf, synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU-only hosts, never run there
    pytest.skip("needs a GPU", allow_module_level=True)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def rel_l2(a, b):
    return O.rel_l2(np.asarray(a, np.float64), np.asarray(b, np.float64))


# ----------------------------------------------------------------------------- unpacking
def _int4_kernel_rule(w):
    """The GPU's INT4 dequantisation decision, taken in the same (f16) arithmetic:
    f16(f16(q - z) * s), each operation rounded to nearest even."""
    n, k = w["n"], w["k"]
    q = np.empty((n, k), np.float16)
    q[:, 0::2] = w["codes"] & 15
    q[:, 1::2] = w["codes"] >> 4
    z = np.repeat(w["zeros"], 128, axis=1)
    s = np.repeat(w["scales"], 128, axis=1)
    return (q - z) * s


@pytest.mark.parametrize("fmt", ["q1", "int4"])
@pytest.mark.parametrize("n,k", [(256, 128), (300, 384), (1000, 4096), (24576, 128)])
def test_dequant_bit_exact(fmt, n, k):
    w = synth.quant_weight(fmt, synth.rng_for(11, n, k), n, k)
    packed = dev(pf.pf_pack_weights_host(w))
    out = torch.full((n, k), float("nan"), dtype=torch.float16, device="cuda")
    pf.pf_op_dequant(pf._WFMT[fmt], packed, n, k, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    if fmt == "q1":
        ref = O.dequant_q1(w["bits"], w["scales"]).astype(np.float16)  # +-s: exact in f16
        np.testing.assert_array_equal(got.view(np.uint16), ref.view(np.uint16))
    else:
        ref = _int4_kernel_rule(w)
        np.testing.assert_array_equal(got.view(np.uint16), ref.view(np.uint16))
        exact = O.dequant_int4(w["codes"], w["scales"], w["zeros"])
        err = np.abs(got.astype(np.float64) - exact)
        assert np.all(err <= 2.0 ** -10 * np.abs(exact) + 2.0 ** -24)


def test_pack_interleave_gate_up():
    # dequantising an interleaved gate_up tile gives gate rows then the matching up rows
    I, k = 256, 256
    w = synth.q1_weight(synth.rng_for(12), 2 * I, k)
    packed = dev(pf.pf_pack_weights_host(w, interleave_gate_up=True))
    out = torch.empty((2 * I, k), dtype=torch.float16, device="cuda")
    pf.pf_op_dequant(pf.W_Q1, packed, 2 * I, k, out)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    ref = O.dequant_q1(w["bits"], w["scales"]).astype(np.float16)
    for t in range(4):  # each 128 packed rows: 64 gate rows, then the 64 matching up rows
        np.testing.assert_array_equal(got[128 * t: 128 * t + 64], ref[64 * t: 64 * t + 64])
        np.testing.assert_array_equal(got[128 * t + 64: 128 * t + 128], ref[I + 64 * t: I + 64 * t + 64])


# ----------------------------------------------------------------------------- GEMM
# (M, N, K, most CTAs): 0 = one per SM. Few CTAs over many k-blocks split tiles between
# CTAs in every way the k-range partition allows (head / tail / middle / three-way).
GEMM_CASES = [
    (1, 256, 128, 1), (16, 512, 256, 0), (127, 768, 384, 2), (129, 256, 1024, 3),
    (300, 6144, 4096, 0), (512, 4096, 4096, 7), (512, 4096, 12288, 0), (64, 1280, 512, 5),
    (200, 512, 1024, 9), (40, 24576, 256, 0),
    # 8 < M <= 64: weight rows as the MMA's M side (tokens padded to 16 / 32 / 64)
    (12, 1280, 512, 0), (33, 6144, 1024, 0), (64, 4096, 14336, 0),
    # M <= 8: the warp-MMA GEMV (ragged M and N, long K, several CTAs per row block)
    (4, 4096, 4096, 0), (2, 24576, 4096, 3), (3, 768, 384, 0), (8, 2048, 1024, 0), (5, 776, 640, 0),
    (1, 4096, 14336, 0),
]


def assert_counters_zero(scratch, m, n):
    """Every launch that completes leaves the per-tile arrival counters zero (one per
    128 x 256 tile, or two per 256 x 256 tile of a CTA pair)."""
    tiles = max(-(-m // 128), 2 * -(-m // 256)) * -(-n // 256)
    counters = scratch[scratch.numel() - 4 * tiles:].view(torch.int32)
    assert int(counters.abs().sum()) == 0


@pytest.mark.parametrize("fmt", ["q1", "int4"])
@pytest.mark.parametrize("m,n,k,ctas", GEMM_CASES)
@pytest.mark.parametrize("epi", [pf.EPI_STORE_F32, pf.EPI_RESID_ADD, pf.EPI_SWIGLU])
def test_gemm_vs_oracle(fmt, m, n, k, ctas, epi):
    if epi == pf.EPI_SWIGLU and n % 256:
        pytest.skip("SwiGLU needs N = 2I with I % 128 == 0")
    rng = synth.rng_for(13, m, n, k)
    a = rng.standard_normal((m, k)).astype(np.float16)
    w = synth.quant_weight(fmt, rng, n, k)
    W = O.dequant(w)
    ref = a.astype(np.float64) @ W.T
    packed = dev(pf.pf_pack_weights_host(w, interleave_gate_up=(epi == pf.EPI_SWIGLU)))
    a_d = dev(a)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    scratch = pf.gemm_scratch(m, n, ctas)
    # Q1: exact f16 products, f32 accumulation of up to 12288 of them in the tensor core
    # (and, for a tile split between CTAs, in the f32 partial sums): ~sqrt(K) * 2^-24 plus the
    # tensor core's internal
    # alignment -> 5e-5. INT4: the f16 rounding of each weight (2^-11) dominates -> 1e-3.
    tol = 5e-5 if fmt == "q1" else 1e-3
    if epi == pf.EPI_SWIGLU:
        out = torch.full((m, n // 2), float("nan"), dtype=torch.float16, device="cuda")
        pf.pf_op_gemm(pf._WFMT[fmt], epi, a_d, packed, m, n, k, out, scratch, ctas, status)
        pf.pf_status_read(status)
        assert_counters_zero(scratch, m, n)
        g, u = ref[:, : n // 2], ref[:, n // 2:]
        exp = O.silu(g) * u
        assert rel_l2(out.cpu().numpy(), exp) <= 2e-3
        return
    x0 = rng.standard_normal((m, n)).astype(np.float32)
    if epi == pf.EPI_RESID_ADD:
        out = dev(x0)
        exp = x0.astype(np.float64) + ref
    else:
        out = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
        exp = ref
    pf.pf_op_gemm(pf._WFMT[fmt], epi, a_d, packed, m, n, k, out, scratch, ctas, status)
    pf.pf_status_read(status)
    assert_counters_zero(scratch, m, n)
    got = out.cpu().numpy()
    if epi == pf.EPI_RESID_ADD:
        assert rel_l2(got - x0, ref) <= tol
    assert rel_l2(got, exp) <= tol


# ----------------------------------------------------------------------------- RMSNorm
@pytest.mark.parametrize("m,h", [(1, 256), (16, 256), (512, 4096), (37, 12288)])
def test_rmsnorm_within_1e3(m, h):
    rng = synth.rng_for(14, m, h)
    x = rng.standard_normal((m, h)).astype(np.float32) * 3
    w = synth.norm_weight(rng, h)
    y = torch.empty((m, h), dtype=torch.float16, device="cuda")
    pf.pf_op_rmsnorm(dev(x), dev(w), 1e-6, y)
    torch.cuda.synchronize()
    ref = O.rmsnorm(x, w, 1e-6)
    err = np.abs(y.cpu().numpy().astype(np.float64) - ref)
    assert np.all(err <= 1e-3 * np.abs(ref) + 1e-6)


# ----------------------------------------------------------------------------- QK-norm + RoPE + KV
SENT = {"f32": 0x7FC00001, "bf16": 0x7FC1, "f16": 0x7E01}


def _kv_case(shape, m, start, seed=15):
    rng = synth.rng_for(seed, m, start)
    s = shape
    qkv = rng.standard_normal((m, s.qkv_rows)).astype(np.float32)
    qn = synth.norm_weight(rng, s.head_dim)
    kn = synth.norm_weight(rng, s.head_dim)
    return qkv, qn, kn


@pytest.mark.parametrize("shape,m,start,layer,nl", [
    (synth.TINY, 16, 0, 0, 1), (synth.TINY, 7, 5, 1, 2),
    (synth.QWEN3_8B_LAYER, 512, 0, 0, 1), (synth.QWEN3_8B_LAYER, 33, 3000, 0, 1),
    (synth.LLAMA3_8B_INT4_LAYER, 16, 8192, 0, 1),
])
def test_qk_norm_rope_kv(shape, m, start, layer, nl):
    import dataclasses
    s = dataclasses.replace(shape, n_layers=nl)
    cfg = pf.make_config(s, max_chunk=max(m, 16))
    qkv, qn, kn = _kv_case(s, m, start)
    nq, nkv, hd = s.n_q_heads, s.n_kv_heads, s.head_dim
    rope = dev(pf.pf_rope_table_host(s.rope_theta, hd, s.max_seq))
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[s.kv_dtype]
    qdt = torch.bfloat16 if s.kv_dtype == "bf16" else torch.float16
    ib = torch.int32 if s.kv_dtype == "f32" else torch.int16
    kc = torch.empty((nl, nkv, s.max_seq, hd), dtype=tdt, device="cuda")
    vc = torch.empty_like(kc)
    kc.view(ib).fill_(SENT[s.kv_dtype])
    vc.view(ib).fill_(SENT[s.kv_dtype])
    q = torch.empty((m, nq, hd), dtype=qdt, device="cuda")
    pf.pf_op_qk_norm_rope_kv(cfg, dev(qkv), dev(qn) if s.qk_norm else None,
                             dev(kn) if s.qk_norm else None, rope, layer, start, m, q, kc, vc)
    torch.cuda.synchronize()
    # oracle
    qr = qkv[:, : nq * hd].reshape(m, nq, hd)
    kr = qkv[:, nq * hd:(nq + nkv) * hd].reshape(m, nkv, hd)
    vr = qkv[:, (nq + nkv) * hd:].reshape(m, nkv, hd)
    if s.qk_norm:
        qr = O.rmsnorm(qr, qn, s.eps).astype(np.float32)
        kr = O.rmsnorm(kr, kn, s.eps).astype(np.float32)
    ang = O.rope_angles(np.arange(start, start + m), hd, s.rope_theta)
    q_ref = O.apply_rope(qr, ang)
    k_ref = O.apply_rope(kr, ang)
    # q (kernel operand type): within 1e-3 relative before rounding, i.e. within one
    # ulp of the operand type of the rounded oracle value
    qg = q.float().cpu().numpy().astype(np.float64)
    ulp = 2.0 ** -8 if qdt == torch.bfloat16 else 2.0 ** -10
    assert np.all(np.abs(qg - q_ref) <= (1e-3 + ulp) * np.abs(q_ref) + 1e-6)
    # cache slots: bit-exact placement; values = the oracle's rounded to the cache type
    kg = kc.float().cpu().numpy()
    vg = vc.float().cpu().numpy()
    kb = kc.view(ib).cpu().numpy()
    vb = vc.view(ib).cpu().numpy()
    written = np.zeros(kb.shape, bool)
    written[layer, :, start:start + m, :] = True
    assert np.all(kb[~written] == np.array(SENT[s.kv_dtype]).astype(kb.dtype))
    assert np.all(vb[~written] == np.array(SENT[s.kv_dtype]).astype(vb.dtype))
    k_sl = kg[layer, :, start:start + m, :].transpose(1, 0, 2).astype(np.float64)
    v_sl = vg[layer, :, start:start + m, :].transpose(1, 0, 2).astype(np.float64)
    cu = {"f32": 0.0, "bf16": 2.0 ** -8, "f16": 2.0 ** -10}[s.kv_dtype]
    assert np.all(np.abs(k_sl - k_ref) <= (1e-3 + cu) * np.abs(k_ref) + 1e-6)
    np.testing.assert_array_equal(v_sl, O.round_to_cache(vr, s.kv_dtype))
    if s.kv_dtype == "f32":  # RoPE / norm arithmetic itself within 1e-3
        assert np.all(np.abs(k_sl - k_ref) <= 1e-3 * np.abs(k_ref) + 1e-7)


# ----------------------------------------------------------------------------- attention
@pytest.mark.parametrize("shape,m,start,qscale", [
    (synth.TINY, 16, 0, 1), (synth.TINY, 9, 40, 1),
    (synth.QWEN3_8B_LAYER, 512, 0, 1), (synth.QWEN3_8B_LAYER, 37, 100, 1),
    (synth.QWEN3_8B_LAYER_LONG, 512, 3584, 1),
    (synth.LLAMA3_8B_INT4_LAYER, 1, 8192, 1), (synth.LLAMA3_8B_INT4_LAYER, 64, 8192, 1),
    # large scores: row maxima jump by more than 2^8 between key tiles, so the running
    # max is raised and the partial output rescaled (for some rows of a warp only)
    (synth.QWEN3_8B_LAYER, 200, 300, 8), (synth.LLAMA3_8B_INT4_LAYER, 1, 8192, 8),
    (synth.TINY, 16, 40, 8),
])
def test_attention_vs_oracle(shape, m, start, qscale):
    s = shape
    nq, nkv, hd = s.n_q_heads, s.n_kv_heads, s.head_dim
    cfg = pf.make_config(s, max_chunk=max(m, 16))
    rng = synth.rng_for(16, m, start)
    L = start + m
    qdt = torch.bfloat16 if s.kv_dtype == "bf16" else torch.float16
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16, "f16": torch.float16}[s.kv_dtype]
    q = torch.from_numpy(qscale * rng.standard_normal((m, nq, hd)).astype(np.float32)).to(qdt).cuda()
    kc = torch.full((1, nkv, s.max_seq, hd), float("nan"), dtype=tdt, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    kc[0, :, :L] = torch.from_numpy(rng.standard_normal((nkv, L, hd)).astype(np.float32)).to(tdt).cuda()
    vc[0, :, :L] = torch.from_numpy(rng.standard_normal((nkv, L, hd)).astype(np.float32)).to(tdt).cuda()
    out = torch.full((m, nq * hd), float("nan"), dtype=torch.float16, device="cuda")
    pf.pf_op_attention(cfg, q, kc, vc, 0, start, m, out)
    torch.cuda.synchronize()
    ref = O.causal_gqa_attention(q.float().cpu().numpy(), kc[0].float().cpu().numpy(),
                                 vc[0].float().cpu().numpy(), start)
    got = out.float().cpu().numpy().reshape(m, nq, hd)
    assert np.all(np.isfinite(got))
    assert rel_l2(got, ref) <= 5e-3


@pytest.mark.parametrize("shape,m,start,n_split,qscale", [
    (synth.LLAMA3_8B_INT4_LAYER, 1, 8192, 19, 1), (synth.LLAMA3_8B_INT4_LAYER, 1, 8192, 19, 8),
    (synth.LLAMA3_8B_INT4_LAYER, 16, 8192, 9, 1), (synth.LLAMA3_8B_INT4_LAYER, 64, 5000, 4, 1),
    # more parts than key tiles: most parts are empty and must not disturb the merge
    (synth.QWEN3_8B_LAYER, 7, 100, 64, 1), (synth.QWEN3_8B_LAYER, 512, 0, 2, 1),
    (dataclasses.replace(synth.TINY, kv_dtype="bf16"), 9, 40, 3, 1),
])
def test_attention_split_vs_oracle(shape, m, start, n_split, qscale):
    # split-KV: the key tiles cut into n_split parts whose partial results are merged by a
    # second kernel (for chunks of at most 2 tokens, by the part that finishes last); the
    # same result as the one-pass kernel up to f32 addition order
    s = shape
    nq, nkv, hd = s.n_q_heads, s.n_kv_heads, s.head_dim
    cfg = pf.make_config(s, max_chunk=max(m, 16))
    rng = synth.rng_for(18, m, start)
    L = start + m
    tdt = torch.bfloat16
    q = torch.from_numpy(qscale * rng.standard_normal((m, nq, hd)).astype(np.float32)).to(tdt).cuda()
    kc = torch.full((1, nkv, s.max_seq, hd), float("nan"), dtype=tdt, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    kc[0, :, :L] = torch.from_numpy(rng.standard_normal((nkv, L, hd)).astype(np.float32)).to(tdt).cuda()
    vc[0, :, :L] = torch.from_numpy(rng.standard_normal((nkv, L, hd)).astype(np.float32)).to(tdt).cuda()
    nbytes = pf.pf_attention_scratch_bytes(cfg, m, n_split)
    assert nbytes == -(-nkv * 4 // 16) * 16 + n_split * m * nq * (hd + 2) * 4
    scratch = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device="cuda")  # NaN-filled partials
    out = torch.full((m, nq * hd), float("nan"), dtype=torch.float16, device="cuda")
    pf.pf_op_attention_split(cfg, q, kc, vc, 0, start, m, n_split, scratch, out)
    if m <= 2:  # merged in the kernel: the arrival counters are left at zero
        assert int(scratch[: nkv * 4].view(torch.int32).abs().sum()) == 0
    one = torch.full_like(out, float("nan"))
    pf.pf_op_attention(cfg, q, kc, vc, 0, start, m, one)
    torch.cuda.synchronize()
    ref = O.causal_gqa_attention(q.float().cpu().numpy(), kc[0].float().cpu().numpy(),
                                 vc[0].float().cpu().numpy(), start)
    got = out.float().cpu().numpy().reshape(m, nq, hd)
    assert np.all(np.isfinite(got))
    assert rel_l2(got, ref) <= 5e-3
    assert rel_l2(got, one.float().cpu().numpy().reshape(m, nq, hd)) <= 5e-3


def test_attention_split_rejects_bad_arguments():
    s = synth.QWEN3_8B_LAYER
    cfg = pf.make_config(s, max_chunk=16)
    q = torch.zeros((4, s.n_q_heads, s.head_dim), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((1, s.n_kv_heads, s.max_seq, s.head_dim), dtype=torch.bfloat16, device="cuda")
    out = torch.zeros((4, s.n_q_heads * s.head_dim), dtype=torch.float16, device="cuda")
    small = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(pf.PfError) as e:
        pf.pf_op_attention_split(cfg, q, kc, kc, 0, 0, 4, 8, small, out)
    assert e.value.status == 11  # PF_ERR_WORKSPACE
    with pytest.raises(pf.PfError) as e:
        pf.pf_op_attention_split(cfg, q, kc, kc, 0, 0, 4, 65, small, out)
    assert e.value.status == 1


# ----------------------------------------------------------------------------- embed / head
def test_embed_bit_exact():
    E = synth.rng_for(17).standard_normal((1000, 256)).astype(np.float32)
    toks = synth.tokens(37, 1000, seed=3)
    x = torch.empty((37, 256), dtype=torch.float32, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    pf.pf_op_embed(dev(E), dev(toks), 37, 256, 1000, x, status)
    pf.pf_status_read(status)
    np.testing.assert_array_equal(x.cpu().numpy(), E[toks])
    # an id outside the vocabulary: zero row and a recorded status, other rows intact
    bad = toks.copy()
    bad[5] = 1000
    pf.pf_op_embed(dev(E), dev(bad), 37, 256, 1000, x, status)
    with pytest.raises(pf.PfError) as e:
        pf.pf_status_read(status)
    assert e.value.status == 5
    got = x.cpu().numpy()
    assert np.all(got[5] == 0) and np.array_equal(np.delete(got, 5, 0), np.delete(E[toks], 5, 0))


@pytest.mark.parametrize("fmt,vocab,h", [("q1", 1000, 256), ("int4", 1000, 256), ("q1", 151936, 4096),
                                         ("q1", 77777, 1024), ("q1", 300, 16384)])
def test_lm_head_vs_oracle(fmt, vocab, h):
    rng = synth.rng_for(18, vocab, h)
    w = synth.quant_weight(fmt, rng, vocab, h)
    x = rng.standard_normal(h).astype(np.float32) * 5
    nw = synth.norm_weight(rng, h)
    logits = torch.full((vocab,), float("nan"), dtype=torch.float32, device="cuda")
    pf.pf_op_lm_head(pf._WFMT[fmt], dev(x), dev(nw), 1e-6, dev(pf.pf_pack_weights_host(w)), vocab,
                     h, logits)
    torch.cuda.synchronize()
    y = O.rmsnorm(x, nw, 1e-6).astype(np.float32)
    ref = O.dequant(w) @ y.astype(np.float64)
    assert rel_l2(logits.cpu().numpy(), ref) <= 1e-4


# ----------------------------------------------------------------------------- greedy argmax
@pytest.mark.parametrize("rows,n,ld", [(1, 151936, 151936), (3, 5000, 5000), (4, 1031, 1040), (2, 1, 1)])
def test_argmax_rows_exact(rows, n, ld):
    """pf_op_argmax (one 1024-thread CTA per row) against the oracle's argmax on the same f32
    values: integer results, so bit-exact; planted ties, NaN and -inf included."""
    rng = synth.rng_for(77, rows, n)
    x = np.full((rows, ld), np.nan, np.float32)  # padding past n must never be read
    x[:, :n] = rng.standard_normal((rows, n)).astype(np.float32)
    if n > 8:
        x[0, n - 1] = x[0, :n].max()      # a tie with an earlier maximum
        x[-1, 3] = np.nan                  # NaN never wins
        x[-1, 5] = np.float32(1e30)        # but a later number may
    if rows > 2:
        x[1, :n] = -np.inf                 # a row of -inf gives 0
    out = torch.full((rows,), -7, dtype=torch.int32, device="cuda")
    pf.pf_op_argmax(dev(x), rows, n, ld, out)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.cpu().numpy(), O.argmax_first(x[:, :n]))
