"""Whole-path parity through the C ABI sessions: one layer (tiny and Qwen3-8B-shaped),
chunked vs one-shot vs token-by-token, the INT4 Llama-3-8B layer over a filled cache,
a multi-layer stack with embedding and LM head, and the host-side checks of a session.

Per-layer hidden states and logits: relative L2 <= 2e-2 against the oracle (the bound
the target states for the f16/bf16 tensor-core path). KV slot placement: bit-exact
(sentinel bit patterns outside the written range)."""
import dataclasses

import numpy as np
import pytest

from oracle import prefill_oracle as O
from quantized_transformer_prefill_q1_gb300 import pf, synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

TOL = 2e-2
SENT = {"f32": 0x7FC00001, "bf16": 0x7FC1, "f16": 0x7E01}


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def kv_bits(t, kv_dtype):
    return t.view(torch.int32 if kv_dtype == "f32" else torch.int16).cpu().numpy()


def check_kv(sess, model, shape, lo, hi, tol=TOL):
    """Slots [lo, hi) of every layer hold the oracle's values; the rest keep the sentinel."""
    for name, gpu_t, ref in (("k", sess.k, model.k_cache), ("v", sess.v, model.v_cache)):
        bits = kv_bits(gpu_t, shape.kv_dtype)
        written = np.zeros(bits.shape, bool)
        written[:, :, lo:hi] = True
        assert np.all(bits[~written] == np.array(SENT[shape.kv_dtype]).astype(bits.dtype)), name
        got = gpu_t.float().cpu().numpy()[:, :, lo:hi]
        assert O.rel_l2(got, ref[:, :, lo:hi]) <= tol, name


@pytest.mark.parametrize("shape,m", [(synth.TINY, 16), (synth.QWEN3_8B_LAYER, 512)])
@pytest.mark.parametrize("graphs", [True, False])
def test_layer_one_chunk(shape, m, graphs):
    layers, _ = synth.model_inputs(shape)
    x = synth.hidden_input(m, shape.hidden)
    om = O.OracleModel(shape, layers)
    ref, _ = om.prefill(x, [m], False, False)
    sess = pf.Session(pf.DeviceModel(shape, layers, max_chunk=m), kv_fill_bits=SENT[shape.kv_dtype],
                      graphs=graphs)
    xd = dev(x)
    sess.prefill_hidden(xd, 0)
    sess.sync()
    assert sess.position == m
    assert O.rel_l2(xd.cpu().numpy(), ref) <= TOL
    check_kv(sess, om, shape, 0, m)


def test_layer_forward_entry_point():
    s = synth.TINY
    layers, _ = synth.model_inputs(s)
    x = synth.hidden_input(16, s.hidden)
    om = O.OracleModel(s, layers)
    ref = om.layer_forward(0, x, 0)
    sess = pf.Session(pf.DeviceModel(s, layers, max_chunk=16))
    xd = dev(x)
    sess.layer_forward(0, xd, 0)
    sess.sync()
    assert sess.position == 0  # the per-layer call leaves the position to the caller
    assert O.rel_l2(xd.cpu().numpy(), ref) <= TOL


@pytest.mark.parametrize("shape,n,chunks", [
    (synth.TINY, 48, [16, 16, 16]),
    (synth.QWEN3_8B_LAYER_LONG, 4096, [512] * 8),
])
def test_chunked_equals_one_shot_and_oracle(shape, n, chunks):
    layers, _ = synth.model_inputs(shape)
    x = synth.hidden_input(n, shape.hidden)
    om = O.OracleModel(shape, layers)
    ref, _ = om.prefill(x, [n], False, False)
    # one shot: the whole prompt as one micro-batch
    one = pf.Session(pf.DeviceModel(shape, layers, max_chunk=n), kv_fill_bits=SENT[shape.kv_dtype])
    x1 = dev(x)
    one.prefill_hidden(x1, 0)
    one.sync()
    del one
    torch.cuda.empty_cache()
    # chunked: consecutive chunks against the growing cache
    ch = pf.Session(pf.DeviceModel(shape, layers, max_chunk=max(chunks)), kv_fill_bits=SENT[shape.kv_dtype])
    x2 = dev(x)
    off = 0
    for c in chunks:
        ch.prefill_hidden(x2[off:off + c], off)
        off += c
    ch.sync()
    assert ch.position == n
    g1, g2 = x1.cpu().numpy(), x2.cpu().numpy()
    assert O.rel_l2(g1, ref) <= TOL and O.rel_l2(g2, ref) <= TOL
    assert O.rel_l2(g2, g1) <= TOL
    check_kv(ch, om, shape, 0, n)


@pytest.mark.parametrize("shape,n", [(synth.TINY, 24), (synth.QWEN3_8B_LAYER_LONG, 64)])
def test_token_by_token_equals_one_shot(shape, n):
    layers, _ = synth.model_inputs(shape)
    x = synth.hidden_input(n, shape.hidden)
    om = O.OracleModel(shape, layers)
    dec = O.decode_prompt(om, x)
    sess = pf.Session(pf.DeviceModel(shape, layers, max_chunk=16))
    xd = dev(x)
    for t in range(n):
        sess.prefill_hidden(xd[t:t + 1], t)
    sess.sync()
    om2 = O.OracleModel(shape, layers)
    one, _ = om2.prefill(x, [n], False, False)
    assert O.rel_l2(dec, one) <= 1e-6
    assert O.rel_l2(xd.cpu().numpy(), dec) <= TOL


@pytest.mark.parametrize("m", [1, 4, 16, 64, 512])
def test_int4_llama_layer_over_filled_cache(m):
    s = synth.LLAMA3_8B_INT4_LAYER
    P = 8192
    layers, _ = synth.model_inputs(s)
    x = synth.hidden_input(m, s.hidden)
    kvp = synth.kv_prefill_bf16_bits(1, s.n_kv_heads, P, s.head_dim)
    om = O.OracleModel(s, layers)
    om.k_cache[:, :, :P] = synth.bf16_bits_to_f32(kvp["k"])
    om.v_cache[:, :, :P] = synth.bf16_bits_to_f32(kvp["v"])
    om.position = P
    ref, _ = om.prefill(x, [m], False, False)
    sess = pf.Session(pf.DeviceModel(s, layers, max_chunk=m))
    sess.k[:, :, :P].view(torch.int16).copy_(dev(kvp["k"].view(np.int16)))
    sess.v[:, :, :P].view(torch.int16).copy_(dev(kvp["v"].view(np.int16)))
    sess.set_position(P)
    xd = dev(x)
    sess.prefill_hidden(xd, P)
    sess.sync()
    assert sess.position == P + m
    assert O.rel_l2(xd.cpu().numpy(), ref) <= TOL


def _small_stack(n_layers=3, vocab=5000):
    return dataclasses.replace(synth.TINY, n_layers=n_layers, vocab=vocab, max_seq=128)


def test_stack_tokens_logits_and_chunking():
    s = _small_stack()
    layers, extra = synth.model_inputs(s)
    toks = synth.tokens(96, s.vocab)
    om = O.OracleModel(s, layers, extra)
    _, ref_logits = om.prefill(toks, [96], True, True)
    dm = pf.DeviceModel(s, layers, extra, max_chunk=32)
    sess = pf.Session(dm, kv_fill_bits=SENT[s.kv_dtype])
    logits = torch.full((s.vocab,), float("nan"), dtype=torch.float32, device="cuda")
    sess.prefill_chunk(toks[:40], 0)          # split internally into 32 + 8
    sess.prefill_chunk(toks[40:], 40, logits)  # 32 + 24, head on the last micro-batch
    sess.sync()
    assert sess.position == 96
    assert O.rel_l2(logits.cpu().numpy(), ref_logits) <= TOL
    check_kv(sess, om, s, 0, 96)
    # end to end from host memory
    sess.set_position(0)
    host = np.full(s.vocab, np.nan, np.float32)
    sess.prefill_tokens_host(toks, 0, host)
    assert O.rel_l2(host, ref_logits) <= TOL


def test_decode_steps_match_oracle_prefixes():
    """pf_decode_step: after a 32-token prefill, each step feeds the next token from device
    memory at the session's position; its logits equal the oracle's last-position logits of
    the prefix (prefill = decode, the pages' token-by-token path)."""
    s = _small_stack()
    layers, extra = synth.model_inputs(s)
    toks = synth.tokens(38, s.vocab)
    om = O.OracleModel(s, layers, extra)
    dm = pf.DeviceModel(s, layers, extra, max_chunk=32)
    sess = pf.Session(dm, kv_fill_bits=SENT[s.kv_dtype])
    logits = torch.full((s.vocab,), float("nan"), dtype=torch.float32, device="cuda")
    sess.prefill_chunk(toks[:32], 0)
    tok_d = torch.from_numpy(toks.astype(np.int32)).cuda()
    for n in range(32, 38):
        sess.decode_step(tok_d[n:n + 1], logits)
        sess.sync()
        assert sess.position == n + 1
        _, ref = O.OracleModel(s, layers, extra).prefill(toks[:n + 1], [n + 1], True, True)
        assert O.rel_l2(logits.cpu().numpy(), ref) <= TOL
    om.prefill(toks, [38], True, True)
    check_kv(sess, om, s, 0, 38)
    with pytest.raises(pf.PfError) as e:  # a decode step needs a logits buffer
        pf.check(pf.lib().pf_decode_step(sess.h, tok_d.data_ptr(), None, None))
    assert e.value.status == 7  # PF_ERR_LOGITS
    assert sess.position == 38


def test_session_validation_leaves_state_unchanged():
    s = _small_stack(n_layers=1, vocab=100)
    layers, extra = synth.model_inputs(s)
    sess = pf.Session(pf.DeviceModel(s, layers, extra, max_chunk=16))
    logits = torch.empty(s.vocab, dtype=torch.float32, device="cuda")
    with pytest.raises(pf.PfError) as e:
        sess.prefill_chunk(np.array([], np.int32), 0)
    assert e.value.status == 3
    with pytest.raises(pf.PfError) as e:
        sess.prefill_chunk(np.array([1, 2], np.int32), 5)
    assert e.value.status == 4
    with pytest.raises(pf.PfError) as e:
        sess.prefill_chunk(np.array([1, 100], np.int32), 0)
    assert e.value.status == 5
    with pytest.raises(pf.PfError) as e:
        sess.prefill_chunk(np.arange(129, dtype=np.int32) % 100, 0)
    assert e.value.status == 6
    assert sess.position == 0
    sess.prefill_chunk(np.array([1, 2, 3], np.int32), 0, logits)
    sess.sync()
    assert sess.position == 3
    with pytest.raises(pf.PfError) as e:
        sess.prefill_chunk(np.array([1], np.int32), 0)
    assert e.value.status == 4 and sess.position == 3


@pytest.mark.parametrize("m", [8, 24, 72])
def test_verify_tail_matches_oracle(m):
    """pf_prefill_verify after a 16-token prefill: logits of every position against the
    oracle's verify tail (the LM head as a GEMV, small-M and large GEMM by M), and ids equal
    to the argmax of the GPU's own logits (the decision taken in the kernel's precision);
    the oracle's choice is the GPU's or within the tolerance of it."""
    s = _small_stack()
    layers, extra = synth.model_inputs(s)
    toks = synth.tokens(16 + m, s.vocab)
    om = O.OracleModel(s, layers, extra)
    om.prefill(toks[:16], [16], True, False)
    ref, _ = om.prefill_verify(toks[16:])
    sess = pf.Session(pf.DeviceModel(s, layers, extra, max_chunk=72), kv_fill_bits=SENT[s.kv_dtype])
    sess.prefill_chunk(toks[:16], 0)
    lg = torch.full((m, s.vocab), float("nan"), dtype=torch.float32, device="cuda")
    ids = torch.full((m,), -1, dtype=torch.int32, device="cuda")
    sess.prefill_verify(dev(toks[16:].astype(np.int32)), 16, lg, ids)
    sess.sync()
    assert sess.position == 16 + m
    got = lg.cpu().numpy()
    assert np.isfinite(got).all()
    for t in range(m):
        assert O.rel_l2(got[t], ref[t]) <= TOL, t
        top = int(O.argmax_first(ref[t]))
        assert got[t, top] >= got[t].max() - TOL * np.abs(got[t]).max()
    np.testing.assert_array_equal(ids.cpu().numpy(), O.argmax_first(got))
    check_kv(sess, om, s, 0, 16 + m)


def test_greedy_decode_chain_on_device():
    """pf_decode_step_greedy: five steps enqueued back to back, each reading the token the
    previous one chose on the device; every chosen token is the argmax of its step's logits,
    and the logits match the oracle's last-position logits of the prefix actually fed."""
    s = _small_stack()
    layers, extra = synth.model_inputs(s)
    toks = synth.tokens(16, s.vocab)
    sess = pf.Session(pf.DeviceModel(s, layers, extra, max_chunk=16), kv_fill_bits=SENT[s.kv_dtype])
    sess.prefill_chunk(toks[:15], 0)
    K = 5
    chain = torch.zeros(K + 1, dtype=torch.int32, device="cuda")
    chain[0] = int(toks[15])
    lg = torch.full((K, s.vocab), float("nan"), dtype=torch.float32, device="cuda")
    for i in range(K):
        sess.decode_step_greedy(chain[i:i + 1], chain[i + 1:i + 2], lg[i])
    sess.sync()
    assert sess.position == 15 + K
    got = lg.cpu().numpy()
    ch = chain.cpu().numpy()
    np.testing.assert_array_equal(ch[1:], O.argmax_first(got))
    fed = np.concatenate([toks[:15], ch[:K]]).astype(np.int64)
    for i in range(K):
        _, ref = O.OracleModel(s, layers, extra).prefill(fed[:16 + i], [16 + i], True, True)
        assert O.rel_l2(got[i], ref) <= TOL, i
