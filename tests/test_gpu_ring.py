"""Ring / sink KV cache on the GPU (turbospark-runtime 0.3.0 families/llama/prefill.rs, the
batch-attention input contract's ring_capacity R and sink_count S) against the oracle's ring
reading: positions 0 .. S-1 keep slots 0 .. S-1, a later position p goes to slot
S + (p - S) mod (R - S), and the query at p attends to the sinks and the R - S most recent
positions up to p, RoPE at absolute positions.

Checked through the C ABI sessions:
  * hidden rows after the layers: relative L2 <= 2e-2 against the oracle's batched form (a
    linear history with the window + sink mask), for one-shot, chunked and token-by-token
    runs, the last against the oracle's per-token form that reads a physical ring;
  * the ring's slots after the prompt: slots the oracle never wrote keep the NaN sentinel
    bits (placement exact), written slots hold the oracle's values of the right position
    (relative L2 <= 2e-2 per slot, the per-layer bound);
  * GPU one-shot = GPU chunked on the Qwen3-8B-shaped layer (R 1024, S 4, 2048 positions).
"""
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
SENT_BF16 = 0x7FC1


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def check_ring(sess, om, shape):
    """Every layer's ring slots against the oracle's ring after the same positions."""
    for l in range(shape.n_layers):
        rk, rv = om.ring_cache(l)
        for name, gpu_t, ref in (("k", sess.k, rk), ("v", sess.v, rv)):
            bits = gpu_t[l].view(torch.int16).cpu().numpy()
            got = gpu_t[l].float().cpu().numpy()
            empty = np.isnan(ref)
            assert np.all(bits[empty] == np.int16(SENT_BF16)), (name, l)
            for h in range(ref.shape[0]):
                for slot in range(ref.shape[1]):
                    if not empty[h, slot, 0]:
                        assert O.rel_l2(got[h, slot], ref[h, slot]) <= TOL, (name, l, h, slot)


TINY_RING = dataclasses.replace(synth.TINY, kv_dtype="bf16", n_layers=2, max_seq=64)


@pytest.mark.parametrize("R,S,n,chunks,max_chunk", [
    (10, 2, 40, [16, 5, 19], 16),   # wraps several times; chunks longer than the window
    (10, 0, 23, [23], 32),          # no sinks, one chunk of more than the ring
    (32, 3, 20, [7, 13], 16),       # never wraps: slots past position 19 stay unwritten
    (65, 1, 64, [64], 64),          # a window wider than the chunk's CTA tile of 64 tokens
])
def test_ring_prefill_tiny(R, S, n, chunks, max_chunk):
    s = TINY_RING
    layers, _ = synth.model_inputs(s)
    x = synth.hidden_input(n, s.hidden)
    om = O.OracleModel(s, layers, ring_capacity=R, sink_count=S)
    ref, _ = om.prefill(x, chunks, False, False)
    dm = pf.DeviceModel(s, layers, max_chunk=max_chunk, ring_capacity=R, sink_count=S)
    sess = pf.Session(dm, kv_fill_bits=SENT_BF16)
    assert tuple(sess.k.shape) == (s.n_layers, s.n_kv_heads, R, s.head_dim)
    xd = dev(x)
    off = 0
    for c in chunks:
        sess.prefill_hidden(xd[off:off + c], off)
        off += c
    sess.sync()
    assert sess.position == n
    assert O.rel_l2(xd.cpu().numpy(), ref) <= TOL
    check_ring(sess, om, s)


def test_ring_token_by_token_matches_physical_ring():
    # the GPU prefills 6 tokens, then takes one token per call past the ring's capacity
    # several times; the oracle runs every position through its per-token form, which reads a
    # physical ring (one-shot = chunked = per-token is pinned for the oracle itself)
    R, S = 10, 2
    s = TINY_RING
    layers, _ = synth.model_inputs(s)
    x = synth.hidden_input(30, s.hidden, stream=3)
    om = O.OracleModel(s, layers, ring_capacity=R, sink_count=S)
    ref = O.decode_prompt(om, x, start=0)  # every position through the physical ring
    dm = pf.DeviceModel(s, layers, max_chunk=8, ring_capacity=R, sink_count=S)
    sess = pf.Session(dm, kv_fill_bits=SENT_BF16)
    xd = dev(x)
    sess.prefill_hidden(xd[:6], 0)
    for t in range(6, 30):
        sess.prefill_hidden(xd[t:t + 1], t)
    sess.sync()
    assert sess.position == 30
    got = xd.cpu().numpy()
    assert O.rel_l2(got[:6], ref[:6]) <= TOL
    assert O.rel_l2(got[6:], ref[6:]) <= TOL
    for l in range(s.n_layers):  # the physical ring the per-token form kept
        for name, gpu_t, ring in (("k", sess.k, om.ring_k), ("v", sess.v, om.ring_v)):
            g = gpu_t[l].float().cpu().numpy()
            for h in range(s.n_kv_heads):
                for slot in range(R):
                    assert O.rel_l2(g[h, slot], ring[l, h, slot]) <= TOL, (name, l, h, slot)


def test_ring_qwen3_layer_one_shot_equals_chunked_and_oracle():
    R, S, n = 1024, 4, 2048
    s = dataclasses.replace(synth.QWEN3_8B_LAYER, max_seq=n)
    layers, _ = synth.model_inputs(s)
    x = synth.hidden_input(n, s.hidden, stream=5)
    om = O.OracleModel(s, layers, ring_capacity=R, sink_count=S)
    ref, _ = om.prefill(x, [512] * 4, False, False)
    outs = []
    for max_chunk, chunks in ((512, [512] * 4), (2048, [2048])):
        sess = pf.Session(pf.DeviceModel(s, layers, max_chunk=max_chunk, ring_capacity=R, sink_count=S),
                          kv_fill_bits=SENT_BF16)
        xd = dev(x)
        off = 0
        for c in chunks:
            sess.prefill_hidden(xd[off:off + c], off)
            off += c
        sess.sync()
        assert sess.position == n
        got = xd.cpu().numpy()
        assert O.rel_l2(got, ref) <= TOL
        check_ring(sess, om, s)
        outs.append(got)
        sess.close()
    # the GPU's own one-shot and chunked runs: same arithmetic up to GEMM split order
    assert O.rel_l2(outs[1], outs[0]) <= 5e-3


def test_ring_config_checks():
    s = TINY_RING
    layers, _ = synth.model_inputs(s)
    for R, S in ((4, 4), (4, 5), (0, 1), (-1, 0)):
        with pytest.raises(pf.PfError):
            pf.Session(pf.DeviceModel(s, layers, max_chunk=8, ring_capacity=R, sink_count=S))
    f32 = dataclasses.replace(s, kv_dtype="f32")
    with pytest.raises(pf.PfError) as e:
        pf.Session(pf.DeviceModel(f32, synth.model_inputs(f32)[0], max_chunk=8, ring_capacity=8, sink_count=1))
    assert e.value.status == 8  # PF_ERR_UNSUPPORTED: the ring needs the 16-bit tensor-core kernel
    assert pf.lib().pf_kv_bytes(pf.ctypes.byref(pf.make_config(s, 8, ring_capacity=12, sink_count=2))) == \
        s.n_layers * s.n_kv_heads * 12 * s.head_dim * 2
