"""Paged KV cache: blocks of 128 positions placed through a per-session block table.

The layout changes where K / V live, not what is computed, so a paged session must match a
linear session fed the same inputs: the chunked prefill of a Qwen3-8B-shaped layer, and two
sessions of a small stack sharing one pool with disjoint tables, prefill then decode. The
match is to the run-to-run noise of the GEMMs' f32 reduce-adds (their order varies between
launches, and a flipped bf16 rounding of one cached K / V element follows; two linear sessions
differ by 2-3e-4 in the small stack's logits): relative L2 <= 1e-4 for the 8B-shaped layer's
hidden states, <= 2e-3 for the small stack's logits, K / V per head within 5e-3 relative L2;
a K / V row in the wrong slot would be off by the whole row. Slot placement is exact: physical
blocks outside the table keep a sentinel bit pattern. Also the host-side refusals: an
unassigned block, and malformed tables."""
import dataclasses

import numpy as np
import pytest

from quantized_transformer_prefill_q1_gb300 import pf, synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

B = pf.KV_BLOCK
SENT_BF16 = 0x7FC1


def rel_l2(a, b):
    a, b = a.double(), b.double()
    return float((a - b).norm() / b.norm())


def assert_kv_close(got, ref):
    """Per (layer, kv head): relative L2 <= 5e-3 and every element within 5 % of the largest
    |value| (bf16 roundings that flip with the GEMMs' summation order, carried one layer on,
    stay far below both; a K / V row in the wrong slot is off by the whole row)."""
    g, r = got.float(), ref.float()
    for l in range(r.shape[0]):
        for h in range(r.shape[1]):
            gg, rr = g[l, h], r[l, h]
            assert rel_l2(gg, rr) <= 5e-3, (l, h, rel_l2(gg, rr))
            assert float((gg - rr).abs().max()) <= 0.05 * float(rr.abs().max()), (l, h)


def gather(cache, table, n_blocks):
    """The first n_blocks position blocks of a paged cache, in position order."""
    return torch.cat([cache[:, :, t * B:(t + 1) * B] for t in table[:n_blocks]], dim=2)


def test_paged_layer_chunks_match_linear():
    shape = synth.QWEN3_8B_LAYER  # max_seq 4096: 32 position blocks
    layers, _ = synth.model_inputs(shape)
    n = 2048
    x = torch.from_numpy(synth.hidden_input(n, shape.hidden)).cuda()
    lin = pf.Session(pf.DeviceModel(shape, layers, max_chunk=512))
    pool = 40
    table = np.random.default_rng(7).permutation(pool)[:32].astype(np.int32)
    pag = pf.Session(pf.DeviceModel(shape, layers, max_chunk=512, kv_block_pool=pool), block_table=table,
                     kv_fill_bits=SENT_BF16)
    xl, xp = x.clone(), x.clone()
    for off in range(0, n, 512):  # four chunks into a cache holding the earlier ones
        lin.prefill_hidden(xl[off:off + 512], off)
        pag.prefill_hidden(xp[off:off + 512], off)
    lin.sync()
    pag.sync()
    assert pag.position == n
    assert rel_l2(xp, xl) <= 1e-4
    nb = n // B
    assert_kv_close(gather(pag.k, table, nb), lin.k[:, :, :n])
    assert_kv_close(gather(pag.v, table, nb), lin.v[:, :, :n])
    # blocks of positions not yet written, and blocks outside the table, keep the sentinel
    untouched = sorted(set(range(pool)) - set(table[:nb].tolist()))
    for c in (pag.k, pag.v):
        bits = c.view(torch.int16)
        for t in untouched:
            assert bool((bits[:, :, t * B:(t + 1) * B] == SENT_BF16).all()), t


def _stack():
    return dataclasses.replace(synth.TINY, n_layers=2, vocab=5000, max_seq=512, kv_dtype=synth.KV_BF16)


def test_two_sessions_share_one_pool():
    s = _stack()
    layers, extra = synth.model_inputs(s)
    toks_a = synth.tokens(203, s.vocab, seed=1)
    toks_b = synth.tokens(306, s.vocab, seed=2)
    dm_lin = pf.DeviceModel(s, layers, extra, max_chunk=128)
    dm_pag = pf.DeviceModel(s, layers, extra, max_chunk=128, kv_block_pool=8)
    la, lb = pf.Session(dm_lin), pf.Session(dm_lin)
    ta, tb = [5, 2, 7, 0], [1, 6, 3, 4]
    pa = pf.Session(dm_pag, block_table=ta)
    pb = pf.Session(dm_pag, kv=(pa.k, pa.v), block_table=tb)  # one pool, disjoint blocks
    out = {k: torch.empty(s.vocab, dtype=torch.float32, device="cuda") for k in ("la", "lb", "pa", "pb")}
    # interleaved: A's prompt, B's prompt, then decode steps of each in turn
    for sess, toks, key in ((la, toks_a, "la"), (pa, toks_a, "pa"), (lb, toks_b, "lb"), (pb, toks_b, "pb")):
        sess.prefill_chunk(toks[:200] if key[1] == "a" else toks[:300], 0, out[key])
    for sess in (la, pa, lb, pb):
        sess.sync()
    assert rel_l2(out["pa"], out["la"]) <= 2e-3 and rel_l2(out["pb"], out["lb"]) <= 2e-3
    ids_a = torch.from_numpy(toks_a.astype(np.int32)).cuda()
    ids_b = torch.from_numpy(toks_b.astype(np.int32)).cuda()
    for i in range(3):
        la.decode_step(ids_a[200 + i:201 + i], out["la"])
        pa.decode_step(ids_a[200 + i:201 + i], out["pa"])
        lb.decode_step(ids_b[300 + i:301 + i], out["lb"])
        pb.decode_step(ids_b[300 + i:301 + i], out["pb"])
        for sess in (la, pa, lb, pb):
            sess.sync()
        assert rel_l2(out["pa"], out["la"]) <= 2e-3 and rel_l2(out["pb"], out["lb"]) <= 2e-3
    assert pa.position == 203 and pb.position == 303
    assert_kv_close(gather(pa.k, ta, 2)[:, :, :203], la.k[:, :, :203])
    assert_kv_close(gather(pb.v, tb, 3)[:, :, :303], lb.v[:, :, :303])


def test_unassigned_block_is_refused():
    s = _stack()
    layers, extra = synth.model_inputs(s)
    sess = pf.Session(pf.DeviceModel(s, layers, extra, max_chunk=128, kv_block_pool=4),
                      block_table=[3, 1, -1, -1])
    toks = synth.tokens(300, s.vocab, seed=3)
    sess.prefill_chunk(toks[:200], 0)  # positions 0 .. 199: blocks 0 and 1
    sess.sync()
    with pytest.raises(pf.PfError) as e:
        sess.prefill_chunk(toks[200:300], 200)  # reaches block 2
    assert e.value.status == 6  # PF_ERR_KV_CAPACITY
    assert sess.position == 200
    sess.set_block_table([3, 1, 0, -1])
    sess.prefill_chunk(toks[200:300], 200)
    sess.sync()
    assert sess.position == 300


def test_block_table_checks():
    s = _stack()
    layers, extra = synth.model_inputs(s)
    sess = pf.Session(pf.DeviceModel(s, layers, extra, max_chunk=128, kv_block_pool=4))
    for bad in ([0, 1, 2], [0, 1, 2, 4], [0, 1, 1, 2], [0, -2, 1, 2]):
        with pytest.raises(pf.PfError) as e:
            sess.set_block_table(bad)
        assert e.value.status == 2, bad  # PF_ERR_SHAPE
    lin = pf.Session(pf.DeviceModel(s, layers, extra, max_chunk=128))
    with pytest.raises(pf.PfError) as e:
        lin.set_block_table([0, 1, 2, 3])
    assert e.value.status == 8  # PF_ERR_UNSUPPORTED
