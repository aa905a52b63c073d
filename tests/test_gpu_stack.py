"""Full-size parity: the 36-layer Qwen3-8B-shaped Q1 stack on a 2048-token prompt fed as four
512-token chunks, final RMSNorm + Q1 LM head on the last position, against the oracle's values
stored in tests/golden/qwen3_8b_q1_stack_2048_seed0.npz (written by
tests/golden/make_stack_golden.py, which calls only the oracle and the seeded generator).

Checked element by element:
  * all 151936 logits: relative L2 <= 2e-2 (the bound of the f16 / bf16 tensor-core path),
    and the oracle's top token scores within that tolerance of the GPU's maximum;
  * the last position's hidden row after layer 35: relative L2 <= 2e-2;
  * K and V cache slots of layers 0, 17 and 35 at positions 0, 511, 512, 1535 and 2047 (the
    chunk edges). Layer 0 sees the exact embedding rows, so its slots differ from the
    oracle's only by the f16 GEMM operand rounding (about 2^-12 relative) and the two sides'
    rounding to bf16: every element within 1e-3 of its slot's largest magnitude plus one
    bf16 ulp of the oracle's value. Deeper layers carry the accumulated f16 / bf16 error of
    the layers before them: relative L2 <= 2e-2 over the layer's sampled slots (the per-layer
    hidden-state bound), and <= 4e-2 for any single slot of 128 values.
"""
import json
import os

import numpy as np
import pytest

from quantized_transformer_prefill_q1_gb300 import pf, synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
GOLDEN = os.path.join(HERE, "qwen3_8b_q1_stack_2048_seed0.npz")
GOLDEN_META = os.path.join(HERE, "qwen3_8b_q1_stack_2048_seed0.json")
TOL = 2e-2


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def bf16_ulp(v):
    """Spacing of bf16 numbers at |v| (8 significant bits)."""
    a = np.maximum(np.abs(np.asarray(v, np.float64)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


@pytest.fixture(scope="module")
def stack_run():
    gold = dict(np.load(GOLDEN))
    meta = json.load(open(GOLDEN_META))
    s = synth.QWEN3_8B_STACK
    layers, extra = synth.model_inputs(s, seed=0)
    toks = synth.tokens(2048, s.vocab, seed=0)
    emb_rows = extra["embed"][toks]
    dm = pf.DeviceModel(s, layers, extra, max_chunk=512)
    del layers
    sess = pf.Session(dm)
    logits = torch.full((s.vocab,), float("nan"), dtype=torch.float32, device="cuda")
    for c in range(4):  # token ids from the host, the embedding on the GPU
        sess.prefill_chunk(toks[512 * c: 512 * (c + 1)], 512 * c, logits if c == 3 else None)
    sess.sync()
    assert sess.position == 2048
    li = torch.as_tensor(gold["kv_layers"], dtype=torch.long, device="cuda")
    pi = torch.as_tensor(gold["kv_positions"], dtype=torch.long, device="cuda")
    k = sess.k[li][:, :, pi].float().cpu().numpy()
    v = sess.v[li][:, :, pi].float().cpu().numpy()
    got_logits = logits.cpu().numpy()
    # the last hidden row: the same prompt again from its embedding rows (hidden input, the
    # rows updated in place), which leaves the final hidden rows in the caller's buffer
    sess.set_position(0)
    x = torch.from_numpy(np.ascontiguousarray(emb_rows)).cuda()
    sess.prefill_hidden(x, 0)
    sess.sync()
    last = x[-1].cpu().numpy()
    sess.close()
    return gold, meta, got_logits, last, k, v


def test_full_stack_logits_match_the_oracle(stack_run):
    gold, meta, got, _, _, _ = stack_run
    ref = gold["logits"].astype(np.float64)
    assert np.isfinite(got).all()
    assert rel_l2(got, ref) <= TOL
    top = meta["logits_argmax"]
    assert top == int(np.argmax(ref))
    assert got[top] >= got.max() - TOL * np.abs(got).max()


def test_full_stack_last_hidden_matches_the_oracle(stack_run):
    gold, _, _, last, _, _ = stack_run
    assert np.isfinite(last).all()
    assert rel_l2(last, gold["last_hidden"]) <= TOL


@pytest.mark.parametrize("name", ["k", "v"])
def test_full_stack_kv_slots_match_the_oracle(stack_run, name):
    gold, _, _, _, k, v = stack_run
    got = {"k": k, "v": v}[name]
    ref = gold[name + "_slots"].astype(np.float64)
    assert got.shape == ref.shape
    for i, layer in enumerate(gold["kv_layers"]):
        if layer != 0:
            assert rel_l2(got[i], ref[i]) <= TOL, (name, int(layer))
        for h in range(ref.shape[1]):
            for j, pos in enumerate(gold["kv_positions"]):
                g, r = got[i, h, j], ref[i, h, j]
                if layer == 0:
                    bound = 1e-3 * np.abs(r).max() + bf16_ulp(r)
                    assert np.all(np.abs(g - r) <= bound), (name, int(layer), h, int(pos))
                else:
                    assert rel_l2(g, r) <= 2 * TOL, (name, int(layer), h, int(pos))
