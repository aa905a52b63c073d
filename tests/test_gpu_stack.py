"""Full-size parity: the 36-layer Qwen3-8B-shaped Q1 stack on a 2048-token prompt fed as four
512-token chunks, final RMSNorm + Q1 LM head on the last position, against the oracle's
logits stored in tests/golden/qwen3_8b_q1_stack_2048_seed0.json (written by
tests/golden/make_stack_golden.py, which calls only the oracle and the seeded generator).

The stored values are every 74th logit, the full logits' L2 norm and argmax. The bar is the
2e-2 relative L2 bound of the f16 / bf16 tensor-core path."""
import json
import os

import numpy as np
import pytest

from quantized_transformer_prefill_q1_gb300 import pf, synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "qwen3_8b_q1_stack_2048_seed0.json")
TOL = 2e-2


def test_full_stack_logits_match_the_oracle():
    gold = json.load(open(GOLDEN))
    s = synth.QWEN3_8B_STACK
    layers, extra = synth.model_inputs(s, seed=0)
    toks = synth.tokens(2048, s.vocab, seed=0)
    dm = pf.DeviceModel(s, layers, extra, max_chunk=512)
    sess = pf.Session(dm)
    logits = torch.full((s.vocab,), float("nan"), dtype=torch.float32, device="cuda")
    for c in range(4):
        sess.prefill_chunk(toks[512 * c: 512 * (c + 1)], 512 * c, logits if c == 3 else None)
    sess.sync()
    assert sess.position == 2048
    got = logits.cpu().numpy().astype(np.float64)
    assert np.isfinite(got).all()
    ref = np.asarray(gold["logits_sample"], np.float64)
    sample = got[::gold["stride"]]
    rel = np.linalg.norm(sample - ref) / np.linalg.norm(ref)
    assert rel <= TOL, rel
    assert abs(np.linalg.norm(got) - gold["logits_l2"]) <= TOL * gold["logits_l2"]
    # the oracle's top token is the GPU's top token or within the tolerance of it
    top = gold["logits_argmax"]
    assert got[top] >= got.max() - TOL * np.abs(got).max()
