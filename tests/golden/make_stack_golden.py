"""Writes the expected values for the full-size stack test from the CPU oracle.

Workload: the 36-layer Qwen3-8B-shaped Q1 stack (seed 0), a 2048-token prompt of seeded
token ids fed as 4 chunks of 512, final RMSNorm + Q1 LM head on the last position.
Stored: the logits at every 74th vocabulary index, the full logits' L2 norm and argmax,
and the last position's final hidden row. Calls only the oracle and the seeded input
generator. Run from the repository root: python tests/golden/make_stack_golden.py
"""
import json
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from oracle import prefill_oracle as O  # noqa: E402
from quantized_transformer_prefill_q1_gb300 import synth  # noqa: E402

OUT = os.path.join(ROOT, "tests", "golden", "qwen3_8b_q1_stack_2048_seed0.json")
STRIDE = 74


def main():
    s = synth.QWEN3_8B_STACK
    t0 = time.time()
    layers, extra = synth.model_inputs(s, seed=0)
    toks = synth.tokens(2048, s.vocab, seed=0)
    model = O.OracleModel(s, layers, extra, cache_dequant=False)
    x, logits = model.prefill_layer_major(toks, [512] * 4, True, True)
    idx = np.arange(0, s.vocab, STRIDE)
    rec = {
        "workload": "qwen3-8b-shaped 36-layer Q1 stack, seed 0, 2048 tokens as 4x512 chunks",
        "source": "oracle/prefill_oracle.py via tests/golden/make_stack_golden.py",
        "stride": STRIDE,
        "logits_sample": [float(v) for v in logits[idx]],
        "logits_l2": float(np.linalg.norm(logits.astype(np.float64))),
        "logits_argmax": int(np.argmax(logits)),
        "last_hidden": [float(v) for v in x[-1]],
        "oracle_seconds": round(time.time() - t0, 1),
    }
    with open(OUT, "w") as f:
        json.dump(rec, f)
    print(OUT, rec["oracle_seconds"], "s")


if __name__ == "__main__":
    main()
