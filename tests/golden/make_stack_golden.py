"""Writes the expected values for the full-size stack test from the CPU oracle.

Workload: the 36-layer Qwen3-8B-shaped Q1 stack (seed 0), a 2048-token prompt of seeded
token ids fed as 4 chunks of 512, final RMSNorm + Q1 LM head on the last position.

Stored in qwen3_8b_q1_stack_2048_seed0.npz:
  logits       f32 [151936]        every logit of the last position
  last_hidden  f32 [4096]          the last position's hidden row after layer 35
  kv_layers    int [3]             layers 0, 17, 35
  kv_positions int [5]             positions 0, 511, 512, 1535, 2047 (chunk edges)
  k_slots      f32 [3, 8, 5, 128]  K cache slots [layer][kv head][position][hd], values
  v_slots      f32 [3, 8, 5, 128]  already rounded to bf16 (the cache's element type)
plus a small JSON beside it (workload, argmax, norms, oracle time).

Calls only the oracle and the seeded input generator. Run from the repository root:
python tests/golden/make_stack_golden.py (about 15-30 minutes of CPU).
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

HERE = os.path.join(ROOT, "tests", "golden")
OUT_NPZ = os.path.join(HERE, "qwen3_8b_q1_stack_2048_seed0.npz")
OUT_JSON = os.path.join(HERE, "qwen3_8b_q1_stack_2048_seed0.json")
KV_LAYERS = (0, 17, 35)
KV_POSITIONS = (0, 511, 512, 1535, 2047)


def main():
    s = synth.QWEN3_8B_STACK
    t0 = time.time()
    layers, extra = synth.model_inputs(s, seed=0)
    toks = synth.tokens(2048, s.vocab, seed=0)
    model = O.OracleModel(s, layers, extra, cache_dequant=False)
    x, logits = model.prefill_layer_major(toks, [512] * 4, True, True)
    li = np.asarray(KV_LAYERS)
    pi = np.asarray(KV_POSITIONS)
    k_slots = model.k_cache[li][:, :, pi, :].astype(np.float32)
    v_slots = model.v_cache[li][:, :, pi, :].astype(np.float32)
    np.savez(OUT_NPZ, logits=logits.astype(np.float32), last_hidden=x[-1].astype(np.float32),
             kv_layers=li, kv_positions=pi, k_slots=k_slots, v_slots=v_slots)
    rec = {
        "workload": "qwen3-8b-shaped 36-layer Q1 stack, seed 0, 2048 tokens as 4x512 chunks",
        "source": "oracle/prefill_oracle.py via tests/golden/make_stack_golden.py",
        "arrays": os.path.basename(OUT_NPZ),
        "logits_l2": float(np.linalg.norm(logits.astype(np.float64))),
        "logits_argmax": int(np.argmax(logits)),
        "last_hidden_l2": float(np.linalg.norm(x[-1].astype(np.float64))),
        "oracle_seconds": round(time.time() - t0, 1),
    }
    with open(OUT_JSON, "w") as f:
        json.dump(rec, f, indent=1)
    print(OUT_NPZ, rec["oracle_seconds"], "s")


if __name__ == "__main__":
    main()
