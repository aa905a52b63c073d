"""bench.py's output contract, checked on the CPU through its reference arm (the oracle
timed on the host): one JSON line whose keys and types the round-end tooling reads."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert "workload" in d["config"]


def test_timeline_labels_follow_the_layer_order():
    """bench.py's timeline case names each launch by its place in the layer: the first
    RMSNorm of a layer precedes the QKV GEMM, attention precedes the O GEMM, gate_up
    precedes down."""
    sys.path.insert(0, ROOT)
    import bench
    layer = ["rmsnorm_reg", "gemm_pair_resid", "qk_norm_rope_kv", "attention_tc", "gemm_pair_resid",
             "rmsnorm_reg", "gemm_pair_swiglu", "gemm_pair_resid"]
    got = bench.timeline_classes(["set_int", "embed"] + layer * 2 + ["lm_head_q1"])
    one = ["rmsnorm_attn", "gemm_qkv", "qk_norm_rope_kv", "attention", "gemm_o", "rmsnorm_ffn", "gemm_gate_up",
           "gemm_down"]
    assert got == ["set_int", "embed"] + one * 2 + ["lm_head_q1"]
    # with the norms as the GEMMs' prologues (no norm kernels), and a ring store after attention
    fused = ["gemm_pair_resid", "qk_norm_rope_kv", "attention_tc", "ring_store", "gemm_pair_resid",
             "gemm_pair_swiglu", "gemm_pair_resid"]
    got = bench.timeline_classes(["embed"] + fused * 2)
    one = ["gemm_qkv", "qk_norm_rope_kv", "attention", "ring_store", "gemm_o", "gemm_gate_up", "gemm_down"]
    assert got == ["embed"] + one * 2
