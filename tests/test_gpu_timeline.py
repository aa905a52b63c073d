"""The per-CTA kernel timeline (pf_timeline_set): one record per CTA of every kernel a
Qwen3-8B-shaped layer launches (graph replay included), well-formed stamps, the capacity
bound, and recording off again once the buffer is unset."""
import numpy as np
import pytest

from quantized_transformer_prefill_q1_gb300 import pf, synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)

M = 512  # four 128-token blocks: the GEMMs run on CTA pairs


@pytest.fixture(scope="module")
def layer_session():
    shape = synth.QWEN3_8B_LAYER
    layers, _ = synth.model_inputs(shape)
    sess = pf.Session(pf.DeviceModel(shape, layers, max_chunk=M), graphs=True)
    x = torch.from_numpy(synth.hidden_input(M, shape.hidden)).cuda()
    sess.prefill_hidden(x.clone(), 0)  # records the graph
    sess.sync()
    return shape, sess, x


def run(sess, x, buf, cap):
    pf.pf_timeline_set(buf, cap)
    sess.set_position(0)
    sess.prefill_hidden(x.clone(), 0)
    sess.sync()
    torch.cuda.synchronize()
    pf.pf_timeline_set(None, 0)


def test_one_record_per_cta(layer_session):
    shape, sess, x = layer_session
    cap = 1 << 16
    buf = torch.zeros(4 + 4 * cap, dtype=torch.int64, device="cuda")
    run(sess, x, buf, cap)
    rec = pf.timeline_records(buf)
    assert int(buf[0]) == len(rec) > 0
    assert np.all(rec["end_ns"] >= rec["start_ns"])
    names = [pf.pf_timeline_kernel_name(int(k)) for k in rec["kernel"]]
    assert None not in names
    count = {n: names.count(n) for n in set(names)}
    # the two RMSNorms: one CTA per token row each
    assert count["rmsnorm_reg"] == 2 * M
    # QKV / O / down on CTA pairs (residual form), gate_up with SwiGLU: an even CTA count
    assert count["gemm_pair_resid"] % 2 == 0 and count["gemm_pair_resid"] > 0
    assert count["gemm_pair_swiglu"] % 2 == 0 and count["gemm_pair_swiglu"] > 0
    g = shape.n_q_heads // shape.n_kv_heads
    assert count["attention_tc"] == (M * g + 127) // 128 * shape.n_kv_heads
    # every CTA index of a launch appears once: the attention's grid has no repeats
    att = rec[np.array(names) == "attention_tc"]
    assert len(np.unique(att["cta"])) == len(att)
    # records end within the prompt's span and the SM ids are plausible
    props = torch.cuda.get_device_properties(0)
    assert np.all(rec["sm"] < props.multi_processor_count)


def test_capacity_and_off(layer_session):
    _, sess, x = layer_session
    cap = 10
    buf = torch.zeros(4 + 4 * cap + 16, dtype=torch.int64, device="cuda")
    run(sess, x, buf, cap)
    total = int(buf[0])
    assert total > cap  # more CTAs ran than the buffer holds ...
    assert len(pf.timeline_records(buf)) == cap  # ... and only `capacity` records were written
    assert int(buf[4 + 4 * cap:].abs().sum()) == 0  # nothing past the last record
    # recording is off once the buffer is unset
    sess.set_position(0)
    sess.prefill_hidden(x.clone(), 0)
    sess.sync()
    torch.cuda.synchronize()
    assert int(buf[0]) == total


def test_rejects_bad_capacity():
    buf = torch.zeros(8, dtype=torch.int64, device="cuda")
    with pytest.raises(pf.PfError):
        pf.pf_timeline_set(buf, 0)
