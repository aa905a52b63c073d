"""Failure detection on the GPU without a fault: a bounded device wait that nothing
completes must give up, record PF_ERR_DEVICE_TIMEOUT in the status word and leave the
context usable (the next launches still run and still match the oracle)."""
import numpy as np
import pytest

from oracle import prefill_oracle as O
from quantized_transformer_prefill_q1_gb300 import pf, synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)


def test_bounded_wait_times_out_and_context_survives():
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    pf.pf_selftest_bounded_wait(status, 1_000_000, arrive=True)   # completes
    pf.pf_status_read(status)
    pf.pf_selftest_bounded_wait(status, 2_000_000, arrive=False)  # nobody arrives: 2 ms
    with pytest.raises(pf.PfError) as e:
        pf.pf_status_read(status)
    assert e.value.status == 10
    pf.pf_status_read(status)  # the read cleared it
    # the context is intact: a GEMM still runs and matches the oracle
    rng = synth.rng_for(31)
    a = rng.standard_normal((64, 256)).astype(np.float16)
    w = synth.q1_weight(rng, 256, 256)
    out = torch.zeros((64, 256), dtype=torch.float32, device="cuda")
    pf.pf_op_gemm(pf.W_Q1, pf.EPI_STORE_F32, torch.from_numpy(a).cuda(),
                  torch.from_numpy(pf.pf_pack_weights_host(w)).cuda(), 64, 256, 256, out,
                  pf.gemm_scratch(64, 256), 0, status)
    pf.pf_status_read(status)
    ref = a.astype(np.float64) @ O.dequant(w).T
    assert O.rel_l2(out.cpu().numpy(), ref) <= 1e-5


def test_session_reports_device_status():
    s = synth.TINY
    layers, _ = synth.model_inputs(s)
    sess = pf.Session(pf.DeviceModel(s, layers, max_chunk=16))
    # a kernel of this session records a status: the session's sync returns it once
    sess.sync()
    ws_status = sess.ws[:16].view(torch.int32)
    pf.pf_selftest_bounded_wait(ws_status, 1_000_000, arrive=False)
    with pytest.raises(pf.PfError) as e:
        sess.sync()
    assert e.value.status == 10
    sess.sync()
