"""The GEMM entry point that allocates nothing (pf_op_gemm_static_scratch), checked against
the ordinary entry point (pf_op_gemm with caller-owned scratch) through the C ABI.

Some callers may not allocate device memory: a plug-in whose host application owns every
device allocation, or a service that cannot afford the device synchronisation an
allocation may cause. For them the library keeps the GEMM's scratch in a fixed array of
its own. This file sorts last so that a run stopping at its first failure has run every
other test before it; it passes alone in a fresh process and after the rest."""
import numpy as np
import pytest

from quantized_transformer_prefill_q1_gb300 import pf, synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a GPU", allow_module_level=True)


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


# tolerances of the GEMM parity tests: Q1 5e-5, INT4 1e-3 (f32 outputs), SwiGLU f16 2e-3
TOL = {"q1": 5e-5, "int4": 1e-3}


@pytest.mark.parametrize("fmt", ["q1", "int4"])
@pytest.mark.parametrize("epi", [pf.EPI_STORE_F32, pf.EPI_RESID_ADD, pf.EPI_SWIGLU])
# (128, 512, 1024): 2 tiles on 16 CTAs, so the M > 64 kernel splits every SwiGLU tile and
# passes the partials through the fixed array; (32, 768, 1024): the 16 < M <= 64 kernel, whose
# SwiGLU splits use the array too; (1, 256, 128): the GEMV, which needs no scratch.
@pytest.mark.parametrize("m,n,k", [(300, 768, 1024), (200, 1280, 512), (128, 512, 1024),
                                   (32, 768, 1024), (1, 256, 128)])
def test_static_scratch_matches_gemm_twice(fmt, epi, m, n, k):
    if epi == pf.EPI_SWIGLU and n % 256:
        pytest.skip("SwiGLU needs N = 2I with I % 128 == 0")
    rng = synth.rng_for(41, m, n, k)
    a = dev(rng.standard_normal((m, k)).astype(np.float16))
    packed = dev(pf.pf_pack_weights_host(synth.quant_weight(fmt, rng, n, k),
                                         interleave_gate_up=(epi == pf.EPI_SWIGLU)))
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    swiglu = epi == pf.EPI_SWIGLU
    shape = (m, n // 2) if swiglu else (m, n)
    dtype = torch.float16 if swiglu else torch.float32
    x0 = torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(dtype).cuda()

    def fresh():  # residual input for epilogue 1, garbage that must be overwritten otherwise
        return x0.clone() if epi == pf.EPI_RESID_ADD else torch.full(shape, float("nan"), dtype=dtype,
                                                                      device="cuda")

    ref = fresh()
    pf.pf_op_gemm(pf._WFMT[fmt], epi, a, packed, m, n, k, ref, pf.gemm_scratch(m, n), 0, status)
    pf.pf_status_read(status)
    ref = ref.float().cpu().numpy()
    tol = 2e-3 if swiglu else TOL[fmt]
    for _ in range(2):  # two calls in a row share (and must leave clean) the fixed scratch
        out = fresh()
        pf.pf_op_gemm_static_scratch(pf._WFMT[fmt], epi, a, packed, m, n, k, out, status)
        pf.pf_status_read(status)
        got = out.float().cpu().numpy()
        assert np.isfinite(got).all()
        if epi == pf.EPI_RESID_ADD:
            base = x0.float().cpu().numpy()
            assert rel_l2(got - base, ref - base) <= tol
        assert rel_l2(got, ref) <= tol


def test_static_scratch_rejects_oversized_output():
    a = torch.zeros(16, dtype=torch.float16, device="cuda")
    w = torch.zeros(16, dtype=torch.uint8, device="cuda")
    out = torch.zeros(16, dtype=torch.float32, device="cuda")
    # 1024 x 128 = 131072 output tiles of 128 x 256, beyond the fixed scratch's 16384
    with pytest.raises(pf.PfError) as e:
        pf.pf_op_gemm_static_scratch(pf.W_Q1, pf.EPI_STORE_F32, a, w, 131072, 32768, 128, out)
    assert e.value.status == 2  # PF_ERR_SHAPE
    assert "static GEMM scratch" in str(e.value)
