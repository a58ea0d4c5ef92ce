"""The bounded device waits on the GPU: a wait that nothing completes gives
up after its limit, the error word reports QMM_EDEVICE_TIMEOUT through
qmm_sync_check, and the context stays usable (the next matvec is correct)."""
import time

import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import block_quantized_weight_q6_gb300 as qmm  # noqa: E402


def _matvec_ok():
    N, K = 64, 1024
    W = synth.q6k_matrix(77, N, K)
    x = synth.normal_bf16(78, (2, K))
    y = torch.empty((2, N), dtype=torch.float32, device="cuda")
    qmm.gemv(qmm.Q6_K, torch.from_numpy(W).cuda(),
             torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16), y, N, K)
    torch.cuda.synchronize()
    qmm.sync_check()
    ref, absum = oracle.gemv_float(qmm.Q6_K, W, x, N, K)
    assert (np.abs(y.cpu().numpy().astype(np.float64) - ref) <= 1e-4 * absum + 1e-6).all()


@pytest.mark.parametrize("limit_us", [1000, 20000])
def test_wait_gives_up_and_reports_timeout(limit_us):
    torch.cuda.synchronize()
    qmm.sync_check()  # nothing pending before the probe
    t0 = time.perf_counter()
    qmm.wait_probe(limit_us)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    with pytest.raises(qmm.QmmError) as ei:
        qmm.sync_check()
    assert ei.value.code == qmm.EDEVICE_TIMEOUT
    # the wait lasted its limit (and not much more: it polls the clock every
    # few sleeping try_waits)
    assert waited >= limit_us * 1e-6
    assert waited < limit_us * 1e-6 + 0.5
    # the flag was cleared by the check, and the context still computes
    qmm.sync_check()
    _matvec_ok()


def test_wait_probe_rejects_bad_limits():
    with pytest.raises(qmm.QmmError) as ei:
        qmm.wait_probe(0)
    assert ei.value.code == qmm.EINVAL
    with pytest.raises(qmm.QmmError):
        qmm.wait_probe(2_000_000)
