"""qmm_gemv_noalloc: the matvec for callers that cannot allocate device memory
when they call (engine-owned memory, allocator-free inference loops). It keeps
its scratch in a fixed array inside the library instead of a caller-provided
workspace. Here it is called through the C interface and compared with
qmm_gemv on the same inputs, twice in a row (the second call finds the first
call's leftovers in the shared array).

This file is collected last on purpose, so that a run stopping at its first
failure has already run every other test."""
import ctypes as C

import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import block_quantized_weight_q6_gb300 as qmm  # noqa: E402


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _x(x):
    return _dev(x.view(np.int16)).view(torch.bfloat16) if x.dtype == np.uint16 else _dev(x)


CASES = [
    # (format, N, K, B, activation mode, activations): short N (split-K
    # partials in scratch), q8 (quantized activation tile and scales in
    # scratch), batch 8 float (bf16 activation tile in scratch)
    (qmm.Q6_K, 1024, 4096, 1, qmm.ACT_FLOAT, "f32"),
    (qmm.Q4_0, 512, 4096, 8, qmm.ACT_Q8, "bf16"),
    (qmm.Q8_0, 256, 2048, 8, qmm.ACT_FLOAT, "bf16"),
]


@pytest.mark.parametrize("fmt,N,K,B,act,xdt", CASES)
def test_noalloc_matches_gemv_twice(fmt, N, K, B, act, xdt):
    W = synth.matrix(fmt, 301 + fmt, N, K)
    x = synth.normal_f32(302, (B, K)) if xdt == "f32" else synth.normal_bf16(302, (B, K))
    Wt, xt = _dev(W), _x(x)
    ref = torch.empty((B, N), dtype=torch.float32, device="cuda")
    qmm.gemv(fmt, Wt, xt, ref, N, K, act)
    torch.cuda.synchronize()
    if act == qmm.ACT_Q8:
        xq, s = oracle.quantize_q8(x)
        _, absum = oracle.gemv_q8(fmt, W, xq, s, N, K)
    else:
        _, absum = oracle.gemv_float(fmt, W, x, N, K)
    bound = 1e-4 * absum + 1e-6
    code = fmt | (qmm.X_BF16 if xdt == "bf16" else qmm.X_F32) | act
    stream = torch.cuda.current_stream()
    assert qmm.lib.qmm_set_stream(C.c_void_p(stream.cuda_stream)) == qmm.OK
    for _ in range(2):
        y = torch.full((B, N), float("nan"), dtype=torch.float32, device="cuda")
        rc = qmm.lib.qmm_gemv_noalloc(code, C.c_void_p(Wt.data_ptr()), C.c_void_p(xt.data_ptr()),
                                      C.c_void_p(y.data_ptr()), N, K, B)
        assert rc == qmm.OK, qmm.lib.qmm_last_error().decode()
        torch.cuda.synchronize()
        qmm.sync_check()
        diff = np.abs(y.cpu().numpy().astype(np.float64) - ref.cpu().numpy().astype(np.float64))
        assert (diff <= bound).all()


def test_noalloc_refuses_shapes_beyond_its_scratch():
    """16 batch rows of 262144 quantized activations (4 MiB of int8 plus their
    scales) need more than the fixed array holds: refused before anything is
    launched"""
    N, K, B = 16, 262144, 16
    code = qmm.Q6_K | qmm.X_BF16 | qmm.ACT_Q8
    assert qmm.lib.qmm_workspace_bytes(code, B, N, K) > 4 << 20
    W = torch.zeros(N * (K // 256) * 210, dtype=torch.uint8, device="cuda")
    x = torch.zeros((B, K), dtype=torch.bfloat16, device="cuda")
    y = torch.zeros((B, N), dtype=torch.float32, device="cuda")
    rc = qmm.lib.qmm_gemv_noalloc(code, C.c_void_p(W.data_ptr()), C.c_void_p(x.data_ptr()),
                                  C.c_void_p(y.data_ptr()), N, K, B)
    assert rc == qmm.ENOWORKSPACE
    assert "scratch" in qmm.lib.qmm_last_error().decode()
