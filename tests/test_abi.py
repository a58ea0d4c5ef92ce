"""The C interface without a GPU: libqmm builds and loads, exports every
function include/qmm.h declares, and rejects bad arguments on the host before
anything is launched (so no CUDA call is made)."""
import ctypes as C
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qmm.h")


@pytest.fixture(scope="module")
def L():
    import importlib
    build = importlib.import_module("block_quantized_weight_q6_gb300.build")
    build.build()
    import block_quantized_weight_q6_gb300 as q
    q.lib.qmm_init()  # forces the load
    return q


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*([A-Za-z_]\w*)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ["qmm_gemv", "qmm_gemm", "moe_gemv", "qmm_plane_build", "qmm_quantize_q8",
              "qmm_route_topk_softmax", "qmm_liveness_read", "qmm_last_error"]:
        assert n in names


def test_library_exports_every_declared_function(L):
    handle = C.CDLL(L.build.LIB)
    missing = [n for n in declared_functions() if not hasattr(handle, n)]
    assert not missing, missing


def _rc(L, fn, *args):
    rc = getattr(L.lib, fn)(*args)
    return rc, L.lib.qmm_last_error().decode()


FAKE = C.c_void_p(0x10000)  # never dereferenced: every case below fails validation first
MIS = C.c_void_p(0x10008)


@pytest.mark.parametrize("case,expect", [
    ("null_W", -1), ("null_y", -1), ("zero_N", -1), ("zero_K", -1), ("B0", -1), ("B17", -1),
    ("bad_fmt", -1), ("bad_x", -1), ("bad_mode", -1), ("unknown_bits", -1),
    ("K_not_block_q6k", -3), ("K_not_block_q4", -3), ("misaligned_W", -3), ("misaligned_x", -3),
])
def test_gemv_argument_errors(L, case, expect):
    fmt, W, x, y, N, K, B = L.Q6_K, FAKE, FAKE, FAKE, 64, 256, 1
    if case == "null_W": W = None
    if case == "null_y": y = None
    if case == "zero_N": N = 0
    if case == "zero_K": K = 0
    if case == "B0": B = 0
    if case == "B17": B = 17
    if case == "bad_fmt": fmt = 0x06
    if case == "bad_x": fmt = L.Q6_K | 0x200
    if case == "bad_mode": fmt = L.Q6_K | 0x2000
    if case == "unknown_bits": fmt = L.Q6_K | 0x10000
    if case == "K_not_block_q6k": K = 288
    if case == "K_not_block_q4": fmt, K = L.Q4_0, 48
    if case == "misaligned_W": W = MIS
    if case == "misaligned_x": x = MIS
    rc, msg = _rc(L, "qmm_gemv", fmt, W, x, y, N, K, B)
    assert rc == expect, (case, rc, msg)
    assert msg


def test_kquant_formats_only_on_the_fp16_mma_matvec(L):
    """Q4_K / Q2_K: accepted by the matvecs for bf16 activations in float
    mode, B <= 8, N % 8 == 0; refused with QMM_EUNSUPPORTED (-2) elsewhere,
    on the host, before anything is launched"""
    bf = L.X_BF16
    for f in (L.Q4_K, L.Q2_K):
        assert _rc(L, "qmm_gemv", f | L.X_F32, FAKE, FAKE, FAKE, 64, 256, 1)[0] == -2   # fp32 x
        assert _rc(L, "qmm_gemv", f | bf | L.ACT_Q8, FAKE, FAKE, FAKE, 64, 256, 1)[0] == -2
        assert _rc(L, "qmm_gemv", f | bf, FAKE, FAKE, FAKE, 64, 256, 9)[0] == -2      # B > 8
        assert _rc(L, "qmm_gemv", f | bf, FAKE, FAKE, FAKE, 12, 256, 1)[0] == -2      # N % 8
        assert _rc(L, "qmm_gemv", f | bf, FAKE, FAKE, FAKE, 64, 288, 1)[0] == -3      # K % 256
        assert _rc(L, "qmm_gemm", f, FAKE, FAKE, FAKE, 128, 64, 256, None)[0] == -2
        assert _rc(L, "qmm_gemv_noalloc", f | bf, FAKE, FAKE, FAKE, 64, 256, 1)[0] == -2
        assert _rc(L, "moe_gemv", f | bf, None, None, None, None, None)[0] == -2
        assert L.lib.qmm_workspace_bytes(f | L.X_F32, 1, 64, 256) == 0


def test_moe_prefill_argument_errors(L):
    """host-side checks of moe_prefill, before anything is launched"""
    P = C.c_void_p * 2
    ptrs = P(FAKE, FAKE)
    m = L.MoeExperts()
    m.n_experts, m.hidden, m.inter, m.top_k, m.n_tokens = 2, 256, 128, 1, 4
    m.w_gate = m.w_up = m.w_down = C.cast(ptrs, C.POINTER(C.c_void_p))
    ok = L.Q4_0 | L.X_BF16
    assert _rc(L, "moe_prefill", L.Q8_0 | L.X_BF16, C.byref(m), FAKE, FAKE, FAKE, FAKE)[0] == -2
    assert _rc(L, "moe_prefill", L.Q4_K | L.X_BF16, C.byref(m), FAKE, FAKE, FAKE, FAKE)[0] == -2
    assert _rc(L, "moe_prefill", ok, None, FAKE, FAKE, FAKE, FAKE)[0] == -1
    assert _rc(L, "moe_prefill", ok, C.byref(m), None, FAKE, FAKE, FAKE)[0] == -1
    assert _rc(L, "moe_prefill", ok, C.byref(m), FAKE, FAKE, MIS, FAKE)[0] == -3
    m.top_k = 3
    assert _rc(L, "moe_prefill", ok, C.byref(m), FAKE, FAKE, FAKE, FAKE)[0] == -1   # top_k > n_experts
    m.top_k, m.hidden = 1, 100
    assert _rc(L, "moe_prefill", ok, C.byref(m), FAKE, FAKE, FAKE, FAKE)[0] == -3   # hidden % 32
    assert L.lib.qmm_moe_prefill_workspace_bytes(ok, C.byref(m)) == 0
    m.hidden = 256
    misaligned = P(MIS, FAKE)
    m.w_down = C.cast(misaligned, C.POINTER(C.c_void_p))
    assert _rc(L, "moe_prefill", ok, C.byref(m), FAKE, FAKE, FAKE, FAKE)[0] == -3
    m.w_down = C.cast(ptrs, C.POINTER(C.c_void_p))
    assert L.lib.qmm_moe_prefill_workspace_bytes(ok, C.byref(m)) > 0


def test_quantize_and_plane_argument_errors(L):
    assert _rc(L, "qmm_quantize_q8", 0x300, FAKE, 4, 64, FAKE, FAKE)[0] == -1
    assert _rc(L, "qmm_quantize_q8", 0x100, FAKE, 4, 48, FAKE, FAKE)[0] == -3
    assert _rc(L, "qmm_quantize_q8", 0x100, FAKE, 0, 64, FAKE, FAKE)[0] == -1
    assert _rc(L, "qmm_plane_build", None, 4, 256, FAKE)[0] == -1
    assert _rc(L, "qmm_plane_build", FAKE, 4, 300, FAKE)[0] == -3
    assert _rc(L, "qmm_plane_build", FAKE, 4, 256, MIS)[0] == -3
    assert _rc(L, "qmm_set_workspace", C.c_void_p(0x10010), 1024)[0] == -3
    assert L.lib.qmm_plane_bytes(4096, 11008) == 45088768
    assert L.lib.qmm_plane_bytes(0, 11008) == 0


def test_liveness_read_argument_errors(L):
    buf = (C.c_int64 * 32)()
    assert _rc(L, "qmm_liveness_read", None, 4)[0] == -1
    assert _rc(L, "qmm_liveness_read", buf, 33)[0] == -1


def _gate_in_fresh_process(env_value):
    code = ("import block_quantized_weight_q6_gb300 as q;"
            "print(q.lib.qmm_plane_wanted(4096, 11008), q.lib.qmm_plane_wanted(4096, 4000))")
    env = dict(os.environ)
    env.pop("QMM_Q6K_EXP", None)
    if env_value is not None:
        env["QMM_Q6K_EXP"] = env_value
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                         text=True, check=True)
    return out.stdout.split()


@pytest.mark.parametrize("value,expect", [(None, ["1", "0"]), ("1", ["1", "0"]), ("", ["1", "0"]),
                                          ("0", ["0", "0"]), ("false", ["1", "0"])])
def test_plane_gate_default_on_zero_opts_out(L, value, expect):
    """unset means on; only an explicit "0" opts out; K % 256 gates it too"""
    assert _gate_in_fresh_process(value) == expect


def test_gemv_group_argument_errors(L):
    P = C.c_void_p * 1
    I64 = C.c_int64 * 1
    W, x, y = P(FAKE), P(FAKE), P(FAKE)
    N, K = I64(64), I64(256)
    fn = L.lib.qmm_gemv_group
    assert _rc(L, "qmm_gemv_group", 0x03, 0, W, x, y, N, K, 1)[0] == -1    # n = 0
    assert _rc(L, "qmm_gemv_group", 0x03, 13, W, x, y, N, K, 1)[0] == -1   # n above 12
    assert _rc(L, "qmm_gemv_group", 0x03, 1, None, x, y, N, K, 1)[0] == -1  # null array
    assert _rc(L, "qmm_gemv_group", 0x03, 1, W, x, y, I64(0), K, 1)[0] == -1  # N = 0
    assert _rc(L, "qmm_gemv_group", 0x03, 1, W, x, y, N, I64(100), 1)[0] == -3  # K not a block multiple
    assert _rc(L, "qmm_gemv_group", 0x03, 1, W, x, y, N, K, 17)[0] == -1   # B above 16
    assert fn is not None
    assert L.lib.qmm_gemv_group_workspace_bytes(0x03, 0, N, K, 1) == 0
