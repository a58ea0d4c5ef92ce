"""Prefill GEMM on the GPU (tcgen05) against the CPU oracle, the W_exp plane
variant against the in-kernel expansion (bitwise), and the path labels.

Float outputs: |Y - Y_ref| <= 1e-4 * sum_k |w_k x^_k| + 1e-6 (x^ = s * x_q).
Integer cases (unit scales, integer activations with amax 127): bitwise.
"""
import os
import subprocess
import sys

import numpy as np
import pytest

import oracle
from oracle import pack
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import block_quantized_weight_q6_gb300 as qmm  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def x_tensor(x):
    if x.dtype == np.uint16:
        return dev(x.view(np.int16)).view(torch.bfloat16)
    return dev(x)


def run_gemm(fmt, W, X, N, K, plane=None, Wt=None):
    M = X.shape[0]
    Y = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    qmm.gemm(fmt, Wt if Wt is not None else dev(W), x_tensor(X), Y, M, N, K, plane)
    torch.cuda.synchronize()
    qmm.sync_check()
    return Y.cpu().numpy()


def assert_within(y, ref, absum, what=""):
    err = np.abs(y.astype(np.float64) - ref)
    bound = 1e-4 * absum + 1e-6
    bad = ~(err <= bound)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} out of bound; first {tuple(i)}: "
                             f"got {y[tuple(i)]}, ref {ref[tuple(i)]}, bound {bound[tuple(i)]}")


def unit_q6k(N, K, rng):
    codes = rng.integers(0, 64, (N, K))
    W = pack.pack_q6k_matrix(codes, np.ones((N, K // 16), int),
                             np.full((N, K // 256), pack.f16_bits(1.0)))
    return W, codes - 32


def int_acts(M, K, rng):
    xi = rng.integers(-127, 128, (M, K))
    xi[:, ::32] = 127
    return xi, xi.astype(np.float32)


@pytest.mark.parametrize("M,N,K", [(128, 128, 256), (200, 136, 512), (1, 8, 256), (300, 260, 768)])
def test_q6k_gemm_unit_scale_bitwise(M, N, K):
    rng = np.random.default_rng(M + N + K)
    W, wint = unit_q6k(N, K, rng)
    xi, X = int_acts(M, K, rng)
    exact = (xi @ wint.T).astype(np.float64)
    Y2 = run_gemm(qmm.Q6_K, W, X, N, K)
    assert np.array_equal(Y2.astype(np.float64), exact)
    Wt = dev(W)
    plane = qmm.plane_build(Wt, N, K)
    Y1 = run_gemm(qmm.Q6_K, W, X, N, K, plane=plane, Wt=Wt)
    qmm.plane_release(Wt)
    assert np.array_equal(Y1.astype(np.float64), exact)


@pytest.mark.parametrize("M,N,K", [(128, 128, 256), (130, 96, 512), (257, 300, 1024)])
def test_q4_0_gemm_unit_scale_bitwise(M, N, K):
    rng = np.random.default_rng(7 * M + N)
    codes = rng.integers(0, 16, (N, K))
    W = pack.pack_q4_0_matrix(codes, np.full((N, K // 32), pack.f16_bits(1.0)))
    xi, X = int_acts(M, K, rng)
    Y = run_gemm(qmm.Q4_0, W, X, N, K)
    assert np.array_equal(Y.astype(np.float64), (xi @ (codes - 8).T).astype(np.float64))


@pytest.mark.parametrize("M,N,K", [(256, 256, 1024), (77, 130, 2048)])
def test_q6k_gemm_random_plane_equals_in_kernel_and_oracle(M, N, K):
    W = synth.q6k_matrix(11 + M, N, K)
    X = synth.normal_bf16(12 + M, (M, K))
    Wt = dev(W)
    Y2 = run_gemm(qmm.Q6_K, W, X, N, K, Wt=Wt)
    plane = qmm.plane_build(Wt, N, K)
    Y1 = run_gemm(qmm.Q6_K, W, X, N, K, plane=plane, Wt=Wt)
    qmm.plane_release(Wt)
    assert np.array_equal(Y1.view(np.uint32), Y2.view(np.uint32)), "W_exp and in-kernel differ"
    xq, s = oracle.quantize_q8(X)
    ref, absum = oracle.gemv_q8(qmm.Q6_K, W, xq, s, N, K)
    assert_within(Y2, ref, absum, f"q6_K gemm {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(128, 128, 512), (200, 72, 4096)])
def test_q4_0_gemm_random(M, N, K):
    W = synth.q4_0_matrix(21 + M, N, K)
    X = synth.normal_bf16(22 + M, (M, K))
    Y = run_gemm(qmm.Q4_0, W, X, N, K)
    xq, s = oracle.quantize_q8(X)
    ref, absum = oracle.gemv_q8(qmm.Q4_0, W, xq, s, N, K)
    assert_within(Y, ref, absum, f"Q4_0 gemm {M}x{N}x{K}")


def test_gemm_rows_match_q8_gemv():
    """a GEMM row is the q8-activation matvec of that row (same definition)"""
    N, K = 256, 1024
    W = synth.q6k_matrix(31, N, K)
    X = synth.normal_bf16(32, (16, K))
    Wt = dev(W)
    Y = run_gemm(qmm.Q6_K, W, X, N, K, Wt=Wt)
    y = torch.empty((16, N), dtype=torch.float32, device="cuda")
    qmm.gemv(qmm.Q6_K, Wt, x_tensor(X), y, N, K, qmm.ACT_Q8)
    torch.cuda.synchronize()
    xq, s = oracle.quantize_q8(X)
    _, absum = oracle.gemv_q8(qmm.Q6_K, W, xq, s, N, K)
    assert (np.abs(Y.astype(np.float64) - y.cpu().numpy()) <= 2e-4 * absum + 2e-6).all()


def test_plane_build_bitwise():
    N, K = 96, 768
    W = synth.q6k_matrix(41, N, K)
    Wt = dev(W)
    plane = qmm.plane_build(Wt, N, K)
    torch.cuda.synchronize()
    qmm.plane_release(Wt)
    assert np.array_equal(plane.cpu().numpy(), oracle.plane_q6k(W, N, K))


def test_full_size_ffn_down_prefill_sampled():
    """q6_K ffn_down 4096 x 11008, 512 bf16 tokens: both variants bitwise
    identical; 1024 sampled outputs against the oracle."""
    M, N, K = 512, 4096, 11008
    W = synth.q6k_matrix(synth.workload_seed(2, 0), N, K)
    X = synth.normal_bf16(synth.workload_seed(2, 1), (M, K))
    Wt = dev(W)
    Y2 = run_gemm(qmm.Q6_K, W, X, N, K, Wt=Wt)
    plane = qmm.plane_build(Wt, N, K)
    Y1 = run_gemm(qmm.Q6_K, W, X, N, K, plane=plane, Wt=Wt)
    qmm.plane_release(Wt)
    del plane
    assert np.array_equal(Y1.view(np.uint32), Y2.view(np.uint32))
    rng = np.random.default_rng(5)
    ms = np.concatenate([rng.integers(0, M, 1020), [0, M - 1, 0, M - 1]])
    ns = np.concatenate([rng.integers(0, N, 1020), [0, N - 1, N - 1, 0]])
    xq, s = oracle.quantize_q8(X)
    ref, absum = oracle.gemm_q8_pairs(qmm.Q6_K, W, K, xq, s, ms, ns)
    assert_within(Y2[ms, ns], ref, absum, "ffn_down prefill")
    assert np.isfinite(Y2).all()


def test_labels_and_plane_errors():
    N, K, M = 64, 512, 16
    W = synth.q6k_matrix(51, N, K)
    X = synth.normal_bf16(52, (M, K))
    Wt = dev(W)
    qmm.liveness_reset()
    run_gemm(qmm.Q6_K, W, X, N, K, Wt=Wt)                 # never registered: in-kernel
    plane = qmm.plane_build(Wt, N, K)
    run_gemm(qmm.Q6_K, W, X, N, K, plane=plane, Wt=Wt)    # the plane path
    run_gemm(qmm.Q6_K, W, X, N, K, Wt=Wt)                 # plane exists but not passed
    live = qmm.liveness()
    assert live["gemm_in_kernel"] == 1 and live["gemm_exp_plane"] == 1
    assert live["gemm_fallback"] == 1 and live["plane_build"] == 1
    # a plane of other geometry is refused, never used silently
    Y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    with pytest.raises(qmm.QmmError) as ei:
        qmm.gemm(qmm.Q6_K, Wt, x_tensor(X), Y, M, N // 2, K, plane)
    assert ei.value.code == qmm.EPLANE
    other = torch.zeros_like(plane)
    with pytest.raises(qmm.QmmError) as ei:
        qmm.gemm(qmm.Q6_K, Wt, x_tensor(X), Y, M, N, K, other)
    assert ei.value.code == qmm.EPLANE
    qmm.plane_release(Wt)
    # registration that could not allocate: later launches count as fallback
    qmm.liveness_reset()
    qmm.plane_register_failed(Wt, N, K)
    run_gemm(qmm.Q6_K, W, X, N, K, Wt=Wt)
    assert qmm.liveness()["gemm_fallback"] == 1
    qmm.plane_release(Wt)


def _fresh(code, env_extra):
    env = dict(os.environ)
    env.update(env_extra)
    return subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                          text=True, timeout=300)


def test_exp_off_label_and_fault_injection_in_fresh_processes():
    code = r"""
import numpy as np, torch, synth, block_quantized_weight_q6_gb300 as qmm
N, K, M = 64, 512, 8
W = torch.from_numpy(synth.q6k_matrix(1, N, K)).cuda()
X = torch.randn(M, K, device="cuda").to(torch.bfloat16)
Y = torch.empty(M, N, device="cuda")
qmm.liveness_reset()
wanted = qmm.plane_wanted(N, K)
if wanted:
    qmm.plane_build(W, N, K)      # QMM_FAULT=plane_alloc: recorded as a failed allocation
qmm.gemm(qmm.Q6_K, W, X, Y, M, N, K, None)
torch.cuda.synchronize()
l = qmm.liveness()
print(int(wanted), l["gemm_exp_off"], l["gemm_fallback"], l["gemm_in_kernel"], l["gemm_exp_plane"])
"""
    r = _fresh(code, {"QMM_Q6K_EXP": "0", "QMM_DEBUG_LABEL": "1"})
    assert r.returncode == 0, r.stderr
    assert r.stdout.split() == ["0", "1", "0", "0", "0"]
    assert "in-kernel-expand(exp=off)" in r.stderr
    r = _fresh(code, {"QMM_FAULT": "plane_alloc", "QMM_DEBUG_LABEL": "1"})
    assert r.returncode == 0, r.stderr
    assert r.stdout.split() == ["1", "0", "1", "0", "0"]
    assert "fallback!" in r.stderr


def full_range_scales(W, N, K, rows, seed):
    """W (N x K q6_K) with the sub-block scales of the given rows drawn on
    the whole int8 range (-128..127), the rest as drawn"""
    W = W.copy()
    blocks = W.reshape(N, K // 256, 210)
    rng = np.random.default_rng(seed)
    rows = np.asarray(rows)
    blocks[rows, :, 192:208] = rng.integers(0, 256, (len(rows), K // 256, 16)).astype(np.uint8)
    return W


@pytest.mark.parametrize("M,N,K,rows", [
    (40, 136, 512, "all"),           # every tile two passes
    (200, 264, 1024, "tile1"),       # only the second 128-row weight tile holds large scales
    (40, 136, 4096, "all"),          # K split over CTAs, each split two passes
])
def test_q6k_gemm_full_int8_scales(M, N, K, rows):
    """Sub-block scales anywhere in -128..127 (a tile holding one beyond 56
    runs its K range a second time for the rest of each scale): both
    variants bitwise equal, within the bound against the oracle, and the
    tiles without large scales unchanged from a matrix where the large ones
    are absent."""
    W0 = synth.q6k_matrix(71 + K, N, K)
    sel = np.arange(N) if rows == "all" else np.arange(128, 256)
    W = full_range_scales(W0, N, K, sel, 72 + N)
    sc = W.reshape(-1, 210)[:, 192:208].view(np.int8)
    assert np.abs(sc.astype(int)).max() > 120
    X = synth.normal_bf16(73 + M, (M, K))
    Wt = dev(W)
    Y2 = run_gemm(qmm.Q6_K, W, X, N, K, Wt=Wt)
    plane = qmm.plane_build(Wt, N, K)
    Y1 = run_gemm(qmm.Q6_K, W, X, N, K, plane=plane, Wt=Wt)
    qmm.plane_release(Wt)
    assert np.array_equal(Y1.view(np.int32), Y2.view(np.int32))
    xq, s = oracle.quantize_q8(X)
    ref, absum = oracle.gemv_q8(qmm.Q6_K, W, xq, s, N, K)
    assert_within(Y2, ref, absum, f"q6_K GEMM, int8 scales, {M}x{N}x{K}")
    if rows != "all":
        # weight tiles 0 and 2 hold the same rows as in W0 and run one pass
        Y0 = run_gemm(qmm.Q6_K, W0, X, N, K)
        keep = np.r_[0:128, 256:N]
        assert np.array_equal(Y0[:, keep].view(np.int32), Y2[:, keep].view(np.int32))


@pytest.mark.parametrize("K", [256, 512])
def test_q6k_gemm_full_int8_scales_integer_exact(K):
    """d = 1, scales on -128..127, codes 30..34 (q - 32 in -2..2), integer
    activations with amax 127 per block (activation scale 1): every pass's
    block partials and the whole sum are integers below 2^24, so Y is the
    exact integer product, bitwise, in both variants"""
    M, N = 40, 136
    rng = np.random.default_rng(K)
    codes = rng.integers(30, 35, (N, K))
    scales = rng.integers(-128, 128, (N, K // 16))
    scales[:, 0] = -128
    scales[:, 1] = 127
    W = pack.pack_q6k_matrix(codes, scales, np.full((N, K // 256), pack.f16_bits(1.0)))
    wint = np.repeat(scales, 16, axis=1) * (codes - 32)
    xi, X = int_acts(M, K, rng)
    exact = (xi @ wint.T).astype(np.float64)
    assert np.abs(exact).max() < 2 ** 24
    Wt = dev(W)
    Y2 = run_gemm(qmm.Q6_K, W, X, N, K, Wt=Wt)
    assert np.array_equal(Y2.astype(np.float64), exact)
    plane = qmm.plane_build(Wt, N, K)
    Y1 = run_gemm(qmm.Q6_K, W, X, N, K, plane=plane, Wt=Wt)
    qmm.plane_release(Wt)
    assert np.array_equal(Y1.astype(np.float64), exact)


def test_q6k_matvec_large_scale():
    """The matvec applies the scales in fp32: a scale of 100 is exact there."""
    M, N, K = 2, 136, 512
    W = synth.q6k_matrix(71, N, K).copy()
    W.reshape(-1, 210)[5, 192 + 2] = np.uint8(100)
    x1 = synth.normal_bf16(73, (M, K))
    y = torch.empty((M, N), dtype=torch.float32, device="cuda")
    qmm.gemv(qmm.Q6_K, dev(W), x_tensor(x1), y, N, K)
    torch.cuda.synchronize()
    qmm.sync_check()
    ref, absum = oracle.gemv_float(qmm.Q6_K, W, x1, N, K)
    assert_within(y.cpu().numpy(), ref, absum, "q6_K matvec, scale 100")


# The 32-layer prefill sweep's GEMM shapes (7B-shaped layer: Q4_0 wq/wk/wo
# 4096 x 4096, w1/w3 11008 x 4096; q6_K attn_v 4096 x 4096 and the output
# matrix 32000 x 4096, both with the plane and with in-kernel expansion; the
# ffn_down shape is covered above), at the sweep's smallest and largest M.
SWEEP_SHAPES = [("wq", "Q4_0", 4096, 4096, 0), ("w1", "Q4_0", 11008, 4096, 3),
                ("attn_v", "q6_K", 4096, 4096, 5), ("output", "q6_K", 32000, 4096, 15)]


@pytest.mark.parametrize("M", [128, 2048])
@pytest.mark.parametrize("name,fmt_name,N,K,mid", SWEEP_SHAPES)
def test_sweep_shapes_vs_oracle(name, fmt_name, N, K, mid, M):
    """Weights drawn on the device as the sweep draws them; 512 sampled
    outputs against the oracle; the q6_K plane and in-kernel outputs bitwise
    equal over the whole Y."""
    fmt = {"Q4_0": qmm.Q4_0, "q6_K": qmm.Q6_K}[fmt_name]
    Wt = synth.matrix_torch(fmt, synth.workload_seed(4, mid), N, K, "cuda")[0]
    X = synth.normal_bf16(synth.workload_seed(4, 100 + K % 97 + M), (M, K))
    Y2 = run_gemm(fmt, None, X, N, K, Wt=Wt)
    if fmt == qmm.Q6_K:
        plane = qmm.plane_build(Wt, N, K)
        Y1 = run_gemm(fmt, None, X, N, K, plane=plane, Wt=Wt)
        qmm.plane_release(Wt)
        del plane
        assert np.array_equal(Y1.view(np.uint32), Y2.view(np.uint32)), f"{name} M={M}: variants differ"
        del Y1
    assert np.isfinite(Y2).all()
    W = Wt.cpu().numpy()
    rng = np.random.default_rng(M + N + mid)
    ms = np.concatenate([rng.integers(0, M, 508), [0, M - 1, 0, M - 1]])
    ns = np.concatenate([rng.integers(0, N, 508), [0, N - 1, N - 1, 0]])
    xq, s = oracle.quantize_q8(X)
    ref, absum = oracle.gemm_q8_pairs(fmt, W, K, xq, s, ms, ns)
    assert_within(Y2[ms, ns], ref, absum, f"sweep {name} {N}x{K} M={M}")


@pytest.mark.parametrize("fmt_name,M,N,K", [("q6_K", 128, 4096, 4096), ("Q4_0", 77, 130, 2048),
                                            ("q6_K", 200, 520, 8192)])
def test_split_k_grid_vs_oracle_deterministic(fmt_name, M, N, K):
    """A grid of fewer tiles than SMs splits K over CTAs and sums the partials
    in a fixed order: the sum-of-partials launch runs, a second call is
    bitwise identical, the q6_K plane and in-kernel variants agree bitwise,
    and sampled outputs (with the corners) are within the bound."""
    fmt = {"Q4_0": qmm.Q4_0, "q6_K": qmm.Q6_K}[fmt_name]
    Wt = synth.matrix_torch(fmt, synth.workload_seed(7, M % 13), N, K, "cuda")[0]
    X = synth.normal_bf16(synth.workload_seed(7, 3 + K % 11), (M, K))
    qmm.liveness_reset()
    Y = run_gemm(fmt, None, X, N, K, Wt=Wt)
    assert qmm.liveness()["gemm_split_reduce"] == 1
    Y2 = run_gemm(fmt, None, X, N, K, Wt=Wt)
    assert np.array_equal(Y.view(np.uint32), Y2.view(np.uint32))
    if fmt == qmm.Q6_K:
        plane = qmm.plane_build(Wt, N, K)
        Y3 = run_gemm(fmt, None, X, N, K, plane=plane, Wt=Wt)
        qmm.plane_release(Wt)
        assert np.array_equal(Y.view(np.uint32), Y3.view(np.uint32))
    rng = np.random.default_rng(M * N)
    ms = np.concatenate([rng.integers(0, M, 252), [0, M - 1, 0, M - 1]])
    ns = np.concatenate([rng.integers(0, N, 252), [0, N - 1, N - 1, 0]])
    xq, s = oracle.quantize_q8(X)
    ref, absum = oracle.gemm_q8_pairs(fmt, Wt.cpu().numpy(), K, xq, s, ms, ns)
    assert_within(Y[ms, ns], ref, absum, f"split-K {fmt_name} {M}x{N}x{K}")


def test_full_grid_does_not_split():
    """M = 512 against N = 4096 makes 128 tiles: one pass over K, no partials."""
    M, N, K = 512, 4096, 2048
    Wt = synth.matrix_torch(qmm.Q6_K, synth.workload_seed(7, 9), N, K, "cuda")[0]
    X = synth.normal_bf16(synth.workload_seed(7, 10), (M, K))
    qmm.liveness_reset()
    run_gemm(qmm.Q6_K, None, X, N, K, Wt=Wt)
    assert qmm.liveness()["gemm_split_reduce"] == 0
