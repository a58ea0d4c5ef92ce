"""Decode matvec on the GPU (through the C interface) against the CPU oracle.

Float paths: |y - y_ref| <= 1e-4 * sum_k |w_k x_k| + 1e-6 per element.
Integer paths (unit scales, integer activations): bitwise equal.
"""
import numpy as np
import pytest

import oracle
from oracle import pack
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU-only containers
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import block_quantized_weight_q6_gb300 as qmm  # noqa: E402

FMTS = {"q6_K": qmm.Q6_K, "Q4_0": qmm.Q4_0, "Q8_0": qmm.Q8_0}


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def x_tensor(x):
    """numpy fp32 or bf16-bits -> torch cuda tensor of the same values"""
    if x.dtype == np.uint16:
        return dev(x.view(np.int16)).view(torch.bfloat16)
    return dev(x)


def run_gemv(fmt, W, x, N, K, act=qmm.ACT_FLOAT):
    B = x.shape[0]
    y = torch.full((B, N), float("nan"), dtype=torch.float32, device="cuda")
    qmm.gemv(fmt, dev(W), x_tensor(x), y, N, K, act)
    torch.cuda.synchronize()
    qmm.sync_check()
    return y.cpu().numpy()


def assert_within(y, ref, absum, what=""):
    err = np.abs(y.astype(np.float64) - ref)
    bound = 1e-4 * absum + 1e-6
    bad = ~(err <= bound)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} elements out of bound; first {tuple(i)}: "
                             f"got {y[tuple(i)]}, ref {ref[tuple(i)]}, bound {bound[tuple(i)]}")


SMALL = [("q6_K", 37, 256 * 19), ("Q4_0", 53, 32 * 71), ("Q8_0", 29, 32 * 45),
         ("q6_K", 5, 256), ("Q4_0", 3, 32)]


@pytest.mark.parametrize("name,N,K", SMALL)
@pytest.mark.parametrize("B", [1, 2, 3, 8, 16])
@pytest.mark.parametrize("xdt", ["f32", "bf16"])
def test_gemv_float_small(name, N, K, B, xdt):
    fmt = FMTS[name]
    W = synth.matrix(fmt, 100 + N, N, K)
    x = synth.normal_f32(7 + B, (B, K)) if xdt == "f32" else synth.normal_bf16(7 + B, (B, K))
    y = run_gemv(fmt, W, x, N, K)
    ref, absum = oracle.gemv_float(fmt, W, x, N, K)
    assert_within(y, ref, absum, f"{name} {N}x{K} B={B} {xdt}")


@pytest.mark.parametrize("name,N,K", SMALL)
@pytest.mark.parametrize("B", [1, 2, 8, 16])
def test_gemv_q8_small(name, N, K, B):
    fmt = FMTS[name]
    W = synth.matrix(fmt, 200 + N, N, K)
    x = synth.normal_bf16(17 + B, (B, K))
    y = run_gemv(fmt, W, x, N, K, qmm.ACT_Q8)
    xq, s = oracle.quantize_q8(x)
    ref, absum = oracle.gemv_q8(fmt, W, xq, s, N, K)
    assert_within(y, ref, absum, f"q8 {name} {N}x{K} B={B}")


@pytest.mark.parametrize("xdt", ["f32", "bf16"])
@pytest.mark.parametrize("rows,K", [(1, 32), (3, 4096), (16, 11008), (7, 7168)])
def test_quantizer_bitwise(xdt, rows, K):
    x = synth.normal_f32(31, (rows, K)) if xdt == "f32" else synth.normal_bf16(31, (rows, K))
    if xdt == "f32":
        x[0, :32] = np.float32([127, 2.5, -2.5, 3.5, 0.5, 1.5, -0.5, -1.5] * 4)  # exact ties
        if K >= 64:
            x[0, 32:64] = 0.0
    xt = x_tensor(x)
    xq = torch.empty((rows, K), dtype=torch.int8, device="cuda")
    s = torch.empty((rows, K // 32), dtype=torch.float32, device="cuda")
    qmm.quantize_q8(xt, xq, s)
    torch.cuda.synchronize()
    rq, rs = oracle.quantize_q8(x)
    assert np.array_equal(xq.cpu().numpy(), rq)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), rs.view(np.uint32))


def _unit_scale(fmt, N, K, rng):
    one = pack.f16_bits(1.0)
    if fmt == qmm.Q6_K:
        codes = rng.integers(0, 64, (N, K))
        return pack.pack_q6k_matrix(codes, np.ones((N, K // 16), int),
                                    np.full((N, K // 256), one)), codes - 32
    if fmt == qmm.Q4_0:
        codes = rng.integers(0, 16, (N, K))
        return pack.pack_q4_0_matrix(codes, np.full((N, K // 32), one)), codes - 8
    vals = rng.integers(-127, 128, (N, K))
    return pack.pack_q8_0_matrix(vals, np.full((N, K // 32), one)), vals


@pytest.mark.parametrize("name", ["q6_K", "Q4_0", "Q8_0"])
@pytest.mark.parametrize("B", [1, 8])
@pytest.mark.parametrize("K", [512, 2048])
def test_gemv_integer_paths_bitwise(name, B, K):
    """d = 1, sub-scales 1, integer activations with amax 127 per 32: the q8
    path is an exact integer matmul; so is the float path (all partial sums
    are integers below 2^24). Both must equal the oracle bitwise. (K = 2048
    at batch 1 runs every format through the CUDA-core batch-1 matvec.)"""
    fmt = FMTS[name]
    N = 24
    rng = np.random.default_rng(fmt * 10 + B)
    W, wint = _unit_scale(fmt, N, K, rng)
    xi = rng.integers(-127, 128, (B, K))
    xi[:, ::32] = 127
    x = xi.astype(np.float32)
    exact = (xi @ wint.T).astype(np.float64)
    y8 = run_gemv(fmt, W, x, N, K, qmm.ACT_Q8)
    yf = run_gemv(fmt, W, x, N, K, qmm.ACT_FLOAT)
    xq, s = oracle.quantize_q8(x)
    r8, _ = oracle.gemv_q8(fmt, W, xq, s, N, K)
    assert np.array_equal(r8, exact)
    assert np.array_equal(y8.astype(np.float64), exact)
    assert np.array_equal(yf.astype(np.float64), exact)


def test_gemv_identity_returns_x():
    n = 512
    codes = np.full((n, n), 32)
    np.fill_diagonal(codes, 33)
    W = pack.pack_q6k_matrix(codes, np.ones((n, n // 16), int),
                             np.full((n, n // 256), pack.f16_bits(1.0)))
    x = synth.normal_f32(5, (2, n))
    y = run_gemv(qmm.Q6_K, W, x, n, n)
    assert np.array_equal(y, x)


def test_q6k_full_size_1024x4096_b1_fp32_all_outputs():
    """the single-matvec workload: q6_K 1024 x 4096, batch 1, fp32 activations"""
    N, K = 1024, 4096
    W = synth.q6k_matrix(synth.workload_seed(0, 0), N, K)
    x = synth.normal_f32(synth.workload_seed(0, 1), (1, K))
    y = run_gemv(qmm.Q6_K, W, x, N, K)
    ref, absum = oracle.gemv_float(qmm.Q6_K, W, x, N, K)
    assert_within(y, ref, absum, "q6_K 1024x4096")
    # split-K reduction is deterministic: a second run is bitwise identical
    y2 = run_gemv(qmm.Q6_K, W, x, N, K)
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))


DECODE_SET = [("wq", "Q4_0", 4096, 4096), ("w1", "Q4_0", 11008, 4096),
              ("attn_v", "q6_K", 4096, 4096), ("ffn_down", "q6_K", 4096, 11008),
              ("output", "q6_K", 32000, 4096), ("wq_q8_0", "Q8_0", 4096, 4096)]


@pytest.mark.parametrize("mid", range(len(DECODE_SET)))
@pytest.mark.parametrize("B", [1, 8])
@pytest.mark.parametrize("act", ["float", "q8"])
def test_decode_set_full_size_sampled(mid, B, act):
    """7B-shaped decode matrices at full size, batch 1 and 8, bf16 activations:
    512 sampled outputs against the oracle, computed one by one."""
    name, fmt_name, N, K = DECODE_SET[mid]
    fmt = FMTS[fmt_name]
    W = synth.matrix(fmt, synth.workload_seed(1, mid), N, K)
    x = synth.normal_bf16(synth.workload_seed(1, 8 + B), (B, K))
    y = run_gemv(fmt, W, x, N, K, qmm.ACT_Q8 if act == "q8" else qmm.ACT_FLOAT)
    rng = np.random.default_rng(mid)
    bs = rng.integers(0, B, 512)
    ns = np.concatenate([rng.integers(0, N, 508), [0, N - 1, N // 2, N - 2]])
    if act == "float":
        ref, absum = oracle.gemv_float_pairs(fmt, W, K, x, bs, ns)
    else:
        xq, s = oracle.quantize_q8(x)
        ref, absum = oracle.gemm_q8_pairs(fmt, W, K, xq, s, bs, ns)
    assert_within(y[bs, ns], ref, absum, f"{name} B={B} {act}")
    assert np.isfinite(y).all()


def test_tail_bytes_and_tiny_shapes():
    """matrices whose byte size is not a multiple of 16 (tail copied by plain
    loads) and single-block rows"""
    for fmt, N, K in [(qmm.Q4_0, 1, 32), (qmm.Q4_0, 3, 64), (qmm.Q8_0, 1, 32),
                      (qmm.Q8_0, 5, 96), (qmm.Q6_K, 1, 256), (qmm.Q6_K, 3, 512)]:
        W = synth.matrix(fmt, 7, N, K)
        for B in (1, 16):
            x = synth.normal_f32(3, (B, K))
            y = run_gemv(fmt, W, x, N, K)
            ref, absum = oracle.gemv_float(fmt, W, x, N, K)
            assert_within(y, ref, absum, f"tiny fmt={fmt} {N}x{K} B={B}")


def test_liveness_counts_each_launch():
    qmm.liveness_reset()
    N, K = 64, 4096
    W = synth.q6k_matrix(1, N, K)
    x = synth.normal_f32(2, (2, K))  # batch 2: the tensor-core matvec
    run_gemv(qmm.Q6_K, W, x, N, K)
    run_gemv(qmm.Q6_K, W, x[:1], N, K, qmm.ACT_Q8)
    live = qmm.liveness()
    assert live["gemv_float"] == 1 and live["gemv_q8"] == 1 and live["quantize"] == 1
    assert live["gemv_splitk_reduce"] == 2  # short N is split along K
    assert live["x_tile"] == 1              # fp32 float mode lays the activations out once
    run_gemv(qmm.Q6_K, W, synth.normal_bf16(3, (9, K)), N, K)  # batch 9: the tensor-core matvec
    live = qmm.liveness()
    assert live["gemv_float"] == 2 and live["x_tile"] == 1  # bf16: gathered inside the matvec
    assert live["gemv_mv1"] == 0 and live["gemv_splitk_reduce"] == 3
    run_gemv(qmm.Q6_K, W, synth.normal_f32(3, (1, K)), N, K)  # batch 1, fp32: one mv1 launch, no split
    live = qmm.liveness()
    assert live["gemv_mv1"] == 1 and live["gemv_float"] == 2 and live["gemv_splitk_reduce"] == 3
    # batch 1 and 4, bf16, N % 8 == 0: the fp16-MMA matvec, one launch each
    # after one activation layout launch (K split across warps, no reduce)
    run_gemv(qmm.Q6_K, W, synth.normal_bf16(3, (1, K)), N, K)
    run_gemv(qmm.Q6_K, W, synth.normal_bf16(3, (4, K)), N, K)
    live = qmm.liveness()
    assert live["gemv_mv8"] == 2 and live["x_tile"] == 3
    assert live["gemv_mv1"] == 1 and live["gemv_float"] == 2 and live["gemv_splitk_reduce"] == 3


def test_missing_workspace_is_an_error():
    N, K = 64, 1024
    Wt = dev(synth.q6k_matrix(1, N, K))
    xt = x_tensor(synth.normal_f32(2, (1, K)))
    y = torch.empty((1, N), dtype=torch.float32, device="cuda")
    qmm.lib.qmm_set_workspace(None, 0)
    rc = qmm.lib.qmm_gemv(qmm.Q6_K | qmm.ACT_Q8, qmm._ptr(Wt), qmm._ptr(xt), qmm._ptr(y), N, K, 1)
    assert rc == qmm.ENOWORKSPACE


GROUP_SHAPES = {  # ragged rows, several K, more than one 128-row tile
    "q6_K": [(37, 256 * 3), (300, 256 * 5), (129, 256 * 16), (8, 256)],
    "Q4_0": [(53, 32 * 7), (260, 32 * 40), (128, 32 * 128)],
    "Q8_0": [(29, 32 * 9), (200, 32 * 64)],
}


@pytest.mark.parametrize("name", ["q6_K", "Q4_0", "Q8_0"])
@pytest.mark.parametrize("B", [1, 3, 8, 16])
@pytest.mark.parametrize("xdt,act", [("bf16", "float"), ("f32", "float"), ("bf16", "q8")])
def test_gemv_group_matches_oracle(name, B, xdt, act):
    fmt = FMTS[name]
    shapes = GROUP_SHAPES[name]
    Ws = [synth.matrix(fmt, 300 + i, N, K) for i, (N, K) in enumerate(shapes)]
    mk = synth.normal_bf16 if xdt == "bf16" else synth.normal_f32
    xs = [mk(400 + i, (B, K)) for i, (N, K) in enumerate(shapes)]
    ys = [torch.full((B, N), float("nan"), dtype=torch.float32, device="cuda") for N, K in shapes]
    mode = qmm.ACT_Q8 if act == "q8" else qmm.ACT_FLOAT
    grp = qmm.GemvGroup(fmt, [dev(W) for W in Ws], [x_tensor(x) for x in xs], ys,
                        [N for N, K in shapes], [K for N, K in shapes], mode)
    qmm.gemv_group(grp)
    torch.cuda.synchronize()
    qmm.sync_check()
    for (N, K), W, x, y in zip(shapes, Ws, xs, ys):
        if act == "q8":
            xq, s = oracle.quantize_q8(x)
            ref, absum = oracle.gemv_q8(fmt, W, xq, s, N, K)
        else:
            ref, absum = oracle.gemv_float(fmt, W, x, N, K)
        assert_within(y.cpu().numpy(), ref, absum, f"group {name} {N}x{K} B={B} {xdt} {act}")


def test_gemv_group_launches_once_per_step():
    """A grouped call launches the activation layout, the matvec and the
    split-K reduction once each, whatever the number of matrices."""
    fmt = qmm.Q6_K
    shapes = [(37, 256 * 12), (60, 256 * 16), (20, 256 * 8)]  # short N: split along K
    Ws = [synth.matrix(fmt, 500 + i, N, K) for i, (N, K) in enumerate(shapes)]
    xs = [synth.normal_f32(600 + i, (1, K)) for i, (N, K) in enumerate(shapes)]
    ys = [torch.empty((1, N), dtype=torch.float32, device="cuda") for N, K in shapes]
    grp = qmm.GemvGroup(fmt, [dev(W) for W in Ws], [x_tensor(x) for x in xs], ys,
                        [N for N, K in shapes], [K for N, K in shapes], qmm.ACT_Q8)
    qmm.liveness_reset()
    qmm.gemv_group(grp)
    torch.cuda.synchronize()
    qmm.sync_check()
    live = qmm.liveness()
    assert live["gemv_q8"] == 1 and live["quantize"] == 1
    assert live["gemv_splitk_reduce"] == 1
    for (N, K), W, x, y in zip(shapes, Ws, xs, ys):
        xq, s = oracle.quantize_q8(x)
        ref, absum = oracle.gemv_q8(fmt, W, xq, s, N, K)
        assert_within(y.cpu().numpy(), ref, absum, f"group launches {N}x{K}")


# The batch-1 float matvec on the CUDA cores (mv1): taken for B = 1, float
# mode, K % 256 == 0 and rows of whole 16-byte pieces (q6_K: K % 2048 == 0).
# Ragged row counts (not a multiple of the 4-row item), K pieces of 2048 with
# a partial last piece, more items than warps in the grid, fp32 and bf16
# activations.
MV1_SHAPES = [("q6_K", 37, 2048), ("q6_K", 2053, 4096), ("q6_K", 300, 8192), ("q6_K", 3, 6144),
              ("Q4_0", 1001, 4096), ("Q4_0", 70, 2816), ("Q4_0", 19500, 4096), ("Q4_0", 5, 256),
              ("Q8_0", 515, 4096), ("Q8_0", 33, 768), ("Q8_0", 16, 6144)]


@pytest.mark.parametrize("name,N,K", MV1_SHAPES)
@pytest.mark.parametrize("xdt", ["f32", "bf16"])
def test_mv1_matches_oracle(name, N, K, xdt):
    fmt = FMTS[name]
    W = synth.matrix(fmt, 700 + N, N, K)
    x = synth.normal_f32(710 + N, (1, K)) if xdt == "f32" else synth.normal_bf16(710 + N, (1, K))
    qmm.liveness_reset()
    y = run_gemv(fmt, W, x, N, K)
    # bf16 rows with N % 8 == 0 take the fp16-MMA matvec instead
    mvh = xdt == "bf16" and N % 8 == 0
    assert qmm.liveness()["gemv_mv8" if mvh else "gemv_mv1"] == 1
    if N * K <= 4096 * 4096:
        ref, absum = oracle.gemv_float(fmt, W, x, N, K)
        assert_within(y, ref, absum, f"mv1 {name} {N}x{K} {xdt}")
    else:  # large: sampled outputs, computed one by one
        rng = np.random.default_rng(N)
        ns = np.concatenate([rng.integers(0, N, 300), [0, N - 1, N - 16, N - 17]])
        ref, absum = oracle.gemv_float_pairs(fmt, W, K, x, np.zeros(len(ns), int), ns)
        assert_within(y[0, ns], ref, absum, f"mv1 {name} {N}x{K} {xdt}")
    # the order of the sums is fixed: a second call is bitwise identical
    y2 = run_gemv(fmt, W, x, N, K)
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))


def test_mv1_zero_weights_and_identity_are_exact():
    """w = 0 gives exactly 0 and a one-hot row gives exactly its x, through
    the batch-1 matvec of each format"""
    n = 2048
    x = synth.normal_f32(9, (1, n))
    one = pack.f16_bits(1.0)
    codes = np.full((n, n), 32)
    np.fill_diagonal(codes, 33)
    W6 = pack.pack_q6k_matrix(codes, np.ones((n, n // 16), int), np.full((n, n // 256), one))
    c4 = np.full((n, n), 8)
    np.fill_diagonal(c4, 9)
    W4 = pack.pack_q4_0_matrix(c4, np.full((n, n // 32), one))
    v8 = np.zeros((n, n), int)
    np.fill_diagonal(v8, 1)
    W8 = pack.pack_q8_0_matrix(v8, np.full((n, n // 32), one))
    for fmt, W in [(qmm.Q6_K, W6), (qmm.Q4_0, W4), (qmm.Q8_0, W8)]:
        qmm.liveness_reset()
        y = run_gemv(fmt, W, x, n, n)
        assert qmm.liveness()["gemv_mv1"] == 1
        assert np.array_equal(y, x), f"fmt {fmt}"


# The batch 2-8 float matvec on the warp-level MMA (mv8): taken for 2 <= B <= 8,
# bf16 activations, float mode, K % 256 == 0. Ragged rows (not a multiple of
# the 32-row item or of a 16-row MMA tile), activation rows short of 8, K
# split over several warps (short N, long K), q6_K super-blocks at every even
# offset of their 16-byte piece, q6_K rows that are not whole 16-byte pieces
# (each row at its own offset), more items than warps.
MV8_SHAPES = [("q6_K", 37, 2048), ("q6_K", 2053, 4096), ("q6_K", 61, 16384), ("q6_K", 4100, 6144),
              ("q6_K", 61, 11008), ("q6_K", 33, 768), ("q6_K", 4099, 11008),
              ("Q4_0", 1001, 4096), ("Q4_0", 70, 2816), ("Q4_0", 13000, 4096), ("Q4_0", 5, 256),
              ("Q8_0", 515, 4096), ("Q8_0", 33, 768)]


@pytest.mark.parametrize("name,N,K", MV8_SHAPES)
@pytest.mark.parametrize("B", [2, 5, 8])
def test_mv8_matches_oracle(name, N, K, B):
    fmt = FMTS[name]
    W = synth.matrix(fmt, 800 + N, N, K)
    x = synth.normal_bf16(810 + N + B, (B, K))
    qmm.liveness_reset()
    y = run_gemv(fmt, W, x, N, K)
    assert qmm.liveness()["gemv_mv8"] == 1
    if N * K <= 4096 * 4096:
        ref, absum = oracle.gemv_float(fmt, W, x, N, K)
        assert_within(y, ref, absum, f"mv8 {name} {N}x{K} B={B}")
    else:
        rng = np.random.default_rng(N + B)
        ns = np.concatenate([rng.integers(0, N, 200), [0, N - 1, N - 16, N - 33]])
        bs = rng.integers(0, B, len(ns))
        ref, absum = oracle.gemv_float_pairs(fmt, W, K, x, bs, ns)
        assert_within(y[bs, ns], ref, absum, f"mv8 {name} {N}x{K} B={B}")
    y2 = run_gemv(fmt, W, x, N, K)
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))


@pytest.mark.parametrize("name", ["q6_K", "Q4_0", "Q8_0"])
def test_mv8_integer_path_bitwise(name):
    """unit scales and integer activations (exact in bf16): the MMA's sums are
    integers below 2^24, so the batch 2-8 matvec equals the exact product"""
    fmt = FMTS[name]
    N, K, B = 40, 2048, 8
    rng = np.random.default_rng(fmt * 10 + 7)
    W, wint = _unit_scale(fmt, N, K, rng)
    xi = rng.integers(-127, 128, (B, K))
    x = synth.to_bf16_bits(xi.astype(np.float32))  # integers below 256: exact in bf16
    exact = (xi @ wint.T).astype(np.float64)
    qmm.liveness_reset()
    y = run_gemv(fmt, W, x, N, K)
    assert qmm.liveness()["gemv_mv8"] == 1
    assert np.array_equal(y.astype(np.float64), exact)


def test_unaligned_q6k_rows_at_batch_1_take_the_tensor_core_matvec():
    """q6_K rows that are not whole 16-byte pieces (K / 256 not a multiple of
    8) go to the tensor-memory matvec at batch 1 (to the warp-level MMA at
    batch 2-8, above)"""
    N, K = 61, 11008
    W = synth.matrix(qmm.Q6_K, 900, N, K)
    x = synth.normal_bf16(901, (1, K))
    qmm.liveness_reset()
    y = run_gemv(qmm.Q6_K, W, x, N, K)
    live = qmm.liveness()
    assert live["gemv_mv1"] == 0 and live["gemv_mv8"] == 0 and live["gemv_float"] == 1
    ref, absum = oracle.gemv_float(qmm.Q6_K, W, x, N, K)
    assert_within(y, ref, absum, "unaligned q6_K B=1")


def test_group_makes_one_fast_launch_per_k():
    """a grouped batch-8 call over matrices of two K (one of them with rows
    that are not whole 16-byte pieces) makes one warp-MMA launch per K"""
    shapes = [(100, 4096), (70, 11008), (44, 4096)]  # N % 8 != 0: not the fp16-MMA matvec
    Ws = [synth.matrix(qmm.Q6_K, 950 + i, N, K) for i, (N, K) in enumerate(shapes)]
    xs = [synth.normal_bf16(960 + i, (8, K)) for i, (N, K) in enumerate(shapes)]
    ys = [torch.full((8, N), float("nan"), dtype=torch.float32, device="cuda") for N, K in shapes]
    grp = qmm.GemvGroup(qmm.Q6_K, [dev(W) for W in Ws], [x_tensor(x) for x in xs], ys,
                        [N for N, K in shapes], [K for N, K in shapes], qmm.ACT_FLOAT)
    qmm.liveness_reset()
    qmm.gemv_group(grp)
    torch.cuda.synchronize()
    qmm.sync_check()
    live = qmm.liveness()
    assert live["gemv_mv8"] == 2 and live["gemv_float"] == 0
    for (N, K), W, x, y in zip(shapes, Ws, xs, ys):
        ref, absum = oracle.gemv_float(qmm.Q6_K, W, x, N, K)
        assert_within(y.cpu().numpy(), ref, absum, f"group per K {N}x{K}")


def test_fast_paths_opt_out_gate():
    """QMM_MVH=0, QMM_MV1=0 and QMM_MV8=0 (read once per process) send batch
    1 and batch 2-8 to the tensor-memory matvec; the results stay within the
    bound"""
    import os
    import subprocess
    import sys
    code = r"""
import numpy as np, torch, sys
sys.path.insert(0, {root!r})
import block_quantized_weight_q6_gb300 as qmm, oracle, synth
N, K = 48, 2048
W = synth.q6k_matrix(3, N, K)
Wt = torch.from_numpy(W).cuda()
for B in (1, 4):
    x = synth.normal_bf16(4 + B, (B, K))
    xt = torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    y = torch.empty((B, N), dtype=torch.float32, device="cuda")
    qmm.liveness_reset()
    qmm.gemv(qmm.Q6_K, Wt, xt, y, N, K)
    torch.cuda.synchronize()
    live = qmm.liveness()
    assert live["gemv_mv1"] == 0 and live["gemv_mv8"] == 0 and live["gemv_float"] == 1, live
    ref, absum = oracle.gemv_float(qmm.Q6_K, W, x, N, K)
    assert (np.abs(y.cpu().numpy() - ref) <= 1e-4 * absum + 1e-6).all()
print("gate ok")
"""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, QMM_MV1="0", QMM_MV8="0", QMM_MVH="0")
    r = subprocess.run([sys.executable, "-c", code.format(root=root)], env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0 and "gate ok" in r.stdout, r.stdout + r.stderr


# The batch 1-8 matvec on the warp-level MMA with fp16 operands (mvh): taken
# for bf16 activations, 1 <= B <= 8, float mode, K % 256 == 0, N % 8 == 0, any
# mix of formats in one launch. Rows not a multiple of the 256-row block of 8
# stride-8 items (partial items), a single 8-row group, K split over several
# warps (short N, long K), q6_K super-blocks at every even lead (K = 11008:
# rows of 9030 bytes), Q8_0 stages at both leads (K / 128 odd and even).
MVH_SHAPES = [("q6_K", 8, 256), ("q6_K", 264, 768), ("q6_K", 1000, 11008), ("q6_K", 520, 4096),
              ("q6_K", 4104, 2304), ("Q4_0", 8, 256), ("Q4_0", 392, 1280), ("Q4_0", 4104, 512),
              ("Q4_0", 136, 11008), ("Q8_0", 16, 256), ("Q8_0", 264, 2304), ("Q8_0", 8200, 768)]


@pytest.mark.parametrize("name,N,K", MVH_SHAPES)
@pytest.mark.parametrize("B", [1, 3, 8])
def test_mvh_matches_oracle(name, N, K, B):
    fmt = FMTS[name]
    W = synth.matrix(fmt, 1200 + N, N, K)
    x = synth.normal_bf16(1210 + N + B, (B, K))
    qmm.liveness_reset()
    y = run_gemv(fmt, W, x, N, K)
    live = qmm.liveness()
    assert live["gemv_mv8"] == 1 and live["x_tile"] == 1 and live["gemv_float"] == 0
    if N * K <= 2048 * 4096:
        ref, absum = oracle.gemv_float(fmt, W, x, N, K)
        assert_within(y, ref, absum, f"mvh {name} {N}x{K} B={B}")
    else:
        rng = np.random.default_rng(N + B)
        ns = np.concatenate([rng.integers(0, N, 300), [0, N - 1, N - 8, N - 9, 255, 256]])
        bs = rng.integers(0, B, len(ns))
        ref, absum = oracle.gemv_float_pairs(fmt, W, K, x, bs, ns)
        assert_within(y[bs, ns], ref, absum, f"mvh {name} {N}x{K} B={B}")
    # the order of the sums is fixed: a second call is bitwise identical
    y2 = run_gemv(fmt, W, x, N, K)
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))


@pytest.mark.parametrize("name", ["q6_K", "Q4_0", "Q8_0"])
@pytest.mark.parametrize("B", [1, 8])
def test_mvh_integer_path_bitwise(name, B):
    """unit scales, integer activations (exact in bf16 and, scaled by a power
    of two, in fp16): every partial sum is an exact integer multiple of the
    scale, so the fp16-MMA matvec equals the exact product bitwise"""
    fmt = FMTS[name]
    N, K = 48, 2048
    rng = np.random.default_rng(fmt * 10 + B)
    W, wint = _unit_scale(fmt, N, K, rng)
    xi = rng.integers(-127, 128, (B, K))
    x = synth.to_bf16_bits(xi.astype(np.float32))
    qmm.liveness_reset()
    y = run_gemv(fmt, W, x, N, K)
    assert qmm.liveness()["gemv_mv8"] == 1
    assert np.array_equal(y.astype(np.float64), (xi @ wint.T).astype(np.float64))


def test_mvh_identity_and_zero_rows_are_exact():
    """a one-hot row returns its bf16 activation bitwise; an all-zero weight
    row and an all-zero activation row give exactly 0"""
    n = 1024
    one = pack.f16_bits(1.0)
    codes = np.full((n, n), 32)
    np.fill_diagonal(codes, 33)
    codes[5] = 32  # an all-zero weight row
    W = pack.pack_q6k_matrix(codes, np.ones((n, n // 16), int), np.full((n, n // 256), one))
    x = synth.normal_bf16(21, (3, n))
    x[1] = 0  # an all-zero activation row
    y = run_gemv(qmm.Q6_K, W, x, n, n)
    xf = synth.bf16_bits_to_f32(x)
    expect = xf.copy()
    expect[:, 5] = 0.0
    assert np.array_equal(y, expect)


def test_mvh_activation_range_extremes():
    """activation rows of very large and very small magnitude (each row gets
    its own power-of-two scale) and a row mixing magnitudes 2^40 apart"""
    N, K = 64, 4096
    W = synth.q6k_matrix(31, N, K)
    xf = synth.normal_f32(32, (4, K))
    xf[0] *= 1e30
    xf[1] *= 1e-30
    xf[2, ::2] *= 2.0 ** 20
    xf[2, 1::2] *= 2.0 ** -20
    x = synth.to_bf16_bits(xf)
    y = run_gemv(qmm.Q6_K, W, x, N, K)
    ref, absum = oracle.gemv_float(qmm.Q6_K, W, x, N, K)
    assert_within(y, ref, absum, "activation extremes")


@pytest.mark.parametrize("B", [1, 6])
def test_mvh_q6k_large_scales_exact_form(B):
    """q6_K sub-block scales outside -62..62 (up to -128 and 127) take the
    exact two-MMA form of the tile; the result stays within the bound, and
    with unit d and integer activations it is exact"""
    N, K = 96, 1024
    W = synth.q6k_matrix(41, N, K).copy()
    blk = W.reshape(-1, 210)
    blk[::5, 192 + 3] = np.uint8(127)
    blk[2::5, 192 + 11] = np.uint8(128)   # -128
    blk[3::7, 192 + 0] = np.uint8(256 - 90)
    x = synth.normal_bf16(42 + B, (B, K))
    y = run_gemv(qmm.Q6_K, W, x, N, K)
    ref, absum = oracle.gemv_float(qmm.Q6_K, W, x, N, K)
    assert_within(y, ref, absum, "q6_K large scales")
    rng = np.random.default_rng(43)
    codes = rng.integers(0, 64, (N, K))
    sc = rng.integers(-128, 128, (N, K // 16))
    Wu = pack.pack_q6k_matrix(codes, sc, np.full((N, K // 256), pack.f16_bits(1.0)))
    xi = rng.integers(-8, 9, (B, K))
    yu = run_gemv(qmm.Q6_K, Wu, synth.to_bf16_bits(xi.astype(np.float32)), N, K)
    wint = (codes - 32) * np.repeat(sc, 16, axis=1)
    assert np.array_equal(yu.astype(np.float64), (xi @ wint.T).astype(np.float64))


@pytest.mark.parametrize("B", [1, 3, 8])
@pytest.mark.parametrize("xdt", ["bf16", "f32"])
def test_gemv_multi_mixed_formats(B, xdt):
    """matvecs of all three formats in one call: with bf16 activations the
    ones with N % 8 == 0 run in one fp16-MMA launch whatever their format, the
    others per format; with fp32 activations all run per format"""
    spec = [("Q4_0", 264, 512), ("q6_K", 520, 4096), ("Q8_0", 40, 768), ("q6_K", 37, 256 * 5),
            ("Q4_0", 53, 32 * 16), ("q6_K", 256, 11008)]
    Ws = [synth.matrix(FMTS[f], 1300 + i, N, K) for i, (f, N, K) in enumerate(spec)]
    mk = synth.normal_bf16 if xdt == "bf16" else synth.normal_f32
    xs = [mk(1310 + i, (B, K)) for i, (f, N, K) in enumerate(spec)]
    ys = [torch.full((B, N), float("nan"), dtype=torch.float32, device="cuda") for f, N, K in spec]
    multi = qmm.GemvMulti([FMTS[f] for f, N, K in spec], [dev(W) for W in Ws], [x_tensor(x) for x in xs],
                          ys, [N for f, N, K in spec], [K for f, N, K in spec])
    qmm.liveness_reset()
    qmm.gemv_multi(multi)
    torch.cuda.synchronize()
    qmm.sync_check()
    live = qmm.liveness()
    if xdt == "bf16":
        assert live["gemv_mv8"] >= 1 and live["x_tile"] == 1
    for (f, N, K), W, x, y in zip(spec, Ws, xs, ys):
        ref, absum = oracle.gemv_float(FMTS[f], W, x, N, K)
        assert_within(y.cpu().numpy(), ref, absum, f"multi {f} {N}x{K} B={B} {xdt}")


def test_gemv_multi_shares_equal_activations():
    """matvecs that read the same activation tensor (q, k, v of one layer)
    share one fp16 copy of it; results as separate calls within the bound"""
    K, B = 4096, 2
    x = synth.normal_bf16(1400, (B, K))
    xt = x_tensor(x)
    spec = [("Q4_0", 512), ("Q4_0", 512), ("q6_K", 512)]
    Ws = [synth.matrix(FMTS[f], 1410 + i, N, K) for i, (f, N) in enumerate(spec)]
    ys = [torch.empty((B, N), dtype=torch.float32, device="cuda") for f, N in spec]
    multi = qmm.GemvMulti([FMTS[f] for f, N in spec], [dev(W) for W in Ws], [xt, xt, xt], ys,
                          [N for f, N in spec], [K] * 3)
    qmm.gemv_multi(multi)
    torch.cuda.synchronize()
    qmm.sync_check()
    for (f, N), W, y in zip(spec, Ws, ys):
        ref, absum = oracle.gemv_float(FMTS[f], W, x, N, K)
        assert_within(y.cpu().numpy(), ref, absum, f"shared x {f}")


def test_gemv_multi_argument_errors():
    xt = x_tensor(synth.normal_bf16(1, (1, 256)))
    Wt = dev(synth.q6k_matrix(1, 8, 256))
    y = torch.empty((1, 8), dtype=torch.float32, device="cuda")
    # activation bits that differ between entries
    m = qmm.GemvMulti([qmm.Q6_K, qmm.Q6_K], [Wt, Wt], [xt, xt], [y, y], [8, 8], [256, 256])
    m._fmt[1] = qmm.Q6_K | qmm.X_F32
    with pytest.raises(qmm.QmmError) as ei:
        qmm.gemv_multi(m)
    assert ei.value.code == qmm.EINVAL
