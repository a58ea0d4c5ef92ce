"""Q4_K / Q2_K matvecs (the K-quant ladder of quantprobe "LAWS.md", Law 4
amendment L-16) on the GPU, through the C interface, against the CPU oracle.

Float bound, as for the other formats: |y - y_ref| <= 1e-4 * s + 1e-6 per
element, where s is the oracle's magnitude sum; for these formats the weight
is the difference d*scale*q - dmin*min and the kernel sums the two terms
separately, so s = sum_k (|d*scale*q| + |dmin*min|) * |x|.
Integer cases (d = dmin = 1, integer activations): bitwise equal.
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

FMTS = {"Q4_K": qmm.Q4_K, "Q2_K": qmm.Q2_K}
PACK = {qmm.Q4_K: (pack.pack_q4k_block, 15, 32, 63), qmm.Q2_K: (pack.pack_q2k_block, 3, 16, 15)}


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def xbf(x):
    return dev(x.view(np.int16)).view(torch.bfloat16)


def run(fmt, W, x, N, K):
    B = x.shape[0]
    y = torch.full((B, N), float("nan"), dtype=torch.float32, device="cuda")
    qmm.gemv(fmt, dev(W), xbf(x), y, N, K)
    torch.cuda.synchronize()
    qmm.sync_check()
    return y.cpu().numpy()


def assert_within(y, ref, absum, what):
    err = np.abs(y.astype(np.float64) - ref)
    bound = 1e-4 * absum + 1e-6
    bad = ~(err <= bound)
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {bad.sum()} out of bound; first {i}: got {y[i]}, "
                             f"ref {ref[i]}, bound {bound[i]}")
    return float((err / bound).max())


# several items (16 rows at stride 8 in 128-row blocks), ragged N, one stage,
# odd and even super-block counts (Q2_K's 84-byte super-blocks land at every
# lead 0, 4, 8, 12 of a 16-byte line), long K split over warps
KQ_SHAPES = [(8, 256), (24, 512), (136, 11008), (264, 4864), (1000, 2304), (4104, 768)]


@pytest.mark.parametrize("name", ["Q4_K", "Q2_K"])
@pytest.mark.parametrize("N,K", KQ_SHAPES)
@pytest.mark.parametrize("B", [1, 3, 8])
def test_kquant_matches_oracle(name, N, K, B):
    fmt = FMTS[name]
    W = synth.matrix(fmt, 1500 + N, N, K)
    x = synth.normal_bf16(1510 + N + B, (B, K))
    qmm.liveness_reset()
    y = run(fmt, W, x, N, K)
    live = qmm.liveness()
    assert live["gemv_mv8"] == 1 and live["x_tile"] == 1 and live["gemv_float"] == 0
    ref, absum = oracle.gemv_float(fmt, W, x, N, K)
    assert_within(y, ref, absum, f"{name} {N}x{K} B={B}")
    y2 = run(fmt, W, x, N, K)
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))


@pytest.mark.parametrize("name", ["Q4_K", "Q2_K"])
@pytest.mark.parametrize("N,K", [(4096, 4096), (11008, 4096), (4096, 11008)])
@pytest.mark.parametrize("B", [1, 8])
def test_kquant_full_size_sampled(name, N, K, B):
    """the ladder's matrix shapes (a 7B layer's attention, up/gate and down
    projections) at full size, 512 sampled outputs against the oracle"""
    fmt = FMTS[name]
    W = synth.matrix(fmt, synth.workload_seed(5, fmt) + N, N, K)
    x = synth.normal_bf16(synth.workload_seed(5, 8) + B, (B, K))
    y = run(fmt, W, x, N, K)
    rng = np.random.default_rng(N + K + B)
    ns = np.concatenate([rng.integers(0, N, 500), [0, 7, 8, 127, 128, N - 1]])
    bs = rng.integers(0, B, len(ns))
    ref, absum = oracle.gemv_float_pairs(fmt, W, K, x, bs, ns)
    assert_within(y[bs, ns], ref, absum, f"{name} {N}x{K} B={B}")


@pytest.mark.parametrize("name", ["Q4_K", "Q2_K"])
@pytest.mark.parametrize("B", [1, 8])
def test_kquant_integer_path_bitwise(name, B):
    """d = dmin = 1, random scales and mins, integer activations: every
    weight sc*q - m and every partial sum is an integer below 2^24, so the
    result is the exact integer product"""
    fmt = FMTS[name]
    packer, qmax, sub, smax = PACK[fmt]
    N, K = 40, 1024
    rng = np.random.default_rng(fmt * 7 + B)
    codes = rng.integers(0, qmax + 1, (N, K))
    sc = rng.integers(0, smax + 1, (N, K // sub))
    mn = rng.integers(0, smax + 1, (N, K // sub))
    one = np.full((N, K // 256), pack.f16_bits(1.0))
    W = pack.pack_kq_matrix(packer, codes, sc, mn, one, one)
    wint = np.repeat(sc, sub, axis=1) * codes - np.repeat(mn, sub, axis=1)
    xi = rng.integers(-4, 5, (B, K))
    y = run(fmt, W, synth.to_bf16_bits(xi.astype(np.float32)), N, K)
    assert np.array_equal(y.astype(np.float64), (xi @ wint.T).astype(np.float64))


@pytest.mark.parametrize("name", ["Q4_K", "Q2_K"])
def test_kquant_zero_scales_and_one_hot(name):
    """all scales and mins zero give exactly 0; a single nonzero code per row
    (scale 1, d = 1, mins 0) returns that code times its bf16 activation"""
    fmt = FMTS[name]
    packer, qmax, sub, smax = PACK[fmt]
    N, K = 64, 512
    rng = np.random.default_rng(fmt)
    codes = rng.integers(0, qmax + 1, (N, K))
    zero = np.zeros((N, K // sub), int)
    one = np.full((N, K // 256), pack.f16_bits(1.0))
    x = synth.normal_bf16(77, (2, K))
    y = run(fmt, pack.pack_kq_matrix(packer, codes, zero, zero, one, one), x, N, K)
    assert np.array_equal(y, np.zeros_like(y))
    ks = rng.integers(0, K, N)
    oh = np.zeros((N, K), int)
    oh[np.arange(N), ks] = qmax
    y = run(fmt, pack.pack_kq_matrix(packer, oh, np.ones((N, K // sub), int), zero, one, one), x, N, K)
    xf = synth.bf16_bits_to_f32(x)
    assert np.array_equal(y, qmax * xf[:, ks])


@pytest.mark.parametrize("B", [1, 5, 8])
def test_kquant_in_multi_and_group_calls(B):
    """Q4_K and Q2_K beside q6_K / Q4_0 / Q8_0 in one mixed-format call (one
    fp16-MMA launch), and a same-format group call"""
    spec = [("Q4_K", 264, 4096), ("Q2_K", 520, 11008), ("q6_K", 136, 4096), ("Q2_K", 8, 256),
            ("Q4_0", 264, 512), ("Q4_K", 1024, 2304), ("Q8_0", 40, 768)]
    allf = {"Q4_K": qmm.Q4_K, "Q2_K": qmm.Q2_K, "q6_K": qmm.Q6_K, "Q4_0": qmm.Q4_0, "Q8_0": qmm.Q8_0}
    Ws = [synth.matrix(allf[f], 1600 + i, N, K) for i, (f, N, K) in enumerate(spec)]
    xs = [synth.normal_bf16(1610 + i, (B, K)) for i, (f, N, K) in enumerate(spec)]
    ys = [torch.full((B, N), float("nan"), dtype=torch.float32, device="cuda") for f, N, K in spec]
    multi = qmm.GemvMulti([allf[f] for f, N, K in spec], [dev(W) for W in Ws], [xbf(x) for x in xs],
                          ys, [N for f, N, K in spec], [K for f, N, K in spec])
    qmm.liveness_reset()
    qmm.gemv_multi(multi)
    torch.cuda.synchronize()
    qmm.sync_check()
    live = qmm.liveness()
    assert live["gemv_mv8"] == 1 and live["x_tile"] == 1
    for (f, N, K), W, x, y in zip(spec, Ws, xs, ys):
        ref, absum = oracle.gemv_float(allf[f], W, x, N, K)
        assert_within(y.cpu().numpy(), ref, absum, f"multi {f} {N}x{K} B={B}")
    # a group call of one format
    Wg = [synth.matrix(qmm.Q2_K, 1700 + i, 264, 1024) for i in range(3)]
    xg = [synth.normal_bf16(1710 + i, (B, 1024)) for i in range(3)]
    yg = [torch.empty((B, 264), dtype=torch.float32, device="cuda") for _ in range(3)]
    group = qmm.GemvGroup(qmm.Q2_K, [dev(W) for W in Wg], [xbf(x) for x in xg], yg, [264] * 3, [1024] * 3)
    qmm.gemv_group(group)
    torch.cuda.synchronize()
    qmm.sync_check()
    for W, x, y in zip(Wg, xg, yg):
        ref, absum = oracle.gemv_float(qmm.Q2_K, W, x, 264, 1024)
        assert_within(y.cpu().numpy(), ref, absum, f"group Q2_K B={B}")


def test_kquant_refused_outside_the_matvec():
    """fp32 activations or q8 mode with a K-quant format: QMM_EUNSUPPORTED"""
    W = dev(synth.matrix(qmm.Q4_K, 1, 64, 256))
    y = torch.empty((1, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(qmm.QmmError) as ei:
        qmm.gemv(qmm.Q4_K, W, dev(synth.normal_f32(1, (1, 256))), y, 64, 256)
    assert ei.value.code == qmm.EUNSUPPORTED
    with pytest.raises(qmm.QmmError) as ei:
        qmm.gemv(qmm.Q4_K, W, xbf(synth.normal_bf16(1, (1, 256))), y, 64, 256, qmm.ACT_Q8)
    assert ei.value.code == qmm.EUNSUPPORTED
