"""Additive-codebook matvec (qmm_cbk_gemv; "Chasing x100", "The kernel is
ready") on the GPU, through the C interface, against the CPU oracle.

Float bound: |y - y_ref| <= 1e-4 * s + 1e-6 per element, s the oracle's
magnitude sum over every book's term (sum_k sum_m |scale * book term * x|).
Integer case (one-hot books, unit scales, integer activations): bitwise.
"""
import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - CPU-only containers
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import block_quantized_weight_q6_gb300 as qmm  # noqa: E402


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def x_tensor(x):
    if x.dtype == np.uint16:
        return dev(x.view(np.int16)).view(torch.bfloat16)
    return dev(x)


def run(M, codes, books, scales, x, N, K):
    B = x.shape[0]
    y = torch.full((B, N), float("nan"), dtype=torch.float32, device="cuda")
    qmm.cbk_gemv(M, dev(codes), dev(books.view(np.int16)), dev(scales.view(np.int16)), x_tensor(x), y, N, K)
    torch.cuda.synchronize()
    qmm.sync_check()
    return y.cpu().numpy()


def assert_within(y, ref, absum, what):
    err = np.abs(y.astype(np.float64) - ref)
    bound = 1e-4 * absum + 1e-6
    bad = ~(err <= bound)
    if bad.any():
        i = tuple(np.argwhere(bad)[0])
        raise AssertionError(f"{what}: {bad.sum()} out of bound; first {i}: got {y[i]}, ref {ref[i]}")


# one chunk, an odd number of chunks, several row slices and row blocks of
# codes, every batch size class (the chunk width drops to 8 groups where
# batch x books > 8)
SHAPES = [(8, 128), (37, 1152), (300, 640), (1000, 2048)]


@pytest.mark.parametrize("M", [2, 3])
@pytest.mark.parametrize("N,K", SHAPES)
@pytest.mark.parametrize("B", [1, 3, 8])
@pytest.mark.parametrize("xdt", ["bf16", "f32"])
def test_cbk_matches_oracle(M, N, K, B, xdt):
    codes, books, scales = synth.cbk_matrix(4000 + N + M, M, N, K)
    x = synth.normal_bf16(4010 + B, (B, K)) if xdt == "bf16" else synth.normal_f32(4010 + B, (B, K))
    qmm.liveness_reset()
    y = run(M, codes, books, scales, x, N, K)
    assert qmm.liveness()["cbk_gemv"] == 2
    ref, absum = oracle.cbk_gemv(M, codes, books, scales, x, N, K)
    assert_within(y, ref, absum, f"cbk M={M} {N}x{K} B={B} {xdt}")
    y2 = run(M, codes, books, scales, x, N, K)
    assert np.array_equal(y.view(np.uint32), y2.view(np.uint32))


@pytest.mark.parametrize("M", [2, 3])
@pytest.mark.parametrize("N,K", [(4096, 4096), (11008, 4096)])
@pytest.mark.parametrize("B", [1, 8])
def test_cbk_full_size_sampled(M, N, K, B):
    codes, books, scales = synth.cbk_matrix(4100 + N + M, M, N, K)
    x = synth.normal_bf16(4110 + B, (B, K))
    y = run(M, codes, books, scales, x, N, K)
    rng = np.random.default_rng(N + M + B)
    ns = np.sort(np.concatenate([rng.integers(0, N, 60), [0, N - 1]]))
    ref, absum = oracle.cbk_gemv(M, codes[ns], books, scales[ns], x, len(ns), K)
    assert_within(y[:, ns], ref, absum, f"cbk M={M} {N}x{K} B={B}")


@pytest.mark.parametrize("M", [2, 3])
def test_cbk_one_hot_books_integer_exact(M):
    """book 0 entry c = (c % 5 - 2) at position c % 8, the others zero, unit
    scales, integer activations: every table entry and sum is an exact
    integer, so the result equals the integer product bitwise"""
    N, K, B = 200, 1024, 4
    books = np.zeros((M, 256, 8))
    for c in range(256):
        books[0, c, c % 8] = c % 5 - 2
    bbits = books.astype(np.float16).view(np.uint16)
    rng = np.random.default_rng(M)
    codes = rng.integers(0, 256, (N, K // 8, M)).astype(np.uint8)
    scales = np.full(N, 1.0, np.float16).view(np.uint16)
    w = np.zeros((N, K))
    for n in range(N):
        for g in range(K // 8):
            c = int(codes[n, g, 0])
            w[n, 8 * g + c % 8] = c % 5 - 2
    xi = rng.integers(-50, 51, (B, K))
    y = run(M, codes, bbits, scales, synth.to_bf16_bits(xi.astype(np.float32)), N, K)
    assert np.array_equal(y.astype(np.float64), (xi @ w.T).astype(np.float64))


def test_cbk_argument_errors():
    codes, books, scales = synth.cbk_matrix(1, 2, 8, 128)
    y = torch.empty((1, 8), dtype=torch.float32, device="cuda")
    x = x_tensor(synth.normal_bf16(1, (1, 128)))
    for M, K, B, code in [(4, 128, 1, qmm.EINVAL), (2, 120, 1, qmm.EALIGN), (2, 128, 9, qmm.EINVAL)]:
        with pytest.raises(qmm.QmmError) as ei:
            xb = x if B == 1 else x_tensor(synth.normal_bf16(1, (B, 128)))
            qmm.cbk_gemv(M, dev(codes), dev(books.view(np.int16)), dev(scales.view(np.int16)), xb, y, 8, K)
        assert ei.value.code == code
