"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test checks the oracle against something independent: hand-built blocks
with hand-derived values (tests/golden), closed forms over every code and
scale, textbook facts (IEEE binary16/bfloat16 via numpy), library routines
(numpy matmul / integer matmul, stable argsort, scipy softmax), identity and
one-hot matrices, and brute force on small inputs.
"""
import os

import numpy as np
import pytest

import oracle
from oracle import pack
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_fixture(name):
    hexs, rows = None, []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("hex "):
                hexs = bytes.fromhex(line[4:])
            else:
                rows.append(line.split())
    return np.frombuffer(hexs, np.uint8).copy(), rows


# --------------------------------------------------------------- scalars

def test_fp16_decode_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # textbook values: 1.0, smallest subnormal, largest normal
    assert oracle.half_to_double(0x3C00) == 1.0
    assert oracle.half_to_double(0x0001) == 2.0 ** -24
    assert oracle.half_to_double(0x7BFF) == 65504.0


def test_bf16_decode():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 65536, 4000).astype(np.uint16)
    with np.errstate(invalid="ignore"):
        ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    got = np.array([oracle.bf16_to_double(int(b)) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(got[~nan], ref[~nan])
    assert oracle.bf16_to_double(0x3F80) == 1.0


# --------------------------------------------------------------- block layouts

def test_q6k_hand_block():
    blk, rows = _read_fixture("q6k_block_hand.txt")
    assert blk.size == 210
    codes = oracle.q6k_codes(blk)
    w = oracle.dequant(oracle.Q6_K, blk, 1, 256)[0]
    for i, q, sc, wt in rows:
        i = int(i)
        assert codes[i] == int(q), i
        assert w[i] == float(wt), i
    # same bytes with d = smallest fp16 subnormal: every weight scales by 2^-24
    blk2 = blk.copy()
    blk2[208], blk2[209] = 0x01, 0x00
    w2 = oracle.dequant(oracle.Q6_K, blk2, 1, 256)[0]
    assert np.array_equal(w2, w * 2.0 ** -24)


def test_q4_0_hand_block():
    blk, rows = _read_fixture("q4_0_block_hand.txt")
    w = oracle.dequant(oracle.Q4_0, blk, 1, 32)[0]
    for i, q, wt in rows:
        assert w[int(i)] == float(wt)


def test_q8_0_hand_block():
    blk, rows = _read_fixture("q8_0_block_hand.txt")
    w = oracle.dequant(oracle.Q8_0, blk, 1, 32)[0]
    for i, q, wt in rows:
        assert w[int(i)] == float(wt)


@pytest.mark.parametrize("d", [1.0, 3.0517578125e-05, 1.7881393432617188e-07, -0.000244140625])
def test_q6k_closed_form_all_codes_and_scales(d):
    """w = d * sc * (q - 32) for all 64 codes x 64 scales (normal, subnormal d)."""
    d_bits = pack.f16_bits(d)
    dval = float(np.array([d_bits], np.uint16).view(np.float16)[0])
    codes = np.arange(256) % 64
    for sc in range(-32, 32):
        blk = pack.pack_q6k_block(codes, np.full(16, sc), d_bits)
        w = oracle.dequant(oracle.Q6_K, blk, 1, 256)[0]
        ref = dval * sc * (codes - 32).astype(np.float64)
        assert np.array_equal(w, ref)
        assert np.array_equal(w.astype(np.float32).astype(np.float64), w)  # exact in fp32


def test_q6k_codes_permuted():
    """every element position decodes its own code (no index mix-up)"""
    rng = np.random.default_rng(7)
    for _ in range(8):
        codes = rng.integers(0, 64, 256)
        scales = rng.integers(-32, 32, 16)
        blk = pack.pack_q6k_block(codes, scales, pack.f16_bits(1.0))
        assert np.array_equal(oracle.q6k_codes(blk), codes)
        w = oracle.dequant(oracle.Q6_K, blk, 1, 256)[0]
        assert np.array_equal(w, scales[np.arange(256) // 16] * (codes - 32.0))


def test_q4_0_and_q8_0_closed_form():
    for d in [0.5, 6.103515625e-05, 5.960464477539063e-08]:
        db = pack.f16_bits(d)
        dv = float(np.array([db], np.uint16).view(np.float16)[0])
        codes = np.arange(32) % 16
        w = oracle.dequant(oracle.Q4_0, pack.pack_q4_0_block(codes, db), 1, 32)[0]
        assert np.array_equal(w, dv * (codes - 8.0))
        vals = np.concatenate([np.arange(-127, -111), np.arange(112, 128)])
        w = oracle.dequant(oracle.Q8_0, pack.pack_q8_0_block(vals, db), 1, 32)[0]
        assert np.array_equal(w, dv * vals)


def test_synth_fields_land_where_the_layout_says():
    """generator draws: q6_K codes cover 0..63, scales -32..31, d >= 0 fp16"""
    W = synth.q6k_matrix(5, 64, 512)
    blocks = W.reshape(-1, 210)
    sc = blocks[:, 192:208].view(np.int8)
    assert sc.min() == -32 and sc.max() == 31
    d = blocks[:, 208:210].copy().view(np.float16).astype(np.float64)
    assert (d >= 0).all() and d.max() < 2e-3
    codes = np.concatenate([oracle.q6k_codes(b) for b in blocks[:16]])
    assert codes.min() == 0 and codes.max() == 63


# --------------------------------------------------------------- K-quant ladder formats

def _f16(v):
    return float(np.array([pack.f16_bits(v)], np.uint16).view(np.float16)[0])


@pytest.mark.parametrize("fmt,name", [(oracle.Q4_K, "q4k_block_hand.txt"),
                                      (oracle.Q2_K, "q2k_block_hand.txt")])
def test_kq_hand_block(fmt, name):
    blk, rows = _read_fixture(name)
    assert blk.size == oracle.BLOCK_BYTES[fmt]
    codes = oracle.kq_codes(fmt, blk)
    w = oracle.dequant(fmt, blk, 1, 256)[0]
    for i, q, j, wt in rows:
        assert codes[int(i)] == int(q), i
        assert w[int(i)] == float(wt), i


def test_q4k_hand_block_scales_and_mins():
    blk, _ = _read_fixture("q4k_block_hand.txt")
    got = [oracle.kq_scale_min(oracle.Q4_K, blk, j) for j in range(8)]
    assert got == list(zip([1, 2, 3, 4, 17, 33, 50, 63], [0, 5, 10, 63, 16, 31, 47, 2]))


def test_q2k_hand_block_scales_and_mins():
    blk, _ = _read_fixture("q2k_block_hand.txt")
    assert [oracle.kq_scale_min(oracle.Q2_K, blk, j) for j in range(16)] == \
        [(j, 15 - j) for j in range(16)]


KQ = [(oracle.Q4_K, pack.pack_q4k_block, 15, 32, 63), (oracle.Q2_K, pack.pack_q2k_block, 3, 16, 15)]


@pytest.mark.parametrize("fmt,packer,qmax,sub,smax", KQ)
def test_kq_one_hot_positions(fmt, packer, qmax, sub, smax):
    """a single nonzero code at position i decodes to a single nonzero weight
    at i (unit scales, zero mins): the element order of the layout"""
    ones, zeros = np.ones(256 // sub, int), np.zeros(256 // sub, int)
    for i in range(256):
        codes = np.zeros(256, int)
        codes[i] = qmax
        w = oracle.dequant(fmt, packer(codes, ones, zeros, pack.f16_bits(1.0), 0), 1, 256)[0]
        assert w[i] == qmax and np.count_nonzero(w) == 1, i


@pytest.mark.parametrize("fmt,packer,qmax,sub,smax", KQ)
def test_kq_closed_form_every_scale_and_min(fmt, packer, qmax, sub, smax):
    """w = d * scale_j * q - dmin * min_j for every scale and min value of
    every sub-block (the others random), d and dmin exact fp16 values"""
    rng = np.random.default_rng(11)
    codes = rng.integers(0, qmax + 1, 256)
    d, dmin = _f16(0.0078125), _f16(3.0517578125e-05)
    for j in range(256 // sub):
        for v in range(smax + 1):
            for which in (0, 1):
                sc = rng.integers(0, smax + 1, 256 // sub)
                mn = rng.integers(0, smax + 1, 256 // sub)
                (sc if which == 0 else mn)[j] = v
                blk = packer(codes, sc, mn, pack.f16_bits(d), pack.f16_bits(dmin))
                assert oracle.kq_scale_min(fmt, blk, j) == (sc[j], mn[j])
                if v % 8 == 0:
                    w = oracle.dequant(fmt, blk, 1, 256)[0]
                    e = np.arange(256) // sub
                    assert np.array_equal(w, d * sc[e] * codes - dmin * mn[e].astype(float))


@pytest.mark.parametrize("fmt", [oracle.Q4_K, oracle.Q2_K])
def test_kq_gemv_brute_force_4x512(fmt):
    """float matvec = numpy matmul of the dequantized rows built by the
    independent encoder; the bound's scale is the two-term magnitude sum"""
    packer, qmax, sub, smax = {oracle.Q4_K: (pack.pack_q4k_block, 15, 32, 63),
                               oracle.Q2_K: (pack.pack_q2k_block, 3, 16, 15)}[fmt]
    N, K = 4, 512
    rng = np.random.default_rng(5)
    codes = rng.integers(0, qmax + 1, (N, K))
    sc = rng.integers(0, smax + 1, (N, K // sub))
    mn = rng.integers(0, smax + 1, (N, K // sub))
    dv = np.array([[_f16(0.001 * (n + 1) + 0.0002 * b) for b in range(K // 256)] for n in range(N)])
    mv = np.array([[_f16(0.0005 * (n + 2) + 0.0001 * b) for b in range(K // 256)] for n in range(N)])
    W = pack.pack_kq_matrix(packer, codes, sc, mn,
                            np.vectorize(pack.f16_bits)(dv), np.vectorize(pack.f16_bits)(mv))
    e, blk = np.arange(K) // sub, np.arange(K) // 256
    pos = dv[:, blk] * sc[:, e] * codes
    neg = mv[:, blk] * mn[:, e]
    dense = pos - neg
    assert np.array_equal(oracle.dequant(fmt, W, N, K), dense)
    x = synth.normal_f32(21, (3, K))
    y, a = oracle.gemv_float(fmt, W, x, N, K)
    ref = x.astype(np.float64) @ dense.T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(a, np.abs(x.astype(np.float64)) @ (np.abs(pos) + np.abs(neg)).T, rtol=1e-12)


def test_kq_synth_fields_land_where_the_layout_says():
    for fmt, qmax, smax, nsub in [(oracle.Q4_K, 15, 63, 8), (oracle.Q2_K, 3, 15, 16)]:
        W = synth.matrix(fmt, 6, 32, 1024).reshape(-1, oracle.BLOCK_BYTES[fmt])
        sm = np.array([oracle.kq_scale_min(fmt, b, j) for b in W[:64] for j in range(nsub)])
        assert sm.min() == 0 and sm.max() == smax
        codes = np.concatenate([oracle.kq_codes(fmt, b) for b in W[:8]])
        assert codes.min() == 0 and codes.max() == qmax
        o = synth.KQ_D_OFF[fmt]
        for off in (o, o + 2):
            v = W[:, off:off + 2].copy().view(np.float16).astype(np.float64)
            assert (v >= 0).all() and v.max() < 2e-3 and v.max() > 0


def test_kq_q8_path_is_refused():
    W = synth.matrix(oracle.Q4_K, 1, 8, 256)
    xq, s = oracle.quantize_q8(synth.normal_f32(1, (1, 256)))
    with pytest.raises(ValueError):
        oracle.gemv_q8(oracle.Q4_K, W, xq, s, 8, 256)


# --------------------------------------------------------------- float matvec

def _identity_q6k(n):
    codes = np.full((n, n), 32)
    np.fill_diagonal(codes, 33)
    return pack.pack_q6k_matrix(codes, np.ones((n, n // 16), int),
                                np.full((n, n // 256), pack.f16_bits(1.0)))


def test_gemv_identity_returns_x_bitwise():
    n = 256
    W = _identity_q6k(n)
    x = synth.normal_f32(3, (2, n))
    y, _ = oracle.gemv_float(oracle.Q6_K, W, x, n, n)
    assert np.array_equal(y, x.astype(np.float64))
    xb = synth.normal_bf16(4, (1, n))
    y, _ = oracle.gemv_float(oracle.Q6_K, W, xb, n, n)
    assert np.array_equal(y[0], synth.bf16_bits_to_f32(xb[0]).astype(np.float64))


def test_gemv_one_hot_rows():
    N, K = 4, 512
    rng = np.random.default_rng(3)
    codes = np.full((N, K), 32)
    ks = rng.integers(0, K, N)
    qs = rng.integers(0, 64, N)
    for n in range(N):
        codes[n, ks[n]] = qs[n]
    scales = rng.integers(-32, 32, (N, K // 16))
    d = np.full((N, K // 256), pack.f16_bits(0.0078125))
    W = pack.pack_q6k_matrix(codes, scales, d)
    x = synth.normal_f32(9, (1, K))
    y, _ = oracle.gemv_float(oracle.Q6_K, W, x, N, K)
    for n in range(N):
        w = 0.0078125 * scales[n, ks[n] // 16] * (qs[n] - 32)
        assert y[0, n] == w * float(x[0, ks[n]])


@pytest.mark.parametrize("fmt", [oracle.Q6_K, oracle.Q4_0, oracle.Q8_0])
def test_gemv_brute_force_4x256(fmt):
    """blocked oracle vs numpy matmul of the dense matrix built from logical values"""
    N, K = 4, 256
    rng = np.random.default_rng(fmt)
    if fmt == oracle.Q6_K:
        codes = rng.integers(0, 64, (N, K))
        scales = rng.integers(-32, 32, (N, K // 16))
        dv = np.abs(rng.normal(size=(N, K // 256))) * 2e-4
        db = dv.astype(np.float16).view(np.uint16)
        W = pack.pack_q6k_matrix(codes, scales, db)
        dense = (db.view(np.float16).astype(np.float64).repeat(256, 1)
                 * scales.repeat(16, 1) * (codes - 32))
    elif fmt == oracle.Q4_0:
        codes = rng.integers(0, 16, (N, K))
        db = (np.abs(rng.normal(size=(N, K // 32))) * 2e-4).astype(np.float16).view(np.uint16)
        W = pack.pack_q4_0_matrix(codes, db)
        dense = db.view(np.float16).astype(np.float64).repeat(32, 1) * (codes - 8)
    else:
        vals = rng.integers(-127, 128, (N, K))
        db = (np.abs(rng.normal(size=(N, K // 32))) * 2e-4).astype(np.float16).view(np.uint16)
        W = pack.pack_q8_0_matrix(vals, db)
        dense = db.view(np.float16).astype(np.float64).repeat(32, 1) * vals
    assert np.array_equal(oracle.dequant(fmt, W, N, K), dense)
    x = rng.normal(size=(3, K)).astype(np.float32)
    y, a = oracle.gemv_float(fmt, W, x, N, K)
    ref = x.astype(np.float64) @ dense.T
    assert np.allclose(y, ref, rtol=1e-13, atol=1e-18)
    assert np.allclose(a, np.abs(x.astype(np.float64)) @ np.abs(dense).T, rtol=1e-13)
    # integer-valued activations: every partial sum is exact, so equality is exact
    xi = rng.integers(-8, 9, (2, K)).astype(np.float32)
    yi, _ = oracle.gemv_float(fmt, W, xi, N, K)
    assert np.array_equal(yi, xi.astype(np.float64) @ dense.T)


# --------------------------------------------------------------- q8 quantizer

def test_quantizer_hand_vectors():
    with open(os.path.join(GOLDEN, "q8_quantizer_hand.txt")) as f:
        lines = [l.split() for l in f if l.strip() and not l.startswith("#")]
    xs = [np.array(l[1:], np.float32) for l in lines if l[0] == "x"]
    qs = [np.array(l[1:], np.int64) for l in lines if l[0] == "q"]
    x = np.concatenate(xs)[None, :]
    xq, s = oracle.quantize_q8(x)
    assert np.array_equal(xq[0], np.concatenate(qs))
    assert s[0, 0] == np.float32(1.0)
    assert s[0, 1] == np.float32(0.0)
    assert s[0, 2] == np.float32(3.0) / np.float32(127.0)


def test_quantizer_scale_underflow_gives_zeros():
    """amax so small that amax/127 rounds to 0 in fp32: the block is all zeros"""
    x = np.zeros((1, 32), np.float32)
    x[0, 5] = np.float32(1e-45)  # smallest fp32 subnormal
    x[0, 6] = -np.float32(1e-45)
    xq, s = oracle.quantize_q8(x)
    assert s[0, 0] == 0.0 and not xq.any()
    x[0, 5] = np.float32(2e-38)  # normal tiny amax: scale stays non-zero
    xq, s = oracle.quantize_q8(x)
    assert s[0, 0] == np.float32(2e-38) / np.float32(127.0) and xq[0, 5] == 127


def test_quantizer_amax_maps_to_127_and_range():
    x = synth.normal_f32(11, (8, 1024))
    xq, s = oracle.quantize_q8(x)
    blocks = x.reshape(8, 32, 32)
    qb = xq.reshape(8, 32, 32).astype(np.int64)
    amax_pos = np.abs(blocks).argmax(axis=2)
    got = np.take_along_axis(qb, amax_pos[..., None], 2)[..., 0]
    sign = np.sign(np.take_along_axis(blocks, amax_pos[..., None], 2)[..., 0])
    assert np.array_equal(got, (127 * sign).astype(np.int64))
    assert xq.min() >= -127
    # reconstruction error within half a quantization step
    rec = qb * s.reshape(8, 32, 1).astype(np.float64)
    assert (np.abs(rec - blocks) <= 0.5 * s.reshape(8, 32, 1) * (1 + 1e-6)).all()


def test_quantizer_bf16_equals_f32_of_same_values():
    xb = synth.normal_bf16(12, (4, 256))
    xf = synth.bf16_bits_to_f32(xb).reshape(4, 256)
    a = oracle.quantize_q8(xb)
    b = oracle.quantize_q8(xf)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


# --------------------------------------------------------------- integer matvec

@pytest.mark.parametrize("fmt", [oracle.Q6_K, oracle.Q4_0, oracle.Q8_0])
def test_q8_gemv_unit_scale_is_exact_integer(fmt):
    """d = 1, sub-block scales 1 and activation scale 1 (x integer, amax 127):
    the quantized path reduces to an integer matmul, exactly."""
    N, K = 5, 512
    rng = np.random.default_rng(20 + fmt)
    one = pack.f16_bits(1.0)
    if fmt == oracle.Q6_K:
        codes = rng.integers(0, 64, (N, K))
        W = pack.pack_q6k_matrix(codes, np.ones((N, K // 16), int), np.full((N, K // 256), one))
        wint = codes - 32
    elif fmt == oracle.Q4_0:
        codes = rng.integers(0, 16, (N, K))
        W = pack.pack_q4_0_matrix(codes, np.full((N, K // 32), one))
        wint = codes - 8
    else:
        wint = rng.integers(-127, 128, (N, K))
        W = pack.pack_q8_0_matrix(wint, np.full((N, K // 32), one))
    x = rng.integers(-127, 128, (3, K))
    x[:, ::32] = 127  # every 32-block has amax 127 -> s = 1
    xq, s = oracle.quantize_q8(x.astype(np.float32))
    assert np.array_equal(xq, x) and (s == 1.0).all()
    y, _ = oracle.gemv_q8(fmt, W, xq, s, N, K)
    assert np.array_equal(y, (x @ wint.T).astype(np.float64))


def test_q6k_group_int_brute_force():
    rng = np.random.default_rng(5)
    codes = rng.integers(0, 64, (1, 512))
    W = pack.pack_q6k_matrix(codes, rng.integers(-32, 32, (1, 32)),
                             np.full((1, 2), pack.f16_bits(1.0)))
    xq = rng.integers(-127, 128, 512).astype(np.int8)
    for g in range(32):
        ref = int(np.dot(xq[16 * g:16 * g + 16].astype(np.int64), codes[0, 16 * g:16 * g + 16] - 32))
        assert oracle.group_int(oracle.Q6_K, W, xq, g) == ref


@pytest.mark.parametrize("fmt", [oracle.Q6_K, oracle.Q4_0, oracle.Q8_0])
def test_q8_gemv_equals_float_definition_on_dequantized_x(fmt):
    """y_q8 = W_dense @ (s * x_q): the integer path is a regrouping of the
    float definition applied to the quantized activations"""
    N, K = 6, 512
    W = synth.matrix(fmt, 31, N, K)
    x = synth.normal_f32(32, (2, K))
    xq, s = oracle.quantize_q8(x)
    y, a = oracle.gemv_q8(fmt, W, xq, s, N, K)
    xhat = xq.astype(np.float64) * np.repeat(s.astype(np.float64), 32, axis=1)
    dense = oracle.dequant(fmt, W, N, K)
    ref = xhat @ dense.T
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-20)
    assert np.allclose(a, np.abs(xhat) @ np.abs(dense).T, rtol=1e-12)


def test_gemm_pairs_match_gemv_rows():
    N, K, M = 16, 512, 4
    W = synth.q6k_matrix(40, N, K)
    X = synth.normal_bf16(41, (M, K))
    xq, s = oracle.quantize_q8(X)
    y, _ = oracle.gemv_q8(oracle.Q6_K, W, xq, s, N, K)
    ms, ns = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    yp, _ = oracle.gemm_q8_pairs(oracle.Q6_K, W, K, xq, s, ms.ravel(), ns.ravel())
    assert np.array_equal(yp.reshape(M, N), y)


def test_gemv_float_pairs_match_full():
    N, K = 8, 512
    W = synth.q4_0_matrix(42, N, K)
    x = synth.normal_f32(43, (3, K))
    y, a = oracle.gemv_float(oracle.Q4_0, W, x, N, K)
    bs, ns = np.meshgrid(np.arange(3), np.arange(N), indexing="ij")
    yp, ap = oracle.gemv_float_pairs(oracle.Q4_0, W, K, x, bs.ravel(), ns.ravel())
    assert np.array_equal(yp.reshape(3, N), y) and np.array_equal(ap.reshape(3, N), a)


# --------------------------------------------------------------- plane

def test_plane_is_centered_codes():
    rng = np.random.default_rng(8)
    N, K = 3, 768
    codes = rng.integers(0, 64, (N, K))
    W = pack.pack_q6k_matrix(codes, rng.integers(-32, 32, (N, K // 16)),
                             np.full((N, K // 256), pack.f16_bits(0.5)))
    assert np.array_equal(oracle.plane_q6k(W, N, K), (codes - 32).astype(np.int8))


# --------------------------------------------------------------- routing / MoE

def test_route_topk_matches_stable_sort_and_scipy_softmax():
    from scipy.special import softmax
    logits = synth.normal_f32(50, (16, 256))
    logits[3, 10] = logits[3, 200] = 9.0  # a tie: the lower index must come first
    idx, gate = oracle.route_topk_softmax(logits, 8)
    for t in range(16):
        ref = np.argsort(-logits[t].astype(np.float64), kind="stable")[:8]
        assert np.array_equal(idx[t], ref)
        assert np.allclose(gate[t], softmax(logits[t, ref].astype(np.float64)), rtol=1e-14)
    assert list(idx[3, :2]) == [10, 200]
    assert np.allclose(gate.sum(1), 1.0, rtol=1e-15)


def _dense_ffn(fmt, wg, wu, wd, H, I, x):
    g = oracle.dequant(fmt, wg, I, H) @ x
    u = oracle.dequant(fmt, wu, I, H) @ x
    h = g / (1.0 + np.exp(-g)) * u
    return oracle.dequant(fmt, wd, H, I) @ h


def test_moe_single_expert_is_plain_swiglu_ffn():
    H, I, E = 64, 96, 4
    fmt = oracle.Q4_0
    wg = [synth.q4_0_matrix(60 + e, I, H) for e in range(E)]
    wu = [synth.q4_0_matrix(70 + e, I, H) for e in range(E)]
    wd = [synth.q4_0_matrix(80 + e, H, I) for e in range(E)]
    x = synth.normal_f32(61, (2, H))
    idx = np.array([[2], [0]], np.int32)
    gate = np.ones((2, 1))
    y, bound = oracle.moe_float(fmt, H, I, wg, wu, wd, idx, gate, x)
    for t in range(2):
        ref = _dense_ffn(fmt, wg[idx[t, 0]], wu[idx[t, 0]], wd[idx[t, 0]], H, I,
                         x[t].astype(np.float64))
        assert np.allclose(y[t], ref, rtol=1e-12, atol=1e-15)
    assert (bound > 0).all()


def test_moe_identical_experts_sum_of_gates_is_one():
    H, I, E, k = 64, 32, 8, 4
    fmt = oracle.Q4_0
    g0 = synth.q4_0_matrix(90, I, H)
    u0 = synth.q4_0_matrix(91, I, H)
    d0 = synth.q4_0_matrix(92, H, I)
    x = synth.normal_bf16(93, (3, H))
    logits = synth.normal_f32(94, (3, E))
    idx, gate = oracle.route_topk_softmax(logits, k)
    y, _ = oracle.moe_float(fmt, H, I, [g0] * E, [u0] * E, [d0] * E, idx, gate, x)
    for t in range(3):
        ref = _dense_ffn(fmt, g0, u0, d0, H, I, synth.bf16_bits_to_f32(x[t]).astype(np.float64))
        assert np.allclose(y[t], ref, rtol=1e-12, atol=1e-15)


# --------------------------------------------------------------- MoE prefill (quantized activations)

def _moe_q8_single(fmt, Wg, Wu, Wd, H, I, x_row):
    """one expert's FFN composed from the pinned primitives: quantize, q8
    matvec, numpy silu, quantize of fp32 h, q8 matvec"""
    xq, sx = oracle.quantize_q8(x_row[None, :])
    g, _ = oracle.gemv_q8(fmt, Wg, xq, sx, I, H)
    u, _ = oracle.gemv_q8(fmt, Wu, xq, sx, I, H)
    with np.errstate(over="ignore"):
        h = (g / (1.0 + np.exp(-g))) * u
    hq, sh = oracle.quantize_q8(h.astype(np.float32))
    o, _ = oracle.gemv_q8(fmt, Wd, hq, sh, H, I)
    return o[0]


@pytest.mark.parametrize("fmt", [oracle.Q4_0, oracle.Q6_K])
def test_moe_q8_is_the_composition_of_pinned_steps(fmt):
    E, H, I, T, k = 3, 512, 256, 4, 2
    wg = [synth.matrix(fmt, 60 + e, I, H) for e in range(E)]
    wu = [synth.matrix(fmt, 70 + e, I, H) for e in range(E)]
    wd = [synth.matrix(fmt, 80 + e, H, I) for e in range(E)]
    x = synth.to_bf16_bits(synth.normal_f32(90, (T, H)) * 1000)
    idx = np.array([[0, 2], [1, 0], [2, 1], [1, 2]], np.int32)
    gate = np.array([[0.25, 0.75], [0.5, 0.5], [1.0, 0.0], [0.125, 0.875]])
    y, tight, loose = oracle.moe_q8(fmt, H, I, wg, wu, wd, idx, gate, x)
    xf = synth.bf16_bits_to_f32(x)
    for t in range(T):
        ref = sum(gate[t, j] * _moe_q8_single(fmt, wg[idx[t, j]], wu[idx[t, j]], wd[idx[t, j]], H, I, xf[t])
                  for j in range(k))
        assert np.allclose(y[t], ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max()), t
    assert (tight > 0).all() and (loose >= tight).all()


# --------------------------------------------------------------- additive codebooks

def _f16bits(vals):
    return np.asarray(vals, np.float64).astype(np.float16).view(np.uint16)


def test_cbk_hand_matrix():
    """M = 2, one row of two groups, scale 2, hand-derived weights"""
    books = np.zeros((2, 256, 8))
    books[0, 3] = [1, 2, 3, 4, 0.5, 0.25, -1, -2]
    books[0, 200] = [0.125, 0, 0, 0, 0, 0, 0, 8]
    books[1, 7] = [-1, -1, -1, -1, 1, 1, 1, 1]
    books[1, 255] = [0, 0.5, 0, 0.5, 0, 0.5, 0, 0.5]
    codes = np.array([[[3, 7], [200, 255]]], np.uint8)
    w = oracle.cbk_dequant(2, codes, _f16bits(books), _f16bits([2.0]), 1, 16)[0]
    assert list(w) == [0, 2, 4, 6, 3, 2.5, 0, -2, 0.25, 1, 0, 1, 0, 1, 0, 17]


@pytest.mark.parametrize("M", [2, 3])
def test_cbk_one_hot_books_reveal_the_codes(M):
    """book 0 entry c = (c + 1) at position c % 8, the other books zero: each
    weight shows which code of which group the layout picked"""
    N, K = 3, 64
    books = np.zeros((M, 256, 8))
    for c in range(256):
        books[0, c, c % 8] = c + 1
    rng = np.random.default_rng(M)
    codes = rng.integers(0, 256, (N, K // 8, M)).astype(np.uint8)
    w = oracle.cbk_dequant(M, codes, _f16bits(books), _f16bits([1.0, 0.5, 4.0]), N, K)
    sc = [1.0, 0.5, 4.0]
    for n in range(N):
        for g in range(K // 8):
            c = int(codes[n, g, 0])
            expect = np.zeros(8)
            expect[c % 8] = sc[n] * (c + 1)
            assert np.array_equal(w[n, 8 * g:8 * g + 8], expect), (n, g)


def test_cbk_books_add_and_scales_multiply():
    """three books = the sum of the one-book matrices; a row's scale
    multiplies its weights"""
    codes, books, scales = synth.cbk_matrix(9, 3, 4, 128)
    w3 = oracle.cbk_dequant(3, codes, books, scales, 4, 128)
    parts = []
    for m in range(3):
        bm = np.zeros_like(books)
        bm[0] = books[m]
        cm = np.zeros_like(codes[:, :, :2])
        cm[:, :, 0] = codes[:, :, m]
        parts.append(oracle.cbk_dequant(2, cm, bm[:2], scales, 4, 128))
    assert np.allclose(w3, parts[0] + parts[1] + parts[2], rtol=0, atol=1e-15)
    s2 = _f16bits(2.0 * scales.view(np.float16).astype(np.float64))
    assert np.array_equal(oracle.cbk_dequant(3, codes, books, s2, 4, 128), 2.0 * w3)


@pytest.mark.parametrize("M", [2, 3])
def test_cbk_gemv_brute_force(M):
    codes, books, scales = synth.cbk_matrix(11 + M, M, 5, 256)
    w = oracle.cbk_dequant(M, codes, books, scales, 5, 256)
    x = synth.normal_f32(12, (3, 256))
    y, a = oracle.cbk_gemv(M, codes, books, scales, x, 5, 256)
    assert np.allclose(y, x.astype(np.float64) @ w.T, rtol=1e-12, atol=1e-15)
    assert (a >= np.abs(x.astype(np.float64)) @ np.abs(w).T * (1 - 1e-12)).all()
