"""Planted mistakes: each mutant of the oracle's C source (a dropped term, a
wrong shift or index, a wrong rounding) is compiled on the CPU and must be
caught by the same hand-built fixtures and closed forms the pins use."""
import ctypes as C
import os
import subprocess

import numpy as np
import pytest

import oracle
from oracle import pack

SRC = os.path.join(os.path.dirname(oracle.__file__), "qmm_oracle.c")

MUTANTS = {
    "nibble_select": ("(ql[i % 128] >> (4 * (i / 128)))", "(ql[i % 128] >> (4 * (i / 64 % 2)))"),
    "qh_shift": ("(qh[i % 64] >> (2 * (i / 64)))", "(qh[i % 64] >> (2 * (i / 32 % 4)))"),
    "no_center": ("return sc * (orc_q6k_code(blk, i) - 32);", "return sc * orc_q6k_code(blk, i);"),
    "scale_index": ("int sc = (int8_t)blk[192 + i / 16];", "int sc = (int8_t)blk[192 + i / 32];"),
    "q4_offset": ("return q - 8;", "return q - 7;"),
    "round_away": ("float rq = nearbyintf(t);", "float rq = roundf(t);"),
    "d_offset": ("int off = (fmt == ORC_Q6_K) ? 208 : 0;", "int off = (fmt == ORC_Q6_K) ? 206 : 0;"),
    "q4k_scale_top_bits": ("*scale = (b[j + 4] & 15) | ((b[j - 4] >> 6) << 4);",
                           "*scale = (b[j + 4] & 15) | ((b[j] >> 6) << 4);"),
    "q4k_nibble": ("(qs[32 * (i / 64) + i % 32] >> (4 * ((i / 32) % 2)))",
                   "(qs[32 * (i / 64) + i % 32] >> (4 * ((i / 64) % 2)))"),
    "q2k_shift": ("(qs[32 * (i / 128) + i % 32] >> (2 * ((i % 128) / 32)))",
                  "(qs[32 * (i / 128) + i % 32] >> (2 * ((i % 64) / 16)))"),
    "q2k_min_nibble": ("*min = blk[j] >> 4;", "*min = blk[j] & 15;"),
    "kq_min_sign": ("return pos - neg;", "return pos + neg;"),
    "cbk_code_order": ("int c = codes[(n * (K / 8) + g) * M + m];", "int c = codes[(n * (K / 8) + m) * M + g % M];"),
    "cbk_lane_flip": ("t[m] = s * orc_half_to_double(books[((int64_t)m * 256 + c) * 8 + j]);",
                      "t[m] = s * orc_half_to_double(books[((int64_t)m * 256 + c) * 8 + (7 - j)]);"),
}


def _build(name, tmp_path):
    src = open(SRC).read()
    a, b = MUTANTS[name]
    assert a in src, name
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(a, b))
    so = tmp_path / f"{name}.so"
    subprocess.run(["gcc", "-O1", "-fPIC", "-shared", "-ffp-contract=off", "-o", str(so),
                    str(path), "-lm"], check=True)
    L = C.CDLL(str(so))
    L.orc_dequant_row.argtypes = [C.c_int, C.c_void_p, C.c_int64, C.c_void_p]
    L.orc_quantize_q8.argtypes = [C.c_void_p, C.c_int, C.c_int64, C.c_int64, C.c_void_p,
                                  C.c_void_p]
    return L


def _dequant(L, fmt, blk, K):
    out = np.empty(K, np.float64)
    b = np.ascontiguousarray(blk)
    L.orc_dequant_row(fmt, b.ctypes.data, K, out.ctypes.data)
    return out


def _pins_pass(L) -> bool:
    rng = np.random.default_rng(0)
    codes = rng.integers(0, 64, 256)
    scales = rng.integers(-32, 32, 16)
    blk = pack.pack_q6k_block(codes, scales, pack.f16_bits(0.5))
    if not np.array_equal(_dequant(L, oracle.Q6_K, blk, 256),
                          0.5 * scales[np.arange(256) // 16] * (codes - 32.0)):
        return False
    c4 = np.arange(32) % 16
    if not np.array_equal(_dequant(L, oracle.Q4_0, pack.pack_q4_0_block(c4, pack.f16_bits(1.0)), 32),
                          c4 - 8.0):
        return False
    for fmt, packer, qmax, sub, smax in [(oracle.Q4_K, pack.pack_q4k_block, 15, 32, 63),
                                         (oracle.Q2_K, pack.pack_q2k_block, 3, 16, 15)]:
        kc = rng.integers(0, qmax + 1, 256)
        ks = rng.integers(0, smax + 1, 256 // sub)
        km = rng.integers(0, smax + 1, 256 // sub)
        blk = packer(kc, ks, km, pack.f16_bits(0.5), pack.f16_bits(0.25))
        e = np.arange(256) // sub
        if not np.array_equal(_dequant(L, fmt, blk, 256), 0.5 * ks[e] * kc - 0.25 * km[e]):
            return False
    # additive codebooks: one-hot books reveal the code and lane order
    cb = np.zeros((2, 256, 8))
    for c in range(256):
        cb[0, c, c % 8] = c + 1
    cbits = cb.astype(np.float16).view(np.uint16)
    codes = rng.integers(0, 256, (1, 4, 2)).astype(np.uint8)
    sc = np.array([1.0], np.float16).view(np.uint16)
    L.orc_cbk_weight.restype = C.c_double
    L.orc_cbk_weight.argtypes = [C.c_int, C.c_void_p, C.c_void_p, C.c_void_p, C.c_int64, C.c_int64, C.c_int64]
    for k in range(32):
        c = int(codes[0, k // 8, 0])
        want = (c + 1.0) if k % 8 == c % 8 else 0.0
        if L.orc_cbk_weight(2, codes.ctypes.data, cbits.ctypes.data, sc.ctypes.data, 32, 0, k) != want:
            return False
    x = np.array([[127, 2.5, -2.5, 3.5] + [0.0] * 28], np.float32)
    xq = np.empty((1, 32), np.int8)
    s = np.empty((1, 1), np.float32)
    L.orc_quantize_q8(x.ctypes.data, 0, 1, 32, xq.ctypes.data, s.ctypes.data)
    return list(xq[0, :4]) == [127, 2, -2, 4]


def test_unmutated_oracle_passes_mutant_harness(tmp_path):
    assert _pins_pass(oracle.lib())


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    assert not _pins_pass(_build(name, tmp_path))
