"""Block encoders: logical values -> packed bytes (test infrastructure).

Written from the layout definition, independently of both the C oracle's
decoder and the CUDA decoders, so that tests can build structured matrices
(identity, one-hot, unit scales) and check the decoders against values chosen
by the test.

q6_K super-block (210 B): ql[128] | qh[64] | scales[16] (int8) | d (fp16 LE).
  element i: low 4 bits in ql[i % 128] (low nibble if i < 128, else high),
             high 2 bits in qh[i % 64] at bit 2 * (i // 64),
             scale scales[i // 16]; weight = d * scale * (q - 32).
Q4_0 block (18 B): d (fp16 LE) | qs[16]; element i in qs[i % 16], low nibble
  if i < 16 else high; weight = d * (q - 8).
Q8_0 block (34 B): d (fp16 LE) | qs[32] (int8); weight = d * q.
Q4_K super-block (144 B): d | dmin (fp16 LE) | 12 bytes of 6-bit scales and
  mins | qs[128]. Sub-block j (32 weights): j < 4: scale in bits 0-5 of byte
  j, min in bits 0-5 of byte j + 4; j >= 4: byte j + 4 = (scale & 15) |
  (min & 15) << 4, scale >> 4 in bits 6-7 of byte j - 4, min >> 4 in bits 6-7
  of byte j. Element i: nibble (i // 32) % 2 of qs[32 * (i // 64) + i % 32];
  weight = d * scale * q - dmin * min.
Q2_K super-block (84 B): scales[16] (low nibble scale, high nibble min of
  sub-block i // 16) | qs[64] | d | dmin (fp16 LE). Element i: bits
  2 * ((i % 128) // 32) of qs[32 * (i // 128) + i % 32].
"""
from __future__ import annotations

import numpy as np


def f16_bits(v: float) -> int:
    return int(np.array([v], np.float16).view(np.uint16)[0])


def pack_q6k_block(codes, scales, d_bits: int) -> np.ndarray:
    codes = np.asarray(codes, np.int64)
    scales = np.asarray(scales, np.int64)
    assert codes.shape == (256,) and scales.shape == (16,)
    assert codes.min() >= 0 and codes.max() <= 63
    assert scales.min() >= -128 and scales.max() <= 127
    blk = np.zeros(210, np.uint8)
    for i in range(256):
        q = int(codes[i])
        blk[i % 128] |= (q & 0xF) << (4 * (i // 128))
        blk[128 + i % 64] |= (q >> 4) << (2 * (i // 64))
    blk[192:208] = scales.astype(np.int8).view(np.uint8)
    blk[208] = d_bits & 0xFF
    blk[209] = (d_bits >> 8) & 0xFF
    return blk


def pack_q4_0_block(codes, d_bits: int) -> np.ndarray:
    codes = np.asarray(codes, np.int64)
    assert codes.shape == (32,) and codes.min() >= 0 and codes.max() <= 15
    blk = np.zeros(18, np.uint8)
    blk[0] = d_bits & 0xFF
    blk[1] = (d_bits >> 8) & 0xFF
    for i in range(32):
        blk[2 + i % 16] |= int(codes[i]) << (4 * (i // 16))
    return blk


def pack_q8_0_block(vals, d_bits: int) -> np.ndarray:
    vals = np.asarray(vals, np.int64)
    assert vals.shape == (32,) and vals.min() >= -128 and vals.max() <= 127
    blk = np.zeros(34, np.uint8)
    blk[0] = d_bits & 0xFF
    blk[1] = (d_bits >> 8) & 0xFF
    blk[2:34] = vals.astype(np.int8).view(np.uint8)
    return blk


def pack_q6k_matrix(codes, scales, d_bits) -> np.ndarray:
    """codes [N][K] (0..63), scales [N][K/16], d_bits [N][K/256] -> bytes."""
    codes = np.asarray(codes)
    N, K = codes.shape
    scales = np.asarray(scales).reshape(N, K // 16)
    d_bits = np.asarray(d_bits).reshape(N, K // 256)
    out = []
    for n in range(N):
        for b in range(K // 256):
            out.append(pack_q6k_block(codes[n, 256 * b:256 * (b + 1)],
                                      scales[n, 16 * b:16 * (b + 1)], int(d_bits[n, b])))
    return np.concatenate(out)


def pack_q4_0_matrix(codes, d_bits) -> np.ndarray:
    codes = np.asarray(codes)
    N, K = codes.shape
    d_bits = np.asarray(d_bits).reshape(N, K // 32)
    return np.concatenate([pack_q4_0_block(codes[n, 32 * b:32 * (b + 1)], int(d_bits[n, b]))
                           for n in range(N) for b in range(K // 32)])


def pack_q8_0_matrix(vals, d_bits) -> np.ndarray:
    vals = np.asarray(vals)
    N, K = vals.shape
    d_bits = np.asarray(d_bits).reshape(N, K // 32)
    return np.concatenate([pack_q8_0_block(vals[n, 32 * b:32 * (b + 1)], int(d_bits[n, b]))
                           for n in range(N) for b in range(K // 32)])


def pack_q4k_block(codes, scales, mins, d_bits: int, dmin_bits: int) -> np.ndarray:
    codes = np.asarray(codes, np.int64)
    scales = np.asarray(scales, np.int64)
    mins = np.asarray(mins, np.int64)
    assert codes.shape == (256,) and codes.min() >= 0 and codes.max() <= 15
    assert scales.shape == (8,) and mins.shape == (8,)
    assert min(scales.min(), mins.min()) >= 0 and max(scales.max(), mins.max()) <= 63
    blk = np.zeros(144, np.uint8)
    blk[0], blk[1] = d_bits & 0xFF, (d_bits >> 8) & 0xFF
    blk[2], blk[3] = dmin_bits & 0xFF, (dmin_bits >> 8) & 0xFF
    b = np.zeros(12, np.int64)
    for j in range(8):
        sc, mn = int(scales[j]), int(mins[j])
        if j < 4:
            b[j] |= sc
            b[j + 4] |= mn
        else:
            b[j + 4] |= (sc & 15) | ((mn & 15) << 4)
            b[j - 4] |= (sc >> 4) << 6
            b[j] |= (mn >> 4) << 6
    blk[4:16] = b.astype(np.uint8)
    for i in range(256):
        blk[16 + 32 * (i // 64) + i % 32] |= int(codes[i]) << (4 * ((i // 32) % 2))
    return blk


def pack_q2k_block(codes, scales, mins, d_bits: int, dmin_bits: int) -> np.ndarray:
    codes = np.asarray(codes, np.int64)
    scales = np.asarray(scales, np.int64)
    mins = np.asarray(mins, np.int64)
    assert codes.shape == (256,) and codes.min() >= 0 and codes.max() <= 3
    assert scales.shape == (16,) and mins.shape == (16,)
    assert min(scales.min(), mins.min()) >= 0 and max(scales.max(), mins.max()) <= 15
    blk = np.zeros(84, np.uint8)
    blk[0:16] = (scales | (mins << 4)).astype(np.uint8)
    for i in range(256):
        blk[16 + 32 * (i // 128) + i % 32] |= int(codes[i]) << (2 * ((i % 128) // 32))
    blk[80], blk[81] = d_bits & 0xFF, (d_bits >> 8) & 0xFF
    blk[82], blk[83] = dmin_bits & 0xFF, (dmin_bits >> 8) & 0xFF
    return blk


def pack_kq_matrix(pack_block, codes, scales, mins, d_bits, dmin_bits) -> np.ndarray:
    """codes [N][K], scales / mins [N][K / sub-block], d_bits / dmin_bits
    [N][K / 256] -> bytes, with pack_block one of the two K-quant packers."""
    codes = np.asarray(codes)
    N, K = codes.shape
    nsub = np.asarray(scales).size // (N * (K // 256))
    scales = np.asarray(scales).reshape(N, K // 256, nsub)
    mins = np.asarray(mins).reshape(N, K // 256, nsub)
    d_bits = np.asarray(d_bits).reshape(N, K // 256)
    dmin_bits = np.asarray(dmin_bits).reshape(N, K // 256)
    return np.concatenate([pack_block(codes[n, 256 * b:256 * (b + 1)], scales[n, b], mins[n, b],
                                      int(d_bits[n, b]), int(dmin_bits[n, b]))
                           for n in range(N) for b in range(K // 256)])
