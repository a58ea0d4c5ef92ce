"""Seeded synthetic inputs for block-quantized weight matmul.

This module only draws random numbers and places them in the byte fields of
the block formats; it holds none of the matmul arithmetic (no decoding, no
dot products, no quantization). Both the CUDA tests/bench and the CPU oracle
consume what it produces.

Generator: splitmix64 on a counter (z = seed + (i+1) * 0x9E3779B97F4A7C15,
then the published splitmix64 finalizer), one independent stream per tensor
and field. Normals: Box-Muller in float64 from two uniforms of 53 bits.

Value distributions (per block of each format):
  q6_K (210 B): ql[128] and qh[64] uniform random bytes, so every 6-bit code
      q is uniform on 0..63; scales[16] uniform on -32..31; d =
      fp16(|N(0,1)| * 2e-4) little-endian.
  Q4_0 (18 B):  d as above, then 16 uniform bytes (every nibble q uniform on
      0..15).
  Q8_0 (34 B):  d as above, then 32 int8 uniform on -127..127.
  Q4_K (144 B): d and dmin as d above, then 12 + 128 uniform bytes (every
      6-bit scale and min uniform on 0..63, every code on 0..15).
  Q2_K (84 B):  16 + 64 uniform bytes (every 4-bit scale and min uniform on
      0..15, every code on 0..3), then d and dmin as d above.
  additive codebooks: codes uniform bytes; codebook entries fp16(N(0,1) *
      0.05); row scales fp16(0.5 + U(0,1)).
  activations:  N(0,1) as float32, or rounded to bfloat16 (ties to even).
"""
from __future__ import annotations

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

Q4_0, Q8_0, Q6_K, Q4_K, Q2_K = 1, 2, 3, 4, 5
BLOCK_ELEMS = {Q4_0: 32, Q8_0: 32, Q6_K: 256, Q4_K: 256, Q2_K: 256}
BLOCK_BYTES = {Q4_0: 18, Q8_0: 34, Q6_K: 210, Q4_K: 144, Q2_K: 84}
# byte offsets of the fp16 d and dmin in a K-quant super-block
KQ_D_OFF = {Q4_K: 0, Q2_K: 80}

_CHUNK = 1 << 22  # draws per numpy pass (bounded temporaries)


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def substream(seed: int, tag: int) -> int:
    """A seed for an independent stream, derived from (seed, tag)."""
    with np.errstate(over="ignore"):
        z = _mix(np.array([np.uint64(seed & 0xFFFFFFFFFFFFFFFF) ^ np.uint64(tag * 0x100000001B3)],
                          dtype=np.uint64))
    return int(z[0])


def splitmix64(seed: int, n: int) -> np.ndarray:
    """n uint64 draws of the counter-based splitmix64 stream `seed`."""
    out = np.empty(n, np.uint64)
    s = np.uint64(seed & 0xFFFFFFFFFFFFFFFF)
    with np.errstate(over="ignore"):
        for i0 in range(0, n, _CHUNK):
            i = np.arange(i0 + 1, min(n, i0 + _CHUNK) + 1, dtype=np.uint64)
            out[i0:i0 + len(i)] = _mix(s + i * _GOLDEN)
    return out


def uniform_bytes(seed: int, nbytes: int) -> np.ndarray:
    words = splitmix64(seed, (nbytes + 7) // 8)
    return words.view(np.uint8)[:nbytes].copy()


def uniform_ints(seed: int, n: int, lo: int, hi: int) -> np.ndarray:
    """n integers uniform on [lo, hi] (multiply-shift range reduction)."""
    u = splitmix64(seed, n) >> np.uint64(32)
    span = np.uint64(hi - lo + 1)
    with np.errstate(over="ignore"):
        v = (u * span) >> np.uint64(32)
    return v.astype(np.int64) + lo


def normals(seed: int, n: int) -> np.ndarray:
    """n standard normals (float64), Box-Muller."""
    m = (n + 1) // 2
    u = splitmix64(seed, 2 * m)
    u1 = ((u[0::2] >> np.uint64(11)).astype(np.float64) + 0.5) * 2.0 ** -53
    u2 = ((u[1::2] >> np.uint64(11)).astype(np.float64) + 0.5) * 2.0 ** -53
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * m, np.float64)
    z[0::2] = r * np.cos(2.0 * np.pi * u2)
    z[1::2] = r * np.sin(2.0 * np.pi * u2)
    return z[:n]


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (uint16), round to nearest even."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + np.uint64(0x7FFF) + ((b >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return b.astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _scale_d(seed: int, nblocks: int) -> np.ndarray:
    """d = fp16(|N(0,1)| * 2e-4) as little-endian byte pairs [nblocks][2]."""
    d = (np.abs(normals(seed, nblocks)) * 2e-4).astype(np.float16)
    return d.view(np.uint8).reshape(nblocks, 2)


def q6k_matrix(seed: int, N: int, K: int) -> np.ndarray:
    """N x K q6_K weights, rows of K/256 consecutive 210-byte super-blocks."""
    assert K % 256 == 0
    nb = N * (K // 256)
    out = np.empty((nb, 210), np.uint8)
    out[:, 0:192] = uniform_bytes(substream(seed, 1), nb * 192).reshape(nb, 192)
    out[:, 192:208] = uniform_ints(substream(seed, 2), nb * 16, -32, 31).astype(
        np.int8).view(np.uint8).reshape(nb, 16)
    out[:, 208:210] = _scale_d(substream(seed, 3), nb)
    return out.reshape(-1)


def q4_0_matrix(seed: int, N: int, K: int) -> np.ndarray:
    """N x K Q4_0 weights, rows of K/32 consecutive 18-byte blocks."""
    assert K % 32 == 0
    nb = N * (K // 32)
    out = np.empty((nb, 18), np.uint8)
    out[:, 0:2] = _scale_d(substream(seed, 3), nb)
    out[:, 2:18] = uniform_bytes(substream(seed, 1), nb * 16).reshape(nb, 16)
    return out.reshape(-1)


def q8_0_matrix(seed: int, N: int, K: int) -> np.ndarray:
    """N x K Q8_0 weights, rows of K/32 consecutive 34-byte blocks."""
    assert K % 32 == 0
    nb = N * (K // 32)
    out = np.empty((nb, 34), np.uint8)
    out[:, 0:2] = _scale_d(substream(seed, 3), nb)
    out[:, 2:34] = uniform_ints(substream(seed, 1), nb * 32, -127, 127).astype(
        np.int8).view(np.uint8).reshape(nb, 32)
    return out.reshape(-1)


def kq_matrix(fmt: int, seed: int, N: int, K: int) -> np.ndarray:
    """N x K Q4_K or Q2_K weights, rows of K/256 consecutive super-blocks."""
    assert K % 256 == 0
    nb, bb, o = N * (K // 256), BLOCK_BYTES[fmt], KQ_D_OFF[fmt]
    out = uniform_bytes(substream(seed, 1), nb * bb).reshape(nb, bb)
    out[:, o:o + 2] = _scale_d(substream(seed, 3), nb)
    out[:, o + 2:o + 4] = _scale_d(substream(seed, 4), nb)
    return out.reshape(-1)


def matrix(fmt: int, seed: int, N: int, K: int) -> np.ndarray:
    if fmt in KQ_D_OFF:
        return kq_matrix(fmt, seed, N, K)
    return {Q4_0: q4_0_matrix, Q8_0: q8_0_matrix, Q6_K: q6k_matrix}[fmt](seed, N, K)


def matrix_bytes(fmt: int, N: int, K: int) -> int:
    return N * (K // BLOCK_ELEMS[fmt]) * BLOCK_BYTES[fmt]


def normal_f32(seed: int, shape) -> np.ndarray:
    n = int(np.prod(shape))
    return normals(substream(seed, 7), n).astype(np.float32).reshape(shape)


def normal_bf16(seed: int, shape) -> np.ndarray:
    """N(0,1) activations as bfloat16 bit patterns (uint16)."""
    return to_bf16_bits(normal_f32(seed, shape)).reshape(shape)


def workload_seed(config_id: int, matrix_id: int) -> int:
    return 0x5EED0000 + config_id * 16 + matrix_id


def matrix_torch(fmt: int, seed: int, N: int, K: int, device, count: int = 1):
    """`count` N x K matrices of format `fmt` drawn on `device` with torch's
    seeded generator (for workloads too large to draw on the host): the same
    per-field distributions as the numpy generators above, but a different
    random stream. Returns a uint8 tensor [count, bytes per matrix]."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(seed & 0x7FFFFFFFFFFFFFFF)
    be, bb = BLOCK_ELEMS[fmt], BLOCK_BYTES[fmt]
    nb = N * (K // be)
    out = torch.randint(0, 256, (count, nb, bb), dtype=torch.uint8, device=device, generator=g)
    d = (torch.randn((count, nb), generator=g, device=device).abs() * 2e-4).half()
    d_bytes = d.view(torch.uint8).view(count, nb, 2)
    if fmt == Q6_K:
        sc = torch.randint(-32, 32, (count, nb, 16), dtype=torch.int8, device=device, generator=g)
        out[:, :, 192:208] = sc.view(torch.uint8)
        out[:, :, 208:210] = d_bytes
    elif fmt == Q4_0:
        out[:, :, 0:2] = d_bytes
    elif fmt in KQ_D_OFF:
        o = KQ_D_OFF[fmt]
        dm = (torch.randn((count, nb), generator=g, device=device).abs() * 2e-4).half()
        out[:, :, o:o + 2] = d_bytes
        out[:, :, o + 2:o + 4] = dm.view(torch.uint8).view(count, nb, 2)
    else:
        qs = torch.randint(-127, 128, (count, nb, 32), dtype=torch.int8, device=device, generator=g)
        out[:, :, 2:34] = qs.view(torch.uint8)
        out[:, :, 0:2] = d_bytes
    return out.view(count, nb * bb)


def cbk_matrix(seed: int, M: int, N: int, K: int):
    """An N x K additive-codebook matrix with M codebooks: (codes [N][K/8][M]
    uint8, books [M][256][8] fp16 bits, scales [N] fp16 bits)."""
    assert K % 8 == 0 and M in (2, 3)
    codes = uniform_bytes(substream(seed, 1), N * (K // 8) * M).reshape(N, K // 8, M)
    books = (normals(substream(seed, 2), M * 256 * 8) * 0.05).astype(np.float16).view(np.uint16).reshape(M, 256, 8)
    u = (splitmix64(substream(seed, 3), N) >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    scales = (0.5 + u).astype(np.float16).view(np.uint16)
    return codes, books, scales
