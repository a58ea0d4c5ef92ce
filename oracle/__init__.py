"""Plain CPU oracle for block-quantized weight matmul (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package. The product library never does, and
the two share no code: the C source here is compiled on its own with gcc.

Each function is a thin numpy wrapper around ``qmm_oracle.c``; see that file
for the definitions and the passages they follow.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qmm_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

Q4_0, Q8_0, Q6_K, Q4_K, Q2_K = 1, 2, 3, 4, 5
X_F32, X_BF16 = 0, 1

BLOCK_ELEMS = {Q4_0: 32, Q8_0: 32, Q6_K: 256, Q4_K: 256, Q2_K: 256}
BLOCK_BYTES = {Q4_0: 18, Q8_0: 34, Q6_K: 210, Q4_K: 144, Q2_K: 84}
# formats whose quantized-activation (integer) path the oracle defines
Q8_FORMATS = (Q4_0, Q8_0, Q6_K)

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        L = C.CDLL(build())
        P, I64, I, D = C.c_void_p, C.c_int64, C.c_int, C.c_double
        sig = {
            "orc_half_to_double": (D, [C.c_uint16]),
            "orc_bf16_to_double": (D, [C.c_uint16]),
            "orc_block_elems": (I, [I]),
            "orc_block_bytes": (I, [I]),
            "orc_q6k_code": (I, [P, I]),
            "orc_kq_code": (I, [I, P, I]),
            "orc_kq_scale_min": (None, [I, P, I, P, P]),
            "orc_weight": (D, [I, P, I64]),
            "orc_dequant_row": (None, [I, P, I64, P]),
            "orc_gemv_float": (None, [I, P, I64, I64, P, I, I, P, P]),
            "orc_quantize_q8": (None, [P, I, I64, I64, P, P]),
            "orc_group_int": (I64, [I, P, P, I64]),
            "orc_gemv_q8": (None, [I, P, I64, I64, P, P, I, P, P]),
            "orc_gemm_q8_pairs": (None, [I, P, I64, P, P, P, P, I64, P, P]),
            "orc_gemv_float_pairs": (None, [I, P, I64, P, I, P, P, I64, P, P]),
            "orc_plane_q6k": (None, [P, I64, I64, P]),
            "orc_route_topk_softmax": (None, [P, I, I, I, P, P]),
            "orc_moe_float": (None, [I, I, I, P, P, P, I, I, P, P, P, I, P, P, P]),
            "orc_moe_q8": (None, [I, I, I, P, P, P, I, I, P, P, P, I, P, P, P]),
            "orc_cbk_weight": (D, [I, P, P, P, I64, I64, I64]),
            "orc_cbk_gemv": (None, [I, P, P, P, I64, I64, P, I, I, P, P]),
        }
        for name, (res, args) in sig.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(C.c_void_p)


def _xkind(x: np.ndarray) -> int:
    if x.dtype == np.float32:
        return X_F32
    if x.dtype == np.uint16:  # raw bfloat16 bits
        return X_BF16
    raise TypeError(f"activations must be float32 or bf16 bits (uint16), got {x.dtype}")


def half_to_double(h: int) -> float:
    return lib().orc_half_to_double(h)


def bf16_to_double(h: int) -> float:
    return lib().orc_bf16_to_double(h)


def dequant(fmt: int, W: np.ndarray, N: int, K: int) -> np.ndarray:
    """Dense [N][K] float64 weights (each value is exactly an fp32 number)."""
    out = np.empty((N, K), np.float64)
    rb = K // BLOCK_ELEMS[fmt] * BLOCK_BYTES[fmt]
    Wb = np.ascontiguousarray(W).view(np.uint8).reshape(-1)
    for n in range(N):
        row = np.ascontiguousarray(Wb[n * rb:(n + 1) * rb])
        lib().orc_dequant_row(fmt, _p(row), K, _p(out[n]))
    return out


def q6k_codes(block: np.ndarray) -> np.ndarray:
    """The 256 unsigned 6-bit codes of one q6_K super-block."""
    b = np.ascontiguousarray(block, dtype=np.uint8)
    return np.array([lib().orc_q6k_code(_p(b), i) for i in range(256)], np.int64)


def kq_codes(fmt: int, block: np.ndarray) -> np.ndarray:
    """The 256 unsigned codes of one Q4_K / Q2_K super-block."""
    b = np.ascontiguousarray(block, dtype=np.uint8)
    return np.array([lib().orc_kq_code(fmt, _p(b), i) for i in range(256)], np.int64)


def kq_scale_min(fmt: int, block: np.ndarray, j: int):
    """(scale, min) of sub-block j of one Q4_K / Q2_K super-block."""
    b = np.ascontiguousarray(block, dtype=np.uint8)
    sc, mn = C.c_int(), C.c_int()
    lib().orc_kq_scale_min(fmt, _p(b), j, C.byref(sc), C.byref(mn))
    return sc.value, mn.value


def _q8_only(fmt):
    if fmt not in Q8_FORMATS:
        raise ValueError(f"the quantized-activation path is defined for q6_K, Q4_0, Q8_0 only")


def gemv_float(fmt, W, x, N, K):
    """x: [B][K] float32 or bf16 bits -> (y [B][N] float64, sum|w x| [B][N])."""
    x = np.ascontiguousarray(x)
    B = x.shape[0]
    y = np.empty((B, N), np.float64)
    a = np.empty((B, N), np.float64)
    lib().orc_gemv_float(fmt, _p(np.ascontiguousarray(W)), N, K, _p(x), _xkind(x), B,
                         _p(y), _p(a))
    return y, a


def quantize_q8(x):
    """x: [R][K] float32 or bf16 bits -> (x_q int8 [R][K], s float32 [R][K/32])."""
    x = np.ascontiguousarray(x)
    R, K = x.shape
    xq = np.empty((R, K), np.int8)
    s = np.empty((R, K // 32), np.float32)
    lib().orc_quantize_q8(_p(x), _xkind(x), R, K, _p(xq), _p(s))
    return xq, s


def group_int(fmt, row: np.ndarray, xq_row: np.ndarray, g: int) -> int:
    _q8_only(fmt)
    return lib().orc_group_int(fmt, _p(np.ascontiguousarray(row)),
                               _p(np.ascontiguousarray(xq_row)), g)


def gemv_q8(fmt, W, xq, s, N, K):
    _q8_only(fmt)
    xq = np.ascontiguousarray(xq)
    s = np.ascontiguousarray(s, dtype=np.float32)
    B = xq.shape[0]
    y = np.empty((B, N), np.float64)
    a = np.empty((B, N), np.float64)
    lib().orc_gemv_q8(fmt, _p(np.ascontiguousarray(W)), N, K, _p(xq), _p(s), B, _p(y), _p(a))
    return y, a


def gemm_q8_pairs(fmt, W, K, xq, s, ms, ns):
    _q8_only(fmt)
    ms = np.ascontiguousarray(ms, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    y = np.empty(len(ms), np.float64)
    a = np.empty(len(ms), np.float64)
    lib().orc_gemm_q8_pairs(fmt, _p(np.ascontiguousarray(W)), K, _p(np.ascontiguousarray(xq)),
                            _p(np.ascontiguousarray(s, dtype=np.float32)), _p(ms), _p(ns),
                            len(ms), _p(y), _p(a))
    return y, a


def gemv_float_pairs(fmt, W, K, x, bs, ns):
    x = np.ascontiguousarray(x)
    bs = np.ascontiguousarray(bs, dtype=np.int64)
    ns = np.ascontiguousarray(ns, dtype=np.int64)
    y = np.empty(len(bs), np.float64)
    a = np.empty(len(bs), np.float64)
    lib().orc_gemv_float_pairs(fmt, _p(np.ascontiguousarray(W)), K, _p(x), _xkind(x), _p(bs),
                               _p(ns), len(bs), _p(y), _p(a))
    return y, a


def plane_q6k(W, N, K):
    plane = np.empty((N, K), np.int8)
    lib().orc_plane_q6k(_p(np.ascontiguousarray(W)), N, K, _p(plane))
    return plane


def route_topk_softmax(logits: np.ndarray, k: int):
    logits = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = logits.shape
    idx = np.empty((T, k), np.int32)
    gate = np.empty((T, k), np.float64)
    lib().orc_route_topk_softmax(_p(logits), T, E, k, _p(idx), _p(gate))
    return idx, gate


def moe_float(fmt, H, I, wg, wu, wd, idx, gate, x, want_h=False):
    """wg/wu/wd: lists (one per expert) of packed matrices; x [T][H]."""
    x = np.ascontiguousarray(x)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    gate = np.ascontiguousarray(gate, dtype=np.float64)
    T, k = idx.shape
    keep = [np.ascontiguousarray(m) for m in list(wg) + list(wu) + list(wd)]
    E = len(wg)
    arr = (C.c_void_p * E)
    pg = arr(*[m.ctypes.data for m in keep[:E]])
    pu = arr(*[m.ctypes.data for m in keep[E:2 * E]])
    pd = arr(*[m.ctypes.data for m in keep[2 * E:]])
    y = np.empty((T, H), np.float64)
    bound = np.empty((T, H), np.float64)
    h = np.empty((T, k, I), np.float64) if want_h else None
    lib().orc_moe_float(fmt, H, I, C.cast(pg, C.c_void_p), C.cast(pu, C.c_void_p),
                        C.cast(pd, C.c_void_p), T, k, _p(idx), _p(gate), _p(x), _xkind(x),
                        _p(y), _p(bound), _p(h) if want_h else None)
    return (y, bound, h) if want_h else (y, bound)


def moe_q8(fmt, H, I, wg, wu, wd, idx, gate, x):
    """The expert FFN with quantized activations (the prefill GEMM's
    arithmetic): returns (y [T][H], tight bound, loose bound)."""
    _q8_only(fmt)
    x = np.ascontiguousarray(x)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    gate = np.ascontiguousarray(gate, dtype=np.float64)
    T, k = idx.shape
    keep = [np.ascontiguousarray(m) for m in list(wg) + list(wu) + list(wd)]
    E = len(wg)
    arr = (C.c_void_p * E)
    pg = arr(*[m.ctypes.data for m in keep[:E]])
    pu = arr(*[m.ctypes.data for m in keep[E:2 * E]])
    pd = arr(*[m.ctypes.data for m in keep[2 * E:]])
    y = np.empty((T, H), np.float64)
    tight = np.empty((T, H), np.float64)
    loose = np.empty((T, H), np.float64)
    lib().orc_moe_q8(fmt, H, I, C.cast(pg, C.c_void_p), C.cast(pu, C.c_void_p), C.cast(pd, C.c_void_p),
                     T, k, _p(idx), _p(gate), _p(x), _xkind(x), _p(y), _p(tight), _p(loose))
    return y, tight, loose


def cbk_dequant(M, codes, books, scales, N, K):
    """Dense [N][K] weights of an additive-codebook matrix (codes [N][K/8][M]
    uint8, books [M][256][8] fp16 bits, scales [N] fp16 bits)."""
    c, bk, sc = (np.ascontiguousarray(codes, np.uint8), np.ascontiguousarray(books, np.uint16),
                 np.ascontiguousarray(scales, np.uint16))
    return np.array([[lib().orc_cbk_weight(M, _p(c), _p(bk), _p(sc), K, n, k) for k in range(K)]
                     for n in range(N)])


def cbk_gemv(M, codes, books, scales, x, N, K):
    """x: [B][K] float32 or bf16 bits -> (y [B][N] float64, tolerance scale)."""
    x = np.ascontiguousarray(x)
    B = x.shape[0]
    y = np.empty((B, N), np.float64)
    a = np.empty((B, N), np.float64)
    lib().orc_cbk_gemv(M, _p(np.ascontiguousarray(codes, np.uint8)), _p(np.ascontiguousarray(books, np.uint16)),
                       _p(np.ascontiguousarray(scales, np.uint16)), N, K, _p(x), _xkind(x), B, _p(y), _p(a))
    return y, a
