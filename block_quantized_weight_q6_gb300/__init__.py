"""GB300-native matrix multiplication against block-quantized LLM weights.

Python binding of libqmm (include/qmm.h). Every function here only marshals
arguments (torch tensors -> device pointers, the current stream, a cached
workspace) and calls the C interface; all arithmetic runs in the library's
sm_103a kernels. There is no CPU or PyTorch fallback: if libqmm.so is not
built, importing this package raises.
"""
from __future__ import annotations

import ctypes as C
import os

from .build import LIB as _LIB_PATH

Q4_0, Q8_0, Q6_K, Q4_K, Q2_K = 0x01, 0x02, 0x03, 0x04, 0x05
X_F32, X_BF16 = 0x000, 0x100
ACT_FLOAT, ACT_Q8 = 0x0000, 0x1000

OK, EINVAL, EUNSUPPORTED, EALIGN, ECUDA, EPLANE, EDEVICE_TIMEOUT, ENOWORKSPACE = (
    0, -1, -2, -3, -4, -5, -6, -7)

LIVE = {
    "gemv_float": 0, "gemv_q8": 1, "gemv_splitk_reduce": 2, "quantize": 3, "plane_build": 4,
    "gemm_exp_plane": 5, "gemm_in_kernel": 6, "gemm_exp_off": 7, "gemm_fallback": 8,
    "gemm_q4_0": 9, "route": 10, "moe_gate_up": 11, "moe_down": 12, "moe_combine": 13,
    "x_tile": 14, "moe_plan": 15, "moe_gather": 16, "gemv_mv1": 17, "gemv_mv8": 18, "moe_silu": 19,
    "gemm_split_reduce": 20, "moe_prefill_plan": 21, "moe_prefill_rows": 22, "moe_prefill_silu": 23,
    "cbk_gemv": 24,
}
LIVE_COUNT = 32

BLOCK_ELEMS = {Q4_0: 32, Q8_0: 32, Q6_K: 256, Q4_K: 256, Q2_K: 256}
BLOCK_BYTES = {Q4_0: 18, Q8_0: 34, Q6_K: 210, Q4_K: 144, Q2_K: 84}


class QmmError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"qmm error {code}: {msg}")
        self.code = code


class MoeExperts(C.Structure):
    _fields_ = [("n_experts", C.c_int), ("hidden", C.c_int), ("inter", C.c_int),
                ("top_k", C.c_int), ("n_tokens", C.c_int),
                ("w_gate", C.POINTER(C.c_void_p)), ("w_up", C.POINTER(C.c_void_p)),
                ("w_down", C.POINTER(C.c_void_p))]


def _load():
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"{_LIB_PATH} is not built; run block_quantized_weight_q6_gb300.build.build()")
    L = C.CDLL(_LIB_PATH)
    P, I, I64, U32, SZ = C.c_void_p, C.c_int, C.c_int64, C.c_uint32, C.c_size_t
    sig = {
        "qmm_init": (I, []),
        "qmm_set_stream": (I, [P]),
        "qmm_set_workspace": (I, [P, SZ]),
        "qmm_workspace_bytes": (SZ, [U32, I64, I64, I64]),
        "qmm_gemv": (I, [U32, P, P, P, I64, I64, I]),
        "qmm_quantize_q8": (I, [U32, P, I64, I64, P, P]),
        "qmm_gemv_noalloc": (I, [U32, P, P, P, I64, I64, I]),
        "qmm_gemv_group": (I, [U32, I, C.POINTER(C.c_void_p), C.POINTER(C.c_void_p),
                               C.POINTER(C.c_void_p), C.POINTER(C.c_int64), C.POINTER(C.c_int64), I]),
        "qmm_gemv_group_workspace_bytes": (SZ, [U32, I, C.POINTER(C.c_int64), C.POINTER(C.c_int64), I]),
        "qmm_gemv_multi": (I, [I, C.POINTER(C.c_uint32), C.POINTER(C.c_void_p), C.POINTER(C.c_void_p),
                               C.POINTER(C.c_void_p), C.POINTER(C.c_int64), C.POINTER(C.c_int64), I]),
        "qmm_gemv_multi_workspace_bytes": (SZ, [I, C.POINTER(C.c_uint32), C.POINTER(C.c_int64),
                                                C.POINTER(C.c_int64), I]),
        "qmm_gemm": (I, [U32, P, P, P, I64, I64, I64, P]),
        "qmm_plane_bytes": (SZ, [I64, I64]),
        "qmm_plane_wanted": (I, [I64, I64]),
        "qmm_plane_build": (I, [P, I64, I64, P]),
        "qmm_plane_release": (I, [P]),
        "moe_gemv": (I, [U32, C.POINTER(MoeExperts), P, P, P, P]),
        "qmm_moe_workspace_bytes": (SZ, [C.POINTER(MoeExperts)]),
        "moe_prefill": (I, [U32, C.POINTER(MoeExperts), P, P, P, P]),
        "qmm_cbk_gemv": (I, [I, P, P, P, U32, P, P, I64, I64, I]),
        "qmm_cbk_workspace_bytes": (SZ, [I, I64, I64, I]),
        "qmm_moe_prefill_workspace_bytes": (SZ, [U32, C.POINTER(MoeExperts)]),
        "qmm_route_topk_softmax": (I, [P, I, I, I, P, P]),
        "qmm_liveness_read": (I, [C.POINTER(C.c_int64), I]),
        "qmm_liveness_reset": (I, []),
        "qmm_sync_check": (I, []),
        "qmm_wait_probe": (I, [U32]),
        "qmm_last_error": (C.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    return L


class _Lib:
    """libqmm, loaded on first use (raises if the library is not built)."""
    _handle = None

    def __getattr__(self, name):
        if _Lib._handle is None:
            _Lib._handle = _load()
        return getattr(_Lib._handle, name)


lib = _Lib()


def _check(rc: int):
    if rc != OK:
        raise QmmError(rc, lib.qmm_last_error().decode())


# ---------------------------------------------------------------- marshalling

_ws = {}
_ws_outgrown = []


def _torch():
    import torch
    return torch


def _prepare(device, nbytes: int):
    """Point the library at torch's current stream and a workspace of at least
    nbytes on `device` (cached per device, grown on demand). A workspace that
    is outgrown stays allocated: CUDA graphs captured earlier still hold its
    address."""
    torch = _torch()
    stream = torch.cuda.current_stream(device)
    _check(lib.qmm_set_stream(C.c_void_p(stream.cuda_stream)))
    key = device.index if device.index is not None else torch.cuda.current_device()
    buf = _ws.get(key)
    if nbytes and (buf is None or buf.numel() < nbytes):
        if buf is not None:
            _ws_outgrown.append(buf)
        buf = torch.empty(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
        _ws[key] = buf
    if buf is not None:
        _check(lib.qmm_set_workspace(C.c_void_p(buf.data_ptr()), buf.numel()))
    else:
        _check(lib.qmm_set_workspace(None, 0))


def _ptr(t):
    return C.c_void_p(t.data_ptr()) if t is not None else None


def _act_bits(x) -> int:
    torch = _torch()
    if x.dtype == torch.float32:
        return X_F32
    if x.dtype == torch.bfloat16:
        return X_BF16
    raise TypeError(f"activations must be float32 or bfloat16, got {x.dtype}")


def gemv(fmt: int, W, x, y, N: int, K: int, act: int = ACT_FLOAT):
    """y[B][N] = W (N x K, packed `fmt` blocks) times x[B][K] per batch row."""
    B = x.shape[0]
    code = fmt | _act_bits(x) | act
    _prepare(x.device, lib.qmm_workspace_bytes(code, B, N, K))
    with _torch().cuda.device(x.device):
        _check(lib.qmm_gemv(code, _ptr(W), _ptr(x), _ptr(y), N, K, B))


class GemvGroup:
    """A fixed set of matvecs of one format and batch for gemv_group: the
    host arrays of the call, built once (keep the object while it is used)."""

    def __init__(self, fmt: int, Ws, xs, ys, Ns, Ks, act: int = ACT_FLOAT):
        n = len(Ws)
        if not (len(xs) == len(ys) == len(Ns) == len(Ks) == n):
            raise ValueError("Ws, xs, ys, Ns, Ks must have the same length")
        B = xs[0].shape[0]
        self.n, self.B, self.device = n, B, xs[0].device
        self.code = fmt | _act_bits(xs[0]) | act
        P = C.c_void_p * n
        L = C.c_int64 * n
        self._W = P(*[t.data_ptr() for t in Ws])
        self._x = P(*[t.data_ptr() for t in xs])
        self._y = P(*[t.data_ptr() for t in ys])
        self._N = L(*Ns)
        self._K = L(*Ks)
        self._keep = (list(Ws), list(xs), list(ys))
        self.ws = lib.qmm_gemv_group_workspace_bytes(self.code, n, self._N, self._K, B)


def gemv_group(group: GemvGroup):
    """y[i] = W[i] x[i] for every matvec of the group, in one launch."""
    _prepare(group.device, group.ws)
    with _torch().cuda.device(group.device):
        _check(lib.qmm_gemv_group(group.code, group.n, group._W, group._x, group._y, group._N,
                                  group._K, group.B))


class GemvMulti:
    """A fixed set of matvecs of possibly different weight formats (the same
    activation type, mode and batch) for gemv_multi: the host arrays of the
    call, built once (keep the object while it is used)."""

    def __init__(self, fmts, Ws, xs, ys, Ns, Ks, act: int = ACT_FLOAT):
        n = len(Ws)
        if not (len(fmts) == len(xs) == len(ys) == len(Ns) == len(Ks) == n):
            raise ValueError("fmts, Ws, xs, ys, Ns, Ks must have the same length")
        B = xs[0].shape[0]
        self.n, self.B, self.device = n, B, xs[0].device
        self._fmt = (C.c_uint32 * n)(*[f | _act_bits(x) | act for f, x in zip(fmts, xs)])
        P = C.c_void_p * n
        L = C.c_int64 * n
        self._W = P(*[t.data_ptr() for t in Ws])
        self._x = P(*[t.data_ptr() for t in xs])
        self._y = P(*[t.data_ptr() for t in ys])
        self._N = L(*Ns)
        self._K = L(*Ks)
        self._keep = (list(Ws), list(xs), list(ys))
        self.ws = lib.qmm_gemv_multi_workspace_bytes(n, self._fmt, self._N, self._K, B)


def gemv_multi(multi: GemvMulti):
    """y[i] = W[i] x[i] for every matvec of the set (formats may differ)."""
    _prepare(multi.device, multi.ws)
    with _torch().cuda.device(multi.device):
        _check(lib.qmm_gemv_multi(multi.n, multi._fmt, multi._W, multi._x, multi._y, multi._N,
                                  multi._K, multi.B))


def quantize_q8(x, xq, s):
    """xq[rows][K] int8, s[rows][K/32] fp32 = per-32 quantization of x."""
    rows, K = x.shape
    _prepare(x.device, 0)
    with _torch().cuda.device(x.device):
        _check(lib.qmm_quantize_q8(_act_bits(x), _ptr(x), rows, K, _ptr(xq), _ptr(s)))


def gemv_workspace_bytes(fmt: int, B: int, N: int, K: int, x_bits: int = X_F32,
                         act: int = ACT_FLOAT) -> int:
    return lib.qmm_workspace_bytes(fmt | x_bits | act, B, N, K)


def gemm(fmt: int, W, X, Y, M: int, N: int, K: int, plane=None):
    """Y[M][N] = quantized-activation GEMM of X[M][K] (bf16 or fp32) with W."""
    code = fmt | _act_bits(X) | ACT_Q8
    _prepare(X.device, lib.qmm_workspace_bytes(code, M, N, K))
    with _torch().cuda.device(X.device):
        _check(lib.qmm_gemm(code, _ptr(W), _ptr(X), _ptr(Y), M, N, K, _ptr(plane)))


def plane_bytes(N: int, K: int) -> int:
    return lib.qmm_plane_bytes(N, K)


def plane_wanted(N: int, K: int) -> bool:
    return bool(lib.qmm_plane_wanted(N, K))


def plane_build(W, N: int, K: int, plane=None):
    """Builds W's centered-int8 plane into `plane` (allocated with torch when
    None) and registers it. Returns the plane tensor."""
    torch = _torch()
    if plane is None:
        plane = torch.empty((N, K), dtype=torch.int8, device=W.device)
    _prepare(W.device, 0)
    with torch.cuda.device(W.device):
        _check(lib.qmm_plane_build(_ptr(W), N, K, _ptr(plane)))
    return plane


def plane_register_failed(W, N: int, K: int):
    """Records that W's plane was wanted but could not be allocated."""
    _check(lib.qmm_plane_build(_ptr(W), N, K, None))


def plane_release(W):
    _check(lib.qmm_plane_release(_ptr(W)))


def route_topk_softmax(logits, k: int, idx, gate_w):
    T, E = logits.shape
    _prepare(logits.device, 0)
    with _torch().cuda.device(logits.device):
        _check(lib.qmm_route_topk_softmax(_ptr(logits), T, E, k, _ptr(idx), _ptr(gate_w)))


def moe_experts(w_gate, w_up, w_down, hidden: int, inter: int, top_k: int, n_tokens: int):
    """Host-side expert table (keeps the pointer arrays, and the tensors they
    point into, alive on the object)."""
    E = len(w_gate)
    arr = C.c_void_p * E
    m = MoeExperts()
    m._keep = (arr(*[t.data_ptr() for t in w_gate]), arr(*[t.data_ptr() for t in w_up]),
               arr(*[t.data_ptr() for t in w_down]))
    m._tensors = (list(w_gate), list(w_up), list(w_down))  # the device memory the pointers name
    m.n_experts, m.hidden, m.inter, m.top_k, m.n_tokens = E, hidden, inter, top_k, n_tokens
    m.w_gate = C.cast(m._keep[0], C.POINTER(C.c_void_p))
    m.w_up = C.cast(m._keep[1], C.POINTER(C.c_void_p))
    m.w_down = C.cast(m._keep[2], C.POINTER(C.c_void_p))
    return m


def moe(fmt: int, experts: MoeExperts, idx, gate_w, x, y):
    code = fmt | _act_bits(x) | ACT_FLOAT
    _prepare(x.device, lib.qmm_moe_workspace_bytes(C.byref(experts)))
    with _torch().cuda.device(x.device):
        _check(lib.moe_gemv(code, C.byref(experts), _ptr(idx), _ptr(gate_w), _ptr(x), _ptr(y)))


def liveness() -> dict:
    buf = (C.c_int64 * LIVE_COUNT)()
    _check(lib.qmm_liveness_read(buf, LIVE_COUNT))
    return {name: int(buf[i]) for name, i in LIVE.items()}


def liveness_reset():
    _torch().cuda.synchronize()
    _check(lib.qmm_set_stream(None))
    _check(lib.qmm_liveness_reset())
    _torch().cuda.synchronize()


def sync_check():
    _check(lib.qmm_sync_check())


def wait_probe(limit_us: int, device=None):
    """Launches the bounded-wait probe (a wait that must give up after
    limit_us microseconds) on torch's current stream."""
    torch = _torch()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else device
    _prepare(dev, 0)
    with torch.cuda.device(dev):
        _check(lib.qmm_wait_probe(limit_us))


def moe_prefill(fmt: int, experts: MoeExperts, idx, gate_w, x, y):
    """The routed expert FFN of `moe` for many tokens, grouped by expert
    through the prefill GEMM (quantized activations); not graph-capturable.
    Experts whose matrices lie at one stride per projection (e.g. the rows
    of one [E, bytes] tensor each) run one grouped GEMM launch per
    projection; any other table runs one per expert."""
    code = fmt | _act_bits(x)
    _prepare(x.device, lib.qmm_moe_prefill_workspace_bytes(code, C.byref(experts)))
    with _torch().cuda.device(x.device):
        _check(lib.moe_prefill(code, C.byref(experts), _ptr(idx), _ptr(gate_w), _ptr(x), _ptr(y)))


def cbk_gemv(n_books: int, codes, books, scales, x, y, N: int, K: int):
    """y[B][N] = the additive-codebook matrix (codes uint8 [N][K/8][n_books],
    books fp16 bits [n_books][256][8], scales fp16 bits [N]) times x[B][K]."""
    B = x.shape[0]
    xt = _act_bits(x)
    _prepare(x.device, lib.qmm_cbk_workspace_bytes(n_books, N, K, B))
    with _torch().cuda.device(x.device):
        _check(lib.qmm_cbk_gemv(n_books, _ptr(codes), _ptr(books), _ptr(scales), xt, _ptr(x), _ptr(y), N, K, B))
