"""ctypes binding of libboost_block.so (argument marshalling only).

Every function here checks the torch tensors it is given (dtype, device,
contiguity, shape), passes raw pointers and sizes to the C ABI declared in
``include/boost_block.h`` and raises ``BoostError`` on a non-OK status. No
arithmetic of the block happens in Python; there is no CPU fallback: if the
library is missing, ``lib()`` raises.
"""

from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

_LIB = None

BOOST_OK = 0
STATUS_NAMES = {
    0: "BOOST_OK", 1: "BOOST_ERR_INVALID_ARG", 2: "BOOST_ERR_UNSUPPORTED_SHAPE",
    3: "BOOST_ERR_ALIGNMENT", 4: "BOOST_ERR_WORKSPACE", 5: "BOOST_ERR_CUDA",
    6: "BOOST_ERR_TIMEOUT", 7: "BOOST_ERR_DEVICE_CHECK",
}
ACT = {"identity": 0, "silu": 1}

EXPORTS = (
    "boost_block_workspace_bytes", "boost_block_ws_init", "boost_block_fwd", "boost_block_bwd",
    "boost_rmsnorm_stats", "boost_block_layout", "boost_block_check", "boost_status_string",
    "boost_swiglu_fwd", "boost_swiglu_bwd", "boost_add", "boost_debug_wait_timeout",
    "boost_block_ws_layout", "boost_profile_enable", "boost_profile_kernel_count",
    "boost_profile_read", "boost_rmsnorm_rstd_noalloc", "boost_block_bwd_swiglu",
    "boost_profile_read_kernels", "boost_block_fwd_swiglu", "boost_block_fwd_btp",
    "boost_block_up", "boost_debug_count_writes", "boost_debug_count_log",
    "boost_profile_only", "boost_block_fwd_residual", "boost_block_bwd_residual",
)


class BoostError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        name = STATUS_NAMES.get(status, str(status))
        msg = lib().boost_status_string(status).decode() if _LIB is not None else name
        super().__init__(f"{what}: {name} ({msg})")


class Desc(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("d", ctypes.c_int64), ("r", ctypes.c_int64),
                ("k", ctypes.c_int64), ("n", ctypes.c_int64), ("S", ctypes.c_int32),
                ("eps", ctypes.c_float), ("act", ctypes.c_int32), ("has_norm", ctypes.c_int32)]


def lib_path() -> str:
    return _build.LIB


def lib():
    """Load the library once; raise if it has not been built."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "`python -m rank_bottleneck_online_gb300.build`")
    L = ctypes.CDLL(path)
    vp, sz, i64, u32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int64, ctypes.c_uint32
    dp = ctypes.POINTER(Desc)
    L.boost_block_workspace_bytes.argtypes = [dp]
    L.boost_block_workspace_bytes.restype = sz
    L.boost_block_ws_init.argtypes = [vp, sz, vp]
    L.boost_block_fwd.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.boost_block_fwd_swiglu.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.boost_block_fwd_btp.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.boost_block_up.argtypes = [dp, vp, vp, vp, vp, vp, sz, vp]
    L.boost_debug_count_writes.argtypes = [vp, i64]
    L.boost_debug_count_log.argtypes = [ctypes.POINTER(i64), i64]
    L.boost_debug_count_log.restype = i64
    L.boost_block_bwd.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.boost_block_fwd_residual.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.boost_block_bwd_residual.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                           sz, vp]
    L.boost_rmsnorm_stats.argtypes = [dp, vp, vp, vp, vp]
    L.boost_block_layout.argtypes = [dp, ctypes.POINTER(i64), ctypes.POINTER(i64),
                                     ctypes.POINTER(i64)]
    L.boost_block_check.argtypes = [vp, vp]
    L.boost_status_string.argtypes = [ctypes.c_int]
    L.boost_status_string.restype = ctypes.c_char_p
    L.boost_swiglu_fwd.argtypes = [i64, i64, vp, vp, vp, vp]
    L.boost_swiglu_bwd.argtypes = [i64, i64, vp, vp, vp, vp, vp, vp]
    L.boost_add.argtypes = [i64, vp, vp, vp, vp]
    L.boost_debug_wait_timeout.argtypes = [vp, sz, u32, vp]
    szp = ctypes.POINTER(sz)
    L.boost_block_ws_layout.argtypes = [dp, szp, szp, szp, szp]
    L.boost_rmsnorm_rstd_noalloc.argtypes = [dp, vp, vp, vp]
    L.boost_block_bwd_swiglu.argtypes = [dp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    L.boost_profile_enable.argtypes = [ctypes.c_int]
    L.boost_profile_only.argtypes = [ctypes.c_int]
    L.boost_profile_kernel_count.argtypes = []
    dbl = ctypes.POINTER(ctypes.c_double)
    L.boost_profile_read.argtypes = [ctypes.c_int, ctypes.POINTER(ctypes.c_char_p),
                                     ctypes.POINTER(i64), dbl, dbl, dbl]
    L.boost_profile_read_kernels.argtypes = [ctypes.c_int, ctypes.POINTER(i64)]
    for name in EXPORTS:
        if name not in ("boost_block_workspace_bytes", "boost_status_string",
                        "boost_debug_count_log"):
            getattr(L, name).restype = ctypes.c_int
    _LIB = L
    return L


def _check(status: int, what: str):
    if status != BOOST_OK:
        raise BoostError(status, what)


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, name, dtype, shape=None):
    if t is None:
        raise ValueError(f"{name} is required")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t


def make_desc(T, d, r, k, n, *, S=1, eps=1e-5, act="silu", has_norm=True) -> Desc:
    return Desc(int(T), int(d), int(r), int(k), int(n), int(S), float(eps),
                ACT[act] if isinstance(act, str) else int(act), 1 if has_norm else 0)


def workspace_bytes(desc: Desc) -> int:
    return int(lib().boost_block_workspace_bytes(ctypes.byref(desc)))


class Workspace:
    """Caller-owned device workspace (torch memory), error word cleared on creation."""

    def __init__(self, nbytes: int, device=None, stream=None):
        self.nbytes = max(int(nbytes), 256)
        self.buf = torch.empty(self.nbytes, dtype=torch.uint8,
                               device=device or torch.device("cuda"))
        _check(lib().boost_block_ws_init(_ptr(self.buf), self.nbytes, _stream(stream)),
               "boost_block_ws_init")

    @property
    def ptr(self):
        return _ptr(self.buf)

    def ensure(self, nbytes: int):
        if nbytes > self.nbytes:
            self.__init__(nbytes, self.buf.device)
        return self


def layout(desc: Desc):
    """Shard offsets [S+1], group column offsets [k+1], exchange element count (host)."""
    S = desc.S if desc.has_norm else 1
    so = (ctypes.c_int64 * (S + 1))()
    go = (ctypes.c_int64 * (desc.k + 1))()
    ex = ctypes.c_int64(0)
    _check(lib().boost_block_layout(ctypes.byref(desc), so, go, ctypes.byref(ex)),
           "boost_block_layout")
    return list(so), list(go), ex.value


def ws_layout(desc: Desc):
    """Byte offsets of a, dzs, A' and rstd inside a workspace for ``desc``."""
    o = [ctypes.c_size_t(0) for _ in range(4)]
    _check(lib().boost_block_ws_layout(ctypes.byref(desc), *(ctypes.byref(v) for v in o)),
           "boost_block_ws_layout")
    return {"a": o[0].value, "dzs": o[1].value, "Ap": o[2].value, "rstd": o[3].value}


def ws_view(ws: "Workspace", offset: int, shape, dtype):
    """A torch view of workspace bytes (for tests and inspection)."""
    n = 1
    for s in shape:
        n *= s
    nbytes = n * torch.tensor([], dtype=dtype).element_size()
    return ws.buf[offset:offset + nbytes].view(dtype).view(*shape)


def rmsnorm_stats(desc: Desc, x, ssq=None, rstd=None, stream=None):
    _need(x, "x", torch.bfloat16, (desc.T, desc.d))
    if ssq is None:
        ssq = torch.empty(desc.S, desc.T, dtype=torch.float32, device=x.device)
    if rstd is None:
        rstd = torch.empty(desc.T, dtype=torch.float32, device=x.device)
    _check(lib().boost_rmsnorm_stats(ctypes.byref(desc), _ptr(x), _ptr(ssq), _ptr(rstd),
                                     _stream(stream)), "boost_rmsnorm_stats")
    return ssq, rstd


def rmsnorm_rstd_noalloc(desc: Desc, x, rstd=None, stream=None):
    """Row scales through the allocation-free entry point (for callers that cannot
    allocate device memory; the partials use the library's fixed device array)."""
    _need(x, "x", torch.bfloat16, (desc.T, desc.d))
    if rstd is None:
        rstd = torch.empty(desc.T, dtype=torch.float32, device=x.device)
    _need(rstd, "rstd", torch.float32, (desc.T,))
    _check(lib().boost_rmsnorm_rstd_noalloc(ctypes.byref(desc), _ptr(x), _ptr(rstd),
                                            _stream(stream)), "boost_rmsnorm_rstd_noalloc")
    return rstd


def block_fwd(desc: Desc, x, gamma, A, B, ws: Workspace, *, y=None, rstd=None, stream=None,
              residual=None):
    """y [k,T,n] (and the row scale into ``rstd`` if given). With ``residual`` [T,n]
    (k == 1): y = residual + block(x), added in the up-projection's epilogue."""
    bf = torch.bfloat16
    _need(x, "x", bf, (desc.T, desc.d))
    _need(A, "A", bf, (desc.d, desc.k * desc.r))
    _need(B, "B", bf, (desc.k, desc.r, desc.n))
    if desc.has_norm:
        _need(gamma, "gamma", bf, (desc.d,))
    if y is None:
        y = torch.empty(desc.k, desc.T, desc.n, dtype=bf, device=x.device)
    _need(y, "y", bf, (desc.k, desc.T, desc.n))
    if rstd is not None:
        _need(rstd, "rstd", torch.float32, (desc.T,))
    if residual is not None:
        _need(residual, "residual", bf, (desc.T, desc.n))
        _check(lib().boost_block_fwd_residual(ctypes.byref(desc), _ptr(x), _ptr(gamma), _ptr(A),
                                              _ptr(B), _ptr(residual), _ptr(y), _ptr(rstd),
                                              ws.ptr, ws.nbytes, _stream(stream)),
               "boost_block_fwd_residual")
        return y
    _check(lib().boost_block_fwd(ctypes.byref(desc), _ptr(x), _ptr(gamma), _ptr(A), _ptr(B),
                                 _ptr(y), _ptr(rstd), ws.ptr, ws.nbytes, _stream(stream)),
           "boost_block_fwd")
    return y


def block_fwd_swiglu(desc: Desc, x, gamma, A, B, ws: Workspace, *, y=None, h=None, rstd=None,
                     stream=None):
    """Gate/up block (k == 2) forward with the SwiGLU forward fused in: returns
    (y [2,T,n] = gate, up; h [T,n] = silu(gate) * up)."""
    bf = torch.bfloat16
    if desc.k != 2:
        raise ValueError("block_fwd_swiglu needs k == 2 (gate and up groups)")
    _need(x, "x", bf, (desc.T, desc.d))
    _need(A, "A", bf, (desc.d, desc.k * desc.r))
    _need(B, "B", bf, (desc.k, desc.r, desc.n))
    if desc.has_norm:
        _need(gamma, "gamma", bf, (desc.d,))
    if y is None:
        y = torch.empty(desc.k, desc.T, desc.n, dtype=bf, device=x.device)
    if h is None:
        h = torch.empty(desc.T, desc.n, dtype=bf, device=x.device)
    _need(y, "y", bf, (desc.k, desc.T, desc.n))
    _need(h, "h", bf, (desc.T, desc.n))
    if rstd is not None:
        _need(rstd, "rstd", torch.float32, (desc.T,))
    _check(lib().boost_block_fwd_swiglu(ctypes.byref(desc), _ptr(x), _ptr(gamma), _ptr(A),
                                        _ptr(B), _ptr(y), _ptr(h), _ptr(rstd), ws.ptr, ws.nbytes,
                                        _stream(stream)),
           "boost_block_fwd_swiglu")
    return y, h


def block_up(desc: Desc, a, B, ws: Workspace, *, y=None, h=None, stream=None):
    """The up-projection alone from a given bottleneck activation a [T, k*r]; with h
    (k == 2) also h = silu(y[0]) * y[1]. Returns y (and h)."""
    bf = torch.bfloat16
    _need(a, "a", bf, (desc.T, desc.k * desc.r))
    _need(B, "B", bf, (desc.k, desc.r, desc.n))
    if y is None:
        y = torch.empty(desc.k, desc.T, desc.n, dtype=bf, device=a.device)
    _need(y, "y", bf, (desc.k, desc.T, desc.n))
    if h is not None:
        _need(h, "h", bf, (desc.T, desc.n))
    _check(lib().boost_block_up(ctypes.byref(desc), _ptr(a), _ptr(B), _ptr(y), _ptr(h), ws.ptr,
                                ws.nbytes, _stream(stream)), "boost_block_up")
    return y if h is None else (y, h)


def btp_payload_elems(desc: Desc) -> int:
    """fp32 values of the emulated exchange payload: S*T*k*r partial products, then
    (normed blocks) S*T sums of squares."""
    return desc.S * desc.T * (desc.k * desc.r + (1 if desc.has_norm else 0))


def block_fwd_btp(desc: Desc, x, gamma, A, B, ws: Workspace, *, y=None, rstd=None,
                  payload=None, stream=None):
    """Forward with the down-projection as the emulated bottleneck-aware TP exchange.
    Returns (y [k,T,n], zpart [S,T,k*r], ssq [S,T] or None), the last two views of the
    payload buffer."""
    bf = torch.bfloat16
    _need(x, "x", bf, (desc.T, desc.d))
    _need(A, "A", bf, (desc.d, desc.k * desc.r))
    _need(B, "B", bf, (desc.k, desc.r, desc.n))
    if desc.has_norm:
        _need(gamma, "gamma", bf, (desc.d,))
    if y is None:
        y = torch.empty(desc.k, desc.T, desc.n, dtype=bf, device=x.device)
    _need(y, "y", bf, (desc.k, desc.T, desc.n))
    n_pay = btp_payload_elems(desc)
    if payload is None:
        payload = torch.empty(n_pay, dtype=torch.float32, device=x.device)
    _need(payload, "payload", torch.float32, (n_pay,))
    if rstd is not None:
        _need(rstd, "rstd", torch.float32, (desc.T,))
    _check(lib().boost_block_fwd_btp(ctypes.byref(desc), _ptr(x), _ptr(gamma), _ptr(A), _ptr(B),
                                     _ptr(y), _ptr(rstd), _ptr(payload), ws.ptr, ws.nbytes,
                                     _stream(stream)),
           "boost_block_fwd_btp")
    S, T, kr = desc.S, desc.T, desc.k * desc.r
    zpart = payload[:S * T * kr].view(S, T, kr)
    ssq = payload[S * T * kr:].view(S, T) if desc.has_norm else None
    return y, zpart, ssq


def block_bwd(desc: Desc, x, gamma, A, B, dy, ws: Workspace, *, rstd=None, dx=None,
              dgamma=None, dA=None, dB=None, stream=None, dx_residual=None):
    """Returns (dx, dgamma or None, dA, dB). With ``dx_residual`` [T,d]: dx =
    dx_residual + the block's input gradient, added in the dx epilogue."""
    bf = torch.bfloat16
    _need(x, "x", bf, (desc.T, desc.d))
    _need(A, "A", bf, (desc.d, desc.k * desc.r))
    _need(B, "B", bf, (desc.k, desc.r, desc.n))
    _need(dy, "dy", bf, (desc.k, desc.T, desc.n))
    dev = x.device
    if dx is None:
        dx = torch.empty(desc.T, desc.d, dtype=bf, device=dev)
    if dA is None:
        dA = torch.empty(desc.d, desc.k * desc.r, dtype=bf, device=dev)
    if dB is None:
        dB = torch.empty(desc.k, desc.r, desc.n, dtype=bf, device=dev)
    if desc.has_norm:
        _need(gamma, "gamma", bf, (desc.d,))
        if dgamma is None:
            dgamma = torch.empty(desc.d, dtype=bf, device=dev)
    if rstd is not None:
        _need(rstd, "rstd", torch.float32, (desc.T,))
    if dx_residual is not None:
        _need(dx_residual, "dx_residual", bf, (desc.T, desc.d))
        _check(lib().boost_block_bwd_residual(ctypes.byref(desc), _ptr(x), _ptr(gamma), _ptr(A),
                                              _ptr(B), _ptr(rstd), _ptr(dy), _ptr(dx_residual),
                                              _ptr(dx), _ptr(dgamma), _ptr(dA), _ptr(dB),
                                              ws.ptr, ws.nbytes, _stream(stream)),
               "boost_block_bwd_residual")
        return dx, dgamma, dA, dB
    _check(lib().boost_block_bwd(ctypes.byref(desc), _ptr(x), _ptr(gamma), _ptr(A), _ptr(B),
                                 _ptr(rstd), _ptr(dy), _ptr(dx), _ptr(dgamma), _ptr(dA),
                                 _ptr(dB), ws.ptr, ws.nbytes, _stream(stream)),
           "boost_block_bwd")
    return dx, dgamma, dA, dB


def block_bwd_swiglu(desc: Desc, h, A, B, dy, gate, up, ws: Workspace, *, dgate=None,
                     dup=None, dA=None, dB=None, stream=None):
    """Backward of a no-norm block whose input is h = silu(gate)*up: (dgate, dup, dA, dB)."""
    bf = torch.bfloat16
    _need(h, "h", bf, (desc.T, desc.d))
    _need(A, "A", bf, (desc.d, desc.k * desc.r))
    _need(B, "B", bf, (desc.k, desc.r, desc.n))
    _need(dy, "dy", bf, (desc.k, desc.T, desc.n))
    _need(gate, "gate", bf, (desc.T, desc.d))
    _need(up, "up", bf, (desc.T, desc.d))
    dev = h.device
    if dgate is None:
        dgate = torch.empty(desc.T, desc.d, dtype=bf, device=dev)
    if dup is None:
        dup = torch.empty(desc.T, desc.d, dtype=bf, device=dev)
    if dA is None:
        dA = torch.empty(desc.d, desc.k * desc.r, dtype=bf, device=dev)
    if dB is None:
        dB = torch.empty(desc.k, desc.r, desc.n, dtype=bf, device=dev)
    _check(lib().boost_block_bwd_swiglu(ctypes.byref(desc), _ptr(h), _ptr(A), _ptr(B), _ptr(dy),
                                        _ptr(gate), _ptr(up), _ptr(dgate), _ptr(dup), _ptr(dA),
                                        _ptr(dB), ws.ptr, ws.nbytes, _stream(stream)),
           "boost_block_bwd_swiglu")
    return dgate, dup, dA, dB


def swiglu_fwd(gate, up, h=None, stream=None):
    bf = torch.bfloat16
    _need(gate, "gate", bf)
    _need(up, "up", bf, gate.shape)
    T, n = gate.shape
    if h is None:
        h = torch.empty_like(gate)
    _check(lib().boost_swiglu_fwd(T, n, _ptr(gate), _ptr(up), _ptr(h), _stream(stream)),
           "boost_swiglu_fwd")
    return h


def swiglu_bwd(gate, up, dh, dgate=None, dup=None, stream=None):
    bf = torch.bfloat16
    _need(gate, "gate", bf)
    _need(up, "up", bf, gate.shape)
    _need(dh, "dh", bf, gate.shape)
    T, n = gate.shape
    if dgate is None:
        dgate = torch.empty_like(gate)
    if dup is None:
        dup = torch.empty_like(gate)
    _check(lib().boost_swiglu_bwd(T, n, _ptr(gate), _ptr(up), _ptr(dh), _ptr(dgate), _ptr(dup),
                                  _stream(stream)), "boost_swiglu_bwd")
    return dgate, dup


def add(a, b, out=None, stream=None):
    bf = torch.bfloat16
    _need(a, "a", bf)
    _need(b, "b", bf, a.shape)
    if out is None:
        out = torch.empty_like(a)
    _check(lib().boost_add(a.numel(), _ptr(a), _ptr(b), _ptr(out), _stream(stream)), "boost_add")
    return out


def check(ws: Workspace, stream=None):
    """Synchronise and raise if a kernel recorded a device-side error."""
    _check(lib().boost_block_check(ws.ptr, _stream(stream)), "boost_block_check")


def profile_enable(on: bool):
    _check(lib().boost_profile_enable(1 if on else 0), "boost_profile_enable")


def profile_only(name=None):
    """Time only the named kernel's operations (None: every kernel)."""
    L = lib()
    idx = -1
    if name is not None:
        names = {}
        for i in range(L.boost_profile_kernel_count()):
            nm = ctypes.c_char_p()
            _check(L.boost_profile_read(i, ctypes.byref(nm), None, None, None, None),
                   "boost_profile_read")
            names[nm.value.decode()] = i
        if name not in names:
            raise KeyError(name)
        idx = names[name]
    _check(L.boost_profile_only(idx), "boost_profile_only")


def profile_kernels():
    """{kernel name: kernels launched} for kernels that ran (an operation split over
    concurrent launches counts each of them)."""
    L = lib()
    out = {}
    for i in range(L.boost_profile_kernel_count()):
        name = ctypes.c_char_p()
        n = ctypes.c_int64(0)
        _check(L.boost_profile_read(i, ctypes.byref(name), None, None, None, None),
               "boost_profile_read")
        _check(L.boost_profile_read_kernels(i, ctypes.byref(n)), "boost_profile_read_kernels")
        if n.value:
            out[name.value.decode()] = n.value
    return out


def profile_read():
    """{kernel name: (launches, total_ms, total_flops, total_bytes)} for kernels that ran."""
    L = lib()
    out = {}
    for i in range(L.boost_profile_kernel_count()):
        name = ctypes.c_char_p()
        n = ctypes.c_int64(0)
        ms, fl, by = ctypes.c_double(0), ctypes.c_double(0), ctypes.c_double(0)
        _check(L.boost_profile_read(i, ctypes.byref(name), ctypes.byref(n), ctypes.byref(ms),
                                    ctypes.byref(fl), ctypes.byref(by)), "boost_profile_read")
        if n.value:
            out[name.value.decode()] = (n.value, ms.value, fl.value, by.value)
    return out


def debug_count_writes(counts=None):
    """Start (with a zeroed int32 CUDA tensor) or stop (None) write counting."""
    if counts is None:
        _check(lib().boost_debug_count_writes(None, 0), "boost_debug_count_writes")
        return
    if counts.dtype != torch.int32 or not counts.is_cuda or not counts.is_contiguous():
        raise TypeError("counts must be a contiguous int32 CUDA tensor")
    _check(lib().boost_debug_count_writes(_ptr(counts), counts.numel()),
           "boost_debug_count_writes")


def debug_count_log():
    """[(offset, M, N, ld, planes, splits, plane_stride, split_stride)] of the recorded
    GEMM operations; raises if the count buffer ran out."""
    L = lib()
    n = L.boost_debug_count_log(None, 0)
    if n < 0:
        raise RuntimeError("write-count buffer too small")
    buf = (ctypes.c_int64 * (8 * max(n, 1)))()
    L.boost_debug_count_log(buf, n)
    return [tuple(buf[8 * i:8 * i + 8]) for i in range(n)]


def debug_wait_timeout(ws: Workspace, limit_us: int, stream=None):
    _check(lib().boost_debug_wait_timeout(ws.ptr, ws.nbytes, int(limit_us), _stream(stream)),
           "boost_debug_wait_timeout")
