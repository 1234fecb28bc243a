"""Python binding of the wq4 C ABI (include/wq4.h): W4A16 GEMM for GB300 (sm_103a).

Argument marshalling only: every step of the computation runs in the CUDA kernels of libwq4.so.
Tensors are passed by device pointer together with torch's current CUDA stream; torch supplies
device memory and streams and nothing else. There is no CPU fallback: the calls raise if the
library is missing or a tensor is not on a CUDA device.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import List, Optional, Sequence

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libwq4.so")
DEBUG_LIB_PATH = os.path.join(PKG, "libwq4_debug.so")   # the bounds-checking build (build(debug=True))
HEADER = os.path.join(os.path.dirname(PKG), "include", "wq4.h")

OK, ERR_INVALID, ERR_ALIGN, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT, ERR_BOUNDS = 0, -1, -2, -3, -4, -5, -6, -7
DTYPES = {"bf16": 0, "fp16": 1}
QTYPES = {"u4b8": 0, "u4_zp": 1, "u4_fzp": 2}
OPT_TOKEN_TILE, OPT_GRID, OPT_SPLIT_ALL, OPT_TIMEOUT_CYCLES, OPT_TRACE, OPT_A_IN_SMEM, OPT_CLUSTER = 1, 2, 3, 4, 5, 6, 7
OPT_DECODE, OPT_PDL, OPT_TEST_STALL = 8, 9, 10
OPT_CONST_WEIGHTS, OPT_DECODE_DEPTH, OPT_DECODE_TRIGGER, OPT_VERIFY_DEV_PTRS = 11, 12, 13, 14
GROUP = 128

_lib = None


class Wq4Error(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s: %s (status %d)" % (what, _lib.wq4_status_string(status).decode() if _lib else "?", status))


def build(force: bool = False, debug: bool = False) -> str:
    """Build libwq4.so (or, with debug=True, the bounds-checking libwq4_debug.so)."""
    from .builder import build as _build
    return _build(force=force, debug=debug)


def load_library(path: str = LIB_PATH):
    """Load libwq4.so (raises if it has not been built); every call of this module goes through
    the library loaded first (use_library swaps it)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError("%s is not built: run `python -m weight_only_quantized_wq4_gb300.builder`" %
                           os.path.basename(path))
    lib = ctypes.CDLL(path)
    c_int, c_size, vp, ll = ctypes.c_int, ctypes.c_size_t, ctypes.c_void_p, ctypes.c_longlong
    ip = ctypes.POINTER(ctypes.c_int)
    vpp = ctypes.POINTER(ctypes.c_void_p)
    sigs = {
        "wq4_version": (c_int, []),
        "wq4_status_string": (ctypes.c_char_p, [c_int]),
        "wq4_prepacked_bytes": (c_size, [c_int, c_int, c_int, c_int]),
        "wq4_prepack": (c_int, [vp, vp, vp, c_int, c_int, c_int, c_int, c_int, vp, vp]),
        "wq4_unprepack": (c_int, [vp, c_int, c_int, c_int, c_int, c_int, vp, vp, vp, vp]),
        "wq4_workspace_bytes": (c_int, [c_int, c_int, c_int, c_int, ctypes.POINTER(c_size)]),
        "wq4_workspace_bytes_ex": (c_int, [c_int, c_int, c_int, c_int, c_int, ctypes.POINTER(c_size)]),
        "wq4_mm": (c_int, [vp, vp, vp, c_int, c_int, c_int, c_int, c_int, c_int, vp, c_size, vp]),
        "wq4_mm_ex": (c_int, [vp, vp, vp, c_int, c_int, c_int, c_int, c_int, c_int, ctypes.c_float, vp,
                              ctypes.c_float, vp, vp, c_size, vp]),
        "wq4_grouped_workspace_bytes": (c_int, [c_int, ip, ip, ip, c_int, ctypes.POINTER(c_size)]),
        "wq4_grouped_mm": (c_int, [c_int, ip, ip, ip, vpp, vpp, vpp, c_int, c_int, c_int, vp, c_size, vp]),
        "wq4_grouped_workspace_bytes_ex": (c_int, [c_int, ip, ip, ip, c_int, c_int, ctypes.POINTER(c_size)]),
        "wq4_mm_static_scratch": (c_int, [vp, vp, vp, c_int, c_int, c_int, c_int, c_int, c_int, vp]),
        "wq4_grouped_device_m_workspace_bytes": (c_int, [c_int, ctypes.POINTER(c_size)]),
        "wq4_grouped_mm_device_m": (c_int, [c_int, vp, ip, ip, ip, vpp, vpp, vpp, c_int, c_int, c_int, vp, c_size, vp]),
        "wq4_grouped_dev_ptrs_workspace_bytes": (c_int, [c_int, ip, ip, ip, c_int, ctypes.POINTER(c_size)]),
        "wq4_grouped_mm_dev_ptrs": (c_int, [c_int, ip, ip, ip, vp, vp, vp, c_int, c_int, c_int, vp, c_size, vp]),
        "wq4_get_last_error": (c_int, [vp]),
        "wq4_debug_checks": (c_int, []),
        "wq4_last_violation": (c_int, [ip]),
        "wq4_set_option": (c_int, [c_int, ll]),
        "wq4_get_option": (ll, [c_int]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def use_library(path: str):
    """Route every call of this module through the library at `path` (libwq4_debug.so, say), loading
    it if needed; returns the library it replaces (None if none was loaded), for restore_library."""
    global _lib
    old = _lib
    _lib = None
    try:
        load_library(path)
    except Exception:
        _lib = old
        raise
    return old


def restore_library(old) -> None:
    """Undo use_library: route the calls through `old` again."""
    global _lib
    _lib = old


def debug_checks() -> bool:
    """True when the library in use is the bounds-checking debug build."""
    return bool(load_library().wq4_debug_checks())


def last_violation():
    """(site, value, context, context) of the first bounds violation the last ERR_BOUNDS report read
    back, or None; clears it."""
    rec = (ctypes.c_int * 4)()
    seen = load_library().wq4_last_violation(rec)
    return tuple(rec) if seen == 1 else None


def header_functions(path: str = HEADER) -> List[str]:
    """Names of the functions include/wq4.h declares."""
    with open(path) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(wq4_[a-z_]+)\s*\(", text)))


def _check(status: int, what: str) -> None:
    if status != OK:
        raise Wq4Error(status, what)


def _torch():
    import torch
    return torch


def _stream(device) -> ctypes.c_void_p:
    torch = _torch()
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _cuda(t, name: str):
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return ctypes.c_void_p(t.data_ptr())


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return DTYPES["bf16"]
    if t.dtype == torch.float16:
        return DTYPES["fp16"]
    raise ValueError("activations and scales must be bfloat16 or float16")


# ------------------------------------------------------------------------------------ API
def set_option(key: int, value: int) -> None:
    _check(load_library().wq4_set_option(key, value), "wq4_set_option")


def get_option(key: int) -> int:
    return int(load_library().wq4_get_option(key))


def get_last_error(device=None) -> int:
    """Synchronise torch's current stream and return the library's status (0 = ok)."""
    return int(load_library().wq4_get_last_error(_stream(device)))


def prepacked_bytes(N: int, K: int, qtype: str = "u4b8", group_size: int = GROUP) -> int:
    return int(load_library().wq4_prepacked_bytes(N, K, group_size, QTYPES[qtype]))


def prepack(Wq, scales, zeros=None, qtype: str = "u4b8", group_size: int = GROUP, dtype: str = "bf16"):
    """Wq: int32 [N][K/8] (packed codes), scales: bf16/fp16 [K/G][N] or None (no scales, uint4b8
    only; ``dtype`` then names the activation type), zeros: int32 [K/G][N/8] (u4_zp), bf16/fp16
    float zeros [K/G][N] (u4_fzp) or None. Returns the prepacked blob (uint8 CUDA tensor)."""
    torch = _torch()
    lib = load_library()
    N, K = Wq.shape[0], Wq.shape[1] * 8
    nbytes = prepacked_bytes(N, K, qtype, group_size)
    if nbytes == 0:
        raise Wq4Error(ERR_UNSUPPORTED, "wq4_prepacked_bytes")
    blob = torch.empty(nbytes, dtype=torch.uint8, device=Wq.device)
    zp = _cuda(zeros, "zeros") if zeros is not None else None
    sp = _cuda(scales, "scales") if scales is not None else None
    code = _dtype_code(scales) if scales is not None else DTYPES[dtype]
    _check(lib.wq4_prepack(_cuda(Wq, "Wq"), sp, zp, N, K, group_size, code, QTYPES[qtype], _cuda(blob, "blob"),
                           _stream(Wq.device)), "wq4_prepack")
    return blob


def unprepack(blob, N: int, K: int, dtype: str = "bf16", qtype: str = "u4b8", group_size: int = GROUP):
    """Inverse of prepack: (Wq int32 [N][K/8], scales [K/G][N], zeros: int32 [K/G][N/8] (u4_zp),
    float zeros [K/G][N] (u4_fzp) or None)."""
    torch = _torch()
    lib = load_library()
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    Wq = torch.empty((N, K // 8), dtype=torch.int32, device=blob.device)
    sc = torch.empty((K // group_size, N), dtype=tdt, device=blob.device)
    zs = None
    if qtype == "u4_zp":
        zs = torch.empty((K // group_size, N // 8), dtype=torch.int32, device=blob.device)
    elif qtype == "u4_fzp":
        zs = torch.empty((K // group_size, N), dtype=tdt, device=blob.device)
    _check(lib.wq4_unprepack(_cuda(blob, "blob"), N, K, group_size, DTYPES[dtype], QTYPES[qtype], _cuda(Wq, "Wq"),
                             _cuda(sc, "scales"), _cuda(zs, "zeros") if zs is not None else None,
                             _stream(blob.device)), "wq4_unprepack")
    return Wq, sc, zs


def workspace_bytes(M: int, N: int, K: int, group_size: int = GROUP, qtype: str = "u4b8") -> int:
    out = ctypes.c_size_t(0)
    _check(load_library().wq4_workspace_bytes_ex(M, N, K, group_size, QTYPES[qtype], ctypes.byref(out)),
           "wq4_workspace_bytes_ex")
    return int(out.value)


def grouped_workspace_bytes(Ms: Sequence[int], Ns: Sequence[int], Ks: Sequence[int], group_size: int = GROUP,
                            qtype: str = "u4b8") -> int:
    P = len(Ms)
    arr = ctypes.c_int * P
    out = ctypes.c_size_t(0)
    _check(load_library().wq4_grouped_workspace_bytes_ex(P, arr(*Ms), arr(*Ns), arr(*Ks), group_size, QTYPES[qtype],
                                                         ctypes.byref(out)),
           "wq4_grouped_workspace_bytes_ex")
    return int(out.value)


def alloc_workspace(nbytes: int, device="cuda"):
    """A zero-filled workspace (the library needs it zeroed once; calls keep it so)."""
    torch = _torch()
    return torch.zeros(max(nbytes, 16), dtype=torch.uint8, device=device)


def mm(X, blob, N: int, qtype: str = "u4b8", workspace=None, out=None, group_size: int = GROUP,
       alpha: float = 1.0, C=None, beta: float = 0.0, bias=None):
    """Y[M,N] = X[M,K] . dequant(W)^T for a prepacked weight blob (prepacked with group_size).
    With alpha / C / beta / bias given: Y = alpha (X . dequant(W)^T) + beta C + bias (wq4_mm_ex)."""
    torch = _torch()
    lib = load_library()
    M, K = X.shape
    if out is None:
        out = torch.empty((M, N), dtype=X.dtype, device=X.device)
    if workspace is None and M > 0:
        nbytes = workspace_bytes(M, N, K, group_size, qtype)
        workspace = alloc_workspace(nbytes, X.device) if nbytes > 0 else None   # decode sizes need none
    ws_ptr = _cuda(workspace, "workspace") if workspace is not None else None
    ws_n = workspace.numel() if workspace is not None else 0
    if alpha == 1.0 and beta == 0.0 and C is None and bias is None:
        _check(lib.wq4_mm(_cuda(X, "X"), _cuda(blob, "blob"), _cuda(out, "Y") if M > 0 else None, M, N, K,
                          group_size, _dtype_code(X), QTYPES[qtype], ws_ptr, ws_n, _stream(X.device)), "wq4_mm")
        return out
    cp = _cuda(C, "C") if C is not None else None
    bp = _cuda(bias, "bias") if bias is not None else None
    _check(lib.wq4_mm_ex(_cuda(X, "X"), _cuda(blob, "blob"), _cuda(out, "Y") if M > 0 else None, M, N, K,
                         group_size, _dtype_code(X), QTYPES[qtype], float(alpha), cp, float(beta), bp, ws_ptr, ws_n,
                         _stream(X.device)), "wq4_mm_ex")
    return out


def grouped_mm(Xs: Sequence, blobs: Sequence, N: Sequence[int], qtype: str = "u4b8", workspace=None,
               outs: Optional[Sequence] = None, group_size: int = GROUP):
    """Independent problems Y_p = X_p . dequant(W_p)^T in one launch (every blob prepacked with
    group_size)."""
    torch = _torch()
    lib = load_library()
    P = len(Xs)
    Ms = [int(x.shape[0]) for x in Xs]
    Ks = [int(x.shape[1]) for x in Xs]
    Ns = [int(n) for n in N]
    if outs is None:
        outs = [torch.empty((m, n), dtype=x.dtype, device=x.device) for x, m, n in zip(Xs, Ms, Ns)]
    if workspace is None:
        workspace = alloc_workspace(grouped_workspace_bytes(Ms, Ns, Ks, group_size, qtype), Xs[0].device)
    arr = ctypes.c_int * P
    ptrs = ctypes.c_void_p * P
    xp = ptrs(*[x.data_ptr() if m > 0 else None for x, m in zip(Xs, Ms)])
    wp = ptrs(*[b.data_ptr() for b in blobs])
    yp = ptrs(*[y.data_ptr() if m > 0 else None for y, m in zip(outs, Ms)])
    _check(lib.wq4_grouped_mm(P, arr(*Ms), arr(*Ns), arr(*Ks), xp, wp, yp, group_size, _dtype_code(Xs[0]), QTYPES[qtype],
                              _cuda(workspace, "workspace"), workspace.numel(), _stream(Xs[0].device)),
           "wq4_grouped_mm")
    return list(outs)


def grouped_device_m_workspace_bytes(P: int) -> int:
    """Workspace of wq4_grouped_mm_device_m for P problems (the device tile table)."""
    nb = ctypes.c_size_t(0)
    _check(load_library().wq4_grouped_device_m_workspace_bytes(P, ctypes.byref(nb)),
           "wq4_grouped_device_m_workspace_bytes")
    return int(nb.value)


def grouped_mm_device_m(Xs: Sequence, blobs: Sequence, M_dev, N: Sequence[int], qtype: str = "u4b8",
                        workspace=None, outs: Optional[Sequence] = None, group_size: int = GROUP):
    """Grouped GEMM with the token counts in device memory (``M_dev``: int32 CUDA tensor [P]).
    Xs[p] holds M_cap = Xs[p].shape[0] rows (its capacity); only the first M_dev[p] rows of each
    Y[p] are written."""
    torch = _torch()
    lib = load_library()
    P = len(Xs)
    caps = [int(x.shape[0]) for x in Xs]
    Ks = [int(x.shape[1]) for x in Xs]
    Ns = [int(n) for n in N]
    if M_dev.dtype != torch.int32 or not M_dev.is_cuda or M_dev.numel() != P:
        raise ValueError("M_dev must be an int32 CUDA tensor with one entry per problem")
    if outs is None:
        outs = [torch.empty((c, n), dtype=x.dtype, device=x.device) for x, c, n in zip(Xs, caps, Ns)]
    if workspace is None:
        workspace = torch.empty(grouped_device_m_workspace_bytes(P), dtype=torch.uint8, device=Xs[0].device)
    arr = ctypes.c_int * P
    ptrs = ctypes.c_void_p * P
    xp = ptrs(*[x.data_ptr() if c > 0 else None for x, c in zip(Xs, caps)])
    wp = ptrs(*[b.data_ptr() for b in blobs])
    yp = ptrs(*[y.data_ptr() if c > 0 else None for y, c in zip(outs, caps)])
    _check(lib.wq4_grouped_mm_device_m(P, _cuda(M_dev, "M_dev"), arr(*caps), arr(*Ns), arr(*Ks), xp, wp, yp, group_size,
                                       _dtype_code(Xs[0]), QTYPES[qtype], _cuda(workspace, "workspace"),
                                       workspace.numel(), _stream(Xs[0].device)), "wq4_grouped_mm_device_m")
    return list(outs)


def grouped_dev_ptrs_workspace_bytes(M: Sequence[int], N: Sequence[int], K: Sequence[int],
                                     group_size: int = GROUP) -> int:
    """Workspace of wq4_grouped_mm_dev_ptrs for these shapes."""
    P = len(M)
    arr = ctypes.c_int * P
    nb = ctypes.c_size_t(0)
    _check(load_library().wq4_grouped_dev_ptrs_workspace_bytes(P, arr(*M), arr(*N), arr(*K), group_size,
                                                                ctypes.byref(nb)),
           "wq4_grouped_dev_ptrs_workspace_bytes")
    return int(nb.value)


def grouped_mm_dev_ptrs(M: Sequence[int], N: Sequence[int], K: Sequence[int], X_ptrs, W_ptrs, Y_ptrs,
                        dtype: str = "bf16", qtype: str = "u4b8", workspace=None, group_size: int = GROUP):
    """Grouped GEMM whose per-problem pointers are in device memory: X_ptrs, W_ptrs, Y_ptrs are int64
    CUDA tensors [P] of device addresses (written by any kernel earlier on the stream); the shapes
    M, N, K are host lists. Results land in the Y buffers the addresses name."""
    torch = _torch()
    lib = load_library()
    P = len(M)
    for t, nm in ((X_ptrs, "X_ptrs"), (W_ptrs, "W_ptrs"), (Y_ptrs, "Y_ptrs")):
        if t.dtype != torch.int64 or not t.is_cuda or t.numel() != P:
            raise ValueError("%s must be an int64 CUDA tensor with one address per problem" % nm)
    dev = X_ptrs.device
    if workspace is None:
        workspace = alloc_workspace(grouped_dev_ptrs_workspace_bytes(M, N, K, group_size), dev)
    arr = ctypes.c_int * P
    _check(lib.wq4_grouped_mm_dev_ptrs(P, arr(*M), arr(*N), arr(*K), _cuda(X_ptrs, "X_ptrs"), _cuda(W_ptrs, "W_ptrs"),
                                       _cuda(Y_ptrs, "Y_ptrs"), group_size, DTYPES[dtype], QTYPES[qtype],
                                       _cuda(workspace, "workspace"), workspace.numel(), _stream(dev)),
           "wq4_grouped_mm_dev_ptrs")
