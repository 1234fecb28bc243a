"""Helpers shared by the GPU tests: move seeded numpy inputs to torch CUDA tensors and back."""
import numpy as np

import oracle as O


def torch_dtype(dtype):
    import torch
    return torch.bfloat16 if dtype == "bf16" else torch.float16


def to_cuda16(bits: np.ndarray, dtype: str):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch_dtype(dtype)).cuda()


def to_cuda32(words: np.ndarray):
    import torch
    return torch.from_numpy(np.ascontiguousarray(words).view(np.int32)).cuda()


def from_cuda16(t) -> np.ndarray:
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def from_cuda32(t) -> np.ndarray:
    return t.contiguous().cpu().numpy().view(np.uint32)


def gpu_prepack(wq4, p):
    Z = None
    if p.Z is not None:
        Z = to_cuda16(p.Z, p.dtype) if p.qtype == "u4_fzp" else to_cuda32(p.Z)
    S = to_cuda16(p.S_bits, p.dtype) if p.S_bits is not None else None
    return wq4.prepack(to_cuda32(p.Wq), S, Z, qtype=p.qtype, group_size=p.group_size, dtype=p.dtype)


def gpu_mm(wq4, p, blob=None, **kw):
    blob = gpu_prepack(wq4, p) if blob is None else blob
    Y = wq4.mm(to_cuda16(p.X_bits, p.dtype), blob, p.N, qtype=p.qtype, group_size=p.group_size, **kw)
    return Y


def y_as_f64(Y, dtype: str) -> np.ndarray:
    return O.decode16(from_cuda16(Y), dtype)


def assert_parity(Y_gpu_f64: np.ndarray, Y_ref: np.ndarray, what: str = ""):
    st = O.check_tolerance(Y_gpu_f64, Y_ref)
    assert st["violations"] == 0, "%s: %s" % (what, st)
    return st
