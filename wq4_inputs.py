"""Seeded synthetic inputs for the W4A16 GEMM, shared by the oracle tests, the GPU tests and the bench.

This module draws random numbers and stores them in the input formats of the library's API. It
holds none of the method's arithmetic: no unpacking, no dequantisation, no products. The CPU
oracle (``oracle/``) and the CUDA path both receive what this module produces and nothing else.

Input formats (the layouts the public API takes):

* ``X_bits``  uint16 [M][K]      activations as raw bf16 or fp16 bit patterns, row-major.
* ``Wq``      uint32 [N][K/8]    4-bit weight codes q in [0, 15], eight per word along K; code of
                                 element k = 8*j + i sits in bits [4i, 4i+4) of word j.
* ``S_bits``  uint16 [K/G][N]    one scale per (group, weight row), N contiguous, raw 16-bit bits.
* ``Z``       uint32 [K/G][N/8]  (uint4 + zero-point mode) zero points z in [0, 15], eight per
                                 word along N with the same little-endian nibble order;
              uint16 [K/G][N]    (uint4 + float-zero mode) one pre-scaled float zero per (group,
                                 weight row), raw 16-bit bits, like the scales.

Draw recipe (seed = 1000 + the workload's 1-based index): one ``numpy.random.default_rng(seed)``
draws, in this order, X ~ N(0, 1) in fp32, the codes q ~ U{0..15}, the scales s ~ U[0.005, 0.02]
in fp32, the zero points z ~ U{6..9} (zero-point mode) or the float zeros ~ U[-0.18, -0.03] in
fp32 (float-zero mode). The grouped workload draws X for
all sum_M rows first, then each problem's q, s (and z) in problem order, then the token split
M_p ~ Multinomial(sum_M, uniform); problem p takes the next M_p rows of X. fp32 draws are rounded
to the 16-bit type with round-to-nearest-even.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np

GROUP = 128
BF16 = "bf16"
FP16 = "fp16"
U4B8 = "u4b8"      # stored code minus 8
U4_ZP = "u4_zp"    # stored code minus a per-group zero point
U4_FZP = "u4_fzp"  # stored code times the scale plus a per-group float zero (pre-scaled)


def f32_to_bits(a: np.ndarray, dtype: str) -> np.ndarray:
    """Round fp32 values to bf16/fp16 (round-to-nearest-even) and return the raw uint16 bits."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    if dtype == FP16:
        return a.astype(np.float16).view(np.uint16)
    if dtype != BF16:
        raise ValueError(dtype)
    u = a.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def pack_u4(codes: np.ndarray) -> np.ndarray:
    """Pack 4-bit codes along the last axis, eight per uint32, element 8j+i in bits [4i, 4i+4)."""
    codes = np.asarray(codes)
    if codes.shape[-1] % 8:
        raise ValueError("last axis must be a multiple of 8")
    c = codes.astype(np.uint32).reshape(codes.shape[:-1] + (codes.shape[-1] // 8, 8))
    shifts = (4 * np.arange(8, dtype=np.uint32))
    return np.bitwise_or.reduce(c << shifts, axis=-1).astype(np.uint32)


@dataclasses.dataclass
class Problem:
    """One GEMM problem Y[M,N] = X[M,K] . dequant(Wq)[N,K]^T in API formats."""
    M: int
    N: int
    K: int
    dtype: str
    qtype: str
    X_bits: np.ndarray               # uint16 [M][K]
    q: np.ndarray                    # uint8  [N][K]  (the codes before packing, for tests)
    Wq: np.ndarray                   # uint32 [N][K/8]
    S_bits: Optional[np.ndarray]     # uint16 [K/G][N]; None = no scales (direct conversion)
    z: Optional[np.ndarray] = None   # uint8  [K/G][N] (u4_zp)
    Z: Optional[np.ndarray] = None   # zero points as the API takes them: uint32 [K/G][N/8] of 4-bit
                                     # values (u4_zp), or uint16 [K/G][N] float zeros (u4_fzp)
    group_size: int = GROUP


def problem_from_codes(X_bits, q, S_bits, z, dtype, qtype, group_size=GROUP) -> Problem:
    """Build a Problem from explicit arrays (used by hand-made test cases)."""
    X_bits = np.ascontiguousarray(X_bits, dtype=np.uint16)
    q = np.ascontiguousarray(q, dtype=np.uint8)
    S_bits = None if S_bits is None else np.ascontiguousarray(S_bits, dtype=np.uint16)
    M, K = X_bits.shape
    N = q.shape[0]
    Z = None
    if qtype == U4_ZP:
        z = np.ascontiguousarray(z, dtype=np.uint8)
        Z = pack_u4(z)
    elif qtype == U4_FZP:                   # z holds the float zeros' 16-bit patterns
        Z = np.ascontiguousarray(z, dtype=np.uint16)
        z = None
    else:
        z = None
    return Problem(M, N, K, dtype, qtype, X_bits, q, pack_u4(q), S_bits, z, Z, group_size)


def _draw(rng, M, N, K, dtype, qtype, X_bits=None, group_size=GROUP, scaled=True):
    if X_bits is None:
        X_bits = f32_to_bits(rng.standard_normal((M, K), dtype=np.float32), dtype)
    q = rng.integers(0, 16, size=(N, K), dtype=np.uint8)
    ng = K // group_size
    S_bits = f32_to_bits(rng.uniform(0.005, 0.02, size=(ng, N)).astype(np.float32), dtype) if scaled else None
    z = rng.integers(6, 10, size=(ng, N), dtype=np.uint8) if qtype == U4_ZP else None
    if qtype == U4_FZP:                     # about -z s for z in 6..9 and s in the scale range
        z = f32_to_bits(rng.uniform(-0.18, -0.03, size=(ng, N)).astype(np.float32), dtype)
    return problem_from_codes(X_bits, q, S_bits, z, dtype, qtype, group_size)


def make_problem(M: int, N: int, K: int, dtype: str = BF16, qtype: str = U4B8, seed: int = 0,
                 group_size: int = GROUP, scaled: bool = True) -> Problem:
    """One seeded problem of the given shape, drawn by the recipe in the module docstring; one
    scale (and zero point) row per ``group_size`` K elements, or no scales if not ``scaled``."""
    if K % group_size:
        raise ValueError("K must be a multiple of the group size")
    rng = np.random.default_rng(seed)
    return _draw(rng, M, N, K, dtype, qtype, group_size=group_size, scaled=scaled)


def make_grouped(sum_M: int, P: int, N: int, K: int, dtype: str = BF16, qtype: str = U4B8,
                 seed: int = 0, M_list: Optional[List[int]] = None) -> List[Problem]:
    """P independent problems sharing (N, K); the token split is a seeded multinomial of sum_M
    over P equal probabilities unless ``M_list`` gives it explicitly."""
    rng = np.random.default_rng(seed)
    X_all = f32_to_bits(rng.standard_normal((sum_M, K), dtype=np.float32), dtype)
    weights = [_draw(rng, 0, N, K, dtype, qtype, X_bits=np.zeros((0, K), np.uint16)) for _ in range(P)]
    if M_list is None:
        M_list = [int(v) for v in rng.multinomial(sum_M, [1.0 / P] * P)]
    if sum(M_list) != sum_M or len(M_list) != P:
        raise ValueError("M_list must have P entries summing to sum_M")
    out, row = [], 0
    for p, Mp in enumerate(M_list):
        w = weights[p]
        w.X_bits = np.ascontiguousarray(X_all[row:row + Mp])
        w.M = Mp
        row += Mp
        out.append(w)
    return out


# The five workloads: name -> constructor arguments. Seeds are 1000 + the 1-based index.
WORKLOADS = {
    "tiny_m16_n256_k512_fp16_u4b8": dict(kind="mm", M=16, N=256, K=512, dtype=FP16, qtype=U4B8, seed=1001),
    "decode_m8_n4096_k4096_bf16_u4b8": dict(kind="mm", M=8, N=4096, K=4096, dtype=BF16, qtype=U4B8, seed=1002),
    "asym_m128_n14336_k4096_bf16_u4zp": dict(kind="mm", M=128, N=14336, K=4096, dtype=BF16, qtype=U4_ZP, seed=1003),
    "prefill_m4096_n4096_k14336_bf16_u4b8": dict(kind="mm", M=4096, N=4096, K=14336, dtype=BF16, qtype=U4B8, seed=1004),
    "grouped_8x_n14336_k4096_summ1024_bf16_u4b8": dict(kind="grouped", sum_M=1024, P=8, N=14336, K=4096,
                                                       dtype=BF16, qtype=U4B8, seed=1005),
}


def make_workload(name: str):
    """Problem (or list of Problems for the grouped workload) for one named workload."""
    spec = dict(WORKLOADS[name])
    kind = spec.pop("kind")
    if kind == "mm":
        return make_problem(**spec)
    return make_grouped(**spec)


def algorithmic_bytes(M: int, N: int, K: int, qtype: str, group_size: int = GROUP) -> int:
    """Bytes the method must move at minimum: X + packed W + scales (+ zeros) + Y, each once."""
    ng = K // group_size
    b = 2 * M * K + N * K // 2 + 2 * ng * N + 2 * M * N
    if qtype == U4_ZP:
        b += ng * N // 2
    if qtype == U4_FZP:
        b += 2 * ng * N
    return b


def algorithmic_flops(M: int, N: int, K: int) -> int:
    return 2 * M * N * K
