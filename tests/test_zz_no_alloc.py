"""wq4_mm_static_scratch: the variant of wq4_mm for callers that cannot allocate device memory
(its K-split scratch is a fixed array inside the library). Called through the C ABI, call after
call, it must give wq4_mm's bits where wq4_mm's plan fits the array, and the same sums within the
parity tolerance where it keeps the tiles whole instead. This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

import oracle as O
import wq4_inputs as I
from tests.wq4_testutil import from_cuda16, gpu_prepack, to_cuda16

pytestmark = pytest.mark.gpu


def _call(lib, X, blob, Y, p):
    clib = lib.load_library()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return clib.wq4_mm_static_scratch(ctypes.c_void_p(X.data_ptr()), ctypes.c_void_p(blob.data_ptr()),
                                      ctypes.c_void_p(Y.data_ptr()), p.M, p.N, p.K, 128, lib.DTYPES[p.dtype],
                                      lib.QTYPES[p.qtype], stream)


STATIC_SCRATCH_BYTES = 24 << 20

# (M, N, K, dtype, qtype): the decode kernel (M = 8), cluster-split and whole tiles (M = 128), two
# K-split plans whose scratch would exceed the fixed array (M = 1024 and the 4096-token prefill
# shape), which then keep their tiles whole, and float zeros (the activation-sum table in the array).
SHAPES = [(8, 4096, 4096, "bf16", "u4b8"), (128, 14336, 4096, "bf16", "u4_zp"),
          (1024, 4096, 4096, "bf16", "u4b8"), (4096, 4096, 14336, "bf16", "u4b8"),
          (300, 512, 1024, "bf16", "u4_fzp")]


@pytest.mark.parametrize("M,N,K,dtype,qtype", SHAPES)
def test_static_scratch_default_options(lib, M, N, K, dtype, qtype):
    p = I.make_problem(M, N, K, dtype, qtype, seed=3000 + M)
    blob = gpu_prepack(lib, p)
    X = to_cuda16(p.X_bits, p.dtype)
    ws = lib.workspace_bytes(M, N, K, qtype=qtype)
    want_bits = from_cuda16(lib.mm(X, blob, p.N, qtype=p.qtype))
    rows = None if M <= 128 else np.random.default_rng(M).choice(M, 48, replace=False)
    ref = O.mm_problem(p, rows)
    for _ in range(2):
        Y = torch.full((p.M, p.N), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _call(lib, X, blob, Y, p) == lib.OK
        assert lib.get_last_error() == lib.OK
        got_bits = from_cuda16(Y)
        if ws <= STATIC_SCRATCH_BYTES:
            # the same plan as wq4_mm: the same bits
            assert np.array_equal(got_bits, want_bits)
        else:
            # tiles kept whole: the same sums in another order
            st = O.check_tolerance(O.decode16(got_bits, p.dtype), O.decode16(want_bits, p.dtype))
            assert st["violations"] == 0, st
        got = O.decode16(got_bits, p.dtype)
        st = O.check_tolerance(got if rows is None else got[rows], ref)
        assert st["violations"] == 0, st
    if M >= 1024:
        assert ws > STATIC_SCRATCH_BYTES   # the re-planned case is the one exercised


def test_static_scratch_split_matches_wq4_mm_twice(lib):
    # Every tile goes through the K-split path (split over CTAs, partial sums and tile counters
    # in scratch), whatever the planner would pick for this shape on its own.
    p = I.make_problem(128, 14336, 1024, "bf16", "u4_zp", seed=2024)
    lib.set_option(lib.OPT_SPLIT_ALL, 1)
    try:
        assert lib.workspace_bytes(p.M, p.N, p.K) > 0
        blob = gpu_prepack(lib, p)
        X = to_cuda16(p.X_bits, p.dtype)
        want = O.decode16(from_cuda16(lib.mm(X, blob, p.N, qtype=p.qtype)), p.dtype)
        for _ in range(2):
            Y = torch.full((p.M, p.N), float("nan"), dtype=torch.bfloat16, device="cuda")
            assert _call(lib, X, blob, Y, p) == lib.OK
            assert lib.get_last_error() == lib.OK
            got = O.decode16(from_cuda16(Y), p.dtype)
            st = O.check_tolerance(got, want)
            assert st["violations"] == 0, st
            assert O.check_tolerance(got, O.mm_problem(p))["violations"] == 0
    finally:
        lib.set_option(lib.OPT_SPLIT_ALL, 0)


def test_static_scratch_rejects_plans_beyond_its_size(lib):
    p = I.make_problem(128, 14336, 1024, "bf16", "u4_zp", seed=2025)
    blob = gpu_prepack(lib, p)
    X = to_cuda16(p.X_bits, p.dtype)
    Y = torch.empty((p.M, p.N), dtype=torch.bfloat16, device="cuda")
    lib.set_option(lib.OPT_GRID, 4096)          # 4096 persistent CTAs need far more than the fixed array
    try:
        assert _call(lib, X, blob, Y, p) == lib.ERR_WORKSPACE
    finally:
        lib.set_option(lib.OPT_GRID, 0)
    assert lib.get_last_error() == lib.OK
