"""The bounds-checking debug build (libwq4_debug.so, compiled with WQ4_DEBUG=1) on every kernel path.

Each case runs through the same Python API with the debug library swapped in, and checks three
things: parity with the oracle, WQ4_OK from wq4_get_last_error, and no recorded violation. Between
them the cases reach every check site:
  - the decode kernel's weight stages, activation pieces and output columns;
  - the GEMM's scheduled tiles, activation tiles, weight records and output columns;
  - the K-split slots and counters;
  - the activation-sum panels and their pre-pass;
  - the epilogue's C copies, both into the C buffer and into the activation ring;
  - the problem index of the grouped calls.
A check that fires is covered on the CPU (tests/test_check_predicates.py) and by the host-side
record plumbing. No case here plants an out-of-range coordinate in a kernel."""
import numpy as np
import pytest

import oracle as O
import wq4_inputs as I
from tests.wq4_testutil import assert_parity, gpu_mm, gpu_prepack, to_cuda16, y_as_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dbg(lib):
    """The package with every call routed through the debug library for this module."""
    lib.build(debug=True)
    old = lib.use_library(lib.DEBUG_LIB_PATH)
    try:
        assert lib.debug_checks(), "libwq4_debug.so was built without its checks"
        yield lib
    finally:
        lib.restore_library(old)


@pytest.fixture
def d(dbg):
    yield dbg
    for key in (dbg.OPT_TOKEN_TILE, dbg.OPT_GRID, dbg.OPT_SPLIT_ALL, dbg.OPT_CLUSTER, dbg.OPT_DECODE):
        dbg.set_option(key, 0)
    assert dbg.last_violation() is None


def clean(lib, what):
    rc = lib.get_last_error()
    assert rc == lib.OK, "%s: status %d, violation %s" % (what, rc, lib.last_violation())


def test_release_library_has_no_checks(lib):
    old = lib.use_library(lib.LIB_PATH)
    try:
        assert not lib.debug_checks()
    finally:
        lib.restore_library(old)


@pytest.mark.parametrize("M,N,K,dtype,qtype,G", [
    (8, 512, 1024, "bf16", "u4b8", 128), (5, 384, 768, "fp16", "u4_zp", 128), (3, 256, 1024, "bf16", "u4_fzp", 64),
    (32, 128, 4096, "fp16", "u4b8", 128), (1, 1024, 512, "bf16", "u4_zp", 64)])
def test_decode_paths(d, M, N, K, dtype, qtype, G):
    p = I.make_problem(M, N, K, dtype, qtype, seed=M + N, group_size=G)
    Y = gpu_mm(d, p)
    clean(d, "decode %s" % ((M, N, K, qtype, G),))
    assert_parity(y_as_f64(Y, dtype), O.mm_problem(p), "decode")


@pytest.mark.parametrize("token_tile", [16, 64, 128, 160, 192])
@pytest.mark.parametrize("split_all,grid,cluster", [(0, 0, 0), (1, 7, 0), (0, 0, 4)])
def test_gemm_schedules(d, token_tile, split_all, grid, cluster):
    """Whole tiles (a ragged last m-tile), K-split tiles over 7 CTAs, and cluster splits."""
    d.set_option(d.OPT_TOKEN_TILE, token_tile)
    d.set_option(d.OPT_SPLIT_ALL, split_all)
    d.set_option(d.OPT_GRID, grid)
    d.set_option(d.OPT_CLUSTER, cluster)
    d.set_option(d.OPT_DECODE, -1)
    M = 100 if cluster else 300
    p = I.make_problem(M, 384, 1280, "bf16", "u4_zp", seed=token_tile + grid + cluster)
    Y = gpu_mm(d, p)
    clean(d, "tile %d split %d grid %d cluster %d" % (token_tile, split_all, grid, cluster))
    assert_parity(y_as_f64(Y, "bf16"), O.mm_problem(p), "schedules")


@pytest.mark.parametrize("token_tile,G,split_all", [(64, 128, 0), (128, 64, 0), (192, 128, 1), (160, 64, 0)])
def test_gemm_float_zeros(d, token_tile, G, split_all):
    """The activation-sum pre-pass and the zero steps' panel copies."""
    d.set_option(d.OPT_TOKEN_TILE, token_tile)
    d.set_option(d.OPT_SPLIT_ALL, split_all)
    p = I.make_problem(200, 256, 1536, "fp16", "u4_fzp", seed=token_tile + G, group_size=G)
    Y = gpu_mm(d, p)
    clean(d, "float zeros tile %d G %d" % (token_tile, G))
    assert_parity(y_as_f64(Y, "fp16"), O.mm_problem(p), "float zeros")


@pytest.mark.parametrize("M,token_tile,split_all", [(300, 128, 0), (300, 192, 0), (200, 64, 1), (8, 0, 0)])
def test_epilogue_c_copies(d, M, token_tile, split_all):
    """C through the C buffer (token tiles with room for it), through the activation ring (192),
    from global memory (K-split), and in the decode kernel (M = 8)."""
    import torch
    d.set_option(d.OPT_TOKEN_TILE, token_tile)
    d.set_option(d.OPT_SPLIT_ALL, split_all)
    N, K, dtype = 384, 1024, "bf16"
    p = I.make_problem(M, N, K, dtype, "u4b8", seed=M + token_tile)
    rng = np.random.default_rng(M)
    C_bits = I.f32_to_bits(rng.standard_normal((M, N)).astype(np.float32), dtype)
    bias_bits = I.f32_to_bits(rng.standard_normal(N).astype(np.float32), dtype)
    blob = gpu_prepack(d, p)
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    Y = d.mm(to_cuda16(p.X_bits, dtype), blob, N, out=out, alpha=0.75, C=to_cuda16(C_bits, dtype), beta=-0.5,
             bias=to_cuda16(bias_bits, dtype))
    clean(d, "epilogue %s" % ((M, token_tile, split_all),))
    ref = O.epilogue(O.mm_problem(p), dtype, 0.75, C_bits, -0.5, bias_bits)
    assert_parity(y_as_f64(Y, dtype), ref, "epilogue")


@pytest.mark.parametrize("qtype,G,M_list", [("u4b8", 128, [40, 0, 150, 7]), ("u4_fzp", 64, [64, 9, 0]),
                                            ("u4_zp", 128, [8, 3, 16])])
def test_grouped(d, qtype, G, M_list):
    """Host pointer arrays: the tcgen05 GEMM, and the decode kernel when every M is small."""
    Ns = [256, 128, 384, 256][:len(M_list)]
    Ks = [1024, 512, 768, 512][:len(M_list)]
    probs = [I.make_problem(m, n, k, "bf16", qtype, seed=70 + i, group_size=G)
             for i, (m, n, k) in enumerate(zip(M_list, Ns, Ks))]
    blobs = [gpu_prepack(d, p) for p in probs]
    outs = d.grouped_mm([to_cuda16(p.X_bits, "bf16") for p in probs], blobs, Ns, qtype=qtype, group_size=G)
    clean(d, "grouped %s" % (M_list,))
    for p, Y in zip(probs, outs):
        if p.M:
            assert_parity(y_as_f64(Y, "bf16"), O.mm_problem(p), "grouped M=%d" % p.M)


def test_grouped_device_m(d):
    import torch
    M_true, caps = [30, 0, 77], [64, 16, 128]
    Ns, Ks = [256, 128, 384], [512, 1024, 512]
    probs = [I.make_problem(c, n, k, "bf16", "u4b8", seed=80 + i) for i, (c, n, k) in enumerate(zip(caps, Ns, Ks))]
    blobs = [gpu_prepack(d, p) for p in probs]
    M_dev = torch.tensor(M_true, dtype=torch.int32, device="cuda")
    outs = d.grouped_mm_device_m([to_cuda16(p.X_bits, "bf16") for p in probs], blobs, M_dev, Ns)
    clean(d, "device m")
    for p, m, Y in zip(probs, M_true, outs):
        if m:
            assert_parity(y_as_f64(Y[:m], "bf16"), O.mm_problem(p)[:m], "device m M=%d" % m)


def test_grouped_dev_ptrs(d):
    from tests.test_gpu_dev_ptrs import Case
    c = Case(d, [33, 0, 5, 120, 64, 1], [(256, 512), (128, 1024)], seed=11)
    c.run()
    clean(d, "device pointers")
    c.check("device pointers")
