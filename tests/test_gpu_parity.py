"""GPU path vs the CPU oracle through the C ABI: prepack bit-exact, GEMM within
|Y - Y_ref| <= 1e-2 + 1e-2 |Y_ref| (fp32 accumulation, output rounded to bf16/fp16 once)."""
import ctypes

import numpy as np
import pytest

import oracle as O
import wq4_inputs as I
from tests.wq4_testutil import (assert_parity, from_cuda16, from_cuda32, gpu_mm, gpu_prepack, to_cuda16, to_cuda32,
                                y_as_f64)

pytestmark = pytest.mark.gpu


@pytest.fixture
def opts(lib):
    """Options set inside a test are reset afterwards."""
    yield lib
    for key in (lib.OPT_TOKEN_TILE, lib.OPT_GRID, lib.OPT_SPLIT_ALL, lib.OPT_A_IN_SMEM, lib.OPT_TIMEOUT_CYCLES,
                lib.OPT_CLUSTER, lib.OPT_DECODE, lib.OPT_PDL, lib.OPT_TEST_STALL, lib.OPT_CONST_WEIGHTS,
                lib.OPT_DECODE_DEPTH, lib.OPT_DECODE_TRIGGER):
        lib.set_option(key, 0)


# ------------------------------------------------------------------------------ prepack
PREPACK_SHAPES = [(128, 128, "bf16", "u4b8"), (256, 512, "fp16", "u4b8"), (384, 256, "bf16", "u4_zp"),
                  (512, 640, "fp16", "u4_zp"), (384, 256, "bf16", "u4_fzp"), (512, 640, "fp16", "u4_fzp"),
                  (4096, 4096, "bf16", "u4b8"), (14336, 4096, "bf16", "u4_zp"), (4096, 4096, "bf16", "u4_fzp")]


@pytest.mark.parametrize("N,K,dtype,qtype", PREPACK_SHAPES)
def test_prepack_bit_exact(lib, N, K, dtype, qtype):
    p = I.make_problem(1, N, K, dtype, qtype, seed=N + K)
    blob = gpu_prepack(lib, p).cpu().numpy()
    ref = O.prepack(p.Wq, p.S_bits, N, K, dtype, qtype, p.Z)
    assert blob.shape == ref.shape
    assert np.array_equal(blob, ref)


@pytest.mark.parametrize("N,K,dtype,qtype", PREPACK_SHAPES[:6])
def test_unprepack_round_trip(lib, N, K, dtype, qtype):
    p = I.make_problem(1, N, K, dtype, qtype, seed=3 * N + K)
    Wq, S, Z = lib.unprepack(gpu_prepack(lib, p), N, K, dtype, qtype)
    assert np.array_equal(from_cuda32(Wq), p.Wq)
    assert np.array_equal(from_cuda16(S), p.S_bits)
    if qtype == "u4_zp":
        assert np.array_equal(from_cuda32(Z), p.Z)
    elif qtype == "u4_fzp":
        assert np.array_equal(from_cuda16(Z), p.Z)
    else:
        assert Z is None


# ------------------------------------------------------------------------------ GEMM
SMALL = [
    (1, 128, 128, "bf16", "u4b8"),
    (8, 256, 512, "bf16", "u4b8"),
    (16, 256, 512, "fp16", "u4b8"),
    (17, 384, 640, "bf16", "u4_zp"),
    (33, 128, 256, "fp16", "u4_zp"),
    (64, 256, 384, "bf16", "u4b8"),
    (65, 384, 256, "bf16", "u4b8"),
    (128, 256, 512, "bf16", "u4_zp"),
    (129, 128, 384, "fp16", "u4b8"),
    (300, 512, 1024, "bf16", "u4b8"),
    (777, 256, 256, "bf16", "u4_zp"),
]


# group sizes other than 128 (a multiple of 128 dividing K; G = K is channel-wise) and weights
# without scales (uint4b8 direct conversion)
GROUP_MODES = [
    (256, 512, "bf16", "u4_zp", 256, True), (384, 640, "fp16", "u4b8", 640, True),
    (256, 384, "bf16", "u4b8", 128, False), (128, 1024, "fp16", "u4b8", 512, False),
    (256, 1024, "bf16", "u4_fzp", 512, True), (256, 512, "bf16", "u4b8", 64, True), (384, 640, "fp16", "u4_zp", 64, True),
    (256, 384, "bf16", "u4_fzp", 64, True), (128, 256, "fp16", "u4b8", 64, False),
]


@pytest.mark.parametrize("N,K,dtype,qtype,G,scaled", GROUP_MODES)
def test_prepack_group_sizes_bit_exact(lib, N, K, dtype, qtype, G, scaled):
    p = I.make_problem(1, N, K, dtype, qtype, seed=N + K + G, group_size=G, scaled=scaled)
    blob = gpu_prepack(lib, p)
    assert np.array_equal(blob.cpu().numpy(), O.prepack(p.Wq, p.S_bits, N, K, dtype, qtype, p.Z, group_size=G))
    Wq, S, Z = lib.unprepack(blob, N, K, dtype, qtype, group_size=G)
    assert np.array_equal(from_cuda32(Wq), p.Wq)
    if scaled:
        assert np.array_equal(from_cuda16(S), p.S_bits)
    if qtype == "u4_zp":
        assert np.array_equal(from_cuda32(Z), p.Z)
    if qtype == "u4_fzp":
        assert np.array_equal(from_cuda16(Z), p.Z)


GROUP_MM = [
    (40, 256, 1024, "bf16", "u4_zp", 256, True), (200, 384, 512, "fp16", "u4b8", 512, True),
    (64, 256, 768, "bf16", "u4b8", 128, False), (130, 256, 2048, "bf16", "u4b8", 2048, True),
    (8, 512, 1024, "bf16", "u4_zp", 512, True), (5, 256, 640, "fp16", "u4b8", 128, False),
    (6, 256, 1024, "bf16", "u4_fzp", 512, True), (150, 384, 1024, "fp16", "u4_fzp", 1024, True),
    (8, 4096, 4096, "bf16", "u4b8", 64, True), (5, 2944, 8960, "bf16", "u4_zp", 64, True),
    (16, 768, 1408, "fp16", "u4_fzp", 64, True), (100, 1024, 2048, "bf16", "u4b8", 64, True),
    (300, 384, 512, "fp16", "u4_zp", 64, True), (777, 256, 1024, "bf16", "u4_fzp", 64, True),
    (129, 512, 768, "bf16", "u4b8", 64, False), (500, 384, 1024, "bf16", "u4_zp", 64, True),
    (1000, 256, 512, "fp16", "u4b8", 64, True), (384, 512, 640, "bf16", "u4_fzp", 64, True),
]


@pytest.mark.parametrize("M,N,K,dtype,qtype,G,scaled", GROUP_MM)
def test_mm_group_sizes(lib, M, N, K, dtype, qtype, G, scaled):
    """Both kernels (M <= 32 takes the decode kernel) on every mode."""
    p = I.make_problem(M, N, K, dtype, qtype, seed=M + N + G, group_size=G, scaled=scaled)
    assert_parity(y_as_f64(gpu_mm(lib, p), dtype), O.mm_problem(p), "G=%d scaled=%s" % (G, scaled))


@pytest.mark.parametrize("M,N,K,dtype,qtype", SMALL)
def test_mm_small(lib, M, N, K, dtype, qtype):
    p = I.make_problem(M, N, K, dtype, qtype, seed=M * 7 + N + K)
    Y = gpu_mm(lib, p)
    assert_parity(y_as_f64(Y, dtype), O.mm_problem(p), str((M, N, K, dtype, qtype)))


@pytest.mark.parametrize("token_tile", [16, 64, 128, 160, 192])
@pytest.mark.parametrize("grid", [0, 3, 7])
@pytest.mark.parametrize("split_all", [0, 1])
def test_mm_schedules(opts, token_tile, grid, split_all):
    """Every token tile with whole tiles, K-split tiles and tiles split over 2+ CTAs."""
    lib = opts
    lib.set_option(lib.OPT_TOKEN_TILE, token_tile)
    lib.set_option(lib.OPT_GRID, grid)
    lib.set_option(lib.OPT_SPLIT_ALL, split_all)
    p = I.make_problem(250, 384, 1280, "bf16", "u4_zp", seed=token_tile + grid)
    Y = gpu_mm(lib, p)
    assert_parity(y_as_f64(Y, "bf16"), O.mm_problem(p), "tile %d grid %d split %d" % (token_tile, grid, split_all))


@pytest.mark.parametrize("token_tile", [16, 64, 128, 160, 192])
@pytest.mark.parametrize("cluster", [2, 3, 4, 8])
def test_mm_cluster_split(opts, token_tile, cluster):
    """Each tile's K range split over a cluster; partials added through distributed shared memory."""
    lib = opts
    lib.set_option(lib.OPT_TOKEN_TILE, token_tile)
    lib.set_option(lib.OPT_CLUSTER, cluster)
    p = I.make_problem(100, 256, 1152, "bf16", "u4b8", seed=cluster * 100 + token_tile)
    assert_parity(y_as_f64(gpu_mm(lib, p), "bf16"), O.mm_problem(p), "cluster %d tile %d" % (cluster, token_tile))


@pytest.mark.parametrize("token_tile", [16, 64, 128, 160, 192])
def test_mm_long_k(opts, token_tile):
    """64 groups per tile: the operand buffers (2, 3 or 4 of them, by token tile) and both MMA
    issuers cycle through many phases; two m-tiles, one of them ragged."""
    lib = opts
    lib.set_option(lib.OPT_TOKEN_TILE, token_tile)
    p = I.make_problem(token_tile + 37, 256, 8192, "bf16", "u4b8", seed=token_tile * 3 + 1)
    assert_parity(y_as_f64(gpu_mm(lib, p), "bf16"), O.mm_problem(p), "long K, tile %d" % token_tile)


@pytest.mark.parametrize("M,qtype", [(8, "u4b8"), (200, "u4_zp"), (64, "u4_fzp")])
def test_mm_longest_k(lib, M, qtype):
    """K = 65536 (512 groups) on the tensor-core path. One or two tiles on 152 SMs, so the planner
    splits K (over a cluster, or through the workspace) into long group ranges. With float zeros
    there are 8 zero steps per tile."""
    p = I.make_problem(M, 128, 65536, "bf16", qtype, seed=M + 65536)
    assert_parity(y_as_f64(gpu_mm(lib, p), "bf16"), O.mm_problem(p), "K = 65536, M = %d" % M)


DECODE = [
    (1, 128, 128, "bf16", "u4b8"), (5, 256, 384, "fp16", "u4_zp"), (8, 4096, 4096, "bf16", "u4b8"),
    (8, 384, 8960, "bf16", "u4_zp"), (9, 512, 1024, "bf16", "u4b8"), (16, 1024, 2048, "fp16", "u4b8"),
    (17, 256, 640, "bf16", "u4_zp"), (24, 128, 1024, "fp16", "u4b8"), (32, 2048, 2048, "bf16", "u4_zp"),
    (3, 14336, 512, "bf16", "u4b8"),
    # 17..32 tokens whose activations do not fit at once: two launches of at most 16 rows
    (24, 512, 4096, "bf16", "u4b8"), (32, 384, 2560, "fp16", "u4_zp"), (17, 256, 4096, "bf16", "u4_zp"),
    # three row blocks per CTA (one warp idle), long K at 8 tokens
    (7, 7296, 3840, "fp16", "u4_zp"), (2, 6144, 1024, "fp16", "u4b8"), (8, 256, 8960, "bf16", "u4b8"),
    (8, 4096, 6144, "bf16", "u4_zp"),
]


@pytest.mark.parametrize("const", [0, 1])
@pytest.mark.parametrize("M,N,K,dtype,qtype", DECODE)
def test_decode_kernel(opts, M, N, K, dtype, qtype, const):
    """The warp-level-MMA kernel for at most 32 tokens (forced on), in stream order and with
    constant weights (weights copied before the kernel ahead completes)."""
    lib = opts
    lib.set_option(lib.OPT_DECODE, 1)
    lib.set_option(lib.OPT_CONST_WEIGHTS, const)
    p = I.make_problem(M, N, K, dtype, qtype, seed=M * 13 + N + K)
    assert_parity(y_as_f64(gpu_mm(lib, p), dtype), O.mm_problem(p), "decode %s" % ((M, N, K, dtype, qtype),))


@pytest.mark.parametrize("M,K", [(1, 12288), (8, 12288), (8, 12416), (16, 6144), (16, 6272), (32, 6144), (32, 6272)])
def test_decode_at_its_largest_k(lib, M, K):
    """Decode-sized M at the largest K whose activations fit in the decode kernel's shared memory at
    once: 12288 up to 8 tokens and 6144 up to 16, with 17..32 tokens as two 16-row launches at
    6144. Also one 128-K group beyond it, where the call takes the tensor-core GEMM instead."""
    dtype, qtype = ("bf16" if M % 2 == 0 else "fp16"), ("u4_zp" if K % 256 else "u4b8")
    p = I.make_problem(M, 256, K, dtype, qtype, seed=M + K)
    assert_parity(y_as_f64(gpu_mm(lib, p), dtype), O.mm_problem(p), "largest K %s" % ((M, K),))


@pytest.mark.parametrize("depth,trigger,const", [(2, 0, 0), (3, 1, 0), (2, 0, 1), (5, 0, 1), (16, 1, 1), (0, 0, 1)])
@pytest.mark.parametrize("M,N,K,qtype", [(8, 4096, 4096, "u4b8"), (5, 2944, 8960, "u4_zp"), (16, 768, 1408, "u4b8"),
                                         (7, 4864, 4096, "u4_zp"), (12, 2432, 8192, "u4b8"), (3, 11264, 2048, "u4b8")])
def test_decode_ring_and_modes(opts, depth, trigger, const, M, N, K, qtype):
    """The decode kernel's weight ring (forced depths, so the ring wraps many times; K not a
    multiple of 8 groups leaves a short last stage), the two trigger points and the constant-weights
    mode (header check and first weight copies before the wait on the kernel ahead); depth 0 is the
    automatic ring, and N = 11264 gives a CTA 4 or 5 blocks."""
    lib = opts
    lib.set_option(lib.OPT_DECODE, 1)
    lib.set_option(lib.OPT_DECODE_DEPTH, depth)
    lib.set_option(lib.OPT_DECODE_TRIGGER, trigger)
    lib.set_option(lib.OPT_CONST_WEIGHTS, const)
    p = I.make_problem(M, N, K, "bf16", qtype, seed=M + N + K + depth)
    assert_parity(y_as_f64(gpu_mm(lib, p), "bf16"), O.mm_problem(p), "decode ring %s" % ((depth, trigger, const),))
    assert lib.get_last_error() == lib.OK


def _mismatched_calls(lib, p, blob, X):
    """Calls whose arguments disagree with the blob's header (nothing else wrong)."""
    yield "qtype", dict(qtype="u4_zp" if p.qtype == "u4b8" else "u4b8")
    yield "group size", dict(qtype=p.qtype, group_size=p.K)
    yield "N", dict(qtype=p.qtype, N=p.N // 2)


@pytest.mark.parametrize("M,const", [(8, 0), (8, 1), (100, 0), (300, 0)])
def test_blob_header_mismatch_is_reported(opts, M, const):
    """A blob passed with a qtype, group size or N other than the ones it was prepacked with: the
    kernels compare the blob's header with the call before they read any record, record
    WQ4_ERR_INVALID and stop; the next correct call is fine. Decode (M = 8, stream order and
    constant weights), cluster split (M = 100) and data-parallel (M = 300) paths."""
    import torch
    lib = opts
    lib.set_option(lib.OPT_CONST_WEIGHTS, const)
    p = I.make_problem(M, 1024, 1024, "bf16", "u4b8", seed=M + 17)
    blob = gpu_prepack(lib, p)
    X = to_cuda16(p.X_bits, "bf16")
    torch.cuda.synchronize()
    for what, kw in _mismatched_calls(lib, p, blob, X):
        N = kw.get("N", p.N)
        Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
        lib.mm(X, blob, N, qtype=kw["qtype"], out=Y, group_size=kw.get("group_size", 128))
        assert lib.get_last_error() == lib.ERR_INVALID, what
        assert lib.get_last_error() == lib.OK
    assert_parity(y_as_f64(lib.mm(X, blob, p.N), "bf16"), O.mm_problem(p), "after a header mismatch")


@pytest.mark.parametrize("M,N,K", [(8, 4096, 4096), (100, 256, 1152), (300, 512, 1024)])
def test_header_check_paths_agree(opts, M, N, K):
    """A blob written by wq4_prepack for these arguments is streamed while its header is checked; a
    copy of it made by other means (here a tensor clone) is checked before any record is read. Both
    paths give the same bits, on the decode, cluster-split and data-parallel plans."""
    lib = opts
    p = I.make_problem(M, N, K, "bf16", "u4_zp", seed=M + N)
    blob = gpu_prepack(lib, p)
    copy = blob.clone()
    X = to_cuda16(p.X_bits, "bf16")
    for const in (0, 1):
        lib.set_option(lib.OPT_CONST_WEIGHTS, const)
        a = from_cuda16(lib.mm(X, blob, N, qtype="u4_zp"))
        b = from_cuda16(lib.mm(X, copy, N, qtype="u4_zp"))
        assert np.array_equal(a, b)
        assert lib.get_last_error() == lib.OK
    assert_parity(O.decode16(a, "bf16"), O.mm_problem(p), "header check paths")


def test_decode_const_weights_chain_matches_stream_order(opts):
    """With constant weights the decode kernel reads the blob before the kernel ahead completes;
    in a graph of calls where each call's activations are the previous call's output, the result
    must equal plain stream order bit for bit."""
    import torch
    lib = opts
    M, K = 8, 4096
    ps = [I.make_problem(M, K, K, "bf16", "u4b8", seed=950 + i) for i in range(6)]
    blobs = [gpu_prepack(lib, p) for p in ps]
    X0 = to_cuda16(ps[0].X_bits, "bf16")
    torch.cuda.synchronize()

    def chain(const, pdl):
        lib.set_option(lib.OPT_CONST_WEIGHTS, const)
        lib.set_option(lib.OPT_PDL, pdl)
        st = torch.cuda.Stream()
        outs = [torch.empty((M, K), dtype=torch.bfloat16, device="cuda") for _ in ps]
        with torch.cuda.stream(st):
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=st):
                x = X0
                for i in range(len(ps)):
                    lib.mm(x, blobs[i], K, qtype="u4b8", out=outs[i])
                    x = outs[i]
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize()
        assert lib.get_last_error() == lib.OK
        return [from_cuda16(o) for o in outs]

    a = chain(1, 0)
    b = chain(0, -1)
    for i in range(len(ps)):
        assert np.array_equal(a[i], b[i]), "call %d differs with constant weights" % i
    assert_parity(O.decode16(a[0], "bf16"), O.mm_problem(ps[0]), "const-weights chain call 0")


def test_decode_chain_in_a_graph(opts):
    """Programmatic dependent launch on the decode kernel: a graph of calls, each call's activations
    the previous call's output (N = K). The same bits as plain stream order, and the first call
    matches the oracle."""
    import torch
    lib = opts
    M, K = 8, 4096
    ps = [I.make_problem(M, K, K, "bf16", "u4b8", seed=900 + i) for i in range(6)]
    blobs = [gpu_prepack(lib, p) for p in ps]
    X0 = to_cuda16(ps[0].X_bits, "bf16")
    torch.cuda.synchronize()

    def chain(pdl):
        lib.set_option(lib.OPT_PDL, pdl)
        st = torch.cuda.Stream()
        outs = [torch.empty((M, K), dtype=torch.bfloat16, device="cuda") for _ in ps]
        with torch.cuda.stream(st):
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=st):
                x = X0
                for i in range(len(ps)):
                    lib.mm(x, blobs[i], K, qtype="u4b8", out=outs[i])
                    x = outs[i]
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize()
        assert lib.get_last_error() == lib.OK
        return [from_cuda16(o) for o in outs]

    a = chain(0)
    b = chain(-1)
    for i in range(len(ps)):
        assert np.array_equal(a[i], b[i]), "call %d differs with programmatic launch" % i
    assert_parity(O.decode16(a[0], "bf16"), O.mm_problem(ps[0]), "decode chain call 0")


@pytest.mark.parametrize("M,N,K,mode", [(128, 14336, 1024, "whole"), (300, 512, 2048, "split"),
                                         (40, 512, 1024, "cluster"), (200, 1024, 512, "grouped")])
def test_gemm_const_weights(opts, M, N, K, mode):
    """With the constant-weights promise the GEMM copies weight records before the kernel ahead
    completes; activations produced by a kernel right before the call still keep stream order."""
    import torch
    lib = opts
    lib.set_option(lib.OPT_CONST_WEIGHTS, 1)
    if mode == "split":
        lib.set_option(lib.OPT_SPLIT_ALL, 1)
        lib.set_option(lib.OPT_GRID, 9)
    elif mode == "cluster":
        lib.set_option(lib.OPT_CLUSTER, 4)
    probs = ([I.make_problem(M, N, K, "bf16", "u4_zp", seed=M + K)] if mode != "grouped" else
             I.make_grouped(M, 3, N, K, "bf16", "u4b8", seed=M, M_list=[M - 70, 0, 70]))
    blobs = [gpu_prepack(lib, p) for p in probs]
    torch.cuda.synchronize()
    for rep in range(3):
        # the activations are written on the stream just before each call
        Xs = [to_cuda16(p.X_bits, "bf16") if p.M else to_cuda16(np.zeros((0, p.K), np.uint16), "bf16") for p in probs]
        Xs = [(x.float() * 1.0).to(torch.bfloat16) for x in Xs]
        if mode == "grouped":
            outs = lib.grouped_mm(Xs, blobs, [p.N for p in probs], qtype="u4b8")
        else:
            outs = [lib.mm(Xs[0], blobs[0], N, qtype="u4_zp")]
        for p, Y in zip(probs, outs):
            if p.M:
                assert_parity(y_as_f64(Y, "bf16"), O.mm_problem(p), "const weights %s rep %d" % (mode, rep))
    assert lib.get_last_error() == lib.OK


def test_decode_kernel_deterministic(opts):
    lib = opts
    lib.set_option(lib.OPT_DECODE, 1)
    p = I.make_problem(8, 2048, 4096, "bf16", "u4b8", seed=99)
    blob = gpu_prepack(lib, p)
    a = from_cuda16(gpu_mm(lib, p, blob))
    b = from_cuda16(gpu_mm(lib, p, blob))
    assert np.array_equal(a, b)
    lib.set_option(lib.OPT_PDL, -1)                                   # plain stream order: same bits
    c = from_cuda16(gpu_mm(lib, p, blob))
    assert np.array_equal(a, c)


def test_decode_after_prepack_same_stream(opts):
    """prepack and the decode call back to back on one stream (no synchronisation between them):
    the decode kernel may start early under programmatic launch but reads the weights only after
    the prepack kernel has finished."""
    import torch
    lib = opts
    lib.set_option(lib.OPT_DECODE, 1)
    p = I.make_problem(8, 4096, 4096, "bf16", "u4b8", seed=7)
    ref = O.mm_problem(p)
    for _ in range(3):
        Wq, S, X = to_cuda32(p.Wq), to_cuda16(p.S_bits, "bf16"), to_cuda16(p.X_bits, "bf16")
        torch.cuda.synchronize()
        blob = lib.prepack(Wq, S, None, qtype="u4b8")
        y = lib.mm(X, blob, p.N, qtype="u4b8")
        assert_parity(y_as_f64(y, "bf16"), ref, "decode right after prepack")


@pytest.mark.parametrize("M,split_all", [(128, 0), (500, 0), (500, 1)])
def test_gemm_back_to_back_in_a_graph(opts, M, split_all):
    """Programmatic dependent launch: a graph of GEMM calls where each call's activations are the
    previous call's output (Y_i feeds X_{i+1}, N = K) and one weight is prepacked inside the
    graph right before its use. The result must equal the same chain run with plain stream order."""
    import torch
    lib = opts
    K = 1024
    ps = [I.make_problem(M, K, K, "bf16", "u4b8", seed=700 + i) for i in range(4)]
    Wq = [to_cuda32(p.Wq) for p in ps]
    S = [to_cuda16(p.S_bits, "bf16") for p in ps]
    blobs = [gpu_prepack(lib, p) for p in ps[:3]]
    X0 = to_cuda16(ps[0].X_bits, "bf16")

    lib.set_option(lib.OPT_SPLIT_ALL, split_all)   # 1: every tile split, counters reused call to call

    def chain(pdl):
        lib.set_option(lib.OPT_PDL, pdl)
        st = torch.cuda.Stream()
        outs = [torch.empty((M, K), dtype=torch.bfloat16, device="cuda") for _ in range(4)]
        blob3 = torch.empty(lib.prepacked_bytes(K, K), dtype=torch.uint8, device="cuda")
        ws = lib.alloc_workspace(max(lib.workspace_bytes(M, K, K), 16))
        clib = lib.load_library()
        with torch.cuda.stream(st):
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=st):
                x = X0
                for i in range(4):
                    if i == 3:   # prepack the last weight inside the graph, right before its use
                        assert clib.wq4_prepack(ctypes.c_void_p(Wq[3].data_ptr()), ctypes.c_void_p(S[3].data_ptr()),
                                                None, K, K, 128, 0, 0, ctypes.c_void_p(blob3.data_ptr()),
                                                ctypes.c_void_p(st.cuda_stream)) == lib.OK
                    lib.mm(x, blobs[i] if i < 3 else blob3, K, qtype="u4b8", workspace=ws, out=outs[i])
                    x = outs[i]
            for _ in range(3):
                g.replay()
            torch.cuda.synchronize()
        assert lib.get_last_error() == lib.OK
        return [from_cuda16(o) for o in outs]

    a = chain(0)
    b = chain(-1)
    for i in range(4):
        assert np.array_equal(a[i], b[i]), "call %d differs with programmatic launch" % i
    # and the first call of the chain matches the oracle
    assert_parity(O.decode16(a[0], "bf16"), O.mm_problem(ps[0]), "chain call 0")


@pytest.mark.parametrize("M,N,K,split_all", [(100, 256, 1152, 0), (200, 14336, 256, 0), (200, 14336, 256, 1),
                                           (8, 512, 1024, 0), (24, 256, 512, 0), (4, 14336, 4096, 0)])
def test_wait_timeout_reports_status_and_recovers(opts, M, N, K, split_all):
    """Failure detection without a fault: each CTA waits once on a barrier that nothing arrives on
    (WQ4_OPT_TEST_STALL) under a short bound (2e5 cycles, ~0.1 ms); the wait runs out, the CTA
    stops, lets its copies and MMAs finish, frees its tensor memory and exits. The host reads
    WQ4_ERR_TIMEOUT, the status word is cleared, and the next call (normal bound, fresh
    workspace) is correct. Cluster (M=100), data-parallel, K-split and decode shapes (one and six
    row blocks per CTA)."""
    import torch
    lib = opts
    p = I.make_problem(M, N, K, "bf16", "u4b8", seed=M + N + K)
    blob = gpu_prepack(lib, p)
    X = to_cuda16(p.X_bits, "bf16")
    torch.cuda.synchronize()
    lib.set_option(lib.OPT_SPLIT_ALL, split_all)
    lib.set_option(lib.OPT_TIMEOUT_CYCLES, 200000)
    lib.set_option(lib.OPT_TEST_STALL, 1)
    try:
        lib.mm(X, blob, p.N)
        status = lib.get_last_error()
    finally:
        lib.set_option(lib.OPT_TEST_STALL, 0)
        lib.set_option(lib.OPT_TIMEOUT_CYCLES, 0)
    assert status == lib.ERR_TIMEOUT
    assert lib.get_last_error() == lib.OK
    assert_parity(y_as_f64(lib.mm(X, blob, p.N), "bf16"), O.mm_problem(p), "after a timeout")


@pytest.mark.parametrize("M,N,K,dtype,split_all,in_place", [
    (200, 14336, 256, "bf16", 0, False), (200, 14336, 256, "bf16", 1, False), (100, 256, 1152, "fp16", 0, False),
    (8, 512, 1024, "bf16", 0, False), (24, 256, 512, "fp16", 0, True), (300, 384, 512, "bf16", 0, True),
    (28, 256, 4096, "fp16", 0, True), (6, 14336, 4096, "bf16", 0, True),
    # one whole tile per CTA (C through the activation stage after the last group), in place
    (128, 14336, 1024, "bf16", 0, True),
    # 192-token tiles (C through its own buffer) and K-split tiles (C from global memory)
    (1000, 8192, 512, "fp16", 0, False), (256, 14336, 512, "bf16", 0, False)])
def test_mm_epilogue(opts, M, N, K, dtype, split_all, in_place):
    """Y = alpha acc + beta C + bias on the data-parallel, K-split, cluster and decode paths, and
    in place (C is Y)."""
    import torch
    lib = opts
    lib.set_option(lib.OPT_SPLIT_ALL, split_all)
    p = I.make_problem(M, N, K, dtype, "u4_zp", seed=M * 3 + N + K)
    rng = np.random.default_rng(M + N)
    C_bits = I.f32_to_bits(rng.standard_normal((M, N)).astype(np.float32), dtype)
    bias_bits = I.f32_to_bits(rng.standard_normal(N).astype(np.float32), dtype)
    alpha, beta = 0.5, -1.25
    blob = gpu_prepack(lib, p)
    X = to_cuda16(p.X_bits, dtype)
    C = to_cuda16(C_bits, dtype)
    bias = to_cuda16(bias_bits, dtype)
    out = C if in_place else torch.empty((M, N), dtype=C.dtype, device="cuda")
    Y = lib.mm(X, blob, N, qtype="u4_zp", out=out, alpha=alpha, C=C, beta=beta, bias=bias)
    ref = O.epilogue(O.mm_problem(p), dtype, alpha, C_bits, beta, bias_bits)
    assert_parity(y_as_f64(Y, dtype), ref, "epilogue %s" % ((M, N, K, split_all, in_place),))


@pytest.mark.parametrize("token_tile,split_all,cluster,qtype", [
    (16, 0, 0, "u4b8"), (64, 1, 0, "u4_zp"), (128, 0, 0, "u4b8"), (64, 0, 4, "u4_fzp"), (16, 1, 0, "u4_fzp"),
    (128, 1, 0, "u4_zp"), (160, 0, 0, "u4b8"), (192, 0, 0, "u4_zp"), (192, 1, 0, "u4b8"), (192, 0, 2, "u4b8"),
    (128, 0, 0, "u4_fzp"), (192, 0, 0, "u4_fzp"), (160, 1, 0, "u4_fzp")])
def test_mm_group_64_schedules(opts, token_tile, split_all, cluster, qtype):
    """G = 64 (two scale sets per record, a partial per 64-K half, MMA warp h issuing half h of
    every group): every token tile, K-split and cluster plans."""
    lib = opts
    lib.set_option(lib.OPT_TOKEN_TILE, token_tile)
    lib.set_option(lib.OPT_SPLIT_ALL, split_all)
    lib.set_option(lib.OPT_CLUSTER, cluster)
    p = I.make_problem(150, 512, 2048, "bf16", qtype, seed=token_tile + 3 * split_all + cluster, group_size=64)
    assert_parity(y_as_f64(gpu_mm(lib, p), "bf16"), O.mm_problem(p), "G=64 %s" % ((token_tile, split_all, cluster),))


# ------------------------------------------------------------------------------ float zeros
FZP_MM = [(1, 128, 128, "bf16"), (8, 4096, 4096, "bf16"), (5, 2944, 8960, "bf16"), (16, 768, 1408, "fp16"),
          (33, 256, 512, "fp16"), (100, 1024, 2048, "bf16"), (300, 384, 512, "fp16"), (128, 14336, 4096, "bf16"),
          (777, 256, 1024, "bf16")]


@pytest.mark.parametrize("M,N,K,dtype", FZP_MM)
def test_mm_float_zeros(lib, M, N, K, dtype):
    """value = q s + zf (zero added after the scale) on both kernels: decode sizes (activation
    sums from an all-ones MMA) and the tensor-core path (activation sums from a pre-pass)."""
    p = I.make_problem(M, N, K, dtype, "u4_fzp", seed=M + 2 * N + K)
    assert_parity(y_as_f64(gpu_mm(lib, p), dtype), O.mm_problem(p), "float zeros %s" % ((M, N, K, dtype),))


@pytest.mark.parametrize("token_tile,split_all,cluster", [(128, 1, 0), (192, 0, 0), (64, 0, 4), (16, 0, 0),
                                                          (160, 1, 0)])
def test_mm_float_zeros_schedules(opts, token_tile, split_all, cluster):
    """Each CTA adds the zero term of its own groups: K-split, cluster and whole-tile plans."""
    lib = opts
    lib.set_option(lib.OPT_TOKEN_TILE, token_tile)
    lib.set_option(lib.OPT_SPLIT_ALL, split_all)
    lib.set_option(lib.OPT_CLUSTER, cluster)
    p = I.make_problem(150, 512, 2048, "bf16", "u4_fzp", seed=token_tile + split_all + cluster)
    assert_parity(y_as_f64(gpu_mm(lib, p), "bf16"), O.mm_problem(p), "schedule %s" % ((token_tile, split_all, cluster),))


@pytest.mark.parametrize("M,N", [(6, 384), (200, 384), (128, 14336)])
def test_mm_float_zeros_epilogue(opts, M, N):
    lib = opts
    K, dtype = 1024, "fp16"
    p = I.make_problem(M, N, K, dtype, "u4_fzp", seed=M + 5)
    rng = np.random.default_rng(M)
    C_bits = I.f32_to_bits(rng.standard_normal((M, N)).astype(np.float32), dtype)
    bias_bits = I.f32_to_bits(rng.standard_normal(N).astype(np.float32), dtype)
    Y = lib.mm(to_cuda16(p.X_bits, dtype), gpu_prepack(lib, p), N, qtype="u4_fzp", alpha=0.5,
               C=to_cuda16(C_bits, dtype), beta=-1.25, bias=to_cuda16(bias_bits, dtype))
    ref = O.epilogue(O.mm_problem(p), dtype, 0.5, C_bits, -1.25, bias_bits)
    assert_parity(y_as_f64(Y, dtype), ref, "float zeros epilogue M=%d" % M)


def test_float_zeros_contract(lib):
    """The activation-sum tables are in the workspace query of the tensor-core path only (a table
    per non-empty problem in the grouped query); device-resident shapes refuse the mode; a
    float-zero blob read as another qtype is reported."""
    import torch
    assert lib.workspace_bytes(8, 4096, 4096, qtype="u4_fzp") == 0
    # at least 300 rows (M rounded up to the token tile) x 2 x 64 padded zero groups x 2 bytes
    assert lib.workspace_bytes(300, 512, 1024, qtype="u4_fzp") >= 300 * 2 * 64 * 2
    assert lib.workspace_bytes(300, 512, 1024, qtype="u4_fzp") > lib.workspace_bytes(300, 512, 1024)
    Ms, Ns, Ks = [30, 0, 34], [256, 256, 256], [512, 512, 512]
    assert (lib.grouped_workspace_bytes(Ms, Ns, Ks, qtype="u4_fzp")
            >= lib.grouped_workspace_bytes(Ms, Ns, Ks) + 2 * 64 * 2 * 64 * 2)
    probs = I.make_grouped(64, 2, 256, 512, "bf16", "u4_fzp", seed=4, M_list=[30, 34])
    Xs = [to_cuda16(q.X_bits, "bf16") for q in probs]
    with pytest.raises(lib.Wq4Error) as e:
        lib.grouped_mm_device_m(Xs, [gpu_prepack(lib, q) for q in probs],
                                torch.tensor([30, 34], dtype=torch.int32, device="cuda"), [256, 256], qtype="u4_fzp")
    assert e.value.status == lib.ERR_UNSUPPORTED
    p = I.make_problem(40, 256, 512, "bf16", "u4_fzp", seed=41)
    blob = gpu_prepack(lib, p)
    lib.mm(to_cuda16(p.X_bits, "bf16"), blob, p.N, qtype="u4_zp")
    assert lib.get_last_error() == lib.ERR_INVALID
    assert_parity(y_as_f64(gpu_mm(lib, p, blob=blob), "bf16"), O.mm_problem(p), "after the mismatch")


@pytest.mark.parametrize("qtype,dtype", [("u4b8", "bf16"), ("u4_zp", "fp16")])
def test_grouped_device_resident_counts(lib, qtype, dtype):
    """Token counts in device memory, written by a kernel right before the call: clamped to the
    capacity, zero-count problems skipped, rows past each count untouched."""
    import torch
    caps = [64, 16, 256, 160, 128, 40]
    Ns = [256, 384, 256, 128, 256, 128]
    Ks = [512, 1024, 512, 768, 512, 256]
    want = [37, 0, 256, 129, 5, 999]                   # 999 > capacity 40: clamped
    probs = [I.make_problem(c, n, k, dtype, qtype, seed=300 + i) for i, (c, n, k) in enumerate(zip(caps, Ns, Ks))]
    Xs = [to_cuda16(p.X_bits, dtype) for p in probs]
    blobs = [gpu_prepack(lib, p) for p in probs]
    outs = [torch.full((c, n), float("nan"), dtype=Xs[0].dtype, device="cuda") for c, n in zip(caps, Ns)]
    for o in outs:
        o.view(torch.int16).fill_(0x7E01)
    M_host = torch.tensor(want, dtype=torch.int32)
    M_dev = M_host.cuda() * 1 - 0                       # produced by kernels on the stream
    lib.grouped_mm_device_m(Xs, blobs, M_dev, Ns, qtype=qtype, outs=outs)
    assert lib.get_last_error() == lib.OK
    for p, o, c, w in zip(probs, outs, caps, want):
        m = max(0, min(w, c))
        got = from_cuda16(o)
        if m:
            ref = O.mm_problem(p, rows=range(m))
            assert_parity(O.decode16(got[:m], dtype), ref, "device counts, M=%d" % m)
        assert np.all(got[m:] == 0x7E01), "rows past the count were written"


def test_mm_cluster_larger_than_groups(opts):
    """A cluster never gets more CTAs than the tile has groups (here K = 256: two groups)."""
    lib = opts
    lib.set_option(lib.OPT_CLUSTER, 8)
    p = I.make_problem(12, 384, 256, "fp16", "u4_zp", seed=4)
    assert_parity(y_as_f64(gpu_mm(lib, p), "fp16"), O.mm_problem(p), "cluster capped")


def test_grouped_cluster_split(opts):
    lib = opts
    lib.set_option(lib.OPT_CLUSTER, 4)
    probs = I.make_grouped(30, 3, 256, 768, "bf16", "u4_zp", seed=21, M_list=[7, 0, 23])
    outs = _grouped(lib, probs, "u4_zp")
    for p, Y in zip(probs, outs):
        if p.M:
            assert_parity(y_as_f64(Y, "bf16"), O.mm_problem(p), "grouped cluster M=%d" % p.M)


@pytest.mark.parametrize("token_tile", [16, 128, 160, 192])
def test_mm_a_operand_in_smem(opts, token_tile):
    lib = opts
    lib.set_option(lib.OPT_A_IN_SMEM, 1)
    lib.set_option(lib.OPT_TOKEN_TILE, token_tile)
    p = I.make_problem(40, 256, 512, "fp16", "u4b8", seed=5)
    assert_parity(y_as_f64(gpu_mm(lib, p), "fp16"), O.mm_problem(p), "A in smem")


def test_mm_deterministic(opts):
    lib = opts
    lib.set_option(lib.OPT_GRID, 5)
    lib.set_option(lib.OPT_SPLIT_ALL, 1)
    p = I.make_problem(24, 256, 2048, "bf16", "u4b8", seed=11)
    blob = gpu_prepack(lib, p)
    a = from_cuda16(gpu_mm(lib, p, blob))
    b = from_cuda16(gpu_mm(lib, p, blob))
    assert np.array_equal(a, b)


def test_mm_m0_is_noop(lib):
    import torch
    p = I.make_problem(0, 128, 128, "bf16", "u4b8", seed=1)
    blob = gpu_prepack(lib, p)
    X = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    Y = lib.mm(X, blob, 128)
    assert Y.shape == (0, 128)
    assert lib.get_last_error() == 0


def test_workspace_reuse_keeps_counters_zero(opts):
    """A K-split call leaves its arrival counters at zero, so the workspace can be reused."""
    lib = opts
    lib.set_option(lib.OPT_GRID, 6)
    p = I.make_problem(10, 256, 1024, "bf16", "u4b8", seed=12)
    blob = gpu_prepack(lib, p)
    ws = lib.alloc_workspace(lib.workspace_bytes(10, 256, 1024))
    for _ in range(3):
        Y = lib.mm(to_cuda16(p.X_bits, "bf16"), blob, 256, workspace=ws)
        assert_parity(y_as_f64(Y, "bf16"), O.mm_problem(p), "reuse")
    assert lib.get_last_error() == 0


# ------------------------------------------------------------------------------ grouped
def _grouped(lib, probs, qtype):
    blobs = [gpu_prepack(lib, p) for p in probs]
    Xs = [to_cuda16(p.X_bits, p.dtype) if p.M > 0 else to_cuda16(np.zeros((0, p.K), np.uint16), p.dtype)
          for p in probs]
    return lib.grouped_mm(Xs, blobs, [p.N for p in probs], qtype=qtype)


@pytest.mark.parametrize("M_list", [[0, 17, 0, 40], [5], [130, 1, 64, 0, 200], [0, 0, 33]])
def test_grouped_small(lib, M_list):
    probs = I.make_grouped(sum(M_list), len(M_list), 256, 384, "bf16", "u4b8", seed=len(M_list), M_list=M_list)
    outs = _grouped(lib, probs, "u4b8")
    for p, Y in zip(probs, outs):
        assert Y.shape == (p.M, p.N)
        if p.M:
            assert_parity(y_as_f64(Y, "bf16"), O.mm_problem(p), "grouped M=%d" % p.M)


@pytest.mark.parametrize("dtype,G,M_list", [("bf16", 128, [0, 17, 40, 0, 200]), ("fp16", 128, [5, 130, 64]),
                                             ("bf16", 64, [33, 0, 150, 8]), ("fp16", 512, [70, 1, 0])])
def test_grouped_float_zeros(lib, dtype, G, M_list):
    """Float zeros in the grouped call: every problem's zero steps read its own sums table."""
    Ks = [1024, 512, 2048, 1024, 512][:len(M_list)]
    Ns = [256, 384, 128, 256, 128][:len(M_list)]
    probs = [I.make_problem(m, n, k, dtype, "u4_fzp", seed=60 + i, group_size=G)
             for i, (m, n, k) in enumerate(zip(M_list, Ns, Ks))]
    blobs = [gpu_prepack(lib, p) for p in probs]
    Xs = [to_cuda16(p.X_bits, dtype) for p in probs]
    outs = lib.grouped_mm(Xs, blobs, Ns, qtype="u4_fzp", group_size=G)
    assert lib.get_last_error() == lib.OK
    for p, Y in zip(probs, outs):
        if p.M:
            assert_parity(y_as_f64(Y, dtype), O.mm_problem(p), "grouped float zeros %s" % ((p.M, p.N, p.K, G),))


def test_trace_names_each_path(opts, capfd):
    """WQ4_OPT_TRACE = 1: each call prints its plan on stderr, one line per path; 0: nothing."""
    lib = opts
    try:
        lib.set_option(lib.OPT_TRACE, 1)
        p = I.make_problem(8, 256, 512, "bf16", "u4b8", seed=1)
        gpu_mm(lib, p)
        lib.set_option(lib.OPT_TOKEN_TILE, 128)
        q = I.make_problem(200, 256, 512, "bf16", "u4b8", seed=2)
        gpu_mm(lib, q)
        lib.set_option(lib.OPT_TOKEN_TILE, 0)
        probs = I.make_grouped(20, 2, 256, 512, "bf16", "u4b8", seed=3, M_list=[12, 8])
        lib.grouped_mm([to_cuda16(r.X_bits, "bf16") for r in probs], [gpu_prepack(lib, r) for r in probs], [256, 256])
        assert lib.get_last_error() == lib.OK
        err = capfd.readouterr().err
        assert "[wq4] decode kernel: M=8" in err, err
        assert "[wq4] problems=1 token_tile=128" in err, err
        assert "[wq4] grouped decode kernel: problems=2" in err, err
        lib.set_option(lib.OPT_TRACE, 0)
        gpu_mm(lib, p)
        assert lib.get_last_error() == lib.OK
        assert "[wq4]" not in capfd.readouterr().err
    finally:
        lib.set_option(lib.OPT_TRACE, 0)


def test_grouped_calls_with_every_problem_empty(lib):
    """Every problem with M = 0: host pointer arrays (with and without float zeros), device-resident
    counts that are all zero, and device pointer arrays. Each call reports OK and leaves its
    outputs untouched."""
    import torch
    from tests.test_gpu_dev_ptrs import SENTINEL, Case
    Ns, Ks = [256, 128, 384], [512, 1024, 256]
    for qtype in ("u4_zp", "u4_fzp"):
        probs = [I.make_problem(4, n, k, "bf16", qtype, seed=90 + i) for i, (n, k) in enumerate(zip(Ns, Ks))]
        blobs = [gpu_prepack(lib, p) for p in probs]
        Xs = [to_cuda16(p.X_bits, "bf16") for p in probs]
        outs = lib.grouped_mm([x[:0] for x in Xs], blobs, Ns, qtype=qtype)
        assert lib.get_last_error() == lib.OK
        assert all(o.shape[0] == 0 for o in outs)
    Ys = [torch.full((4, n), SENTINEL, dtype=torch.int16, device="cuda") for n in Ns]
    probs = [I.make_problem(4, n, k, "bf16", "u4b8", seed=95 + i) for i, (n, k) in enumerate(zip(Ns, Ks))]
    M_dev = torch.zeros(3, dtype=torch.int32, device="cuda")
    lib.grouped_mm_device_m([to_cuda16(p.X_bits, "bf16") for p in probs], [gpu_prepack(lib, p) for p in probs], M_dev,
                            Ns, outs=[y.view(torch.bfloat16) for y in Ys])
    assert lib.get_last_error() == lib.OK
    assert all(bool((y == SENTINEL).all()) for y in Ys), "a zero-count problem was written"
    c = Case(lib, [0, 0, 0], [(256, 512), (128, 1024)], seed=12)
    c.run()
    assert lib.get_last_error() == lib.OK
    assert bool((c.Y == SENTINEL).all())


GROUPED_DECODE = [
    ("bf16", "u4b8", 128, [8, 8, 8, 8]),
    ("fp16", "u4_zp", 128, [1, 0, 16, 5, 0]),
    ("bf16", "u4_fzp", 128, [3, 32, 17]),
    ("bf16", "u4b8", 64, [12, 0, 7]),
    ("fp16", "u4_fzp", 64, [2, 9]),
    ("bf16", "u4_zp", 128, [24, 1]),
]


@pytest.mark.parametrize("dtype,qtype,G,M_list", GROUPED_DECODE)
def test_grouped_decode_kernel(opts, dtype, qtype, G, M_list):
    """Grouped calls whose problems all have at most 32 tokens take the decode kernel in one launch
    (no workspace); the same call with the decode kernel switched off takes the GEMM."""
    lib = opts
    Ns = [4096, 512, 1024, 384, 256, 640][:len(M_list)]
    Ks = [1024, 2048, 512, 1024, 768, 1536][:len(M_list)]
    probs = [I.make_problem(m, n, k, dtype, qtype, seed=80 + i, group_size=G)
             for i, (m, n, k) in enumerate(zip(M_list, Ns, Ks))]
    blobs = [gpu_prepack(lib, p) for p in probs]
    Xs = [to_cuda16(p.X_bits, dtype) for p in probs]
    assert lib.grouped_workspace_bytes(M_list, Ns, Ks, G, qtype) == 0
    for decode in (0, -1):
        lib.set_option(lib.OPT_DECODE, decode)
        outs = lib.grouped_mm(Xs, blobs, Ns, qtype=qtype, group_size=G)
        assert lib.get_last_error() == lib.OK
        for p, Y in zip(probs, outs):
            if p.M:
                assert_parity(y_as_f64(Y, dtype), O.mm_problem(p), "grouped decode=%d %s" % (decode, (p.M, p.N, p.K)))


def test_grouped_decode_many_problems(lib):
    """64 decode-sized problems in one launch, every CTA on blocks of its own problem."""
    rng = np.random.default_rng(64)
    M_list = [int(v) for v in rng.integers(0, 9, size=64)]
    probs = [I.make_problem(m, 256, 512, "bf16", "u4b8", seed=200 + i) for i, m in enumerate(M_list)]
    outs = _grouped(lib, probs, "u4b8")
    assert lib.get_last_error() == lib.OK
    for p, Y in zip(probs, outs):
        if p.M:
            assert_parity(y_as_f64(Y, "bf16"), O.mm_problem(p), "64 problems, M=%d" % p.M)


def test_grouped_mixed_shapes(lib):
    """Per-problem N and K differ."""
    shapes = [(9, 128, 256), (70, 384, 128), (0, 256, 512), (150, 256, 640)]
    probs = [I.make_problem(m, n, k, "fp16", "u4_zp", seed=i) for i, (m, n, k) in enumerate(shapes)]
    outs = _grouped(lib, probs, "u4_zp")
    for p, Y in zip(probs, outs):
        if p.M:
            assert_parity(y_as_f64(Y, "fp16"), O.mm_problem(p), "mixed %s" % ((p.M, p.N, p.K),))


# ------------------------------------------------------------------------------ workloads
@pytest.mark.slow
@pytest.mark.parametrize("name", ["tiny_m16_n256_k512_fp16_u4b8", "decode_m8_n4096_k4096_bf16_u4b8",
                                  "asym_m128_n14336_k4096_bf16_u4zp", "prefill_m4096_n4096_k14336_bf16_u4b8"])
def test_workload_full(lib, name):
    p = I.make_workload(name)
    Y = y_as_f64(gpu_mm(lib, p), p.dtype)
    st = assert_parity(Y, O.mm_problem(p), name)
    print(name, st)


@pytest.mark.slow
def test_grouped_workload_full(lib):
    probs = I.make_workload("grouped_8x_n14336_k4096_summ1024_bf16_u4b8")
    outs = _grouped(lib, probs, "u4b8")
    for i, (p, Y) in enumerate(zip(probs, outs)):
        assert_parity(y_as_f64(Y, "bf16"), O.mm_problem(p), "problem %d M=%d" % (i, p.M))
