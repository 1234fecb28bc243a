"""Grouped GEMM with its per-problem pointers in device memory (wq4_grouped_mm_dev_ptrs) against the
oracle, through the C ABI: the activation tensor maps the set-up kernel patches on the device
(byte for byte against the host encoder), parity for up to 4096 problems with empty ones and with
pointer arrays written by a kernel, problems that fail the device-side check, the K-split and
cluster plans, bit-identity with wq4_grouped_mm, and a captured graph replayed with new pointers.

The problems of a case share a few base problems ("sm90_gemm_array_tma_warpspecialized_cooperative.hpp":
the grouped call takes any pointer per problem, aliasing included): problem i uses base b's weight
blob and rows [r0, r0 + M_i) of base b's activations, so its reference is those rows of the
oracle's result for base b."""
import numpy as np
import pytest

import oracle as O
import wq4_inputs as I
from tests.wq4_testutil import assert_parity, from_cuda16, gpu_prepack, to_cuda16

pytestmark = pytest.mark.gpu

SENTINEL = 0x7E01      # a NaN pattern no GEMM result has


@pytest.fixture
def opts(lib):
    yield lib
    for key in (lib.OPT_VERIFY_DEV_PTRS, lib.OPT_GRID, lib.OPT_SPLIT_ALL, lib.OPT_CLUSTER, lib.OPT_TOKEN_TILE):
        lib.set_option(key, 0)


class Case:
    """P problems over a few base problems, their buffers on the device and the pointer arrays."""

    def __init__(self, lib, M_list, shapes, dtype="bf16", qtype="u4b8", seed=0, group_size=128, base_of=None):
        import torch
        rng = np.random.default_rng(seed)
        self.lib, self.dtype, self.qtype, self.G = lib, dtype, qtype, group_size
        rows = max(1, max(M_list))
        self.bases = [I.make_problem(rows, n, k, dtype, qtype, seed=seed * 31 + j, group_size=group_size)
                      for j, (n, k) in enumerate(shapes)]
        self.X = [to_cuda16(b.X_bits, dtype) for b in self.bases]
        self.W = [gpu_prepack(lib, b) for b in self.bases]
        self._refs = {}
        P = len(M_list)
        self.M = [int(m) for m in M_list]
        self.base = [int(v) for v in (base_of if base_of is not None else rng.integers(0, len(shapes), size=P))]
        self.N = [self.bases[b].N for b in self.base]
        self.K = [self.bases[b].K for b in self.base]
        self.r0 = [int(rng.integers(0, rows - m + 1)) for m in self.M]
        self.y_off = np.zeros(P, np.int64)
        off = 0
        for i in range(P):
            self.y_off[i] = off
            off += self.M[i] * self.N[i]
        self.Y = torch.empty(max(off, 8), dtype=torch.int16, device="cuda")
        self.Y.fill_(SENTINEL)
        # the pointer arrays are written by kernels on the stream: a gather of the bases' addresses
        # plus per-problem byte offsets
        self._xb = torch.tensor([x.data_ptr() for x in self.X], dtype=torch.int64, device="cuda")
        wb = torch.tensor([w.data_ptr() for w in self.W], dtype=torch.int64, device="cuda")
        self._idx = torch.tensor(self.base, dtype=torch.int64, device="cuda")
        self.W_ptrs = wb[self._idx]
        self.X_ptrs = torch.empty(P, dtype=torch.int64, device="cuda")
        self.set_rows(self.r0)
        self.Y_ptrs = torch.from_numpy(2 * self.y_off).cuda() + self.Y.data_ptr()

    def set_rows(self, r0):
        """Point problem i at rows [r0[i], r0[i] + M_i) of its base's activations (on the device)."""
        import torch
        self.r0 = [int(r) for r in r0]
        off = torch.from_numpy(np.array([2 * r * k for r, k in zip(self.r0, self.K)], np.int64)).cuda()
        self.X_ptrs.copy_(self._xb[self._idx] + off)

    def run(self, workspace=None):
        self.lib.grouped_mm_dev_ptrs(self.M, self.N, self.K, self.X_ptrs, self.W_ptrs, self.Y_ptrs, dtype=self.dtype,
                                     qtype=self.qtype, workspace=workspace, group_size=self.G)

    def out(self, i) -> np.ndarray:
        o, m, n = int(self.y_off[i]), self.M[i], self.N[i]
        return from_cuda16(self.Y[o:o + m * n].view(m, n) if m else self.Y[:0].view(0, n))

    def ref(self, i) -> np.ndarray:
        b = self.base[i]
        if b not in self._refs:
            self._refs[b] = O.mm_problem(self.bases[b])
        return self._refs[b][self.r0[i]:self.r0[i] + self.M[i]]

    def check(self, what, skip=()):
        for i in range(len(self.M)):
            if not self.M[i]:
                continue
            got = self.out(i)
            if i in skip:
                assert np.all(got == SENTINEL), "%s: problem %d was written" % (what, i)
            else:
                assert_parity(O.decode16(got, self.dtype), self.ref(i), "%s, problem %d (M=%d N=%d K=%d)" % (
                    what, i, self.M[i], self.N[i], self.K[i]))


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_patched_maps_match_host_encoder(opts, dtype):
    """The set-up kernel's maps (a template encoded on the host for the problem's rows and K, its
    address replaced on the device) equal the host encoder's maps for the same activations, byte
    for byte; the GEMM is not launched."""
    lib = opts
    rng = np.random.default_rng(7)
    M_list = [int(v) for v in rng.integers(0, 200, size=40)]
    M_list[3] = M_list[17] = 0
    M_list[5], M_list[9] = 1, 192
    # tensors just under and at 128 KiB (the encoder derives a flag from the total size)
    M_list[10:14] = [127, 128, 63, 64]
    c = Case(lib, M_list, [(128, 256), (256, 512), (128, 1024)], dtype=dtype, seed=1,
             base_of=[i % 3 for i in range(40)][:10] + [1, 1, 2, 2] + [i % 3 for i in range(26)])
    lib.set_option(lib.OPT_VERIFY_DEV_PTRS, 1)
    c.run()
    assert lib.get_last_error() == lib.OK
    assert bool((c.Y == SENTINEL).all()), "verification mode must not launch the GEMM"


@pytest.mark.parametrize("P,dtype,qtype", [(1, "bf16", "u4b8"), (128, "bf16", "u4b8"), (128, "fp16", "u4_zp"),
                                           (600, "bf16", "u4_zp")])
def test_dev_ptrs_parity(lib, P, dtype, qtype):
    """Empty problems among them (about a third); 600 problems take two set-up launches."""
    rng = np.random.default_rng(P)
    M_list = [int(v) if rng.random() > 0.33 else 0 for v in rng.integers(1, 70, size=P)]
    M_list[0] = max(M_list[0], 1)
    c = Case(lib, M_list, [(256, 512), (128, 256), (384, 768)], dtype=dtype, qtype=qtype, seed=P)
    c.run()
    assert lib.get_last_error() == lib.OK
    c.check("P=%d" % P)


def test_dev_ptrs_4096_problems(lib):
    rng = np.random.default_rng(4096)
    M_list = [int(v) for v in rng.integers(0, 5, size=4096)]
    c = Case(lib, M_list, [(128, 128), (128, 256), (256, 128), (128, 512)], seed=2)
    c.run()
    assert lib.get_last_error() == lib.OK
    c.check("P=4096")


@pytest.mark.parametrize("mode", ["split_all", "cluster", "token_tile_16", "wide"])
def test_dev_ptrs_schedules(opts, mode):
    lib = opts
    if mode == "split_all":
        lib.set_option(lib.OPT_SPLIT_ALL, 1)
        lib.set_option(lib.OPT_GRID, 7)
    elif mode == "cluster":
        lib.set_option(lib.OPT_CLUSTER, 4)
    elif mode == "token_tile_16":
        lib.set_option(lib.OPT_TOKEN_TILE, 16)
    M_list = [300, 0, 150, 7, 0, 64] if mode == "wide" else [9, 0, 30, 1, 0, 17]
    c = Case(lib, M_list, [(256, 1024), (128, 512)], dtype="fp16", qtype="u4_zp", seed=3)
    c.run()
    assert lib.get_last_error() == lib.OK
    c.check(mode)


def test_dev_ptrs_group_size(lib):
    c = Case(lib, [40, 0, 129, 3], [(256, 1024), (128, 512)], qtype="u4_zp", seed=5, group_size=256)
    c.run()
    assert lib.get_last_error() == lib.OK
    c.check("G=256")
    c = Case(lib, [40, 0, 300, 3], [(256, 512)], seed=6, group_size=64)
    c.run()
    assert lib.get_last_error() == lib.OK
    c.check("G=64")


def test_dev_ptrs_bit_identical_to_grouped_mm(lib):
    """At most 64 problems: the same plan and kernel as wq4_grouped_mm, the same bits."""
    import torch
    M_list = [33, 0, 5, 120, 64, 1, 0, 250]
    c = Case(lib, M_list, [(256, 512), (128, 1024)], seed=8, base_of=[0, 1, 0, 1, 1, 0, 0, 1])
    c.run()
    assert lib.get_last_error() == lib.OK
    Xs = [c.X[b][r:r + m] if m else c.X[b][:0] for b, r, m in zip(c.base, c.r0, c.M)]
    outs = lib.grouped_mm(Xs, [c.W[b] for b in c.base], c.N)
    for i, o in enumerate(outs):
        if c.M[i]:
            assert np.array_equal(from_cuda16(o), c.out(i)), "problem %d" % i
    torch.cuda.synchronize()


def test_dev_ptrs_bad_problems_are_skipped(lib):
    """A null activation pointer, a misaligned output pointer and a blob of another shape each
    make their own problem invalid; the others are computed; the call reports WQ4_ERR_INVALID."""
    M_list = [20, 31, 8, 50, 12]
    c = Case(lib, M_list, [(256, 512), (128, 512)], seed=9, base_of=[0, 0, 1, 1, 0])
    c.X_ptrs[1] = 0                                   # null X
    c.Y_ptrs[2] = c.Y_ptrs[2] + 8                     # misaligned Y
    c.W_ptrs[3] = c.W[0].data_ptr()                   # header says N = 256, the call N = 128
    c.run()
    assert lib.get_last_error() == lib.ERR_INVALID
    c.Y_ptrs[2] = c.Y_ptrs[2] - 8
    c.check("bad problems", skip=(1, 2, 3))
    assert lib.get_last_error() == lib.OK            # the status was cleared


def test_dev_ptrs_graph_replay_with_new_pointers(lib):
    """A captured call reads the pointer arrays at each replay: rewriting them between replays
    (same shapes) moves the work to other buffers."""
    import torch
    M_list = [17, 0, 40, 3]
    c = Case(lib, M_list, [(256, 512), (128, 512)], seed=10, base_of=[0, 1, 1, 0])
    ws = lib.alloc_workspace(lib.grouped_dev_ptrs_workspace_bytes(c.M, c.N, c.K))
    c.run(ws)                                          # first call outside the capture
    assert lib.get_last_error() == lib.OK
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            c.run(ws)
    torch.cuda.current_stream().wait_stream(s)
    c.Y.fill_(SENTINEL)
    g.replay()
    torch.cuda.synchronize()
    c.check("first replay")
    # other rows of the same bases and another output buffer
    c.set_rows([2, 0, 0, 9])
    Y2 = torch.full_like(c.Y, SENTINEL)
    c.Y_ptrs.copy_(torch.from_numpy(2 * c.y_off).cuda() + Y2.data_ptr())
    c.Y.fill_(SENTINEL)
    g.replay()
    torch.cuda.synchronize()
    assert bool((c.Y == SENTINEL).all()), "the old output buffer was written"
    c.Y = Y2
    c.check("second replay")
    assert lib.get_last_error() == lib.OK
