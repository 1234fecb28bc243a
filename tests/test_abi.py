"""The C-ABI library builds, loads and exports every function include/wq4.h declares, and its
argument checks (after "machete_mainloop.cuh", can_implement) reject bad calls before any
CUDA work — these run without a GPU."""
import ctypes

import pytest

import weight_only_quantized_wq4_gb300 as wq4


@pytest.fixture(scope="module")
def clib():
    wq4.build()
    return wq4.load_library()


def test_exports_every_declared_symbol(clib):
    names = wq4.header_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(clib, n), n


def test_status_strings(clib):
    for code in (0, -1, -2, -3, -4, -5, -6, -7):
        assert clib.wq4_status_string(code) != b"unknown status", code
    assert clib.wq4_version() >= 100


def test_unprepack_argument_rules(clib):
    """wq4_unprepack rejects bad calls before any CUDA work."""
    up = clib.wq4_unprepack
    assert up(None, 128, 128, 128, 0, 0, A16b, A16c, None, None) == wq4.ERR_INVALID       # no blob
    assert up(A16, 128, 128, 128, 0, 0, None, A16c, None, None) == wq4.ERR_INVALID        # no code output
    assert up(A16, 128, 128, 128, 0, 0, A16b, A16c, A16c, None) == wq4.ERR_INVALID        # zeros for u4b8
    assert up(A16, 128, 128, 128, 0, 1, A16b, A16c, None, None) == wq4.ERR_INVALID        # zp without zeros
    assert up(A16, 128, 128, 128, 0, 3, A16b, A16c, None, None) == wq4.ERR_INVALID        # no such qtype
    assert up(A16, 100, 128, 128, 0, 0, A16b, A16c, None, None) == wq4.ERR_UNSUPPORTED    # N not a multiple of 128
    assert up(A16, 128, 256, 384, 0, 0, A16b, A16c, None, None) == wq4.ERR_UNSUPPORTED    # G does not divide K
    assert up(MIS, 128, 128, 128, 0, 0, A16b, A16c, None, None) == wq4.ERR_ALIGN
    assert up(A16, 128, 128, 128, 0, 0, MIS, A16c, None, None) == wq4.ERR_ALIGN
    assert up(A16, 128, 128, 128, 0, 0, A16b, MIS, None, None) == wq4.ERR_ALIGN
    assert up(A16, 128, 128, 128, 0, 1, A16b, A16c, MIS, None) == wq4.ERR_ALIGN


def test_every_declared_status_has_its_own_text(clib):
    """Each WQ4_ERR_* code include/wq4.h declares maps to a text of its own, and the binding's
    constants agree with the header."""
    import re
    with open(wq4.HEADER) as f:
        codes = {n: int(v) for n, v in re.findall(r"\b(WQ4_(?:OK|ERR_[A-Z]+))\s*=\s*(-?\d+)", f.read())}
    assert len(codes) >= 8
    texts = {clib.wq4_status_string(v) for v in codes.values()}
    assert len(texts) == len(codes) and b"unknown status" not in texts
    for name, v in codes.items():
        assert getattr(wq4, name[len("WQ4_"):]) == v, name


def test_every_declared_option_matches_the_binding(clib):
    """Each WQ4_OPT_* key include/wq4.h declares has the binding's value and reads back as set."""
    import re
    with open(wq4.HEADER) as f:
        keys = {n: int(v) for n, v in re.findall(r"\b(WQ4_OPT_[A-Z_]+)\s*=\s*(\d+)", f.read())}
    assert len(keys) >= 14
    for name, v in keys.items():
        assert getattr(wq4, name[len("WQ4_"):]) == v, name
    assert clib.wq4_set_option(keys["WQ4_OPT_TOKEN_TILE"], 64) == wq4.OK
    assert clib.wq4_get_option(keys["WQ4_OPT_TOKEN_TILE"]) == 64
    assert clib.wq4_set_option(keys["WQ4_OPT_TOKEN_TILE"], 0) == wq4.OK


def test_release_library_has_no_bounds_checks(clib):
    assert clib.wq4_debug_checks() == 0
    rec = (ctypes.c_int * 4)(7, 7, 7, 7)
    assert clib.wq4_last_violation(rec) == 0 and list(rec) == [0, 0, 0, 0]
    assert clib.wq4_last_violation(None) == wq4.ERR_INVALID


def test_debug_library_builds_and_exports(clib):
    """libwq4_debug.so: the same sources with the kernels' bounds checks compiled in."""
    path = wq4.build(debug=True)
    assert path == wq4.DEBUG_LIB_PATH
    dlib = ctypes.CDLL(path)
    for n in wq4.header_functions():
        assert hasattr(dlib, n), n
    assert dlib.wq4_debug_checks() == 1


def test_binding_swaps_to_the_debug_library(clib):
    """use_library routes the binding's calls through the debug build; restore_library undoes it."""
    wq4.build(debug=True)
    assert not wq4.debug_checks()
    old = wq4.use_library(wq4.DEBUG_LIB_PATH)
    try:
        assert wq4.debug_checks()
        assert wq4.last_violation() is None
        assert wq4.prepacked_bytes(4096, 4096) == 256 + 32 * 32 * 8448     # the same ABI through it
    finally:
        wq4.restore_library(old)
    assert not wq4.debug_checks()
    with pytest.raises(RuntimeError):
        wq4.use_library(wq4.DEBUG_LIB_PATH + ".missing")
    assert wq4.load_library() is old                                      # a failed swap keeps the old one


def test_prepacked_bytes(clib):
    assert clib.wq4_prepacked_bytes(4096, 4096, 128, 0) == 256 + 32 * 32 * 8448
    assert clib.wq4_prepacked_bytes(14336, 4096, 128, 1) == 256 + 112 * 32 * 8576
    assert clib.wq4_prepacked_bytes(100, 4096, 128, 0) == 0       # N not a multiple of 128
    assert clib.wq4_prepacked_bytes(128, 4096, 64, 0) == 256 + 32 * 8 * 1088   # G = 64: two scale sets
    assert clib.wq4_prepacked_bytes(128, 4096, 64, 1) == 256 + 32 * 8 * 1104
    assert clib.wq4_prepacked_bytes(128, 4096, 64, 2) == 256 + 32 * 8 * 1152
    assert clib.wq4_prepacked_bytes(128, 4096, 32, 0) == 0        # group size 32 not built
    assert clib.wq4_prepacked_bytes(128, 1024, 384, 0) == 0       # 384 does not divide K
    assert clib.wq4_prepacked_bytes(128, 1024, 256, 0) == 256 + 8 * 8448   # one record per 128 K
    assert clib.wq4_prepacked_bytes(128, 640, 640, 1) == 256 + 5 * 8576    # channel-wise (G = K)
    assert clib.wq4_prepacked_bytes(256, 512, 128, 2) == 256 + 2 * 4 * 8704  # float zeros: 1088-byte blocks
    assert clib.wq4_prepacked_bytes(128, 128, 128, 3) == 0                   # no such qtype


A16 = ctypes.c_void_p(0x10000)     # 16-byte aligned fake device addresses (never dereferenced)
A16b = ctypes.c_void_p(0x20000)
A16c = ctypes.c_void_p(0x30000)
MIS = ctypes.c_void_p(0x10008)


def _mm(clib, X=A16, W=A16b, Y=A16c, M=8, N=128, K=128, G=128, dt=0, qt=0):
    return clib.wq4_mm(X, W, Y, M, N, K, G, dt, qt, None, 0, None)


def test_mm_argument_rules(clib):
    assert _mm(clib, M=-1) == wq4.ERR_INVALID
    assert _mm(clib, N=0) == wq4.ERR_INVALID
    assert _mm(clib, N=100) == wq4.ERR_UNSUPPORTED
    assert _mm(clib, K=200) == wq4.ERR_UNSUPPORTED
    assert _mm(clib, G=0) == wq4.ERR_INVALID                      # group size must be non-zero
    assert _mm(clib, G=32) == wq4.ERR_UNSUPPORTED                 # neither 64 nor a multiple of 128
    assert _mm(clib, dt=7) == wq4.ERR_INVALID
    assert _mm(clib, qt=9) == wq4.ERR_INVALID
    assert _mm(clib, X=None) == wq4.ERR_INVALID
    assert _mm(clib, W=None) == wq4.ERR_INVALID
    assert _mm(clib, X=MIS) == wq4.ERR_ALIGN                      # 128-bit alignment for TMA
    assert _mm(clib, Y=MIS) == wq4.ERR_ALIGN
    assert _mm(clib, M=0, X=None, W=None, Y=None) == wq4.OK       # empty problem: nothing to do


def test_prepack_argument_rules(clib):
    pp = clib.wq4_prepack
    assert pp(A16, A16b, None, 128, 128, 128, 0, 0, A16c, None) != wq4.ERR_INVALID   # valid (fails later, no GPU)
    assert pp(A16, A16b, A16c, 128, 128, 128, 0, 0, A16c, None) == wq4.ERR_INVALID   # zeros given in u4b8 mode
    assert pp(A16, A16b, None, 128, 128, 128, 0, 1, A16c, None) == wq4.ERR_INVALID   # zeros missing in zp mode
    assert pp(A16, None, None, 128, 128, 128, 0, 0, A16c, None) != wq4.ERR_INVALID   # no scales: direct conversion
    assert pp(A16, None, A16c, 128, 128, 128, 0, 1, A16c, None) == wq4.ERR_INVALID   # zero points need scales
    assert pp(A16, A16b, None, 128, 256, 256, 0, 0, A16c, None) != wq4.ERR_UNSUPPORTED  # G = 256 divides K
    assert pp(A16, A16b, None, 128, 256, 384, 0, 0, A16c, None) == wq4.ERR_UNSUPPORTED  # G does not divide K
    assert pp(A16, A16b, None, 128, 256, 32, 0, 0, A16c, None) == wq4.ERR_UNSUPPORTED   # G neither 64 nor a multiple of 128
    assert pp(A16, A16b, None, 128, 256, 64, 0, 0, A16c, None) != wq4.ERR_UNSUPPORTED   # G = 64
    assert pp(MIS, A16b, None, 128, 128, 128, 0, 0, A16c, None) == wq4.ERR_ALIGN
    assert pp(A16, A16b, MIS, 128, 128, 128, 0, 1, A16c, None) == wq4.ERR_ALIGN
    assert pp(A16, MIS, None, 128, 128, 128, 0, 0, A16c, None) == wq4.ERR_ALIGN      # scales ("can_implement")
    assert pp(A16, A16b, None, 128, 128, 128, 0, 0, MIS, None) == wq4.ERR_ALIGN      # the blob
    assert pp(A16, A16b, MIS, 128, 128, 128, 0, 2, A16c, None) == wq4.ERR_ALIGN      # float zeros
    assert pp(A16, A16b, A16c, 128, 128, 128, 0, 2, A16c, None) != wq4.ERR_INVALID   # float zeros with scales
    assert pp(A16, A16b, None, 128, 128, 128, 0, 2, A16c, None) == wq4.ERR_INVALID   # float zeros missing
    assert pp(A16, None, A16c, 128, 128, 128, 0, 2, A16c, None) == wq4.ERR_INVALID   # float zeros need scales


def test_mm_ex_argument_rules(clib):
    ex = clib.wq4_mm_ex
    assert ex(A16, A16b, A16c, 8, 128, 128, 128, 0, 0, 1.0, None, 0.5, None, None, 0, None) == wq4.ERR_INVALID  # beta needs C
    assert ex(A16, A16b, A16c, 8, 128, 128, 128, 0, 0, 1.0, MIS, 0.5, None, None, 0, None) == wq4.ERR_ALIGN
    assert ex(A16, A16b, A16c, 8, 128, 128, 128, 0, 0, 1.0, None, 0.0, MIS, None, 0, None) == wq4.ERR_ALIGN
    assert ex(A16, A16b, A16c, 8, 128, 128, 32, 0, 0, 1.0, None, 0.0, None, None, 0, None) == wq4.ERR_UNSUPPORTED
    assert ex(A16, A16b, A16c, 0, 128, 128, 128, 0, 0, 1.0, None, 0.0, None, None, 0, None) == wq4.OK  # M = 0


def test_grouped_argument_rules(clib):
    arr = ctypes.c_int * 2
    ptrs = ctypes.c_void_p * 2
    g = clib.wq4_grouped_mm
    X, W, Y = ptrs(A16, A16), ptrs(A16b, A16b), ptrs(A16c, A16c)
    assert g(0, arr(8, 8), arr(128, 128), arr(128, 128), X, W, Y, 128, 0, 0, None, 0, None) == wq4.ERR_INVALID
    assert g(65, arr(8, 8), arr(128, 128), arr(128, 128), X, W, Y, 128, 0, 0, None, 0, None) == wq4.ERR_UNSUPPORTED
    assert g(2, arr(8, -1), arr(128, 128), arr(128, 128), X, W, Y, 128, 0, 0, None, 0, None) == wq4.ERR_INVALID
    assert g(2, arr(8, 8), arr(128, 96), arr(128, 128), X, W, Y, 128, 0, 0, None, 0, None) == wq4.ERR_UNSUPPORTED
    Xbad = ptrs(A16, MIS)
    assert g(2, arr(8, 8), arr(128, 128), arr(128, 128), Xbad, W, Y, 128, 0, 0, None, 0, None) == wq4.ERR_ALIGN
    # an empty problem's pointers are never looked at
    Xnull = ptrs(A16, None)
    rc = g(2, arr(8, 0), arr(128, 128), arr(128, 128), Xnull, W, ptrs(A16c, None), 128, 0, 0, None, 0, None)
    assert rc not in (wq4.ERR_INVALID, wq4.ERR_ALIGN)


def test_device_m_argument_rules(clib):
    """wq4_grouped_mm_device_m rejects bad calls before any CUDA work."""
    arr = ctypes.c_int * 2
    ptrs = ctypes.c_void_p * 2
    d = clib.wq4_grouped_mm_device_m
    nb = ctypes.c_size_t(0)
    assert clib.wq4_grouped_device_m_workspace_bytes(2, ctypes.byref(nb)) == wq4.OK and nb.value > 0
    ws, wsn = ctypes.c_void_p(0x40000), nb.value
    X, W, Y = ptrs(A16, A16), ptrs(A16b, A16b), ptrs(A16c, A16c)
    Mdev = ctypes.c_void_p(0x50000)

    def call(P=2, M_dev=Mdev, cap=(8, 8), N=(128, 128), K=(128, 128), X=X, qtype=0, ws=ws, wsn=wsn):
        return d(P, M_dev, arr(*cap), arr(*N), arr(*K), X, W, Y, 128, 0, qtype, ws, wsn, None)

    assert call(qtype=2) == wq4.ERR_UNSUPPORTED                 # float zeros need host-known shapes
    assert call(P=0) == wq4.ERR_INVALID
    assert call(M_dev=None) == wq4.ERR_INVALID
    assert call(P=65) == wq4.ERR_UNSUPPORTED
    assert call(M_dev=ctypes.c_void_p(0x50002)) == wq4.ERR_ALIGN   # int counts: 4-byte aligned
    assert call(ws=None) == wq4.ERR_WORKSPACE
    assert call(wsn=16) == wq4.ERR_WORKSPACE
    assert call(ws=ctypes.c_void_p(0x40008)) == wq4.ERR_ALIGN
    assert call(cap=(8, -1)) == wq4.ERR_INVALID
    assert call(N=(128, 96)) == wq4.ERR_UNSUPPORTED
    assert call(X=ptrs(A16, MIS)) == wq4.ERR_ALIGN


def test_workspace_query_argument_rules(clib):
    """The workspace queries and the static-scratch call reject bad arguments before they look at
    the device."""
    nb = ctypes.c_size_t(0)
    out = ctypes.byref(nb)
    arr = ctypes.c_int * 2
    assert clib.wq4_workspace_bytes(8, 128, 128, 128, None) == wq4.ERR_INVALID
    assert clib.wq4_workspace_bytes(-1, 128, 128, 128, out) == wq4.ERR_INVALID
    assert clib.wq4_workspace_bytes(8, 100, 128, 128, out) == wq4.ERR_UNSUPPORTED
    assert clib.wq4_workspace_bytes(8, 128, 256, 384, out) == wq4.ERR_UNSUPPORTED     # G does not divide K
    assert clib.wq4_workspace_bytes(8, 128, 128, 0, out) == wq4.ERR_INVALID
    assert clib.wq4_workspace_bytes_ex(8, 128, 128, 128, 3, out) == wq4.ERR_INVALID   # no such qtype
    g = clib.wq4_grouped_workspace_bytes
    assert g(0, arr(8, 8), arr(128, 128), arr(128, 128), 128, out) == wq4.ERR_INVALID
    assert g(65, arr(8, 8), arr(128, 128), arr(128, 128), 128, out) == wq4.ERR_INVALID
    assert g(2, arr(8, -2), arr(128, 128), arr(128, 128), 128, out) == wq4.ERR_INVALID
    assert g(2, arr(8, 8), arr(128, 128), arr(128, 200), 128, out) == wq4.ERR_UNSUPPORTED
    assert clib.wq4_grouped_workspace_bytes_ex(2, arr(8, 8), arr(128, 128), arr(128, 128), 128, 7, out) == wq4.ERR_INVALID
    dp = clib.wq4_grouped_dev_ptrs_workspace_bytes
    assert dp(0, arr(8, 8), arr(128, 128), arr(128, 128), 128, out) == wq4.ERR_INVALID
    big = ctypes.c_int * 4097
    assert dp(4097, big(), big(*([128] * 4097)), big(*([128] * 4097)), 128, out) == wq4.ERR_UNSUPPORTED
    assert dp(2, arr(8, 8), arr(128, 128), arr(128, 128), 128, None) == wq4.ERR_INVALID
    st = clib.wq4_mm_static_scratch
    assert st(A16, A16b, A16c, 8, 128, 128, 128, 2, 0, None) == wq4.ERR_INVALID          # no such dtype
    assert st(A16, A16b, A16c, 8, 128, 128, 0, 0, 0, None) == wq4.ERR_INVALID            # group size 0


def test_dev_ptrs_argument_rules(clib):
    """Host-side checks of wq4_grouped_mm_dev_ptrs: every one answers before any device work."""
    g = clib.wq4_grouped_mm_dev_ptrs

    def call(P=2, M=(8, 8), N=(128, 128), K=(128, 128), X=A16, W=A16b, Y=A16c, G=128, qt=0):
        arr = ctypes.c_int * len(M)
        return g(P, arr(*M), arr(*N), arr(*K), X, W, Y, G, 0, qt, None, 0, None)

    assert call(P=0) == wq4.ERR_INVALID
    assert call(P=4097, M=(8,) * 4097, N=(128,) * 4097, K=(128,) * 4097) == wq4.ERR_UNSUPPORTED
    assert call(M=(8, -1)) == wq4.ERR_INVALID
    assert call(N=(128, 96)) == wq4.ERR_UNSUPPORTED
    assert call(K=(128, 384), G=256) == wq4.ERR_UNSUPPORTED
    assert call(qt=2) == wq4.ERR_UNSUPPORTED                          # float zeros: single problems
    assert call(X=None) == wq4.ERR_INVALID
    assert call(Y=ctypes.c_void_p(0x10004)) == wq4.ERR_ALIGN           # pointer arrays: 8-byte aligned
    rc = call(P=5, M=(1, 9, 300, 2, 0), N=(128,) * 5, K=(128, 256, 384, 512, 640))   # shapes all differ
    assert rc not in (wq4.ERR_INVALID, wq4.ERR_ALIGN, wq4.ERR_UNSUPPORTED)


def test_options(clib):
    assert clib.wq4_set_option(1, 64) == wq4.OK
    assert clib.wq4_get_option(1) == 64
    assert clib.wq4_set_option(1, 48) == wq4.ERR_INVALID
    assert clib.wq4_set_option(1, 160) == wq4.OK
    assert clib.wq4_set_option(1, 0) == wq4.OK
    assert clib.wq4_set_option(wq4.OPT_PDL, 1) == wq4.ERR_INVALID
    assert clib.wq4_set_option(wq4.OPT_PDL, -1) == wq4.OK
    assert clib.wq4_get_option(wq4.OPT_PDL) == -1
    assert clib.wq4_set_option(wq4.OPT_PDL, 0) == wq4.OK
    assert clib.wq4_set_option(wq4.OPT_TEST_STALL, 2) == wq4.ERR_INVALID
    assert clib.wq4_set_option(wq4.OPT_TEST_STALL, 0) == wq4.OK
    assert clib.wq4_set_option(wq4.OPT_CONST_WEIGHTS, 2) == wq4.ERR_INVALID
    assert clib.wq4_set_option(wq4.OPT_CONST_WEIGHTS, 1) == wq4.OK
    assert clib.wq4_get_option(wq4.OPT_CONST_WEIGHTS) == 1
    assert clib.wq4_set_option(wq4.OPT_CONST_WEIGHTS, 0) == wq4.OK
    assert clib.wq4_set_option(wq4.OPT_DECODE_DEPTH, 1) == wq4.ERR_INVALID
    assert clib.wq4_set_option(wq4.OPT_DECODE_DEPTH, 17) == wq4.ERR_INVALID
    assert clib.wq4_set_option(wq4.OPT_DECODE_DEPTH, 4) == wq4.OK
    assert clib.wq4_set_option(wq4.OPT_DECODE_DEPTH, 0) == wq4.OK
    assert clib.wq4_set_option(wq4.OPT_DECODE_TRIGGER, 2) == wq4.ERR_INVALID
    assert clib.wq4_set_option(wq4.OPT_DECODE_TRIGGER, 0) == wq4.OK
    assert clib.wq4_set_option(wq4.OPT_VERIFY_DEV_PTRS, 2) == wq4.ERR_INVALID
    assert clib.wq4_set_option(wq4.OPT_VERIFY_DEV_PTRS, 0) == wq4.OK
    assert clib.wq4_set_option(99, 1) == wq4.ERR_INVALID
    assert clib.wq4_get_option(99) == -1
