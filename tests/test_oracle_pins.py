"""Pins for the CPU oracle: each test checks it against something other than its own formulas.

* exact rational brute force, decoding bf16/fp16 bit patterns by the format definitions and
  reading nibbles as hexadecimal digits (a different route for every step);
* closed forms: one-hot codes, an identity weight, codes equal to their zero point;
* invariants: the per-group scale, uint4b8 == zero-point mode with z = 8, linearity in X;
* IEEE / bfloat16 bit patterns and the API's nibble order;
* the blob layout placed element by element versus the vectorised ``prepack``.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle as O
import wq4_inputs as I

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ---------------------------------------------------------------- independent decoders
def bf16_exact(bits: int) -> Fraction:
    """bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits."""
    sign = -1 if bits & 0x8000 else 1
    e, f = (bits >> 7) & 0xFF, bits & 0x7F
    assert e != 0xFF
    if e == 0:
        return sign * Fraction(f, 1 << 7) * Fraction(1, 1 << 126)
    return sign * (1 + Fraction(f, 1 << 7)) * (Fraction(2) ** (e - 127))


def fp16_exact(bits: int) -> Fraction:
    """IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits."""
    sign = -1 if bits & 0x8000 else 1
    e, f = (bits >> 10) & 0x1F, bits & 0x3FF
    assert e != 0x1F
    if e == 0:
        return sign * Fraction(f, 1 << 10) * Fraction(1, 1 << 14)
    return sign * (1 + Fraction(f, 1 << 10)) * (Fraction(2) ** (e - 15))


def exact16(bits: int, dtype: str) -> Fraction:
    return bf16_exact(bits) if dtype == "bf16" else fp16_exact(bits)


def nibble_hex(word: int, i: int) -> int:
    """Element i of a packed word read as the i-th hexadecimal digit from the right."""
    return int(("%08x" % int(word))[7 - i], 16)


def brute_force(p):
    """Y[m][n] as exact Fractions, one multiply-add at a time, and sum_k |term| per output."""
    G = p.group_size
    Y, A = [], []
    for m in range(p.M):
        row, arow = [], []
        for n in range(p.N):
            acc, aabs = Fraction(0), Fraction(0)
            for k in range(p.K):
                qv = nibble_hex(p.Wq[n, k // 8], k % 8)
                g = k // G
                sv = exact16(int(p.S_bits[g, n]), p.dtype) if p.S_bits is not None else Fraction(1)
                xv = exact16(int(p.X_bits[m, k]), p.dtype)
                if p.qtype == "u4_fzp":                     # code times scale, plus the float zero
                    wv = qv * sv + exact16(int(p.Z[g, n]), p.dtype)
                else:
                    zv = 8 if p.qtype == "u4b8" else nibble_hex(p.Z[g, n // 8], n % 8)
                    wv = (qv - zv) * sv
                acc += xv * wv
                aabs += abs(xv * wv)
            row.append(acc)
            arow.append(aabs)
        Y.append(row)
        A.append(arow)
    return Y, A


# ---------------------------------------------------------------- formats
def test_decode16_bit_patterns():
    bf = {0x3F80: 1.0, 0xBF80: -1.0, 0x4000: 2.0, 0x4300: 128.0, 0x3C00: 2.0 ** -7,
          0x0001: 2.0 ** -133, 0x7F7F: 3.3895313892515355e38}
    for bits, val in bf.items():
        assert O.decode16(np.array([bits], np.uint16), "bf16")[0] == val
        assert float(bf16_exact(bits)) == val
    hf = {0x3C00: 1.0, 0xC000: -2.0, 0x0001: 2.0 ** -24, 0x7BFF: 65504.0, 0x6400: 1024.0, 0x3555: 0.333251953125}
    for bits, val in hf.items():
        assert O.decode16(np.array([bits], np.uint16), "fp16")[0] == val
        assert float(fp16_exact(bits)) == val
    rng = np.random.default_rng(0)
    for dtype in ("bf16", "fp16"):
        bits = rng.integers(0, 0x7800, 2000).astype(np.uint16)
        dec = O.decode16(bits, dtype)
        assert all(dec[i] == float(exact16(int(b), dtype)) for i, b in enumerate(bits))


def test_nibble_order_is_little_endian():
    # element 8j + i sits in bits [4i, 4i + 4) of word j
    words = np.array([[0x76543210, 0xFEDCBA98]], dtype=np.uint32)
    assert O.unpack_u4(words, 16).tolist() == [list(range(16))]
    assert I.pack_u4(np.arange(16, dtype=np.uint8)[None]).tolist() == [[0x76543210, 0xFEDCBA98]]


def test_input_rounding_is_rne():
    vals = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 1.0 + 2 ** -8 + 2 ** -20], np.float32)
    assert I.f32_to_bits(vals, "bf16").tolist() == [0x3F80, 0x3F80, 0x3F82, 0xC020, 0x3F81]
    assert I.f32_to_bits(np.array([1.0 + 2 ** -11], np.float32), "fp16").tolist() == [0x3C00]


# ---------------------------------------------------------------- brute force
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("qtype", ["u4b8", "u4_zp", "u4_fzp"])
@pytest.mark.parametrize("shape", [(1, 8, 128), (3, 16, 256), (2, 8, 384)])
def test_oracle_equals_exact_brute_force(dtype, qtype, shape):
    M, N, K = shape
    p = I.make_problem(M, N, K, dtype, qtype, seed=hash((dtype, qtype, shape)) % 1000)
    Yref = O.mm_problem(p)
    exact, sum_abs = brute_force(p)
    for m in range(M):
        for n in range(N):
            # every product is exact in fp64; any summation order errs by <= K * 2^-53 * sum|terms|
            bound = p.K * 2.0 ** -53 * float(sum_abs[m][n]) * 1.01
            assert abs(Yref[m, n] - float(exact[m][n])) <= bound, (m, n, Yref[m, n], float(exact[m][n]))


# one scale row per 256 K, one per row (G = K), one per 64 K (two per 128-K record), and no
# scales at all (direct conversion)
GMODES = [(256, True), ("K", True), (64, True), (128, False)]


@pytest.mark.parametrize("qtype,gmode", [(q, g) for q in ("u4b8", "u4_zp", "u4_fzp") for g in GMODES
                                          if g[1] or q == "u4b8"])     # direct conversion: no zero points
@pytest.mark.parametrize("shape", [(1, 8, 256), (2, 8, 512)])
def test_oracle_group_sizes_equal_exact_brute_force(qtype, gmode, shape):
    M, N, K = shape
    G, scaled = (K if gmode[0] == "K" else gmode[0]), gmode[1]
    p = I.make_problem(M, N, K, "bf16", qtype, seed=K + G + M, group_size=G, scaled=scaled)
    assert (p.S_bits is None) == (not scaled) and (scaled is False or p.S_bits.shape == (K // G, N))
    Yref = O.mm_problem(p)
    exact, sum_abs = brute_force(p)
    for m in range(M):
        for n in range(N):
            bound = p.K * 2.0 ** -53 * float(sum_abs[m][n]) * 1.01
            assert abs(Yref[m, n] - float(exact[m][n])) <= bound, (m, n)


# ---------------------------------------------------------------- epilogue (alpha, C, beta, bias)
def test_epilogue_exact_brute_force():
    """D[m][n] = alpha * sum_k x w + beta * C[m][n] + bias[n], every term an exact Fraction."""
    p = I.make_problem(2, 8, 256, "bf16", "u4_zp", seed=77)
    rng = np.random.default_rng(5)
    C = I.f32_to_bits(rng.standard_normal((2, 8)).astype(np.float32), "bf16")
    bias = I.f32_to_bits(rng.standard_normal(8).astype(np.float32), "bf16")
    alpha, beta = 0.75, -1.5                                   # both exact in binary
    D = O.epilogue(O.mm_problem(p), "bf16", alpha, C, beta, bias)
    exact, sum_abs = brute_force(p)
    for m in range(2):
        for n in range(8):
            e = Fraction(alpha) * exact[m][n] + Fraction(beta) * bf16_exact(int(C[m, n])) + bf16_exact(int(bias[n]))
            bound = (p.K + 2) * 2.0 ** -53 * (float(sum_abs[m][n]) + abs(beta * float(bf16_exact(int(C[m, n])))) + 1) * 1.01
            assert abs(D[m, n] - float(e)) <= bound


def test_epilogue_closed_forms():
    p = I.make_problem(3, 16, 128, "fp16", "u4b8", seed=78)
    Y = O.mm_problem(p)
    C = I.f32_to_bits(np.full((3, 16), 0.5, np.float32), "fp16")
    assert np.array_equal(O.epilogue(Y, "fp16"), Y)                       # identity epilogue
    assert np.array_equal(O.epilogue(Y, "fp16", 0.0, C, 1.0), np.full((3, 16), 0.5))   # alpha 0: D = C
    bias = I.f32_to_bits(np.arange(16, dtype=np.float32), "fp16")
    assert np.array_equal(O.epilogue(Y, "fp16", 1.0, None, 0.0, bias) - Y, np.tile(np.arange(16.0), (3, 1)))
    # beta = 0 never reads C (a C of NaN changes nothing)
    Cnan = np.full((3, 16), 0x7E00, np.uint16)
    assert np.array_equal(O.epilogue(Y, "fp16", 2.0, Cnan, 0.0), 2.0 * Y)


# ---------------------------------------------------------------- closed forms
def _codes_at_zero(N, K, qtype, rng):
    if qtype == "u4b8":
        return np.full((N, K), 8, np.uint8), None
    z = rng.integers(0, 15, (K // 128, N)).astype(np.uint8)   # <= 14 so that z + 1 is a code
    q = np.repeat(z.T, 128, axis=1).astype(np.uint8)         # q[n, k] = z[k // 128, n]
    return q, z


@pytest.mark.parametrize("qtype", ["u4b8", "u4_zp"])
def test_one_hot_closed_form(qtype):
    """(q - z) = 1 at one (n*, k*), 0 elsewhere  =>  Y[:, n*] = s[k*/G, n*] X[:, k*], rest 0."""
    rng = np.random.default_rng(3)
    M, N, K = 5, 16, 384
    q, z = _codes_at_zero(N, K, qtype, rng)
    n_star, k_star = 11, 300
    q[n_star, k_star] += 1
    X = I.f32_to_bits(rng.standard_normal((M, K)).astype(np.float32), "bf16")
    S = I.f32_to_bits(rng.uniform(0.005, 0.02, (K // 128, N)).astype(np.float32), "bf16")
    p = I.problem_from_codes(X, q, S, z, "bf16", qtype)
    Y = O.mm_problem(p)
    expect = np.zeros((M, N))
    expect[:, n_star] = [float(bf16_exact(int(X[m, k_star])) * bf16_exact(int(S[k_star // 128, n_star])))
                         for m in range(M)]
    assert np.array_equal(Y, expect)


def test_identity_weight_gives_x():
    """N = K = 128, codes 8 + delta_nk (uint4b8), unit scales  =>  Y = X exactly."""
    rng = np.random.default_rng(4)
    X = I.f32_to_bits(rng.standard_normal((7, 128)).astype(np.float32), "fp16")
    q = (8 + np.eye(128)).astype(np.uint8)
    S = np.full((1, 128), 0x3C00, np.uint16)                  # fp16 1.0
    Y = O.mm_problem(I.problem_from_codes(X, q, S, None, "fp16", "u4b8"))
    assert np.array_equal(Y, X.view(np.float16).astype(np.float64))


@pytest.mark.parametrize("qtype", ["u4b8", "u4_zp"])
def test_codes_at_zero_point_give_zero(qtype):
    rng = np.random.default_rng(5)
    q, z = _codes_at_zero(24, 256, qtype, rng)
    X = I.f32_to_bits(rng.standard_normal((3, 256)).astype(np.float32), "bf16")
    S = I.f32_to_bits(rng.uniform(0.005, 0.02, (2, 24)).astype(np.float32), "bf16")
    Y = O.mm_problem(I.problem_from_codes(X, q, S, z, "bf16", qtype))
    assert np.array_equal(Y, np.zeros((3, 24)))


# ---------------------------------------------------------------- invariants
@pytest.mark.parametrize("qtype", ["u4b8", "u4_zp"])
def test_group_scale_invariant(qtype):
    """Doubling s[g0, n0] adds exactly group g0's contribution to column n0 and nothing else."""
    p = I.make_problem(6, 32, 512, "bf16", qtype, seed=7)
    g0, n0 = 2, 19
    Y = O.mm_problem(p)
    S2 = p.S_bits.copy()
    s = O.decode16(S2[g0:g0 + 1, n0], "bf16")[0]
    S2[g0, n0] = I.f32_to_bits(np.array([2 * s], np.float32), "bf16")[0]   # exact: power-of-2 scaling
    Y2 = O.mm_problem(I.problem_from_codes(p.X_bits, p.q, S2, p.z, "bf16", qtype))
    # the group's own contribution, by a different route: codes outside group g0 set to zero point
    z = p.z if qtype == "u4_zp" else np.full((4, 32), 8, np.uint8)
    q_only = np.repeat(z.T, 128, axis=1).astype(np.uint8)
    q_only[:, g0 * 128:(g0 + 1) * 128] = p.q[:, g0 * 128:(g0 + 1) * 128]
    contrib = O.mm_problem(I.problem_from_codes(p.X_bits, q_only, p.S_bits, p.z, "bf16", qtype))
    others = [n for n in range(32) if n != n0]
    assert np.array_equal(Y2[:, others], Y[:, others])
    np.testing.assert_allclose(Y2[:, n0] - Y[:, n0], contrib[:, n0], rtol=1e-12, atol=1e-12)
    assert np.abs(contrib[:, n0]).max() > 0


def test_u4b8_equals_zero_point_8():
    p = I.make_problem(4, 64, 256, "fp16", "u4b8", seed=8)
    z8 = np.full((2, 64), 8, np.uint8)
    pz = I.problem_from_codes(p.X_bits, p.q, p.S_bits, z8, "fp16", "u4_zp")
    assert np.array_equal(O.mm_problem(p), O.mm_problem(pz))


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_float_zero_equals_integer_zero_when_exact(dtype):
    """Float-zero mode with zf = -z s, for scales of at most 4 significant bits (so that z s,
    z <= 9, is exact in the 16-bit type), gives the integer zero-point mode's result bit for bit."""
    rng = np.random.default_rng(21)
    M, N, K = 3, 32, 384
    q = rng.integers(0, 16, (N, K)).astype(np.uint8)
    z = rng.integers(6, 10, (K // 128, N)).astype(np.uint8)
    s = rng.integers(8, 16, (K // 128, N)) * 2.0 ** -10                  # m 2^-10, m in 8..15
    S = I.f32_to_bits(s.astype(np.float32), dtype)
    zs = -z.astype(np.float64) * s
    ZF = I.f32_to_bits(zs.astype(np.float32), dtype)
    assert np.array_equal(O.decode16(ZF, dtype), zs)                     # the premise: exact
    X = I.f32_to_bits(rng.standard_normal((M, K)).astype(np.float32), dtype)
    p_int = I.problem_from_codes(X, q, S, z, dtype, "u4_zp")
    p_flt = I.problem_from_codes(X, q, S, ZF, dtype, "u4_fzp")
    assert np.array_equal(O.mm_problem(p_int), O.mm_problem(p_flt))


def test_float_zero_one_hot_closed_form():
    """X one-hot at k*: Y[m, n] = x_m (q[n, k*] s[g*, n] + zf[g*, n]), g* = k* // 128 (exact)."""
    rng = np.random.default_rng(22)
    M, N, K, k_star = 4, 16, 512, 301
    p0 = I.make_problem(M, N, K, "bf16", "u4_fzp", seed=22)
    X = np.zeros((M, K), np.uint16)
    X[:, k_star] = I.f32_to_bits(rng.standard_normal(M).astype(np.float32), "bf16")
    p = I.problem_from_codes(X, p0.q, p0.S_bits, p0.Z, "bf16", "u4_fzp")
    Y = O.mm_problem(p)
    g = k_star // 128
    for m in range(M):
        for n in range(N):
            w = int(p.q[n, k_star]) * bf16_exact(int(p.S_bits[g, n])) + bf16_exact(int(p.Z[g, n]))
            assert Y[m, n] == float(bf16_exact(int(X[m, k_star])) * w)


def test_float_zero_alone_is_group_sums():
    """Codes all 0: Y[m, n] = sum_g zf[g, n] * (sum of X[m, k] over group g), exact rationals."""
    rng = np.random.default_rng(23)
    M, N, K = 2, 8, 384
    p0 = I.make_problem(M, N, K, "fp16", "u4_fzp", seed=23)
    p = I.problem_from_codes(p0.X_bits, np.zeros((N, K), np.uint8), p0.S_bits, p0.Z, "fp16", "u4_fzp")
    Y = O.mm_problem(p)
    for m in range(M):
        gsum = [sum((fp16_exact(int(p.X_bits[m, k])) for k in range(128 * g, 128 * g + 128)), Fraction(0))
                for g in range(K // 128)]
        for n in range(N):
            exact = sum((fp16_exact(int(p.Z[g, n])) * gsum[g] for g in range(K // 128)), Fraction(0))
            assert abs(Y[m, n] - float(exact)) <= 1e-12 * (1 + abs(float(exact)))
    del rng


def test_linearity_in_x():
    rng = np.random.default_rng(9)
    p = I.make_problem(4, 32, 256, "bf16", "u4b8", seed=9)
    # X1 + X2 exactly representable: small integers
    X1 = rng.integers(-8, 8, (4, 256)).astype(np.float32)
    X2 = rng.integers(-8, 8, (4, 256)).astype(np.float32)
    ys = []
    for X in (X1, X2, X1 + X2):
        ys.append(O.mm_problem(I.problem_from_codes(I.f32_to_bits(X, "bf16"), p.q, p.S_bits, None, "bf16", "u4b8")))
    np.testing.assert_allclose(ys[0] + ys[1], ys[2], rtol=0, atol=1e-12)


def test_transpose_identity():
    """Y^T = W . X^T (the transposed problem the pages compute) equals X . W^T."""
    p = I.make_problem(5, 32, 256, "bf16", "u4_zp", seed=10)
    W = O.dequantize(p.Wq, p.S_bits, p.N, p.K, p.dtype, p.qtype, p.Z)
    X = O.decode16(p.X_bits, "bf16")
    np.testing.assert_allclose((W @ X.T).T, O.mm_problem(p), rtol=1e-13, atol=1e-13)


def test_grouped_is_per_problem_and_handles_empty():
    probs = I.make_grouped(40, 4, 128, 256, "bf16", "u4b8", seed=11, M_list=[0, 17, 0, 23])
    outs = O.grouped_mm(probs)
    assert [o.shape for o in outs] == [(0, 128), (17, 128), (0, 128), (23, 128)]
    np.testing.assert_array_equal(outs[1], O.mm_problem(probs[1]))


def test_tolerance_check():
    rng = np.random.default_rng(12)
    Y = rng.standard_normal(1000) * 10
    rounded = O.decode16(I.f32_to_bits(Y.astype(np.float32), "bf16"), "bf16")   # correctly rounded output
    assert O.check_tolerance(rounded, Y)["violations"] == 0
    bad = Y.copy()
    bad[17] += 2 * (1e-2 + 1e-2 * abs(Y[17]))
    st = O.check_tolerance(bad, Y)
    assert st["violations"] == 1 and st["max_err_over_tol"] == pytest.approx(2.0)
    assert O.check_tolerance(np.array([np.nan]), np.array([0.0]))["violations"] == 1


# ---------------------------------------------------------------- blob layout
def _brute_blob(p) -> np.ndarray:
    """The blob built one element at a time straight from the layout's wording (no scales: 1.0 =
    0x3F80 / 0x3C00): record (nt, g) is eight 16-row blocks; a block has H scale sets (H = 2 for
    G = 64, else 1), set h covering the record's K elements from 64 h and carrying the scale (and
    zero) of quantisation group (128 g + 64 h) // G; block bytes 1024 + 32 H (uint4b8), plus 8 H
    padded to 16 (zero points) or plus 32 H (float zeros); in block b, row rr's K elements
    32 j + [0, 32) form 16-byte chunk 16 j + rr, its scale of set h sits at byte
    1024 + 32 h + 4 (rr % 8) + 2 (rr // 8), its zero point of set h in byte 1024 + 32 H + 8 h + rr % 8
    (high nibble for rr >= 8), its float zero of set h at byte 1024 + 32 H + 32 h + 4 (rr % 8) + 2 (rr // 8)."""
    G = p.group_size
    H = 2 if G == 64 else 1
    bb = 1024 + 32 * H + {"u4b8": 0, "u4_zp": 8 * H, "u4_fzp": 32 * H}[p.qtype]
    bb = (bb + 15) // 16 * 16
    tb = 8 * bb
    nG = p.K // 128
    blob = np.zeros(256 + (p.N // 128) * nG * tb, np.uint8)
    assert blob.size == O.prepacked_bytes(p.N, p.K, p.qtype, G)
    hdr = [O.BLOB_MAGIC, 2, p.N, p.K, G, O.DTYPE_CODE[p.dtype], O.QTYPE_CODE[p.qtype], tb, p.N // 128, nG]
    for i, v in enumerate(hdr):
        blob[4 * i:4 * i + 4] = list(int(v).to_bytes(4, "little"))
    pos = {0: 0, 2: 1, 4: 2, 6: 3, 1: 4, 3: 5, 5: 6, 7: 7}
    for n in range(p.N):
        nt, b, rr = n // 128, (n % 128) // 16, n % 16
        for k in range(p.K):
            g, kk = k // 128, k % 128
            j, w, e = kk // 32, (kk % 32) // 8, kk % 8
            blk = 256 + (nt * nG + g) * tb + b * bb
            byte_off = blk + (16 * j + rr) * 16 + 4 * w + pos[e] // 2
            shift = 4 * (pos[e] % 2)
            blob[byte_off] |= int(p.q[n, k]) << shift
    for g in range(nG):
        for h in range(H):
            src = (128 * g + 64 * h) // G
            for n in range(p.N):
                nt, b, rr = n // 128, (n % 128) // 16, n % 16
                blk = 256 + (nt * nG + g) * tb + b * bb
                sbits = int(p.S_bits[src, n]) if p.S_bits is not None else (0x3F80 if p.dtype == "bf16" else 0x3C00)
                so = blk + 1024 + 32 * h + 4 * (rr % 8) + 2 * (rr // 8)
                blob[so:so + 2] = list(sbits.to_bytes(2, "little"))
                if p.qtype == "u4_zp":
                    blob[blk + 1024 + 32 * H + 8 * h + rr % 8] |= int(p.z[src, n]) << (4 * (rr // 8))
                if p.qtype == "u4_fzp":                     # float zeros placed like the scales
                    zo = blk + 1024 + 32 * H + 32 * h + 4 * (rr % 8) + 2 * (rr // 8)
                    blob[zo:zo + 2] = list(int(p.Z[src, n]).to_bytes(2, "little"))
    return blob


@pytest.mark.parametrize("qtype", ["u4b8", "u4_zp", "u4_fzp"])
def test_blob_layout_brute_force(qtype):
    p = I.make_problem(1, 256, 256, "bf16", qtype, seed=13)
    assert np.array_equal(O.prepack(p.Wq, p.S_bits, p.N, p.K, p.dtype, p.qtype, p.Z), _brute_blob(p))


@pytest.mark.parametrize("qtype,G,scaled,dtype", [("u4_zp", 256, True, "bf16"), ("u4b8", 512, True, "fp16"),
                                                  ("u4_fzp", 256, True, "fp16"), ("u4b8", 64, True, "bf16"),
                                                  ("u4_zp", 64, True, "fp16"), ("u4_fzp", 64, True, "bf16"),
                                                  ("u4b8", 64, False, "fp16"),
                                                  ("u4b8", 128, False, "bf16"), ("u4b8", 256, False, "fp16")])
def test_blob_layout_group_sizes_brute_force(qtype, G, scaled, dtype):
    p = I.make_problem(1, 256, 512, dtype, qtype, seed=G + 1, group_size=G, scaled=scaled)
    blob = O.prepack(p.Wq, p.S_bits, p.N, p.K, p.dtype, p.qtype, p.Z, group_size=G)
    assert np.array_equal(blob, _brute_blob(p))
    Wq, S, Z = O.unprepack(blob, p.N, p.K, dtype, qtype, group_size=G)
    assert np.array_equal(Wq, p.Wq)
    if scaled:
        assert np.array_equal(S, p.S_bits)
    if qtype in ("u4_zp", "u4_fzp"):
        assert np.array_equal(Z, p.Z)


def test_blob_rejects_unsupported_group_sizes():
    p = I.make_problem(1, 128, 512, "bf16", "u4b8", seed=3)
    for G in (32, 384, 192):
        with pytest.raises(ValueError):
            O.prepack(p.Wq, np.zeros((512 // 32, 128), np.uint16), p.N, p.K, p.dtype, p.qtype, group_size=G)


@pytest.mark.parametrize("qtype", ["u4b8", "u4_zp", "u4_fzp"])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_blob_round_trip(qtype, dtype):
    p = I.make_problem(1, 384, 640, dtype, qtype, seed=14)
    blob = O.prepack(p.Wq, p.S_bits, p.N, p.K, dtype, qtype, p.Z)
    assert blob.size == O.prepacked_bytes(p.N, p.K, qtype)
    Wq, S, Z = O.unprepack(blob, p.N, p.K, dtype, qtype)
    assert np.array_equal(Wq, p.Wq) and np.array_equal(S, p.S_bits)
    if qtype in ("u4_zp", "u4_fzp"):
        assert np.array_equal(Z, p.Z)
    hdr = blob[:40].view(np.uint32)
    assert hdr.tolist() == [O.BLOB_MAGIC, 2, 384, 640, 128, O.DTYPE_CODE[dtype], O.QTYPE_CODE[qtype],
                            O.tile_bytes(qtype), 3, 5]
