"""The pins are sharp: each plausible mistake planted in the oracle (on the CPU, by patching one
of its functions for the duration of a test) makes at least one pin fail."""
import numpy as np
import pytest

import oracle as OP
import oracle.wq4_oracle as W
import tests.test_oracle_pins as pins

_good_dequantize = W.dequantize
_good_unpack = W.unpack_u4
_good_decode = W.decode16
_good_epilogue = W.epilogue
_good_prepack = W.prepack


def _dq_zero_index_mod(Wq, S_bits, N, K, dtype, qtype, Z_words=None, group_size=128):
    q = W.unpack_u4(Wq, K).astype(np.int64)
    z = W.zero_points(N, K, qtype, Z_words, group_size)
    s = W.decode16(S_bits, dtype)
    g = np.arange(K) // group_size
    gz = np.arange(K) % (K // group_size)          # wrong index for the zero point
    return (q - z[gz, :].T).astype(np.float64) * s[g, :].T


def _dq_sign(Wq, S_bits, N, K, dtype, qtype, Z_words=None, group_size=128):
    return -_good_dequantize(Wq, S_bits, N, K, dtype, qtype, Z_words, group_size)


def _dq_drop_zero(Wq, S_bits, N, K, dtype, qtype, Z_words=None, group_size=128):
    q = W.unpack_u4(Wq, K).astype(np.float64)
    s = W.decode16(S_bits, dtype)
    return q * s[np.arange(K) // group_size, :].T


def _dq_group_64(Wq, S_bits, N, K, dtype, qtype, Z_words=None, group_size=128):
    q = W.unpack_u4(Wq, K).astype(np.int64)
    z = W.zero_points(N, K, qtype, Z_words, group_size)
    s = W.decode16(S_bits, dtype)
    g = np.minimum(np.arange(K) // 64, K // group_size - 1)   # wrong group size
    return (q - z[g, :].T).astype(np.float64) * s[g, :].T


def _dq_scale_rows_swapped(Wq, S_bits, N, K, dtype, qtype, Z_words=None, group_size=128):
    out = _good_dequantize(Wq, S_bits, N, K, dtype, qtype, Z_words, group_size)
    return out[::-1].copy()                          # rows of W attached to the wrong outputs


def _fzp_parts(Wq, S_bits, N, K, dtype, Z_words, group_size):
    q = W.unpack_u4(Wq, K).astype(np.float64)
    g = np.arange(K) // group_size
    s = W.decode16(S_bits, dtype)[g, :].T
    zf = W.decode16(Z_words, dtype).reshape(K // group_size, N)[g, :].T
    return q, s, zf


def _dq_fzp_zero_before_scale(Wq, S_bits, N, K, dtype, qtype, Z_words=None, group_size=128):
    if qtype != "u4_fzp":
        return _good_dequantize(Wq, S_bits, N, K, dtype, qtype, Z_words, group_size)
    q, s, zf = _fzp_parts(Wq, S_bits, N, K, dtype, Z_words, group_size)
    return (q + zf) * s


def _dq_fzp_zero_dropped(Wq, S_bits, N, K, dtype, qtype, Z_words=None, group_size=128):
    if qtype != "u4_fzp":
        return _good_dequantize(Wq, S_bits, N, K, dtype, qtype, Z_words, group_size)
    q, s, zf = _fzp_parts(Wq, S_bits, N, K, dtype, Z_words, group_size)
    return q * s


def _dq_fzp_zero_subtracted(Wq, S_bits, N, K, dtype, qtype, Z_words=None, group_size=128):
    if qtype != "u4_fzp":
        return _good_dequantize(Wq, S_bits, N, K, dtype, qtype, Z_words, group_size)
    q, s, zf = _fzp_parts(Wq, S_bits, N, K, dtype, Z_words, group_size)
    return q * s - zf


def _dq_with_groups_at_64(gmap):
    """The oracle's dequantisation, but at G = 64 with group index gmap(k) in place of k // 64."""
    def dq(Wq, S_bits, N, K, dtype, qtype, Z_words=None, group_size=128):
        if group_size != 64:
            return _good_dequantize(Wq, S_bits, N, K, dtype, qtype, Z_words, group_size)
        q = W.unpack_u4(Wq, K).astype(np.int64)
        z = W.zero_points(N, K, qtype, Z_words, group_size)
        s = W.decode16(S_bits, dtype) if S_bits is not None else np.ones((K // group_size, N))
        g = gmap(np.arange(K))
        out = (q - z[g, :].T).astype(np.float64) * s[g, :].T
        if qtype == "u4_fzp":
            out = out + W.decode16(Z_words, dtype).reshape(K // group_size, N)[g, :].T
        return out
    return dq


def _epi_bias_scaled(Y_acc, dtype, alpha=1.0, C_bits=None, beta=0.0, bias_bits=None):
    D = float(alpha) * _good_epilogue(Y_acc, dtype, 1.0, None, 0.0, bias_bits)   # alpha (acc + bias)
    if beta != 0.0:
        D = D + float(beta) * W.decode16(np.asarray(C_bits).reshape(D.shape), dtype)
    return D


def _epi_alpha_beta_swapped(Y_acc, dtype, alpha=1.0, C_bits=None, beta=0.0, bias_bits=None):
    return _good_epilogue(Y_acc, dtype, beta if C_bits is not None else alpha, C_bits,
                          alpha if C_bits is not None else beta, bias_bits)


def _epi_bias_per_token(Y_acc, dtype, alpha=1.0, C_bits=None, beta=0.0, bias_bits=None):
    D = _good_epilogue(Y_acc, dtype, alpha, C_bits, beta, None)
    if bias_bits is not None:
        b = W.decode16(np.asarray(bias_bits), dtype)
        D = D + b[np.arange(D.shape[0]) % b.size][:, None]       # indexed by token, not by weight row
    return D


def _epi_c_transposed(Y_acc, dtype, alpha=1.0, C_bits=None, beta=0.0, bias_bits=None):
    if C_bits is None or beta == 0.0:
        return _good_epilogue(Y_acc, dtype, alpha, C_bits, beta, bias_bits)
    Ct = np.ascontiguousarray(np.asarray(C_bits).reshape(np.shape(Y_acc)).T).reshape(np.shape(Y_acc))
    return _good_epilogue(Y_acc, dtype, alpha, Ct, beta, bias_bits)


def _pp_from_good(edit):
    """The oracle's blob with `edit(records, qtype, group_size)` applied to its tile records
    [N/128][K/128][record bytes] in place."""
    def pp(Wq, S_bits, N, K, dtype, qtype, Z_words=None, group_size=128):
        blob = _good_prepack(Wq, S_bits, N, K, dtype, qtype, Z_words, group_size=group_size).copy()
        recs = blob[W.HEADER_BYTES:].reshape(N // 128, K // 128, W.tile_bytes(qtype, group_size))
        edit(recs, qtype, group_size)
        return blob
    return pp


def _records_k_major(recs, qtype, G):
    recs[...] = recs.transpose(1, 0, 2).reshape(recs.shape).copy()   # (g, nt) order instead of (nt, g)


def _scale_sets_swapped(recs, qtype, G):
    if G != 64:
        return
    bb = W.block_bytes(qtype, G)
    for b in range(8):
        s0 = b * bb + 1024
        a = recs[:, :, s0:s0 + 32].copy()
        recs[:, :, s0:s0 + 32] = recs[:, :, s0 + 32:s0 + 64]
        recs[:, :, s0 + 32:s0 + 64] = a


def _scale_rows_paired_wrong(recs, qtype, G):
    bb = W.block_bytes(qtype, G)
    for b in range(8):
        for w in range(8):                           # rows r and r + 8 of each scale word swapped
            o = b * bb + 1024 + 4 * w
            lo = recs[:, :, o:o + 2].copy()
            recs[:, :, o:o + 2] = recs[:, :, o + 2:o + 4]
            recs[:, :, o + 2:o + 4] = lo


def _unpack_big_endian(words, length):
    words = np.asarray(words, dtype=np.uint32)
    shifts = 28 - 4 * np.arange(8, dtype=np.uint32)
    nib = (words[..., :, None] >> shifts) & np.uint32(0xF)
    return nib.reshape(words.shape[:-1] + (words.shape[-1] * 8,)).astype(np.uint8)


def _decode_bf16_as_fp16(bits, dtype):
    return _good_decode(bits, "fp16")


MUTANTS = {
    "zero point indexed by k mod groups": ("dequantize", _dq_zero_index_mod),
    "sign flipped": ("dequantize", _dq_sign),
    "zero point dropped": ("dequantize", _dq_drop_zero),
    "group size 64": ("dequantize", _dq_group_64),
    "weight rows permuted": ("dequantize", _dq_scale_rows_swapped),
    "big-endian nibbles": ("unpack_u4", _unpack_big_endian),
    "bf16 decoded as fp16": ("decode16", _decode_bf16_as_fp16),
    "float zero added before the scale": ("dequantize", _dq_fzp_zero_before_scale),
    "float zero dropped": ("dequantize", _dq_fzp_zero_dropped),
    "float zero subtracted": ("dequantize", _dq_fzp_zero_subtracted),
    # G = 64 (two scale sets per 128-K record): the first set used for both halves, or the halves swapped
    "G = 64 with one scale set per 128 K": ("dequantize", _dq_with_groups_at_64(lambda k: (k // 128) * 2)),
    "G = 64 with the halves swapped": ("dequantize", _dq_with_groups_at_64(lambda k: (k // 64) ^ 1)),
    # the epilogue D = alpha acc + beta C + bias[n]
    "epilogue: bias scaled by alpha": ("epilogue", _epi_bias_scaled),
    "epilogue: alpha and beta swapped": ("epilogue", _epi_alpha_beta_swapped),
    "epilogue: bias indexed by token": ("epilogue", _epi_bias_per_token),
    "epilogue: C read transposed": ("epilogue", _epi_c_transposed),
    # the prepacked blob's layout
    "blob records in k-major order": ("prepack", _pp_from_good(_records_k_major)),
    "blob G = 64 scale sets swapped": ("prepack", _pp_from_good(_scale_sets_swapped)),
    "blob scales of rows r and r + 8 swapped": ("prepack", _pp_from_good(_scale_rows_paired_wrong)),
}


def _pins_all_pass():
    checks = [
        lambda: pins.test_oracle_equals_exact_brute_force("bf16", "u4_zp", (2, 8, 384)),
        lambda: pins.test_oracle_equals_exact_brute_force("bf16", "u4b8", (3, 16, 256)),
        lambda: pins.test_one_hot_closed_form("u4_zp"),
        lambda: pins.test_group_scale_invariant("u4b8"),
        lambda: pins.test_decode16_bit_patterns(),
        lambda: pins.test_nibble_order_is_little_endian(),
        lambda: pins.test_oracle_equals_exact_brute_force("fp16", "u4_fzp", (1, 8, 128)),
        lambda: pins.test_float_zero_one_hot_closed_form(),
        lambda: pins.test_float_zero_alone_is_group_sums(),
        lambda: pins.test_oracle_group_sizes_equal_exact_brute_force("u4_zp", (64, True), (1, 8, 256)),
        lambda: pins.test_epilogue_exact_brute_force(),
        lambda: pins.test_epilogue_closed_forms(),
        lambda: pins.test_blob_layout_brute_force("u4_zp"),
        lambda: pins.test_blob_layout_group_sizes_brute_force("u4_zp", 64, True, "fp16"),
    ]
    for c in checks:
        try:
            c()
        except Exception:
            return False
    return True


def test_unmutated_oracle_passes():
    assert _pins_all_pass()


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(W, attr, fn)
    if hasattr(OP, attr):                            # the package's own name for it, which the pins call
        monkeypatch.setattr(OP, attr, fn)
    assert not _pins_all_pass(), name
