"""Plant plausible mistakes in the oracle (on the CPU) and check that the pins catch them.

Each mutant replaces one oracle function with a subtly wrong variant (a wrong
sign, a swapped index, a dropped term, another rounding rule); at least one
pin must then fail.  This shows the pins constrain every part of the oracle.
"""

import numpy as np
import pytest

from oracle import kvq_oracle as ko
import test_oracle_outliers as opins
import test_oracle_pins as pins

F32 = np.float32


_orig = {"fwht": ko.fwht, "pack_q4_0": ko.pack_q4_0, "quantize_q4_0": ko.quantize_q4_0,
         "quantize_q8_0": ko.quantize_q8_0, "bf16_bits": ko.bf16_bits,
         "signed_max_magnitude": ko.signed_max_magnitude, "rotation_matrix": ko.rotation_matrix,
         "sylvester_hadamard": ko.sylvester_hadamard, "pack_q5_0": ko.pack_q5_0,
         "dequantize": ko.dequantize, "softmax_attention": ko.softmax_attention}


def _fwht_transposed_pairs(x, group):
    # butterfly with (a-b, a+b): a sign/ordering slip
    y = np.array(x, dtype=np.float64, copy=True)
    shape, d, h = y.shape, y.shape[-1], 1
    while h < group:
        v = y.reshape(-1, d // group, group // (2 * h), 2, h)
        a, b = v[:, :, :, 0, :].copy(), v[:, :, :, 1, :].copy()
        v[:, :, :, 0, :], v[:, :, :, 1, :] = a - b, a + b
        y = v.reshape(shape)
        h *= 2
    return y / np.sqrt(group)


def _pack_q4_swapped(codes):
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 16:] | (c[..., :16] << 4)).astype(np.uint8)


def _pack_q4_interleaved(codes):
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def _q4_rounding(y):
    b = ko._blocks(y)
    m, _ = ko.signed_max_magnitude(b)
    d = (m / F32(-8)).astype(F32)
    inv = ko._inverse(d)
    v = (b * inv[..., None]).astype(F32) + F32(8.0)
    codes = np.clip(np.rint(v), 0, 15)   # round-half-even instead of trunc(x + 8.5)
    return ko.f16_bits(d), codes.astype(np.uint8)


def _q4_amax_scale(y):
    b = ko._blocks(y)
    _, amax = ko.signed_max_magnitude(b)
    d = (amax / F32(-8)).astype(F32)       # sign of the max dropped
    inv = ko._inverse(d)
    v = ((b * inv[..., None]).astype(F32) + F32(8.5)).astype(F32)
    return ko.f16_bits(d), np.minimum(15, np.trunc(v)).astype(np.uint8)


def _q8_half_even(y):
    b = ko._blocks(y)
    amax = np.max(np.abs(b), axis=-1).astype(F32)
    d = (amax / F32(127)).astype(F32)
    v = (b * ko._inverse(d)[..., None]).astype(F32)
    return ko.f16_bits(d), np.rint(v).astype(np.int8)


def _bf16_truncate(x):
    u = np.asarray(x, dtype=F32).view(np.uint32)
    return (u >> 16).astype(np.uint16)


def _signed_max_last_tie(blocks):
    a = np.abs(blocks)
    idx = blocks.shape[-1] - 1 - np.argmax(a[..., ::-1], axis=-1)
    amax = np.take_along_axis(a, idx[..., None], axis=-1)[..., 0]
    m = np.take_along_axis(blocks, idx[..., None], axis=-1)[..., 0]
    return np.where(amax > 0, m, F32(0)).astype(F32), amax.astype(F32)


def _rotation_unnormalized(d):
    return _orig["rotation_matrix"](d) * np.sqrt(ko.rotation_group(d))


def _rotation_natural_blocks(d):
    # block-diagonal built with the wrong block size for non-power-of-two d
    if ko.is_power_of_two(d):
        return _orig["rotation_matrix"](d)
    g = 32
    hg = ko.sylvester_hadamard(g) / np.sqrt(g)
    r = np.zeros((d, d))
    for i in range(d // g):
        r[i * g:(i + 1) * g, i * g:(i + 1) * g] = hg
    return r


def _pack_q5_high_bits_reversed(codes):
    qs, qh = _orig["pack_q5_0"](codes)
    rev = np.zeros_like(qh)
    for j in range(32):
        rev |= ((qh >> np.uint32(j)) & np.uint32(1)) << np.uint32(31 - j)
    return qs, rev


def _dequant_no_offset(qtype, d_bits, codes):
    dv = ko.f16_value(d_bits)[..., None]
    x = np.asarray(codes).astype(np.float64) * dv
    return x.reshape(x.shape[:-2] + (x.shape[-2] * 32,))


def _softmax_no_max_shift_scale(q, K, V, scale):
    return _orig["softmax_attention"](q, K, V, scale * 1.01)


def _min_no_half(y, top=15):
    """q4_1 without the +0.5 (codes truncated instead of rounded)."""
    b = ko._blocks(y)
    lo = np.min(b, axis=-1).astype(np.float32)
    d = ((np.max(b, axis=-1) - lo) / np.float32(top)).astype(np.float32)
    inv = ko._inverse(d)
    v = ((b - lo[..., None]).astype(np.float32) * inv[..., None]).astype(np.float32)
    codes = np.minimum(top, np.trunc(v.astype(np.float64)))
    word = ko.f16_bits(d).astype(np.uint32) | (ko.f16_bits(lo).astype(np.uint32) << np.uint32(16))
    return word, codes.astype(np.uint8)


def _min_word_swapped(y):
    """q5_1 with d and the minimum swapped in the scale word."""
    word, codes = ko._quantize_min(y, 31)
    return ((word >> np.uint32(16)) | (word << np.uint32(16))).astype(np.uint32), codes


def _dequant_min_dropped(qtype, d_bits, codes):
    """Scale + minimum blocks decoded without the minimum."""
    if qtype in ko.MIN_TYPES:
        dv, _ = ko.scale_and_min(qtype, d_bits)
        x = np.asarray(codes).astype(np.float64) * dv[..., None]
        return x.reshape(x.shape[:-2] + (x.shape[-2] * 32,))
    return _ORIG_DEQUANT(qtype, d_bits, codes)


_ORIG_DEQUANT = ko.dequantize
_ORIG_SPLIT = ko.split_outliers
_ORIG_OVALS = ko.outlier_values


def _split_rest_not_zeroed(x, oidx):
    """Outlier values taken but left in the vector that gets rotated."""
    xo, _ = _ORIG_SPLIT(x, oidx)
    return xo, np.asarray(x, dtype=np.float32).copy()


def _split_slots_reversed(x, oidx):
    """Outlier values stored in decreasing channel order."""
    xo, rest = _ORIG_SPLIT(x, oidx)
    return xo[..., ::-1].copy(), rest


def _ovals_shifted(d_bits, codes, chans, head_dim):
    """Outlier values scattered one channel off."""
    return np.roll(_ORIG_OVALS(d_bits, codes, chans, head_dim), 1, axis=-1)


def _ovals_negated(d_bits, codes, chans, head_dim):
    return -_ORIG_OVALS(d_bits, codes, chans, head_dim)


_ORIG_GGML = ko.to_ggml_bytes


def _f16_truncating(x):
    """float32 -> fp16 by truncating the mantissa instead of rounding to nearest even."""
    x = np.asarray(x, dtype=F32)
    t = x.astype(np.float16)
    up = np.abs(t.astype(F32)) > np.abs(x)            # RNE rounded away from zero: step back one ulp
    bits = t.view(np.uint16).copy()
    bits[up & (x != 0)] -= 1
    return bits


def _q5_divisor_15(y):
    """q5_0 scale m / -15 instead of m / -16."""
    return ko._quantize_offset(y, -15.0, 16.5, 31)


def _ggml_qs_before_d(qtype, d_bits, codes):
    """Block fields in the wrong order: quants first, then the scale."""
    img = _ORIG_GGML(qtype, d_bits, codes)
    hd = 4 if qtype in ko.MIN_TYPES else 2
    return np.concatenate([img[..., hd:], img[..., :hd]], axis=-1)


def _enable_rule_32(head_dim):
    """Rotation enabled from head_dim 32 in steps of 32."""
    return head_dim >= 32 and head_dim % 32 == 0


def _inverse_unguarded(d):
    """1/d without the d == 0 case (an all-zero block then divides by zero)."""
    with np.errstate(divide="ignore", invalid="ignore"):
        return (F32(1.0) / np.asarray(d, dtype=F32)).astype(F32)


# -- the cache and the attention functions -----------------------------------
_ORIG_STORED = ko.OracleCache.stored
_ORIG_APPEND = ko.OracleCache.append
_ORIG_DECODE = ko.decode_attention
_ORIG_PREFILL = ko.prefill_attention


def _stored_tail_one_short(self, which, b, h):
    """Body / tail boundary one position late: position n - T read from the body."""
    n = int(self.seq_len[b])
    split = min(n, max(0, n - self.T + 1))
    out = np.empty((n, self.d), dtype=np.float64)
    out[:split] = self.body_values(which, b, h, 0, split)
    if n > split:
        out[split:] = self.tail_values(which, b, h, np.arange(split, n))
    return out


def _tail_slot_shifted(self, which, b, h, positions):
    """Ring slot off by one: (pos + 1) % T."""
    slots = (np.asarray(positions, dtype=np.int64) + 1) % self.T
    return ko.bf16_value(self.tail[which][b, h, slots])


def _append_not_write_through(self, k, v, n_new_per_seq=None, prerotated=False):
    """Tokens that go to the tail are not quantized into the body."""
    n_before = self.seq_len.copy()
    _ORIG_APPEND(self, k, v, n_new_per_seq, prerotated)
    if self.T == 0:
        return
    for b in range(self.B):
        n0, n1 = int(n_before[b]), int(self.seq_len[b])
        first = max(n0, n1 - self.T)
        for w in ("k", "v"):
            self.codes[w][b, :, first:n1] = 0
            self.dbits[w][b, :, first:n1] = 0


def _decode_heads_interleaved(cache, q, scale=None, pairs=None):
    """Query head h reads KV head h % Hkv instead of h // (Hq / Hkv)."""
    q = np.asarray(q, dtype=np.float64)
    B, Hq, d = q.shape
    perm = np.array([(h % cache.H) * (Hq // cache.H) + h // cache.H for h in range(Hq)])
    out = _ORIG_DECODE(cache, q[:, perm], scale, pairs)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(Hq)
    return out[:, inv]


def _decode_not_rotated_back(cache, q, scale=None, pairs=None):
    """The output is left in the rotated basis."""
    out = _ORIG_DECODE(cache, q, scale, pairs)
    if cache.rot["v"]:
        out = out @ ko.rotation_matrix(out.shape[-1])   # H is its own inverse: undoes the back-rotation
    return out


def _prefill_strictly_causal(cache, q, q_pos0=None, causal=True, scale=None, heads=None):
    """A query does not see the key at its own position (t < p)."""
    B, n_tok = np.asarray(q).shape[:2]
    if not causal:
        return _ORIG_PREFILL(cache, q, q_pos0, causal, scale, heads)
    p0 = cache.seq_len - n_tok if q_pos0 is None else np.asarray(q_pos0)
    return _ORIG_PREFILL(cache, q, p0 - 1, causal, scale, heads)


def _prefill_positions_shifted(cache, q, q_pos0=None, causal=True, scale=None, heads=None):
    """Default query positions one too far: n - n_tok + 1."""
    n_tok = np.asarray(q).shape[1]
    p0 = cache.seq_len - n_tok + 1 if q_pos0 is None else np.asarray(q_pos0)
    return _ORIG_PREFILL(cache, q, p0, causal, scale, heads)


MUTANTS = [
    ("fwht", _fwht_transposed_pairs, [pins.test_rotate_golden_vectors]),
    ("pack_q4_0", _pack_q4_swapped, [pins.test_packing_golden]),
    ("pack_q4_0", _pack_q4_interleaved, [pins.test_packing_golden]),
    ("quantize_q4_0", _q4_rounding, [pins.test_golden_blocks]),
    ("quantize_q4_0", _q4_amax_scale, [pins.test_golden_blocks]),
    ("quantize_q8_0", _q8_half_even, [pins.test_golden_blocks]),
    ("bf16_bits", _bf16_truncate, [pins.test_bf16_rounding_matches_torch]),
    ("signed_max_magnitude", _signed_max_last_tie, [pins.test_signed_max_first_index_on_ties, pins.test_golden_blocks]),
    ("rotation_matrix", _rotation_unnormalized, [lambda: pins.test_rotation_orthonormal_symmetric(128)]),
    ("rotation_matrix", _rotation_natural_blocks, [lambda: pins.test_rotation_orthonormal_symmetric(192)]),
    ("pack_q5_0", _pack_q5_high_bits_reversed, [pins.test_packing_golden]),
    ("dequantize", _dequant_no_offset, [lambda: pins.test_quantizer_error_bounds("q4_0")]),
    ("softmax_attention", _softmax_no_max_shift_scale, [pins.test_decode_gqa_bruteforce]),
    ("quantize_q4_1", _min_no_half, [pins.test_golden_blocks]),
    ("quantize_q5_1", _min_word_swapped, [pins.test_golden_blocks]),
    ("dequantize", _dequant_min_dropped, [lambda: pins.test_min_quantizer_error_bounds("q4_1")]),
    ("split_outliers", _split_rest_not_zeroed, [lambda: opins.test_exact_reconstruction_through_rotation(True)]),
    ("split_outliers", _split_slots_reversed, [lambda: opins.test_exact_reconstruction_through_rotation(False)]),
    ("outlier_values", _ovals_shifted, [opins.test_outlier_only_vectors_are_q8_0_alone]),
    ("outlier_values", _ovals_negated, [lambda: opins.test_reconstruction_error_within_the_two_quantizations("q4_0")]),
    ("f16_bits", _f16_truncating, [pins.test_golden_blocks]),
    ("rotation_enabled", _enable_rule_32, [pins.test_enable_rule]),
    ("_inverse", _inverse_unguarded, [lambda: pins.test_all_zero_block("q4_0", 0x8000, 8)]),
    ("quantize_q5_0", _q5_divisor_15, [pins.test_golden_blocks]),
    ("to_ggml_bytes", _ggml_qs_before_d, [pins.test_packing_golden]),
    ("decode_attention", _decode_heads_interleaved, [pins.test_decode_gqa_bruteforce]),
    ("decode_attention", _decode_not_rotated_back, [pins.test_decode_gqa_bruteforce]),
    ("prefill_attention", _prefill_strictly_causal, [pins.test_prefill_causal_bruteforce_and_decode_consistency]),
    ("prefill_attention", _prefill_positions_shifted, [pins.test_prefill_causal_bruteforce_and_decode_consistency]),
]

# mutants of OracleCache methods: (method name, replacement, pins)
CACHE_MUTANTS = [
    ("stored", _stored_tail_one_short, [pins.test_tail_ring_wraparound_many_appends]),
    ("tail_values", _tail_slot_shifted, [pins.test_tail_ring_wraparound_many_appends]),
    ("append", _append_not_write_through, [pins.test_tail_ring_wraparound_many_appends]),
]


@pytest.mark.parametrize("i", range(len(MUTANTS)))
def test_pins_catch_planted_mistake(monkeypatch, i):
    name, fn, checks = MUTANTS[i]
    monkeypatch.setattr(ko, name, fn)
    failed = 0
    for chk in checks:
        try:
            with np.errstate(all="ignore"):   # a planted mistake may divide by zero
                chk()
        except (AssertionError, ValueError):
            failed += 1
    assert failed >= 1, f"mutant of {name} ({fn.__name__}) passed every pin"


@pytest.mark.parametrize("i", range(len(CACHE_MUTANTS)))
def test_pins_catch_planted_cache_mistake(monkeypatch, i):
    name, fn, checks = CACHE_MUTANTS[i]
    monkeypatch.setattr(ko.OracleCache, name, fn)
    failed = 0
    for chk in checks:
        try:
            with np.errstate(all="ignore"):   # a planted mistake may divide by zero
                chk()
        except (AssertionError, ValueError):
            failed += 1
    assert failed >= 1, f"mutant of OracleCache.{name} ({fn.__name__}) passed every pin"
