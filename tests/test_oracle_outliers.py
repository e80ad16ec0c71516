"""Pins of the oracle's outlier-channel path (8-bit outlier channels beside the
rotated low-bit rest) against what the mathematics fixes: exact reconstruction
when every quantization step is exact, the special cases that reduce to the
plain cache (no outlier energy) or to q8_0 alone (no rest), brute-force
attention in the original basis, the bf16 tail left whole, and the error bound
of the two quantizations.  No GPU needed."""

import numpy as np
import pytest

from oracle import kvq_oracle as ko
from test_oracle_pins import _loops_attention

F32 = np.float32


def _exact_case(upper: bool, ntok=6, seed=0):
    """d = 64, one KV head, outlier channels = one half of the head.  The rest
    lives in the other half as u = H_32 z (z integers with |z| <= 127 and one
    127 per vector), so R x_rest = (4z, +-4z): q8_0 blocks with scale exactly 4
    and codes z.  Outlier values are integers * 2^-3 with one 127 * 2^-3, so
    their q8_0 scale is exactly 2^-3.  Both quantizations are then exact."""
    rng = np.random.default_rng(seed)
    d = 64
    h32 = ko.sylvester_hadamard(32)
    x = np.zeros((1, ntok, 1, d), F32)
    for t in range(ntok):
        z = rng.integers(-127, 128, 32)
        z[rng.integers(32)] = 127 * rng.choice([-1, 1])
        zo = rng.integers(-127, 128, 32)
        zo[rng.integers(32)] = 127 * rng.choice([-1, 1])
        rest, outl = (h32 @ z).astype(F32), (zo * 0.125).astype(F32)
        x[0, t, 0] = np.concatenate([rest, outl]) if upper else np.concatenate([outl, rest])
    chans = np.arange(32, 64) if upper else np.arange(0, 32)
    return x, chans[None, :]


@pytest.mark.parametrize("upper", [True, False])
def test_exact_reconstruction_through_rotation(upper):
    x, oidx = _exact_case(upper)
    c = ko.OracleCache(1, 1, 64, 16, 0, "q8_0", "q8_0", True, True, outliers=oidx)
    c.append(x, x)
    R = ko.rotation_matrix(64)
    for w in ("k", "v"):
        khat = c.stored(w, 0, 0) @ R          # original basis
        assert np.max(np.abs(khat - x[0, :, 0])) < 1e-9
        # codes: the rest is 4z in the rotated basis, the outliers are 8 * value
        assert np.all(ko.f16_value(c.odbits[w][0, 0, :6]) == 0.125)
        assert np.array_equal(c.ocodes[w][0, 0, :6, 0].astype(np.float64), x[0, :, 0][:, oidx[0]] * 8)
        assert np.all(ko.f16_value(c.dbits[w][0, 0, :6]) == 4.0)


def test_outlier_only_vectors_are_q8_0_alone():
    """x_rest = 0: the body holds all-zero blocks and what attention sees is
    the q8_0 round trip of the outlier values at their channels."""
    rng = np.random.default_rng(1)
    d, n, H = 128, 9, 2
    oidx = np.stack([np.sort(rng.choice(d, 32, replace=False)) for _ in range(H)])
    x = np.zeros((1, n, H, d), F32)
    for h in range(H):
        x[0, :, h][:, oidx[h]] = rng.standard_normal((n, 32)).astype(F32) * 10
    c = ko.OracleCache(1, H, d, 16, 0, "q4_0", "q5_1", True, True, outliers=oidx)
    c.append(x, x)
    R = ko.rotation_matrix(d)
    for h in range(H):
        db, cd = ko.quantize_q8_0(x[0, :, h][:, oidx[h]])
        want = np.zeros((n, d))
        want[:, oidx[h]] = ko.dequantize("q8_0", db, cd)
        for w in ("k", "v"):
            assert np.max(np.abs(c.stored(w, 0, h) @ R - want)) < 1e-9
    assert np.all(ko.f16_value(c.dbits["k"][0, :, :n]) == 0)       # q4_0 all-zero blocks


def test_zero_outlier_channels_give_the_plain_cache():
    rng = np.random.default_rng(2)
    d, n, H, T = 128, 20, 2, 4
    oidx = np.stack([np.sort(rng.choice(d, 32, replace=False)) for _ in range(H)])
    x = rng.standard_normal((2, n, H, d)).astype(F32)
    for h in range(H):
        x[:, :, h][..., oidx[h]] = 0.0
    a = ko.OracleCache(2, H, d, 32, T, "q5_0", "q8_0", True, True, outliers=oidx)
    b = ko.OracleCache(2, H, d, 32, T, "q5_0", "q8_0", True, True)
    a.append(x, x * 0.5)
    b.append(x, x * 0.5)
    for w in ("k", "v"):
        assert np.array_equal(a.codes[w], b.codes[w]) and np.array_equal(a.dbits[w], b.dbits[w])
        assert np.array_equal(a.tail[w], b.tail[w])
        assert not a.ocodes[w].any() and not a.odbits[w].any()
    q = rng.standard_normal((2, H * 3, d))
    assert np.max(np.abs(ko.decode_attention(a, q) - ko.decode_attention(b, q))) < 1e-12


def test_decode_bruteforce_in_the_original_basis():
    """Attention with the rotated query over the rotated stored values, rotated
    back, equals textbook attention of q over k_hat, v_hat in the original basis."""
    rng = np.random.default_rng(3)
    B, H, g, d, T = 2, 2, 2, 64, 3
    oidx = np.stack([np.sort(rng.choice(d, 32, replace=False)) for _ in range(H)])
    c = ko.OracleCache(B, H, d, 32, T, "q4_0", "q8_0", True, True, outliers=oidx)
    k = rng.standard_normal((B, 11, H, d)).astype(F32)
    v = rng.standard_normal((B, 11, H, d)).astype(F32)
    k[..., 7] *= 25
    c.append(k, v, n_new_per_seq=[11, 6])
    q = rng.standard_normal((B, H * g, d))
    out = ko.decode_attention(c, q)
    R = ko.rotation_matrix(d)
    for b in range(B):
        for hq in range(H * g):
            kv = hq // g
            Ks = [list(r) for r in c.stored("k", b, kv) @ R]
            Vs = [list(r) for r in c.stored("v", b, kv) @ R]
            o = np.array(_loops_attention(list(q[b, hq]), Ks, Vs, 1 / 8.0))
            assert np.max(np.abs(out[b, hq] - o)) < 1e-12


def test_tail_keeps_the_whole_rotated_vector():
    rng = np.random.default_rng(4)
    d, n, T = 64, 10, 16
    oidx = np.arange(0, 64, 2)[None, :]
    x = rng.standard_normal((1, n, 1, d)).astype(F32)
    a = ko.OracleCache(1, 1, d, 16, T, "q4_0", "q4_0", True, True, outliers=oidx)
    b = ko.OracleCache(1, 1, d, 16, T, "q4_0", "q4_0", True, True)
    a.append(x, x)
    b.append(x, x)
    assert np.array_equal(a.tail["k"], b.tail["k"]) and np.array_equal(a.tail["v"], b.tail["v"])
    q = rng.standard_normal((1, 1, d))
    assert np.max(np.abs(ko.decode_attention(a, q) - ko.decode_attention(b, q))) < 1e-12


@pytest.mark.parametrize("qtype", ["q4_0", "q5_0", "q8_0", "q4_1", "q5_1"])
def test_reconstruction_error_within_the_two_quantizations(qtype):
    """||k_hat - x|| <= ||e_rest|| + ||e_O||: the error of the rotated rest (the
    rotation keeps its norm) plus the q8_0 error of the outlier values."""
    rng = np.random.default_rng(5)
    d, n = 128, 16
    oidx = np.sort(rng.choice(d, 32, replace=False))[None, :]
    x = rng.standard_normal((1, n, 1, d)).astype(F32)
    x[..., oidx[0, :3]] *= 40
    c = ko.OracleCache(1, 1, d, 16, 0, qtype, qtype, True, True, outliers=oidx)
    c.append(x, x)
    plain = ko.OracleCache(1, 1, d, 16, 0, qtype, qtype, True, True)
    plain.append(x, x)
    R = ko.rotation_matrix(d)
    rest = x[0, :, 0].copy()
    rest[:, oidx[0]] = 0
    yr = ko.rotate(rest).astype(F32)
    db, cd = ko.quantize(qtype, yr)
    e_rest = np.linalg.norm(ko.dequantize(qtype, db, cd) - yr, axis=-1)
    xo = x[0, :, 0][:, oidx[0]]
    ob, oc = ko.quantize_q8_0(xo)
    e_o = np.linalg.norm(ko.dequantize("q8_0", ob, oc) - xo, axis=-1)
    err = np.linalg.norm(c.stored("k", 0, 0) @ R - x[0, :, 0], axis=-1)
    assert np.all(err <= e_rest + e_o + 1e-9)
    assert np.all(err >= np.abs(e_rest - e_o) - 1e-9)
    # at 4 bits the planted outliers dominate the plain cache's error, not this
    # one's (at 8 bits the coarser q8_0 block of the outliers can cost more)
    err_plain = np.linalg.norm(plain.stored("k", 0, 0) @ R - x[0, :, 0], axis=-1)
    if qtype in ("q4_0", "q4_1"):
        assert np.mean(err) < np.mean(err_plain)


def test_outlier_arguments_rejected():
    with pytest.raises(ValueError):   # not strictly increasing
        ko.OracleCache(1, 1, 64, 16, 0, "q4_0", "q4_0", True, True, outliers=[[1] * 32])
    with pytest.raises(ValueError):   # O not a multiple of 32
        ko.OracleCache(1, 1, 64, 16, 0, "q4_0", "q4_0", True, True, outliers=[list(range(16))])
    with pytest.raises(ValueError):   # channel out of range
        ko.OracleCache(1, 1, 64, 16, 0, "q4_0", "q4_0", True, True, outliers=[list(range(40, 72))])
    c = ko.OracleCache(1, 1, 64, 16, 0, "q4_0", "q4_0", True, True, outliers=[list(range(32))])
    with pytest.raises(ValueError):   # outliers are picked in the original basis
        c.append(np.zeros((1, 1, 1, 64), F32), np.zeros((1, 1, 1, 64), F32), prerotated=True)
