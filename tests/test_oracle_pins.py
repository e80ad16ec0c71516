"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: hand-worked
golden values, closed forms, invariants, brute force, or a library routine
(numpy / torch) for a special case.  No GPU needed.
"""

import json
import math

import numpy as np
import pytest

from oracle import kvq_oracle as ko
from rotated_bit_kv_kvq_gb300 import workloads as wl
from conftest import golden_path


def _golden(name):
    with open(golden_path(name)) as f:
        return json.load(f)


def _dense(block_spec, default):
    out = np.full(32, default, dtype=np.float64)
    for k, v in block_spec.items():
        out[int(k)] = v
    return out


# ---------------------------------------------------------------- rotation

def test_sylvester_golden():
    g = _golden("hadamard.json")
    assert np.array_equal(ko.sylvester_hadamard(2), np.array(g["H2"]))
    assert np.array_equal(ko.sylvester_hadamard(4), np.array(g["H4"]))
    h8 = ko.sylvester_hadamard(8)
    assert np.array_equal(h8[3], np.array(g["H8_row3"]))
    assert np.array_equal(h8[5], np.array(g["H8_row5"]))


def test_rotate_golden_vectors():
    g = _golden("hadamard.json")
    r4 = ko.sylvester_hadamard(4) / 2.0
    for case in g["rotate4"]:
        x = np.array(case["x"], dtype=np.float64)
        assert np.allclose(x @ r4, case["y"], atol=1e-15)
        assert np.allclose(ko.fwht(x, 4), case["y"], atol=1e-15)


@pytest.mark.parametrize("d", [64, 128, 256, 512, 192, 320])
def test_rotation_orthonormal_symmetric(d):
    r = ko.rotation_matrix(d)
    assert np.max(np.abs(r @ r.T - np.eye(d))) < 1e-14
    assert np.array_equal(r, r.T)
    # entries are +-1/sqrt(G) inside the Hadamard blocks and 0 outside
    g = ko.rotation_group(d)
    nz = np.abs(r[r != 0])
    assert np.allclose(nz, 1 / math.sqrt(g))
    assert np.count_nonzero(r) == d * g


@pytest.mark.parametrize("d", [64, 128, 256, 192, 320])
def test_fwht_equals_matrix_product(d):
    rng = np.random.default_rng(1)
    x = rng.standard_normal((7, d))
    assert np.max(np.abs(ko.fwht(x, ko.rotation_group(d)) - ko.rotate(x))) < 1e-12


def test_hadamard_is_self_inverse_transform():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((5, 256))
    assert np.max(np.abs(ko.rotate(ko.rotate(x)) - x)) < 1e-12


@pytest.mark.parametrize("d", [64, 128, 256, 192])
def test_dot_products_preserved(d):
    """Orthogonal rotation keeps q.k (velog 아다마르 회전: the score is a dot product)."""
    rng = np.random.default_rng(3)
    q = rng.standard_normal((9, d)) * 3
    k = rng.standard_normal((11, d))
    k[:, :3] *= 20
    a = q @ k.T
    b = ko.rotate(q) @ ko.rotate(k).T
    assert np.max(np.abs(a - b) / (np.abs(a) + 1)) < 1e-12


def test_exact_attention_same_with_and_without_rotation():
    """Unquantized attention in the rotated basis, rotated back, equals plain attention."""
    rng = np.random.default_rng(4)
    d = 128
    q = rng.standard_normal((4, d))
    K = rng.standard_normal((300, d)); K[:, [5, 77]] *= 20
    V = rng.standard_normal((300, d)); V[:, [9]] *= 20
    s = ko.default_scale(d)
    plain = ko.softmax_attention(q, K, V, s)
    rot = ko.rotate(ko.softmax_attention(ko.rotate(q), ko.rotate(K), ko.rotate(V), s))
    assert np.max(np.abs(plain - rot)) < 1e-12


def test_enable_rule():
    assert ko.rotation_enabled(64) and ko.rotation_enabled(128) and ko.rotation_enabled(192)
    assert not ko.rotation_enabled(32) and not ko.rotation_enabled(96) and not ko.rotation_enabled(80)
    assert ko.rotation_group(192) == 64 and ko.rotation_group(256) == 256
    with pytest.raises(ValueError):
        ko.rotation_group(96)


# ------------------------------------------------------------ fp16 / bf16

def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * 100,
        # exact ties: low 16 bits 0x8000 with even and odd upper halves
        (np.arange(1000, dtype=np.uint32) << 16 | 0x8000).view(np.float32) + 0,
        np.array([0.0, -0.0, 1e-40, -3e38, 3.3e38], dtype=np.float32),
    ]).astype(np.float32)
    x = x[np.isfinite(x)]
    ours = ko.bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_f16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(6)
    x = np.concatenate([rng.standard_normal(20000) * 10, rng.standard_normal(2000) * 1e-6,
                        [2.0 ** -24 * 1.5, 2.0 ** -25, 65519.0, 1 / 127]]).astype(np.float32)
    ours = ko.f16_bits(x)
    ref = torch.from_numpy(x).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


# ------------------------------------------------------------ quantizers

def test_golden_blocks():
    g = _golden("quant_blocks.json")
    for blk in g["blocks"]:
        x = _dense(blk["x"], 0.0).astype(np.float32)
        dbits, codes = ko.quantize(blk["type"], x)
        exp_codes = _dense(blk["codes"], blk["default_code"]).astype(np.int64)
        assert int(dbits[0]) == blk["d_bits"], blk["name"]
        assert np.array_equal(codes[0].astype(np.int64), exp_codes), blk["name"]


def _random_blocks(rng, n, outliers=True):
    x = rng.standard_normal((n, 32)).astype(np.float32)
    if outliers:
        x[::3, 5] *= 20
        x[1::3] *= np.float32(1e-3)
    return x


def _d_exact(qtype, x):
    """The float32 scale d before fp16 rounding, restated from the definition."""
    xf = x.astype(np.float32)
    if qtype == "q8_0":
        return (np.max(np.abs(xf), axis=-1) / np.float32(127)).astype(np.float64)
    idx = np.argmax(np.abs(xf), axis=-1)
    m = xf[np.arange(len(xf)), idx]
    return (m / np.float32(-8 if qtype == "q4_0" else -16)).astype(np.float64)


@pytest.mark.parametrize("qtype", ["q8_0", "q4_0", "q5_0"])
def test_quantizer_error_bounds(qtype):
    """|x - deq(q(x))| <= |d|/2 off the clamp (|d| on the clamped code), plus
    the fp16 rounding of d times the code magnitude and a few ulps."""
    rng = np.random.default_rng(7)
    x = _random_blocks(rng, 4000)
    dbits, codes = ko.quantize(qtype, x)
    deq = ko.dequantize(qtype, dbits, codes).reshape(-1, 32)
    d = _d_exact(qtype, x)[:, None]
    D = ko.f16_value(dbits).reshape(-1, 1)
    off = {"q8_0": 0, "q4_0": 8, "q5_0": 16}[qtype]
    top = {"q8_0": 127, "q4_0": 15, "q5_0": 31}[qtype]
    c = codes.reshape(-1, 32).astype(np.float64) - off
    slack = np.abs(c) * np.abs(d - D) + np.abs(d) * 1e-5 + 1e-30
    err = np.abs(x.astype(np.float64) - deq)
    clamped = (codes.reshape(-1, 32) == top) & (qtype != "q8_0")
    bound = np.where(clamped, np.abs(d), np.abs(d) / 2) + slack
    assert np.all(err <= bound)
    if qtype != "q8_0":
        # the clamp only hits values of the same sign as d, i.e. opposite to m
        xs = np.broadcast_to(x.astype(np.float64), clamped.shape)
        ds = np.broadcast_to(d, clamped.shape)
        assert np.all(np.sign(xs[clamped]) == np.sign(ds[clamped]))


@pytest.mark.parametrize("qtype", ["q4_0", "q5_0"])
def test_max_element_round_trips(qtype):
    """The element of largest magnitude gets code 0, i.e. deq = -8*D (-16*D) = m up to D rounding."""
    rng = np.random.default_rng(8)
    x = _random_blocks(rng, 2000)
    dbits, codes = ko.quantize(qtype, x)
    idx = np.argmax(np.abs(x), axis=-1)
    c = codes.reshape(-1, 32)
    assert np.all(c[np.arange(len(x)), idx] == 0)


@pytest.mark.parametrize("qtype", ["q8_0", "q4_0", "q5_0"])
def test_codes_are_nearest_levels_bruteforce(qtype):
    """Brute force over every code: the chosen one is a nearest level of
    (code - offset) * d to x, except the clamped top code of q4_0/q5_0."""
    rng = np.random.default_rng(9)
    x = _random_blocks(rng, 600)
    dbits, codes = ko.quantize(qtype, x)
    codes = codes.reshape(-1, 32).astype(np.int64)
    d = _d_exact(qtype, x)
    off = {"q8_0": 0, "q4_0": 8, "q5_0": 16}[qtype]
    levels = {"q8_0": np.arange(-127, 128), "q4_0": np.arange(16), "q5_0": np.arange(32)}[qtype]
    top = levels[-1]
    for i in range(len(x)):
        if d[i] == 0:
            continue
        for j in range(32):
            dist = np.abs(x[i, j] - (levels - off) * d[i])
            best = dist.min()
            chosen = codes[i, j]
            if qtype != "q8_0" and chosen == top and x[i, j] / d[i] + off > top + 0.5:
                continue  # clamped: the nearest level lies beyond the code range
            k = int(np.where(levels == chosen)[0][0])
            assert dist[k] <= best + abs(d[i]) * 1e-6, (qtype, i, j)


@pytest.mark.parametrize("qtype,zero_bits,zero_code", [("q8_0", 0x0000, 0), ("q4_0", 0x8000, 8), ("q5_0", 0x8000, 16)])
def test_all_zero_block(qtype, zero_bits, zero_code):
    dbits, codes = ko.quantize(qtype, np.zeros((3, 64), np.float32))
    assert np.all(dbits == zero_bits)
    assert np.all(codes == zero_code)
    assert np.all(ko.dequantize(qtype, dbits, codes) == 0)


# ---- scale + minimum formats (q4_1 / q5_1)

def _lo_d_exact(qtype, x):
    """float32 lo and d = (hi - lo)/top before fp16 rounding, restated from the definition."""
    xf = x.astype(np.float32)
    lo = xf.min(axis=-1)
    top = 15 if qtype == "q4_1" else 31
    return lo.astype(np.float64), ((xf.max(axis=-1) - lo) / np.float32(top)).astype(np.float64), top


@pytest.mark.parametrize("qtype", ["q4_1", "q5_1"])
def test_min_quantizer_error_bounds(qtype):
    """|x - (code*D + M)| <= d/2 + code*|d - D| + |lo - M| (+ ulps): every code is the
    rounded position of x on the grid lo + k*d, and the grid fits the block exactly."""
    rng = np.random.default_rng(17)
    x = _random_blocks(rng, 4000)
    word, codes = ko.quantize(qtype, x)
    deq = ko.dequantize(qtype, word, codes).reshape(-1, 32)
    lo, d, top = _lo_d_exact(qtype, x)
    D, M = ko.scale_and_min(qtype, word)
    c = codes.reshape(-1, 32).astype(np.float64)
    assert c.max() <= top
    slack = c * np.abs(d - D.reshape(-1))[:, None] + np.abs(lo - M.reshape(-1))[:, None] \
        + (np.abs(d) * 1e-5 + np.abs(lo) * 1e-6)[:, None] + 1e-30
    err = np.abs(x.astype(np.float64) - deq)
    assert np.all(err <= (d / 2)[:, None] + slack)


@pytest.mark.parametrize("qtype", ["q4_1", "q5_1"])
def test_min_quantizer_extremes(qtype):
    """The smallest value gets code 0 and the largest the top code (the grid spans the block)."""
    rng = np.random.default_rng(18)
    x = _random_blocks(rng, 2000)
    word, codes = ko.quantize(qtype, x)
    c = codes.reshape(-1, 32)
    top = 15 if qtype == "q4_1" else 31
    rows = np.arange(len(x))
    assert np.all(c[rows, np.argmin(x, axis=-1)] == 0)
    assert np.all(c[rows, np.argmax(x, axis=-1)] == top)


@pytest.mark.parametrize("qtype", ["q4_1", "q5_1"])
def test_min_codes_are_nearest_levels_bruteforce(qtype):
    """Brute force over every code: the chosen one is a nearest grid level lo + k*d."""
    rng = np.random.default_rng(19)
    x = _random_blocks(rng, 600)
    word, codes = ko.quantize(qtype, x)
    codes = codes.reshape(-1, 32).astype(np.int64)
    lo, d, top = _lo_d_exact(qtype, x)
    levels = np.arange(top + 1)
    for i in range(len(x)):
        if d[i] == 0:
            assert np.all(codes[i] == 0)
            continue
        for j in range(32):
            dist = np.abs(x[i, j] - (lo[i] + levels * d[i]))
            assert dist[codes[i, j]] <= dist.min() + abs(d[i]) * 1e-5, (qtype, i, j)


@pytest.mark.parametrize("qtype", ["q4_1", "q5_1"])
def test_min_constant_and_zero_blocks(qtype):
    x = np.zeros((3, 64), np.float32)
    x[1] = -2.5
    word, codes = ko.quantize(qtype, x)
    assert np.all(codes == 0)
    assert np.all((word & 0xFFFF) == 0)
    assert np.array_equal(ko.dequantize(qtype, word, codes), x.astype(np.float64))


def test_signed_max_first_index_on_ties():
    x = np.zeros((3, 32), np.float32)
    x[0, [4, 9]] = [5, -5]
    x[1, [4, 9]] = [-5, 5]
    x[2, :] = -0.0
    m, amax = ko.signed_max_magnitude(x)
    assert m[0] == 5 and m[1] == -5 and amax[0] == 5
    assert m[2] == 0 and not np.signbit(m[2])


# ------------------------------------------------------------ packing

def test_packing_golden():
    g = _golden("packing.json")
    c = np.array(g["q4_0_codes_up_down"]["codes"], np.uint8)
    assert ko.pack_q4_0(c).tobytes().hex() == g["q4_0_codes_up_down"]["qs_hex"]
    for key in ("q5_0_codes_0_to_31", "q5_0_alternating_high"):
        c = np.array(g[key]["codes"], np.uint8)
        qs, qh = ko.pack_q5_0(c)
        assert qs.tobytes().hex() == g[key]["qs_hex"]
        assert int(qh) == g[key]["qh"]
    for key, qt in (("ggml_q4_0_block", "q4_0"), ("ggml_q5_0_block", "q5_0"), ("ggml_q8_0_block", "q8_0"),
                    ("ggml_q4_1_block", "q4_1"), ("ggml_q5_1_block", "q5_1")):
        e = g[key]
        codes = np.array(e["codes"], np.int64).astype(np.int8 if qt == "q8_0" else np.uint8)[None]
        word = np.uint32 if qt in ko.MIN_TYPES else np.uint16
        b = ko.to_ggml_bytes(qt, np.array([e["d_bits"]], word), codes)
        assert b.tobytes().hex() == e["bytes_hex"], key
        assert b.shape[-1] == ko.GGML_BLOCK_BYTES[qt]


def test_pack_round_trip():
    rng = np.random.default_rng(10)
    c4 = rng.integers(0, 16, (50, 32)).astype(np.uint8)
    assert np.array_equal(ko.unpack_q4_0(ko.pack_q4_0(c4)), c4)
    c5 = rng.integers(0, 32, (50, 32)).astype(np.uint8)
    qs, qh = ko.pack_q5_0(c5)
    assert np.array_equal(ko.unpack_q5_0(qs, qh), c5)


# ------------------------------------------------------------ benefit of rotation

def _c1_like(seed):
    w = wl.WORKLOADS["decode_d64_ctx256"]
    inp = wl.make_inputs(w, seed)
    return w, inp


def _rotation_errors(seed):
    """(reconstruction MSE of K+V, attention-output rel-L2) for q4_0 without
    and with rotation, on the 64-channel outlier workload with its query."""
    w, inp = _c1_like(seed)
    K = inp.k_hist[0, :, 0]  # [n][64]
    V = inp.v_hist[0, :, 0]
    q = inp.q[0, 0]
    res = {}
    for rot in (False, True):
        errs = []
        recon = {}
        for name, X in (("k", K), ("v", V)):
            Y = ko.rotate(X).astype(np.float32) if rot else X.astype(np.float32)
            dbits, codes = ko.quantize_q4_0(Y)
            deq = ko.dequantize("q4_0", dbits, codes)
            back = ko.rotate(deq) if rot else deq
            recon[name] = back
            errs.append(np.mean((back - X) ** 2))
        out = ko.softmax_attention(q[None], recon["k"], recon["v"], ko.default_scale(64))[0]
        exact = ko.softmax_attention(q[None], K, V, ko.default_scale(64))[0]
        res[rot] = (sum(errs), np.linalg.norm(out - exact) / np.linalg.norm(exact))
    return res


def test_rotation_lowers_q4_error():
    """velog 아다마르 회전: rotation spreads the outlier channels, so 4-bit
    blocks lose much less.  Direction pin on the outlier workload, seeds 0..9:
    the block reconstruction error drops on every seed; the attention-output
    error drops on average and on at least 9 of the 10 seeds (with the query
    sharing K's outlier channels, one seed's single query is better served by
    the unrotated blocks, whose scale is set by those very channels)."""
    res = [_rotation_errors(s) for s in range(10)]
    assert all(r[True][0] < r[False][0] for r in res)
    assert all(r[True][0] < 0.5 * r[False][0] for r in res)
    wins = sum(r[True][1] < r[False][1] for r in res)
    assert wins >= 9
    assert np.mean([r[True][1] for r in res]) < 0.5 * np.mean([r[False][1] for r in res])


# ------------------------------------------------------------ cache, tail, attention

def _tiny_cache(rng, T, k_type="q4_0", v_type="q8_0", B=2, H=2, d=64, max_ctx=128, rot=True):
    return ko.OracleCache(B, H, d, max_ctx, T, k_type, v_type, rot, rot)


def test_tail_covering_everything_is_bf16_attention():
    """T >= n: every key/value is the bf16 rounding of its rotated input."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(11)
    B, H, d, n, g = 1, 2, 64, 40, 3
    c = ko.OracleCache(B, H, d, 64, 64, "q4_0", "q4_0", True, True)
    k = rng.standard_normal((B, n, H, d)).astype(np.float32)
    v = rng.standard_normal((B, n, H, d)).astype(np.float32)
    c.append(k, v)
    q = rng.standard_normal((B, H * g, d))
    out = ko.decode_attention(c, q)
    R = ko.rotation_matrix(d)
    for h in range(H * g):
        kr = torch.from_numpy((k[0, :, h // g] @ R).astype(np.float32)).to(torch.bfloat16).double().numpy()
        vr = torch.from_numpy((v[0, :, h // g] @ R).astype(np.float32)).to(torch.bfloat16).double().numpy()
        ref = ko.softmax_attention((q[0, h] @ R)[None], kr, vr, 1 / 8.0)[0] @ R
        assert np.max(np.abs(out[0, h] - ref)) < 1e-12


def test_tail_zero_is_body_only():
    rng = np.random.default_rng(12)
    B, H, d, n = 1, 1, 128, 50
    c = ko.OracleCache(B, H, d, 64, 0, "q8_0", "q5_0", True, True)
    k = rng.standard_normal((B, n, H, d)).astype(np.float32)
    v = rng.standard_normal((B, n, H, d)).astype(np.float32)
    c.append(k, v)
    q = rng.standard_normal((B, H, d))
    R = ko.rotation_matrix(d)
    dk, ck = ko.quantize_q8_0((k[0, :, 0] @ R).astype(np.float32))
    dv, cv = ko.quantize_q5_0((v[0, :, 0] @ R).astype(np.float32))
    ref = ko.softmax_attention((q[0] @ R), ko.dequantize("q8_0", dk, ck), ko.dequantize("q5_0", dv, cv),
                               1 / math.sqrt(d)) @ R
    assert np.max(np.abs(ko.decode_attention(c, q)[0] - ref)) < 1e-12


def test_tail_ring_wraparound_many_appends():
    """Many small appends: the last T positions come from ring slots pos % T
    holding bf16 of the rotated inputs; older positions from the body."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(13)
    B, H, d, T = 2, 1, 64, 16
    c = ko.OracleCache(B, H, d, 256, T, "q4_0", "q4_0", True, True)
    R = ko.rotation_matrix(d)
    allk = [[], []]
    for step in range(23):
        nn = [int(rng.integers(0, 6)), int(rng.integers(0, 6))]
        k = rng.standard_normal((B, 5, H, d)).astype(np.float32)
        v = rng.standard_normal((B, 5, H, d)).astype(np.float32)
        c.append(k, v, n_new_per_seq=nn)
        for b in range(B):
            allk[b].extend(list(k[b, :nn[b], 0]))
    for b in range(B):
        n = int(c.seq_len[b])
        assert n == len(allk[b])
        st = c.stored("k", b, 0)
        for t in range(n):
            y = (allk[b][t] @ R).astype(np.float32)
            if t >= n - T:
                exp = torch.from_numpy(y).to(torch.bfloat16).double().numpy()
            else:
                db, cd = ko.quantize_q4_0(y)
                exp = ko.dequantize("q4_0", db, cd)
            assert np.array_equal(st[t], exp)


def _loops_attention(qv, Ks, Vs, scale):
    """Pure-Python softmax attention of one query vector."""
    s = [scale * sum(qv[c] * K[c] for c in range(len(qv))) for K in Ks]
    if not s:
        return [0.0] * len(qv)
    mx = max(s)
    e = [math.exp(x - mx) for x in s]
    tot = sum(e)
    return [sum(e[t] / tot * Vs[t][c] for t in range(len(Vs))) for c in range(len(qv))]


def test_decode_gqa_bruteforce():
    rng = np.random.default_rng(14)
    B, H, g, d, T = 2, 2, 3, 64, 5
    c = ko.OracleCache(B, H, d, 64, T, "q5_0", "q4_0", True, True)
    k = rng.standard_normal((B, 12, H, d)).astype(np.float32)
    v = rng.standard_normal((B, 12, H, d)).astype(np.float32)
    c.append(k, v, n_new_per_seq=[12, 7])
    q = rng.standard_normal((B, H * g, d))
    out = ko.decode_attention(c, q)
    R = ko.rotation_matrix(d)
    for b in range(B):
        for h in range(H * g):
            kv = h // g
            Ks = [list(r) for r in c.stored("k", b, kv)]
            Vs = [list(r) for r in c.stored("v", b, kv)]
            o = np.array(_loops_attention(list(q[b, h] @ R), Ks, Vs, 1 / 8.0)) @ R
            assert np.max(np.abs(out[b, h] - o)) < 1e-12


def test_prefill_causal_bruteforce_and_decode_consistency():
    rng = np.random.default_rng(15)
    B, H, g, d, T, n = 2, 1, 2, 64, 4, 9
    c = ko.OracleCache(B, H, d, 64, T, "q8_0", "q4_0", True, True)
    k = rng.standard_normal((B, n, H, d)).astype(np.float32)
    v = rng.standard_normal((B, n, H, d)).astype(np.float32)
    c.append(k, v)
    q = rng.standard_normal((B, 6, H * g, d))
    out = ko.prefill_attention(c, q, causal=True)
    R = ko.rotation_matrix(d)
    for b in range(B):
        Ks = [list(r) for r in c.stored("k", b, 0)]
        Vs = [list(r) for r in c.stored("v", b, 0)]
        for i in range(6):
            p = n - 6 + i
            for h in range(H * g):
                o = np.array(_loops_attention(list(q[b, i, h] @ R), Ks[:p + 1], Vs[:p + 1], 1 / 8.0)) @ R
                assert np.max(np.abs(out[b, i, h] - o)) < 1e-12
    # the last prompt row sees every key, like a decode step with the same query
    dec = ko.decode_attention(c, q[:, -1])
    assert np.max(np.abs(dec - out[:, -1])) < 1e-12
    # non-causal: every row equals the decode result for its query
    nc = ko.prefill_attention(c, q, causal=False)
    for i in range(6):
        assert np.max(np.abs(nc[:, i] - ko.decode_attention(c, q[:, i]))) < 1e-12


def test_rotation_switches():
    """K rotation off: q is not rotated and K is stored as is; V rotation off:
    no inverse rotation.  With exact (tail) storage every switch combination
    gives the same attention result up to bf16 rounding."""
    rng = np.random.default_rng(16)
    d, n = 64, 20
    k = rng.standard_normal((1, n, 1, d)).astype(np.float32)
    v = rng.standard_normal((1, n, 1, d)).astype(np.float32)
    q = rng.standard_normal((1, 1, d))
    outs = []
    for rk in (False, True):
        for rv in (False, True):
            c = ko.OracleCache(1, 1, d, 64, 64, "q4_0", "q4_0", rk, rv)
            c.append(k, v)
            outs.append(ko.decode_attention(c, q))
            sk = c.stored("k", 0, 0)
            assert np.max(np.abs(sk - (ko.rotate(k[0, :, 0]) if rk else k[0, :, 0]))) < 0.05
    for o in outs[1:]:
        assert np.max(np.abs(o - outs[0])) < 2e-2


def test_empty_sequence_gives_zeros():
    c = ko.OracleCache(2, 1, 64, 64, 4, "q4_0", "q4_0", True, True)
    k = np.ones((2, 3, 1, 64), np.float32)
    c.append(k, k, n_new_per_seq=[0, 3])
    out = ko.decode_attention(c, np.ones((2, 1, 64)))
    assert np.all(out[0] == 0) and np.any(out[1] != 0)


def test_append_rejects_overflow():
    c = ko.OracleCache(1, 1, 64, 64, 4, "q4_0", "q4_0", True, True)
    with pytest.raises(ValueError):
        c.append(np.zeros((1, 65, 1, 64), np.float32), np.zeros((1, 65, 1, 64), np.float32))
