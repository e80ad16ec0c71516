"""Plain CPU oracle: rotated, block-quantized KV cache and exact attention over it.

TEST INFRASTRUCTURE ONLY -- used by ``tests/``, ``__graft_entry__.smoke()`` and
the CPU legs of ``bench.py``; never by the product path.  It shares no code
with the CUDA library.

Sources (pages are cited by title and section):

* [P1] velog post "fix-kv-cache-quantization-outliers" (llama.cpp KV rotation
  patch).  Section "아다마르 회전" (Hadamard rotation): Q, K and V are multiplied
  by a normalized Hadamard matrix and stored rotated; after attention the
  result is rotated back; the Hadamard matrix is orthogonal so dot products
  (and hence attention scores) are unchanged; the GGUF block formats are not
  changed.  Section "적용 및 배경 기술" (application): rotation switches on
  automatically when head_dim >= 64 and a multiple of 64, and K / V rotation
  can each be switched off.
* [P2] aitrends.kr summary "KV 캐시 양자화 벤치마크: KVarN과 Precision Tail",
  sections "섹션별 상세" and "용어 해설" (Precision Tail): the most recent X
  tokens are kept in BF16, the rest in the low-bit format.
* The q8_0 / q5_0 / q4_0 blocks are the GGUF block formats [P1] says stay
  unchanged: 32 values per block with an fp16 scale.  q8_0 scale = amax/127,
  codes round-half-away-from-zero; q5_0 / q4_0 scale = (signed value of
  largest magnitude) / -16 or -8, codes = trunc(x/scale + 16.5 or 8.5)
  clamped to 31 or 15.
* q4_1 / q5_1 (scale + minimum), which [P2] benchmarks beside them (its
  tables of K/V type pairs, e.g. q5_0-q4_1 and q8_0-q5_1, section "섹션별
  상세"): 32 values, fp16 scale d = (max - min) / 15 or 31 and fp16 minimum;
  codes = min(top, trunc((x - min) / d + 0.5)); value = code * d + min.  The
  pages name these types without restating them; the reading is the GGUF
  definition of the same names, as for the _0 types.

* Outlier channels kept at 8 bits ([P1] section "적용 및 배경 기술" names, as a
  direction of the work the patch comes from, mixed precision that keeps only
  the outlier channels at 8 bits; it gives no selection rule, count or
  interplay with the rotation).  Reading used here: per KV head the caller
  names O channels (O a multiple of 32) of the *original* basis.  On the
  write path those O values are stored as q8_0 blocks, unrotated, in slot
  order (increasing channel); they are set to zero in the vector, and the
  rest is rotated and quantized in the cache's format as before.  The bf16
  tail keeps the whole rotated vector.  What attention sees for a body
  position is the rotated, dequantized rest plus the rotated scatter of the
  dequantized outlier values -- in the original basis,
  k_hat = R^T deq(R k_rest) + scatter(deq8(k_O)), which is k up to the two
  quantization errors.

Precision: rotation and attention in float64; quantizer arithmetic in IEEE
float32 exactly as the block definition states (one rounding per operation,
no fused multiply-add); fp16 and bf16 round-to-nearest-even.

Parity pins (tests/test_oracle_pins.py and tests/test_oracle_outliers.py):
every function below is pinned by closed forms, invariants, brute force or
hand-worked golden values; tests/test_oracle_mutations.py plants plausible
mistakes in these functions and checks that a pin fails for each.  No
function is "parity unpinned".
"""

from __future__ import annotations

import math

import numpy as np

F32 = np.float32
F64 = np.float64

QK = 32  # values per quantization block

TYPE_Q4_0 = "q4_0"
TYPE_Q5_0 = "q5_0"
TYPE_Q8_0 = "q8_0"
TYPE_Q4_1 = "q4_1"
TYPE_Q5_1 = "q5_1"
TYPES = (TYPE_Q4_0, TYPE_Q5_0, TYPE_Q8_0, TYPE_Q4_1, TYPE_Q5_1)
MIN_TYPES = (TYPE_Q4_1, TYPE_Q5_1)   # scale + minimum per block

# bytes of one block in the GGUF array-of-structs layout: scale (+ minimum) + payload
GGML_BLOCK_BYTES = {TYPE_Q4_0: 18, TYPE_Q5_0: 22, TYPE_Q8_0: 34, TYPE_Q4_1: 20, TYPE_Q5_1: 24}


# ---------------------------------------------------------------------------
# Hadamard rotation  ([P1] 아다마르 회전; enable rule from [P1] 적용 및 배경 기술)
# ---------------------------------------------------------------------------

def is_power_of_two(n: int) -> bool:
    return n > 0 and (n & (n - 1)) == 0


def sylvester_hadamard(n: int) -> np.ndarray:
    """Unnormalized Hadamard matrix in Sylvester order:
    H_1 = [1],  H_2n = [[H_n, H_n], [H_n, -H_n]]."""
    if not is_power_of_two(n):
        raise ValueError("Sylvester Hadamard needs a power-of-two size")
    h = np.ones((1, 1), dtype=F64)
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def rotation_enabled(head_dim: int) -> bool:
    """[P1] 적용 및 배경 기술: automatic when head_dim >= 64 and a multiple of 64."""
    return head_dim >= 64 and head_dim % 64 == 0


def rotation_group(head_dim: int) -> int:
    """Size of the Hadamard blocks used for one head.

    A power-of-two head_dim uses one H_d.  Any other multiple of 64 uses a
    block diagonal of H_64 blocks (the page only fixes "a multiple of 64";
    the 64-wide blocks are the plainest rotation that exists for every such
    size)."""
    if not rotation_enabled(head_dim):
        raise ValueError(f"head_dim {head_dim} is not eligible for rotation")
    return head_dim if is_power_of_two(head_dim) else 64


def rotation_matrix(head_dim: int) -> np.ndarray:
    """R = blockdiag(H_G / sqrt(G), ...): orthonormal and symmetric, so R^-1 = R."""
    g = rotation_group(head_dim)
    hg = sylvester_hadamard(g) / math.sqrt(g)
    r = np.zeros((head_dim, head_dim), dtype=F64)
    for i in range(head_dim // g):
        r[i * g:(i + 1) * g, i * g:(i + 1) * g] = hg
    return r


def rotate(x: np.ndarray) -> np.ndarray:
    """Row vectors x (last axis = head_dim) times R, in float64."""
    x = np.asarray(x, dtype=F64)
    return x @ rotation_matrix(x.shape[-1])


def fwht(x: np.ndarray, group: int) -> np.ndarray:
    """Fast Walsh-Hadamard transform of each `group`-wide slice of the last
    axis, normalized by 1/sqrt(group), in float64.

    Butterfly form of the same product as `rotate`: for h = 1, 2, 4, ...,
    each pair (j, j+h) inside every 2h-wide chunk becomes (a+b, a-b)."""
    y = np.array(x, dtype=F64, copy=True)
    shape = y.shape
    d = shape[-1]
    if d % group or not is_power_of_two(group):
        raise ValueError("bad FWHT group")
    h = 1
    while h < group:
        v = y.reshape(-1, d // group, group // (2 * h), 2, h)
        a = v[:, :, :, 0, :].copy()
        b = v[:, :, :, 1, :].copy()
        v[:, :, :, 0, :] = a + b
        v[:, :, :, 1, :] = a - b
        y = v.reshape(shape)
        h *= 2
    return y / math.sqrt(group)


# ---------------------------------------------------------------------------
# fp16 / bf16 rounding
# ---------------------------------------------------------------------------

def f16_bits(x) -> np.ndarray:
    """float32 -> IEEE binary16 bits, round to nearest even."""
    return np.asarray(x, dtype=F32).astype(np.float16).view(np.uint16)


def f16_value(bits) -> np.ndarray:
    return np.asarray(bits, dtype=np.uint16).view(np.float16).astype(F64)


def bf16_bits(x) -> np.ndarray:
    """float32 -> bfloat16 bits, round to nearest even (finite inputs)."""
    u = np.asarray(x, dtype=F32).view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_value(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(F32).astype(F64)


# ---------------------------------------------------------------------------
# Block quantizers (GGUF q8_0 / q5_0 / q4_0, which [P1] says are unchanged)
# ---------------------------------------------------------------------------

def _blocks(y: np.ndarray) -> np.ndarray:
    y = np.asarray(y, dtype=F32)
    if y.shape[-1] % QK:
        raise ValueError("last axis must be a multiple of 32")
    return y.reshape(y.shape[:-1] + (y.shape[-1] // QK, QK))


def signed_max_magnitude(blocks: np.ndarray):
    """Per block: the value with the largest |x|, the first one on ties
    (a strict '>' scan that starts from +0.0).  Returns (m, amax) in float32."""
    a = np.abs(blocks)
    idx = np.argmax(a, axis=-1)  # first occurrence of the maximum
    amax = np.take_along_axis(a, idx[..., None], axis=-1)[..., 0]
    m = np.take_along_axis(blocks, idx[..., None], axis=-1)[..., 0]
    # a block whose magnitudes are all zero never replaces the initial +0.0
    m = np.where(amax > 0, m, F32(0.0)).astype(F32)
    return m, amax.astype(F32)


def _inverse(d: np.ndarray) -> np.ndarray:
    """id = 1/d in float32, 0 where d == 0."""
    out = np.zeros_like(d, dtype=F32)
    nz = d != 0
    out[nz] = F32(1.0) / d[nz]
    return out


def _round_half_away(v: np.ndarray) -> np.ndarray:
    """roundf(): nearest integer, halves away from zero (evaluated exactly in float64)."""
    v64 = v.astype(F64)
    return np.sign(v64) * np.floor(np.abs(v64) + 0.5)


def quantize_q8_0(y):
    """q8_0: d = amax/127, codes = roundf(x * (1/d)) in [-127, 127], D = fp16(d).

    Returns (D bits uint16 [..., nb], codes int8 [..., nb, 32])."""
    b = _blocks(y)
    amax = np.max(np.abs(b), axis=-1).astype(F32)
    d = (amax / F32(127.0)).astype(F32)
    inv = _inverse(d)
    v = (b * inv[..., None]).astype(F32)
    codes = _round_half_away(v)
    assert np.all(np.abs(codes) <= 127)
    return f16_bits(d), codes.astype(np.int8)


def _quantize_offset(y, qmax_neg: float, offset: float, top: int):
    b = _blocks(y)
    m, _ = signed_max_magnitude(b)
    d = (m / F32(qmax_neg)).astype(F32)
    inv = _inverse(d)
    v = ((b * inv[..., None]).astype(F32) + F32(offset)).astype(F32)
    codes = np.minimum(top, np.trunc(v.astype(F64)))
    assert np.all(codes >= 0)
    return f16_bits(d), codes.astype(np.uint8)


def quantize_q4_0(y):
    """q4_0: d = m/-8, codes = min(15, trunc(x*(1/d) + 8.5)), D = fp16(d).

    Returns (D bits uint16 [..., nb], codes uint8 0..15 [..., nb, 32])."""
    return _quantize_offset(y, -8.0, 8.5, 15)


def quantize_q5_0(y):
    """q5_0: d = m/-16, codes = min(31, trunc(x*(1/d) + 16.5)), D = fp16(d).

    Returns (D bits uint16 [..., nb], codes uint8 0..31 [..., nb, 32])."""
    return _quantize_offset(y, -16.0, 16.5, 31)


def _quantize_min(y, top: int):
    """Scale + minimum blocks: lo / hi = smallest / largest value (float32; the
    first one in block order on ties, which only decides the sign of a zero
    minimum), d = (hi - lo) / top, id = 1/d (0 when d == 0), code = min(top,
    trunc((x - lo) * id + 0.5)) with one float32 rounding per operation.  Returns
    the scale word (fp16 bits of d in bits 0-15, of lo in bits 16-31) and the codes."""
    b = _blocks(y)
    lo = np.take_along_axis(b, np.argmin(b, axis=-1)[..., None], axis=-1)[..., 0].astype(F32)
    hi = np.take_along_axis(b, np.argmax(b, axis=-1)[..., None], axis=-1)[..., 0].astype(F32)
    d = ((hi - lo) / F32(top)).astype(F32)
    inv = _inverse(d)
    v = (((b - lo[..., None]).astype(F32) * inv[..., None]).astype(F32) + F32(0.5)).astype(F32)
    codes = np.minimum(top, np.trunc(v.astype(F64)))
    assert np.all(codes >= 0)
    word = f16_bits(d).astype(np.uint32) | (f16_bits(lo).astype(np.uint32) << np.uint32(16))
    return word, codes.astype(np.uint8)


def quantize_q4_1(y):
    """q4_1: d = (max - min)/15, codes = min(15, trunc((x - min)*(1/d) + 0.5)).

    Returns (scale word uint32 [..., nb]: fp16 d | fp16 min << 16, codes uint8 0..15)."""
    return _quantize_min(y, 15)


def quantize_q5_1(y):
    """q5_1: d = (max - min)/31, codes = min(31, trunc((x - min)*(1/d) + 0.5))."""
    return _quantize_min(y, 31)


def quantize(qtype: str, y):
    return {TYPE_Q4_0: quantize_q4_0, TYPE_Q5_0: quantize_q5_0, TYPE_Q8_0: quantize_q8_0,
            TYPE_Q4_1: quantize_q4_1, TYPE_Q5_1: quantize_q5_1}[qtype](y)


def scale_and_min(qtype: str, d_bits):
    """(fp16 scale, fp16 minimum) values of stored blocks, float64 (minimum 0 for the _0 types)."""
    if qtype in MIN_TYPES:
        w = np.asarray(d_bits, dtype=np.uint32)
        return (f16_value((w & np.uint32(0xFFFF)).astype(np.uint16)),
                f16_value((w >> np.uint32(16)).astype(np.uint16)))
    dv = f16_value(d_bits)
    return dv, np.zeros_like(dv)


def dequantize(qtype: str, d_bits, codes) -> np.ndarray:
    """code -> value with the stored fp16 scale (and minimum), in float64,
    flattened back to head_dim."""
    c = np.asarray(codes).astype(F64)
    if qtype in MIN_TYPES:
        dv, mv = scale_and_min(qtype, d_bits)
        x = c * dv[..., None] + mv[..., None]
        return x.reshape(x.shape[:-2] + (x.shape[-2] * QK,))
    dv = f16_value(d_bits)[..., None]
    if qtype == TYPE_Q8_0:
        x = c * dv
    elif qtype == TYPE_Q4_0:
        x = (c - 8.0) * dv
    elif qtype == TYPE_Q5_0:
        x = (c - 16.0) * dv
    else:
        raise ValueError(qtype)
    return x.reshape(x.shape[:-2] + (x.shape[-2] * QK,))


# ---- packing (GGUF block payloads) ----------------------------------------

def pack_q4_0(codes) -> np.ndarray:
    """byte k (0..15) = code_k | code_{k+16} << 4."""
    c = np.asarray(codes, dtype=np.uint8)
    return (c[..., :16] | (c[..., 16:] << 4)).astype(np.uint8)


def unpack_q4_0(qs) -> np.ndarray:
    q = np.asarray(qs, dtype=np.uint8)
    return np.concatenate([q & 0x0F, q >> 4], axis=-1)


def pack_q5_0(codes):
    """qs byte k = low nibble of code_k | low nibble of code_{k+16} << 4;
    qh bit j = bit 4 of code_j (j = 0..31), stored little-endian."""
    c = np.asarray(codes, dtype=np.uint8)
    qs = ((c[..., :16] & 0x0F) | ((c[..., 16:] & 0x0F) << 4)).astype(np.uint8)
    bits = ((c >> 4) & 1).astype(np.uint64)
    qh = np.zeros(c.shape[:-1], dtype=np.uint64)
    for j in range(QK):
        qh |= bits[..., j] << np.uint64(j)
    return qs, qh.astype(np.uint32)


def unpack_q5_0(qs, qh) -> np.ndarray:
    low = unpack_q4_0(qs)
    h = np.asarray(qh, dtype=np.uint32)[..., None]
    hi = ((h >> np.arange(QK, dtype=np.uint32)) & 1).astype(np.uint8)
    return low | (hi << 4)


def to_ggml_bytes(qtype: str, d_bits, codes) -> np.ndarray:
    """Array-of-structs GGUF byte image of blocks [..., nb]:
    q4_0 = [d:2][qs:16], q5_0 = [d:2][qh:4 LE][qs:16], q8_0 = [d:2][qs:32],
    q4_1 = [d:2][min:2][qs:16], q5_1 = [d:2][min:2][qh:4 LE][qs:16]."""
    if qtype in MIN_TYPES:
        w = np.asarray(d_bits, dtype="<u4")
        dbytes = w[..., None].view(np.uint8).reshape(w.shape + (4,))   # d then min, little-endian
    else:
        d = np.asarray(d_bits, dtype=np.uint16)
        dbytes = d[..., None].view(np.uint8).reshape(d.shape + (2,))
    if qtype in (TYPE_Q4_0, TYPE_Q4_1):
        parts = [dbytes, pack_q4_0(codes)]
    elif qtype in (TYPE_Q5_0, TYPE_Q5_1):
        qs, qh = pack_q5_0(codes)
        qhb = qh.astype("<u4")[..., None].view(np.uint8).reshape(qh.shape + (4,))
        parts = [dbytes, qhb, qs]
    elif qtype == TYPE_Q8_0:
        parts = [dbytes, np.asarray(codes, dtype=np.int8).view(np.uint8)]
    else:
        raise ValueError(qtype)
    return np.concatenate(parts, axis=-1)


# ---------------------------------------------------------------------------
# Outlier channels ([P1] 적용 및 배경 기술: 8-bit outlier channels; reading in
# the module docstring)
# ---------------------------------------------------------------------------

def split_outliers(x: np.ndarray, oidx: np.ndarray):
    """x [..., H, d] (float32), oidx [H][O] -> (x_O [..., H, O]: the values of
    each head's outlier channels in slot order, x_rest: x with those channels
    set to zero)."""
    x = np.asarray(x, dtype=F32)
    xo = np.stack([x[..., h, oidx[h]] for h in range(x.shape[-2])], axis=-2)
    rest = x.copy()
    for h in range(x.shape[-2]):
        rest[..., h, oidx[h]] = 0.0
    return xo, rest


def outlier_values(d_bits, codes, chans, head_dim: int) -> np.ndarray:
    """q8_0 outlier blocks of one head ([n][O/32], [n][O/32][32]) -> float64
    [n][head_dim]: slot i's dequantized value at channel chans[i], zeros
    elsewhere (original basis)."""
    v = dequantize(TYPE_Q8_0, d_bits, codes)
    out = np.zeros(v.shape[:-1] + (head_dim,), dtype=F64)
    out[..., np.asarray(chans)] = v
    return out


# ---------------------------------------------------------------------------
# The rotated, quantized KV cache with a BF16 precision tail
# ---------------------------------------------------------------------------

class OracleCache:
    """Per sequence and KV head, every appended token is rotated (if enabled),
    quantized into the body at its position and -- if it is among the last
    `tail_len` tokens written -- also kept as bf16 in ring slot pos % tail_len.
    Attention reads positions [n - T, n) from the tail and the rest from the
    body ([P2] 용어 해설, Precision Tail).

    Reading of unstated details: the tail holds the *rotated* values, so one
    query basis and one inverse rotation serve body and tail; the body is
    written for every token ("write-through"), so codes never depend on T."""

    def __init__(self, batch, n_kv_heads, head_dim, max_ctx, tail_len,
                 k_type, v_type, rot_k, rot_v, outliers=None):
        if head_dim % QK:
            raise ValueError("head_dim must be a multiple of 32")
        # outlier channels: [n_kv_heads][O], strictly increasing, O a multiple of 32
        self.oidx = None if outliers is None else np.asarray(outliers, dtype=np.int64)
        self.O = 0 if self.oidx is None else self.oidx.shape[1]
        if self.O:
            if (self.oidx.shape[0] != n_kv_heads or self.O % QK or self.O >= head_dim
                    or np.any(self.oidx < 0) or np.any(self.oidx >= head_dim)
                    or np.any(np.diff(self.oidx, axis=1) <= 0)):
                raise ValueError("outlier channels: [n_kv_heads][O], O a multiple of 32 below head_dim, "
                                 "strictly increasing channels")
        if (rot_k or rot_v) and not rotation_enabled(head_dim):
            raise ValueError("rotation requested on an ineligible head_dim")
        self.B, self.H, self.d = batch, n_kv_heads, head_dim
        self.max_ctx, self.T = max_ctx, tail_len
        self.types = {"k": k_type, "v": v_type}
        self.rot = {"k": bool(rot_k), "v": bool(rot_v)}
        nb = head_dim // QK
        self.codes = {w: np.zeros((batch, n_kv_heads, max_ctx, nb, QK), np.uint8 if self.types[w] != TYPE_Q8_0 else np.int8)
                      for w in ("k", "v")}
        self.dbits = {w: np.zeros((batch, n_kv_heads, max_ctx, nb),
                                  np.uint32 if self.types[w] in MIN_TYPES else np.uint16) for w in ("k", "v")}
        self.tail = {w: np.zeros((batch, n_kv_heads, max(tail_len, 1), head_dim), np.uint16)
                     for w in ("k", "v")}
        no = max(self.O, QK) // QK
        self.ocodes = {w: np.zeros((batch, n_kv_heads, max_ctx, no, QK), np.int8) for w in ("k", "v")}
        self.odbits = {w: np.zeros((batch, n_kv_heads, max_ctx, no), np.uint16) for w in ("k", "v")}
        self.seq_len = np.zeros(batch, dtype=np.int64)

    # -- write path -------------------------------------------------------
    def stored_input(self, which: str, x: np.ndarray, prerotated: bool) -> np.ndarray:
        """The float32 vectors that get quantized: x (float32) rotated in
        float64 when rotation is on, then rounded to float32."""
        x = np.asarray(x, dtype=F32)
        if self.rot[which] and not prerotated:
            return rotate(x).astype(F32)
        return x

    def append(self, k, v, n_new_per_seq=None, prerotated=False):
        """k, v: [B][n_new][H][d] (float32 values).  Appends n_new_per_seq[b]
        (default n_new) tokens of each sequence at positions seq_len[b]..."""
        k = np.asarray(k, dtype=F32)
        v = np.asarray(v, dtype=F32)
        n_new = k.shape[1]
        if self.O and prerotated:
            raise ValueError("outlier channels are picked in the original basis: no prerotated input")
        for b in range(self.B):
            nb = n_new if n_new_per_seq is None else int(n_new_per_seq[b])
            n0 = int(self.seq_len[b])
            if nb < 0 or nb > n_new or n0 + nb > self.max_ctx:
                raise ValueError("append out of range")
            if nb == 0:
                continue
            for which, x in (("k", k), ("v", v)):
                y = self.stored_input(which, x[b, :nb], prerotated)  # [nb][H][d], the tail's values
                yb = y
                if self.O:
                    # outlier values (unrotated) -> q8_0; the rest, zeroed there, is rotated
                    xo, rest = split_outliers(x[b, :nb], self.oidx)
                    od, oc = quantize_q8_0(xo)
                    self.ocodes[which][b, :, n0:n0 + nb] = oc.transpose(1, 0, 2, 3)
                    self.odbits[which][b, :, n0:n0 + nb] = od.transpose(1, 0, 2)
                    yb = self.stored_input(which, rest, False)
                dbits, codes = quantize(self.types[which], yb)
                self.codes[which][b, :, n0:n0 + nb] = codes.transpose(1, 0, 2, 3)
                self.dbits[which][b, :, n0:n0 + nb] = dbits.transpose(1, 0, 2)
                if self.T > 0:
                    first = max(n0, n0 + nb - self.T)
                    for pos in range(first, n0 + nb):
                        self.tail[which][b, :, pos % self.T] = bf16_bits(y[pos - n0])
            self.seq_len[b] = n0 + nb

    # -- what attention reads --------------------------------------------
    def body_values(self, which, b, h, t0=0, t1=None) -> np.ndarray:
        """float64 [t1 - t0][d] in the basis attention works in (rotated when
        rotation is on): the dequantized body, plus -- with outlier channels --
        the dequantized q8_0 outlier values scattered to their channels and
        rotated like the rest."""
        t1 = int(self.seq_len[b]) if t1 is None else t1
        x = dequantize(self.types[which], self.dbits[which][b, h, t0:t1],
                       self.codes[which][b, h, t0:t1])
        if self.O:
            xo = outlier_values(self.odbits[which][b, h, t0:t1], self.ocodes[which][b, h, t0:t1],
                                self.oidx[h], self.d)
            x = x + (rotate(xo) if self.rot[which] else xo)
        return x

    def tail_values(self, which, b, h, positions) -> np.ndarray:
        slots = np.asarray(positions, dtype=np.int64) % self.T
        return bf16_value(self.tail[which][b, h, slots])

    def stored(self, which, b, h) -> np.ndarray:
        """float64 [n][d]: the value attention sees for every position < n."""
        n = int(self.seq_len[b])
        split = max(0, n - self.T)
        out = np.empty((n, self.d), dtype=F64)
        out[:split] = self.body_values(which, b, h, 0, split)
        if n > split:
            out[split:] = self.tail_values(which, b, h, np.arange(split, n))
        return out

    def ggml_blocks(self, which, b, h, t0, count) -> np.ndarray:
        return to_ggml_bytes(self.types[which], self.dbits[which][b, h, t0:t0 + count],
                             self.codes[which][b, h, t0:t0 + count])


# ---------------------------------------------------------------------------
# Attention (float64)
# ---------------------------------------------------------------------------

def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)


def softmax_attention(q, K, V, scale) -> np.ndarray:
    """Textbook attention of query rows q [m][d] over keys K [n][d] and values
    V [n][d] with an optional boolean visibility mask; float64.  A query that
    sees no key returns zeros."""
    q = np.asarray(q, dtype=F64)
    s = scale * (q @ np.asarray(K, dtype=F64).T)
    if s.shape[-1] == 0:
        return np.zeros((q.shape[0], np.asarray(V).shape[-1]))
    s = s - s.max(axis=-1, keepdims=True)
    p = np.exp(s)
    p /= p.sum(axis=-1, keepdims=True)
    return p @ np.asarray(V, dtype=F64)


def decode_attention(cache: OracleCache, q, scale=None, pairs=None) -> np.ndarray:
    """q [B][Hq][d] -> out [B][Hq][d] float64.

    Query head h reads KV head h // (Hq/Hkv).  q is rotated when K rotation
    is on (scores are then dot products in the rotated basis, [P1] 아다마르
    회전); the output is rotated back when V rotation is on.  `pairs`
    optionally restricts the work to a list of (b, kv_head)."""
    q = np.asarray(q, dtype=F64)
    B, Hq, d = q.shape
    g = Hq // cache.H
    scale = default_scale(d) if not scale else scale
    R = rotation_matrix(d) if (cache.rot["k"] or cache.rot["v"]) else None
    qr = q @ R if cache.rot["k"] else q
    out = np.zeros((B, Hq, d), dtype=F64)
    todo = pairs if pairs is not None else [(b, h) for b in range(B) for h in range(cache.H)]
    for b, kvh in todo:
        if cache.seq_len[b] == 0:
            continue
        K = cache.stored("k", b, kvh)
        V = cache.stored("v", b, kvh)
        heads = slice(kvh * g, (kvh + 1) * g)
        o = softmax_attention(qr[b, heads], K, V, scale)
        out[b, heads] = o @ R if cache.rot["v"] else o
    return out


def prefill_attention(cache: OracleCache, q, q_pos0=None, causal=True, scale=None,
                      heads=None) -> np.ndarray:
    """q [B][n_tok][Hq][d] -> out [B][n_tok][Hq][d] float64.

    Query i of sequence b sits at absolute position p = q_pos0[b] + i
    (default: the last n_tok positions of the sequence) and, when causal,
    sees keys t <= p; every query sees only t < seq_len[b]."""
    q = np.asarray(q, dtype=F64)
    B, n_tok, Hq, d = q.shape
    g = Hq // cache.H
    scale = default_scale(d) if not scale else scale
    R = rotation_matrix(d) if (cache.rot["k"] or cache.rot["v"]) else None
    qr = q @ R if cache.rot["k"] else q
    out = np.zeros_like(q)
    heads = range(Hq) if heads is None else heads
    for b in range(B):
        n = int(cache.seq_len[b])
        p0 = n - n_tok if q_pos0 is None else int(q_pos0[b])
        for kvh in range(cache.H):
            hs = [h for h in heads if h // g == kvh]
            if not hs:
                continue
            K = cache.stored("k", b, kvh)
            V = cache.stored("v", b, kvh)
            s = scale * np.einsum("ihd,td->iht", qr[b][:, hs], K)
            pos = p0 + np.arange(n_tok)
            vis = np.ones((n_tok, n), dtype=bool)
            if causal:
                vis = np.arange(n)[None, :] <= pos[:, None]
            s = np.where(vis[:, None, :], s, -np.inf)
            smax = s.max(axis=-1, keepdims=True)
            smax = np.where(np.isfinite(smax), smax, 0.0)
            p = np.exp(s - smax)
            den = p.sum(axis=-1, keepdims=True)
            p = np.divide(p, den, out=np.zeros_like(p), where=den > 0)
            o = np.einsum("iht,td->ihd", p, V)
            out[b][:, hs] = o @ R if cache.rot["v"] else o
    return out
