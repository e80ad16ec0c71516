"""Outlier channels kept at 8 bits (q8_0, original basis) beside the rotated
low-bit rest: GPU write path, decode, the fused step and prefill against the
oracle.

Outlier caches take inputs in the original basis only, so the GPU rotates
the rest itself.  To keep both sides' caches identical the inputs are dyadic
(multiples of 2^-3 with small numerators) at head_dim 64 and 256, where the
fp32 butterfly and the 1/8 or 1/16 normalisation are exact; at head_dim 128
the rotation is switched off.  Blocks, outlier planes and tail rows are then
compared bit for bit, and attention within the usual tolerance."""

import numpy as np
import pytest

from oracle import kvq_oracle as ko
from kvq_testlib import assert_close, gpu_blocks, gpu_decode, require_gpu, to_dev

pytestmark = pytest.mark.gpu

PAIRS = [(k, v) for k in ("q4_0", "q5_0", "q8_0") for v in ("q4_0", "q5_0", "q8_0")]


def _outliers(rng, H, d):
    return np.stack([np.sort(rng.choice(d, 32, replace=False)) for _ in range(H)]).astype(np.int64)


def _dyadic(rng, shape, oidx):
    x = rng.integers(-64, 65, shape).astype(np.float32) * np.float32(0.125)
    for h in range(shape[2]):
        x[:, :, h][..., oidx[h][:4]] *= 16     # a few large outlier channels per head
    return x


def _caches(kvq, B, H, d, max_ctx, T, kt, vt, rot, oidx, **kw):
    flags = kvq.KVQ_ROT_AUTO if rot else (kvq.KVQ_ROT_K_OFF | kvq.KVQ_ROT_V_OFF)
    gc = kvq.KVCache(B, H, d, max_ctx, T, kt, vt, flags=flags, outliers=oidx.tolist(), **kw)
    oc = ko.OracleCache(B, H, d, max_ctx, T, kt, vt, rot, rot, outliers=oidx)
    return gc, oc


def _append(kvq, torch, gc, oc, k, v, nps=None):
    nps_dev = None if nps is None else torch.tensor(np.asarray(nps, np.int32)).cuda()
    kvq.kvq_rotate_quantize_append(gc.desc, to_dev(k, "f32", torch), to_dev(v, "f32", torch), n_new_per_seq=nps_dev)
    oc.append(k, v, n_new_per_seq=nps)
    st, bits = kvq.kvq_sync_status(gc.desc)
    assert st == 0, (st, bits)


def _outlier_rows(gc, which, rows, torch):
    """int8 codes [rows][32] and fp16 scale bits [rows] of K or V in the outlier
    plane (groups of 16 rows: K codes [16][32], V codes [16][32], K scales [16],
    V scales [16])."""
    grp = gc.planes["outl"].cpu().numpy().reshape(-1, 1088)
    w = 0 if which == "k" else 1
    g, i = rows // 16, rows % 16
    codes = grp[:, w * 512:(w + 1) * 512].reshape(-1, 16, 32).view(np.int8)
    scales = grp[:, 1024 + w * 32:1024 + (w + 1) * 32].copy().view(np.uint16)
    return codes[g, i], scales[g, i]


def _check_cache(torch, gc, oc, kt, vt, d, page_of=None):
    B, H = oc.B, oc.H
    for b in range(B):
        n = int(oc.seq_len[b])
        for h in range(H):
            assert np.array_equal(gpu_blocks(gc, b, h, 0, 0, n, kt, d, torch), oc.ggml_blocks("k", b, h, 0, n))
            assert np.array_equal(gpu_blocks(gc, b, h, 1, 0, n, vt, d, torch), oc.ggml_blocks("v", b, h, 0, n))
            t = np.arange(n)
            if page_of is None:
                rows = (b * H + h) * oc.max_ctx + t
            else:
                pt = oc.max_ctx // page_of[0]
                rows = (page_of[1][b * pt + t // page_of[0]] * H + h) * page_of[0] + t % page_of[0]
            for w in ("k", "v"):
                qs, dd = _outlier_rows(gc, w, rows, torch)
                assert np.array_equal(qs, oc.ocodes[w][b, h, :n, 0]), (w, b, h)
                assert np.array_equal(dd, oc.odbits[w][b, h, :n, 0]), (w, b, h)
            if oc.T:
                lo = max(0, n - oc.T)
                for w in ("k", "v"):
                    tail = gc.planes[f"{w}_tail"].cpu().numpy().view(np.uint16).reshape(B, H, oc.T, d)
                    assert np.array_equal(tail[b, h, np.arange(lo, n) % oc.T], oc.tail[w][b, h, np.arange(lo, n) % oc.T])


@pytest.mark.parametrize("d,rot", [(64, True), (256, True), (128, False)])
def test_append_bit_exact(d, rot):
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    rng = np.random.default_rng(81)
    B, H, T = 2, 2, 8
    oidx = _outliers(rng, H, d)
    gc, oc = _caches(kvq, B, H, d, 128, T, "q4_0", "q8_0", rot, oidx)
    for step in range(3):   # ragged appends
        n = [40, 3, 17][step]
        nps = [n, max(0, n - 2)]
        k = _dyadic(rng, (B, n, H, d), oidx) if rot else rng.standard_normal((B, n, H, d)).astype(np.float32)
        v = _dyadic(rng, (B, n, H, d), oidx) if rot else rng.standard_normal((B, n, H, d)).astype(np.float32)
        _append(kvq, torch, gc, oc, k, v, nps)
    _check_cache(torch, gc, oc, "q4_0", "q8_0", d)


@pytest.mark.parametrize("kt,vt", PAIRS)
def test_decode_every_pair(kt, vt):
    """head_dim 128, rotation off: every q4_0 / q5_0 / q8_0 pair, GQA 4, ragged lengths."""
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    rng = np.random.default_rng(82)
    B, H, g, d, T = 2, 2, 4, 128, 16
    oidx = _outliers(rng, H, d)
    gc, oc = _caches(kvq, B, H, d, 1024, T, kt, vt, False, oidx)
    k = rng.standard_normal((B, 700, H, d)).astype(np.float32)
    v = rng.standard_normal((B, 700, H, d)).astype(np.float32)
    for h in range(H):
        k[:, :, h][..., oidx[h][:3]] *= 25
        v[:, :, h][..., oidx[h][:3]] *= 10
    _append(kvq, torch, gc, oc, k, v, [700, 333])
    q = rng.standard_normal((B, H * g, d)).astype(np.float32)
    assert_close(gpu_decode(gc, q, "f32", torch), ko.decode_attention(oc, q), what=f"{kt}/{vt}")


@pytest.mark.parametrize("d,kt,vt,T", [(64, "q4_0", "q4_0", 8), (64, "q8_0", "q5_0", 0), (256, "q4_0", "q8_0", 32),
                                       (256, "q5_0", "q4_0", 0)])
def test_decode_rotated(d, kt, vt, T):
    """Rotation on (exact dyadic inputs): the merge rotates the rest back and adds
    the outlier channels in the original basis."""
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    rng = np.random.default_rng(83)
    B, H, g = 2, 2, 3
    oidx = _outliers(rng, H, d)
    gc, oc = _caches(kvq, B, H, d, 512, T, kt, vt, True, oidx)
    k, v = _dyadic(rng, (B, 300, H, d), oidx), _dyadic(rng, (B, 300, H, d), oidx)
    _append(kvq, torch, gc, oc, k, v, [300, 129])
    _check_cache(torch, gc, oc, kt, vt, d)
    for qd in ("f32", "bf16"):
        q = rng.standard_normal((B, H * g, d)).astype(np.float32)
        if qd == "bf16":
            q = torch.from_numpy(q).to(torch.bfloat16).float().numpy()
        assert_close(gpu_decode(gc, q, qd, torch), ko.decode_attention(oc, q), what=f"d{d} {kt}/{vt} T{T} {qd}")


def test_paged_outliers():
    """Outlier planes follow the page table like the body."""
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    rng = np.random.default_rng(84)
    B, H, g, d, T, P = 2, 2, 2, 64, 8, 64
    max_ctx = 256
    n_pages = B * max_ctx // P + 3
    table = rng.permutation(n_pages)[:B * max_ctx // P].astype(np.int32)
    oidx = _outliers(rng, H, d)
    gc, oc = _caches(kvq, B, H, d, max_ctx, T, "q4_0", "q8_0", True, oidx, page_tokens=P, n_pages=n_pages,
                     page_table=torch.from_numpy(table))
    k, v = _dyadic(rng, (B, 200, H, d), oidx), _dyadic(rng, (B, 200, H, d), oidx)
    _append(kvq, torch, gc, oc, k, v, [200, 90])
    _check_cache(torch, gc, oc, "q4_0", "q8_0", d, page_of=(P, table))
    q = rng.standard_normal((B, H * g, d)).astype(np.float32)
    assert_close(gpu_decode(gc, q, "f32", torch), ko.decode_attention(oc, q), what="paged")


def test_fused_steps():
    """kvq_append_decode on an outlier cache: the tail CTA writes the new tokens
    (outlier planes included) inside the decode launch."""
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    rng = np.random.default_rng(85)
    B, H, g, d, T = 2, 2, 4, 64, 8
    oidx = _outliers(rng, H, d)
    gc, oc = _caches(kvq, B, H, d, 256, T, "q5_0", "q4_0", True, oidx)
    k, v = _dyadic(rng, (B, 90, H, d), oidx), _dyadic(rng, (B, 90, H, d), oidx)
    _append(kvq, torch, gc, oc, k, v, [90, 41])
    for step in range(10):
        k, v = _dyadic(rng, (B, 1, H, d), oidx), _dyadic(rng, (B, 1, H, d), oidx)
        q = rng.standard_normal((B, H * g, d)).astype(np.float32)
        out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
        ws = torch.empty(kvq.kvq_decode_workspace_bytes(gc.desc, H * g), dtype=torch.uint8, device="cuda")
        kvq.kvq_append_decode(gc.desc, to_dev(k, "f32", torch), to_dev(v, "f32", torch), to_dev(q, "f32", torch),
                              out, ws)
        st, bits = kvq.kvq_sync_status(gc.desc)
        assert st == 0, (st, bits)
        oc.append(k, v)
        assert_close(out.cpu().numpy().astype(np.float64), ko.decode_attention(oc, q), what=f"step {step}")
    assert np.array_equal(gc.seq_len.cpu().numpy(), oc.seq_len)
    _check_cache(torch, gc, oc, "q5_0", "q4_0", d)


def test_invalid_outlier_list_sets_status():
    """A list that is not strictly increasing: status bit, and the calls finish."""
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    rng = np.random.default_rng(86)
    B, H, d = 1, 1, 64
    bad = np.arange(32)[None, :].copy()
    bad[0, 5] = 3                          # repeats an earlier channel
    gc = kvq.KVCache(B, H, d, 64, 0, "q4_0", "q4_0", outliers=bad.tolist())
    x = to_dev(rng.standard_normal((B, 4, H, d)).astype(np.float32), "f32", torch)
    kvq.kvq_rotate_quantize_append(gc.desc, x, x)
    st, bits = kvq.kvq_sync_status(gc.desc)
    assert st == kvq.KVQ_ERR_DEVICE_RANGE and bits & kvq.KVQ_DEV_ERR_OUTLIER
    q = to_dev(rng.standard_normal((B, 2, d)).astype(np.float32), "f32", torch)
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    ws = torch.empty(kvq.kvq_decode_workspace_bytes(gc.desc, 2), dtype=torch.uint8, device="cuda")
    kvq.kvq_decode_attention(gc.desc, q, out, ws)
    st, bits = kvq.kvq_sync_status(gc.desc)
    assert bits & kvq.KVQ_DEV_ERR_OUTLIER
    assert torch.isfinite(out).all()


@pytest.mark.parametrize("d,rot,kt,vt,T", [(64, True, "q4_0", "q8_0", 16), (64, True, "q5_0", "q4_0", 0),
                                           (128, False, "q4_0", "q4_0", 32), (128, False, "q8_0", "q5_0", 0)])
def test_prefill(d, rot, kt, vt, T):
    """The staging adds each body key's and value's rotated outlier part to the
    dequantized rest; causal and non-causal, GQA 4, ragged lengths."""
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    from test_gpu_prefill import gpu_prefill
    rng = np.random.default_rng(87)
    B, H, g, n = 2, 2, 4, 200
    oidx = _outliers(rng, H, d)
    gc, oc = _caches(kvq, B, H, d, 256, T, kt, vt, rot, oidx)
    if rot:
        k, v = _dyadic(rng, (B, n, H, d), oidx), _dyadic(rng, (B, n, H, d), oidx)
    else:
        k = rng.standard_normal((B, n, H, d)).astype(np.float32)
        v = rng.standard_normal((B, n, H, d)).astype(np.float32)
        for h in range(H):
            k[:, :, h][..., oidx[h][:3]] *= 25
    _append(kvq, torch, gc, oc, k, v, [n, 150])
    q = rng.standard_normal((B, 150, H * g, d)).astype(np.float32)
    for causal in (True, False):
        assert_close(gpu_prefill(gc, q, "f32", torch, causal=causal),
                     ko.prefill_attention(oc, q, causal=causal), what=f"d{d} {kt}/{vt} T{T} causal={causal}")


def test_prefill_paged():
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    from test_gpu_prefill import gpu_prefill
    rng = np.random.default_rng(88)
    B, H, g, d, T, P, max_ctx = 2, 2, 2, 64, 8, 64, 256
    n_pages = B * max_ctx // P + 2
    table = rng.permutation(n_pages)[:B * max_ctx // P].astype(np.int32)
    oidx = _outliers(rng, H, d)
    gc, oc = _caches(kvq, B, H, d, max_ctx, T, "q8_0", "q4_0", True, oidx, page_tokens=P, n_pages=n_pages,
                     page_table=torch.from_numpy(table))
    k, v = _dyadic(rng, (B, 180, H, d), oidx), _dyadic(rng, (B, 180, H, d), oidx)
    _append(kvq, torch, gc, oc, k, v, [180, 77])
    q = rng.standard_normal((B, 77, H * g, d)).astype(np.float32)
    assert_close(gpu_prefill(gc, q, "f32", torch), ko.prefill_attention(oc, q), what="paged prefill")


@pytest.mark.parametrize("d,rot,kt,vt", [(64, True, "q4_0", "q8_0"), (256, True, "q5_0", "q4_0"),
                                         (128, False, "q8_0", "q5_0")])
def test_bulk_append_bit_exact(d, rot, kt, vt):
    """Appends of at least 2,048 vectors (the block-per-lane kernel with the
    outlier slots staged in shared memory): blocks, outlier planes and tail rows
    bit-exact after two ragged calls, then decode."""
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    rng = np.random.default_rng(89)
    B, H, g, T = 2, 4, 2, 16
    oidx = _outliers(rng, H, d)
    gc, oc = _caches(kvq, B, H, d, 640, T, kt, vt, rot, oidx)
    for n, nps in ((300, [300, 280]), (290, [250, 290])):
        if rot:
            k, v = _dyadic(rng, (B, n, H, d), oidx), _dyadic(rng, (B, n, H, d), oidx)
        else:
            k = rng.standard_normal((B, n, H, d)).astype(np.float32)
            v = rng.standard_normal((B, n, H, d)).astype(np.float32)
        _append(kvq, torch, gc, oc, k, v, nps)
    _check_cache(torch, gc, oc, kt, vt, d)
    q = rng.standard_normal((B, H * g, d)).astype(np.float32)
    assert_close(gpu_decode(gc, q, "f32", torch), ko.decode_attention(oc, q), what=f"bulk d{d}")


def test_decode_two_head_groups():
    """12 query heads per KV head: two CTAs along the head axis share one KV
    head's outlier list; the merge finds each query head's list by its KV head."""
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    rng = np.random.default_rng(90)
    B, H, g, d, T = 2, 2, 12, 128, 8
    oidx = _outliers(rng, H, d)
    gc, oc = _caches(kvq, B, H, d, 512, T, "q4_0", "q8_0", False, oidx)
    k = rng.standard_normal((B, 400, H, d)).astype(np.float32)
    v = rng.standard_normal((B, 400, H, d)).astype(np.float32)
    for h in range(H):
        v[:, :, h][..., oidx[h][:2]] *= 15
    _append(kvq, torch, gc, oc, k, v, [400, 211])
    q = rng.standard_normal((B, H * g, d)).astype(np.float32)
    assert_close(gpu_decode(gc, q, "f32", torch), ko.decode_attention(oc, q), what="two head groups")
