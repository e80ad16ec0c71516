"""Paged body layout (block table) vs the oracle's logical cache: a pool of
pages shared by the sequences, pages handed out in a shuffled order.  The
blocks read back through the page table must equal the oracle's bit for bit,
and decode, prefill and the fused step must match the oracle's attention."""

import numpy as np
import pytest

from oracle import kvq_oracle as ko
from kvq_testlib import append_both, assert_close, gpu_blocks, gpu_decode, prerotate, require_gpu, to_dev

pytestmark = pytest.mark.gpu


def _paged_pair(torch, kvq, rng, B, H, d, max_ctx, T, kt, vt, page_tokens, spare=7):
    per_seq = max_ctx // page_tokens
    n_pages = B * per_seq + spare
    pages = rng.permutation(n_pages)[:B * per_seq].astype(np.int32)   # shuffled, with unused pages in the pool
    gc = kvq.KVCache(B, H, d, max_ctx, T, kt, vt, page_tokens=page_tokens, n_pages=n_pages,
                     page_table=torch.tensor(pages))
    oc = ko.OracleCache(B, H, d, max_ctx, T, kt, vt, True, True)
    return gc, oc


def _kv(rng, B, n, H, d):
    k = rng.standard_normal((B, n, H, d)).astype(np.float32)
    v = rng.standard_normal((B, n, H, d)).astype(np.float32)
    k[..., 9 % d] *= 20
    v[..., 4] *= 20
    return k, v


@pytest.mark.parametrize("kt,vt,d,page_tokens", [("q8_0", "q4_0", 128, 64), ("q5_1", "q4_0", 256, 128),
                                                 ("q4_0", "q5_0", 64, 64)])
def test_paged_blocks_and_decode(kt, vt, d, page_tokens):
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    rng = np.random.default_rng(71)
    B, H, g, max_ctx, T = 3, 2, 4, 512, 24
    gc, oc = _paged_pair(torch, kvq, rng, B, H, d, max_ctx, T, kt, vt, page_tokens)
    k, v = _kv(rng, B, 500, H, d)
    append_both(gc, oc, k, v, n_new_per_seq=[500, 77, 300], torch=torch)
    for b, n in enumerate([500, 77, 300]):
        for h in range(H):
            assert np.array_equal(gpu_blocks(gc, b, h, 0, 0, n, kt, d, torch), oc.ggml_blocks("k", b, h, 0, n))
            assert np.array_equal(gpu_blocks(gc, b, h, 1, 0, n, vt, d, torch), oc.ggml_blocks("v", b, h, 0, n))
    q = rng.standard_normal((B, H * g, d)).astype(np.float32)
    assert_close(gpu_decode(gc, q, "f32", torch), ko.decode_attention(oc, q), what=f"paged decode {kt}/{vt}")


def test_paged_prefill_and_fused_steps():
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    rng = np.random.default_rng(72)
    B, H, g, d, max_ctx, T, n = 2, 2, 4, 128, 384, 32, 300
    gc, oc = _paged_pair(torch, kvq, rng, B, H, d, max_ctx, T, "q4_0", "q8_0", 64)
    k, v = _kv(rng, B, n, H, d)
    append_both(gc, oc, k, v, torch=torch)
    # causal prefill of the whole prompt
    q = rng.standard_normal((B, n, H * g, d)).astype(np.float32)
    qd = to_dev(q, "f32", torch)
    out = torch.empty_like(qd)
    ws = torch.empty(kvq.kvq_prefill_workspace_bytes(gc.desc, H * g, n), dtype=torch.uint8, device="cuda")
    kvq.kvq_prefill_attention(gc.desc, qd, out, ws)
    st, bits = kvq.kvq_sync_status(gc.desc)
    assert st == 0, (st, bits)
    assert_close(out.cpu().numpy().astype(np.float64), ko.prefill_attention(oc, q), what="paged prefill")
    # decode steps with the append fused into the decode launch
    for step in range(5):
        kn, vn = _kv(rng, B, 1, H, d)
        yk, yv = prerotate(kn, True), prerotate(vn, True)
        qs = rng.standard_normal((B, H * g, d)).astype(np.float32)
        o = torch.empty((B, H * g, d), dtype=torch.float32, device="cuda")
        wsd = torch.empty(kvq.kvq_decode_workspace_bytes(gc.desc, H * g), dtype=torch.uint8, device="cuda")
        kvq.kvq_append_decode(gc.desc, to_dev(yk, "f32", torch), to_dev(yv, "f32", torch), to_dev(qs, "f32", torch),
                              o, wsd, prerotated=True)
        st, bits = kvq.kvq_sync_status(gc.desc)
        assert st == 0, (st, bits)
        oc.append(yk, yv, prerotated=True)
        assert_close(o.cpu().numpy().astype(np.float64), ko.decode_attention(oc, qs), what=f"paged step {step}")
    assert np.array_equal(gc.seq_len.cpu().numpy(), oc.seq_len)


@pytest.mark.parametrize("H", [1, 8])
def test_page_outside_pool_is_reported(H):
    """A page-table entry outside the pool: nothing is written or read through it,
    and append and decode report KVQ_DEV_ERR_PAGE (H = 8: 3,200 vectors, the
    bulk append kernel; H = 1: one warp per vector)."""
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    rng = np.random.default_rng(73)
    B, d, max_ctx = 1, 64, 256
    table = torch.tensor([0, 1, 99, 2], dtype=torch.int32)   # page 2 of the sequence points outside 4 pages
    gc = kvq.KVCache(B, H, d, max_ctx, 0, "q8_0", "q8_0", page_tokens=64, n_pages=4, page_table=table)
    k, v = _kv(rng, B, 200, H, d)
    kvq.kvq_rotate_quantize_append(gc.desc, to_dev(k, "f32", torch), to_dev(v, "f32", torch))
    st, bits = kvq.kvq_sync_status(gc.desc)
    assert st == kvq.KVQ_ERR_DEVICE_RANGE and bits == kvq.KVQ_DEV_ERR_PAGE
    q = to_dev(rng.standard_normal((B, 4 * H, d)).astype(np.float32), "f32", torch)
    out = torch.empty_like(q)
    ws = torch.empty(kvq.kvq_decode_workspace_bytes(gc.desc, 4 * H), dtype=torch.uint8, device="cuda")
    kvq.kvq_decode_attention(gc.desc, q, out, ws)
    st, bits = kvq.kvq_sync_status(gc.desc)
    assert st == kvq.KVQ_ERR_DEVICE_RANGE and bits == kvq.KVQ_DEV_ERR_PAGE
    assert bool(torch.isfinite(out).all())
