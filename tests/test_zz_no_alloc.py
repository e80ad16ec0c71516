"""kvq_decode_attention_noalloc: decode attention for callers that cannot
allocate device memory (so cannot hand the library a workspace).  It uses the
library's fixed device scratch array instead; its results must match
kvq_decode_attention's, call after call, and a decode that would need more
scratch than the fixed array must be refused before anything is launched.

This file is collected last on purpose: if it fails, every other test has
already run."""

import numpy as np
import pytest

from kvq_testlib import append_both, assert_close, gpu_decode, require_gpu, to_dev
from oracle import kvq_oracle as ko

pytestmark = pytest.mark.gpu


def _filled_cache(torch, kvq, rng, B, H, d, n, T, kt, vt):
    gc = kvq.KVCache(B, H, d, (n + 63) // 64 * 64, T, kt, vt)
    k = rng.standard_normal((B, n, H, d)).astype(np.float32)
    v = rng.standard_normal((B, n, H, d)).astype(np.float32)
    k[..., 3] *= 20
    v[..., 9] *= 20
    kvq.kvq_rotate_quantize_append(gc.desc, to_dev(k, "bf16", torch), to_dev(v, "bf16", torch))
    torch.cuda.synchronize()
    return gc


@pytest.mark.parametrize("B,H,g,d,n,T,kt,vt", [(2, 4, 6, 256, 3000, 256, "q8_0", "q4_0"),
                                               (3, 2, 4, 128, 1500, 64, "q5_0", "q5_0")])
def test_noalloc_matches_workspace_entry_point_twice(B, H, g, d, n, T, kt, vt):
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    rng = np.random.default_rng(42)
    gc = _filled_cache(torch, kvq, rng, B, H, d, n, T, kt, vt)
    assert kvq.kvq_decode_workspace_bytes(gc.desc, H * g) <= kvq.KVQ_NOALLOC_SCRATCH_BYTES
    for call in range(2):  # the second call finds the first call's leftovers in the scratch
        q_np = rng.standard_normal((B, H * g, d)).astype(np.float32)
        ref = gpu_decode(gc, q_np, "f32", torch)          # kvq_decode_attention with a workspace
        q = to_dev(q_np, "f32", torch)
        out = torch.full_like(q, float("nan"))
        kvq.kvq_decode_attention_noalloc(gc.desc, q, out)
        st, bits = kvq.kvq_sync_status(gc.desc)
        assert st == 0, (st, bits)
        assert_close(out.cpu().numpy().astype(np.float64), ref, what=f"noalloc call {call}")


def test_noalloc_refuses_more_scratch_than_it_has():
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    gc = kvq.KVCache(128, 8, 256, 64, 64, "q8_0", "q8_0")   # body + tail splits: 16.9 MB of partials
    need = kvq.kvq_decode_workspace_bytes(gc.desc, 64)
    assert need > kvq.KVQ_NOALLOC_SCRATCH_BYTES
    q = torch.zeros((128, 64, 256), dtype=torch.float32, device="cuda")
    out = torch.full_like(q, 7.0)
    with pytest.raises(kvq.KvqError) as e:
        kvq.kvq_decode_attention_noalloc(gc.desc, q, out)
    assert e.value.status == kvq.KVQ_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert bool((out == 7.0).all())   # nothing was launched


def test_noalloc_drops_what_an_earlier_call_of_another_shape_left():
    """A call does not write the partial rows of a split whose token range came out
    empty; whatever an earlier call left there (here a call of another head_dim,
    batch and format, with large scores, so that its rows sit at other offsets and
    hold large values) must be dropped by its weight.  The decode covers an empty
    sequence, a tail-only one and long ones, and is checked against the oracle and
    against kvq_decode_attention given a workspace full of NaN bytes."""
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    rng = np.random.default_rng(7)
    other = _filled_cache(torch, kvq, rng, 3, 2, 128, 1500, 64, "q5_0", "q5_0")
    q_other = to_dev(rng.standard_normal((3, 8, 128)).astype(np.float32) * 50.0, "f32", torch)
    out_other = torch.empty_like(q_other)
    kvq.kvq_decode_attention_noalloc(other.desc, q_other, out_other)
    st, bits = kvq.kvq_sync_status(other.desc)
    assert st == 0, (st, bits)

    B, H, g, d, T = 4, 2, 4, 256, 64
    gc = kvq.KVCache(B, H, d, 2048, T, "q8_0", "q4_0")
    st, rk, rv = kvq.kvq_resolve_rotation(gc.desc)
    assert st == 0
    oc = ko.OracleCache(B, H, d, 2048, T, "q8_0", "q4_0", bool(rk), bool(rv))
    lens = [0, 5, 700, 2000]
    k = rng.standard_normal((B, max(lens), H, d)).astype(np.float32)
    v = rng.standard_normal((B, max(lens), H, d)).astype(np.float32)
    k[..., 7] *= 20
    v[..., 11] *= 20
    append_both(gc, oc, k, v, n_new_per_seq=lens, torch=torch)
    q_np = rng.standard_normal((B, H * g, d)).astype(np.float32)
    ref = ko.decode_attention(oc, q_np)
    q = to_dev(q_np, "f32", torch)
    # the workspace entry point over NaN bytes
    wsb = kvq.kvq_decode_workspace_bytes(gc.desc, H * g)
    ws = torch.full((wsb,), 0xFF, dtype=torch.uint8, device="cuda")
    out_ws = torch.empty_like(q)
    kvq.kvq_decode_attention(gc.desc, q, out_ws, ws)
    st, bits = kvq.kvq_sync_status(gc.desc)
    assert st == 0, (st, bits)
    got_ws = out_ws.cpu().numpy().astype(np.float64)
    assert_close(got_ws, ref, what="workspace of NaN bytes")
    assert np.all(got_ws[0] == 0.0)   # the empty sequence's output
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        kvq.kvq_decode_attention_noalloc(gc.desc, q, out)
        st, bits = kvq.kvq_sync_status(gc.desc)
        assert st == 0, (st, bits)
        got = out.cpu().numpy().astype(np.float64)
        assert_close(got, ref, what=f"noalloc after another shape, call {call}")
        assert_close(got, got_ws, what=f"noalloc vs workspace entry point, call {call}")
