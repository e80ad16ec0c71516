"""kvq_append_decode (one decode step: append the new tokens, then attend) vs the
oracle doing the same two operations.  When fusable, the new tokens are written
inside the decode launch; the cache must then hold exactly what a separate
append would have written (bit-exact blocks and tail rows, seq_len), and every
step's output must match the oracle's attention over the updated cache."""

import numpy as np
import pytest

from oracle import kvq_oracle as ko
from kvq_testlib import assert_close, gpu_blocks, gpu_values, prerotate, require_gpu, to_dev

pytestmark = pytest.mark.gpu


def _tokens(rng, B, n, H, d):
    x = rng.standard_normal((B, n, H, d)).astype(np.float32)
    x[..., 5 % d] *= 20
    return x


def _step(kvq, torch, gc, oc, k, v, q, nps=None):
    """One GPU step through kvq_append_decode and the oracle's append + decode."""
    yk, yv = prerotate(k, oc.rot["k"]), prerotate(v, oc.rot["v"])
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    ws = torch.empty(kvq.kvq_decode_workspace_bytes(gc.desc, q.shape[1]), dtype=torch.uint8, device="cuda")
    nps_dev = None if nps is None else torch.tensor(np.asarray(nps, np.int32)).cuda()
    kvq.kvq_append_decode(gc.desc, to_dev(yk, "f32", torch), to_dev(yv, "f32", torch), to_dev(q, "f32", torch),
                          out, ws, n_new_per_seq=nps_dev, prerotated=True)
    st, bits = kvq.kvq_sync_status(gc.desc)
    oc.append(yk, yv, n_new_per_seq=nps, prerotated=True)
    return st, bits, out.cpu().numpy().astype(np.float64), ko.decode_attention(oc, q)


def _check_cache(torch, gc, oc, B, H, d, kt, vt):
    lens = gc.seq_len.cpu().numpy()
    assert np.array_equal(lens, oc.seq_len)
    for b in range(B):
        n = int(lens[b])
        for h in range(H):
            assert np.array_equal(gpu_blocks(gc, b, h, 0, 0, n, kt, d, torch), oc.ggml_blocks("k", b, h, 0, n))
            assert np.array_equal(gpu_blocks(gc, b, h, 1, 0, n, vt, d, torch), oc.ggml_blocks("v", b, h, 0, n))
            if oc.T == 0:
                continue
            lo = max(0, n - oc.T)
            for which, w in ((2, "k"), (3, "v")):
                got = gpu_values(gc, b, h, which, lo, n - lo, d, torch)
                assert np.array_equal(got, oc.tail_values(w, b, h, np.arange(lo, n)))


@pytest.mark.parametrize("kt,vt,d", [("q8_0", "q4_0", 128), ("q5_0", "q4_1", 256), ("q4_0", "q5_1", 64)])
def test_fused_steps_match_oracle_and_separate_append(kt, vt, d):
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    rng = np.random.default_rng(61)
    B, H, g, T = 2, 2, 6, 8
    gc = kvq.KVCache(B, H, d, 256, T, kt, vt)
    oc = ko.OracleCache(B, H, d, 256, T, kt, vt, True, True)
    pre = _tokens(rng, B, 100, H, d)  # a history appended the ordinary way
    yk, yv = prerotate(pre, True), prerotate(pre * 0.5, True)
    kvq.kvq_rotate_quantize_append(gc.desc, to_dev(yk, "f32", torch), to_dev(yv, "f32", torch),
                                   n_new_per_seq=torch.tensor([100, 37], dtype=torch.int32, device="cuda"),
                                   prerotated=True)
    oc.append(yk, yv, n_new_per_seq=[100, 37], prerotated=True)
    for step in range(12):  # wraps the 8-slot tail ring
        k, v = _tokens(rng, B, 1, H, d), _tokens(rng, B, 1, H, d)
        q = rng.standard_normal((B, H * g, d)).astype(np.float32)
        st, bits, got, ref = _step(kvq, torch, gc, oc, k, v, q)
        assert st == 0, (st, bits)
        assert_close(got, ref, what=f"step {step}")
    _check_cache(torch, gc, oc, B, H, d, kt, vt)


def test_fused_steps_ragged_counts():
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    rng = np.random.default_rng(62)
    B, H, g, d, T = 3, 2, 4, 128, 16
    gc = kvq.KVCache(B, H, d, 192, T, "q8_0", "q4_0")
    oc = ko.OracleCache(B, H, d, 192, T, "q8_0", "q4_0", True, True)
    for step in range(10):
        nps = [int(x) for x in rng.integers(0, 5, B)]
        k, v = _tokens(rng, B, 4, H, d), _tokens(rng, B, 4, H, d)
        q = rng.standard_normal((B, H * g, d)).astype(np.float32)
        st, bits, got, ref = _step(kvq, torch, gc, oc, k, v, q, nps=nps)
        assert st == 0, (st, bits)
        assert_close(got, ref, what=f"step {step} {nps}")
    _check_cache(torch, gc, oc, B, H, d, "q8_0", "q4_0")


@pytest.mark.parametrize("case", ["group_16", "n_new_over_tail", "no_tail"])
def test_not_fusable_falls_back(case):
    """More than 8 query heads per KV head, more new tokens than tail slots, or
    no tail: the step runs as append + decode and gives the same results."""
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    rng = np.random.default_rng(63)
    B, H, d = 2, 2, 128
    g = 16 if case == "group_16" else 4
    T = {"group_16": 8, "n_new_over_tail": 4, "no_tail": 0}[case]
    n_new = 6 if case == "n_new_over_tail" else 2
    gc = kvq.KVCache(B, H, d, 128, T, "q4_0", "q8_0")
    oc = ko.OracleCache(B, H, d, 128, T, "q4_0", "q8_0", True, True)
    for step in range(4):
        k, v = _tokens(rng, B, n_new, H, d), _tokens(rng, B, n_new, H, d)
        q = rng.standard_normal((B, H * g, d)).astype(np.float32)
        st, bits, got, ref = _step(kvq, torch, gc, oc, k, v, q)
        assert st == 0, (st, bits)
        assert_close(got, ref, what=f"{case} step {step}")
    _check_cache(torch, gc, oc, B, H, d, "q4_0", "q8_0")


def test_fused_step_range_error_leaves_full_sequence():
    """A sequence whose new tokens would pass max_ctx is not appended (status bit),
    the other sequence is, and the decode attends over what each one holds."""
    torch = require_gpu()
    from rotated_bit_kv_kvq_gb300 import kvq
    rng = np.random.default_rng(64)
    B, H, g, d, T = 2, 1, 4, 64, 16
    gc = kvq.KVCache(B, H, d, 64, T, "q8_0", "q8_0")
    oc = ko.OracleCache(B, H, d, 64, T, "q8_0", "q8_0", True, True)
    pre = _tokens(rng, B, 64, H, d)
    y = prerotate(pre, True)
    kvq.kvq_rotate_quantize_append(gc.desc, to_dev(y, "f32", torch), to_dev(y, "f32", torch),
                                   n_new_per_seq=torch.tensor([64, 10], dtype=torch.int32, device="cuda"),
                                   prerotated=True)
    oc.append(y, y, n_new_per_seq=[64, 10], prerotated=True)
    k, v = _tokens(rng, B, 1, H, d), _tokens(rng, B, 1, H, d)
    q = rng.standard_normal((B, H * g, d)).astype(np.float32)
    yk, yv = prerotate(k, True), prerotate(v, True)
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    ws = torch.empty(kvq.kvq_decode_workspace_bytes(gc.desc, H * g), dtype=torch.uint8, device="cuda")
    kvq.kvq_append_decode(gc.desc, to_dev(yk, "f32", torch), to_dev(yv, "f32", torch), to_dev(q, "f32", torch),
                          out, ws, prerotated=True)
    st, bits = kvq.kvq_sync_status(gc.desc)
    assert st == kvq.KVQ_ERR_DEVICE_RANGE and bits == kvq.KVQ_DEV_ERR_APPEND_RANGE
    assert gc.seq_len.cpu().numpy().tolist() == [64, 11]
    oc.append(yk, yv, n_new_per_seq=[0, 1], prerotated=True)   # the oracle appends what fits
    assert_close(out.cpu().numpy().astype(np.float64), ko.decode_attention(oc, q), what="range error step")
